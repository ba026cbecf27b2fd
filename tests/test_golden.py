"""Hand-worked fixtures under tests/golden/ (each file names the passage it follows)."""
import json
import os

import numpy as np

from oracle import lmoe_oracle as O

G = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(G, name)) as f:
        return json.load(f)


def test_route_hand_examples():
    for c in _load("route_hand_examples.json")["cases"]:
        if isinstance(c["logits"], str):
            E = c["E"]
            logits = np.full((1, E), float(c["logits"].split(":")[1]), np.float32)
            bias = np.zeros(E, np.float32)
        else:
            logits = np.array(c["logits"], np.float32)
            bias = np.array(c["bias"], np.float32)
        ids, w = O.route(logits, bias, c["topk"], c["rsf"], c["renormalize"])
        assert ids.tolist() == c["ids"], c["name"]
        if "weights" in c:
            assert np.allclose(w, c["weights"], rtol=1e-15), c["name"]
        if "weights_all" in c:
            assert np.allclose(w, c["weights_all"], rtol=1e-15), c["name"]
        if "weights_are_sigmoid_of" in c:
            x = np.array(c["weights_are_sigmoid_of"], np.float64)
            assert np.allclose(w, c["rsf"] / (1 + np.exp(-x)), rtol=3e-7), c["name"]


def test_situ_limits():
    d = _load("situ_limits.json")
    for c in d["cases"]:
        got = O.situ(np.array([c["gate"]]), np.array([c["up"]]), d["beta"], c["linear_beta"])[0]
        assert abs(got - c["out"]) <= 1e-12 * max(1.0, abs(c["out"])), c
