"""The C ABI library on the CPU: it loads, exports every declared function, and
its host-side validation rejects bad arguments before touching any device."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from latent_mixture_experts_sigmoid_gb300 import build
    build.build()
    import latent_mixture_experts_sigmoid_gb300 as lm
    return lm.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s+(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_function_is_exported(lib):
    from latent_mixture_experts_sigmoid_gb300 import build, ABI_FUNCTIONS
    decl = declared_functions()
    assert set(ABI_FUNCTIONS) <= set(decl)
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [n for n in decl if n not in exported]
    assert not missing, missing
    for n in decl:
        getattr(lib, n)


def test_status_strings(lib):
    for st in range(-8, 1):
        assert lib.lmoe_status_string(st)
    assert lib.lmoe_status_string(-99) == b"unknown status"
    assert lib.lmoe_abi_version() == 103


def test_route_validation(lib):
    p = ctypes.c_void_p(16)       # never dereferenced: validation fails first
    assert lib.moe_route(p, None, 4, 8, 2, 2, 1, 1, 1.0, p, p, None) == -3
    assert lib.moe_route(p, None, 4, 8, 2, 1, 3, 1, 1.0, p, p, None) == -3
    assert lib.moe_route(p, None, 4, 8, 9, 1, 1, 1, 1.0, p, p, None) == -2    # topk > E
    assert lib.moe_route(p, None, 4, 2000, 8, 1, 1, 1, 1.0, p, p, None) == -2  # E > 1024
    assert lib.moe_route(p, None, 4, 64, 33, 1, 1, 1, 1.0, p, p, None) == -2   # topk > 32
    assert lib.moe_route(None, None, 4, 8, 2, 1, 1, 1, 1.0, p, p, None) == -1
    assert lib.moe_route(ctypes.c_void_p(20), None, 4, 8, 2, 1, 1, 1, 1.0, p, p, None) == -7
    assert lib.moe_route(None, None, 0, 8, 2, 1, 1, 1, 1.0, None, None, None) == 0  # empty


def test_situ_validation(lib):
    p = ctypes.c_void_p(16)
    assert lib.situ_and_mul(p, p, 4, 8, 0.0, 8.0, None) == -4
    assert lib.situ_and_mul(p, p, 4, 8, float("nan"), 8.0, None) == -4
    assert lib.situ_and_mul(p, p, 4, 12, 4.0, 8.0, None) == -2
    assert lib.situ_and_mul(p, p, 0, 8, 4.0, 8.0, None) == 0
    assert lib.masked_situ_and_mul(p, p, p, 4, 8, 8, -1.0, 8.0, None) == -4
    assert lib.masked_situ_and_mul(p, p, None, 4, 8, 8, 4.0, 8.0, None) == -1
    assert lib.masked_situ_and_mul(p, p, p, 0, 8, 8, 4.0, 8.0, None) == 0


def test_layer_validation_and_workspace(lib):
    import workloads as W
    import latent_mixture_experts_sigmoid_gb300 as lm
    d = lm.make_dims(W.TINY)
    n = lib.latent_moe_workspace_bytes(ctypes.byref(d))
    assert n > 0 and n % 256 == 0
    big = lm.make_dims(W.PREFILL)
    assert lib.latent_moe_workspace_bytes(ctypes.byref(big)) > 800 * 2 ** 20
    bad = lm.make_dims(W.TINY)
    bad.beta = 0.0
    assert lib.latent_moe_workspace_bytes(ctypes.byref(bad)) == 0
    w = lm.LmoeWeights()
    p = ctypes.c_void_p(256)
    assert lib.latent_moe_forward(ctypes.byref(bad), ctypes.byref(w), p, p, p, p, n, None, None) == -4
    bad = lm.make_dims(W.TINY)
    bad.n_group = 8
    assert lib.latent_moe_forward(ctypes.byref(bad), ctypes.byref(w), p, p, p, p, n, None, None) == -3
    bad = lm.make_dims(W.TINY)
    bad.T = (1 << 30) // bad.topk + 1          # more expert-major rows than 2^30
    assert lib.latent_moe_workspace_bytes(ctypes.byref(bad)) == 0
    bad = lm.make_dims(W.TINY)
    bad.latent = 100
    assert lib.latent_moe_forward(ctypes.byref(bad), ctypes.byref(w), p, p, p, p, n, None, None) == -2
    # missing weights
    assert lib.latent_moe_forward(ctypes.byref(d), ctypes.byref(w), p, p, p, p, n, None, None) == -1
    w2 = lm.LmoeWeights(256, 256, 256, None, None, None, 256, None)
    # workspace misaligned / too small
    assert lib.latent_moe_forward(ctypes.byref(d), ctypes.byref(w2), p, p, p,
                                  ctypes.c_void_p(272), n, None, None) == -5
    assert lib.latent_moe_forward(ctypes.byref(d), ctypes.byref(w2), p, p, p, p, n - 256, None,
                                  None) == -5
    # shared expert half given
    w3 = lm.LmoeWeights(256, 256, 256, 256, None, None, 256, None)
    assert lib.latent_moe_forward(ctypes.byref(d), ctypes.byref(w3), p, p, p, p, n, None, None) == -1
    z = lm.make_dims(W.TINY)
    z.T = 0
    assert lib.latent_moe_forward(ctypes.byref(z), ctypes.byref(w), None, None, None, None, 0,
                                  None, None) == 0
    # pre-routed form: ids and weights replace the logits
    fr = lib.latent_moe_forward_routed
    assert fr(ctypes.byref(d), ctypes.byref(w2), p, None, p, p, p, n, None, None) == -1
    assert fr(ctypes.byref(d), ctypes.byref(w2), p, p, None, p, p, n, None, None) == -1
    assert fr(ctypes.byref(d), ctypes.byref(w2), p, ctypes.c_void_p(260), p, p, p, n, None,
              None) == -7
    assert fr(ctypes.byref(d), ctypes.byref(w2), p, p, p, p, ctypes.c_void_p(272), n, None,
              None) == -5
    assert fr(ctypes.byref(z), ctypes.byref(w), None, None, None, None, None, 0, None, None) == 0


def test_linear_validation(lib):
    p = ctypes.c_void_p(16)
    assert lib.lmoe_linear(p, p, None, p, 4, 100, 64, None) == -2
    assert lib.lmoe_linear(p, p, None, p, 4, 128, 60, None) == -2
    assert lib.lmoe_linear(None, p, None, p, 4, 128, 64, None) == -1
    assert lib.lmoe_linear(p, p, None, p, 0, 128, 64, None) == 0


def test_package_fails_loudly_without_library(tmp_path):
    import latent_mixture_experts_sigmoid_gb300._binding as b
    saved = b._lib
    try:
        b._lib = None
        with pytest.raises(ImportError):
            b.load_library(str(tmp_path / "missing.so"))
    finally:
        b._lib = saved


def _host_buffer(nbytes, align=256):
    """An aligned view into a numpy host allocation (and the array that owns it)."""
    import numpy as np
    raw = np.zeros(nbytes + align, dtype=np.uint8)
    off = (-raw.ctypes.data) % align
    return raw[off:off + nbytes], raw


def test_host_memory_is_refused_before_any_launch(lib):
    # Every argument valid except where the memory lives: host (pageable)
    # buffers are not device memory of the current device, so each entry point
    # refuses them with LMOE_ERR_DEVICE (-8) and launches nothing.
    import workloads as W
    import latent_mixture_experts_sigmoid_gb300 as lm
    d = lm.make_dims(W.TINY)
    T, H, L, E, k, dI, ds = 8, 256, 128, 64, 4, 128, 128
    keep = []

    def buf(nbytes):
        v, raw = _host_buffer(max(nbytes, 16))
        keep.append(raw)
        return ctypes.c_void_p(v.ctypes.data)

    x, lg, out = buf(T * H * 2), buf(T * E * 4), buf(T * H * 2)
    w = lm.LmoeWeights(buf(L * H * 2).value, buf(E * 2 * dI * L * 2).value,
                       buf(E * L * dI * 2).value, buf(2 * ds * H * 2).value, buf(H * ds * 2).value,
                       None, buf(H * L * 2).value, None)
    n = lib.latent_moe_workspace_bytes(ctypes.byref(d))
    ws = buf(n)
    assert lib.latent_moe_forward(ctypes.byref(d), ctypes.byref(w), x, lg, out, ws, n, None,
                                  None) == -8
    ids, tw = buf(T * k * 4), buf(T * k * 4)
    assert lib.latent_moe_forward_routed(ctypes.byref(d), ctypes.byref(w), x, ids, tw, out, ws, n,
                                         None, None) == -8
    assert lib.latent_moe_forward_noalloc(ctypes.byref(d), ctypes.byref(w), x, lg, out, None,
                                          None) in (-8, -6)   # -6: no device to hold the scratch
    assert lib.moe_route(lg, None, T, E, k, 1, 1, 1, 2.5, ids, tw, None) == -8
    assert lib.situ_and_mul(x, out, 4, 16, 4.0, 8.0, None) == -8
    cnt = buf(16)
    assert lib.masked_situ_and_mul(x, out, cnt, 2, 2, 16, 4.0, 8.0, None) == -8
    assert lib.lmoe_linear(x, buf(128 * 256 * 2), None, out, 8, 128, 256, None) == -8


def test_router_validation(lib):
    p = ctypes.c_void_p(256)
    assert lib.lmoe_router_logits_workspace_bytes(8, 64, 256) > 0
    assert lib.lmoe_router_logits_workspace_bytes(8, 0, 256) == 0          # E < 1
    assert lib.lmoe_router_logits_workspace_bytes(8, 2000, 256) == 0       # E > 1024
    assert lib.lmoe_router_logits_workspace_bytes(8, 64, 100) == 0         # H % 64
    n = lib.lmoe_router_logits_workspace_bytes(8, 64, 256)
    assert lib.lmoe_router_logits(p, p, p, 8, 64, 100, p, n, None) == -2
    assert lib.lmoe_router_logits(None, p, p, 8, 64, 256, p, n, None) == -1
    assert lib.lmoe_router_logits(p, p, ctypes.c_void_p(260), 8, 64, 256, p, n, None) == -7
    assert lib.lmoe_router_logits(p, p, p, 8, 64, 256, p, n - 256, None) == -5
    assert lib.lmoe_router_logits(None, None, None, 0, 64, 256, None, 0, None) == 0
    import workloads as W
    import latent_mixture_experts_sigmoid_gb300 as lm
    d = lm.make_dims(W.TINY)
    w = lm.LmoeWeights(256, 256, 256, None, None, None, 256, None)
    nb = lib.latent_moe_workspace_bytes(ctypes.byref(d))
    fr = lib.latent_moe_forward_router
    assert fr(ctypes.byref(d), ctypes.byref(w), None, p, p, p, nb, None, None) == -1
    assert fr(ctypes.byref(d), ctypes.byref(w), ctypes.c_void_p(264), p, p, p, nb, None,
              None) == -7
    assert fr(ctypes.byref(d), ctypes.byref(w), p, p, p, ctypes.c_void_p(272), nb, None,
              None) == -5
    assert lib.latent_moe_launch_count_router(ctypes.byref(d), 1) == \
        lib.latent_moe_launch_count(ctypes.byref(d), 1) + 1


def test_mxfp4_validation(lib):
    # host-side checks of the MXFP4 entry points, all before any device access
    import dataclasses
    import workloads as W
    import latent_mixture_experts_sigmoid_gb300 as lm
    p = ctypes.c_void_p(256)
    assert lib.lmoe_dequant_mxfp4(p, p, p, 4, 48, None) == -2             # K % 32
    assert lib.lmoe_dequant_mxfp4(p, p, p, -1, 64, None) == -2            # rows < 0
    assert lib.lmoe_dequant_mxfp4(None, p, p, 4, 64, None) == -1
    assert lib.lmoe_dequant_mxfp4(p, p, ctypes.c_void_p(264), 4, 64, None) == -7
    assert lib.lmoe_dequant_mxfp4(None, None, None, 0, 64, None) == 0     # empty
    d = lm.make_dims(W.TINY)
    nb = lib.latent_moe_workspace_bytes_mxfp4(ctypes.byref(d))
    assert nb >= lib.latent_moe_workspace_bytes(ctypes.byref(d))
    # at 300 tokens the T*k/17 slots are every expert
    dp = lm.make_dims(dataclasses.replace(W.TINY, T=300))
    E, L, dI = W.TINY.num_experts, W.TINY.latent, W.TINY.inter
    # above 16 tokens the T*k/17 heavy-expert slots (bf16 weights + tables)
    for T in (16, 17, 128, 129, 256):
        dm = lm.make_dims(dataclasses.replace(W.TINY, T=T))
        extra = (lib.latent_moe_workspace_bytes_mxfp4(ctypes.byref(dm)) -
                 lib.latent_moe_workspace_bytes(ctypes.byref(dm)))
        H = min(E, T * W.TINY.topk // 17) if T > 16 else 0
        assert H * 3 * dI * L * 2 <= extra <= H * 3 * dI * L * 2 + (E + 4 * H + 2) * 4 + 8 * 256
    assert (lib.latent_moe_workspace_bytes_mxfp4(ctypes.byref(dp)) -
            lib.latent_moe_workspace_bytes(ctypes.byref(dp))) >= E * 3 * dI * L * 2
    big = lm.make_dims(dataclasses.replace(W.TINY, inter=4160))
    assert lib.latent_moe_workspace_bytes_mxfp4(ctypes.byref(big)) == 0   # inter > 4096
    wide = lm.make_dims(dataclasses.replace(W.TINY, latent=4224))
    assert lib.latent_moe_workspace_bytes_mxfp4(ctypes.byref(wide)) == 0  # latent > 4096
    w = lm.LmoeWeights(256, None, None, None, None, None, 256, None)     # w13 / w2 unused
    q = lm.LmoeMxfp4Experts(256, 256, 256, 256)
    fwd = lib.latent_moe_forward_mxfp4
    assert fwd(ctypes.byref(d), ctypes.byref(w), None, p, p, p, p, nb, None, None) == -1
    qn = lm.LmoeMxfp4Experts(256, None, 256, 256)
    assert fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(qn), p, p, p, p, nb, None,
               None) == -1
    qa = lm.LmoeMxfp4Experts(264, 256, 256, 256)                          # codes misaligned
    assert fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(qa), p, p, p, p, nb, None,
               None) == -7
    qs = lm.LmoeMxfp4Experts(256, 260, 256, 256)                          # scales misaligned
    assert fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(qs), p, p, p, p, nb, None,
               None) == -7
    assert fwd(ctypes.byref(big), ctypes.byref(w), ctypes.byref(q), p, p, p, p, nb, None,
               None) == -2
    assert fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(q), p, p, p, ctypes.c_void_p(272),
               nb, None, None) == -5
    # without a device the pointers cannot be device memory
    assert fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(q), p, p, p, p, nb, None,
               None) == -8
    # launches: decode replaces GEMM1 + SituGLU and GEMM2 by one kernel each;
    # above 16 tokens (where an expert can get more than 16) the compact
    # dequantization of the heavy experts and their two grouped GEMMs follow;
    # with inter % 128 != 0 above 128 tokens one dequantization kernel of
    # every expert with tokens comes first
    n_bf16 = lib.latent_moe_launch_count(ctypes.byref(d), 1)
    assert lib.latent_moe_launch_count_mxfp4(ctypes.byref(d), 1) == n_bf16
    for T, extra in ((16, 0), (17, 3), (128, 3), (129, 3), (256, 3), (300, 3)):
        dm = lm.make_dims(dataclasses.replace(W.TINY, T=T))
        assert lib.latent_moe_launch_count_mxfp4(ctypes.byref(dm), 1) == \
            lib.latent_moe_launch_count(ctypes.byref(dm), 1) + extra
    dq = lm.make_dims(dataclasses.replace(W.TINY, T=300, inter=192))
    assert lib.latent_moe_launch_count_mxfp4(ctypes.byref(dq), 1) == \
        lib.latent_moe_launch_count(ctypes.byref(dq), 1) + 1
