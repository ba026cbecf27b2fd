"""Thin ctypes binding of liblmoe.so (include/lmoe.h).

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of the computation runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liblmoe.so")

LMOE_OK = 0
LMOE_ERR_NULL = -1
LMOE_ERR_DIM = -2
LMOE_ERR_UNSUPPORTED = -3
LMOE_ERR_BETA = -4
LMOE_ERR_WORKSPACE = -5
LMOE_ERR_CUDA = -6
LMOE_ERR_ALIGN = -7
LMOE_ERR_DEVICE = -8

ABI_FUNCTIONS = ("moe_route", "situ_and_mul", "masked_situ_and_mul", "latent_moe_forward",
                 "latent_moe_forward_routed",
                 "latent_moe_forward_noalloc", "latent_moe_workspace_bytes", "latent_moe_workspace_offsets",
                 "latent_moe_launch_count", "lmoe_linear", "lmoe_status_string",
                 "lmoe_device_error", "lmoe_abi_version", "lmoe_gemm_unit_walk",
                 "lmoe_router_logits", "lmoe_router_logits_workspace_bytes",
                 "latent_moe_forward_router", "latent_moe_launch_count_router",
                 "lmoe_dequant_mxfp4", "latent_moe_workspace_bytes_mxfp4",
                 "latent_moe_forward_mxfp4", "latent_moe_launch_count_mxfp4")


class LmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class LmoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("hidden", ctypes.c_int), ("latent", ctypes.c_int),
                ("num_experts", ctypes.c_int), ("topk", ctypes.c_int), ("inter", ctypes.c_int),
                ("shared_inter", ctypes.c_int), ("n_group", ctypes.c_int),
                ("topk_group", ctypes.c_int), ("renormalize", ctypes.c_int),
                ("routed_scaling_factor", ctypes.c_float), ("beta", ctypes.c_float),
                ("linear_beta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


class LmoeWeights(ctypes.Structure):
    _fields_ = [("w_down", ctypes.c_void_p), ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("ws13", ctypes.c_void_p), ("ws2", ctypes.c_void_p), ("norm_w", ctypes.c_void_p),
                ("w_up", ctypes.c_void_p), ("e_score_correction_bias", ctypes.c_void_p)]


class LmoeMxfp4Experts(ctypes.Structure):
    _fields_ = [("w13_codes", ctypes.c_void_p), ("w13_scales", ctypes.c_void_p),
                ("w2_codes", ctypes.c_void_p), ("w2_scales", ctypes.c_void_p)]


class LmoeDebug(ctypes.Structure):
    _fields_ = [("topk_ids", ctypes.c_void_p), ("topk_weights", ctypes.c_void_p),
                ("expert_num_tokens", ctypes.c_void_p), ("expert_offsets", ctypes.c_void_p),
                ("row_of", ctypes.c_void_p), ("stage_events", ctypes.c_void_p)]


NUM_STAGES = 11
STAGE_NAMES = ("route", "down", "permute", "scatter", "gemm1", "situ", "gemm2", "combine_norm",
               "shared1", "shared2", "up")


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load liblmoe.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"liblmoe.so not built at {p}; run __graft_entry__.build() "
                          "or python -m latent_mixture_experts_sigmoid_gb300.build")
    lib = ctypes.CDLL(p)
    vp, i32, f32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
    lib.moe_route.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, vp, vp]
    lib.moe_route.restype = i32
    lib.situ_and_mul.argtypes = [vp, vp, i64, i32, f32, f32, vp]
    lib.situ_and_mul.restype = i32
    lib.masked_situ_and_mul.argtypes = [vp, vp, vp, i32, i32, i32, f32, f32, vp]
    lib.masked_situ_and_mul.restype = i32
    lib.latent_moe_workspace_bytes.argtypes = [ctypes.POINTER(LmoeDims)]
    lib.latent_moe_workspace_bytes.restype = ctypes.c_size_t
    lib.latent_moe_workspace_offsets.argtypes = [ctypes.POINTER(LmoeDims),
                                                 ctypes.POINTER(ctypes.c_size_t)]
    lib.latent_moe_workspace_offsets.restype = i32
    lib.latent_moe_forward_noalloc.argtypes = [ctypes.POINTER(LmoeDims),
                                               ctypes.POINTER(LmoeWeights), vp, vp, vp,
                                               ctypes.POINTER(LmoeDebug), vp]
    lib.latent_moe_forward_noalloc.restype = i32
    lib.latent_moe_launch_count.argtypes = [ctypes.POINTER(LmoeDims), i32]
    lib.latent_moe_launch_count.restype = i32
    lib.latent_moe_forward.argtypes = [ctypes.POINTER(LmoeDims), ctypes.POINTER(LmoeWeights), vp,
                                       vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(LmoeDebug), vp]
    lib.latent_moe_forward.restype = i32
    lib.latent_moe_forward_routed.argtypes = [ctypes.POINTER(LmoeDims), ctypes.POINTER(LmoeWeights),
                                              vp, vp, vp, vp, vp, ctypes.c_size_t,
                                              ctypes.POINTER(LmoeDebug), vp]
    lib.latent_moe_forward_routed.restype = i32
    lib.lmoe_linear.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
    lib.lmoe_linear.restype = i32
    lib.lmoe_status_string.argtypes = [i32]
    lib.lmoe_status_string.restype = ctypes.c_char_p
    lib.lmoe_device_error.argtypes = [i32]
    lib.lmoe_device_error.restype = i32
    lib.lmoe_abi_version.argtypes = []
    lib.lmoe_abi_version.restype = i32
    lib.lmoe_gemm_unit_walk.argtypes = [i32, vp, i32, i32, vp, i32]
    lib.lmoe_gemm_unit_walk.restype = i32
    lib.lmoe_router_logits_workspace_bytes.argtypes = [i32, i32, i32]
    lib.lmoe_router_logits_workspace_bytes.restype = ctypes.c_size_t
    lib.lmoe_router_logits.argtypes = [vp, vp, vp, i32, i32, i32, vp, ctypes.c_size_t, vp]
    lib.lmoe_router_logits.restype = i32
    lib.latent_moe_forward_router.argtypes = [ctypes.POINTER(LmoeDims), ctypes.POINTER(LmoeWeights),
                                              vp, vp, vp, vp, ctypes.c_size_t,
                                              ctypes.POINTER(LmoeDebug), vp]
    lib.latent_moe_forward_router.restype = i32
    lib.latent_moe_launch_count_router.argtypes = [ctypes.POINTER(LmoeDims), i32]
    lib.latent_moe_launch_count_router.restype = i32
    lib.lmoe_dequant_mxfp4.argtypes = [vp, vp, vp, i64, i32, vp]
    lib.lmoe_dequant_mxfp4.restype = i32
    lib.latent_moe_workspace_bytes_mxfp4.argtypes = [ctypes.POINTER(LmoeDims)]
    lib.latent_moe_workspace_bytes_mxfp4.restype = ctypes.c_size_t
    lib.latent_moe_forward_mxfp4.argtypes = [ctypes.POINTER(LmoeDims), ctypes.POINTER(LmoeWeights),
                                             ctypes.POINTER(LmoeMxfp4Experts), vp, vp, vp, vp,
                                             ctypes.c_size_t, ctypes.POINTER(LmoeDebug), vp]
    lib.latent_moe_forward_mxfp4.restype = i32
    lib.latent_moe_launch_count_mxfp4.argtypes = [ctypes.POINTER(LmoeDims), i32]
    lib.latent_moe_launch_count_mxfp4.restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().lmoe_status_string(int(status)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_BF16 = (torch.bfloat16, torch.int16)   # bf16 values, or their raw 16-bit patterns


def _dev(t, name: str, dtypes, numel: int) -> int | None:
    """Device address of a tensor argument, after checking that the kernels can
    access it as the C ABI describes: a contiguous tensor on the current CUDA
    device, of one of `dtypes`, holding at least `numel` elements.  None and raw
    integer addresses pass through unchecked (the caller vouches for them)."""
    if t is None or isinstance(t, int):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor, an address or None")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (got device {t.device})")
    if t.get_device() != torch.cuda.current_device():
        raise ValueError(f"{name}: on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.dtype not in (dtypes if isinstance(dtypes, tuple) else (dtypes,)):
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtypes}")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, needs at least {numel}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != LMOE_OK:
        raise LmoeError(status, what)


def moe_route(router_logits, e_score_correction_bias, topk: int, routed_scaling_factor: float,
              topk_ids, topk_weights, renormalize: int = 1, n_group: int = 1,
              topk_group: int = 1, stream=None, T: int | None = None, E: int | None = None):
    """Single-group sigmoid top-k routing; writes topk_ids [T,k] and topk_weights [T,k]."""
    if T is None:
        T, E = router_logits.shape
    T, E, k = int(T), int(E), int(topk)
    st = load_library().moe_route(_dev(router_logits, "router_logits", torch.float32, T * E),
                                  _dev(e_score_correction_bias, "e_score_correction_bias",
                                       torch.float32, E),
                                  T, E, k, int(n_group), int(topk_group),
                                  int(renormalize), float(routed_scaling_factor),
                                  _dev(topk_ids, "topk_ids", torch.int32, T * k),
                                  _dev(topk_weights, "topk_weights", torch.float32, T * k),
                                  _stream(stream))
    _check(st, "moe_route")


def situ_and_mul(inp, out, beta: float, linear_beta: float, stream=None,
                 N: int | None = None, d: int | None = None):
    """SituGLU over a dense [N, 2d] bf16 tensor into out [N, d]."""
    if N is None:
        d = inp.shape[-1] // 2
        N = inp.numel() // (2 * d)
    N, d = int(N), int(d)
    st = load_library().situ_and_mul(_dev(inp, "input", _BF16, N * 2 * d),
                                      _dev(out, "out", _BF16, N * d), N, d, float(beta),
                                      float(linear_beta), _stream(stream))
    _check(st, "situ_and_mul")


def masked_situ_and_mul(inp, out, expert_num_tokens, beta: float, linear_beta: float,
                        stream=None, shape: tuple | None = None):
    """SituGLU over the batched [E, T_max, 2d] layout; padded rows untouched."""
    E, T_max, two_d = (int(v) for v in (shape if shape is not None else tuple(inp.shape)))
    st = load_library().masked_situ_and_mul(
        _dev(inp, "input", _BF16, E * T_max * two_d),
        _dev(out, "out", _BF16, E * T_max * (two_d // 2)),
        _dev(expert_num_tokens, "expert_num_tokens", torch.int32, E),
        E, T_max, two_d // 2, float(beta), float(linear_beta), _stream(stream))
    _check(st, "masked_situ_and_mul")


def make_dims(d) -> LmoeDims:
    """LmoeDims from any object with the lmoe_dims field names."""
    return LmoeDims(int(d.T), int(d.hidden), int(d.latent), int(d.num_experts), int(d.topk),
                    int(d.inter), int(d.shared_inter), int(d.n_group), int(d.topk_group),
                    int(d.renormalize), float(d.routed_scaling_factor), float(d.beta),
                    float(d.linear_beta), float(d.rms_eps))


def make_weights(w: dict, dims=None) -> LmoeWeights:
    """LmoeWeights from a dict of tensors (or addresses); with `dims` every
    tensor is checked against the size lmoe_weights documents for it."""
    if dims is None:
        g = lambda k: _ptr(w.get(k))  # noqa: E731
        return LmoeWeights(g("w_down"), g("w13"), g("w2"), g("ws13"), g("ws2"), g("norm_w"),
                           g("w_up"), g("bias"))
    H, L, E, dI, ds = (int(dims.hidden), int(dims.latent), int(dims.num_experts),
                       int(dims.inter), int(dims.shared_inter))
    need = {"w_down": L * H, "w13": E * 2 * dI * L, "w2": E * L * dI, "ws13": 2 * ds * H,
            "ws2": H * ds, "norm_w": L, "w_up": H * L}
    g = {k: _dev(w.get(k), k, _BF16, n) for k, n in need.items()}
    return LmoeWeights(g["w_down"], g["w13"], g["w2"], g["ws13"], g["ws2"], g["norm_w"],
                       g["w_up"], _dev(w.get("bias"), "bias", torch.float32, E))


def _workspace(workspace, workspace_bytes):
    """(address, byte count) of a workspace tensor, checked to hold the bytes
    claimed for it (the whole tensor when workspace_bytes is None)."""
    if workspace is None or isinstance(workspace, int):
        return workspace, int(workspace_bytes or 0)
    have = workspace.numel() * workspace.element_size()
    n = have if workspace_bytes is None else int(workspace_bytes)
    if n > have:
        raise ValueError(f"workspace: {have} bytes, {n} claimed")
    _dev(workspace, "workspace", (workspace.dtype,), 0)
    return workspace.data_ptr(), n


def latent_moe_workspace_bytes(dims) -> int:
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    return int(load_library().latent_moe_workspace_bytes(ctypes.byref(dd)))


def latent_moe_forward(dims, weights, hidden, router_logits, out, workspace,
                       workspace_bytes: int | None = None, debug: dict | None = None,
                       stream=None):
    """The latent-MoE layer forward; writes out [T, hidden] bf16."""
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    ww = weights if isinstance(weights, LmoeWeights) else make_weights(weights, dd)
    T, H, E = int(dd.T), int(dd.hidden), int(dd.num_experts)
    wsp, wsn = _workspace(workspace, workspace_bytes)
    dbg, keep = _debug_struct(debug, dd)
    st = load_library().latent_moe_forward(
        ctypes.byref(dd), ctypes.byref(ww), _dev(hidden, "hidden", _BF16, T * H),
        _dev(router_logits, "router_logits", torch.float32, T * E),
        _dev(out, "out", _BF16, T * H), wsp, wsn,
        ctypes.byref(dbg) if dbg is not None else None, _stream(stream))
    _check(st, "latent_moe_forward")


def _debug_struct(debug, dd):
    """LmoeDebug for a dict of optional outputs (and the event array it points to)."""
    if not debug:
        return None, None
    T, k, E = int(dd.T), int(dd.topk), int(dd.num_experts)
    ev = debug.get("stage_events")
    ev_arr = None
    if ev is not None:
        for e in ev:                  # torch creates the CUDA event on first record
            if not e.cuda_event:
                e.record()
        ev_arr = (ctypes.c_void_p * len(ev))(*[e.cuda_event for e in ev])
    dbg = LmoeDebug(_dev(debug.get("topk_ids"), "topk_ids", torch.int32, T * k),
                    _dev(debug.get("topk_weights"), "topk_weights", torch.float32, T * k),
                    _dev(debug.get("expert_num_tokens"), "expert_num_tokens", torch.int32, E),
                    _dev(debug.get("expert_offsets"), "expert_offsets", torch.int32, E + 1),
                    _dev(debug.get("row_of"), "row_of", torch.int32, T * k),
                    ctypes.cast(ev_arr, ctypes.c_void_p) if ev_arr is not None else None)
    return dbg, ev_arr


def latent_moe_forward_routed(dims, weights, hidden, topk_ids, topk_weights, out, workspace,
                              workspace_bytes: int | None = None, debug: dict | None = None,
                              stream=None):
    """The layer forward on routing done ahead (topk_ids [T,k] int32 and
    topk_weights [T,k] fp32 as moe_route writes them); skips the routing kernel."""
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    ww = weights if isinstance(weights, LmoeWeights) else make_weights(weights, dd)
    T, H, k = int(dd.T), int(dd.hidden), int(dd.topk)
    wsp, wsn = _workspace(workspace, workspace_bytes)
    dbg, keep = _debug_struct(debug, dd)
    st = load_library().latent_moe_forward_routed(
        ctypes.byref(dd), ctypes.byref(ww), _dev(hidden, "hidden", _BF16, T * H),
        _dev(topk_ids, "topk_ids", torch.int32, T * k),
        _dev(topk_weights, "topk_weights", torch.float32, T * k),
        _dev(out, "out", _BF16, T * H), wsp, wsn,
        ctypes.byref(dbg) if dbg is not None else None, _stream(stream))
    _check(st, "latent_moe_forward_routed")


def lmoe_linear(x, w, out, add=None, stream=None, T: int | None = None, N: int | None = None,
                K: int | None = None):
    """out [T,N] = bf16(x [T,K] @ w [N,K]^T (+ add)) on the tensor-core GEMM."""
    if T is None:
        T, K = x.shape
        N = w.shape[0]
    T, N, K = int(T), int(N), int(K)
    st = load_library().lmoe_linear(_dev(x, "x", _BF16, T * K), _dev(w, "w", _BF16, N * K),
                                    _dev(add, "add", _BF16, T * N), _dev(out, "out", _BF16, T * N),
                                    T, N, K, _stream(stream))
    _check(st, "lmoe_linear")


def latent_moe_forward_noalloc(dims, weights, hidden, router_logits, out, stream=None):
    """The layer forward with the library's own 32 MiB device scratch instead
    of a caller workspace, for callers that cannot allocate device memory.
    Calls that need more scratch raise LmoeError (LMOE_ERR_WORKSPACE); calls
    that overlap on the GPU share the scratch and race."""
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    ww = weights if isinstance(weights, LmoeWeights) else make_weights(weights, dd)
    T, H, E = int(dd.T), int(dd.hidden), int(dd.num_experts)
    st = load_library().latent_moe_forward_noalloc(
        ctypes.byref(dd), ctypes.byref(ww), _dev(hidden, "hidden", _BF16, T * H),
        _dev(router_logits, "router_logits", torch.float32, T * E),
        _dev(out, "out", _BF16, T * H), None, _stream(stream))
    _check(st, "latent_moe_forward_noalloc")


WS_NAMES = ("topk_ids", "topk_weights", "counts", "offsets", "row_of", "Z", "A", "G", "act",
            "Y", "N", "Gs", "As", "Sh", "logits")


def latent_moe_workspace_offsets(dims) -> dict:
    """Byte offsets of the intermediate buffers inside the workspace."""
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    arr = (ctypes.c_size_t * len(WS_NAMES))()
    _check(load_library().latent_moe_workspace_offsets(ctypes.byref(dd), arr),
           "latent_moe_workspace_offsets")
    return dict(zip(WS_NAMES, [int(v) for v in arr]))


def latent_moe_launch_count(dims, has_shared_expert: bool = True) -> int:
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    return int(load_library().latent_moe_launch_count(ctypes.byref(dd), 1 if has_shared_expert else 0))


def lmoe_device_error(clear: bool = False) -> int:
    return int(load_library().lmoe_device_error(1 if clear else 0))


def lmoe_abi_version() -> int:
    return int(load_library().lmoe_abi_version())


def gemm_unit_walk(counts, nfeat: int, paired: bool):
    """Work-unit walk of the grouped GEMM (tokens on M) for per-group token
    counts: int32 [units, 1 + paired, 5] of (first token row, valid rows,
    first weight row, feature tile, shares-token-tile).  Host only."""
    import numpy as np
    c = np.ascontiguousarray(counts, dtype=np.int32)
    lib = load_library()
    n = lib.lmoe_gemm_unit_walk(len(c), c.ctypes.data, nfeat, int(paired), None, 0)
    if n < 0:
        raise LmoeError(n, "lmoe_gemm_unit_walk")
    out = np.zeros((n, 1 + int(paired), 5), dtype=np.int32)
    _check(min(0, lib.lmoe_gemm_unit_walk(len(c), c.ctypes.data, nfeat, int(paired),
                                          out.ctypes.data, n)), "lmoe_gemm_unit_walk")
    return out


def lmoe_router_logits_workspace_bytes(T: int, E: int, H: int) -> int:
    return int(load_library().lmoe_router_logits_workspace_bytes(int(T), int(E), int(H)))


def lmoe_router_logits(hidden, w_router, logits, workspace, stream=None,
                       T: int | None = None, E: int | None = None, H: int | None = None):
    """Router GEMM: logits [T, E] fp32 = hidden [T, H] @ w_router [E, H]^T."""
    if T is None:
        T, H = hidden.shape
        E = w_router.shape[0]
    T, E, H = int(T), int(E), int(H)
    wsp, wsn = _workspace(workspace, None)
    st = load_library().lmoe_router_logits(_dev(hidden, "hidden", _BF16, T * H),
                                           _dev(w_router, "w_router", _BF16, E * H),
                                           _dev(logits, "logits", torch.float32, T * E),
                                           T, E, H, wsp, wsn, _stream(stream))
    _check(st, "lmoe_router_logits")


def latent_moe_forward_router(dims, weights, w_router, hidden, out, workspace,
                              workspace_bytes: int | None = None, debug: dict | None = None,
                              stream=None):
    """The layer forward with its router GEMM (logits = hidden @ w_router^T)."""
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    ww = weights if isinstance(weights, LmoeWeights) else make_weights(weights, dd)
    T, H, E = int(dd.T), int(dd.hidden), int(dd.num_experts)
    wsp, wsn = _workspace(workspace, workspace_bytes)
    dbg, keep = _debug_struct(debug, dd)
    st = load_library().latent_moe_forward_router(
        ctypes.byref(dd), ctypes.byref(ww), _dev(w_router, "w_router", _BF16, E * H),
        _dev(hidden, "hidden", _BF16, T * H), _dev(out, "out", _BF16, T * H), wsp, wsn,
        ctypes.byref(dbg) if dbg is not None else None, _stream(stream))
    _check(st, "latent_moe_forward_router")


def latent_moe_launch_count_router(dims, has_shared_expert: bool = True) -> int:
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    return int(load_library().latent_moe_launch_count_router(ctypes.byref(dd),
                                                              1 if has_shared_expert else 0))


# --- block-scaled (MXFP4) routed experts -------------------------------------------


def lmoe_dequant_mxfp4(codes, scales, out, stream=None, rows: int | None = None,
                       K: int | None = None):
    """out [rows, K] bf16 = E2M1(codes) * 2^(scales - 127); codes uint8
    [rows, K/2] (element 2i in the low nibble), scales uint8 [rows, K/32]."""
    if rows is None:
        K = out.shape[-1]
        rows = out.numel() // K
    rows, K = int(rows), int(K)
    st = load_library().lmoe_dequant_mxfp4(_dev(codes, "codes", torch.uint8, rows * K // 2),
                                           _dev(scales, "scales", torch.uint8, rows * K // 32),
                                           _dev(out, "out", _BF16, rows * K), rows, K,
                                           _stream(stream))
    _check(st, "lmoe_dequant_mxfp4")


def make_mxfp4_experts(q: dict, dims=None) -> LmoeMxfp4Experts:
    """LmoeMxfp4Experts from a dict with w13_q, w13_s, w2_q, w2_s (uint8
    tensors; with `dims` each is checked against its documented size)."""
    names = ("w13_q", "w13_s", "w2_q", "w2_s")
    if dims is None:
        return LmoeMxfp4Experts(*[_ptr(q.get(n)) for n in names])
    E, L, dI = int(dims.num_experts), int(dims.latent), int(dims.inter)
    need = (E * 2 * dI * L // 2, E * 2 * dI * L // 32, E * L * dI // 2, E * L * dI // 32)
    return LmoeMxfp4Experts(*[_dev(q.get(n), n, torch.uint8, c) for n, c in zip(names, need)])


def latent_moe_workspace_bytes_mxfp4(dims) -> int:
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    return int(load_library().latent_moe_workspace_bytes_mxfp4(ctypes.byref(dd)))


def latent_moe_forward_mxfp4(dims, weights, experts, hidden, router_logits, out, workspace,
                             workspace_bytes: int | None = None, debug: dict | None = None,
                             stream=None):
    """The layer forward with MXFP4 routed experts (weights' w13 / w2 unused)."""
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    if isinstance(weights, LmoeWeights):
        ww = weights
    else:
        ww = make_weights(dict(weights, w13=None, w2=None), dd)
    qq = experts if isinstance(experts, LmoeMxfp4Experts) else make_mxfp4_experts(experts, dd)
    T, H, E = int(dd.T), int(dd.hidden), int(dd.num_experts)
    wsp, wsn = _workspace(workspace, workspace_bytes)
    dbg, keep = _debug_struct(debug, dd)
    st = load_library().latent_moe_forward_mxfp4(
        ctypes.byref(dd), ctypes.byref(ww), ctypes.byref(qq), _dev(hidden, "hidden", _BF16, T * H),
        _dev(router_logits, "router_logits", torch.float32, T * E),
        _dev(out, "out", _BF16, T * H), wsp, wsn,
        ctypes.byref(dbg) if dbg is not None else None, _stream(stream))
    _check(st, "latent_moe_forward_mxfp4")


def latent_moe_launch_count_mxfp4(dims, has_shared_expert: bool = True) -> int:
    dd = dims if isinstance(dims, LmoeDims) else make_dims(dims)
    return int(load_library().latent_moe_launch_count_mxfp4(ctypes.byref(dd),
                                                             1 if has_shared_expert else 0))
