"""Python binding of libmoe.so -- the fused MoE expert layer for one GB300.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmoe.so (see include/moe.h for the C ABI).  Functions carry the C names and
take torch tensors on the current CUDA device; they return nothing and raise
``MoEError`` on a non-OK status.  There is no fallback: if the shared library
is missing or fails to load, importing the functions raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MoEError", "MoEProblem", "make_problem", "load_library", "moe_workspace_bytes",
    "moe_router_logits", "moe_route", "moe_permute", "moe_permute_static", "moe_expert_ffn",
    "moe_unpermute", "moe_latent_down", "moe_router_topk",
    "moe_forward", "moe_get_last_error", "moe_launch_count", "moe_profile_enable",
    "moe_profile_read", "moe_pack_weights", "moe_watchdog_selftest", "moe_describe", "STAGES",
    "W_FP8",
    "W_MXFP4", "W_FP8_BLOCK", "F_ROUTER_BIAS", "F_SHARED_BF16", "F_PACKED_WEIGHTS",
    "F_SIGMOID_ROUTING", "F_SITU", "F_FUSED_COMBINE", "MoETuning", "moe_get_tuning",
    "moe_set_tuning", "tuned",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe.so")

W_FP8 = 0
W_MXFP4 = 1
W_FP8_BLOCK = 2
F_ROUTER_BIAS = 0x1
F_SHARED_BF16 = 0x2
F_PACKED_WEIGHTS = 0x4
F_SIGMOID_ROUTING = 0x8
F_SITU = 0x10
F_FUSED_COMBINE = 0x20
STAGES = ("router", "topk", "index", "scatter", "ffn1", "requant", "ffn2", "combine",
          "latent_down", "shared", "latent_up")
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class MoEProblem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("latent", ctypes.c_int32), ("wfmt", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class MoETuning(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("tile_n", "ffn1_gather", "index_3pass", "gemm_1cta",
                                             "pair_small", "mx_1cta", "router_tile", "pdl")]


ROUTER_TILES = {"auto": 0, "8x8": 1, "8x16": 2, "8x16s4": 3, "12w8x16": 4, "tc": 6}


def make_problem(T, H, I, E, top_k, I_shared=0, latent=0, wfmt=W_FP8, flags=0) -> MoEProblem:
    return MoEProblem(T=T, H=H, I=I, E=E, top_k=top_k, I_shared=I_shared, latent=latent,
                      wfmt=wfmt, flags=flags)


_lib = None
_EXPORTS = ("moe_status_string", "moe_workspace_bytes", "moe_router_logits", "moe_route",
            "moe_permute", "moe_permute_static", "moe_expert_ffn", "moe_unpermute", "moe_forward",
            "moe_get_last_error", "moe_launch_count", "moe_profile_enable", "moe_profile_read",
            "moe_pack_weights", "moe_watchdog_selftest", "moe_describe", "moe_latent_down",
            "moe_get_tuning", "moe_set_tuning", "moe_router_topk")


def load_library(path: str = LIB_PATH):
    """Load libmoe.so (build it with moe_expert_layer_02_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so not built at {path}; run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    P, PP = ctypes.c_void_p, ctypes.POINTER(MoEProblem)
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_workspace_bytes.restype = ctypes.c_size_t
    L.moe_workspace_bytes.argtypes = [PP]
    L.moe_router_logits.argtypes = [PP, P, P, P, P, P]
    L.moe_route.argtypes = [PP, P, P, P, P, P]
    L.moe_permute.argtypes = [PP, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    L.moe_permute_static.argtypes = [PP, P, P, P, P, P, P, P, P, P]
    L.moe_pack_weights.argtypes = [PP, P, P, P, P, P, P, P, P, P]
    L.moe_watchdog_selftest.argtypes = [P, P]
    L.moe_describe.argtypes = [PP, ctypes.c_char_p, ctypes.c_size_t]
    L.moe_expert_ffn.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    L.moe_unpermute.argtypes = [PP, P, P, P, P, P]
    L.moe_latent_down.argtypes = [PP, P, P, P, P, ctypes.c_size_t, P]
    L.moe_router_topk.argtypes = [PP, P, P, P, P, P, P, ctypes.c_size_t, P]
    L.moe_get_tuning.argtypes = [ctypes.POINTER(MoETuning)]
    L.moe_set_tuning.argtypes = [ctypes.POINTER(MoETuning)]
    L.moe_forward.argtypes = [PP] + [P] * 16 + [ctypes.c_size_t, P]
    L.moe_get_last_error.argtypes = [P]
    L.moe_launch_count.restype = ctypes.c_int64
    L.moe_profile_enable.argtypes = [ctypes.c_int]
    L.moe_profile_read.argtypes = [P, P]
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def _check(rc: int, where: str):
    if rc != 0:
        raise MoEError(rc, where)


def moe_workspace_bytes(p: MoEProblem) -> int:
    return int(load_library().moe_workspace_bytes(ctypes.byref(p)))


def moe_router_logits(p, x, router_w, bias, logits, stream=None):
    _check(load_library().moe_router_logits(ctypes.byref(p), _ptr(x), _ptr(router_w), _ptr(bias),
                                            _ptr(logits), _stream(stream)), "moe_router_logits")


def moe_route(p, logits, bias, topk_idx, topk_w, stream=None):
    _check(load_library().moe_route(ctypes.byref(p), _ptr(logits), _ptr(bias), _ptr(topk_idx),
                                    _ptr(topk_w), _stream(stream)), "moe_route")


def moe_permute(p, topk_idx, x, counts, offsets, perm, src_row, xq_perm, xscale_perm, ws,
                stream=None):
    _check(load_library().moe_permute(ctypes.byref(p), _ptr(topk_idx), _ptr(x), _ptr(counts),
                                      _ptr(offsets), _ptr(perm), _ptr(src_row), _ptr(xq_perm),
                                      _ptr(xscale_perm), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream)), "moe_permute")


def moe_permute_static(p, topk_idx, x, counts, offsets, perm, src_row, xq_perm, xscale_perm,
                       stream=None):
    """moe_permute for callers that cannot allocate: no workspace argument; the
    scratch is a fixed array inside the library (limit E * ceil(T/32) <= 2^19,
    else MoEError MOE_ERR_WORKSPACE).  Calls that overlap on the GPU race on
    that array; the first call on a device should precede any stream capture."""
    _check(load_library().moe_permute_static(ctypes.byref(p), _ptr(topk_idx), _ptr(x),
                                             _ptr(counts), _ptr(offsets), _ptr(perm),
                                             _ptr(src_row), _ptr(xq_perm), _ptr(xscale_perm),
                                             _stream(stream)), "moe_permute_static")


def moe_expert_ffn(p, offsets, xq_perm, xscale_perm, row_w, w13, w13_scale, w2, w2_scale, y, ws,
                   stream=None):
    _check(load_library().moe_expert_ffn(ctypes.byref(p), _ptr(offsets), _ptr(xq_perm),
                                         _ptr(xscale_perm), _ptr(row_w), _ptr(w13),
                                         _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(y),
                                         _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream)), "moe_expert_ffn")


def moe_pack_weights(p, w13, w2, w13_scale, w2_scale, w13_packed, w2_packed,
                     w13_scale_packed=None, w2_scale_packed=None, stream=None):
    _check(load_library().moe_pack_weights(ctypes.byref(p), _ptr(w13), _ptr(w2), _ptr(w13_scale),
                                           _ptr(w2_scale), _ptr(w13_packed), _ptr(w2_packed),
                                           _ptr(w13_scale_packed), _ptr(w2_scale_packed),
                                           _stream(stream)), "moe_pack_weights")


def moe_unpermute(p, y_rows, perm, shared, out, stream=None):
    _check(load_library().moe_unpermute(ctypes.byref(p), _ptr(y_rows), _ptr(perm), _ptr(shared),
                                        _ptr(out), _stream(stream)), "moe_unpermute")


def moe_router_topk(p, x, router_w, bias, topk_idx, topk_w, ws, stream=None):
    _check(load_library().moe_router_topk(ctypes.byref(p), _ptr(x), _ptr(router_w), _ptr(bias),
                                          _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream)),
           "moe_router_topk")


def moe_latent_down(p, x, latent_down, z, ws, stream=None):
    _check(load_library().moe_latent_down(ctypes.byref(p), _ptr(x), _ptr(latent_down), _ptr(z),
                                          _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(stream)), "moe_latent_down")


def moe_forward(p, x, router_w, router_bias, w13, w13_scale, w2, w2_scale, shared_w13,
                shared_w13_scale, shared_w2, shared_w2_scale, latent_down, latent_up,
                latent_gamma, out, ws, stream=None):
    _check(load_library().moe_forward(
        ctypes.byref(p), _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(w13), _ptr(w13_scale),
        _ptr(w2), _ptr(w2_scale), _ptr(shared_w13), _ptr(shared_w13_scale), _ptr(shared_w2),
        _ptr(shared_w2_scale), _ptr(latent_down), _ptr(latent_up), _ptr(latent_gamma), _ptr(out),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")


def moe_get_last_error(stream=None) -> int:
    return int(load_library().moe_get_last_error(_stream(stream)))


def moe_watchdog_selftest(role_status=None, stream=None):
    _check(load_library().moe_watchdog_selftest(_ptr(role_status), _stream(stream)),
           "moe_watchdog_selftest")


def moe_describe(p) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(load_library().moe_describe(ctypes.byref(p), buf, len(buf)), "moe_describe")
    return buf.value.decode()


def moe_get_tuning() -> dict:
    """The library's launch choices (moe_tuning) as a dict."""
    t = MoETuning()
    _check(load_library().moe_get_tuning(ctypes.byref(t)), "moe_get_tuning")
    return {n: getattr(t, n) for n, _ in MoETuning._fields_}


def moe_set_tuning(**kw):
    """Change some launch choices (names of moe_tuning's fields; router_tile also
    takes the names in ROUTER_TILES); the others keep their current values."""
    cur = moe_get_tuning()
    for k, v in kw.items():
        if k not in cur:
            raise KeyError(k)
        cur[k] = ROUTER_TILES[v] if (k == "router_tile" and isinstance(v, str)) else int(v)
    t = MoETuning(**cur)
    _check(load_library().moe_set_tuning(ctypes.byref(t)), "moe_set_tuning")


class tuned:
    """Context manager: ``with tuned(tile_n=32): ...`` restores the previous
    launch choices on exit."""

    def __init__(self, **kw):
        self.kw = kw

    def __enter__(self):
        self.saved = moe_get_tuning()
        moe_set_tuning(**self.kw)
        return self

    def __exit__(self, *exc):
        moe_set_tuning(**self.saved)
        return False


def moe_launch_count() -> int:
    return int(load_library().moe_launch_count())


def moe_profile_enable(on: bool = True, stages=None):
    """Time every stage (on), the named STAGES only (stages=[...]), or none."""
    mask = 0 if not on else -1 if stages is None else sum(1 << STAGES.index(s) for s in stages)
    load_library().moe_profile_enable(mask)


def moe_profile_read():
    """(ms per stage, launches per stage), each a dict keyed by STAGES names."""
    ms = (ctypes.c_double * len(STAGES))()
    n = (ctypes.c_int64 * len(STAGES))()
    _check(load_library().moe_profile_read(ms, n), "moe_profile_read")
    return dict(zip(STAGES, list(ms))), dict(zip(STAGES, list(n)))
