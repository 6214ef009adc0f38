"""CPU oracle for the fused MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
``--impl reference`` leg may import this package.  The product path
(``moe_expert_layer_02_gb300``) never imports it, and this package never imports
the product: the two share no code, header, table or constant.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 except where the method
itself rounds); this module is argument marshalling over ``ctypes`` with numpy
arrays.  Sources and readings are listed in the C file's header.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
(exhaustive codec checks against torch casts, brute-force routing, permutation
invariants and a sort by (expert, token), an independent dense all-experts
formulation, an fp64 numpy formulation, a single-expert closed form, and the
printed cost-model numbers).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

FP8 = 0
MXFP4 = 1
FP8_BLOCK = 2
SWIGLU = 0
SITU = 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (plain gcc, no CUDA)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E", ctypes.c_int64), ("k", ctypes.c_int64), ("I_s", ctypes.c_int64),
                ("L", ctypes.c_int64), ("wfmt", ctypes.c_int32), ("shared_bf16", ctypes.c_int32),
                ("rms_eps", ctypes.c_double), ("routing", ctypes.c_int32), ("act", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("x", "router_w", "router_bias", "w13", "w13_scale", "w2", "w2_scale",
                 "sw13", "sw13_scale", "sw2", "sw2_scale", "wd", "wu", "gamma")]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_bf16_decode.restype = ctypes.c_double
        L.orc_bf16_decode.argtypes = [ctypes.c_uint16]
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e8m0_decode.restype = ctypes.c_double
        L.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode_array.argtypes = [P, P, i64]
        L.orc_bf16_from_double_array.argtypes = [P, P, i64]
        L.orc_default_threads.restype = ctypes.c_int
        L.orc_router_logits.argtypes = [i64, i64, i64, P, P, P, P, ctypes.c_int]
        L.orc_topk.argtypes = [i64, i64, ctypes.c_int, P, P, P]
        L.orc_topk_sigmoid.argtypes = [i64, i64, ctypes.c_int, P, P, P, P]
        L.orc_exp_canon.restype = ctypes.c_float
        L.orc_exp_canon.argtypes = [ctypes.c_float]
        L.orc_sigmoid_canon.restype = ctypes.c_float
        L.orc_sigmoid_canon.argtypes = [ctypes.c_float]
        L.orc_permute.argtypes = [i64, i64, ctypes.c_int, P, P, P, P, P]
        L.orc_quant_rows.argtypes = [i64, i64, P, P, P]
        L.orc_moe_forward.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Weights), P, i64,
                                      P, P, P, P, ctypes.c_int]
        L.orc_expert_rows.argtypes = [i32, i32, i64, i64, i64, P, P, P, P, P, P, P, P, P, P, P, P,
                                      ctypes.c_int]
        L.orc_combine.argtypes = [i64, i64, ctypes.c_int, P, P, P, P]
        L.orc_latent_down.argtypes = [i64, i64, P, P, P, i64, P, ctypes.c_int]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    return int(lib().orc_default_threads())


# ----------------------------------------------------------------------------- codecs
def e4m3_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib().orc_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[codes]


def e4m3_encode(v) -> np.ndarray:
    shape = np.shape(v)
    v = _c(v, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_p(v), _p(out), v.size)
    return out.reshape(shape)


def bf16_decode(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_from_double(v) -> np.ndarray:
    shape = np.shape(v)
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_bf16_from_double_array(_p(v), _p(out), v.size)
    return out.reshape(shape)


def e2m1_decode(nibbles) -> np.ndarray:
    nibbles = np.asarray(nibbles, dtype=np.uint8)
    table = np.array([lib().orc_e2m1_decode(c) for c in range(16)], dtype=np.float64)
    return table[nibbles & 15]


def e8m0_decode(s) -> np.ndarray:
    s = np.asarray(s, dtype=np.uint8)
    table = np.array([lib().orc_e8m0_decode(c) for c in range(256)], dtype=np.float64)
    return table[s]


# ----------------------------------------------------------------------------- stages
def router_logits(x_bf16_u16, router_w, bias=None, nthreads: int = 0) -> np.ndarray:
    """S1: fp32 logits [T, E] in the canonical order (see moe_oracle.c)."""
    x = _c(x_bf16_u16, np.uint16)
    wr = _c(router_w, np.float32)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), dtype=np.float32)
    lib().orc_router_logits(T, H, E, _p(x), _p(wr), _p(b), _p(out), nthreads)
    return out


def topk(logits, k: int, routing: str = "softmax", bias=None):
    """S2: (idx int32 [T, k], weights float64 [T, k]).

    routing "softmax": the k largest logits, softmax over them (a bias, if any,
    is already inside the logits).  "sigmoid" (noaux_tc): the k largest
    sigmoid(logit) + bias, weights = the chosen sigmoid scores renormalised."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    if routing == "sigmoid":
        b = None if bias is None else _c(bias, np.float32)
        lib().orc_topk_sigmoid(T, E, k, _p(lg), _p(b), _p(idx), _p(w))
    else:
        assert bias is None
        lib().orc_topk(T, E, k, _p(lg), _p(idx), _p(w))
    return idx, w


def exp_canon(a) -> np.ndarray:
    """The canonical fp32 exp(a), a <= 0, used by sigmoid routing's selection."""
    f = lib().orc_exp_canon
    return np.array([f(float(v)) for v in np.asarray(a, dtype=np.float32).ravel()],
                    dtype=np.float32).reshape(np.shape(a))


def sigmoid_canon(l) -> np.ndarray:
    """The canonical fp32 sigmoid used by sigmoid routing's selection."""
    f = lib().orc_sigmoid_canon
    return np.array([f(float(v)) for v in np.asarray(l, dtype=np.float32).ravel()],
                    dtype=np.float32).reshape(np.shape(l))


def permute(idx, E: int):
    """S3/S4 indices: (cnt [E], off [E+1], perm [T, k], src [T*k])."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    cnt = np.empty(E, dtype=np.int32)
    off = np.empty(E + 1, dtype=np.int32)
    perm = np.empty((T, k), dtype=np.int32)
    src = np.empty(T * k, dtype=np.int32)
    lib().orc_permute(T, E, k, _p(idx), _p(cnt), _p(off), _p(perm), _p(src))
    return cnt, off, perm, src


def quant_rows(x_bf16_u16):
    """Per-token fp8: (scale float32 [T], codes uint8 [T, H])."""
    x = _c(x_bf16_u16, np.uint16)
    T, H = x.shape
    s = np.empty(T, dtype=np.float32)
    q = np.empty((T, H), dtype=np.uint8)
    lib().orc_quant_rows(T, H, _p(x), _p(s), _p(q))
    return s, q


def latent_down(x_bf16_u16, wd_bf16_u16, tokens=None, nthreads: int = 0):
    """LatentMoE down projection z = bf16(x Wd^T) (exact products, fp64 sum,
    one nearest-even rounding) for the listed tokens: uint16 [n, L]."""
    x = _c(x_bf16_u16, np.uint16)
    wd = _c(wd_bf16_u16, np.uint16)
    T, H = x.shape
    L = wd.shape[0]
    assert wd.shape[1] == H
    toks = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    z = np.empty((toks.shape[0], L), dtype=np.uint16)
    lib().orc_latent_down(H, L, _p(x), _p(wd), _p(toks), toks.shape[0], _p(z), nthreads)
    return z


def expert_rows(wfmt, off, xq, xs, row_w, w13, w13_scale, w2, w2_scale, want_h=False,
                nthreads: int = 0, act: int = 0):
    """y[r] = row_w[r] * FFN_{e(r)}(xq[r]) for expert-contiguous rows (fp64);
    act = SWIGLU (0) or SITU (1)."""
    off = _c(off, np.int32)
    xq = _c(xq, np.uint8)
    R, K = xq.shape
    E = off.shape[0] - 1
    I = w13.shape[1] // 2
    xs = _c(xs, np.float32)
    row_w = _c(row_w, np.float32)
    w13 = np.ascontiguousarray(w13)
    w2 = np.ascontiguousarray(w2)
    w13_scale = np.ascontiguousarray(w13_scale)
    w2_scale = np.ascontiguousarray(w2_scale)
    y = np.empty((R, K), dtype=np.float64)
    h = np.empty((R, I), dtype=np.uint16) if want_h else None
    hq = np.empty((R, I), dtype=np.uint8) if want_h else None
    hs = np.empty(R, dtype=np.float32) if want_h else None
    lib().orc_expert_rows(wfmt, act, K, I, E, _p(off), _p(xq), _p(xs), _p(row_w), _p(w13),
                          _p(w13_scale), _p(w2), _p(w2_scale), _p(y), _p(h), _p(hq), _p(hs),
                          nthreads)
    return (y, h, hq, hs) if want_h else y


def combine(y_bf16_u16, perm, shared_bf16_u16=None):
    """S7: out[t] = bf16(sum_j y[perm[t,j]] + shared[t]) (fp64 sum), uint16 bits."""
    y = _c(y_bf16_u16, np.uint16)
    perm = _c(perm, np.int32)
    T, k = perm.shape
    H = y.shape[1]
    sh = None if shared_bf16_u16 is None else _c(shared_bf16_u16, np.uint16)
    out = np.empty((T, H), dtype=np.uint16)
    lib().orc_combine(T, H, k, _p(y), _p(perm), _p(sh), _p(out))
    return out


def moe_forward(prob: dict, w: dict, tokens=None, nthreads: int = 0):
    """The whole layer for the listed tokens.

    ``prob``: T, H, I, E, k, I_s, L, wfmt ('fp8'|'mxfp4'), shared_bf16, rms_eps,
    routing ('softmax'|'sigmoid'), act ('swiglu'|'situ').
    ``w``: numpy arrays keyed like the C struct (bf16 as uint16, fp8/fp4 as uint8).
    Returns (out_f64 [n, H], out_bf16_u16 [n, H], idx [n, k], weights [n, k]).
    """
    P = Problem(T=prob["T"], H=prob["H"], I=prob["I"], E=prob["E"], k=prob["k"],
                I_s=prob.get("I_s", 0), L=prob.get("L", 0),
                wfmt={"fp8": FP8, "mxfp4": MXFP4, "fp8_block": FP8_BLOCK}[prob.get("wfmt", "fp8")],
                shared_bf16=int(bool(prob.get("shared_bf16", False))),
                rms_eps=float(prob.get("rms_eps", 1e-6)),
                routing=1 if prob.get("routing", "softmax") == "sigmoid" else 0,
                act=SITU if prob.get("act", "swiglu") == "situ" else SWIGLU)
    keep = {}

    def ptr(name, dtype=None):
        a = w.get(name)
        if a is None:
            return None
        a = np.ascontiguousarray(a) if dtype is None else _c(a, dtype)
        keep[name] = a
        return a.ctypes.data

    W = Weights(x=ptr("x", np.uint16), router_w=ptr("router_w", np.float32),
                router_bias=ptr("router_bias", np.float32), w13=ptr("w13"),
                w13_scale=ptr("w13_scale"), w2=ptr("w2"), w2_scale=ptr("w2_scale"),
                sw13=ptr("sw13"), sw13_scale=ptr("sw13_scale", np.float32), sw2=ptr("sw2"),
                sw2_scale=ptr("sw2_scale", np.float32), wd=ptr("wd", np.uint16),
                wu=ptr("wu", np.uint16), gamma=ptr("gamma", np.uint16))
    T, H, k = prob["T"], prob["H"], prob["k"]
    toks = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    n = toks.shape[0]
    out_f = np.empty((n, H), dtype=np.float64)
    out_b = np.empty((n, H), dtype=np.uint16)
    idx = np.empty((n, k), dtype=np.int32)
    wt = np.empty((n, k), dtype=np.float64)
    lib().orc_moe_forward(ctypes.byref(P), ctypes.byref(W), _p(toks), n, _p(out_f), _p(out_b),
                          _p(idx), _p(wt), nthreads)
    return out_f, out_b, idx, wt
