"""Shared helpers for the -m gpu parity tests: seeded inputs on the device, their
host copies for the oracle, the C-ABI problem struct, and the output tolerance.

Tolerance (fp32-accumulated output, stated for this layer): relative L2 error
<= 1e-2 and max-abs error <= 5e-2 x RMS(reference).  Integer and byte outputs
(routing indices, counts, offsets, permutation, fp8 codes) are compared
bit for bit.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import moe_inputs as mi

REL_L2 = 1e-2
MAX_ABS_RMS = 5e-2


@functools.lru_cache(maxsize=None)
def lib():
    from moe_expert_layer_02_gb300 import build
    build.build()
    import moe_expert_layer_02_gb300 as m
    m.load_library()
    return m


_weights_cache: dict = {}


def gpu_inputs(cfg: mi.MoEConfig, seed: int = 0) -> dict:
    """Inputs on cuda:0; expert weights are shared between configs of equal shape."""
    key = (cfg.E, cfg.I, cfg.K, cfg.I_s, cfg.wfmt, cfg.shared_bf16, cfg.H, cfg.L, seed)
    reuse = _weights_cache.get(key)
    inp = mi.make_inputs(cfg, device="cuda", seed=seed, expert_weights=reuse)
    if reuse is None:
        _weights_cache.clear()  # keep at most one large weight set resident
        _host_cache.clear()     # its host copies go with it
        _weights_cache[key] = inp
    return inp


_host_cache: dict = {}


def host(inp: dict, keys=None) -> dict:
    """numpy copies for the oracle.  Weight copies are cached per device tensor;
    each entry keeps its tensor alive, so the address in the key cannot be
    handed to a different tensor while the entry exists."""
    out = {}
    for k, v in inp.items():
        if keys is not None and k not in keys:
            continue
        if v is None:
            out[k] = None
            continue
        ck = (k, v.data_ptr(), tuple(v.shape), v.dtype)
        hit = _host_cache.get(ck)
        if k not in ("x", "router_w", "router_bias") and hit is not None and hit[0] is v:
            out[k] = hit[1]
            continue
        a = mi.to_numpy({k: v})[k]
        if k not in ("x", "router_w", "router_bias"):
            _host_cache[ck] = (v, a)
        out[k] = a
    return out


def pack(cfg: mi.MoEConfig, inp: dict) -> dict:
    """The same inputs with expert weights in moe_pack_weights' tile order."""
    m = lib()
    out = dict(inp)
    p = problem(cfg)
    w13p, w2p = torch.empty_like(inp["w13"]), torch.empty_like(inp["w2"])
    if cfg.wfmt == "mxfp4":
        s13p, s2p = torch.empty_like(inp["w13_scale"]), torch.empty_like(inp["w2_scale"])
        m.moe_pack_weights(p, inp["w13"], inp["w2"], inp["w13_scale"], inp["w2_scale"], w13p, w2p,
                           s13p, s2p)
        out.update(w13_scale=s13p, w2_scale=s2p)
    else:
        m.moe_pack_weights(p, inp["w13"], inp["w2"], None, None, w13p, w2p)
    out.update(w13=w13p, w2=w2p)
    if cfg.I_s and not cfg.shared_bf16:
        ps = m.make_problem(cfg.T, cfg.H, cfg.I_s, 1, 1)
        s13, s2 = torch.empty_like(inp["sw13"]), torch.empty_like(inp["sw2"])
        m.moe_pack_weights(ps, inp["sw13"], inp["sw2"], None, None, s13, s2)
        out.update(sw13=s13, sw2=s2)
    torch.cuda.synchronize()
    return out


def problem(cfg: mi.MoEConfig, packed: bool = False):
    m = lib()
    flags = m.F_ROUTER_BIAS if (cfg.zipf_bias or cfg.sel_bias) else 0
    if cfg.routing == "sigmoid":
        flags |= m.F_SIGMOID_ROUTING
    if cfg.act == "situ":
        flags |= m.F_SITU
    if packed:
        flags |= m.F_PACKED_WEIGHTS
    if cfg.shared_bf16:
        flags |= m.F_SHARED_BF16
    return m.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, I_shared=cfg.I_s, latent=cfg.L,
                          wfmt=wfmt_code(cfg), flags=flags)


def wfmt_code(cfg: mi.MoEConfig) -> int:
    m = lib()
    return {"fp8": m.W_FP8, "mxfp4": m.W_MXFP4, "fp8_block": m.W_FP8_BLOCK}[cfg.wfmt]


def workspace(p) -> torch.Tensor:
    n = lib().moe_workspace_bytes(p)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """The bars on the fp32-accumulated output: relative L2 <= REL_L2 and
    max-abs <= MAX_ABS_RMS x output RMS.  ``got`` is the layer's stored bf16
    output, whose final rounding adds at most half a bf16 ulp of each element
    on top of the accumulated value, so the max-abs bar allows that too."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(ref ** 2))
    err = got - ref
    rel = np.sqrt(np.sum(err ** 2)) / max(np.sqrt(np.sum(ref ** 2)), 1e-30)
    excess = np.abs(err) - bf16_half_ulp(got)
    mx = np.max(excess) if err.size else 0.0
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_RMS * rms, (
        f"{what}: max-abs error beyond the bf16 store {mx:.3e} > {MAX_ABS_RMS} x RMS {rms:.3e}")
    return rel, mx / max(rms, 1e-30)


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    """Token sample for full-size checks: first, last and random tokens."""
    if T <= n:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, n - 2, replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(pick), dtype=np.int32)
