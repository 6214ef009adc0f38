"""Shared helpers for the -m gpu parity tests: seeded inputs on the device, their
host copies for the oracle, the C-ABI problem struct, and the output tolerance.

Tolerance (stated for this layer): relative L2 error <= 1e-2 and max-abs
error <= 5e-2 x RMS(reference), on the stored bf16 output against the oracle's
unrounded output (block-wise fp8 weights: see assert_close).  Integer and byte outputs
(routing indices, counts, offsets, permutation, fp8 codes) are compared
bit for bit.
"""
from __future__ import annotations

import functools

import re

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


def routing_launches(p) -> int:
    """Kernel launches of S1 + S2 for problem p, from the plan moe_describe
    reports: on the tensor cores prep, GEMM, the sum of its K ranges when there
    are several, top-k; on the CUDA cores router and top-k."""
    mt = re.search(r"router=tensor-cores,k_ranges=(\d+)", lib().moe_describe(p))
    return 2 if mt is None else 3 + (int(mt[1]) > 1)


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


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "",
                 bf16_store_allowance: bool = False):
    """The layer's bars: relative L2 <= REL_L2 and max-abs <= MAX_ABS_RMS x
    output RMS, on the stored bf16 output against the oracle's exact (fp64,
    unrounded) output.

    ``bf16_store_allowance`` is for block-wise fp8 weights only: their 16x block
    gains give outputs of up to ~25x RMS, where the final bf16 store alone
    moves an element by up to half an ulp, ~5% of RMS.  There the max-abs bar
    is applied to |got - ref| minus half a bf16 ulp of ``got``.  Every other
    weight format meets the bar on the raw difference.  The message reports
    both figures."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(ref ** 2))
    err = got - ref
    rel = np.sqrt(np.sum(err ** 2)) / max(np.sqrt(np.sum(ref ** 2)), 1e-30)
    raw = np.max(np.abs(err)) if err.size else 0.0
    adj = np.max(np.abs(err) - bf16_half_ulp(got)) if err.size else 0.0
    mx = adj if bf16_store_allowance else raw
    rms_ = max(rms, 1e-30)
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_RMS * rms, (
        f"{what}: max-abs error {raw / rms_:.4f} x RMS (beyond the bf16 store {adj / rms_:.4f} x RMS)"
        f" > {MAX_ABS_RMS}" + (" [bar applied beyond the bf16 store]" if bf16_store_allowance else ""))
    return rel, raw / rms_


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    """Token sample for full-size checks: first, last and random tokens."""
    if T <= n:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, n - 2, replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(pick), dtype=np.int32)


def edge_tokens(orc, cfg: mi.MoEConfig, h: dict, n: int, seed: int = 0,
                max_experts: int = 1024) -> np.ndarray:
    """Token sample for full-size checks that reaches the kernels' edge paths:
    the token of every expert's last routed row (its last, usually partly
    filled, tile item; at most ``max_experts`` experts, a seeded choice), up to
    32 tokens of the most loaded expert, the first and last tokens, and a
    seeded random fill up to ``n``.  The routing is the oracle's."""
    if cfg.routing == "sigmoid":
        lg = orc.router_logits(h["x"], h["router_w"])
        idx, _ = orc.topk(lg, cfg.k, routing="sigmoid", bias=h["router_bias"])
    else:
        lg = orc.router_logits(h["x"], h["router_w"], h["router_bias"])
        idx, _ = orc.topk(lg, cfg.k)
    cnt, off, _, src = orc.permute(idx, cfg.E)
    rng = np.random.default_rng(seed)
    experts = np.nonzero(cnt)[0]
    if len(experts) > max_experts:
        experts = np.sort(rng.choice(experts, max_experts, replace=False))
    pick = {int(src[off[e + 1] - 1]) for e in experts}
    hot = int(np.argmax(cnt))
    pick |= {int(t) for t in src[off[hot]:off[hot + 1]][:32]}
    pick |= {0, cfg.T - 1}
    rest = np.setdiff1d(np.arange(cfg.T), np.fromiter(pick, np.int64))
    if len(pick) < n and len(rest):
        pick |= {int(t) for t in rng.choice(rest, min(n - len(pick), len(rest)), replace=False)}
    return np.array(sorted(pick), dtype=np.int32)
