"""Seeded synthetic inputs for the fused MoE expert layer.

This module is the one thing the CUDA path's tests and the CPU oracle share: it
draws the inputs and prepares the weight bytes, and holds none of the layer's
own arithmetic (no routing, no activation quantisation, no GEMM, no combine).
Weight quantisation here is input preparation (the layer consumes weights that
are already quantised); it uses torch's own float8 cast for fp8 and the OCP MX
v1.0 recipe for MXFP4, and both sides read the same resulting bytes.

Workloads (shapes from the Ling-2.6-1T Fused MoE V2 write-up, s.1 cost model,
and the Kimi-K3 feasibility report, s.2.4 LatentMoE / s.2.5 MXFP4):

=========  =====  ====  ====  ===  ==  ====  ====  ======  ====================
name         T     H     I     E   k   I_s    L   weights  notes
=========  =====  ====  ====  ===  ==  ====  ====  ======  ====================
toy           64   256   128    8   2     0     0  fp8     CPU-sized
decode       512  8192  2048  256   8  2048     0  fp8     Ling decode batch
prefill    16384  8192  2048  256   8  2048     0  fp8     Ling prefill
latent      4096  7168  3072  896  16  6144  3584  mxfp4   K3 LatentMoE
skewed      8192  8192  2048  256   8  2048     0  fp8     Zipf(1.2) router bias
=========  =====  ====  ====  ===  ==  ====  ====  ======  ====================

Recipe (seed 0 unless stated): x ~ N(0,1) -> bf16; router W ~ N(0, 1/H) fp32;
W1/W3 [E, I, K] ~ N(0, 1/K), W2 [E, K, I] ~ N(0, 1/I) (K = H, or L for the
latent case); fp8 weights use a per-output-channel fp32 scale amax/448; MXFP4
weights use a shared e8m0 exponent floor(log2 amax) - 2 per 32 elements along
the reduction axis, elements rounded to nearest-even e2m1 and clamped to +-6,
two nibbles per byte with the even index in the low nibble.  The skewed case
adds bias[e] = 2 * log p_{rank(e)}, p_r proportional to r^-1.2, rank a seeded
permutation.  x, router and bias come from one CPU generator; each expert's
weights come from a generator on the target device seeded with
(seed << 20) + e, so multi-GB weight sets never need an fp32 host copy.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    I_s: int = 0          # shared-expert intermediate width; 0 = none
    L: int = 0            # latent width; 0 = no latent projection
    wfmt: str = "fp8"     # routed expert weights: "fp8" | "mxfp4" | "fp8_block" (128 x 128)
    shared_bf16: bool = False
    zipf_bias: bool = False
    rms_eps: float = 1e-6
    routing: str = "softmax"  # "softmax" top-k | "sigmoid" (noaux_tc, selection bias)
    act: str = "swiglu"       # "swiglu" | "situ" (beta = 4)
    sel_bias: bool = False    # noaux_tc selection bias ~ N(0, 0.005^2) per expert

    @property
    def K(self) -> int:   # expert input/output width
        return self.L if self.L else self.H

    @property
    def R(self) -> int:   # routed rows
        return self.T * self.k

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)

    def oracle_problem(self) -> dict:
        return dict(T=self.T, H=self.H, I=self.I, E=self.E, k=self.k, I_s=self.I_s, L=self.L,
                    wfmt=self.wfmt, shared_bf16=self.shared_bf16, rms_eps=self.rms_eps,
                    routing=self.routing, act=self.act)


CONFIGS = {
    "toy": MoEConfig("toy", T=64, H=256, I=128, E=8, k=2),
    "decode": MoEConfig("decode", T=512, H=8192, I=2048, E=256, k=8, I_s=2048),
    "prefill": MoEConfig("prefill", T=16384, H=8192, I=2048, E=256, k=8, I_s=2048),
    "latent": MoEConfig("latent", T=4096, H=7168, I=3072, E=896, k=16, I_s=6144, L=3584,
                        wfmt="mxfp4", shared_bf16=True),
    "skewed": MoEConfig("skewed", T=8192, H=8192, I=2048, E=256, k=8, I_s=2048, zipf_bias=True),
    # the decode workload with block-wise fp8 experts (128 x 128 weight blocks,
    # the format tpu-inference requires)
    "decode_block": MoEConfig("decode_block", T=512, H=8192, I=2048, E=256, k=8, I_s=2048,
                              wfmt="fp8_block"),
    # the LatentMoE workload with Kimi K3's own routing and activation (noaux_tc
    # sigmoid routing with a selection bias, SiTU experts)
    "latent_k3": MoEConfig("latent_k3", T=4096, H=7168, I=3072, E=896, k=16, I_s=6144, L=3584,
                           wfmt="mxfp4", shared_bf16=True, routing="sigmoid", act="situ",
                           sel_bias=True),
    # profiling stand-in for "decode": same expert shapes and ~16 rows per
    # expert, 32 experts (1.6 GB of weights: above L2, small enough to capture)
    "decode_e32": MoEConfig("decode_e32", T=64, H=8192, I=2048, E=32, k=8, I_s=2048),
    # profiling stand-in for "latent": ~72 rows per expert, 64 experts
    "latent_e64": MoEConfig("latent_e64", T=288, H=7168, I=3072, E=64, k=16, I_s=6144, L=3584,
                            wfmt="mxfp4", shared_bf16=True),
    # profiling stand-in for "prefill": ~512 rows per expert, 32 experts
    "prefill_e32": MoEConfig("prefill_e32", T=2048, H=8192, I=2048, E=32, k=8, I_s=2048),
    # between decode and prefill: Ling shapes, ~64 rows per expert (64-row
    # tiles on single SMs)
    "mid": MoEConfig("mid", T=2048, H=8192, I=2048, E=256, k=8, I_s=2048),
}


# ----------------------------------------------------------------------------- weight prep
def quantize_fp8_rows(w: torch.Tensor):
    """Per-row (output channel) fp8 e4m3: scale = amax/448, bytes via torch's cast."""
    w = w.float()
    amax = w.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (w / scale[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale.float()


def quantize_fp8_blocks(w: torch.Tensor):
    """Block-wise fp8 e4m3 over 128 x 128 blocks: scale [R/128, C/128] = amax/448
    of the block (1 if zero), bytes via torch's cast of w / scale."""
    w = w.float()
    R, C = w.shape
    b = w.view(R // 128, 128, C // 128, 128)
    amax = b.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (b / scale[:, None, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(R, C)
    return q.view(torch.uint8), scale.float()


def _block_gain(R: int, C: int, gen, device):
    """A seeded gain 2^u, u ~ U(-2, 2), per 128 x 128 block, so that block scales
    differ (up to 16x) as they do in trained weights."""
    u = torch.rand(R // 128, C // 128, generator=gen, device=device) * 4.0 - 2.0
    return torch.pow(2.0, u).repeat_interleave(128, 0).repeat_interleave(128, 1)


_E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def quantize_mxfp4_rows(w: torch.Tensor):
    """OCP MX v1.0 MXFP4 along each row (blocks of 32): packed bytes + e8m0 scales."""
    w = w.float()
    rows, K = w.shape
    assert K % 32 == 0
    blk = w.view(rows, K // 32, 32)
    amax = blk.abs().amax(dim=2)
    safe = torch.where(amax > 0, amax, torch.ones_like(amax))
    exp = (torch.floor(torch.log2(safe)) - 2).clamp(-127, 127)
    exp = torch.where(amax > 0, exp, torch.full_like(exp, -127))
    v = blk / torch.exp2(exp)[..., None]
    mids = torch.tensor(_E2M1_MIDS, device=w.device)
    a = v.abs()
    code = torch.bucketize(a, mids, right=False)
    tie = (code < 7) & (a == mids[code.clamp(max=6)])
    code = torch.where(tie & (code % 2 == 1), code + 1, code)
    nib = (code | torch.where(v < 0, 8, 0)).to(torch.uint8).view(rows, K)
    packed = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return packed.contiguous(), (exp + 127).to(torch.uint8).contiguous()


def _bf16_randn(shape, fan_in, gen, device):
    return (torch.randn(shape, generator=gen, device=device) / math.sqrt(fan_in)).to(torch.bfloat16)


def make_inputs(cfg: MoEConfig, device="cpu", seed: int = 0, expert_weights: dict | None = None) -> dict:
    """All layer inputs for ``cfg`` as torch tensors on ``device``.

    Keys: x (bf16 [T,H]), router_w (f32 [E,H]), router_bias (f32 [E] or None),
    w13 / w2 (uint8 bytes), w13_scale / w2_scale (f32 for fp8, uint8 e8m0 for
    mxfp4), sw13 / sw2 (+ scales for fp8; bf16 when shared_bf16), wd / wu / gamma
    (latent case, bf16).  ``expert_weights`` (a previous result for the same
    E, I, K, I_s, weight format and seed) is reused instead of regenerating the
    expert, shared and latent weights, which depend only on those.
    """
    device = torch.device(device)
    g = torch.Generator().manual_seed(seed)
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    out = {}
    out["x"] = torch.randn(T, H, generator=g).to(torch.bfloat16).to(device)
    out["router_w"] = (torch.randn(E, H, generator=g) / math.sqrt(H)).to(device)
    out["router_bias"] = None
    if cfg.zipf_bias:
        rank = torch.randperm(E, generator=g).double() + 1.0
        p = rank.pow(-1.2)
        p = p / p.sum()
        out["router_bias"] = (2.0 * torch.log(p)).float().to(device)
    if cfg.sel_bias:
        # noaux_tc's correction bias exists to balance expert load; at this size
        # it changes most tokens' selections (~70% at the K3 shape) while the
        # per-expert load stays near the unbiased spread (max 133 vs 103 rows)
        out["router_bias"] = (0.005 * torch.randn(E, generator=g)).float().to(device)

    if expert_weights is not None:
        for key in ("w13", "w13_scale", "w2", "w2_scale", "sw13", "sw13_scale", "sw2",
                    "sw2_scale", "wd", "wu", "gamma"):
            out[key] = expert_weights[key]
        return out

    if cfg.wfmt == "fp8":
        w13 = torch.empty(E, 2 * I, K, dtype=torch.uint8, device=device)
        w13s = torch.empty(E, 2 * I, dtype=torch.float32, device=device)
        w2 = torch.empty(E, K, I, dtype=torch.uint8, device=device)
        w2s = torch.empty(E, K, dtype=torch.float32, device=device)
    elif cfg.wfmt == "fp8_block":
        w13 = torch.empty(E, 2 * I, K, dtype=torch.uint8, device=device)
        w13s = torch.empty(E, 2 * I // 128, K // 128, dtype=torch.float32, device=device)
        w2 = torch.empty(E, K, I, dtype=torch.uint8, device=device)
        w2s = torch.empty(E, K // 128, I // 128, dtype=torch.float32, device=device)
    else:
        w13 = torch.empty(E, 2 * I, K // 2, dtype=torch.uint8, device=device)
        w13s = torch.empty(E, 2 * I, K // 32, dtype=torch.uint8, device=device)
        w2 = torch.empty(E, K, I // 2, dtype=torch.uint8, device=device)
        w2s = torch.empty(E, K, I // 32, dtype=torch.uint8, device=device)
    quant = {"fp8": quantize_fp8_rows, "mxfp4": quantize_mxfp4_rows,
             "fp8_block": quantize_fp8_blocks}[cfg.wfmt]
    blocks = cfg.wfmt == "fp8_block"
    for e in range(E):
        ge = torch.Generator(device=device).manual_seed((seed << 20) + e)
        a = torch.randn(2 * I, K, generator=ge, device=device) / math.sqrt(K)
        b = torch.randn(K, I, generator=ge, device=device) / math.sqrt(I)
        if blocks:
            a = a * _block_gain(2 * I, K, ge, device)
            b = b * _block_gain(K, I, ge, device)
        w13[e], w13s[e] = quant(a)
        w2[e], w2s[e] = quant(b)
        del a, b
    out.update(w13=w13, w13_scale=w13s, w2=w2, w2_scale=w2s)

    out.update(sw13=None, sw13_scale=None, sw2=None, sw2_scale=None)
    if cfg.I_s:
        gs = torch.Generator(device=device).manual_seed((seed << 20) + E)
        if cfg.shared_bf16:
            out["sw13"] = _bf16_randn((2 * cfg.I_s, H), H, gs, device)
            out["sw2"] = _bf16_randn((H, cfg.I_s), cfg.I_s, gs, device)
        else:
            # an fp8 shared expert takes the routed experts' fp8 format
            a = torch.randn(2 * cfg.I_s, H, generator=gs, device=device) / math.sqrt(H)
            b = torch.randn(H, cfg.I_s, generator=gs, device=device) / math.sqrt(cfg.I_s)
            if cfg.wfmt == "fp8_block":
                a = a * _block_gain(2 * cfg.I_s, H, gs, device)
                b = b * _block_gain(H, cfg.I_s, gs, device)
                out["sw13"], out["sw13_scale"] = quantize_fp8_blocks(a)
                out["sw2"], out["sw2_scale"] = quantize_fp8_blocks(b)
            else:
                out["sw13"], out["sw13_scale"] = quantize_fp8_rows(a)
                out["sw2"], out["sw2_scale"] = quantize_fp8_rows(b)

    out.update(wd=None, wu=None, gamma=None)
    if cfg.L:
        gl = torch.Generator(device=device).manual_seed((seed << 20) + E + 1)
        out["wd"] = _bf16_randn((cfg.L, H), H, gl, device)
        out["wu"] = _bf16_randn((H, cfg.L), cfg.L, gl, device)
        out["gamma"] = torch.ones(cfg.L, dtype=torch.bfloat16, device=device)
    return out


def to_numpy(inputs: dict) -> dict:
    """Host numpy views for the oracle: bf16 -> uint16 bits, fp8/fp4 bytes as uint8."""
    res = {}
    for k, v in inputs.items():
        if v is None:
            res[k] = None
            continue
        v = v.detach().contiguous().cpu()
        if v.dtype == torch.bfloat16:
            v = v.view(torch.int16).numpy().view("uint16")
        else:
            v = v.numpy()
        res[k] = v
    return res
