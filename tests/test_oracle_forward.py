"""Pins for the oracle's full layer (S5-S9).

The oracle (plain C, per token) is checked against formulations that share none
of its code: numpy fp64 matrix products with torch's float8 cast for the fp8
roundings and a bit-level bf16 rounding, the dense all-experts special case
(k = E, no routing code at all), a one-hot single-expert closed form, and the
OCP MX e2m1 table for the MXFP4 LatentMoE case.
"""
import math
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- independent helpers
def e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def e2m1_values(nibbles):
    table = {}
    with open(os.path.join(GOLDEN, "ocp_mx_e2m1.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                table[int(a, 16)] = float(b)
    lut = np.array([table[i] for i in range(16)])
    return lut[np.asarray(nibbles) & 15]


def quant_fp8(v32):
    """Per-row fp8: fp32 scale amax/448, torch's RNE cast of the fp32 quotient."""
    v32 = np.asarray(v32, np.float32)
    amax = np.abs(v32).max(-1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = torch.from_numpy((v32 / s[..., None]).astype(np.float32)).to(torch.float8_e4m3fn)
    return s, q.double().numpy()


def bf16_round(d):
    """Nearest-even bf16 of doubles in the normal range, by integer rounding of the bits."""
    d = np.asarray(d, np.float64)
    b = d.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    out = r.view(np.float64)
    return np.where(d == 0, 0.0, out)


def bf16_bits(d):
    return (np.asarray(bf16_round(d), np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_vals(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def fp8_weight(w_bytes, scale):
    return e4m3_values(w_bytes) * np.asarray(scale, np.float64)[..., None]


def fp8_block_weight(w_bytes, scale):
    """e4m3 values times the fp32 scale of their 128 x 128 block."""
    full = np.repeat(np.repeat(np.asarray(scale, np.float64), 128, -2), 128, -1)
    return e4m3_values(w_bytes) * full


def mxfp4_weight(packed, scales):
    lo, hi = packed & 15, packed >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    vals = e2m1_values(nib)
    sc = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return vals * np.repeat(sc, 32, axis=-1)


def sigm(v):
    return 1.0 / (1.0 + np.exp(-v))


def gated(g, u, act="swiglu"):
    """silu(g) u, or SiTU 4 tanh(g/4) sigmoid(g) u written through the identity
    tanh(v) = 2 sigmoid(2v) - 1 (a different route to the same value)."""
    if act == "situ":
        return 4.0 * (2.0 * sigm(g / 2.0) - 1.0) * sigm(g) * u
    return g / (1.0 + np.exp(-g)) * u


def swiglu_rows(xq, sx, W13, W2, I, act="swiglu"):
    """Rows xq [n, K] (decoded, fp64), sx [n]; W13 [2I, K] and W2 [K, I] fp64."""
    acc = xq @ W13.T
    g = acc[:, :I] * sx[:, None]
    u = acc[:, I:] * sx[:, None]
    h = bf16_round(gated(g, u, act))
    s_h, hq = quant_fp8(h.astype(np.float32))
    return (hq @ W2.T) * s_h[:, None].astype(np.float64)


def numpy_layer(cfg, w, idx, wt):
    """The layer for all tokens, given the routing (idx, weights)."""
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    x = bf16_vals(w["x"])
    if cfg.L:
        z = bf16_round(x @ bf16_vals(w["wd"]).T)
        sx, xq = quant_fp8(z.astype(np.float32))
    else:
        sx, xq = quant_fp8(x.astype(np.float32))
    acc = np.zeros((T, K))
    for e in range(E):
        if cfg.wfmt == "fp8":
            W13 = fp8_weight(w["w13"][e], w["w13_scale"][e])
            W2 = fp8_weight(w["w2"][e], w["w2_scale"][e])
        elif cfg.wfmt == "fp8_block":
            W13 = fp8_block_weight(w["w13"][e], w["w13_scale"][e])
            W2 = fp8_block_weight(w["w2"][e], w["w2_scale"][e])
        else:
            W13 = mxfp4_weight(w["w13"][e], w["w13_scale"][e])
            W2 = mxfp4_weight(w["w2"][e], w["w2_scale"][e])
        y = swiglu_rows(xq, sx.astype(np.float64), W13, W2, I, cfg.act)
        coef = np.where(idx == e, wt, 0.0).sum(1)
        acc += coef[:, None] * y
    if cfg.L:
        ms = (acc ** 2).mean(1)
        yn = bf16_round(acc / np.sqrt(ms + cfg.rms_eps)[:, None] * bf16_vals(w["gamma"])[None, :])
        res = yn @ bf16_vals(w["wu"]).T
    else:
        res = acc
    if cfg.I_s:
        if cfg.shared_bf16:
            W13s = bf16_vals(w["sw13"])
            g = x @ W13s[: cfg.I_s].T
            u = x @ W13s[cfg.I_s:].T
            hs = bf16_round(gated(g, u, cfg.act))
            res = res + hs @ bf16_vals(w["sw2"]).T
        else:
            sxs, xqs = quant_fp8(x.astype(np.float32))
            deq = fp8_block_weight if cfg.wfmt == "fp8_block" else fp8_weight
            res = res + swiglu_rows(xqs, sxs.astype(np.float64), deq(w["sw13"], w["sw13_scale"]),
                                    deq(w["sw2"], w["sw2_scale"]), cfg.I_s, cfg.act)
    return res


def _close(a, b, rtol=1e-12):
    scale = np.sqrt((b ** 2).mean()) + 1e-300
    return np.max(np.abs(a - b)) <= rtol * scale * 10


# ----------------------------------------------------------------------------- tests
SMALL = [
    mi.CONFIGS["toy"],
    mi.MoEConfig("small_shared", T=24, H=256, I=128, E=6, k=3, I_s=128),
    mi.MoEConfig("small_bias", T=16, H=128, I=256, E=5, k=2, I_s=128, zipf_bias=True),
    # Kimi K3 routing and activation: noaux_tc sigmoid routing with a selection
    # bias, SiTU experts (fp8 shared expert here, bf16 in the latent case below)
    mi.MoEConfig("small_k3", T=20, H=256, I=128, E=8, k=3, I_s=128, routing="sigmoid",
                 act="situ", sel_bias=True),
    # block-wise fp8 (128 x 128 weight blocks, scales of differing size); a
    # non-square block grid so that a transposed scale index cannot pass
    mi.MoEConfig("small_block", T=24, H=256, I=384, E=6, k=3, I_s=128, wfmt="fp8_block"),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_forward_matches_numpy_formulation(orc, cfg):
    w = mi.to_numpy(mi.make_inputs(cfg, seed=11))
    of, ob, idx, wt = orc.moe_forward(cfg.oracle_problem(), w)
    ref = numpy_layer(cfg, w, idx, wt)
    assert _close(of, ref)
    mism = np.mean(ob != bf16_bits(ref))
    assert mism <= 1e-3
    # routing agrees with the separately pinned stages
    if cfg.routing == "sigmoid":  # the bias steers selection only
        lg = orc.router_logits(w["x"], w["router_w"])
        idx2, wt2 = orc.topk(lg, cfg.k, "sigmoid", w["router_bias"])
    else:
        lg = orc.router_logits(w["x"], w["router_w"], w["router_bias"])
        idx2, wt2 = orc.topk(lg, cfg.k)
    assert np.array_equal(idx, idx2) and np.allclose(wt, wt2, rtol=0, atol=0)


def test_dense_all_experts_special_case(orc):
    # k = E: every expert is selected, so the layer is sum_e softmax_e(l) FFN_e(x)
    # with no routing decisions at all.
    cfg = mi.CONFIGS["toy"].with_(k=8, I_s=128)
    w = mi.to_numpy(mi.make_inputs(cfg, seed=5))
    of, ob, idx, wt = orc.moe_forward(cfg.oracle_problem(), w)
    lg = orc.router_logits(w["x"], w["router_w"]).astype(np.float64)
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = numpy_layer(cfg, w, np.tile(np.arange(8), (cfg.T, 1)), p)
    assert _close(of, ref)


def test_single_expert_one_hot_closed_form(orc):
    # E = 1, k = 1, x = a * e_i: the quantised row is 448 at i and 0 elsewhere,
    # so g = a * W1[:, i] (per-channel scale 1), u = a * W3[:, i], and
    # out = W2 (bf16(silu(g) u) after per-row fp8), computed here by hand.
    H, I, i = 64, 128, 5
    rng = np.random.default_rng(0)
    vals = np.array([0.5, 1.0, 1.5, -0.5, -1.0, 2.0, 0.25, -2.0])
    W1 = np.zeros((I, H)); W3 = np.zeros((I, H)); W2 = np.zeros((H, I))
    W1[:, i] = rng.choice(vals, I)
    W3[:, i] = rng.choice(vals, I)
    W2[:] = rng.choice(vals, (H, I))
    a = 1.0
    enc = lambda M: torch.from_numpy(M.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    x = np.zeros((1, H), np.float32); x[0, i] = a
    w = dict(x=bf16_bits(x), router_w=np.ones((1, H), np.float32), router_bias=None,
             w13=enc(np.concatenate([W1, W3]))[None], w13_scale=np.ones((1, 2 * I), np.float32),
             w2=enc(W2)[None], w2_scale=np.ones((1, H), np.float32),
             sw13=None, sw13_scale=None, sw2=None, sw2_scale=None, wd=None, wu=None, gamma=None)
    prob = dict(T=1, H=H, I=I, E=1, k=1, I_s=0, L=0, wfmt="fp8")
    of, ob, idx, wt = orc.moe_forward(prob, w)
    sx = np.float32(a) / np.float32(448.0)  # per-token scale; x/s == 448 at i
    g = 448.0 * W1[:, i] * float(sx)
    u = 448.0 * W3[:, i] * float(sx)
    h = np.array([float(torch.tensor(gg / (1 + math.exp(-gg)) * uu, dtype=torch.float64)
                        .float().to(torch.bfloat16).float()) for gg, uu in zip(g, u)])
    s_h = np.float32(np.abs(h).max()) / np.float32(448.0)
    hq = torch.from_numpy((h.astype(np.float32) / s_h).astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    expect = W2 @ hq * float(s_h)
    assert idx[0, 0] == 0 and wt[0, 0] == 1.0
    assert np.allclose(of[0], expect, rtol=1e-12, atol=1e-12)
    # a transposed W1 (row i instead of column i) would give zeros here
    assert np.abs(of[0]).max() > 0.1


@pytest.mark.parametrize("k3", [False, True], ids=["softmax-swiglu", "sigmoid-situ"])
def test_latent_mxfp4_matches_numpy(orc, k3):
    cfg = mi.MoEConfig("latent_small", T=6, H=256, I=128, E=4, k=2, I_s=128, L=128,
                       wfmt="mxfp4", shared_bf16=True)
    if k3:
        cfg = cfg.with_(routing="sigmoid", act="situ", sel_bias=True)
    w = mi.to_numpy(mi.make_inputs(cfg, seed=3))
    of, ob, idx, wt = orc.moe_forward(cfg.oracle_problem(), w)
    ref = numpy_layer(cfg, w, idx, wt)
    assert _close(of, ref, rtol=1e-10)
    assert np.mean(ob != bf16_bits(ref)) <= 1e-2


def test_mxfp4_generator_round_trip():
    # the weight prep (input side) reproduces values exactly representable in MXFP4
    scale = 2.0 ** -3
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -6, -4, -3, -2, -1.5, -1, -0.5, 0] * 2) * scale
    packed, sc = mi.quantize_mxfp4_rows(torch.tensor(vals[None, :], dtype=torch.float32))
    back = mxfp4_weight(packed.numpy(), sc.numpy())
    assert np.array_equal(back[0], vals)


def test_token_independence(orc):
    cfg = SMALL[1]
    w = mi.to_numpy(mi.make_inputs(cfg, seed=2))
    of, ob, _, _ = orc.moe_forward(cfg.oracle_problem(), w)
    sel = np.array([17, 3, 3, 0], np.int32)
    of2, ob2, _, _ = orc.moe_forward(cfg.oracle_problem(), w, tokens=sel)
    assert np.array_equal(ob2, ob[sel]) and np.array_equal(of2, of[sel])


def test_expert_rows_matches_forward_pieces(orc):
    # the grouped-rows stage oracle agrees with the per-token layer
    cfg = SMALL[0]
    w = mi.to_numpy(mi.make_inputs(cfg, seed=4))
    lg = orc.router_logits(w["x"], w["router_w"])
    idx, wt = orc.topk(lg, cfg.k)
    cnt, off, perm, src = orc.permute(idx, cfg.E)
    s, q = orc.quant_rows(w["x"])
    row_w = np.empty(cfg.R, np.float32)
    row_w[perm.reshape(-1)] = wt.reshape(-1).astype(np.float32)
    y = orc.expert_rows(orc.FP8, off, q[src], s[src], np.ones(cfg.R, np.float32), w["w13"],
                        w["w13_scale"], w["w2"], w["w2_scale"])
    of, _, _, _ = orc.moe_forward(cfg.oracle_problem(), w)
    comb = (y[perm] * wt[:, :, None]).sum(1)
    assert _close(comb, of)


def test_situ_one_hot_closed_form(orc):
    # E = 1, k = 1, x = e_i: g = 448 s_x W1[:, i], u likewise; SiTU's h =
    # bf16(4 tanh(g/4) sigmoid(g) u) checked value by value with math.tanh, and
    # its two limits: h -> 4u for large g (tanh, sigmoid -> 1) and h -> g u / 2
    # for small g (4 tanh(g/4) -> g, sigmoid -> 1/2).
    H, I, i = 64, 128, 7
    rng = np.random.default_rng(1)
    vals = np.array([0.03125, 0.0625, 0.5, 1.0, 8.0, 16.0, -0.0625, -8.0])
    W1 = np.zeros((I, H)); W3 = np.zeros((I, H)); W2 = np.eye(H, I)
    W1[:, i] = rng.choice(vals, I)
    W3[:, i] = rng.choice(vals, I)
    enc = lambda M: torch.from_numpy(M.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    x = np.zeros((1, H), np.float32); x[0, i] = 1.0
    w = dict(x=bf16_bits(x), router_w=np.ones((1, H), np.float32), router_bias=None,
             w13=enc(np.concatenate([W1, W3]))[None], w13_scale=np.ones((1, 2 * I), np.float32),
             w2=enc(W2)[None], w2_scale=np.ones((1, H), np.float32),
             sw13=None, sw13_scale=None, sw2=None, sw2_scale=None, wd=None, wu=None, gamma=None)
    prob = dict(T=1, H=H, I=I, E=1, k=1, I_s=0, L=0, wfmt="fp8", routing="sigmoid", act="situ")
    cnt, off, perm, src = orc.permute(np.zeros((1, 1), np.int32), 1)
    s, q = orc.quant_rows(w["x"])
    y, h, hq, hs = orc.expert_rows(orc.FP8, off, q, s, np.ones(1, np.float32), w["w13"],
                                   w["w13_scale"], w["w2"], w["w2_scale"], want_h=True,
                                   act=orc.SITU)
    g = 448.0 * W1[:, i] * float(np.float32(1.0) / np.float32(448.0))
    u = 448.0 * W3[:, i] * float(np.float32(1.0) / np.float32(448.0))
    expect = [4.0 * math.tanh(gg / 4.0) / (1.0 + math.exp(-gg)) * uu for gg, uu in zip(g, u)]
    assert np.array_equal(h[0], bf16_bits(np.array(expect)))
    big = np.abs(g) >= 16
    assert np.allclose(bf16_vals(h[0])[big & (g > 0)], 4.0 * u[big & (g > 0)], rtol=2e-2)
    small = np.abs(g) <= 0.0625
    assert np.allclose(bf16_vals(h[0])[small], g[small] * u[small] / 2.0, rtol=5e-2)
    # the layer uses the same activation
    of, _, _, _ = orc.moe_forward(prob, w)
    assert np.allclose(of[0], y[0], rtol=0, atol=0)


def test_fp8_block_with_uniform_row_scales_is_per_channel(orc):
    # when every block of a 128-row block row has one scale c, the block-wise
    # weight equals the per-channel weight with scale c on each of those rows
    cfg = mi.MoEConfig("blk_uni", T=12, H=256, I=256, E=3, k=2, I_s=128, wfmt="fp8_block")
    w = mi.to_numpy(mi.make_inputs(cfg, seed=6))
    for key in ("w13_scale", "w2_scale", "sw13_scale", "sw2_scale"):
        sc = w[key]
        w[key] = np.repeat(sc[..., :1], sc.shape[-1], axis=-1).astype(np.float32)
    of_b, _, idx_b, _ = orc.moe_forward(cfg.oracle_problem(), w)
    wc = dict(w)
    for key in ("w13_scale", "w2_scale", "sw13_scale", "sw2_scale"):
        wc[key] = np.repeat(w[key][..., 0], 128, axis=-1).astype(np.float32)
    of_c, _, idx_c, _ = orc.moe_forward(cfg.with_(wfmt="fp8").oracle_problem(), wc)
    assert np.array_equal(idx_b, idx_c)
    assert _close(of_b, of_c, rtol=1e-12)
