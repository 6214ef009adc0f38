"""GPU parity for MXFP4 experts and the LatentMoE block ("Kimi K3 ...
feasibility analysis", s.2.4 LatentMoE, s.2.5 MXFP4): the block-scaled grouped
GEMMs stage by stage and the whole layer, against the oracle."""
import numpy as np
import pytest
import torch

import _gpu as G
import moe_inputs as mi

pytestmark = pytest.mark.gpu

LAT_SMALL = mi.MoEConfig("latent_small", T=100, H=512, I=256, E=16, k=4, I_s=384, L=256,
                         wfmt="mxfp4", shared_bf16=True)
LAT_NOSH = mi.MoEConfig("latent_noshared", T=64, H=256, I=128, E=8, k=2, L=256, wfmt="mxfp4")
MX_PLAIN = mi.MoEConfig("mxfp4_plain", T=80, H=256, I=384, E=12, k=3, wfmt="mxfp4")
LAT_FP8 = mi.MoEConfig("latent_fp8", T=72, H=512, I=128, E=8, k=2, I_s=256, L=256,
                       shared_bf16=True)
ids = lambda c: c.name


def _latent_rows(orc, cfg, seed=9):
    """Expert-contiguous quantised rows for a random latent input."""
    inp = G.gpu_inputs(cfg)
    h = G.host(inp)
    lg = orc.router_logits(h["x"], h["router_w"], h["router_bias"])
    idx, w = orc.topk(lg, cfg.k)
    cnt, off, perm, src = orc.permute(idx, cfg.E)
    rng = np.random.default_rng(seed)
    z = torch.from_numpy(rng.standard_normal((cfg.T, cfg.K)).astype(np.float32)).to(torch.bfloat16)
    zb = z.view(torch.int16).numpy().view(np.uint16)
    s, q = orc.quant_rows(zb)
    row_w = np.empty(cfg.R, np.float32)
    row_w[perm.reshape(-1)] = w.reshape(-1).astype(np.float32)
    return inp, h, off, q[src], s[src], row_w


@pytest.mark.parametrize("bn", [32, 64, 96])
@pytest.mark.parametrize("cfg", [MX_PLAIN, LAT_SMALL, MX_PLAIN.with_(name="mx_situ", act="situ")],
                         ids=ids)
def test_mxfp4_expert_ffn(orc, cfg, bn, tuning):
    tuning(tile_n=bn)
    m = G.lib()
    inp, h, off, xq, xs, row_w = _latent_rows(orc, cfg)
    p = G.problem(cfg)
    ws = G.workspace(p)
    y = torch.empty(cfg.R, cfg.K, dtype=torch.bfloat16, device="cuda")
    m.moe_expert_ffn(p, torch.from_numpy(off).cuda(), torch.from_numpy(xq).cuda(),
                     torch.from_numpy(xs).cuda(), torch.from_numpy(row_w).cuda(), inp["w13"],
                     inp["w13_scale"], inp["w2"], inp["w2_scale"], y, ws)
    assert m.moe_get_last_error() == 0
    ref = orc.expert_rows(orc.MXFP4, off, xq, xs, row_w, h["w13"], h["w13_scale"], h["w2"],
                          h["w2_scale"], act=orc.SITU if cfg.act == "situ" else orc.SWIGLU)
    G.assert_close(G.bf16_values(G.bf16_bits(y)), ref, f"mxfp4 expert_ffn {cfg.name}")


def _forward(cfg, inp, packed=False):
    m = G.lib()
    p = G.problem(cfg, packed=packed)
    ws = G.workspace(p)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    m.moe_forward(p, inp["x"], inp["router_w"], inp["router_bias"], inp["w13"], inp["w13_scale"],
                  inp["w2"], inp["w2_scale"], inp["sw13"], inp["sw13_scale"], inp["sw2"],
                  inp["sw2_scale"], inp["wd"], inp["wu"], inp["gamma"], out, ws)
    assert m.moe_get_last_error() == 0
    return out


@pytest.mark.parametrize("cfg", [LAT_SMALL, LAT_NOSH, MX_PLAIN, LAT_FP8], ids=ids)
def test_latent_and_mxfp4_forward_small(orc, cfg):
    inp = G.gpu_inputs(cfg)
    out = _forward(cfg, inp)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref, f"moe_forward {cfg.name}")


def _block_rows(key, cfg, p, b):
    # the 128 weight rows of block b of stage pair p: W1|W3 block p (w13), W2 block 2p+b (w2)
    start = (b * cfg.I + p * 128) if key.startswith("w13") else (2 * p + b) * 128
    return torch.arange(start, start + 128)


def test_mxfp4_pack_is_a_permutation():
    # weights: packed[e, p, kb, b, r, :] == w[e, row(p, b) + r, 64kb : 64kb + 64]  (128 e2m1)
    # scales:  packed[e, p, kb, j, b, i, c, :] == s[e, row(p, b) + 32c + 8j + i, 4kb : 4kb + 4]
    cfg = MX_PLAIN.with_(I=512)
    inp = G.gpu_inputs(cfg)
    pk = G.pack(cfg, inp)
    for key, R, C in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        w, t = inp[key].view(cfg.E, R, C // 2), pk[key].reshape(cfg.E, R // 256, C // 128, 2, 128, 64)
        sk = key + "_scale"
        s = inp[sk].view(cfg.E, R, C // 32)
        img = pk[sk].reshape(cfg.E, R // 256, C // 128, 4, 2, 8, 4, 4)  # e, p, kb, j, b, i, c, byte
        for p in range(R // 256):
            for b in range(2):
                rows = _block_rows(key, cfg, p, b)
                got_w = t[:, p, :, b].permute(0, 2, 1, 3).reshape(cfg.E, 128, C // 2)
                assert torch.equal(got_w, w[:, rows]), (key, p, b)
                # [e, kb, j, i, c, byte] -> rows 32c + 8j + i
                got_s = img[:, p, :, :, b].permute(0, 4, 2, 3, 1, 5).reshape(cfg.E, 128, C // 32)
                assert torch.equal(got_s, s[:, rows]), (sk, p, b)


@pytest.mark.parametrize("cfg", [LAT_SMALL, MX_PLAIN], ids=ids)
def test_mxfp4_packed_forward_small(orc, cfg):
    inp = G.gpu_inputs(cfg)
    out = _forward(cfg, G.pack(cfg, inp), packed=True)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref, f"packed {cfg.name}")


def _latent_full(orc, packed=False):
    cfg = mi.CONFIGS["latent"]
    inp = G.gpu_inputs(cfg)
    out = _forward(cfg, G.pack(cfg, inp) if packed else inp, packed=packed)
    h = G.host(inp)
    # 256 tokens: the last routed row of 200 experts (their last tile items),
    # tokens of the most loaded expert, and a random fill
    toks = G.edge_tokens(orc, cfg, h, 256, seed=5, max_experts=200)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), h, tokens=toks)
    return G.bf16_values(G.bf16_bits(out))[toks], ref


# z = bf16(x Wd^T) is exactly rounded on both sides (moe_latent_down), so the
# per-token fp8 quantisation of z agrees code for code and the whole LatentMoE
# layer meets both bars on the raw difference
@pytest.mark.parametrize("packed", [False, True], ids=["row-major", "packed"])
def test_latent_full_size_sampled(orc, packed):
    got, ref = _latent_full(orc, packed)
    assert len(got) >= 256
    G.assert_close(got, ref, f"moe_forward latent ({'packed' if packed else 'row-major'})")


def test_latent_routing_bit_exact(orc):
    # the router runs on the raw hidden x [T, 7168] over 896 experts
    m = G.lib()
    cfg = mi.CONFIGS["latent"]
    inp = G.gpu_inputs(cfg)
    h = G.host(inp, keys=("x", "router_w", "router_bias"))
    p = G.problem(cfg)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    m.moe_router_logits(p, inp["x"], inp["router_w"], None, logits)
    ref = orc.router_logits(h["x"], h["router_w"])
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref.view(np.uint32))
