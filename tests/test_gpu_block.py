"""GPU parity of block-wise fp8 experts (one fp32 scale per 128 x 128 weight
block): the grouped GEMMs with per-stage promotion of the partial sums, whole
layers, and the full decode-sized layer on sampled tokens."""
import numpy as np
import pytest
import torch

import _gpu as G
import moe_inputs as mi
from test_gpu_stages import _check_expert_ffn

pytestmark = pytest.mark.gpu

ids = lambda c: c.name

BLOCK_SMALL = [
    mi.MoEConfig("blk_toy", T=64, H=256, I=128, E=8, k=2, wfmt="fp8_block"),
    mi.MoEConfig("blk_ragged", T=100, H=512, I=384, E=13, k=4, I_s=384, wfmt="fp8_block"),
    mi.MoEConfig("blk_skew", T=640, H=512, I=256, E=16, k=4, zipf_bias=True, wfmt="fp8_block"),
    mi.MoEConfig("blk_t1", T=1, H=256, I=128, E=8, k=2, I_s=128, wfmt="fp8_block"),
]


@pytest.mark.parametrize("bn", [32, 64])
@pytest.mark.parametrize("cfg", BLOCK_SMALL[:3], ids=ids)
def test_block_expert_ffn(orc, cfg, bn, tuning):
    tuning(tile_n=bn)
    _check_expert_ffn(orc, cfg, rows_sample=None)


def test_block_expert_ffn_situ(orc):
    _check_expert_ffn(orc, BLOCK_SMALL[1].with_(name="blk_situ", act="situ"), rows_sample=None,
                      act=orc.SITU)


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


@pytest.mark.parametrize("packed", [False, True], ids=["row-major", "packed"])
@pytest.mark.parametrize("cfg", BLOCK_SMALL + [
    mi.MoEConfig("blk_latent", T=72, H=512, I=128, E=8, k=2, I_s=256, L=256, wfmt="fp8_block",
                 shared_bf16=True)], ids=ids)
def test_block_forward_small(orc, cfg, packed):
    inp = G.gpu_inputs(cfg)
    out = _forward(cfg, G.pack(cfg, inp) if packed else inp, packed=packed)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref, f"moe_forward {cfg.name}",
                   bf16_store_allowance=True)


def test_block_scales_matter(orc):
    # the same bytes with every block scale doubled in one W1 block row change
    # exactly the features of that block row
    cfg = BLOCK_SMALL[0]
    inp = G.gpu_inputs(cfg)
    base = _forward(cfg, inp).float()
    s13 = inp["w13_scale"].clone()
    s13[:, 0, :] *= 2.0  # W1 rows 0..127 of every expert (gate of features 0..127)
    out = _forward(cfg, dict(inp, w13_scale=s13)).float()
    assert not torch.equal(out, base)
    h = G.host(inp)
    h2 = dict(h, w13_scale=s13.cpu().numpy())
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), h2)
    G.assert_close(G.bf16_values(G.bf16_bits(out.to(torch.bfloat16))), ref, "scaled block row",
                   bf16_store_allowance=True)


def test_block_decode_full_size_sampled(orc):
    cfg = mi.CONFIGS["decode_block"]
    inp = G.gpu_inputs(cfg)
    out = _forward(cfg, G.pack(cfg, inp), packed=True)
    toks = G.sample_tokens(cfg.T, 24, seed=9)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp), tokens=toks)
    G.assert_close(G.bf16_values(G.bf16_bits(out))[toks], ref, "decode_block",
                   bf16_store_allowance=True)
