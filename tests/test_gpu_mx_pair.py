"""GPU parity of the MXFP4 grouped GEMMs on SM pairs (tcgen05 cta_group::2),
which run when the expert weights are in moe_pack_weights' order and the
weight blocks pair up ("Kimi K3 ... feasibility analysis", s.2.5 MXFP4 experts;
s.2.4 LatentMoE).  The whole layer against the oracle, and against the
single-SM kernels on the same inputs."""
import pytest
import torch

import _gpu as G
import moe_inputs as mi

pytestmark = pytest.mark.gpu

MX_PAIR = mi.MoEConfig("mxfp4_pair", T=96, H=512, I=256, E=8, k=2, wfmt="mxfp4")
MX_PAIR_RAGGED = mi.MoEConfig("mxfp4_pair_ragged", T=301, H=1024, I=512, E=12, k=3, wfmt="mxfp4")
LAT_PAIR = mi.MoEConfig("latent_pair", T=100, H=512, I=256, E=16, k=4, I_s=384, L=512,
                        wfmt="mxfp4", shared_bf16=True)
ONE_EXPERT = mi.MoEConfig("mxfp4_pair_one", T=40, H=512, I=256, E=1, k=1, wfmt="mxfp4")
ids = lambda c: c.name


def forward(cfg, inp):
    m = G.lib()
    p = G.problem(cfg, packed=True)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    m.moe_forward(p, inp["x"], inp["router_w"], inp["router_bias"], inp["w13"], inp["w13_scale"],
                  inp["w2"], inp["w2_scale"], inp["sw13"], inp["sw13_scale"], inp["sw2"],
                  inp["sw2_scale"], inp["wd"], inp["wu"], inp["gamma"], out, G.workspace(p))
    assert m.moe_get_last_error() == 0
    return G.bf16_values(G.bf16_bits(out))


@pytest.mark.parametrize("bn", [32, 64, 96])
@pytest.mark.parametrize("cfg", [MX_PAIR, MX_PAIR_RAGGED, LAT_PAIR, ONE_EXPERT], ids=ids)
def test_mx_pair_forward(orc, cfg, bn, tuning):
    tuning(tile_n=bn)
    m = G.lib()
    d = m.moe_describe(G.problem(cfg, packed=True))
    assert "ffn1=grouped_mx_pair_kernel" in d and "ffn2=grouped_mx_pair_kernel" in d, d
    inp = G.gpu_inputs(cfg)
    got = forward(cfg, G.pack(cfg, inp))
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(got, ref, f"mxfp4 pair {cfg.name} BN={bn}")


def test_mx_pair_matches_single_sm(tuning):
    cfg = MX_PAIR_RAGGED
    inp = G.pack(cfg, G.gpu_inputs(cfg))
    pair = forward(cfg, inp)
    tuning(mx_1cta=1)
    assert "grouped_mx_pair_kernel" not in G.lib().moe_describe(G.problem(cfg, packed=True))
    single = forward(cfg, inp)
    G.assert_close(pair, single, "pair vs single-SM")


def test_mx_pair_situ(orc):
    cfg = MX_PAIR.with_(name="mxfp4_pair_situ", act="situ")
    inp = G.gpu_inputs(cfg)
    got = forward(cfg, G.pack(cfg, inp))
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(got, ref, "mxfp4 pair SiTU")
