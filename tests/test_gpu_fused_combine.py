"""GPU parity of the fused combine (MOE_F_FUSED_COMBINE): the FFN2 epilogue adds
each routed row, scaled by its routing weight, and each shared-expert row into
an fp32 sum per token, and a last pass rounds the sums to bf16.  Checked against
the oracle's per-token definition of the layer and against the gather combine
on the same inputs."""
import numpy as np
import pytest
import torch

import _gpu as G
import moe_inputs as mi
from test_gpu_forward import SHARED_SMALL
from test_gpu_stages import BIASED, KE, MAXE, RAGGED, T1

pytestmark = pytest.mark.gpu

SMALL = [mi.CONFIGS["toy"], SHARED_SMALL, RAGGED, MAXE, T1, KE, BIASED.with_(I_s=128)]
ids = lambda c: c.name


def fused_problem(cfg, packed=False):
    p = G.problem(cfg, packed=packed)
    p.flags |= G.lib().F_FUSED_COMBINE
    return p


def run(cfg, inp, p):
    m = G.lib()
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    m.moe_forward(p, inp["x"], inp["router_w"], inp["router_bias"], inp["w13"], inp["w13_scale"],
                  inp["w2"], inp["w2_scale"], inp["sw13"], inp["sw13_scale"], inp["sw2"],
                  inp["sw2_scale"], inp["wd"], inp["wu"], inp["gamma"], out, G.workspace(p))
    assert m.moe_get_last_error() == 0
    return G.bf16_values(G.bf16_bits(out))


@pytest.mark.parametrize("cfg", SMALL, ids=ids)
def test_fused_combine_small(orc, cfg):
    m = G.lib()
    p = fused_problem(cfg)
    assert "combine=fused" in m.moe_describe(p)
    inp = G.gpu_inputs(cfg)
    got = run(cfg, inp, p)
    ref_f, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(got, ref_f, f"fused combine {cfg.name}")


def test_fused_matches_gather_and_repeats():
    cfg = SHARED_SMALL
    inp = G.gpu_inputs(cfg)
    a = run(cfg, inp, fused_problem(cfg))
    b = run(cfg, inp, fused_problem(cfg))
    g = run(cfg, inp, G.problem(cfg))
    # the fp32 sums differ only in the order of k + 1 additions: every element
    # of two fused calls lies within one bf16 unit of the other, and the fused
    # and gather results agree to within the output bars
    assert np.all(np.abs(a - b) <= 2 * G.bf16_half_ulp(np.maximum(np.abs(a), np.abs(b))))
    G.assert_close(a, g, "fused vs gather")


def test_fused_launches_and_zeroing():
    # as many launches as with the gather combine; a second call on a reused
    # workspace must not see the first call's sums (S4 zeroes them)
    m = G.lib()
    cfg = SHARED_SMALL
    inp = G.gpu_inputs(cfg)
    p = fused_problem(cfg)
    ws = G.workspace(p)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    args = (p, inp["x"], inp["router_w"], inp["router_bias"], inp["w13"], inp["w13_scale"],
            inp["w2"], inp["w2_scale"], inp["sw13"], inp["sw13_scale"], inp["sw2"],
            inp["sw2_scale"], None, None, None, out, ws)
    n0 = m.moe_launch_count()
    m.moe_forward(*args)
    first = out.clone()
    assert m.moe_launch_count() - n0 == G.routing_launches(p) + 6
    m.moe_forward(*args)
    assert m.moe_get_last_error() == 0
    d = (out.float() - first.float()).abs()
    assert float(d.max()) <= float(2 * first.float().abs().max() * 2.0 ** -8)


def test_fused_packed_weights(orc):
    cfg = SHARED_SMALL
    inp = G.gpu_inputs(cfg)
    m = G.lib()
    w13p, w2p = torch.empty_like(inp["w13"]), torch.empty_like(inp["w2"])
    m.moe_pack_weights(m.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k), inp["w13"], inp["w2"],
                       None, None, w13p, w2p)
    s13, s2 = torch.empty_like(inp["sw13"]), torch.empty_like(inp["sw2"])
    m.moe_pack_weights(m.make_problem(cfg.T, cfg.H, cfg.I_s, 1, 1), inp["sw13"], inp["sw2"],
                       None, None, s13, s2)
    got = run(cfg, dict(inp, w13=w13p, w2=w2p, sw13=s13, sw2=s2), fused_problem(cfg, packed=True))
    ref_f, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(got, ref_f, "fused combine, packed weights")


def test_fused_decode_full_size_sampled(orc):
    cfg = mi.CONFIGS["decode"]
    m = G.lib()
    p = fused_problem(cfg)
    assert "combine=fused" in m.moe_describe(p)
    inp = G.gpu_inputs(cfg)
    got = run(cfg, inp, p)
    toks = G.sample_tokens(cfg.T, 24, seed=11)
    ref_f, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp), tokens=toks)
    G.assert_close(got[toks], ref_f, "fused combine decode")
