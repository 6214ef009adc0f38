"""GPU parity of Kimi K3's routing and activation options: noaux_tc sigmoid
routing (the selection bit for bit, weights within 1e-6) and SiTU experts (the
grouped GEMMs and whole layers within the stated tolerance)."""
import numpy as np
import pytest
import torch

import _gpu as G
import moe_inputs as mi
from test_gpu_stages import _check_expert_ffn

pytestmark = pytest.mark.gpu

ids = lambda c: c.name


def _route_sigmoid(m, lg, bias, k):
    T, E = lg.shape
    flags = m.F_SIGMOID_ROUTING | (m.F_ROUTER_BIAS if bias is not None else 0)
    p = m.make_problem(T, 128, 128, E, k, flags=flags)
    gi = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    b = None if bias is None else torch.from_numpy(bias).cuda()
    m.moe_route(p, torch.from_numpy(lg).cuda(), b, gi, gw)
    assert m.moe_get_last_error() == 0
    return gi.cpu().numpy(), gw.cpu().numpy()


@pytest.mark.parametrize("T,E,k,bias", [
    (300, 64, 6, True), (300, 64, 6, False), (4096, 896, 16, True), (37, 8, 8, True),
    (50, 1024, 32, True), (1, 3, 1, False)])
def test_sigmoid_topk_bit_exact(orc, T, E, k, bias):
    m = G.lib()
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    b = (0.05 * rng.standard_normal(E)).astype(np.float32) if bias else None
    idx, w = orc.topk(lg, k, "sigmoid", b)
    gi, gw = _route_sigmoid(m, lg, b, k)
    assert np.array_equal(gi, idx)
    assert np.allclose(gw, w, rtol=1e-6, atol=1e-7)


def test_sigmoid_topk_edge_values(orc):
    # saturated scores (sigmoid == 1.0 in fp32 above ~17), flushed ones (below
    # -86), infinities, exact key ties made by the bias, and logits at which
    # the range reduction changes its integer n
    m = G.lib()
    T, E, k = 64, 32, 6
    rng = np.random.default_rng(9)
    lg = rng.choice(np.array([30.0, 17.5, 16.0, -90.0, -86.0, -85.9, np.inf, -np.inf, 0.0,
                              0.34657359, -0.34657359, 1.0397208, -1.0397208, 5e-8],
                             np.float32), size=(T, E))
    lg[0] = 0.0
    b = np.zeros(E, np.float32)
    b[[3, 9, 20]] = 0.25
    idx, w = orc.topk(lg, k, "sigmoid", b)
    gi, gw = _route_sigmoid(m, lg, b, k)
    assert np.array_equal(gi, idx)
    assert list(idx[0][:3]) == [3, 9, 20] and list(idx[0][3:]) == [0, 1, 2]
    assert np.allclose(gw, w, rtol=1e-6, atol=1e-7)


def test_router_bias_is_selection_only_under_sigmoid(orc):
    # with sigmoid routing the logits carry no bias; moe_route applies it
    cfg = mi.MoEConfig("k3_route", T=200, H=512, I=128, E=64, k=6, routing="sigmoid",
                       sel_bias=True)
    m = G.lib()
    inp = G.gpu_inputs(cfg)
    h = G.host(inp, keys=("x", "router_w", "router_bias"))
    p = G.problem(cfg)
    lg = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    m.moe_router_logits(p, inp["x"], inp["router_w"], inp["router_bias"], lg)
    ref = orc.router_logits(h["x"], h["router_w"])  # no bias
    assert np.array_equal(lg.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    idx, w = orc.topk(ref, cfg.k, "sigmoid", h["router_bias"])
    gi = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    gw = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda")
    m.moe_route(p, lg, inp["router_bias"], gi, gw)
    assert np.array_equal(gi.cpu().numpy(), idx)
    assert np.allclose(gw.cpu().numpy(), w, rtol=1e-6, atol=1e-7)


SITU_FP8 = [mi.CONFIGS["toy"].with_(name="toy_situ", act="situ"),
            mi.MoEConfig("ragged_situ", T=100, H=512, I=384, E=13, k=4, I_s=384, act="situ")]


@pytest.mark.parametrize("bn", [32, 128, 256])
@pytest.mark.parametrize("cfg", SITU_FP8, ids=ids)
def test_situ_expert_ffn_fp8(orc, cfg, bn, tuning):
    # SiTU epilogue in the single-SM (32, 128) and SM-pair (256) grouped GEMMs
    tuning(tile_n=bn)
    _check_expert_ffn(orc, cfg, rows_sample=None, act=orc.SITU)


K3_SMALL = [
    mi.MoEConfig("k3_fp8", T=96, H=512, I=256, E=16, k=4, I_s=256, routing="sigmoid",
                 act="situ", sel_bias=True),
    mi.MoEConfig("k3_latent", T=100, H=512, I=256, E=16, k=4, I_s=384, L=256, wfmt="mxfp4",
                 shared_bf16=True, routing="sigmoid", act="situ", sel_bias=True),
    mi.MoEConfig("k3_mx_plain", T=80, H=256, I=384, E=12, k=3, wfmt="mxfp4", routing="sigmoid",
                 act="situ", sel_bias=True),
]


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
@pytest.mark.parametrize("cfg", K3_SMALL, ids=ids)
def test_k3_forward_small(orc, cfg, packed):
    inp = G.gpu_inputs(cfg)
    out = _forward(cfg, G.pack(cfg, inp) if packed else inp, packed=packed)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref, f"moe_forward {cfg.name}")


def test_k3_latent_full_size_sampled(orc):
    cfg = mi.CONFIGS["latent_k3"]
    inp = G.gpu_inputs(cfg)
    out = _forward(cfg, G.pack(cfg, inp), packed=True)
    h = G.host(inp)
    toks = G.edge_tokens(orc, cfg, h, 128, seed=7, max_experts=64)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), h, tokens=toks)
    got = G.bf16_values(G.bf16_bits(out))[toks]
    G.assert_close(got, ref, "moe_forward latent_k3")
