"""GPU parity of moe_router_topk (S1 + S2 in one call): the tensor-core logits
with the selection made exact must give the oracle's canonical routing bit for
bit -- expert indices and their order.  Its weights come from the logits the
selection used: canonical ones on the tokens whose order the margins could not
settle, the tensor-core ones elsewhere, so they are held to the error those
margins bound (below; 1e-5 relative where that is smaller)
("Optimising Ling-2.6-1T on TPU with SGLang-JAX", s.1 top-8 routing; "Kimi K3
... feasibility analysis", s.2.4 renormalised top-k and noaux_tc sigmoid
routing).  Runs the tensor-core path on every shape (forced) and the automatic
choice on the named workloads, including constructed exact ties."""
import numpy as np
import pytest
import torch

import _gpu as G
import moe_inputs as mi
from test_gpu_stages import BIASED, E3, FULL, KE, LATENT, MAXE, RAGGED, SKEW_SMALL, T1

pytestmark = pytest.mark.gpu
ids = lambda c: c.name

K3 = mi.CONFIGS["latent_k3"]
SIG_SMALL = mi.MoEConfig("sig_small", T=300, H=512, I=128, E=40, k=6, routing="sigmoid",
                         sel_bias=True)


ULPS = 8.0  # the kernel's margin, in units of 2^-23 |x_t| |w_e|


def _oracle_routing(orc, cfg, h):
    """(idx, weights, logits) of the oracle; logits fp32 [T, E], unbiased
    for sigmoid routing (the bias steers selection only)."""
    if cfg.routing == "sigmoid":
        lg = orc.router_logits(h["x"], h["router_w"])
        return orc.topk(lg, cfg.k, routing="sigmoid", bias=h["router_bias"]) + (lg,)
    lg = orc.router_logits(h["x"], h["router_w"], h["router_bias"])
    return orc.topk(lg, cfg.k) + (lg,)


def _router_splits(cfg):
    """K ranges of the tensor-core router GEMM: enough for every SM pair when
    its output has few 256 x 256 tiles, at least 8 stages of 64 each."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tiles = -(-cfg.T // 256) * -(-cfg.E // 256)
    kb = 3 * cfg.H // 64
    if tiles * 2 > pairs or kb < 16:
        return 1
    s = min(pairs // tiles, kb // 8)
    kbs = -(-kb // s)
    return -(-kb // kbs)


def _weight_rtol(cfg, h, idx, lg):
    """Per-token, per-slot bound on the relative error of the routing weights
    when each chosen logit l_j is off by at most m_j = ULPS 2^-23 |x_t| |w_j|
    (plus (S - 1) 2^-24 |x_t| |w_j| when the GEMM's K runs in S ranges whose
    sums are added: each running sum is at most |x_t| |w_j|).
    Softmax over the chosen logits: dw_i / w_i <= m_i + max_j m_j.  Sigmoid
    scores s_j, renormalised: ds_j <= m_j / 4 + 2^-20 (the sigmoid's slope is
    at most 1/4, plus its own rounding), so dw_i / w_i <= ds_i / s_i +
    max_j ds_j / s_j.  Doubled for second-order terms and fp32 rounding, and
    never below 1e-5."""
    x = G.bf16_values(np.asarray(h["x"]).view(np.uint16)).reshape(cfg.T, cfg.H)
    xn = np.sqrt((x * x).sum(axis=1))
    wr = np.asarray(h["router_w"], np.float64)
    wn = np.sqrt((wr * wr).sum(axis=1))
    m = (ULPS * 2.0 ** -23 + (_router_splits(cfg) - 1) * 2.0 ** -24) * xn[:, None] * wn[idx]
    if cfg.routing == "sigmoid":
        s = 1.0 / (1.0 + np.exp(-np.take_along_axis(lg.astype(np.float64), idx, axis=1)))
        rel = (m / 4 + 2.0 ** -20) / s
    else:
        rel = m
    return np.maximum(2.0 * (rel + rel.max(axis=1, keepdims=True)), 1e-5)


def _check(orc, cfg, inp):
    m = G.lib()
    h = G.host(inp, keys=("x", "router_w", "router_bias"))
    idx, w, lg = _oracle_routing(orc, cfg, h)
    p = G.problem(cfg)
    ws = G.workspace(p)
    gi = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device="cuda")
    gw = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda")
    m.moe_router_topk(p, inp["x"], inp["router_w"], inp["router_bias"], gi, gw, ws)
    assert m.moe_get_last_error() == 0
    got = gi.cpu().numpy()
    bad = np.nonzero((got != idx).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} of {cfg.T} tokens routed differently, first {bad[:5]}"
    rel = np.abs(gw.cpu().numpy() - w) / np.abs(w)
    tol = _weight_rtol(cfg, h, idx, lg)
    worst = np.unravel_index(np.argmax(rel / tol), rel.shape)
    assert (rel <= tol).all(), (f"weight rel error {rel[worst]:.3g} > bound {tol[worst]:.3g} "
                                f"at token {worst[0]}, slot {worst[1]}; max rel {rel.max():.3g}")


@pytest.mark.parametrize("cfg", [mi.CONFIGS["toy"], RAGGED, MAXE, T1, KE, E3, BIASED, SKEW_SMALL,
                                 SIG_SMALL], ids=ids)
def test_router_topk_tensor_cores_small(orc, cfg, tuning):
    tuning(router_tile="tc")
    _check(orc, cfg, G.gpu_inputs(cfg))


@pytest.mark.parametrize("path", ["auto", "tc"])
@pytest.mark.parametrize("cfg", FULL + [LATENT, K3], ids=ids)
def test_router_topk_full_size(orc, cfg, path, tuning):
    tuning(router_tile=path)
    _check(orc, cfg, G.gpu_inputs(cfg))


def test_router_topk_exact_ties(orc, tuning):
    # duplicated router rows give exactly equal logits: the lower index must
    # come first, and the approximate logits cannot decide that on their own
    tuning(router_tile="tc")
    cfg = mi.MoEConfig("ties", T=256, H=512, I=128, E=24, k=5)
    inp = dict(G.gpu_inputs(cfg))
    wr = inp["router_w"].clone()
    wr[7] = wr[3]
    wr[11] = wr[3]
    wr[20] = wr[15]
    inp["router_w"] = wr
    _check(orc, cfg, inp)


def test_router_topk_run_across_the_boundary(orc, tuning):
    # eight copies of one router row with a bias that puts them first for
    # every token: positions 0..7 tie exactly, the k = 5 boundary falls inside
    # that run, and selection must take more than k + 1 experts out before a
    # cut is proven
    tuning(router_tile="tc")
    cfg = mi.MoEConfig("run8", T=256, H=512, I=128, E=24, k=5, zipf_bias=True)
    inp = dict(G.gpu_inputs(cfg))
    wr = inp["router_w"].clone()
    for e in (2, 5, 6, 9, 13, 17, 20, 23):
        wr[e] = wr[2]
    inp["router_w"] = wr
    bias = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
    bias[[2, 5, 6, 9, 13, 17, 20, 23]] = 50.0
    inp["router_bias"] = bias
    _check(orc, cfg, inp)


def test_router_topk_no_cut_within_32(orc, tuning):
    # forty identical experts ahead of all others: no cut can be proven among
    # the first 32 positions, so every expert that could place is recomputed
    tuning(router_tile="tc")
    cfg = mi.MoEConfig("run40", T=128, H=512, I=128, E=64, k=8, zipf_bias=True)
    inp = dict(G.gpu_inputs(cfg))
    same = [e for e in range(cfg.E) if e % 8 != 0][:40]
    wr = inp["router_w"].clone()
    for e in same:
        wr[e] = wr[same[0]]
    inp["router_w"] = wr
    bias = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
    bias[same] = 50.0
    inp["router_bias"] = bias
    _check(orc, cfg, inp)
    # sigmoid routing with the selection bias doing the lifting
    cfg = cfg.with_(name="run40_sig", routing="sigmoid", sel_bias=True, zipf_bias=False)
    inp2 = dict(G.gpu_inputs(cfg))
    inp2["router_w"] = wr
    inp2["router_bias"] = bias
    _check(orc, cfg, inp2)


@pytest.mark.parametrize("cfg", [
    mi.MoEConfig("k32_e40", T=200, H=512, I=128, E=40, k=32),
    mi.MoEConfig("k32_e1024_sig", T=96, H=512, I=128, E=1024, k=32, routing="sigmoid",
                 sel_bias=True),
    mi.MoEConfig("k31_e1024", T=96, H=1024, I=128, E=1024, k=31)], ids=ids)
def test_router_topk_widest_selection(orc, cfg, tuning):
    # k = 32 fills all 32 lanes with the first candidates, so the only cut that
    # can be proven is after position 31, against every expert not taken out;
    # E = 1024 runs the 32-keys-per-lane kernel
    tuning(router_tile="tc")
    _check(orc, cfg, G.gpu_inputs(cfg))
