"""GPU parity of the whole layer (moe_forward, S1..S8 in one call) against the
oracle's per-token definition, in the launch configuration bench.py uses."""
import numpy as np
import pytest
import torch

import _gpu as G
import moe_inputs as mi
from test_gpu_stages import BIASED, E3, KE, MAXE, RAGGED, SKEW_SMALL, T1

pytestmark = pytest.mark.gpu

SHARED_SMALL = mi.MoEConfig("small_shared", T=96, H=256, I=128, E=6, k=3, I_s=128)
SMALL = [mi.CONFIGS["toy"], SHARED_SMALL, RAGGED, MAXE, T1, KE, E3, BIASED.with_(I_s=128)]
FULL = [mi.CONFIGS["decode"], mi.CONFIGS["prefill"], mi.CONFIGS["skewed"]]
ids = lambda c: c.name


def run_forward(cfg, inp, out=None, ws=None, packed=False):
    m = G.lib()
    p = G.problem(cfg, packed=packed)
    ws = G.workspace(p) if ws is None else ws
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda") if out is None else out
    m.moe_forward(p, inp["x"], inp["router_w"], inp["router_bias"], inp["w13"], inp["w13_scale"],
                  inp["w2"], inp["w2_scale"], inp["sw13"], inp["sw13_scale"], inp["sw2"],
                  inp["sw2_scale"], inp["wd"], inp["wu"], inp["gamma"], out, ws)
    return out


def _check(orc, cfg, n_sample):
    m = G.lib()
    inp = G.gpu_inputs(cfg)
    out = run_forward(cfg, inp)
    assert m.moe_get_last_error() == 0
    h = G.host(inp)
    toks = G.sample_tokens(cfg.T, n_sample, seed=11)
    ref_f, ref_b, _, _ = orc.moe_forward(cfg.oracle_problem(), h, tokens=toks)
    got = G.bf16_values(G.bf16_bits(out))[toks]
    return G.assert_close(got, ref_f, f"moe_forward {cfg.name}")


@pytest.mark.parametrize("bn", [32, 128])
@pytest.mark.parametrize("cfg", [SHARED_SMALL, RAGGED, KE], ids=ids)
def test_forward_small_gathered_rows(orc, cfg, bn, tuning):
    # ffn1_gather: S4 writes one fp8 row per token and the FFN1 producer
    # gathers each tile's rows by token, instead of the default permuted rows
    # that FFN1 reads by TMA
    tuning(ffn1_gather=1)
    tuning(tile_n=bn)
    assert "ffn1_rows=gathered" in G.lib().moe_describe(G.problem(cfg))
    _check(orc, cfg, n_sample=cfg.T)


@pytest.mark.parametrize("rows", ["permuted", "gathered"])
@pytest.mark.parametrize("small", ["m128", "m256"])
@pytest.mark.parametrize("cfg", [SHARED_SMALL, RAGGED, SKEW_SMALL.with_(I_s=256)], ids=ids)
def test_forward_sm_pairs(orc, cfg, small, rows, tuning):
    # 256-row tiles on SM pairs for a small batch: items of <= 128 rows as
    # M = 128 tiles, or as padded M = 256 tiles; FFN1 reads permuted rows or
    # gathers one row per token with four-row TMA copies
    tuning(tile_n=256, ffn1_gather=int(rows == "gathered"))
    if small == "m256":
        tuning(pair_small=0)
    d = G.lib().moe_describe(G.problem(cfg))
    assert "ffn1=pair_gemm_kernel" in d and f"ffn1_rows={rows}" in d, d
    _check(orc, cfg, n_sample=cfg.T)


@pytest.mark.parametrize("cfg", SMALL, ids=ids)
def test_forward_small(orc, cfg):
    _check(orc, cfg, n_sample=10 ** 9)


def test_pack_is_a_tile_permutation():
    # packed[e, rb, kb, r, :] == w[e, rb*128 + r, kb*128 : kb*128 + 128]
    cfg = SHARED_SMALL.with_(I=256, H=384)
    inp = G.gpu_inputs(cfg)
    pk = G.pack(cfg, inp)
    for key, R, C in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        w, p = inp[key], pk[key]
        tiles = p.view(cfg.E, R // 128, C // 128, 128, 128)
        back = tiles.permute(0, 1, 3, 2, 4).reshape(cfg.E, R, C)
        assert torch.equal(back, w), key


@pytest.mark.parametrize("cfg", [SHARED_SMALL, RAGGED, KE], ids=ids)
def test_forward_packed_weights_small(orc, cfg):
    m = G.lib()
    inp = G.gpu_inputs(cfg)
    out = run_forward(cfg, G.pack(cfg, inp), packed=True)
    assert m.moe_get_last_error() == 0
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref, f"packed {cfg.name}")


def full_size_tokens(orc, cfg, h, seed):
    """Every token of the decode batch; for the larger batches at least 256
    tokens, among them the token of every expert's last routed row (its last,
    partly filled tile item) and tokens of the most loaded expert."""
    if cfg.T <= 512:
        return np.arange(cfg.T, dtype=np.int32)
    return G.edge_tokens(orc, cfg, h, 256, seed=seed)


@pytest.mark.parametrize("cfg", FULL, ids=ids)
def test_forward_packed_weights_full_size(orc, cfg):
    m = G.lib()
    inp = G.gpu_inputs(cfg)
    out = run_forward(cfg, G.pack(cfg, inp), packed=True)
    assert m.moe_get_last_error() == 0
    h = G.host(inp)
    toks = full_size_tokens(orc, cfg, h, seed=21)
    assert len(toks) >= min(cfg.T, 256)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), h, tokens=toks)
    G.assert_close(G.bf16_values(G.bf16_bits(out))[toks], ref, f"packed {cfg.name}")


@pytest.mark.parametrize("cfg", FULL, ids=ids)
def test_forward_full_size(orc, cfg):
    m = G.lib()
    inp = G.gpu_inputs(cfg)
    out = run_forward(cfg, inp)
    assert m.moe_get_last_error() == 0
    h = G.host(inp)
    toks = full_size_tokens(orc, cfg, h, seed=11)
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), h, tokens=toks)
    G.assert_close(G.bf16_values(G.bf16_bits(out))[toks], ref, f"moe_forward {cfg.name}")


def test_forward_deterministic_and_counted():
    m = G.lib()
    cfg = SHARED_SMALL
    inp = G.gpu_inputs(cfg)
    n0 = m.moe_launch_count()
    a = G.bf16_bits(run_forward(cfg, inp))
    n1 = m.moe_launch_count()
    b = G.bf16_bits(run_forward(cfg, inp))
    assert np.array_equal(a, b)
    # routing, then index (one launch for a batch this small), scatter, ffn1,
    # requant, ffn2, combine
    assert n1 - n0 == G.routing_launches(G.problem(cfg)) + 6


def test_profile_counts_each_stage():
    m = G.lib()
    cfg = SHARED_SMALL
    inp = G.gpu_inputs(cfg)
    m.moe_profile_read()
    m.moe_profile_enable(True)
    try:
        run_forward(cfg, inp)
        run_forward(cfg, inp)
        ms, n = m.moe_profile_read()
    finally:
        m.moe_profile_enable(False)
    base = ("router", "topk", "index", "scatter", "ffn1", "requant", "ffn2", "combine")
    assert all(n[k] == 2 for k in base), n
    assert all(ms[k] > 0 for k in base), ms
    assert all(n[k] == 0 for k in n if k not in base)  # LatentMoE stages idle
    # a stage mask times the named stages only
    m.moe_profile_enable(True, stages=["ffn1", "combine"])
    try:
        run_forward(cfg, inp)
        ms, n = m.moe_profile_read()
    finally:
        m.moe_profile_enable(False)
    assert n["ffn1"] == 1 and n["combine"] == 1 and sum(n.values()) == 2, n


def test_empty_batch_is_a_noop():
    m = G.lib()
    cfg = mi.CONFIGS["toy"].with_(T=0)
    inp = G.gpu_inputs(mi.CONFIGS["toy"])
    p = G.problem(cfg)
    ws = G.workspace(p)
    n0 = m.moe_launch_count()
    out = torch.empty(0, cfg.H, dtype=torch.bfloat16, device="cuda")
    m.moe_forward(p, inp["x"], inp["router_w"], None, inp["w13"], inp["w13_scale"], inp["w2"],
                  inp["w2_scale"], None, None, None, None, None, None, None,
                  torch.empty(16, dtype=torch.bfloat16, device="cuda"), ws)
    assert m.moe_launch_count() == n0


def test_all_tokens_to_one_expert(orc):
    # a router whose bias sends every token to experts 5 (and 2 for k=2):
    # one expert holds every row, the rest are empty
    m = G.lib()
    cfg = mi.MoEConfig("one_hot_route", T=200, H=256, I=128, E=8, k=2, zipf_bias=True)
    inp = G.gpu_inputs(cfg)
    bias = torch.full((cfg.E,), -100.0, device="cuda")
    bias[5] = 100.0
    bias[2] = 50.0
    inp = dict(inp, router_bias=bias)
    out = run_forward(cfg, inp)
    assert m.moe_get_last_error() == 0
    h = G.host(inp)
    ref_f, _, idx, _ = orc.moe_forward(cfg.oracle_problem(), h)
    assert np.all(idx[:, 0] == 5) and np.all(idx[:, 1] == 2)
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref_f, "one-expert routing")
