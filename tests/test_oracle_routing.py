"""Pins for the oracle's routing and permutation (S1-S4).

S1 is checked against an fp64 matmul within a rigorous fp32 error bound; S2
against a library sort on (-logit, index) and against "softmax over all E, take
top-k, renormalise"; S3/S4 against a stable argsort by expert, bijection and
marker-payload invariants, and the e4m3 rounding bound.
"""
import itertools

import numpy as np
import pytest
import torch

import moe_inputs as mi


def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_val(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("T,H,E", [(7, 256, 8), (33, 200, 13), (5, 8192, 256)])
def test_router_logits_vs_fp64(orc, T, H, E):
    rng = np.random.default_rng(T + H + E)
    x = _bf16_bits(rng.standard_normal((T, H)))
    wr = (rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32)
    xd = _bf16_val(x)
    exact = xd @ wr.astype(np.float64).T
    got = orc.router_logits(x, wr)
    # fp32 summation bound: |err| <= gamma_n * sum |x||w|, n = H/32 + 5 steps
    n = H // 32 + 1 + 5
    u = 2.0 ** -24
    bound = (n * u / (1 - n * u)) * (np.abs(xd) @ np.abs(wr.astype(np.float64)).T) + 1e-30
    assert np.all(np.abs(got - exact) <= bound)
    gb = orc.router_logits(x, wr, bias)
    assert np.array_equal(gb, (got + bias).astype(np.float32))


def test_router_logits_is_the_canonical_order(orc):
    # A case where the fixed order is visible: partial sums that cancel.  Lane 0
    # gets +2^24 then +1 (lost in fp32), lane 16 gets -2^24: tree adds lane 16
    # into lane 0 at the first step, giving 0 (not 1).
    H = 64
    x = np.zeros((1, H), np.float32)
    w = np.zeros((1, H), np.float32)
    x[0, 0], w[0, 0] = 1.0, 2.0 ** 24
    x[0, 32], w[0, 32] = 1.0, 1.0
    x[0, 16], w[0, 16] = 1.0, -(2.0 ** 24)
    got = orc.router_logits(_bf16_bits(x), w)
    assert got[0, 0] == 0.0
    # moving the +1 to lane 1 makes it survive (different partial)
    x[0, 32], x[0, 33], w[0, 33] = 0.0, 1.0, 1.0
    got = orc.router_logits(_bf16_bits(x), w)
    assert got[0, 0] == 1.0


def _topk_by_sort(row, k):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (8, 8), (5, 3), (256, 8), (896, 16), (3, 1)])
def test_topk_vs_library_sort(orc, E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 64
    lg = rng.standard_normal((T, E)).astype(np.float32)
    # constructed exact ties: duplicate some columns
    if E >= 4:
        lg[:, 1] = lg[:, 3]
        lg[: T // 2, 0] = lg[: T // 2, 2]
    idx, w = orc.topk(lg, k)
    for t in range(T):
        assert list(idx[t]) == _topk_by_sort(lg[t], k)
    # weights == softmax over all E, take top-k, renormalise
    full = np.exp(lg.astype(np.float64) - lg.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    sel = np.take_along_axis(full, idx.astype(np.int64), 1)
    ref = sel / sel.sum(1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-12, atol=0)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)


def test_topk_brute_force_subsets(orc):
    rng = np.random.default_rng(7)
    E = 6
    for trial in range(200):
        lg = rng.integers(-3, 3, size=(1, E)).astype(np.float32)  # many ties
        for k in range(1, E + 1):
            idx, _ = orc.topk(lg, k)
            best = None
            for sub in itertools.combinations(range(E), k):
                s = sum(float(lg[0, e]) for e in sub)
                if best is None or s > best[0] or (s == best[0] and sub < best[1]):
                    best = (s, sub)
            assert tuple(sorted(idx[0])) == best[1]
            vals = lg[0, idx[0]]
            assert np.all(vals[:-1] >= vals[1:])


def test_topk_ties_pick_lower_index(orc):
    lg = np.zeros((1, 16), np.float32)
    idx, w = orc.topk(lg, 4)
    assert list(idx[0]) == [0, 1, 2, 3]
    assert np.allclose(w, 0.25)
    idx, w = orc.topk(lg, 1)
    assert idx[0, 0] == 0 and w[0, 0] == 1.0


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (100, 13, 4), (513, 256, 8), (1, 5, 5)])
def test_permute_vs_stable_sort(orc, T, E, k):
    rng = np.random.default_rng(T + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    cnt, off, perm, src = orc.permute(idx, E)
    flat = idx.reshape(-1)
    assert np.array_equal(cnt, np.bincount(flat, minlength=E))
    assert off[0] == 0 and off[-1] == T * k and np.all(np.diff(off) == cnt)
    order = np.argsort(flat, kind="stable")  # sorts (t, j) pairs by expert, keeping token order
    assert np.array_equal(src, order // k)
    rows = np.empty(T * k, np.int64)
    rows[order] = np.arange(T * k)
    assert np.array_equal(perm.reshape(-1), rows)
    assert np.array_equal(np.sort(perm.reshape(-1)), np.arange(T * k))  # bijection
    assert np.all(src[perm] == np.arange(T)[:, None])


def test_permute_marker_payload(orc):
    # x[t,:] = t; scatter rows by perm, gather back by perm -> identity, elementwise
    T, E, k = 50, 7, 3
    rng = np.random.default_rng(3)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    cnt, off, perm, src = orc.permute(idx, E)
    x = np.repeat(np.arange(T, dtype=np.float64)[:, None], 16, axis=1)
    rows = np.empty((T * k, 16))
    rows[perm.reshape(-1)] = np.repeat(x, k, axis=0)
    assert np.array_equal(rows[:, 0], src.astype(np.float64))
    for e in range(E):
        seg = rows[off[e]:off[e + 1], 0]
        assert np.all(np.diff(seg) > 0)  # stable: increasing token ids within an expert
        assert np.all(np.isin(seg.astype(int), np.nonzero((idx == e).any(1))[0]))
    back = rows[perm]  # [T, k, 16]
    assert np.array_equal(back, np.repeat(x[:, None, :], k, axis=1))


def test_quant_rows_bounds(orc):
    rng = np.random.default_rng(4)
    T, H = 40, 512
    xf = rng.standard_normal((T, H)) * rng.uniform(1e-3, 1e3, size=(T, 1))
    xf[3] = 0.0
    x = _bf16_bits(xf)
    s, q = orc.quant_rows(x)
    xv = _bf16_val(x)
    amax = np.abs(xv).max(1)
    assert s[3] == 1.0 and np.all(q[3] == 0)
    nz = amax > 0
    assert np.array_equal(s[nz], (amax[nz].astype(np.float32) / np.float32(448.0)))
    dec = orc.e4m3_decode(q) * s[:, None].astype(np.float64)
    # the largest element maps to +-448 exactly
    am = np.abs(xv).argmax(1)
    assert np.all(np.abs(orc.e4m3_decode(q[np.arange(T), am]))[nz] == 448.0)
    # RNE error: half a quantum of the e4m3 binade (relative 2^-4), or half the
    # subnormal spacing 2^-10 * s
    err = np.abs(dec - xv)
    bound = np.maximum(np.abs(xv) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)


def test_zipf_bias_is_a_valid_log_distribution():
    cfg = mi.CONFIGS["skewed"].with_(T=4, H=128, I=128)
    inp = mi.make_inputs(cfg)
    b = inp["router_bias"].double()
    assert torch.allclose(torch.exp(b / 2).sum(), torch.tensor(1.0, dtype=torch.float64), atol=1e-5)
    r = torch.argsort(-b) + 0  # experts by rank
    p = torch.exp(b / 2)[r]
    ratio = p[0] / p[1]
    assert abs(float(ratio) - 2.0 ** 1.2) < 1e-3


def test_combine_one_hot_rows(orc):
    # y row r is the unit vector e_{r mod H} (bf16 1.0): out[t] counts, at each
    # column, how many of the token's rows land there; plus a shared row of 0.5.
    T, k, H = 9, 3, 16
    rng = np.random.default_rng(8)
    perm = np.stack([rng.permutation(T * k)[:k] for _ in range(T)]).astype(np.int32)
    y = np.zeros((T * k, H), np.float32)
    y[np.arange(T * k), np.arange(T * k) % H] = 1.0
    sh = np.full((T, H), 0.5, np.float32)
    out = orc.combine(_bf16_bits(y), perm, _bf16_bits(sh))
    expect = np.full((T, H), 0.5)
    for t in range(T):
        for j in range(k):
            expect[t, perm[t, j] % H] += 1.0
    assert np.array_equal(_bf16_val(out), expect)
    out2 = orc.combine(_bf16_bits(y), perm)
    assert np.array_equal(_bf16_val(out2), expect - 0.5)


# ----------------------------------------------------------------------------- sigmoid (noaux_tc)
def _ulps(a, ref):
    a = np.asarray(a, np.float64)
    spacing = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return np.abs(a - ref) / spacing


def test_exp_canon_accuracy(orc):
    # the canonical fp32 exp against the mathematics (fp64 exp) on (-86, 0]
    a = np.concatenate([np.linspace(-85.99, 0.0, 40001), -np.logspace(-8, 1.9, 2001),
                        [0.0, -1e-30, -0.5, -1.0, -np.log(2.0)]]).astype(np.float32)
    got = orc.exp_canon(a)
    ref = np.exp(a.astype(np.float64))
    assert _ulps(got, ref).max() <= 2.0
    assert orc.exp_canon(np.float32(0.0)) == 1.0
    assert np.all(np.diff(got[:40001]) >= 0)  # monotone on the increasing grid
    assert orc.exp_canon(np.float32(-86.0)) == 0.0 and orc.exp_canon(np.float32(-200.0)) == 0.0


def test_sigmoid_canon_accuracy_and_symmetry(orc):
    l = np.concatenate([np.linspace(-30, 30, 20001), [0.0, 1e-6, -1e-6, 85.0, -85.0]]).astype(np.float32)
    got = orc.sigmoid_canon(l).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    assert _ulps(got, ref).max() <= 3.0
    assert orc.sigmoid_canon(np.float32(0.0)) == 0.5
    pair = orc.sigmoid_canon(l).astype(np.float64) + orc.sigmoid_canon(-l).astype(np.float64)
    assert np.abs(pair - 1.0).max() <= 2 ** -22


def test_topk_sigmoid_without_bias_follows_the_logits(orc):
    # sigmoid is increasing, so with no bias the selection is the softmax one
    # (the pinned routine above), away from fp32 saturation of the sigmoid
    rng = np.random.default_rng(3)
    lg = rng.uniform(-2, 2, (300, 48)).astype(np.float32)
    i1, w1 = orc.topk(lg, 6, "sigmoid")
    i2, _ = orc.topk(lg, 6)
    assert np.array_equal(i1, i2)
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(lg, i1, 1).astype(np.float64)))
    assert np.allclose(w1, s / s.sum(1, keepdims=True), rtol=1e-6)


def test_topk_sigmoid_with_bias_brute_force(orc):
    # keys = score + bias in fp32; selection by a library sort (descending key,
    # then ascending index); weights are the unbiased scores renormalised
    rng = np.random.default_rng(4)
    T, E, k = 200, 40, 5
    lg = rng.standard_normal((T, E)).astype(np.float32)
    b = (0.05 * rng.standard_normal(E)).astype(np.float32)
    idx, w = orc.topk(lg, k, "sigmoid", b)
    sc = orc.sigmoid_canon(lg)
    key = (sc + b[None, :]).astype(np.float32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -key[t].astype(np.float64)))
        assert list(idx[t]) == list(order[:k])
        chosen = sc[t, idx[t]].astype(np.float64)
        assert np.allclose(w[t], chosen / chosen.sum(), rtol=0, atol=1e-15)
    # the bias changes some selections (it is not ignored)
    i0, _ = orc.topk(lg, k, "sigmoid")
    assert not np.array_equal(i0, idx)


def test_topk_sigmoid_ties_pick_lower_index(orc):
    lg = np.zeros((1, 6), np.float32)
    b = np.array([0.0, 0.1, 0.0, 0.1, 0.0, 0.0], np.float32)
    idx, w = orc.topk(lg, 4, "sigmoid", b)
    assert list(idx[0]) == [1, 3, 0, 2]
    assert np.allclose(w[0], 0.25)
