"""Pins for the oracle's LatentMoE down projection z = bf16(x Wd^T) ("Kimi K3
... feasibility analysis", s.2.4 routed_expert_down_proj): one nearest-even
rounding of the exact dot product.

Checked against exact rational arithmetic (Python Fractions, with a rounding
written here from the definition of round-half-to-even), on constructed ties
and near-ties that distinguish the rounding mode and a single rounding from a
rounding through fp32, and against an fp64 matrix product on a larger case.
"""
from fractions import Fraction

import numpy as np
import torch


def bf16_u16(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_value(bits: int) -> Fraction:
    f = np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]
    return Fraction(float(f))


def bf16_rne_exact(v: Fraction) -> int:
    """Bits of the bf16 nearest to v, ties to the even significand (normal range)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 7)           # bf16 spacing in [2^e, 2^(e+1))
    n = a / q                            # in [128, 256)
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = np.float32(float(fl * q))
    return sign | int(np.array([val]).view(np.uint32)[0] >> 16)


def exact_z(xb: np.ndarray, wb: np.ndarray) -> np.ndarray:
    T, H = xb.shape
    L = wb.shape[0]
    xv = [[bf16_value(int(b)) for b in row] for row in xb]
    wv = [[bf16_value(int(b)) for b in row] for row in wb]
    out = np.empty((T, L), np.uint16)
    for t in range(T):
        for l in range(L):
            out[t, l] = bf16_rne_exact(sum(a * b for a, b in zip(xv[t], wv[l])))
    return out


def test_latent_down_matches_exact_rationals(orc):
    g = torch.Generator().manual_seed(11)
    x = bf16_u16(torch.randn(4, 96, generator=g))
    w = bf16_u16(torch.randn(12, 96, generator=g) / 10)
    assert np.array_equal(orc.latent_down(x, w), exact_z(x, w))


def test_latent_down_ties_and_single_rounding(orc):
    # rows of Wd against x = (1, 1, 1, 0, ...):
    #   1 + 2^-8           exact midpoint of 1 and 1 + 2^-7: ties to even -> 1
    #   1 + 3 * 2^-8       midpoint of 1 + 2^-7 and 1 + 2^-6: to even -> 1 + 2^-6
    #   1 + 2^-8 + 2^-30   just above the midpoint -> 1 + 2^-7, where a rounding
    #                      through fp32 (1 + 2^-8, then ties to even) gives 1
    #   -(1 + 2^-8 + 2^-30) the same with the sign
    #   2^-20 - 2^-20 + 2^-40 cancellation down to a tiny exact value
    H = 8
    x = torch.zeros(1, H)
    x[0, :3] = 1.0
    rows = [[1, 2 ** -8, 0], [1, 2 ** -7, 2 ** -8], [1, 2 ** -8, 2 ** -30],
            [-1, -(2 ** -8), -(2 ** -30)], [2 ** -20, -(2 ** -20), 2 ** -40]]
    w = torch.zeros(len(rows), H)
    for i, r in enumerate(rows):
        w[i, :3] = torch.tensor(r, dtype=torch.float64).float()
    xb, wb = bf16_u16(x), bf16_u16(w)
    got = orc.latent_down(xb, wb)[0]
    want = exact_z(xb, wb)[0]
    assert np.array_equal(got, want)
    assert got[0] == 0x3F80 and got[1] == 0x3F82 and got[2] == 0x3F81 and got[3] == 0xBF81
    assert got[4] == bf16_rne_exact(Fraction(2) ** -40)


def test_latent_down_matches_fp64_matmul(orc):
    # K = 7168 as in the LatentMoE workload; fp64 sums of exact bf16 products in
    # another order, rounded by integer bit arithmetic
    g = torch.Generator().manual_seed(12)
    x = torch.randn(6, 7168, generator=g).to(torch.bfloat16)
    w = (torch.randn(40, 7168, generator=g) / 7168 ** 0.5).to(torch.bfloat16)
    ref = (x.double() @ w.double().T).numpy()
    b = ref.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = ((b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)).view(np.float64)
    want = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    got = orc.latent_down(bf16_u16(x), bf16_u16(w))
    assert np.array_equal(got, want)
    # token subsets give the same rows
    sub = orc.latent_down(bf16_u16(x), bf16_u16(w), tokens=np.array([4, 1], np.int32))
    assert np.array_equal(sub, got[[4, 1]])
