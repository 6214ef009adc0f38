"""GPU parity of the LatentMoE down projection z = bf16(x Wd^T) ("Kimi K3 ...
feasibility analysis", s.2.4 routed_expert_down_proj) through moe_latent_down:
bit for bit against the oracle's exactly rounded z, on the whole LatentMoE
batch, on ragged small shapes, and on constructed ties and near-ties that only
the exact recomputation of flagged elements gets right."""
import numpy as np
import pytest
import torch

import _gpu as G
import moe_inputs as mi

pytestmark = pytest.mark.gpu


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _gpu_z(T, H, L, x, wd):
    m = G.lib()
    p = m.make_problem(T, H, 128, 8, 2, latent=L, wfmt=m.W_MXFP4)
    ws = G.workspace(p)
    z = torch.full((T, L), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    m.moe_latent_down(p, x, wd, z, ws)
    assert m.moe_get_last_error() == 0
    return _u16(z)


def test_latent_down_bit_exact_full_batch(orc):
    cfg = mi.CONFIGS["latent"]
    inp = G.gpu_inputs(cfg)
    got = _gpu_z(cfg.T, cfg.H, cfg.L, inp["x"], inp["wd"])
    want = orc.latent_down(_u16(inp["x"]), _u16(inp["wd"]))
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} of {got.size} z elements differ, first {bad[:4].tolist()}"


@pytest.mark.parametrize("T,H,L,seed", [(1, 256, 256, 1), (100, 512, 256, 2),
                                        (300, 1024, 768, 3), (257, 2048, 512, 4)])
def test_latent_down_bit_exact_ragged(orc, T, H, L, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wd = (torch.randn(L, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    got = _gpu_z(T, H, L, x.cuda(), wd.cuda())
    assert np.array_equal(got, orc.latent_down(_u16(x), _u16(wd)))


def test_latent_down_ties_and_near_ties(orc):
    # Among random rows, token 0 = (1, 1, 1, 0, ...) against weight rows whose
    # exact products sum to a bf16 midpoint (ties to even), to just above one
    # (1 + 2^-8 + 2^-30: a sum rounded to fp32 first would land on the midpoint
    # and round down), or cancel to a tiny value.
    T, H, L = 64, 512, 256
    g = torch.Generator().manual_seed(7)
    x = torch.randn(T, H, generator=g)
    wd = torch.randn(L, H, generator=g) / H ** 0.5
    x[0] = 0.0
    x[0, :3] = 1.0
    rows = [[1, 2 ** -8, 0], [1, 2 ** -7, 2 ** -8], [1, 2 ** -8, 2 ** -30],
            [-1, -(2 ** -8), -(2 ** -30)], [2 ** -20, -(2 ** -20), 2 ** -40]]
    for i, r in enumerate(rows):
        wd[i, :3] = torch.tensor(r, dtype=torch.float64).float()
    x, wd = x.to(torch.bfloat16), wd.to(torch.bfloat16)
    got = _gpu_z(T, H, L, x.cuda(), wd.cuda())
    want = orc.latent_down(_u16(x), _u16(wd))
    assert np.array_equal(got, want)
    assert got[0, 0] == 0x3F80 and got[0, 1] == 0x3F82 and got[0, 2] == 0x3F81
    assert got[0, 3] == 0xBF81
