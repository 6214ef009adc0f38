"""moe_permute_static: the expert permutation for callers that cannot allocate.

Some callers of this library have no device memory to lend it: a host that
plans every byte of GPU memory in advance and gives a plugin only its input and
output buffers, or a latency-critical loop where cudaMalloc is off limits
because it can synchronise the whole device.  moe_permute_static serves them by
keeping its two scratch tables in a fixed array inside libmoe.so instead of a
caller workspace.  These tests call it through the C ABI and require exactly
the results of moe_permute (which uses a caller workspace) on two calls in a
row of different sizes, so stale contents left in the shared array by the
first call would show up in the second; and they check that a problem too big
for the fixed array is refused before anything is launched.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import _gpu as G

STATIC_TABLE = 1 << 19  # entries per scratch table inside the library


def _outputs(T, E, k, H, seed):
    m = G.lib()
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32).cuda()
    x = (torch.randn(T, H, generator=g) * 3).to(torch.bfloat16).cuda()
    p = m.make_problem(T, H, 128, E, k)
    res = []
    for use_static in (False, True):
        d = lambda *shape, dt=torch.int32: torch.full(shape, -7, dtype=dt, device="cuda")
        outs = [d(E), d(E + 1), d(T, k), d(T * k), d(T * k, H, dt=torch.uint8),
                d(T * k, dt=torch.float32)]
        if use_static:
            m.moe_permute_static(p, idx, x, *outs)
        else:
            m.moe_permute(p, idx, x, *outs, G.workspace(p))
        assert m.moe_get_last_error() == 0
        res.append([o.cpu().numpy() for o in outs])
    return res


@pytest.mark.gpu
def test_static_permute_matches_workspace_version_two_calls_in_a_row():
    # first a decode-sized problem, then a smaller ragged one with other E and k
    for T, E, k, H, seed in ((512, 256, 8, 8192, 1), (300, 13, 4, 256, 2)):
        ref, got = _outputs(T, E, k, H, seed)
        names = ("counts", "offsets", "perm", "src_row", "xq_perm", "xscale_perm")
        for name, a, b in zip(names, ref, got):
            if a.dtype == np.float32:
                a, b = a.view(np.uint32), b.view(np.uint32)
            assert np.array_equal(a, b), name


@pytest.mark.gpu
def test_static_permute_fills_its_scratch_exactly():
    # E * ceil(T/32) == 2^19: the largest problem the fixed tables admit, so the
    # last entry of each table (and the second table's start) is used
    T, E, k, H = 16384, 1024, 2, 128
    assert E * ((T + 31) // 32) == STATIC_TABLE
    ref, got = _outputs(T, E, k, H, 3)
    for a, b in zip(ref, got):
        if a.dtype == np.float32:
            a, b = a.view(np.uint32), b.view(np.uint32)
        assert np.array_equal(a, b)


def test_static_permute_refuses_problems_beyond_its_scratch():
    m = G.lib()
    E = 1024
    T = (STATIC_TABLE // E + 1) * 32  # one chunk more than the tables hold
    p = m.make_problem(T, 256, 128, E, 2)
    dummy = torch.empty(16, dtype=torch.int32)  # never touched: refused on the host
    with pytest.raises(m.MoEError) as ei:
        m.moe_permute_static(p, dummy, torch.empty(16, dtype=torch.bfloat16), dummy, dummy, dummy,
                             dummy, torch.empty(16, dtype=torch.uint8),
                             torch.empty(16, dtype=torch.float32), stream=0)
    assert ei.value.status == 3  # MOE_ERR_WORKSPACE
