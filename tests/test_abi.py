"""The C-ABI library loads on the host, exports every symbol include/moe.h
declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import torch  # noqa: F401  (loads the CUDA runtime the library links)
    from moe_expert_layer_02_gb300 import build
    build.build()
    import moe_expert_layer_02_gb300 as mm
    mm.load_library()
    return mm


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(m):
    names = declared_functions()
    assert "moe_forward" in names and "moe_permute" in names and len(names) >= 12
    lib = m.load_library()
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(m):
    lib = m.load_library()
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(5) == b"MOE_ERR_TIMEOUT"


def test_workspace_bytes(m):
    p = m.make_problem(512, 8192, 2048, 256, 8, I_shared=2048)
    ws = m.moe_workspace_bytes(p)
    # the permuted fp8 rows, bf16 intermediate and bf16 expert outputs dominate
    rows = 512 * 8 + 512
    assert ws >= rows * 8192 + rows * 2048 * 3 + rows * 8192 * 2
    assert m.moe_workspace_bytes(m.make_problem(0, 8192, 2048, 256, 8)) > 0
    assert m.moe_workspace_bytes(m.make_problem(4, 100, 2048, 256, 8)) == 0  # H % 128


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(H=100), dict(I=0), dict(E=0), dict(top_k=9, E=8), dict(top_k=33, E=64),
    dict(E=2048), dict(I_shared=100), dict(wfmt=7),
])
def test_invalid_problems_rejected_on_host(m, bad):
    base = dict(T=4, H=256, I=128, E=8, top_k=2)
    base.update(bad)
    p = m.make_problem(**base)
    lib = m.load_library()
    assert lib.moe_forward(ctypes.byref(p), *([ctypes.c_void_p(256)] * 16), 1 << 30, None) == 1
    assert lib.moe_workspace_bytes(ctypes.byref(p)) == 0


def test_null_and_workspace_checks(m):
    lib = m.load_library()
    p = m.make_problem(4, 256, 128, 8, 2)
    args = [ctypes.c_void_p(256)] * 16  # x .. ws
    assert lib.moe_forward(ctypes.byref(p), *([None] + args[1:]), 1 << 30, None) == 1
    assert lib.moe_forward(ctypes.byref(p), *(args[:15] + [None]), 1 << 30, None) == 3
    assert lib.moe_forward(ctypes.byref(p), *args, 16, None) == 3
    # misaligned x
    bad = [ctypes.c_void_p(258)] + args[1:]
    assert lib.moe_forward(ctypes.byref(p), *bad, 1 << 30, None) == 1
    # a latent width that is not a multiple of 256 is valid but not implemented
    q = m.make_problem(4, 256, 128, 8, 2, latent=128, wfmt=m.W_MXFP4)
    assert lib.moe_forward(ctypes.byref(q), *args, 1 << 30, None) == 2
    # MXFP4 experts need K (here H) to be a multiple of 256
    q = m.make_problem(4, 384, 128, 8, 2, wfmt=m.W_MXFP4)
    assert lib.moe_forward(ctypes.byref(q), *args, 1 << 30, None) == 2


def test_pack_weights_checks(m):
    lib = m.load_library()
    a, b, c, d = (ctypes.c_void_p(v) for v in (256, 512, 768, 1024))
    p = m.make_problem(4, 256, 128, 8, 2)
    assert lib.moe_pack_weights(ctypes.byref(p), a, b, None, None, a, d, None, None, None) == 1
    assert lib.moe_pack_weights(ctypes.byref(p), a, None, None, None, c, d, None, None, None) == 1
    assert lib.moe_pack_weights(ctypes.byref(p), ctypes.c_void_p(260), b, None, None, c, d,
                                None, None, None) == 1
    assert lib.moe_pack_weights(ctypes.byref(m.make_problem(4, 256, 100, 8, 2)), a, b, None,
                                None, c, d, None, None, None) == 1
    q = m.make_problem(4, 256, 128, 8, 2, wfmt=7)
    assert lib.moe_pack_weights(ctypes.byref(q), a, b, None, None, c, d, None, None, None) == 1


def test_argument_counts_match_header(m):
    # every binding declares exactly the parameters of its C prototype
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lib = m.load_library()
    for name, params in re.findall(r"\b(moe_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", src):
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        fn = getattr(lib, name)
        if fn.argtypes is not None:
            assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def test_binding_names_match_c_names(m):
    for n in declared_functions():
        if n != "moe_status_string":
            assert hasattr(m, n), n


def test_describe_names_the_kernels(m):
    p = m.make_problem(512, 8192, 2048, 256, 8, I_shared=2048)
    assert m.moe_describe(p).startswith("ffn1=grouped_ffn_kernel<FFN1,BN=128>")
    q = m.make_problem(16384, 8192, 2048, 256, 8, I_shared=2048)
    assert "pair_gemm_kernel<FFN1,BN=256>" in m.moe_describe(q)
    x = m.make_problem(4096, 7168, 3072, 896, 16, I_shared=6144, latent=3584, wfmt=m.W_MXFP4,
                       flags=m.F_SHARED_BF16)
    assert "grouped_mx_kernel<FFN1,BN=96>" in m.moe_describe(x)
    lib = m.load_library()
    buf = ctypes.create_string_buffer(8)
    assert lib.moe_describe(ctypes.byref(p), buf, 8) == 1  # too short
    assert lib.moe_describe(ctypes.byref(m.make_problem(4, 100, 128, 8, 2)), buf, 8) == 1


def test_describe_names_the_router(m, tuning):
    # the tensor-core router with its exact selection by default, at every
    # size; a CUDA-core tile when one is chosen
    for T in (1, 512, 16384):
        assert "router=tensor-cores" in m.moe_describe(m.make_problem(T, 8192, 2048, 256, 8))
    tuning(router_tile="8x16")
    assert "router=cuda-cores" in m.moe_describe(m.make_problem(512, 8192, 2048, 256, 8))


def test_fused_combine_plan(m):
    # honoured on the single-SM fp8 GEMMs: the fp32 sum [T, H] replaces the
    # bf16 y rows [T*k + T, H] in the workspace; ignored on the SM-pair GEMMs
    d = m.make_problem(512, 8192, 2048, 256, 8, I_shared=2048)
    f = m.make_problem(512, 8192, 2048, 256, 8, I_shared=2048, flags=m.F_FUSED_COMBINE)
    assert "combine=gather" in m.moe_describe(d)
    assert "combine=fused" in m.moe_describe(f)
    wd, wf = m.moe_workspace_bytes(d), m.moe_workspace_bytes(f)
    assert wd - wf == (512 * 8 + 512) * 8192 * 2 - 512 * 8192 * 4
    pr = m.make_problem(16384, 8192, 2048, 256, 8, I_shared=2048, flags=m.F_FUSED_COMBINE)
    assert "combine=gather" in m.moe_describe(pr)
    lat = m.make_problem(4096, 7168, 3072, 896, 16, I_shared=6144, latent=3584, wfmt=m.W_MXFP4,
                         flags=m.F_SHARED_BF16 | m.F_FUSED_COMBINE)
    assert "combine=gather-rmsnorm" in m.moe_describe(lat)


def test_mx_pair_plan(m):
    # the MXFP4 GEMMs run on SM pairs only with packed weights and paired blocks
    f = m.F_SHARED_BF16
    lat = dict(I_shared=6144, latent=3584, wfmt=m.W_MXFP4)
    d = m.moe_describe(m.make_problem(4096, 7168, 3072, 896, 16, flags=f, **lat))
    assert "ffn1=grouped_mx_kernel" in d and "ffn2=grouped_mx_kernel" in d
    d = m.moe_describe(m.make_problem(4096, 7168, 3072, 896, 16, flags=f | m.F_PACKED_WEIGHTS, **lat))
    assert "ffn1=grouped_mx_pair_kernel" in d and "ffn2=grouped_mx_pair_kernel" in d
    # I = 384 gives three 128-row blocks: FFN1 stays on single SMs
    d = m.moe_describe(m.make_problem(80, 512, 384, 12, 3, wfmt=m.W_MXFP4, flags=m.F_PACKED_WEIGHTS))
    assert "ffn1=grouped_mx_kernel" in d and "ffn2=grouped_mx_pair_kernel" in d


def test_row_gather_plan(m, tuning):
    # ffn1_gather: the fp8 per-channel FFN1 (single-SM or SM pairs) gathers
    # its rows by token, at any tile height; the block-wise and MXFP4 paths
    # read permuted rows, and so does everything by default
    dec = lambda: m.moe_describe(m.make_problem(512, 8192, 2048, 256, 8, I_shared=2048))
    d = dec()
    assert "ffn1=grouped_ffn_kernel<FFN1,BN=128>" in d and "ffn1_rows=permuted" in d, d
    tuning(ffn1_gather=1)
    assert "ffn1_rows=gathered" in dec()
    tuning(tile_n=32)
    assert "BN=32> " in dec() and "ffn1_rows=gathered" in dec()
    tuning(tile_n=0)
    # SM pairs gather with four-row TMA copies
    assert "ffn1_rows=gathered" in m.moe_describe(m.make_problem(16384, 8192, 2048, 256, 8,
                                                                 I_shared=2048))
    assert "ffn1_rows=permuted" in m.moe_describe(m.make_problem(512, 8192, 2048, 256, 8,
                                                                 wfmt=m.W_FP8_BLOCK))
    assert "ffn1_rows=permuted" in m.moe_describe(m.make_problem(512, 8192, 2048, 256, 8,
                                                                 wfmt=m.W_MXFP4))


@pytest.mark.parametrize("tile,want", [(32, (32, 32, 32)), (64, (64, 64, 64)),
                                       (96, (None, None, 96)), (128, (128, None, None)),
                                       (256, (256, None, None)), (0, (None, None, None))])
def test_tile_override_respects_the_format(m, tuning, tile, want):
    # a tile height is taken only where the format has kernels for it (fp8
    # per-channel 32/64/128/256, block-wise 32/64, MXFP4 32/64/96); anything
    # else, and 0, leaves the automatic choice (~16 rows per expert: 128 for
    # fp8 per-channel, 32 for the others)
    tuning(tile_n=tile)
    for fmt, w, auto in zip((m.W_FP8, m.W_FP8_BLOCK, m.W_MXFP4), want, (128, 32, 32)):
        d = m.moe_describe(m.make_problem(512, 8192, 2048, 256, 8, wfmt=fmt))
        bn = int(re.search(r"ffn1=\w+<FFN1,BN=(\d+)>", d).group(1))
        assert bn == (w if w is not None else auto), (fmt, d)


@pytest.mark.parametrize("T,want", [(1, "grouped_ffn_kernel<FFN1,BN=128>"),
                                    (512, "grouped_ffn_kernel<FFN1,BN=128>"),
                                    (3072, "grouped_ffn_kernel<FFN1,BN=128>"),  # 96 rows / expert
                                    (3104, "pair_gemm_kernel<FFN1,BN=256>"),    # 97 rows / expert
                                    (16384, "pair_gemm_kernel<FFN1,BN=256>")])
def test_tile_height_follows_rows_per_expert(m, T, want):
    # fp8 per-channel: 128-row single-SM tiles up to 96 mean rows per expert
    # (the weight stream is fastest there with a four-stage ring), 256-row
    # tiles on SM pairs above
    d = m.moe_describe(m.make_problem(T, 8192, 2048, 256, 8, I_shared=2048))
    assert d.startswith("ffn1=" + want), d


def test_tuning_round_trip_and_range_checks(m, tuning):
    base = m.moe_get_tuning()
    assert base["pair_small"] in (0, 1) and base["pdl"] in (0, 1)
    tuning(tile_n=64, router_tile="8x16s4", pdl=0)
    t = m.moe_get_tuning()
    assert t["tile_n"] == 64 and t["router_tile"] == 3 and t["pdl"] == 0
    for bad in (dict(tile_n=48), dict(router_tile=5), dict(router_tile=7), dict(ffn1_gather=2),
                dict(pdl=-1)):
        with pytest.raises(m.MoEError) as ei:
            m.moe_set_tuning(**bad)
        assert ei.value.status == 1  # MOE_ERR_INVALID_ARG, nothing changed
        assert m.moe_get_tuning() == t
    lib = m.load_library()
    assert lib.moe_get_tuning(None) == 1 and lib.moe_set_tuning(None) == 1
    with m.tuned(tile_n=32):
        assert m.moe_get_tuning()["tile_n"] == 32
    assert m.moe_get_tuning() == t
