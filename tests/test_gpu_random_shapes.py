"""GPU parity of the whole layer on seeded random shapes and launch choices.

Each case draws, from its own seed, one of six problem kinds (fp8 per-channel
experts with and without the shared expert, the same on SM pairs, block-wise
fp8, MXFP4, LatentMoE) inside the shapes the library accepts (T, H, I, E, k,
the shared expert and the latent projection, softmax or sigmoid routing,
SwiGLU or SiTU, row-major or packed weights) and the launch knobs a caller can
set (tile height, the row path of FFN1, the index kernels, single-SM or
SM-pair GEMMs, the router tile), runs moe_forward once, and compares every
token with the oracle under the layer's tolerance.  The draws cover corners
the named cases do not: one expert, k = E, ragged tails of every tile height,
single-token batches."""
import numpy as np
import pytest

import _gpu as G
import moe_inputs as mi
from test_gpu_forward import run_forward

pytestmark = pytest.mark.gpu

KINDS = ("fp8", "fp8_shared", "fp8_block", "mxfp4", "latent", "fp8_pair")
N_CASES = 150


def draw(seed: int):
    r = np.random.default_rng(7000 + seed)
    kind = KINDS[seed % len(KINDS)]
    wide = kind in ("mxfp4", "latent", "fp8_pair")  # H a multiple of 256
    H = int(256 * r.integers(1, 4)) if wide else int(128 * r.integers(1, 7))
    I = int(128 * r.integers(1, 5))
    E = int(r.choice([1, 2, 3, 5, 8, 13, 24, 40, 64]))
    k = int(r.integers(1, min(E, 8) + 1))
    T = int(r.choice([1, 2, 7, 33, 64, 100, 161, 257, 400]))
    if kind == "fp8_pair":  # enough rows for both M = 256 and M = 128 pair tiles
        T = int(r.choice([64, 257, 400, 700]))
    kw = dict(T=T, H=H, I=I, E=E, k=k)
    if kind in ("fp8_shared", "fp8_pair") or (kind == "fp8_block" and r.random() < 0.5):
        kw["I_s"] = I
    if kind == "fp8_block":
        kw["wfmt"] = "fp8_block"
    if kind == "mxfp4":
        kw["wfmt"] = "mxfp4"
    if kind == "latent":
        kw["L"] = int(256 * r.integers(1, H // 256 + 1))
        kw["wfmt"] = str(r.choice(["mxfp4", "fp8", "fp8_block"]))
        kw["I_s"] = int(128 * r.integers(0, 4))
        kw["shared_bf16"] = kw["I_s"] > 0
    if r.random() < 0.3:
        kw.update(routing="sigmoid", sel_bias=True)
    elif r.random() < 0.3:
        kw["zipf_bias"] = True
    if r.random() < 0.3:
        kw["act"] = "situ"
    cfg = mi.MoEConfig(f"rand{seed}_{kind}", **kw)

    tiles = {"fp8": (32, 64, 128, 256), "fp8_block": (32, 64), "mxfp4": (32, 64, 96)}[
        "mxfp4" if cfg.wfmt == "mxfp4" else cfg.wfmt]
    knobs = {}
    if r.random() < 0.6:
        knobs["tile_n"] = int(r.choice(tiles))
    if r.random() < 0.3:
        knobs["ffn1_gather"] = 1
    if r.random() < 0.3:
        knobs["index_3pass"] = 1
    if kind == "fp8_pair":  # 256-row tiles on SM pairs
        knobs["tile_n"] = 256
    elif r.random() < 0.2:
        knobs["gemm_1cta"] = 1
    if r.random() < 0.2:
        knobs["pair_small"] = 0
    if r.random() < 0.3:
        knobs["mx_1cta"] = 1
    if r.random() < 0.5:
        knobs["router_tile"] = str(r.choice(["8x8", "8x16", "8x16s4", "12w8x16", "tc"]))
    # the MXFP4 SM-pair kernels need packed weights
    packed = bool(r.random() < (0.8 if cfg.wfmt == "mxfp4" else 0.5))
    return cfg, knobs, packed


@pytest.mark.parametrize("seed", range(N_CASES))
def test_forward_random_shape(orc, seed, tuning):
    cfg, knobs, packed = draw(seed)
    tuning(**knobs)
    m = G.lib()
    p = G.problem(cfg, packed=packed)
    what = f"{cfg} tuning={knobs} packed={packed} plan: {m.moe_describe(p)}"
    inp = G.gpu_inputs(cfg)
    out = run_forward(cfg, G.pack(cfg, inp) if packed else inp, packed=packed)
    assert m.moe_get_last_error() == 0, what
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref, what,
                   bf16_store_allowance=cfg.wfmt == "fp8_block")
