"""The FLOP/byte formulas used for the roofline reproduce the numbers printed in
the Ling-2.6-1T cost model and the Kimi-K3 LatentMoE/MXFP4 sections
(tests/golden/ling_cost_model.txt, tests/golden/k3_latent_moe.txt)."""
import math
import os

import pytest

import moe_inputs as mi
from moe_expert_layer_02_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v, _ = line.split()
                d[k] = float(v)
    return d


def _round_to(printed, value):
    """True when ``value`` rounds or truncates to ``printed`` at the printed precision."""
    s = repr(printed)
    dec = len(s.split(".")[1]) if "." in s and not s.endswith(".0") else 0
    trunc = math.floor(value * 10 ** dec + 1e-9) / 10 ** dec
    return round(value, dec) == printed or abs(trunc - printed) < 1e-9


def test_ling_cost_model():
    g = _golden("ling_cost_model.txt")
    H, I, ep, T, k, E = 8192, 2048, 32, 16384, 8, 256
    rows = T * k // ep
    assert rows == g["routed_rows_per_device"]
    local = E // ep
    m = rows // local
    ffn1 = local * (acc.ffn1_flops(m, H, I) // 1)
    ffn2 = local * acc.ffn2_flops(m, H, I)
    assert _round_to(g["ffn1_gflop"], ffn1 / 1e9)
    assert _round_to(g["ffn2_gflop"], ffn2 / 1e9)
    assert _round_to(g["routed_gflop"], (ffn1 + ffn2) / 1e9)
    sh = acc.shared_flops(rows, H, I)
    assert _round_to(g["shared_gflop"], sh / 1e9)
    tot = ffn1 + ffn2 + sh
    assert _round_to(g["total_gflop"], tot / 1e9)
    assert _round_to(g["compute_bound_ms"], tot / (g["fp8_peak_per_device_tflops"] * 1e12) * 1e3)
    assert rows * H == g["scatter_elements"]
    assert _round_to(g["scatter_bf16_mb"], rows * H * 2 / 1e6)
    assert _round_to(g["scatter_fp8_mb"], rows * H * 1 / 1e6)
    wb = acc.expert_weight_bytes(H, I, "fp8", with_scales=False)
    assert _round_to(g["expert_weight_mb"], wb / 1e6)
    assert _round_to(g["local_expert_weights_mb"], local * wb / 1e6)
    t1 = local * wb / (g["hbm_per_device_tbs"] * 1e12) * 1e3
    assert _round_to(g["weight_read_once_ms"], t1)
    tiles = math.ceil(m / 160)
    assert tiles == g["token_tiles_bts160"]
    assert _round_to(g["weight_read_bts160_ms"], tiles * t1)


def test_k3_latent_moe_numbers():
    g = _golden("k3_latent_moe.txt")
    cfg = mi.CONFIGS["latent"]
    assert (cfg.H, cfg.L, cfg.I, cfg.E, cfg.k, cfg.I_s) == (
        g["hidden"], g["latent"], g["expert_intermediate"], g["experts"], g["top_k"],
        g["shared_intermediate"])
    per = 3 * cfg.L * cfg.I
    assert _round_to(g["params_per_expert_m"], per / 1e6)
    assert _round_to(g["params_per_layer_b"], cfg.E * per / 1e9)
    assert acc.bits_per_element("mxfp4") == g["mxfp4_bits_per_element"]
    b = acc.expert_weight_bytes(cfg.L, cfg.I, "mxfp4")
    assert b * 8 / per == g["mxfp4_bits_per_element"]


def test_layer_work_decode():
    cfg = mi.CONFIGS["decode"]
    w = acc.layer_work(cfg, touched_experts=256)
    # 256 experts x 3 x 8192 x 2048 fp8 bytes = 12.88 GB of routed weights
    assert abs(w["bytes_weights_routed"] / 1e9 - 12.89) < 0.01
    assert w["flops_fp8"] == 4 * 4096 * 8192 * 2048 + 2 * 4096 * 2048 * 8192 + 6 * 512 * 8192 * 2048
