"""Algorithmic work of the fused MoE layer: FLOPs and bytes per step.

The formulas follow the cost model of the Ling-2.6-1T Fused MoE V2 write-up
(s.1 "MoE kernel cost model": FFN1 = 2 matrices x 2*M*H*I per expert, FFN2 =
2*M*I*H, shared expert = 3 matrices x 2*T*H*I_s, fp8 expert weights = 3*H*I
bytes) and the Kimi-K3 report (s.2.4 expert size 3*L*I, s.2.5 MXFP4 at 4 bits +
one 8-bit scale per 32 elements).  Only work the method must do is counted:
weights (and scales) of experts that received at least one row, the shared
expert's weights, router weights, the input x and the output; intermediates
(permuted rows, h, y) are excluded.
"""
from __future__ import annotations


def ffn1_flops(rows: int, K: int, I: int) -> int:
    """Gate + up projections for ``rows`` routed rows: 2 matrices x 2*rows*K*I."""
    return 2 * (2 * rows * K * I)


def ffn2_flops(rows: int, K: int, I: int) -> int:
    """Down projection: 2*rows*I*K."""
    return 2 * rows * I * K


def swiglu_ffn_flops(rows: int, K: int, I: int) -> int:
    return ffn1_flops(rows, K, I) + ffn2_flops(rows, K, I)


def shared_flops(T: int, H: int, I_s: int) -> int:
    """Shared expert on every token: 3 matrices x 2*T*H*I_s."""
    return 3 * (2 * T * H * I_s)


def expert_weight_bytes(K: int, I: int, wfmt: str = "fp8", with_scales: bool = True) -> float:
    """Bytes of one routed expert (W1, W3 [I, K] and W2 [K, I])."""
    n = 3 * K * I
    if wfmt == "fp8":
        return n + (4 * (2 * I + K) if with_scales else 0)
    if wfmt == "fp8_block":  # one fp32 scale per 128 x 128 block
        return n + (4 * 3 * (K // 128) * (I // 128) if with_scales else 0)
    if wfmt == "mxfp4":
        return n / 2 + (n / 32 if with_scales else 0)
    raise ValueError(wfmt)


def bits_per_element(wfmt: str) -> float:
    return {"fp8": 8.0, "mxfp4": 4.0 + 8.0 / 32.0, "fp8_block": 8.0 + 32.0 / (128 * 128)}[wfmt]


def router_flops(T: int, H: int, E: int) -> int:
    return 2 * T * H * E


def layer_work(cfg, touched_experts: int) -> dict:
    """FLOPs by precision and algorithmic bytes for one forward step of ``cfg``.

    ``cfg`` is a moe_inputs.MoEConfig-like object (T, H, I, E, k, I_s, L, wfmt,
    shared_bf16); ``touched_experts`` is the number of experts with >= 1 row.
    """
    T, H, I, E, k, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.K
    R = T * k
    flops_routed = swiglu_ffn_flops(R, K, I)
    flops_shared = shared_flops(T, H, cfg.I_s) if cfg.I_s else 0
    flops_bf16 = 0
    if cfg.L:
        flops_bf16 += 2 * (2 * T * H * cfg.L)  # down_proj + up_proj
    if cfg.shared_bf16:
        flops_bf16 += flops_shared
        flops_shared = 0
    w_routed = touched_experts * expert_weight_bytes(K, I, cfg.wfmt)
    if cfg.I_s:
        w_shared = 3 * H * cfg.I_s * (2 if cfg.shared_bf16 else 1)
        if not cfg.shared_bf16:
            w_shared += (4 * 3 * (H // 128) * (cfg.I_s // 128) if cfg.wfmt == "fp8_block"
                         else 4 * (2 * cfg.I_s + H))
    else:
        w_shared = 0
    w_latent = 2 * (2 * H * cfg.L) + 2 * cfg.L if cfg.L else 0
    router = 4 * E * H + (4 * E if getattr(cfg, "zipf_bias", False) else 0)
    io = 2 * T * H * 2  # x in, out, both bf16
    return {
        "flops_fp8": flops_routed + flops_shared,  # e4m3 x e4m3 or e4m3 x e2m1
        "flops_bf16": flops_bf16,
        "flops_router_fp32": router_flops(T, H, E),
        "bytes_weights_routed": w_routed,
        "bytes_weights_shared": w_shared,
        "bytes": w_routed + w_shared + w_latent + router + io,
    }


def _matrix_bytes(rows: int, cols: int, wfmt: str) -> float:
    """Bytes of one weight matrix with its scales (fp8: fp32 per row; fp8_block:
    fp32 per 128 x 128 block; mxfp4: 4-bit elements + one e8m0 byte per 32)."""
    if wfmt == "fp8":
        return rows * cols + 4 * rows
    if wfmt == "fp8_block":
        return rows * cols + 4 * (rows // 128) * (cols // 128)
    return rows * cols / 2 + rows * cols / 32


def ffn1_launch_bytes(cfg, touched_experts: int) -> float:
    """Algorithmic bytes of one grouped FFN1 launch: touched W1|W3 (+ scales),
    shared W1|W3, and the quantised rows it reads / the bf16 h it writes."""
    K, I = cfg.K, cfg.I
    b = touched_experts * _matrix_bytes(2 * I, K, cfg.wfmt)
    rows = cfg.T * cfg.k
    if cfg.I_s and not cfg.shared_bf16:
        b += _matrix_bytes(2 * cfg.I_s, K, "fp8_block" if cfg.wfmt == "fp8_block" else "fp8")
        rows_s = cfg.T
    else:
        rows_s = 0
    b += (rows + rows_s) * K + (rows * I + rows_s * cfg.I_s) * 2
    return b


def ffn2_launch_bytes(cfg, touched_experts: int) -> float:
    K, I = cfg.K, cfg.I
    b = touched_experts * _matrix_bytes(K, I, cfg.wfmt)
    rows = cfg.T * cfg.k
    rows_s = cfg.T if (cfg.I_s and not cfg.shared_bf16) else 0
    if rows_s:
        b += _matrix_bytes(K, cfg.I_s, "fp8_block" if cfg.wfmt == "fp8_block" else "fp8")
    b += rows * I + rows_s * cfg.I_s + (rows + rows_s) * K * 2
    return b
