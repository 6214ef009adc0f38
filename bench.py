"""Benchmark of the fused MoE expert layer on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config decode|prefill|skewed|latent|toy|...]
                    [--also prefill,skewed,latent] [--also-steps 30]
    python bench.py --stage router|route|router_topk|latent_down --dims ... [--steps K]

A step is one moe_forward over one batch (router logits -> top-k -> permute +
fp8 quant -> grouped FFN1 -> requant -> grouped FFN2 -> gather + shared),
inputs resident in HBM.  The default workload is the Ling-style decode batch
(T=512, H=8192, I=2048, 256 experts top-8 + a shared expert, fp8 e4m3
per-channel weights), whose ~12.9 GB of expert weights exceed L2 on every
step, so no flush is needed.  ``value`` is algorithmic bytes per step (touched
expert weights + scales, shared weights, router, x, out) / step time, summed
over ranks; replicas run independent copies (the layer does not shard here).
``--impl reference`` times the CPU oracle on a bounded token sample instead.

On one GPU the line also carries ``workloads``: the other workloads (Ling
prefill T=16384, the skewed-routing T=8192 batch, the Kimi-K3-style LatentMoE
T=4096 batch by default), each timed in the same process after the headline
one, with its own step time, dominant-kernel roofline, grouped-GEMM tensor
rate, clocks and per-stage times.  ``--stage`` times one entry point alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer µs; TFLOP/s (prefill) & weight GB/s (decode) vs GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode")
    ap.add_argument("--no-pack", action="store_true",
                    help="time row-major expert weights instead of the packed tile order")
    ap.add_argument("--fused-combine", action="store_true",
                    help="request MOE_F_FUSED_COMBINE (S7 in the FFN2 epilogue, fp32 sums in "
                         "an order that is not fixed)")
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="tokens per oracle step (default: one per host core)")
    ap.add_argument("--also", default="prefill,skewed,latent",
                    help="other workloads timed after the headline one and reported as nested "
                         "records of the same line (comma list; 'none' for none; one GPU only)")
    ap.add_argument("--also-steps", type=int, default=30,
                    help="timed steps of each nested workload")
    ap.add_argument("--stage", choices=["router", "route", "router_topk", "latent_down"],
                    default=None,
                    help="time one entry point alone instead of the layer (see run_stage)")
    ap.add_argument("--router-tile", default=None,
                    help="router kernel choice (auto, tc or a CUDA-core tile; moe_tuning's "
                         "router_tile); --stage router_topk defaults to tc")
    ap.add_argument("--dims", type=int, nargs="+", default=None,
                    help="with --stage: T H E (router), T E k (route), T H E k (router_topk) "
                         "or T H L (latent_down)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 0.0, "fallback"


def workload_name(cfg):
    kind = {"decode": "Ling-style decode", "prefill": "Ling-style prefill",
            "decode_e32": "Ling-style decode, 32 experts (profiling case)",
            "prefill_e32": "Ling-style prefill, 32 experts (profiling case)",
            "mid": "Ling-style mid-size batch",
            "latent": "Kimi-K3-style LatentMoE",
            "latent_e64": "Kimi-K3-style LatentMoE, 64 experts (profiling case)",
            "latent_k3": "Kimi-K3-style LatentMoE with K3 routing and activation",
            "skewed": "skewed-routing stress (Zipf 1.2 router bias)", "toy": "toy"}.get(cfg.name, cfg.name)
    s = (f"{kind}: T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top-{cfg.k}"
         + (f" + shared expert I_s={cfg.I_s}" if cfg.I_s else "")
         + (f", latent L={cfg.L} (bf16 down/up, RMSNorm)" if cfg.L else "")
         + {"mxfp4": ", MXFP4 e2m1 + e8m0/32 expert weights",
            "fp8_block": ", block-wise fp8 e4m3 weights (fp32 scale per 128x128 block)"}.get(
             cfg.wfmt, ", fp8 e4m3 per-output-channel weights")
         + ", per-token fp8 activations"
         + (", noaux_tc sigmoid routing with selection bias" if cfg.routing == "sigmoid" else "")
         + (", SiTU experts" if cfg.act == "situ" else ""))
    return s


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- helpers
# The sources a committed traffic figure depends on (code only), by the file
# that holds the kernel: the single-SM grouped GEMM by default, the SM-pair
# GEMMs and the MXFP4 GEMMs for the summaries that name them.
DEFAULT_TRAFFIC_SOURCES = ("ffn_gemm.cu", "device.cuh", "internal.h")


def kernel_traffic(kernel: str, cfg_name: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{cfg_name}.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    files = tuple(d.get("source_files", DEFAULT_TRAFFIC_SOURCES))
    try:
        if d.get("source_sha") != source_sha(files):
            return None
    except OSError:
        return None
    return d.get("dram_bytes_per_launch")


def source_sha(files=DEFAULT_TRAFFIC_SOURCES) -> str:
    """Hash of the expert-GEMM sources a traffic figure depends on (by default
    the single-SM grouped GEMM, the device helpers and the argument struct it
    reads), code only (comments and whitespace do not change the kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_expert_layer_02_gb300", "csrc")
    for n in files:
        with open(os.path.join(csrc, n)) as f:
            code = f.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        if n == "internal.h":  # only the kernels' argument struct
            m = re.search(r"struct GroupedFfnArgs \{.*?\};", code, flags=re.S)
            code = m.group(0) if m else code
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def cpu_baseline(cfg, inp_host, n_tokens: int, target_s: float = 10.0):
    """Time the oracle on the first tokens of the batch, sized to about
    ``target_s`` seconds of host work (a one-token-per-core probe sets the
    size) unless ``n_tokens`` fixes it.  Returns (seconds, tokens, threads)."""
    import numpy as np

    import oracle
    threads = oracle.threads()

    def run(n):
        toks = np.arange(min(n, cfg.T), dtype=np.int32)
        t0 = time.perf_counter()
        oracle.moe_forward(cfg.oracle_problem(), inp_host, tokens=toks, nthreads=threads)
        return time.perf_counter() - t0, len(toks)

    if n_tokens:
        dt, n = run(n_tokens)
        return dt, n, threads
    dt, n = run(threads)
    want = int(n * target_s / max(dt, 1e-3)) // threads * threads
    if want > n and n < cfg.T:
        dt, n = run(want)
    return dt, n, threads


def dist_setup(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def max_over_ranks(v: float, ws: int) -> float:
    if ws <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(units_per_rank: float, ms: float, ws: int):
    """Whole-job throughput of ws independent replicas: the units all ranks
    processed over the slowest rank's time.  Returns (value per second, max ms)."""
    ms_max = max_over_ranks(ms, ws)
    return ws * units_per_rank / (ms_max * 1e-3), ms_max


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- arms
def run_reference(args, cfg):
    import torch

    import moe_inputs as mi
    from moe_expert_layer_02_gb300 import accounting as acc
    ws, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = mi.make_inputs(cfg, device=dev)
    host = mi.to_numpy(inp)
    del inp
    import numpy as np

    import oracle
    n = args.ref_tokens or oracle.threads()
    toks = np.arange(min(n, cfg.T), dtype=np.int32)
    for _ in range(args.warmup):
        oracle.moe_forward(cfg.oracle_problem(), host, tokens=toks)
    times = []
    budget_s = 240.0  # keep the whole reference arm within a few minutes
    t_start = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, _, idx, _ = oracle.moe_forward(cfg.oracle_problem(), host, tokens=toks)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    step = statistics.mean(times)
    # per-step work of the sample: the same algorithmic bytes, scaled to the sample
    touched = cfg.E if cfg.T * cfg.k >= 4 * cfg.E else len(np.unique(idx))
    bytes_full = acc.layer_work(cfg, touched)["bytes"]
    frac = len(toks) / cfg.T
    value = bytes_full * frac / step / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(cfg), "parallelism": "replicas",
                   "sample": f"{len(toks)} of {cfg.T} tokens per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"first {len(toks)} of {cfg.T} tokens, whole layer per token "
                                   f"(route, top-{cfg.k} experts, shared), bytes scaled by {frac:.4f}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def load_workload(m, cfg, dev, pack: bool, fused_combine: bool = False, base=None):
    """Device inputs, problem, workspace and output buffer for ``cfg``.  Expert
    weights (and their packed copies) of ``base``, a workload loaded before
    with the same weight shapes, are reused instead of regenerated."""
    import torch

    import moe_inputs as mi
    from moe_expert_layer_02_gb300 import accounting as acc
    shape = (cfg.E, cfg.I, cfg.K, cfg.I_s, cfg.wfmt, cfg.shared_bf16, cfg.H, cfg.L)
    reuse = base if base is not None and base["shape"] == shape else None
    raw = mi.make_inputs(cfg, device=dev, seed=0,
                         expert_weights=reuse["raw"] if reuse is not None else None)
    flags = ((m.F_ROUTER_BIAS if (cfg.zipf_bias or cfg.sel_bias) else 0)
             | (m.F_SHARED_BF16 if cfg.shared_bf16 else 0)
             | (m.F_SIGMOID_ROUTING if cfg.routing == "sigmoid" else 0)
             | (m.F_SITU if cfg.act == "situ" else 0)
             | (m.F_FUSED_COMBINE if fused_combine else 0))
    wfmt = {"fp8": m.W_FP8, "mxfp4": m.W_MXFP4, "fp8_block": m.W_FP8_BLOCK}[cfg.wfmt]
    packed = {}
    if pack and reuse is not None:
        packed = reuse["packed"]
    elif pack:
        # one-time load-time weight preparation (untimed): tile-major expert weights
        pp = m.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, latent=cfg.L, wfmt=wfmt)
        w13p, w2p = torch.empty_like(raw["w13"]), torch.empty_like(raw["w2"])
        packed = dict(w13=w13p, w2=w2p)
        if cfg.wfmt == "mxfp4":  # e8m0 scales regrouped into per-stage tensor-memory images
            s13p, s2p = torch.empty_like(raw["w13_scale"]), torch.empty_like(raw["w2_scale"])
            m.moe_pack_weights(pp, raw["w13"], raw["w2"], raw["w13_scale"], raw["w2_scale"], w13p,
                               w2p, s13p, s2p)
            packed.update(w13_scale=s13p, w2_scale=s2p)
        else:
            m.moe_pack_weights(pp, raw["w13"], raw["w2"], None, None, w13p, w2p)
        if cfg.I_s and not cfg.shared_bf16:
            ps = m.make_problem(cfg.T, cfg.H, cfg.I_s, 1, 1)
            s13, s2 = torch.empty_like(raw["sw13"]), torch.empty_like(raw["sw2"])
            m.moe_pack_weights(ps, raw["sw13"], raw["sw2"], None, None, s13, s2)
            packed.update(sw13=s13, sw2=s2)
        torch.cuda.synchronize()
    if pack:
        flags |= m.F_PACKED_WEIGHTS
    inp = dict(raw, **packed)
    p = m.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, I_shared=cfg.I_s, latent=cfg.L,
                       wfmt=wfmt, flags=flags)
    wsb = torch.empty(m.moe_workspace_bytes(p), dtype=torch.uint8, device=dev)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    # touched experts (for algorithmic bytes): routing through the library itself
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
    tidx = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
    tw = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    m.moe_router_logits(p, raw["x"], raw["router_w"], raw["router_bias"], logits)
    m.moe_route(p, logits, raw["router_bias"], tidx, tw)
    touched = int(torch.unique(tidx).numel())
    del logits, tidx, tw

    def step(x=None, y=None):
        m.moe_forward(p, inp["x"] if x is None else x, inp["router_w"], inp["router_bias"],
                      inp["w13"], inp["w13_scale"], inp["w2"], inp["w2_scale"], inp["sw13"],
                      inp["sw13_scale"], inp["sw2"], inp["sw2_scale"], inp["wd"], inp["wu"],
                      inp["gamma"], out if y is None else y, wsb)

    return {"cfg": cfg, "shape": shape, "raw": raw, "packed": packed, "inp": inp, "p": p,
            "wsb": wsb, "out": out, "touched": touched, "work": acc.layer_work(cfg, touched),
            "step": step, "pack": pack}


def timed_run(m, W, steps: int, warmup: int, ws_n: int, local: int):
    """Warm-up, a per-stage table (every stage timed, up to 20 steps), then the
    timed region: ``steps`` steps bracketed by CUDA events on the launching
    stream, with only the grouped-GEMM launches (FFN1, FFN2) also bracketed
    for their live kernel times, and the SM clocks sampled meanwhile."""
    import torch
    step = W["step"]
    stream = torch.cuda.current_stream()
    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    rc = m.moe_get_last_error()
    if rc != 0:
        raise SystemExit(f"device error word {rc} after warm-up ({W['cfg'].name})")
    m.moe_profile_read()
    m.moe_profile_enable(True)
    for _ in range(min(steps, 20)):
        step()
    torch.cuda.synchronize()
    m.moe_profile_enable(False)
    stage_ms, stage_n = m.moe_profile_read()

    clocks = ClockSampler(local)
    time.sleep(0.2)
    m.moe_profile_enable(True, stages=["ffn1", "ffn2"])
    n0 = m.moe_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_n)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(ws_n)
    launches = m.moe_launch_count() - n0
    m.moe_profile_enable(False)
    live_ms, live_n = m.moe_profile_read()
    clk = clocks.stop()
    rc = m.moe_get_last_error()
    if rc != 0:
        raise SystemExit(f"device error word {rc} after the timed region ({W['cfg'].name})")
    return {"ms": ev0.elapsed_time(ev1) / steps, "launches": launches, "clocks": clk,
            "stages_ms": {k: v / max(stage_n[k], 1) for k, v in stage_ms.items()},
            "ffn1_ms": live_ms["ffn1"] / max(live_n["ffn1"], 1),
            "ffn2_ms": live_ms["ffn2"] / max(live_n["ffn2"], 1)}


def peak_clock_mhz():
    """Median SM clock under which the sustained bf16 peak was measured."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["clocks_under_load"]["sm_mhz_median"])
    except Exception:
        return None


def roofline_record(m, W, R, ms_step):
    """The dominant kernel's roofline (FFN1, from its live CUDA-event time) and
    the grouped GEMMs' tensor rate against the fp8 peak."""
    from moe_expert_layer_02_gb300 import accounting as acc
    cfg, touched = W["cfg"], W["touched"]
    hbm, bf16, bf16_sus, src = peaks()
    rows = cfg.R + (cfg.T if (cfg.I_s and not cfg.shared_bf16) else 0)
    ffn1_bytes = acc.ffn1_launch_bytes(cfg, touched)
    ffn1_flops = acc.ffn1_flops(rows, cfg.K, cfg.I)
    ffn2_flops = acc.ffn2_flops(rows, cfg.K, cfg.I)
    # decode-like batches stream weights (HBM-bound); large batches are bound by
    # the fp8 tensor rate, taken as 2 x the measured bf16 rate (nominal ratio),
    # sustained figure because the kernel runs inside a seconds-long loop
    fp8_peak = 2.0 * (bf16_sus or bf16)
    t_hbm = ffn1_bytes / (hbm * 1e9)
    t_mma = ffn1_flops / (fp8_peak * 1e12)
    ms1 = R["ffn1_ms"]
    if t_hbm >= t_mma:
        ach = ffn1_bytes / (ms1 * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"hbm_gbs of {src}"}
    else:
        ach = ffn1_flops / (ms1 * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": ach / fp8_peak,
                "peak_source": f"2 x bf16_tflops_sustained of {src} (fp8 = 2 x bf16 nominal ratio)"}
    plan = m.moe_describe(W["p"])
    ffn1_kernel = plan.split()[0].split("=", 1)[1]
    work = W["work"]
    roof.update({"kernel": f"{ffn1_kernel} (W1|W3 + SiLU*gate)",
                 "traffic": kernel_traffic("ffn1", cfg.name),
                 "algorithmic_bytes_per_launch": ffn1_bytes, "flops_per_launch": ffn1_flops,
                 "avg_launch_ms": ms1,
                 "layer_hbm_frac": (work["bytes"] / (ms_step * 1e-3) / 1e9) / hbm,
                 "layer_tensor_frac": (work["flops_fp8"] / (ms_step * 1e-3) / 1e12) / fp8_peak})
    # grouped expert GEMMs (FFN1 + FFN2) against the fp8 tensor peak, and the
    # same at the clock the peak was measured under (time x SM MHz on both sides)
    gg_tflops = (ffn1_flops + ffn2_flops) / ((R["ffn1_ms"] + R["ffn2_ms"]) * 1e-3) / 1e12
    pk_mhz = peak_clock_mhz()
    run_mhz = (R["clocks"] or {}).get("sm_mhz")
    gg = {"ffn1_ms": R["ffn1_ms"], "ffn2_ms": R["ffn2_ms"], "flops": ffn1_flops + ffn2_flops,
          "tflops": gg_tflops, "fp8_peak_tflops": fp8_peak, "frac_of_fp8_peak": gg_tflops / fp8_peak,
          "peak_sm_mhz": pk_mhz, "run_sm_mhz": run_mhz,
          "frac_of_fp8_peak_at_run_clock": (gg_tflops / (fp8_peak * run_mhz / pk_mhz)
                                            if (pk_mhz and run_mhz) else None)}
    return roof, gg, plan


def workload_record(m, W, args, ws_n, local, steps):
    """One nested record of the bench line: another workload timed in the same
    process after the headline one."""
    cfg = W["cfg"]
    R = timed_run(m, W, steps, args.warmup, ws_n, local)
    value, ms_max = replica_value(W["work"]["bytes"] / 1e9, R["ms"], ws_n)
    roof, gg, plan = roofline_record(m, W, R, ms_max)
    return {"workload": workload_name(cfg), "steps": steps, "ms_per_step": ms_max,
            "value": value, "unit": "GB/s", "latency_us": ms_max * 1e3,
            "tflops_fp8": W["work"]["flops_fp8"] / (ms_max * 1e-3) / 1e12,
            "touched_experts": W["touched"], "roofline": roof, "grouped_gemms": gg,
            "clocks": R["clocks"], "stages_ms": R["stages_ms"], "gpu_launches": R["launches"],
            "plan": plan}


def run_ours(args, cfg):
    import torch

    import moe_expert_layer_02_gb300 as m
    import moe_inputs as mi
    from moe_expert_layer_02_gb300 import build as mb

    ws_n, rank, local = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    mb.build()
    m.load_library()
    dev = torch.device("cuda", local)
    pack = not args.no_pack
    W = load_workload(m, cfg, dev, pack, fused_combine=args.fused_combine)
    p, inp, out, step = W["p"], W["inp"], W["out"], W["step"]
    work = W["work"]
    stream = torch.cuda.current_stream()
    R = timed_run(m, W, args.steps, args.warmup, ws_n, local)
    ms = R["ms"]

    # the same step replayed from a CUDA graph (as a serving loop would run a
    # captured layer): the kernels' launch cost leaves the host entirely
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
        torch.cuda.synchronize()
        reps = max(min(args.steps, 100), 3)
        gev0, gev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gev0.record(stream)
        for _ in range(reps):
            g.replay()
        gev1.record(stream)
        torch.cuda.synchronize()
        graph_ms = gev0.elapsed_time(gev1) / reps
        del g
    except RuntimeError as e:  # capture refused: report the eager numbers only
        print(f"graph replay not measured: {e}", file=sys.stderr)
    rc = m.moe_get_last_error()
    if rc != 0:
        raise SystemExit(f"device error word {rc} after the graph replays")

    # end to end through the public call with host buffers: every step's x is
    # copied in from pinned host memory and its output copied back, on a copy
    # stream with two device buffers each way, so step i+1's upload and step
    # i's download overlap step i's layer (as a serving loop would run them)
    x_host = inp["x"].cpu().pin_memory()
    out_host = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
    x_dev = [torch.empty_like(inp["x"]) for _ in range(2)]
    y_dev = [torch.empty_like(out) for _ in range(2)]
    copy = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(args.steps // 2, 3)
    barrier(ws_n)
    torch.cuda.synchronize()
    e0.record(copy)
    with torch.cuda.stream(copy):
        x_dev[0].copy_(x_host, non_blocking=True)
        ev_in[0].record(copy)
    for i in range(e2e_steps):
        b = i & 1
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # step i-2's output has left y_dev[b]
        step(x_dev[b], y_dev[b])
        ev_done[b].record(stream)
        with torch.cuda.stream(copy):
            if i + 1 < e2e_steps:
                if i >= 1:
                    copy.wait_event(ev_done[b ^ 1])  # step i-1 no longer reads x_dev[b^1]
                x_dev[b ^ 1].copy_(x_host, non_blocking=True)
                ev_in[b ^ 1].record(copy)
            copy.wait_event(ev_done[b])
            out_host.copy_(y_dev[b], non_blocking=True)
            ev_out[b].record(copy)
    stream.wait_event(ev_out[(e2e_steps - 1) & 1])
    e1.record(stream)
    torch.cuda.synchronize()
    # the pipelined steps computed the same layer (bit for bit, except that the
    # fused combine's fp32 sums add in an order that is not fixed: there the
    # outputs may differ by a bf16 ulp, and by more near zero, where the
    # cancelling terms' rounding shows)
    last = y_dev[(e2e_steps - 1) & 1]
    if not args.fused_combine:
        same = torch.equal(last, out)
    else:
        o = out.float()
        rms = float(o.pow(2).mean().sqrt())
        same = bool(((last.float() - o).abs() <= o.abs() * 2.0 ** -7 + 2.0 ** -7 * rms).all())
    if not same:
        raise SystemExit("end-to-end output differs from the device-timed output")
    bytes_step = work["bytes"]
    value, ms_max = replica_value(bytes_step / 1e9, ms, ws_n)
    e2e_value, e2e_ms = replica_value(bytes_step / 1e9, e0.elapsed_time(e1) / e2e_steps, ws_n)
    roof, gg, plan = roofline_record(m, W, R, ms_max)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E,
                   "top_k": cfg.k, "I_shared": cfg.I_s, "touched_experts": W["touched"],
                   "parallelism": "replicas" if ws_n > 1 else "single",
                   "weights": "tile-major (moe_pack_weights, untimed)" if pack else "row-major",
                   "plan": plan,
                   "l2": "inputs larger than L2 (%.1f GB of weights per step), no flush" % (
                       (work["bytes_weights_routed"] + work["bytes_weights_shared"]) / 1e9)},
        "latency_us": ms_max * 1e3,
        "tflops_fp8": work["flops_fp8"] / (ms_max * 1e-3) / 1e12,
        "roofline": roof,
        "grouped_gemms": gg,
        "stages_ms": R["stages_ms"],
        "gpu_launches": R["launches"],
        "graph_ms_per_step": graph_ms,
        "clocks": R["clocks"],
        "e2e": {"value": e2e_value, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": out_host.numel() * 2},
    }
    del x_dev, y_dev, x_host, out_host
    if rank == 0 and ws_n == 1:
        host = mi.to_numpy({k: v for k, v in W["raw"].items()})
        dt, n, cores = cpu_baseline(cfg, host, args.ref_tokens)
        del host
        frac = n / cfg.T
        line["cpu_baseline"] = {
            "value": bytes_step * frac / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {cfg.T} tokens, whole layer per token, bytes scaled by {frac:.4f}",
            "seconds": dt}
    # the other workloads of the layer, each timed in this process after the
    # headline one (weights of equal shape are shared with it)
    extra = [] if (ws_n > 1 or args.also in ("", "none")) else [
        n for n in args.also.split(",") if n and n != cfg.name]
    if extra:
        line["workloads"] = {}
        for name in extra:
            # a nested workload that fails is recorded as such; the headline
            # record above was measured already and is still printed
            try:
                Wx = load_workload(m, mi.CONFIGS[name], dev, pack, base=W)
                line["workloads"][name] = workload_record(m, Wx, args, ws_n, local,
                                                          args.also_steps)
                del Wx
            except (Exception, SystemExit) as exc:  # noqa: BLE001
                print(f"bench.py: workload {name} failed: {exc!r}", file=sys.stderr, flush=True)
                line["workloads"][name] = {"error": repr(exc)[:300]}
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_stage(args):
    """Time one entry point alone on seeded inputs (for profiling a stage under
    ncu without a whole layer's weights on the device): ``--stage router
    --dims T H E`` (moe_router_logits), ``--stage route --dims T E k``
    (moe_route), ``--stage router_topk --dims T H E k`` (moe_router_topk on
    the tensor-core path) or ``--stage latent_down --dims T H L``
    (moe_latent_down).
    x ~ N(0,1) bf16, router weights ~ N(0,1/H) fp32, logits ~ N(0,1), Wd ~
    N(0,1/H) bf16, generated on the device from seed 0."""
    import torch

    import moe_expert_layer_02_gb300 as m
    from moe_expert_layer_02_gb300 import build as mb
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --stage needs a CUDA device")
    mb.build()
    m.load_library()
    g = torch.Generator(device="cuda").manual_seed(0)
    if args.stage == "router":
        T, H, E = args.dims
        x = torch.randn(T, H, device="cuda", generator=g).to(torch.bfloat16)
        w = torch.randn(E, H, device="cuda", generator=g) / H ** 0.5
        out = torch.empty(T, E, device="cuda")
        p = m.make_problem(T, H, 128, E, 1)
        call = lambda: m.moe_router_logits(p, x, w, None, out)  # noqa: E731
        work, unit = 2.0 * T * H * E, "TFLOP/s"
    elif args.stage == "router_topk":
        T, H, E, k = args.dims
        x = torch.randn(T, H, device="cuda", generator=g).to(torch.bfloat16)
        w = torch.randn(E, H, device="cuda", generator=g) / H ** 0.5
        idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
        wt = torch.empty(T, k, device="cuda")
        m.moe_set_tuning(router_tile=args.router_tile or "tc")
        p = m.make_problem(T, H, 128, E, k)
        wsb = torch.empty(m.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        call = lambda: m.moe_router_topk(p, x, w, None, idx, wt, wsb)  # noqa: E731
        work, unit = 2.0 * T * H * E, "TFLOP/s"
    elif args.stage == "latent_down":
        T, H, L = args.dims
        x = torch.randn(T, H, device="cuda", generator=g).to(torch.bfloat16)
        wd = (torch.randn(L, H, device="cuda", generator=g) / H ** 0.5).to(torch.bfloat16)
        z = torch.empty(T, L, dtype=torch.bfloat16, device="cuda")
        p = m.make_problem(T, H, 128, 8, 1, latent=L, wfmt=m.W_MXFP4)
        wsb = torch.empty(m.moe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        call = lambda: m.moe_latent_down(p, x, wd, z, wsb)  # noqa: E731
        work, unit = 2.0 * T * H * L, "TFLOP/s"
    else:
        T, E, k = args.dims
        logits = torch.randn(T, E, device="cuda", generator=g)
        idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
        wt = torch.empty(T, k, device="cuda")
        p = m.make_problem(T, 128, 128, E, k)
        call = lambda: m.moe_route(p, logits, None, idx, wt)  # noqa: E731
        work, unit = 4.0 * T * E, "GB/s"
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(args.steps):
        call()
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    status = m.moe_get_last_error()
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"stage": args.stage, "dims": args.dims, "us_per_call": ms * 1e3,
                      "rate": rate, "unit": unit, "status": status}), flush=True)
    if status:
        raise SystemExit(f"device error {status}")
    return 0


def main():
    args = parse()
    if args.stage:
        want = 4 if args.stage == "router_topk" else 3
        if not args.dims or len(args.dims) != want:
            raise SystemExit(f"--stage {args.stage} needs --dims with {want} numbers")
        return run_stage(args)
    import moe_inputs as mi
    cfg = mi.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
