"""Time one entry point of libmoe.so on seeded synthetic inputs.

    python -m moe_expert_layer_02_gb300.stagebench router T H E [--iters N]
    python -m moe_expert_layer_02_gb300.stagebench route  T E k [--iters N]

A micro-benchmark of a single stage (e.g. to profile it alone under ncu without
holding a whole layer's weights on the device); the layer itself is timed by
bench.py.  Inputs: x ~ N(0,1) bf16 [T,H], router weights ~ N(0,1/H) fp32
[E,H], logits ~ N(0,1) fp32 [T,E]; generated on the device from seed 0.
Prints one JSON line with the mean time per call (CUDA events) and the rate.
"""
from __future__ import annotations

import argparse
import json


def main(argv=None):
    import torch

    from . import build, load_library, make_problem, moe_get_last_error, moe_route, \
        moe_router_logits

    ap = argparse.ArgumentParser()
    ap.add_argument("stage", choices=["router", "route"])
    ap.add_argument("dims", type=int, nargs=3)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    a = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("stagebench needs a CUDA device")
    build.build()
    load_library()
    g = torch.Generator(device="cuda").manual_seed(0)
    if a.stage == "router":
        T, H, E = a.dims
        x = torch.randn(T, H, device="cuda", generator=g).to(torch.bfloat16)
        w = torch.randn(E, H, device="cuda", generator=g) / H ** 0.5
        out = torch.empty(T, E, device="cuda")
        p = make_problem(T, H, 128, E, 1)
        call = lambda: moe_router_logits(p, x, w, None, out)  # noqa: E731
        work, unit = 2.0 * T * H * E, "TFLOP/s"
    else:
        T, E, k = a.dims
        logits = torch.randn(T, E, device="cuda", generator=g)
        idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
        wt = torch.empty(T, k, device="cuda")
        p = make_problem(T, 128, 128, E, k)
        call = lambda: moe_route(p, logits, None, idx, wt)  # noqa: E731
        work, unit = 4.0 * T * E, "GB/s"
    for _ in range(a.warmup):
        call()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(a.iters):
        call()
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / a.iters
    status = moe_get_last_error()
    print(json.dumps({"stage": a.stage, "dims": a.dims, "us_per_call": ms * 1e3,
                      "rate": work / (ms * 1e-3) / 1e12 if unit == "TFLOP/s" else
                      work / (ms * 1e-3) / 1e9, "unit": unit, "status": status}))
    if status:
        raise SystemExit(f"device error {status}")


if __name__ == "__main__":
    main()
