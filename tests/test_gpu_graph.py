"""The whole layer captured in a CUDA graph and replayed: moe_forward queues
its kernels on the caller's stream with no host round trip and no allocation,
so a serving loop can capture one call and replay it with new inputs written
into the same buffers.  Checked against eager calls on the same inputs."""
import pytest
import torch

import _gpu as G
import moe_inputs as mi
from test_gpu_forward import SHARED_SMALL

pytestmark = pytest.mark.gpu

DECODE_SMALL = mi.MoEConfig("decode_small", T=64, H=1024, I=512, E=32, k=8, I_s=512)


def _args(inp, out, ws, p):
    return (p, inp["x"], inp["router_w"], inp["router_bias"], inp["w13"], inp["w13_scale"],
            inp["w2"], inp["w2_scale"], inp["sw13"], inp["sw13_scale"], inp["sw2"],
            inp["sw2_scale"], inp["wd"], inp["wu"], inp["gamma"], out, ws)


@pytest.mark.parametrize("cfg", [SHARED_SMALL, DECODE_SMALL], ids=lambda c: c.name)
def test_forward_replays_in_a_cuda_graph(cfg):
    m = G.lib()
    inp = G.gpu_inputs(cfg)
    p = G.problem(cfg)
    ws = G.workspace(p)
    eager = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    m.moe_forward(*_args(inp, eager, ws, p))  # first call: per-device set-up
    torch.cuda.synchronize()
    out = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.moe_forward(*_args(inp, out, ws, p))
    g.replay()
    torch.cuda.synchronize()
    assert m.moe_get_last_error() == 0
    assert torch.equal(out, eager)
    # new tokens written into the captured input buffer
    x2 = torch.randn(cfg.T, cfg.H, device="cuda",
                     generator=torch.Generator(device="cuda").manual_seed(7)).to(torch.bfloat16)
    inp["x"].copy_(x2)
    g.replay()
    m.moe_forward(*_args(inp, eager, ws, p))
    torch.cuda.synchronize()
    assert m.moe_get_last_error() == 0
    assert torch.equal(out, eager)
