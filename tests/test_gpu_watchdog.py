"""Failure detection on the GPU without a fault: a CTA whose pipeline waits can
never complete gives up after the kernels' wait limit, reports MOE_ERR_TIMEOUT
through the error word, and leaves the context usable for the next layer."""
import time

import pytest
import torch

import _gpu as G
from test_gpu_forward import SHARED_SMALL, run_forward

pytestmark = pytest.mark.gpu


def test_wait_limit_reports_timeout_and_context_survives(orc):
    m = G.lib()
    assert m.moe_get_last_error() == 0
    roles = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    m.moe_watchdog_selftest(roles)
    status = m.moe_get_last_error()
    elapsed = time.monotonic() - t0
    assert status == 5, m.load_library().moe_status_string(status)  # MOE_ERR_TIMEOUT
    assert roles.tolist() == [0, 0, 0, 0]  # every role gave up, none hung
    assert 1.5 < elapsed < 30.0, elapsed  # the 2 s limit, not an instant return
    assert m.moe_get_last_error() == 0  # reading the word cleared it

    # the same context still runs the layer correctly
    cfg = SHARED_SMALL
    inp = G.gpu_inputs(cfg)
    out = run_forward(cfg, inp)
    assert m.moe_get_last_error() == 0
    ref, _, _, _ = orc.moe_forward(cfg.oracle_problem(), G.host(inp))
    G.assert_close(G.bf16_values(G.bf16_bits(out)), ref, "forward after watchdog expiry")


def test_watchdog_uses_no_memory_of_the_caller():
    # role_status is optional; the error word is the library's own
    m = G.lib()
    m.moe_watchdog_selftest(None)
    assert m.moe_get_last_error() == 5
    torch.cuda.synchronize()
