"""Failure detection on the GPU without a fault: a bounded device wait that nothing
satisfies gives up, flags MOE_DEVERR_TIMEOUT and returns; the host reads the status and
the context stays usable.  Inconsistent segment offsets handed to the grouped GEMM are
flagged and the launch does no work."""

import pytest
import torch

import token_dispatch_expert_gb300 as tde
from gpu_util import cfg_c, new_ws, run_route
from workloads import MoEConfig, gen_logits, gen_inputs_host
from gpu_util import dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    c = MoEConfig("fd", T=64, d=64, E=4, k=2, f=64)
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    tde.moe_selftest_wait_timeout(ws, 20_000_000)     # about 10 ms of SM clocks
    status, flags = tde.moe_status(ws)
    assert status == 5                                 # MOE_ERR_TIMEOUT
    assert flags & tde.DEVERR["TIMEOUT"]
    assert tde.moe_status(ws) == (0, 0)                # read-and-clear
    # the context is still usable: a normal call runs and reports no error
    r, ws2 = run_route(c, dev(gen_logits(c)))
    assert tde.moe_status(ws2) == (0, 0)
    assert int(r["offsets"][-1]) == c.T * c.k


def test_bad_offsets_are_flagged_and_skipped():
    c = MoEConfig("bo", T=256, d=128, E=4, k=2, f=128)
    inp = gen_inputs_host(c)
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    R = c.T * c.k
    xp = torch.zeros((R, c.d), dtype=torch.bfloat16, device="cuda")
    ab = torch.full((R, 2 * c.f), 3.0, dtype=torch.bfloat16, device="cuda")
    h = torch.full((R, c.f), 3.0, dtype=torch.bfloat16, device="cuda")
    yp = torch.full((R, c.d), 3.0, dtype=torch.bfloat16, device="cuda")
    # not monotone, and past the buffer's capacity
    offsets = torch.tensor([0, 300, 100, 400, R + 64], dtype=torch.int32, device="cuda")
    tde.moe_grouped_ffn(cfg, xp, offsets, dev(inp["W1"]), dev(inp["W2"]), ab, h, yp, ws)
    status, flags = tde.moe_status(ws)
    assert status == 4 and flags & tde.DEVERR["BAD_OFFSETS"]
    assert (yp == 3.0).all() and (h == 3.0).all()     # nothing was written
