"""GPU check of the grouped GEMMs' clock trace (moe_gemm_clock_trace / moe_gemm_clock_read):
while on, every bf16 and MXFP8 grouped-GEMM launch adds one loop per MMA-issuing CTA with
a clock between idle and the maximum; turning it on zeroes the sums, turning it off keeps
them, and launches while off add nothing.  The traced layer's outputs are the untraced
layer's, bit for bit."""

import pytest
import torch

import token_dispatch_expert_gb300 as tde
from gpu_util import dev
from workloads import MoEConfig, gen_inputs_host

pytestmark = pytest.mark.gpu

C = MoEConfig("trace", T=1024, d=512, E=8, k=2, f=512, zipf_s=1.1)


def run(layer, g, mx=None):
    if mx is not None:
        y = layer.forward_mx(g["logits"], g["x"], mx)
        gr = layer.backward_mx(g["logits"], g["x"], g["dy"], mx)
    else:
        y = layer.forward(g["logits"], g["x"], g["W1"], g["W2"])
        gr = layer.backward(g["logits"], g["x"], g["dy"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    return y, gr


@pytest.mark.parametrize("mxfp8", [0, 2])
def test_clock_trace_counts_loops_and_leaves_outputs_alone(mxfp8):
    g = {k: dev(v) for k, v in gen_inputs_host(C).items()}
    layer = tde.MoELayer(tde.make_config(C.T, C.d, C.E, C.k, C.f, mxfp8=mxfp8))
    wq = layer.quantize_weights(g["W1"], g["W2"]) if mxfp8 else None
    torch.cuda.synchronize()
    tde.moe_gemm_clock_trace(False)
    y0, gr0 = run(layer, g, wq)

    tde.moe_gemm_clock_trace(True)
    assert tde.moe_gemm_clock_read() == (0, 0, 0)          # zeroed when turned on
    y1, gr1 = run(layer, g, wq)
    tde.moe_gemm_clock_trace(False)
    cycles, ns, loops = tde.moe_gemm_clock_read()
    assert loops > 0 and ns > 0
    mhz = cycles / ns * 1e3
    assert 200.0 < mhz < 2600.0, mhz
    assert layer.status() == (0, 0)
    assert torch.equal(y0, y1)
    for k in gr0:
        assert torch.equal(gr0[k], gr1[k]), k

    run(layer, g, wq)                                       # off: nothing added
    assert tde.moe_gemm_clock_read() == (cycles, ns, loops)
