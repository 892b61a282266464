"""The allocation-free routing entry point, moe_route_noalloc.

It exists for callers that cannot allocate device memory -- code running inside a
framework that owns all device memory through its own pool, or latency-critical code
that cannot afford cudaMalloc's possible device-wide synchronisation -- and therefore
cannot pass the workspace moe_route needs.  Its scratch is a fixed array inside the
library.  These checks call it through the C ABI and compare every output with
moe_route's on the same inputs, for two calls in a row (a large shape, then a small
one, so the second call runs on scratch the first one left behind).

This file is named to be collected last.
"""

import numpy as np
import pytest
import torch

import token_dispatch_expert_gb300 as tde
from gpu_util import alloc_route, cfg_c, dev, new_ws
from workloads import CONFIGS, MoEConfig, gen_logits

pytestmark = pytest.mark.gpu

KEYS = ["topk_idx", "topk_w", "counts", "kept", "offsets", "dest_row", "src_tok", "src_slot",
        "drop_mask"]


def route_both(c, logits, with_flags=True):
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    ref = alloc_route(c)
    tde.moe_route(cfg, logits, *[ref[k] for k in KEYS], ws)
    got = alloc_route(c)
    for t in got.values():
        t.fill_(-7) if t.dtype != torch.float32 else t.fill_(float("nan"))
    flags = torch.zeros(4, dtype=torch.int32, device="cuda")
    tde.moe_route_noalloc(cfg, logits, *[got[k] for k in KEYS], flags if with_flags else None)
    torch.cuda.synchronize()
    return ref, got, flags


def test_noalloc_route_matches_moe_route_twice():
    for c in (CONFIGS["capacity"], CONFIGS["qwen3"].replace(name="q_small", T=1000),
              CONFIGS["capacity"].replace(name="cap_score", drop_by_score=True)):
        logits = dev(gen_logits(c))
        ref, got, flags = route_both(c, logits)
        for k in KEYS:
            # same kernels on the same inputs: identical bits (integers exact, weights too)
            assert torch.equal(ref[k], got[k]), (c.name, k)
        assert int(flags[0]) == 0


def test_noalloc_route_reports_nan_and_rejects_oversize():
    c = MoEConfig("nan", T=64, d=64, E=16, k=4, f=64)
    lg = gen_logits(c)
    lg[5, 3] = np.nan
    ref, got, flags = route_both(c, dev(lg))
    for k in KEYS:
        if k != "topk_w":
            assert torch.equal(ref[k], got[k]), k
    assert int(flags[0]) & tde.DEVERR["NAN_LOGIT"]
    # ceil(T/32) * E * 4 bytes beyond the fixed scratch: refused, nothing enqueued
    big = MoEConfig("big", T=40000, d=64, E=256, k=8, f=64)
    out = alloc_route(big.replace(T=1))   # never touched: the call is refused up front
    with pytest.raises(tde.MoEError) as ei:
        tde.moe_route_noalloc(cfg_c(big), out["topk_w"], *[out[k] for k in KEYS])
    assert ei.value.status == 2


def test_noalloc_route_at_the_size_limit_and_without_flags():
    """Drop-by-score routing with E = 64, k = 8 needs ceil(T/32)*E*4 + (E+1)*4 + T*k*4 bytes
    (each part rounded up to 256): T = 26200 fills the 1 MiB array exactly and runs; one
    token more is refused.  Both calls here pass no flags word (dev_flags = NULL), which
    must leave the outputs unchanged."""
    c = MoEConfig("nal_edge", T=26200, d=64, E=64, k=8, f=64, cap_factor=1.0, zipf_s=1.5,
                  drop_by_score=True)
    logits = dev(gen_logits(c))
    for _ in range(2):
        ref, got, _ = route_both(c, logits, with_flags=False)
        for k in KEYS:
            assert torch.equal(ref[k], got[k]), k
        assert int((got["drop_mask"] != 0).sum()) > 0     # the capacity really cuts
    over = c.replace(T=26201)
    out = alloc_route(over)
    with pytest.raises(tde.MoEError) as ei:
        tde.moe_route_noalloc(cfg_c(over), dev(gen_logits(over)), *[out[k] for k in KEYS])
    assert ei.value.status == 2
