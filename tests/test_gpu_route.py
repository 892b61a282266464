"""GPU parity of the routing step (moe_route) against the oracle: bit-exact for every
integer output (top-k ids, counts, kept, offsets, dest_row, src_tok, src_slot, drop
mask) on all five workload shapes and on the degenerate cases; gate weights within
2^-20 relative; two runs bit-identical."""

import numpy as np
import pytest
import torch

import oracle
import token_dispatch_expert_gb300 as tde
from gpu_util import cfg_c, dev, np_i, run_route
from workloads import CONFIGS, MoEConfig, gen_logits

pytestmark = pytest.mark.gpu

INT_KEYS = ["topk_idx", "counts", "kept", "offsets", "dest_row", "src_tok", "src_slot",
            "drop_mask"]


def compare(c, logits, r):
    o = oracle.route(c, logits)
    for key in INT_KEYS:
        np.testing.assert_array_equal(np_i(r[key]), o[key], err_msg=key)
    w = np_i(r["topk_w"]).astype(np.float64)
    np.testing.assert_allclose(w, o["topk_w"], rtol=2.0 ** -20, atol=1e-30)
    return o


EDGE = {
    "tiny_cap": CONFIGS["tiny"].replace(name="tiny_cap", cap_factor=0.5),
    "ragged_T": MoEConfig("ragged_T", T=1000, d=64, E=37, k=5, f=64, zipf_s=1.3),
    "e1k1": MoEConfig("e1k1", T=333, d=64, E=1, k=1, f=64),
    "kE": MoEConfig("kE", T=130, d=64, E=8, k=8, f=64),
    "E256k8_cap": MoEConfig("E256k8_cap", T=777, d=64, E=256, k=8, f=64, cap_factor=0.9,
                            zipf_s=1.5),
    "sig": MoEConfig("sig", T=513, d=64, E=64, k=6, f=64, gate="sigmoid", route_scale=2.5,
                     zipf_s=1.2),
    "T1": MoEConfig("T1", T=1, d=64, E=3, k=2, f=64),
}


@pytest.mark.parametrize("name", list(CONFIGS) + list(EDGE))
def test_route_parity(name):
    c = CONFIGS.get(name) or EDGE[name]
    logits = gen_logits(c)
    r, ws = run_route(c, dev(logits))
    o = compare(c, logits, r)
    s, flags = tde.moe_status(ws)
    assert s == 0 and flags == 0
    if c.capacity:
        assert int(np_i(r["drop_mask"]).sum()) == o["drops"]


def test_route_deterministic():
    c = CONFIGS["capacity"]
    logits = dev(gen_logits(c))
    r1, _ = run_route(c, logits)
    r2, _ = run_route(c, logits)
    for key in INT_KEYS + ["topk_w"]:
        assert torch.equal(r1[key], r2[key]), key


def test_route_ties_signed_zero_and_all_equal():
    c = MoEConfig("ties", T=70, d=64, E=40, k=4, f=64)
    logits = np.full((70, 40), 0.5, np.float32)
    logits[1] = 0.0
    logits[1, ::2] = -0.0
    logits[2, 5:9] = 3.0          # four-way tie at the top
    logits[3] = np.float32(1e-30) * np.arange(40, dtype=np.float32)
    r, _ = run_route(c, dev(logits))
    compare(c, logits, r)
    assert (np_i(r["topk_idx"])[0] == np.arange(4)).all()


def test_route_nan_logits_flagged():
    c = MoEConfig("nan", T=64, d=64, E=16, k=4, f=64)
    logits = gen_logits(c)
    logits[3, 2] = np.nan
    logits[10, :] = np.nan        # a token with only NaN logits still selects k experts
    r, ws = run_route(c, dev(logits))
    o = oracle.route(c, logits)
    for key in INT_KEYS:
        np.testing.assert_array_equal(np_i(r[key]), o[key], err_msg=key)
    s, flags = tde.moe_status(ws)
    assert s == 4                 # MOE_ERR_DEVICE_FLAG
    assert flags & tde.DEVERR["NAN_LOGIT"]
    # the flag is cleared by the read
    assert tde.moe_status(ws) == (0, 0)
