"""GPU parity of the row movers at the full workload shapes: permute (bit-exact),
combine, combine backward with the gate backward, and the un-permute reduce (within
the bf16 tolerance), each fed the oracle's routing and synthetic rows."""

import numpy as np
import pytest
import torch

import oracle
import token_dispatch_expert_gb300 as tde
from gpu_util import assert_close, cfg_c, dev, f64, new_ws, np_i
from workloads import CONFIGS, MoEConfig, gen_bf16, gen_logits, gen_rows_bf16

pytestmark = pytest.mark.gpu

CASES = dict(CONFIGS)
CASES["tiny_cap"] = CONFIGS["tiny"].replace(name="tiny_cap", cap_factor=0.5)
CASES["odd"] = MoEConfig("odd", T=999, d=192, E=13, k=3, f=64, gate="sigmoid", route_scale=2.5,
                         cap_factor=0.8, zipf_s=1.4)


def routed(c):
    logits = gen_logits(c)
    o = oracle.route(c, logits)
    g = {k: dev(np.ascontiguousarray(v)) for k, v in o.items()
         if isinstance(v, np.ndarray) and k != "topk_w"}
    g["topk_w"] = dev(o["topk_w"].astype(np.float32))
    return logits, o, g


@pytest.mark.parametrize("name", list(CASES))
def test_permute_bit_exact(name):
    c = CASES[name]
    _, o, g = routed(c)
    x = gen_bf16(c, "x", (c.T, c.d))
    xp = torch.zeros((c.T * c.k, c.d), dtype=torch.bfloat16, device="cuda")
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    tde.moe_permute(cfg, dev(x), g["src_tok"], g["offsets"], xp, ws)
    n = int(o["offsets"][-1])
    got = np_i(xp.view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(got[:n], x[o["src_tok"][:n]])
    assert (got[n:] == 0).all()          # rows past offsets[E] are not written
    assert tde.moe_status(ws) == (0, 0)


@pytest.mark.parametrize("name", list(CASES))
def test_combine(name):
    c = CASES[name]
    _, o, g = routed(c)
    R = c.T * c.k
    yp = gen_rows_bf16("yp", R, c.d)
    ys = gen_rows_bf16("ys", c.T, c.d) if c.fs else None
    y = torch.empty((c.T, c.d), dtype=torch.bfloat16, device="cuda")
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    tde.moe_combine(cfg, dev(yp), g["dest_row"], g["topk_w"], None if ys is None else dev(ys),
                    y, ws)
    # the oracle combines with the same fp32 weights the kernel was given
    ref = oracle.combine(c, o["dest_row"], o["topk_w"].astype(np.float32).astype(np.float64),
                         yp, ys)
    assert_close("y", f64(y), ref)
    assert tde.moe_status(ws) == (0, 0)


@pytest.mark.parametrize("name", list(CASES))
def test_combine_bwd_and_gate_bwd(name):
    c = CASES[name]
    logits, o, g = routed(c)
    R = c.T * c.k
    yp = gen_rows_bf16("yp", R, c.d)
    dy = gen_bf16(c, "dy", (c.T, c.d))
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    dyp = torch.zeros((R, c.d), dtype=torch.bfloat16, device="cuda")
    dl = torch.empty((c.T, c.E), dtype=torch.float32, device="cuda")
    tde.moe_combine_bwd(cfg, dev(dy), dev(yp), dev(logits), g["topk_idx"], g["topk_w"],
                        g["dest_row"], dyp, dl, ws)
    r = dict(o)
    r["topk_w"] = o["topk_w"].astype(np.float32).astype(np.float64)
    ref_dyp, ref_dl = oracle.combine_bwd(c, logits, r, dy, yp, n_rows=R)
    n = int(o["offsets"][-1])
    assert_close("dyp", f64(dyp)[:n], ref_dyp[:n])
    assert_close("dlogits", f64(dl), ref_dl)
    # unselected experts get exactly zero
    sel = np.zeros((c.T, c.E), bool)
    np.put_along_axis(sel, o["topk_idx"], True, axis=-1)
    assert (f64(dl)[~sel] == 0).all()
    assert tde.moe_status(ws) == (0, 0)


@pytest.mark.parametrize("name", list(CASES))
def test_unpermute_reduce(name):
    c = CASES[name]
    _, o, g = routed(c)
    R = c.T * c.k
    dxp = gen_rows_bf16("dxp", R, c.d)
    dxs = gen_rows_bf16("dxs", c.T, c.d) if c.fs else None
    dx = torch.empty((c.T, c.d), dtype=torch.bfloat16, device="cuda")
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    tde.moe_unpermute_reduce(cfg, dev(dxp), g["dest_row"], None if dxs is None else dev(dxs),
                             dx, ws)
    ref = oracle.unpermute_reduce(c, o["dest_row"], dxp, dxs)
    assert_close("dx", f64(dx), ref)
    assert tde.moe_status(ws) == (0, 0)


def test_bad_indices_are_flagged_not_faulted():
    c = CASES["odd"]
    _, o, g = routed(c)
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    src = g["src_tok"].clone()
    src[5] = c.T + 7                       # out of range: skipped and flagged
    xp = torch.zeros((c.T * c.k, c.d), dtype=torch.bfloat16, device="cuda")
    tde.moe_permute(cfg, dev(gen_bf16(c, "x", (c.T, c.d))), src, g["offsets"], xp, ws)
    s, flags = tde.moe_status(ws)
    assert s == 4 and flags & tde.DEVERR["BAD_INDEX"]
    dest = g["dest_row"].clone()
    dest[3, 0] = c.T * c.k + 100           # past the buffer: treated as dropped and flagged
    y = torch.empty((c.T, c.d), dtype=torch.bfloat16, device="cuda")
    tde.moe_combine(cfg, dev(gen_rows_bf16("yp", c.T * c.k, c.d)), dest, g["topk_w"], None, y,
                    ws)
    s, flags = tde.moe_status(ws)
    assert s == 4 and flags & tde.DEVERR["BAD_INDEX"]
