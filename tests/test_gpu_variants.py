"""GPU parity of the NEXT rows built so far:

* routing variants -- selection-only bias, negative-score dropping and capacity dropping
  by score: bit-exact routing against the oracle, and the whole layer (fwd + bwd) within
  tolerance;
* selective rematerialisation (recompute = 1): ctx keeps neither ab nor h, the backward
  recomputes FC1; every output is compared with the oracle's layer and must also be
  bit-identical to the saving path."""

import numpy as np
import pytest
import torch

import oracle
import token_dispatch_expert_gb300 as tde
from gpu_util import assert_close, cfg_c, dev, f64, np_i, run_route
from workloads import CONFIGS, MoEConfig, gen_inputs_host, gen_logits, gen_select_bias

pytestmark = pytest.mark.gpu

ROUTE_KEYS = ["topk_idx", "counts", "kept", "offsets", "dest_row", "src_tok", "src_slot",
              "drop_mask"]


def with_bias(c, scale=1.5):
    return c.replace(select_bias=gen_select_bias(c, scale))


ROUTE_CASES = {
    "bias_qwen3": with_bias(CONFIGS["qwen3"]),
    "bias_dsv3": with_bias(CONFIGS["dsv3"], 0.5),
    "neg_capacity": CONFIGS["capacity"].replace(name="neg_capacity", drop_negative=True),
    "bias_neg_ragged": with_bias(MoEConfig("bnr", T=999, d=64, E=37, k=5, f=64, cap_factor=0.8,
                                           zipf_s=1.3, drop_negative=True)),
    # full-size capacity workload: 1920 per expert, Zipf-skewed, several experts overflow
    "score_capacity": CONFIGS["capacity"].replace(name="score_capacity", drop_by_score=True),
    "score_neg_bias": with_bias(MoEConfig("snb", T=3001, d=64, E=24, k=4, f=64,
                                          cap_factor=0.6, zipf_s=1.4, drop_negative=True,
                                          drop_by_score=True)),
    "score_many_experts": MoEConfig("sme", T=4096, d=64, E=256, k=8, f=64, cap_factor=0.5,
                                    zipf_s=1.2, drop_by_score=True),
}


def quantised_logits(c, step):
    """Logits on a coarse grid: many equal scores at every capacity cut."""
    lg = gen_logits(c)
    return (np.round(lg / step) * step).astype(np.float32)


@pytest.mark.parametrize("step", [0.25, 1.0])
def test_drop_by_score_ties_bit_exact(step):
    c = MoEConfig("ties", T=5000, d=64, E=16, k=3, f=64, cap_factor=0.5, zipf_s=1.1,
                  drop_by_score=True)
    logits = quantised_logits(c, step)
    r, ws = run_route(c, dev(logits))
    o = oracle.route(c, logits)
    assert o["drops"] > 0
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(np_i(r[key]), o[key], err_msg=key)
    assert tde.moe_status(ws) == (0, 0)


@pytest.mark.parametrize("name", list(ROUTE_CASES))
def test_variant_routing_bit_exact(name):
    c = ROUTE_CASES[name]
    logits = gen_logits(c)
    r, ws = run_route(c, dev(logits))
    o = oracle.route(c, logits)
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(np_i(r[key]), o[key], err_msg=key)
    np.testing.assert_allclose(np_i(r["topk_w"]).astype(np.float64), o["topk_w"], rtol=2.0 ** -20)
    assert tde.moe_status(ws) == (0, 0)


LAYER_CASES = {
    "bias_mid": with_bias(MoEConfig("bm", T=1024, d=512, E=8, k=2, f=512, zipf_s=1.1)),
    "neg_sig_shared": MoEConfig("nss", T=768, d=384, E=16, k=4, f=256, fs=256, gate="sigmoid",
                                route_scale=2.5, cap_factor=1.0, zipf_s=1.2, drop_negative=True),
    "score_capped": MoEConfig("scc", T=1024, d=256, E=8, k=2, f=320, cap_factor=0.8,
                              zipf_s=1.3, drop_by_score=True),
}


def run_layer(c, g):
    layer = tde.MoELayer(cfg_c(c))
    y = layer.forward(g["logits"], g["x"], g["W1"], g["W2"], g.get("W1s"), g.get("W2s"))
    gr = layer.backward(g["logits"], g["x"], g["dy"], g["W1"], g["W2"], g.get("W1s"), g.get("W2s"))
    torch.cuda.synchronize()
    return layer, y, gr


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_variant_layer_against_oracle(name):
    c = LAYER_CASES[name]
    inp = gen_inputs_host(c)
    layer, y, gr = run_layer(c, {k: dev(v) for k, v in inp.items()})
    assert layer.status() == (0, 0)
    fo = oracle.layer_fwd(c, inp)
    bo = oracle.layer_bwd(c, inp, fo)
    v = layer.views()
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(np_i(v[key]), fo["route"][key], err_msg=key)
    assert_close("y", f64(y), fo["y"])
    assert_close("dx", f64(gr["dx"]), bo["dx"])
    assert_close("dlogits", f64(gr["dlogits"]), bo["dlogits"])
    for e in range(c.E):
        if fo["route"]["kept"][e] == 0:
            assert (f64(gr["dW1"][e]) == 0).all()
            continue
        assert_close(f"dW1[{e}]", f64(gr["dW1"][e]), bo["dW1"][e])
        assert_close(f"dW2[{e}]", f64(gr["dW2"][e]), bo["dW2"][e])


@pytest.mark.parametrize("base", ["mid", "shared"])
def test_recompute_against_oracle(base):
    c = (MoEConfig("rc", T=1024, d=512, E=8, k=2, f=512, zipf_s=1.1, cap_factor=1.2)
         if base == "mid" else
         MoEConfig("rcs", T=768, d=384, E=16, k=4, f=256, fs=256, gate="sigmoid",
                   route_scale=2.5, zipf_s=1.2))
    inp = gen_inputs_host(c)
    g = {k: dev(v) for k, v in inp.items()}
    l0, y0, g0 = run_layer(c, g)
    l1, y1, g1 = run_layer(c.replace(recompute=True), g)
    assert l1.status() == (0, 0)
    # the recomputing layer against the oracle (recomputation changes no arithmetic, so the
    # oracle is the plain layer's)
    fo = oracle.layer_fwd(c, inp)
    bo = oracle.layer_bwd(c, inp, fo)
    v = l1.views()
    for key in ("topk_idx", "offsets", "dest_row", "src_tok"):
        np.testing.assert_array_equal(np_i(v[key]), fo["route"][key], err_msg=key)
    assert_close("recompute y", f64(y1), fo["y"])
    assert_close("recompute dx", f64(g1["dx"]), bo["dx"])
    assert_close("recompute dlogits", f64(g1["dlogits"]), bo["dlogits"])
    for e in range(c.E):
        if fo["route"]["kept"][e] == 0:
            assert (f64(g1["dW1"][e]) == 0).all() and (f64(g1["dW2"][e]) == 0).all()
            continue
        assert_close(f"recompute dW1[{e}]", f64(g1["dW1"][e]), bo["dW1"][e])
        assert_close(f"recompute dW2[{e}]", f64(g1["dW2"][e]), bo["dW2"][e])
    if c.fs:
        assert_close("recompute dW1s", f64(g1["dW1s"]), bo["dW1s"])
        assert_close("recompute dW2s", f64(g1["dW2s"]), bo["dW2s"])
    # and bit for bit the saving path's results
    assert torch.equal(y0, y1)
    for k in g0:
        assert torch.equal(g0[k], g1[k]), k
    # ctx holds neither ab nor h: smaller by their bytes
    R = c.T * c.k
    saved = R * 3 * c.f * 2 + (c.T * 3 * c.fs * 2 if c.fs else 0)
    assert l0.ctx.numel() - l1.ctx.numel() >= saved


ALL_DROPPED = {
    "plain": MoEConfig("alldrop", T=300, d=128, E=8, k=2, f=128, drop_negative=True),
    "sig_shared": MoEConfig("alldrop_s", T=300, d=128, E=8, k=3, f=128, fs=192,
                            gate="sigmoid", route_scale=2.5, drop_negative=True),
}


def all_negative(inp):
    inp = dict(inp)
    inp["logits"] = -(np.abs(inp["logits"]) + np.float32(0.5))
    return inp


@pytest.mark.parametrize("name", list(ALL_DROPPED))
def test_every_assignment_dropped(name):
    """Every router logit negative with negative-score dropping: no row is kept, so the
    grouped GEMMs run with zero rows.  y and dx are the shared expert's alone (zero without
    one), every routed weight gradient and dlogits are zero, and the status stays clean."""
    c = ALL_DROPPED[name]
    inp = all_negative(gen_inputs_host(c))
    layer, y, gr = run_layer(c, {k: dev(v) for k, v in inp.items()})
    assert layer.status() == (0, 0)
    fo = oracle.layer_fwd(c, inp)
    bo = oracle.layer_bwd(c, inp, fo)
    assert fo["route"]["offsets"][-1] == 0
    v = layer.views()
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(np_i(v[key]), fo["route"][key], err_msg=key)
    assert (f64(gr["dW1"]) == 0).all() and (f64(gr["dW2"]) == 0).all()
    assert (f64(gr["dlogits"]) == 0).all()
    if c.fs:
        assert_close("y", f64(y), fo["y"])
        assert_close("dx", f64(gr["dx"]), bo["dx"])
        assert_close("dW1s", f64(gr["dW1s"]), bo["dW1s"])
        assert_close("dW2s", f64(gr["dW2s"]), bo["dW2s"])
    else:
        assert (f64(y) == 0).all() and (f64(gr["dx"]) == 0).all()


@pytest.mark.parametrize("level", [1, 2])
def test_every_assignment_dropped_mx(level):
    """The same degenerate routing through the MXFP8 layer calls (level 2: the MXFP8
    weight-gradient path with zero rows per expert)."""
    c = ALL_DROPPED["plain"]
    inp = all_negative(gen_inputs_host(c))
    g = {k: dev(v) for k, v in inp.items()}
    cfg = tde.make_config(c.T, c.d, c.E, c.k, c.f, drop_negative=True, mxfp8=level)
    layer = tde.MoELayer(cfg)
    wq = layer.quantize_weights(g["W1"], g["W2"])
    y = layer.forward_mx(g["logits"], g["x"], wq)
    gr = layer.backward_mx(g["logits"], g["x"], g["dy"], wq)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    assert int(layer.views()["offsets"][-1]) == 0
    for name, t in [("y", y), ("dx", gr["dx"]), ("dW1", gr["dW1"]), ("dW2", gr["dW2"]),
                    ("dlogits", gr["dlogits"])]:
        assert (f64(t) == 0).all(), name
