"""Pins of the oracle's routing variants (the NEXT-3 row):

* a per-expert selection bias that steers the top-k choice only (DeepSeek-V3-style
  balancing bias; the gate weights stay those of the raw logits);
* negative-score dropping (X-MoE verdict page, major comment on section 5.6, which
  attributes to DeepSpeed-MoE the discarding of assignments scored below zero), read as:
  an assignment
  whose raw router logit is negative is dropped before the capacity ranking;
* capacity dropping by score: an overflowing expert keeps the assignments with the
  largest raw logit (ties: lower token) instead of the earliest tokens.

CPU only.  References: numpy lexsort on the fp32 biased key, closed forms, special cases,
and the dense masked torch formulation with autograd (tests/dense_ref.py)."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from dense_ref import dense_grads, dense_layer, keep_mask, selection
from workloads import MoEConfig, bf16_bits_to_f64, gen_inputs_host, gen_logits, gen_select_bias


def lexsort_topk(key, k):
    T, E = key.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    return np.lexsort((ids, -key.astype(np.float64)), axis=-1)[:, :k]


def test_selection_bias_steers_choice_not_weights():
    c = MoEConfig("sb", T=300, d=64, E=16, k=4, f=64, zipf_s=1.0)
    c = c.replace(select_bias=gen_select_bias(c, 2.0))
    lg = gen_logits(c)
    r = oracle.route(c, lg)
    key = (lg + np.asarray(c.select_bias, np.float32)[None, :]).astype(np.float32)
    np.testing.assert_array_equal(r["topk_idx"], lexsort_topk(key, c.k))
    # the weights: softmax of the RAW logits over the selected experts
    sl = np.take_along_axis(lg.astype(np.float64), r["topk_idx"], axis=-1)
    w = np.exp(sl - sl.max(-1, keepdims=True))
    np.testing.assert_allclose(r["topk_w"], w / w.sum(-1, keepdims=True), rtol=1e-13)
    # the bias changes the choice for some tokens (it is not a no-op)
    assert (r["topk_idx"] != lexsort_topk(lg, c.k)).any()


def test_large_bias_forces_an_expert_into_every_topk():
    c = MoEConfig("force", T=64, d=64, E=8, k=2, f=64)
    bias = [0.0] * 8
    bias[5] = 1e6
    c = c.replace(select_bias=tuple(bias))
    r = oracle.route(c, gen_logits(c))
    assert (r["topk_idx"][:, 0] == 5).all()
    assert r["counts"][5] == 64


def test_negative_score_dropping():
    c = MoEConfig("neg", T=400, d=64, E=8, k=3, f=64, drop_negative=True, cap_factor=0.9)
    lg = gen_logits(c)
    r = oracle.route(c, lg)
    sel_l = np.take_along_axis(lg, r["topk_idx"], axis=-1)
    neg = sel_l < 0
    assert neg.any()
    assert (r["drop_mask"][neg] == 1).all()                    # every negative one dropped
    assert (r["dest_row"][neg] == -1).all()
    # counts: eligible assignments only; capacity ranks among them by token order
    onehot = np.zeros((c.T, c.E), np.int64)
    np.put_along_axis(onehot, r["topk_idx"], (~neg).astype(np.int64), axis=-1)
    np.testing.assert_array_equal(r["counts"], onehot.sum(0))
    rank = np.take_along_axis(np.cumsum(onehot, 0) - 1, r["topk_idx"], axis=-1)
    exp_drop = neg | (rank >= c.capacity)
    np.testing.assert_array_equal(r["drop_mask"].astype(bool), exp_drop)
    assert int(r["offsets"][-1]) == int((~exp_drop).sum())


def test_negative_dropping_special_cases():
    c = MoEConfig("negs", T=50, d=64, E=6, k=2, f=64, drop_negative=True)
    lg = gen_logits(c)
    pos = oracle.route(c, lg + 100.0)                          # nothing negative
    base = oracle.route(c.replace(drop_negative=False), lg + 100.0)
    for key in ("topk_idx", "dest_row", "src_tok", "offsets", "drop_mask"):
        np.testing.assert_array_equal(pos[key], base[key])
    allneg = oracle.route(c, -np.abs(lg) - 1.0)                 # everything negative
    assert int(allneg["offsets"][-1]) == 0 and (allneg["drop_mask"] == 1).all()
    inp = gen_inputs_host(c)
    inp["logits"] = -np.abs(inp["logits"]) - 1.0
    assert (oracle.layer_fwd(c, inp)["y"] == 0).all()          # no expert output at all


HERE = os.path.dirname(os.path.abspath(__file__))
ROUTE_KEYS = ("topk_idx", "counts", "kept", "offsets", "dest_row", "src_tok", "src_slot",
              "drop_mask")


def test_drop_by_score_hand_worked_fixture():
    g = json.load(open(os.path.join(HERE, "golden", "route_drop_by_score_hand_worked.json")))
    for case in g["cases"]:
        c = MoEConfig("hand_score", T=case["T"], d=8, E=case["E"], k=case["k"], f=8,
                      gate=case["gate"], cap_factor=case["cap_factor"], drop_by_score=True)
        assert c.capacity == case["capacity"]
        r = oracle.route(c, np.array(case["logits"], np.float32))
        for key in ROUTE_KEYS:
            np.testing.assert_array_equal(r[key], np.array(case[key]), err_msg=key)
        assert r["drops"] == case["drops"]


def check_by_score(c, lg, r):
    """Independent restatement: per overflowing expert, the kept tokens are the `cap` best
    by numpy lexsort on (logit desc, token asc); rows of a segment in token order."""
    sel = selection(lg, c.k)
    np.testing.assert_array_equal(r["topk_idx"], sel)
    elig = (lg >= 0).astype(np.int64) if c.drop_negative else None
    _, keep = keep_mask(sel, c.E, c.capacity, elig, score=lg)
    kept_slots = np.take_along_axis(keep, sel, axis=-1).astype(bool)
    np.testing.assert_array_equal(r["drop_mask"] == 0, kept_slots)
    np.testing.assert_array_equal(r["kept"], keep.sum(0))
    for e in range(c.E):
        s, t = int(r["offsets"][e]), int(r["offsets"][e + 1])
        np.testing.assert_array_equal(r["src_tok"][s:t], np.flatnonzero(keep[:, e]))


@pytest.mark.parametrize("neg", [False, True])
def test_drop_by_score_matches_lexsort(neg):
    c = MoEConfig("bys", T=600, d=64, E=8, k=2, f=64, cap_factor=0.7, zipf_s=1.3,
                  drop_by_score=True, drop_negative=neg)
    lg = gen_logits(c)
    r = oracle.route(c, lg)
    assert r["drops"] > 0
    check_by_score(c, lg, r)
    # it is not the token-order rule on this input
    t = oracle.route(c.replace(drop_by_score=False), lg)
    assert (t["drop_mask"] != r["drop_mask"]).any()
    # kept scores dominate dropped ones inside every expert
    sl = np.take_along_axis(lg, r["topk_idx"], axis=-1)
    for e in range(c.E):
        on_e = r["topk_idx"] == e
        if neg:
            on_e &= sl >= 0
        kept = sl[on_e & (r["drop_mask"] == 0)]
        dropped = sl[on_e & (r["drop_mask"] == 1)]
        if kept.size and dropped.size:
            assert kept.min() >= dropped.max()


def test_drop_by_score_special_cases():
    c = MoEConfig("bys2", T=200, d=64, E=4, k=2, f=64, cap_factor=0.6, drop_by_score=True)
    lg = gen_logits(c)
    t_order = c.replace(drop_by_score=False)
    # no overflow (capacity above every count): identical to the token-order rule
    big = c.replace(cap_factor=None)
    a, b = oracle.route(big, lg), oracle.route(t_order.replace(cap_factor=None), lg)
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    # every token scores an expert equally (a column of equal logits): the tie rule makes
    # it the token-order rule
    lg_eq = np.tile(np.array([[3.0, 2.0, 1.0, 0.0]], np.float32), (c.T, 1))
    a, b = oracle.route(c, lg_eq), oracle.route(t_order, lg_eq)
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    # scores increasing with the token index: the LAST `cap` tokens are kept
    lg_inc = lg_eq + np.arange(c.T, dtype=np.float32)[:, None] * 1e-3
    a = oracle.route(c, lg_inc)
    cap = c.capacity
    np.testing.assert_array_equal(a["src_tok"][:cap], np.arange(c.T - cap, c.T))


VARIANTS = {
    "bias_softmax": MoEConfig("v_bias", T=48, d=64, E=6, k=2, f=64, cap_factor=0.75),
    "neg_sigmoid": MoEConfig("v_neg", T=40, d=64, E=5, k=3, f=64, gate="sigmoid",
                             route_scale=2.5, drop_negative=True, fs=64),
    "by_score": MoEConfig("v_score", T=48, d=64, E=6, k=2, f=64, cap_factor=0.6,
                          zipf_s=1.2, drop_by_score=True),
}


@pytest.mark.parametrize("name", list(VARIANTS))
def test_variants_match_dense_formulation_and_autograd(name):
    c = VARIANTS[name]
    if name == "bias_softmax":
        c = c.replace(select_bias=gen_select_bias(c, 1.5))
    inp = gen_inputs_host(c)
    f64 = {"logits": inp["logits"]}
    for n, v in inp.items():
        if n != "logits":
            f64[n] = bf16_bits_to_f64(v)
    fo = oracle.layer_fwd(c, f64, rnd=False)
    bo = oracle.layer_bwd(c, f64, fo, rnd=False)
    y_ref, g = dense_grads(c, f64)
    np.testing.assert_allclose(fo["y"], y_ref.numpy(), rtol=1e-11, atol=1e-13)
    pairs = [("dx", "x"), ("dW1", "W1"), ("dW2", "W2"), ("dlogits", "logits")]
    if c.fs:
        pairs += [("dW1s", "W1s"), ("dW2s", "W2s")]
    for ours, leaf in pairs:
        ref = g[leaf].numpy()
        np.testing.assert_allclose(bo[ours], ref, rtol=1e-9, atol=1e-11 * np.abs(ref).max(),
                                   err_msg=ours)
