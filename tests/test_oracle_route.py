"""Pins of the oracle's routing step against what the pages and the mathematics fix.

CPU only.  Each check is independent of the oracle's own code: numpy's lexsort for
the selection, bincount / cumulative counts for the histogram and the capacity rule,
closed forms for the gate weights, and a hand-worked fixture.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import CONFIGS, MoEConfig, gen_logits

HERE = os.path.dirname(os.path.abspath(__file__))


def brute_selection(logits, k):
    T, E = logits.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    return np.lexsort((ids, -logits.astype(np.float64)), axis=-1)[:, :k]


def check_route_invariants(cfg, logits, r):
    T, E, k = cfg.T, cfg.E, cfg.k
    cap = cfg.capacity
    idx = r["topk_idx"]
    # selection = brute force sort on (logit desc, id asc)
    np.testing.assert_array_equal(idx, brute_selection(logits, k))
    # every selected key beats every unselected key
    for t in range(min(T, 64)):
        sel = set(idx[t].tolist())
        worst = max(((-logits[t, e], e) for e in sel))     # the last selected key
        for e in range(E):
            if e not in sel:
                assert (-logits[t, e], e) > worst
    # histogram sums to T*k and equals bincount
    counts = r["counts"]
    assert counts.sum() == T * k
    np.testing.assert_array_equal(counts, np.bincount(idx.reshape(-1), minlength=E))
    # capacity: kept = min(counts, cap); drops; offsets = exclusive scan
    kept = np.minimum(counts, cap) if cap > 0 else counts
    np.testing.assert_array_equal(r["kept"], kept)
    drops = int(np.maximum(0, counts - cap).sum()) if cap > 0 else 0
    assert r["drops"] == drops
    assert int(r["offsets"][-1]) == T * k - drops
    np.testing.assert_array_equal(r["offsets"], np.concatenate([[0], np.cumsum(kept)]))
    # dropped slots are exactly the (cap+1)-th and later tokens of an expert, by token order
    onehot = np.zeros((T, E), np.int64)
    np.put_along_axis(onehot, idx, 1, axis=-1)
    rank_te = np.cumsum(onehot, axis=0) - 1
    rank = np.take_along_axis(rank_te, idx, axis=-1)
    exp_drop = (rank >= cap) if cap > 0 else np.zeros_like(rank, bool)
    np.testing.assert_array_equal(r["drop_mask"].astype(bool), exp_drop)
    # dest_row: offsets[e] + rank for kept, -1 for dropped
    exp_dest = np.where(exp_drop, -1, r["offsets"][idx] + rank)
    np.testing.assert_array_equal(r["dest_row"], exp_dest)
    # inverse maps
    nk = int(r["offsets"][-1])
    tt, jj = np.nonzero(~exp_drop)
    p = exp_dest[tt, jj]
    assert sorted(p.tolist()) == list(range(nk))
    np.testing.assert_array_equal(r["src_tok"][p], tt)
    np.testing.assert_array_equal(r["src_slot"][p], tt * k + jj)
    assert (r["src_tok"][nk:] == -1).all() and (r["src_slot"][nk:] == -1).all()
    # within an expert, dest_row increases strictly with t
    for e in range(E):
        s, t_ = r["offsets"][e], r["offsets"][e + 1]
        toks = r["src_tok"][s:t_]
        assert (np.diff(toks) > 0).all()
        assert (idx.reshape(-1)[r["src_slot"][s:t_]] == e).all()


def check_weights(cfg, logits, r):
    T, k = cfg.T, cfg.k
    w = r["topk_w"]
    sel_l = np.take_along_axis(logits.astype(np.float64), r["topk_idx"], axis=-1)
    if cfg.gate == "softmax":
        np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=4 * 2.0 ** -52)
        # softmax over all E, renormalised over the selected (torch routine)
        p = torch.softmax(torch.tensor(logits, dtype=torch.float64), -1).numpy()
        ps = np.take_along_axis(p, r["topk_idx"], axis=-1)
        np.testing.assert_allclose(w, ps / ps.sum(-1, keepdims=True), rtol=1e-13, atol=1e-300)
    else:
        np.testing.assert_allclose(w.sum(-1), cfg.route_scale, rtol=4 * 2.0 ** -52)
        s = 1.0 / (1.0 + np.exp(-sel_l))
        np.testing.assert_allclose(w, cfg.route_scale * s / s.sum(-1, keepdims=True), rtol=1e-13)


@pytest.mark.parametrize("name", ["tiny", "qwen3", "dsv3", "capacity", "mixtral"])
def test_route_full_configs(name):
    cfg = CONFIGS[name]
    logits = gen_logits(cfg)
    r = oracle.route(cfg, logits)
    check_route_invariants(cfg, logits, r)
    check_weights(cfg, logits, r)
    assert r["nan_logits"] == 0


def test_capacity_config_values():
    cfg = CONFIGS["capacity"]
    assert cfg.capacity == 1920          # floor(1.25 * 16384 * 6 / 64)
    r = oracle.route(cfg, gen_logits(cfg))
    assert r["drops"] > 0                # the skewed load overflows some experts
    assert (r["kept"] <= 1920).all() and (r["kept"] == 1920).any()


def test_hand_worked_fixture():
    g = json.load(open(os.path.join(HERE, "golden", "route_hand_worked.json")))
    cfg = MoEConfig("hand", T=g["T"], d=8, E=g["E"], k=g["k"], f=8, gate=g["gate"],
                    cap_factor=None)
    logits = np.array(g["logits"], np.float32)
    # capacity 2 expressed as a factor: floor(c * 5 * 2 / 4) = 2 for c = 0.8
    cfg = cfg.replace(cap_factor=0.8)
    assert cfg.capacity == g["capacity"]
    r = oracle.route(cfg, logits)
    for key in ("topk_idx", "counts", "kept", "offsets", "dest_row", "src_tok", "src_slot",
                "drop_mask"):
        np.testing.assert_array_equal(r[key], np.array(g[key]), err_msg=key)
    assert r["drops"] == g["drops"]
    np.testing.assert_allclose(r["topk_w"], np.array(g["topk_w"]), rtol=1e-15)


def test_all_equal_logits_pick_lowest_ids():
    cfg = MoEConfig("eq", T=17, d=8, E=9, k=3, f=8)
    logits = np.full((17, 9), 0.25, np.float32)
    r = oracle.route(cfg, logits)
    assert (r["topk_idx"] == np.arange(3)).all()
    np.testing.assert_allclose(r["topk_w"], 1.0 / 3.0, rtol=1e-15)


def test_signed_zero_ties_and_nan():
    cfg = MoEConfig("z", T=2, d=8, E=4, k=2, f=8)
    logits = np.array([[-0.0, 0.0, -1.0, -2.0],
                       [np.nan, -np.inf, 1.0, np.nan]], np.float32)
    r = oracle.route(cfg, logits)
    assert r["topk_idx"][0].tolist() == [0, 1]          # +0 == -0, lower id first
    assert r["topk_idx"][1].tolist() == [2, 1]          # NaN ranks below -inf
    assert r["nan_logits"] == 2


def test_k_equals_E_routes_every_expert():
    cfg = MoEConfig("kE", T=33, d=8, E=5, k=5, f=8)
    logits = gen_logits(cfg)
    r = oracle.route(cfg, logits)
    assert (np.sort(r["topk_idx"], -1) == np.arange(5)).all()
    assert (r["counts"] == 33).all()
    np.testing.assert_allclose(r["topk_w"].sum(-1), 1.0, atol=1e-15)


def test_single_expert_identity_permutation():
    cfg = MoEConfig("e1", T=40, d=8, E=1, k=1, f=8)
    r = oracle.route(cfg, gen_logits(cfg))
    np.testing.assert_array_equal(r["src_tok"], np.arange(40))
    np.testing.assert_array_equal(r["dest_row"].reshape(-1), np.arange(40))
    assert (r["topk_w"] == 1.0).all()                    # k = 1 softmax gives w = 1


def test_two_expert_softmax_closed_form():
    cfg = MoEConfig("two", T=64, d=8, E=2, k=2, f=8)
    logits = gen_logits(cfg)
    r = oracle.route(cfg, logits)
    for t in range(64):
        a, b = r["topk_idx"][t]
        expect = 1.0 / (1.0 + math.exp(float(logits[t, b]) - float(logits[t, a])))
        assert abs(r["topk_w"][t, 0] - expect) < 1e-15


def test_sigmoid_gate_closed_form():
    cfg = MoEConfig("sg", T=3, d=8, E=4, k=2, f=8, gate="sigmoid", route_scale=2.5)
    # sigma(ln 3) = 3/4, sigma(0) = 1/2, sigma(-ln 3) = 1/4
    l3 = math.log(3.0)
    logits = np.array([[l3, 0.0, -l3, -5.0],
                       [0.0, -l3, -5.0, l3],
                       [-l3, -l3, -l3, -l3]], np.float32)
    r = oracle.route(cfg, logits)
    s3 = 1.0 / (1.0 + math.exp(-float(np.float32(l3))))
    assert r["topk_idx"][0].tolist() == [0, 1]
    np.testing.assert_allclose(r["topk_w"][0], [2.5 * s3 / (s3 + 0.5), 2.5 * 0.5 / (s3 + 0.5)],
                               rtol=1e-15)
    assert r["topk_idx"][1].tolist() == [3, 0]
    assert r["topk_idx"][2].tolist() == [0, 1]
    np.testing.assert_allclose(r["topk_w"][2], [1.25, 1.25], rtol=1e-15)


def test_capacity_small_variant():
    # tiny layer with c = 0.5: cap = floor(0.5 * 256 * 2 / 8) = 32
    cfg = CONFIGS["tiny"].replace(name="tiny_cap", cap_factor=0.5)
    assert cfg.capacity == 32
    logits = gen_logits(cfg)
    r = oracle.route(cfg, logits)
    check_route_invariants(cfg, logits, r)
    assert r["drops"] > 0
