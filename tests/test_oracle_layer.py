"""Pins of the oracle's bf16 rounding, expert FFN, combine and whole layer.

CPU only.  The comparisons are against: torch's own fp32->bf16 conversion (a library
routine), hand-derived rounding cases, a dense "every expert on every token, then
mask" formulation in torch float64 (tests/dense_ref.py, no code shared with the
oracle), the textbook dense SwiGLU MLP (E = 1, k = 1), identical experts, identity
experts, and the permute round trip.
"""

import numpy as np
import pytest
import torch

import oracle
from dense_ref import as_t, dense_layer, swiglu
from workloads import CONFIGS, MoEConfig, bf16_bits_to_f64, gen_inputs_host


def rel_l2(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ------------------------------------------------------------------ bf16 rounding
def test_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
        np.array([1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-40, 1e-45, 2.0 ** -126, 65504.0],
                 np.float32),
    ]).astype(np.float32)
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_hand_cases():
    u = 2.0 ** -7                       # bf16 spacing in [1, 2)
    cases = {
        1.0 + u / 2: 1.0,               # tie -> even (1.0)
        1.0 + 3 * u / 2: 1.0 + 2 * u,   # tie -> even (mantissa ...10)
        1.0 + u / 2 + 2.0 ** -40: 1.0 + u,   # just above the tie rounds up (no double rounding)
        -(2.0 + 2 * u / 2): -2.0,       # spacing 2^-6 in [2, 4): tie -> even
        2.0 ** -133 * 1.5: 2.0 ** -132,  # subnormal tie -> even
        2.0 ** 128 * (1 - 2.0 ** -9): np.inf,   # past the largest finite bf16
        (2.0 - u) * 2.0 ** 127: (2.0 - u) * 2.0 ** 127,   # largest finite value is exact
    }
    for x, want in cases.items():
        assert oracle.bf16(np.array([x]))[0] == want, x


# ------------------------------------------------------------------ dense pins
SMALL = {
    "tiny": CONFIGS["tiny"],
    "tiny_cap": CONFIGS["tiny"].replace(name="tiny_cap", cap_factor=0.5),
    "tiny_sig_shared": MoEConfig("tiny_sig_shared", T=96, d=64, E=6, k=3, f=128, fs=64,
                                 gate="sigmoid", route_scale=2.5, cap_factor=0.75,
                                 zipf_s=1.2),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_fwd_equals_dense_masked_formulation(name):
    cfg = SMALL[name]
    inp = gen_inputs_host(cfg)
    o = oracle.layer_fwd(cfg, inp, rnd=False)
    y_ref, _ = dense_layer(cfg, inp, rnd=False)
    np.testing.assert_allclose(o["y"], y_ref.numpy(), rtol=1e-11, atol=1e-13)
    # with the bf16 rounding points on both sides the two agree to within one bf16 ulp
    # almost everywhere (the dense side sums experts in another order)
    o_r = oracle.layer_fwd(cfg, inp, rnd=True)
    y_r, _ = dense_layer(cfg, inp, rnd=True)
    y_r = y_r.numpy()
    ulp = np.abs(y_r) * 2.0 ** -7 + 1e-30
    assert (np.abs(o_r["y"] - y_r) <= ulp).mean() > 0.9995
    assert rel_l2(o_r["y"], y_r) < 2e-3
    # the rounded oracle stays within bf16 noise of the exact layer
    assert rel_l2(o_r["y"], o["y"]) < 1e-2


def test_single_expert_is_dense_swiglu_mlp():
    cfg = MoEConfig("e1k1", T=50, d=64, E=1, k=1, f=96)
    inp = gen_inputs_host(cfg)
    o = oracle.layer_fwd(cfg, inp, rnd=False)
    x = bf16_bits_to_f64(inp["x"]); W1 = bf16_bits_to_f64(inp["W1"][0])
    W2 = bf16_bits_to_f64(inp["W2"][0])
    a = x @ W1[:96].T; b = x @ W1[96:].T
    y = ((a / (1.0 + np.exp(-a))) * b) @ W2.T          # textbook SwiGLU MLP, w = 1
    np.testing.assert_allclose(o["y"], y, rtol=1e-12, atol=1e-14)


def test_identical_experts_give_the_plain_ffn():
    cfg = MoEConfig("same", T=64, d=64, E=5, k=2, f=64)
    inp = gen_inputs_host(cfg)
    inp["W1"] = np.repeat(inp["W1"][:1], 5, axis=0)
    inp["W2"] = np.repeat(inp["W2"][:1], 5, axis=0)
    o = oracle.layer_fwd(cfg, inp, rnd=False)
    y = swiglu(as_t(inp["x"]), as_t(inp["W1"][0]), as_t(inp["W2"][0])).numpy()
    np.testing.assert_allclose(o["y"], y, rtol=1e-12, atol=1e-14)   # sum of weights is 1


def test_identity_experts_round_trip():
    # combine(permute(x)) with the FFN skipped returns x (bf16 values unchanged)
    cfg = CONFIGS["tiny"]
    inp = gen_inputs_host(cfg)
    r = oracle.route(cfg, inp["logits"])
    x = bf16_bits_to_f64(inp["x"])
    xp = x[r["src_tok"][: r["offsets"][-1]]]
    y = oracle.combine(cfg, r["dest_row"], r["topk_w"], xp, rnd=True)
    np.testing.assert_array_equal(y, x)


def test_permute_round_trip_through_dest_row():
    cfg = CONFIGS["tiny"].replace(name="tiny_cap", cap_factor=0.5)
    inp = gen_inputs_host(cfg)
    o = oracle.layer_fwd(cfg, inp, rnd=True)
    r = o["route"]
    x = bf16_bits_to_f64(inp["x"])
    t, j = np.nonzero(r["dest_row"] >= 0)
    np.testing.assert_array_equal(o["xp"][r["dest_row"][t, j]], x[t])


def test_fully_dropped_token_gives_zero():
    cfg = MoEConfig("drop", T=64, d=64, E=4, k=1, f=64, cap_factor=0.25)   # cap = 4
    inp = gen_inputs_host(cfg)
    o = oracle.layer_fwd(cfg, inp, rnd=True)
    dropped = o["route"]["drop_mask"][:, 0] == 1
    assert dropped.any()
    assert (o["y"][dropped] == 0).all()


def test_sampled_layer_matches_full_layer():
    cfg = SMALL["tiny_sig_shared"]
    inp = gen_inputs_host(cfg)
    f = oracle.layer_fwd(cfg, inp, rnd=True)
    b = oracle.layer_bwd(cfg, inp, f, rnd=True)
    toks = [0, 5, 17, 95, 42]
    experts = [0, 3, 5]
    wcols = np.array([0, 7, 63])          # valid for f = 128 and fs = 64
    wrows = np.array([1, 2, 63])
    s = oracle.layer_sampled(cfg, oracle.HostSource(inp), toks, experts, wcols, wrows, rnd=True)
    tk = np.array(sorted(toks))
    np.testing.assert_array_equal(s["y"], f["y"][tk])
    np.testing.assert_array_equal(s["dx"], b["dx"][tk])
    np.testing.assert_allclose(s["dlogits"], b["dlogits"][tk], rtol=1e-12, atol=1e-14)
    one_ulp = 2.0 ** -7      # the two sum the rows in another order before rounding
    for e in experts:
        np.testing.assert_allclose(s["dW1"][e][0], b["dW1"][e][np.ix_(wcols, wrows)], rtol=one_ulp)
        np.testing.assert_allclose(s["dW1"][e][1], b["dW1"][e][np.ix_(wcols + cfg.f, wrows)],
                                   rtol=one_ulp)
        np.testing.assert_allclose(s["dW2"][e], b["dW2"][e][np.ix_(wrows, wcols)], rtol=one_ulp)
    np.testing.assert_allclose(s["dW1s"][0], b["dW1s"][np.ix_(wcols, wrows)], rtol=one_ulp)
    np.testing.assert_allclose(s["dW1s"][1], b["dW1s"][np.ix_(wcols + cfg.fs, wrows)],
                               rtol=one_ulp)
    np.testing.assert_allclose(s["dW2s"], b["dW2s"][np.ix_(wrows, wcols)], rtol=one_ulp)


# ------------------------------------------------- dispatch of dy fused into the FC2 dgrad
def _dispatch_case(seed=3, n=40, d=128, f=192):
    rng = np.random.default_rng(seed)
    bf = lambda a: oracle.bf16(np.asarray(a, np.float64))
    dy = bf(rng.standard_normal((n, d)))
    ab = bf(rng.standard_normal((n, 2 * f)))
    W1 = bf(rng.standard_normal((2 * f, d)) * 0.05)
    W2 = bf(rng.standard_normal((d, f)) * 0.05)
    w = rng.uniform(0.05, 1.0, n).astype(np.float32).astype(np.float64)
    return dy, w, ab, W1, W2


def test_dispatch_bwd_with_exact_weights_equals_the_unfused_rows():
    """With power-of-two gate weights w * dy is exact in bf16, so the fused path (dh from
    w * dy taken exactly) and the unfused one (dh from the stored bf16(w * dy)) agree bit
    for bit."""
    dy, _, ab, W1, W2 = _dispatch_case()
    w = 2.0 ** -(np.arange(dy.shape[0]) % 4)
    fused = oracle.ffn_bwd_rows_dispatch(dy, w, ab, W1, W2)
    plain = oracle.ffn_bwd_rows(oracle.bf16(dy * w[:, None]), ab, W1, W2)
    for a, b in zip(fused, plain):
        np.testing.assert_array_equal(a, b)
    # doubling every weight doubles every output exactly (rounding commutes with 2x)
    fused2 = oracle.ffn_bwd_rows_dispatch(dy, 2.0 * w, ab, W1, W2)
    for a, b in zip(fused2, fused):
        np.testing.assert_array_equal(a, 2.0 * b)


def test_dispatch_bwd_against_torch_autograd():
    """dh = w (dy W2) and the SwiGLU backward by torch float64 autograd (not the closed
    form), rounded to bf16 where the GPU path stores da, db and dxp."""
    dy, w, ab, W1, W2 = _dispatch_case(seed=5)
    f = W2.shape[1]
    dab, dxr = oracle.ffn_bwd_rows_dispatch(dy, w, ab, W1, W2)
    t = lambda a: torch.tensor(a, dtype=torch.float64)
    a = t(ab[:, :f]).requires_grad_(True)
    b = t(ab[:, f:]).requires_grad_(True)
    dh = (t(w)[:, None] * t(dy)) @ t(W2)
    hh = torch.nn.functional.silu(a) * b
    ga, gb = torch.autograd.grad(hh, (a, b), grad_outputs=dh)
    r_dab = oracle.bf16(torch.cat([ga, gb], 1).numpy())
    assert rel_l2(dab, r_dab) < 1e-12
    r_dx = oracle.bf16((torch.tensor(r_dab) @ t(W1)).numpy())
    np.testing.assert_array_equal(dxr, r_dx)
    # and it differs from the unfused rows (bf16-rounded w * dy) only by that rounding
    plain, _ = oracle.ffn_bwd_rows(oracle.bf16(dy * w[:, None]), ab, W1, W2)
    assert 0 < rel_l2(dab, plain) < 1e-2
