"""Pins of the oracle's MXFP8 arithmetic (the NEXT-2 row).

* E4M3 rounding and encoding: every finite code round-trips; random values (normal,
  subnormal, ties) agree with torch's float8_e4m3fn conversion, which rounds to nearest
  even; magnitudes above 448 saturate (torch's cast does not, so those are checked by hand).
* MX block quantisation: hand-worked blocks (tests/golden/mxfp8_blocks_hand_worked.json),
  the scale rule against numpy's frexp, the per-block error bound, and scale invariance
  (multiplying a block by 2^j shifts its scale code by j and keeps its element codes).
* The MXFP8 FFN forward: equal to the plain FFN when every operand is exactly
  representable; otherwise equal to a torch float64 composition of the pinned quantiser.
* The MXFP8 weight gradients: the column quantiser (32-row blocks from a segment's first
  row) on the hand-worked blocks laid down a column, by brute force on a segment with a
  short tail, block locality, exactness on representable operands, and the composition
  Q(dab)^T Q(xp), Q(dyp)^T Q(h).
CPU only."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits_to_f64, gen_rows_bf16

HERE = os.path.dirname(os.path.abspath(__file__))


def torch_e4m3(v):
    return torch.tensor(v, dtype=torch.float64).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_every_finite_code_round_trips():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c, v in enumerate(vals):
        if np.isnan(v):
            assert c in (0x7F, 0xFF)
            continue
        assert oracle.e4m3(v) == v
        assert oracle.e4m3_code(v) == c, (c, v)


def test_rounding_matches_torch_in_range():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(20000) * 50,                       # normals
        rng.standard_normal(5000) * 2.0 ** -8,                 # subnormal range
        (rng.integers(-900, 900, 5000) + 0.5) * 2.0 ** -9,     # subnormal ties
        (rng.integers(16, 31, 3000) * 2 + 1) * 2.0 ** rng.integers(-7, 4, 3000),  # ties
    ])
    v = v[np.abs(v) <= 448.0]
    ours = np.array([oracle.e4m3(x) for x in v])
    np.testing.assert_array_equal(ours, torch_e4m3(v))


def test_saturation():
    for v, q in [(448.0, 448.0), (449.0, 448.0), (463.9, 448.0), (464.0, 448.0),
                 (500.0, 448.0), (1e30, 448.0), (-1e5, -448.0), (-450.0, -448.0)]:
        assert oracle.e4m3(v) == q
    assert oracle.e4m3_code(448.0) == 0x7E and oracle.e4m3_code(-448.0) == 0xFE


def test_hand_worked_blocks():
    g = json.load(open(os.path.join(HERE, "golden", "mxfp8_blocks_hand_worked.json")))
    v = np.zeros((len(g["blocks"]), 32))
    exp_codes = np.zeros((len(g["blocks"]), 32), np.uint8)
    for i, b in enumerate(g["blocks"]):
        for k, x in b["values"].items():
            v[i, int(k)] = x
        for k, c in b["codes"].items():
            exp_codes[i, int(k)] = c
    codes, scales, deq = oracle.mx_quantize_rows(v)
    np.testing.assert_array_equal(scales[:, 0], [b["scale"] for b in g["blocks"]])
    np.testing.assert_array_equal(codes, exp_codes)


def test_scale_rule_error_bound_and_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, (64, 1)))
    x[5, 32:64] = 0.0
    codes, scales, deq = oracle.mx_quantize_rows(x)
    blocks = x.reshape(64, 8, 32)
    amax = np.abs(blocks).max(-1)
    _, e = np.frexp(amax)
    X = np.where(amax > 0, np.clip(e - 1 - 8, -127, 127), -127)
    np.testing.assert_array_equal(scales.astype(int), X + 127)
    err = np.abs(deq - x).reshape(64, 8, 32).max(-1)
    assert (err <= amax / 8 + 1e-300).all()               # saturation costs at most 1/8
    # scale invariance: x * 2^j -> the same element codes, scale codes shifted by j
    c2, s2, d2 = oracle.mx_quantize_rows(x * 2.0 ** 5)
    np.testing.assert_array_equal(c2, codes)
    nz = amax > 0
    np.testing.assert_array_equal(s2.astype(int)[nz], scales.astype(int)[nz] + 5)
    np.testing.assert_array_equal(d2, deq * 2.0 ** 5)


def exactly_representable(shape, rng):
    """Values j/8, |j| <= 14, every block of 32 holding one value of magnitude in [1, 2):
    the block scale is 2^-8 and every element maps to an E4M3 value exactly."""
    j = rng.integers(-14, 15, shape)
    j[..., ::32] = rng.choice([-12, -8, 8, 12], size=j[..., ::32].shape)
    return j / 8.0


def test_mx_ffn_equals_plain_ffn_on_representable_operands():
    rng = np.random.default_rng(9)
    n, d, f = 40, 128, 64
    x = exactly_representable((n, d), rng)
    W1 = exactly_representable((2 * f, d), rng)
    W2 = exactly_representable((d, f), rng)
    for m in (x, W1, W2):
        np.testing.assert_array_equal(oracle.mx_quantize_rows(m)[2], m)
    ab, h, yp, hc, hs = oracle.ffn_fwd_rows_mx(x, W1, W2)
    ab0, h0, _ = oracle.ffn_fwd_rows(x, W1, W2)
    np.testing.assert_array_equal(ab, ab0)
    np.testing.assert_array_equal(h, h0)


def test_mx_ffn_matches_torch_composition():
    n, d, f = 33, 96, 64
    x = bf16_bits_to_f64(gen_rows_bf16("mx_x", n, d))
    W1 = bf16_bits_to_f64(gen_rows_bf16("mx_w1", 2 * f, d, std=0.05))
    W2 = bf16_bits_to_f64(gen_rows_bf16("mx_w2", d, f, std=0.05))
    ab, h, yp, hc, hs = oracle.ffn_fwd_rows_mx(x, W1, W2)

    def bf(t):
        return t.to(torch.bfloat16).to(torch.float64)

    q = lambda m: torch.tensor(oracle.mx_quantize_rows(m)[2])
    ab_t = bf(q(x) @ q(W1).T)
    a, b = ab_t[:, :f], ab_t[:, f:]
    h_t = bf(torch.nn.functional.silu(a) * b)
    hq = oracle.mx_quantize_rows(h_t.numpy())
    y_t = bf(torch.tensor(hq[2]) @ q(W2).T)
    np.testing.assert_allclose(ab, ab_t.numpy(), rtol=0, atol=0)
    np.testing.assert_array_equal(h, h_t.numpy())
    np.testing.assert_array_equal(hc, hq[0])
    np.testing.assert_array_equal(hs, hq[1])
    np.testing.assert_allclose(yp, y_t.numpy(), rtol=2 ** -8, atol=1e-12)


@pytest.mark.parametrize("mx_bwd", [False, True])
def test_sampled_mx_layer_matches_full_mx_layer(mx_bwd):
    """layer_sampled(mx=True[, mx_bwd]) is an exact restriction of layer_fwd(mx=True) +
    layer_bwd(mx=mx_bwd)."""
    from workloads import MoEConfig, gen_inputs_host
    cfg = MoEConfig("mx_sample", T=96, d=128, E=4, k=2, f=128, cap_factor=0.8, zipf_s=1.1)
    inp = gen_inputs_host(cfg)
    f = oracle.layer_fwd(cfg, inp, mx=True)
    b = oracle.layer_bwd(cfg, inp, f, mx=mx_bwd)
    toks = [0, 5, 17, 95, 42]
    experts = [0, 3]
    wcols = np.array([0, 7, 63, 100])
    wrows = np.array([1, 2, 63, 127])
    s = oracle.layer_sampled(cfg, oracle.HostSource(inp), toks, experts, wcols, wrows, mx=True,
                             mx_bwd=mx_bwd)
    tk = np.array(sorted(toks))
    np.testing.assert_array_equal(s["y"], f["y"][tk])
    np.testing.assert_array_equal(s["dx"], b["dx"][tk])
    np.testing.assert_allclose(s["dlogits"], b["dlogits"][tk], rtol=1e-12, atol=1e-14)
    one_ulp = 2.0 ** -7      # rows summed in another order before the final rounding
    for e in experts:
        np.testing.assert_allclose(s["dW1"][e][0], b["dW1"][e][np.ix_(wcols, wrows)],
                                   rtol=one_ulp, atol=1e-30)
        np.testing.assert_allclose(s["dW1"][e][1], b["dW1"][e][np.ix_(wcols + cfg.f, wrows)],
                                   rtol=one_ulp, atol=1e-30)
        np.testing.assert_allclose(s["dW2"][e], b["dW2"][e][np.ix_(wrows, wcols)],
                                   rtol=one_ulp, atol=1e-30)
    # and it differs from the bf16 layer (the quantisation is really applied)
    f16 = oracle.layer_fwd(cfg, inp)
    assert (f16["y"] != f["y"]).any()


def test_mx_bwd_equals_plain_bwd_on_representable_operands():
    """With every GEMM operand exactly representable in MXFP8 (along both axes for the
    weights), the MXFP8 data gradients equal the plain ones exactly."""
    rng = np.random.default_rng(12)
    n, d, f = 32, 128, 64
    W1 = exactly_representable((2 * f, d), rng)
    W2 = exactly_representable((d, f), rng)
    # the transposes must be representable too: a value of magnitude in [1,2) in every
    # 32-block along the other axis as well
    W1[:, ::32] = 1.0
    W1[::32, :] = 1.0
    W2[:, ::32] = 1.0
    W2[::32, :] = 1.0
    for m in (W1, W2, W1.T.copy(), W2.T.copy()):
        np.testing.assert_array_equal(oracle.mx_quantize_rows(m)[2], m)
    dyp = exactly_representable((n, d), rng)
    ab = exactly_representable((n, 2 * f), rng) / 4
    dab_mx, dx_mx, dc, ds = oracle.ffn_bwd_rows_mx(dyp, ab, W1, W2)
    dab, dx = oracle.ffn_bwd_rows(dyp, ab, W1, W2)
    np.testing.assert_array_equal(dab_mx, dab)
    # dab itself is generally not representable: the second GEMM sees its quantisation
    dabq = oracle.mx_quantize_rows(dab)[2]
    dx_ref = oracle.bf16(dabq @ W1)
    np.testing.assert_allclose(dx_mx, dx_ref, rtol=2 ** -8, atol=1e-30)
    np.testing.assert_array_equal(dc, oracle.mx_quantize_rows(dab)[0])
    np.testing.assert_array_equal(ds, oracle.mx_quantize_rows(dab)[1])


def test_mx_bwd_matches_torch_composition():
    n, d, f = 40, 96, 64
    dyp = bf16_bits_to_f64(gen_rows_bf16("mxb_dy", n, d))
    ab = bf16_bits_to_f64(gen_rows_bf16("mxb_ab", n, 2 * f))
    W1 = bf16_bits_to_f64(gen_rows_bf16("mxb_w1", 2 * f, d, std=0.05))
    W2 = bf16_bits_to_f64(gen_rows_bf16("mxb_w2", d, f, std=0.05))
    dab, dx, dc, ds = oracle.ffn_bwd_rows_mx(dyp, ab, W1, W2)

    def bf(t):
        return t.to(torch.bfloat16).to(torch.float64)

    q = lambda m: torch.tensor(oracle.mx_quantize_rows(np.ascontiguousarray(m))[2])
    dh = q(dyp) @ q(W2.T).T                                # contraction over d
    a, b = torch.tensor(ab[:, :f]), torch.tensor(ab[:, f:])
    s = torch.sigmoid(a)
    dab_t = torch.cat([bf(dh * b * s * (1 + a * (1 - s))), bf(dh * a * s)], dim=1)
    np.testing.assert_allclose(dab, dab_t.numpy(), rtol=2 ** -7, atol=1e-12)
    dx_t = bf(q(dab) @ q(W1.T).T)                          # contraction over 2f
    np.testing.assert_allclose(dx, dx_t.numpy(), rtol=2 ** -7, atol=1e-10)


# --------------------------------------------------------------- weight gradients (along tokens)
def test_hand_worked_blocks_down_a_column():
    """The column quantiser on the hand-worked blocks laid down a column: the same scale
    codes and element values as the blocks worked along a row."""
    g = json.load(open(os.path.join(HERE, "golden", "mxfp8_blocks_hand_worked.json")))
    nb = len(g["blocks"])
    col = np.zeros((32 * nb, 3))
    for i, b in enumerate(g["blocks"]):
        for k, x in b["values"].items():
            col[32 * i + int(k), 1] = x
    deq = oracle.mx_quantize_cols(col)
    for i, b in enumerate(g["blocks"]):
        X = b["scale"] - 127
        want = np.zeros(32)
        for k, c in b["codes"].items():
            s, e, m = c >> 7, (c >> 3) & 15, c & 7
            mag = (1 + m / 8) * 2.0 ** (e - 7) if e else m / 8 * 2.0 ** -6
            want[int(k)] = (-mag if s else mag) * 2.0 ** X
        np.testing.assert_array_equal(deq[32 * i:32 * i + 32, 1], want)
    assert (deq[:, 0] == 0).all() and (deq[:, 2] == 0).all()


def test_column_blocks_start_at_row_zero_and_short_tail_ignores_padding():
    """Blocks are rows [32j, 32j + 32) of the segment; the short last block is quantised
    from its own values only (as if zero-padded); a change in one block leaves every other
    block alone."""
    rng = np.random.default_rng(21)
    n = 70                                     # 32 + 32 + 6
    v = rng.standard_normal((n, 5)) * np.exp(rng.uniform(-4, 4, (1, 5)))
    deq = oracle.mx_quantize_cols(v)
    # each block by brute force: the scale rule and E4M3 rounding element by element
    for c in range(5):
        for r0 in (0, 32, 64):
            blk = v[r0:min(r0 + 32, n), c]
            amax = np.abs(blk).max()
            X = max(-127, min(127, int(np.frexp(amax)[1]) - 1 - 8))
            want = np.array([oracle.e4m3(x / 2.0 ** X) for x in blk]) * 2.0 ** X
            np.testing.assert_array_equal(deq[r0:r0 + len(blk), c], want)
    v2 = v.copy()
    v2[40, 2] *= 1000.0                        # only rows 32..63 of column 2 may change
    d2 = oracle.mx_quantize_cols(v2)
    changed = d2 != deq
    assert changed[32:64, 2].any()
    changed[32:64, 2] = False
    assert not changed.any()


def test_mx_wgrad_equals_plain_on_representable_operands():
    """With each operand exactly representable in 32-row column blocks, the MXFP8 weight
    gradients equal the plain ones exactly."""
    rng = np.random.default_rng(31)
    n, d, f = 64, 64, 32
    def col_repr(shape):
        return np.ascontiguousarray(exactly_representable(shape[::-1], rng).T)
    xr, h, dyp, dab = col_repr((n, d)), col_repr((n, f)), col_repr((n, d)), col_repr((n, 2 * f))
    for m in (xr, h, dyp, dab):
        np.testing.assert_array_equal(oracle.mx_quantize_cols(m), m)
    w1, w2 = oracle.ffn_wgrad_rows_mx(xr, h, dyp, dab, d, f)
    p1, p2 = oracle.layer.ffn_wgrad_rows(xr, h, dyp, dab, d, f)
    np.testing.assert_array_equal(w1, p1)
    np.testing.assert_array_equal(w2, p2)


def test_mx_wgrad_matches_numpy_composition():
    """dW1 = Q(dab)^T Q(xp) and dW2 = Q(dyp)^T Q(h), Q the column quantiser, summed over an
    uneven segment (45 rows: one full block and a 13-row tail)."""
    n, d, f = 45, 64, 32
    xr = bf16_bits_to_f64(gen_rows_bf16("mxw_x", n, d))
    h = bf16_bits_to_f64(gen_rows_bf16("mxw_h", n, f))
    dyp = bf16_bits_to_f64(gen_rows_bf16("mxw_dy", n, d))
    dab = bf16_bits_to_f64(gen_rows_bf16("mxw_dab", n, 2 * f))
    w1, w2 = oracle.ffn_wgrad_rows_mx(xr, h, dyp, dab, d, f)
    Q = oracle.mx_quantize_cols
    np.testing.assert_allclose(w1, Q(dab).T @ Q(xr), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(w2, Q(dyp).T @ Q(h), rtol=1e-12, atol=1e-14)
    # the quantisation is applied: differs from the plain gradients
    p1, _ = oracle.layer.ffn_wgrad_rows(xr, h, dyp, dab, d, f)
    assert (w1 != p1).any()
    # an empty segment gives zero gradients
    z1, z2 = oracle.ffn_wgrad_rows_mx(xr[:0], h[:0], dyp[:0], dab[:0], d, f)
    assert not z1.any() and not z2.any()


def test_sampled_mx_wgrad_matches_full():
    from workloads import MoEConfig, gen_inputs_host
    cfg = MoEConfig("mxw_sample", T=96, d=128, E=4, k=2, f=128, cap_factor=0.8, zipf_s=1.1)
    inp = gen_inputs_host(cfg)
    f = oracle.layer_fwd(cfg, inp, mx=True)
    b = oracle.layer_bwd(cfg, inp, f, mx=True, mx_wgrad=True)
    wcols = np.array([0, 7, 63, 100])
    wrows = np.array([1, 2, 63, 127])
    experts = [0, 3]
    s = oracle.layer_sampled(cfg, oracle.HostSource(inp), [0, 5], experts, wcols, wrows,
                             mx=True, mx_bwd=True, mx_wgrad=True)
    one_ulp = 2.0 ** -7
    for e in experts:
        np.testing.assert_allclose(s["dW1"][e][0], b["dW1"][e][np.ix_(wcols, wrows)],
                                   rtol=one_ulp, atol=1e-30)
        np.testing.assert_allclose(s["dW1"][e][1], b["dW1"][e][np.ix_(wcols + cfg.f, wrows)],
                                   rtol=one_ulp, atol=1e-30)
        np.testing.assert_allclose(s["dW2"][e], b["dW2"][e][np.ix_(wrows, wcols)],
                                   rtol=one_ulp, atol=1e-30)
    b0 = oracle.layer_bwd(cfg, inp, f, mx=True)
    assert (b0["dW2"] != b["dW2"]).any()
