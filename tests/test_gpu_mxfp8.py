"""GPU parity of the MXFP8 forward (the NEXT-2 row) against the oracle.

* Quantisation (weights, and activations in the fused permute): E4M3 codes and E8M0
  scales bit-exact -- both sides quantise the same bf16 values with the same rule.
* The block-scaled grouped FFN: ab, h, yp within the bf16 tolerance of the oracle's
  MXFP8 FFN (float64 accumulation of the same dequantised operands).  h's quantisation
  starts from each side's own bf16 h, which may differ by one bf16 step at a few
  elements: its codes must agree wherever both sides quantised the same value, and
  almost everywhere overall.
* The layer: moe_layer_fwd_mx against the oracle's MXFP8 forward, followed by either the
  bf16 backward or moe_layer_bwd_mx (data gradients in MXFP8; with mxfp8 = 2 the weight
  gradients too), each against the oracle's backward of the same kind from the same saved
  tensors.  The MXFP8 weight gradients must also sit much closer to the oracle's MXFP8
  gradient than the unquantised gradient does (a quantisation block misplaced along the
  tokens would not).
"""

import numpy as np
import pytest
import torch

import oracle
import token_dispatch_expert_gb300 as tde
from gpu_util import assert_close, cfg_c, dev, f64, new_ws, np_i, stats
from workloads import MoEConfig, gen_inputs_host, gen_logits

pytestmark = pytest.mark.gpu

CASES = {
    "small": MoEConfig("mx_small", T=512, d=256, E=4, k=2, f=384, zipf_s=1.2),
    "n_tail": MoEConfig("mx_tail", T=700, d=384, E=5, k=2, f=256, cap_factor=0.9, zipf_s=1.0),
    "many": MoEConfig("mx_many", T=1024, d=512, E=16, k=4, f=256, zipf_s=1.1),
    # rows per expert >= 192: the CTA-pair kernels (ragged ends, an N tail in FC2)
    "pair": MoEConfig("mx_pair", T=1500, d=384, E=4, k=2, f=384, zipf_s=1.3),
    "pair_cap": MoEConfig("mx_pair_cap", T=2048, d=256, E=3, k=1, f=512, cap_factor=0.8,
                          zipf_s=1.0),
    # 256 fine-grained experts: the largest expert count, many empty and one-row segments
    "fine": MoEConfig("mx_fine", T=512, d=256, E=256, k=8, f=256, zipf_s=1.2),
    # every token to every expert
    "k_eq_E": MoEConfig("mx_kE", T=200, d=256, E=4, k=4, f=256),
}


def _random_mx_shape(i):
    """A seeded random shape within the MXFP8 limits (d, f multiples of 128)."""
    rng = np.random.default_rng(6000 + i)
    E = int(rng.choice([2, 3, 4, 8, 32]))
    k = int(rng.integers(1, min(4, E) + 1))
    return MoEConfig(f"mx_rand{i}", T=int(rng.integers(64, 2500)),
                     d=int(rng.choice([128, 256, 384, 512])), E=E, k=k,
                     f=int(rng.choice([128, 256, 384, 640])),
                     zipf_s=float(rng.uniform(0.5, 1.5)),
                     cap_factor=float(rng.uniform(0.7, 1.3)) if rng.random() < 0.3 else None)


for _i in range(3):
    CASES[f"rand{_i}"] = _random_mx_shape(_i)


def mx_cfg(c, level=1):
    return tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs, c.gate, c.route_scale, c.capacity,
                           mxfp8=level)


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_layer_mx_wgrad(name, got, mx_ref, plain_ref):
    """Layer-level MXFP8 weight gradients, where each side quantises its own bf16 dab and h:
    those can differ by one bf16 step at a few elements, and an element whose E4M3 code
    flips moves by up to 1/8 of itself, so a single gradient entry summed over a short
    segment can move by a few percent of the gradient's rms.  Checked: rel-L2 within the
    bf16 tolerance, every entry within 0.1 of (rms + |o|), and the whole gradient much
    closer to the MXFP8 reference than the unquantised gradient is."""
    s = stats(got, mx_ref)
    assert np.isfinite(got).all(), name
    assert s["rel_l2"] <= 1e-2 and s["max_scaled"] <= 0.1, (name, s)
    gap = rel_l2(plain_ref, mx_ref)
    if gap > 0:
        assert rel_l2(got, mx_ref) < 0.25 * gap, (name, rel_l2(got, mx_ref), gap)


def assert_mx_wgrad(name, got, mx_ref, plain_ref):
    """got within the tolerance of the MXFP8 reference, and much closer to it than the plain
    (unquantised) gradient is: a quantisation block misplaced along the tokens would land
    about as far away as the plain gradient."""
    assert_close(name, got, mx_ref)
    gap = rel_l2(plain_ref, mx_ref)
    if gap > 0:
        assert rel_l2(got, mx_ref) < 0.25 * gap, (name, rel_l2(got, mx_ref), gap)


def unatom(atoms, n_rows_blocks, KB, rows_fn):
    """Rebuild row-major scales [rows][K/32] from the blob's atoms (the inverse of the
    documented layout: byte 16*(m%32) + 4*(m/32) + j of atom (..., kb, half))."""
    out = {}
    a = atoms.reshape(-1, 512)
    for idx in range(a.shape[0]):
        half = idx % 2
        kb = (idx // 2) % KB
        blk = idx // 2 // KB
        for m in range(128):
            row = rows_fn(blk, half, m)
            if row is None:
                continue
            for j in range(4):
                out[(row, 4 * kb + j)] = a[idx, 16 * (m % 32) + 4 * (m // 32) + j]
    return out


def test_weight_quantisation_bit_exact():
    c = MoEConfig("mx_w", T=64, d=384, E=3, k=1, f=256)
    inp = gen_inputs_host(c)
    cfg = mx_cfg(c)
    nbytes, offs = tde.moe_mx_weights_size(cfg)
    wq = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    tde.moe_mx_quantize_weights(cfg, dev(inp["W1"]), dev(inp["W2"]), wq)
    blob = np_i(wq)
    E, d, f = c.E, c.d, c.f
    w1 = inp["W1"].reshape(E * 2 * f, d)
    w2 = inp["W2"].reshape(E * d, f)
    c1, s1, _ = oracle.mx_quantize_rows(w1)
    c2, s2, _ = oracle.mx_quantize_rows(w2)
    np.testing.assert_array_equal(blob[offs[0]:offs[0] + w1.size].reshape(w1.shape), c1)
    np.testing.assert_array_equal(blob[offs[2]:offs[2] + w2.size].reshape(w2.shape), c2)
    # W1 atoms [E][f/128][d/128][2][512]
    NB, KB = f // 128, d // 128
    g1 = unatom(blob[offs[1]:offs[1] + E * NB * KB * 1024], NB, KB,
                lambda blk, half, m: (blk // NB) * 2 * f + half * f + (blk % NB) * 128 + m)
    for (row, b), v in g1.items():
        assert v == s1[row, b], (row, b)
    assert len(g1) == s1.size
    # W2 atoms [E][ceil(d/256)][f/128][2][512]; rows past d are padding
    NT, KB2 = (d + 255) // 256, f // 128

    def w2_row(blk, half, m):
        e, nt = blk // NT, blk % NT
        r = nt * 256 + half * 128 + m
        return e * d + r if r < d else None

    g2 = unatom(blob[offs[3]:offs[3] + E * NT * KB2 * 1024], NT, KB2, w2_row)
    for (row, b), v in g2.items():
        assert v == s2[row, b], (row, b)
    assert len(g2) == s2.size
    # the backward's transposes: W2^T [E][f][d] along d, W1^T [E][d][2f] along 2f
    w2t = np.concatenate([inp["W2"][e].T for e in range(E)])          # [E*f, d]
    w1t = np.concatenate([inp["W1"][e].T for e in range(E)])          # [E*d, 2f]
    ct2, st2, _ = oracle.mx_quantize_rows(np.ascontiguousarray(w2t))
    ct1, st1, _ = oracle.mx_quantize_rows(np.ascontiguousarray(w1t))
    np.testing.assert_array_equal(blob[offs[4]:offs[4] + w2t.size].reshape(w2t.shape), ct2)
    np.testing.assert_array_equal(blob[offs[6]:offs[6] + w1t.size].reshape(w1t.shape), ct1)
    for off_at, C, K, st in ((offs[5], f, d, st2), (offs[7], d, 2 * f, st1)):
        NTt, KBt = (C + 255) // 256, K // 128

        def t_row(blk, half, m, C=C, NTt=NTt):
            e, nt = blk // NTt, blk % NTt
            r = nt * 256 + half * 128 + m
            return e * C + r if r < C else None

        gt = unatom(blob[off_at:off_at + E * NTt * KBt * 1024], NTt, KBt, t_row)
        for (row, b), v in gt.items():
            assert v == st[row, b], (row, b)
        assert len(gt) == st.size


def act_scales_rowmajor(buf, off, n, K):
    """Row-major [n][K/32] scales from an activation atom array (the inverse of the
    documented layout: atom ((off[e] >> 7) + e + l//128) * (K/128) + kb, byte
    16*(m%32) + 4*(m//32) + j for local row l = p - off[e], m = l % 128)."""
    off = np.asarray(off, np.int64)
    E = len(off) - 1
    p = np.arange(n, dtype=np.int64)
    e = np.minimum(np.searchsorted(off, p, side="right") - 1, E - 1)
    l = p - off[e]
    blk = (off[e] >> 7) + e + (l >> 7)
    m = l & 127
    b = np.arange(K // 32, dtype=np.int64)
    kb, j = b // 4, b % 4
    byte = ((blk[:, None] * (K // 128) + kb[None, :]) * 512 + 16 * (m[:, None] % 32)
            + 4 * (m[:, None] // 32) + j[None, :])
    return np.asarray(buf)[byte]


def route_and_inputs(c):
    inp = gen_inputs_host(c)
    o = oracle.route(c, inp["logits"])
    return inp, o, int(o["offsets"][-1])


@pytest.mark.parametrize("name", list(CASES))
def test_permute_quant_bit_exact(name):
    c = CASES[name]
    inp, o, n = route_and_inputs(c)
    cfg = mx_cfg(c)
    ws = new_ws(cfg)
    R = c.T * c.k
    xq = torch.zeros((R, c.d), dtype=torch.uint8, device="cuda")
    xs = torch.zeros(tde.moe_mx_act_scales_size(cfg, c.d), dtype=torch.uint8, device="cuda")
    xp = torch.zeros((R, c.d), dtype=torch.bfloat16, device="cuda")
    tde.moe_mx_permute_quant(cfg, dev(inp["x"]), dev(o["src_tok"]), dev(o["offsets"]), xp, xq,
                             xs, ws)
    rows = inp["x"][o["src_tok"][:n]]
    codes, scales, _ = oracle.mx_quantize_rows(rows)
    np.testing.assert_array_equal(np_i(xq)[:n], codes)
    np.testing.assert_array_equal(act_scales_rowmajor(np_i(xs), o["offsets"], n, c.d), scales)
    np.testing.assert_array_equal(np_i(xp.view(torch.int16))[:n].view(np.uint16), rows)
    assert tde.moe_status(ws) == (0, 0)


def code_agreement(g_codes, o_codes, g_sf, o_sf):
    """Fractions of equal element codes and of equal scale codes."""
    eq = (g_codes == o_codes).mean()
    sf_eq = (g_sf == o_sf).mean()
    return eq, sf_eq


@pytest.mark.parametrize("name", list(CASES))
def test_grouped_ffn_mx_against_oracle(name):
    c = CASES[name]
    inp, o, n = route_and_inputs(c)
    cfg = mx_cfg(c)
    ws = new_ws(cfg)
    R = c.T * c.k
    nbytes, _ = tde.moe_mx_weights_size(cfg)
    wq = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    tde.moe_mx_quantize_weights(cfg, dev(inp["W1"]), dev(inp["W2"]), wq)
    u8 = dict(dtype=torch.uint8, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    xq = torch.zeros((R, c.d), **u8)
    xs = torch.zeros(tde.moe_mx_act_scales_size(cfg, c.d), **u8)
    d_off = dev(o["offsets"])
    tde.moe_mx_permute_quant(cfg, dev(inp["x"]), dev(o["src_tok"]), d_off, None, xq, xs, ws)
    ab = torch.full((R, 2 * c.f), float("nan"), **bf)
    h = torch.full((R, c.f), float("nan"), **bf)
    yp = torch.full((R, c.d), float("nan"), **bf)
    hq = torch.zeros((R, c.f), **u8)
    hs_atoms = torch.zeros(tde.moe_mx_act_scales_size(cfg, c.f), **u8)
    tde.moe_grouped_ffn_mx(cfg, xq, xs, d_off, wq, ab, h, hq, hs_atoms, yp, ws)
    torch.cuda.synchronize()
    hs = act_scales_rowmajor(np_i(hs_atoms), o["offsets"], n, c.f)
    assert tde.moe_status(ws) == (0, 0)
    off = o["offsets"]
    xp = inp["x"][o["src_tok"][:n]]
    r_ab = np.empty((n, 2 * c.f)); r_h = np.empty((n, c.f)); r_yp = np.empty((n, c.d))
    r_hq = np.empty((n, c.f), np.uint8); r_hs = np.empty((n, c.f // 32), np.uint8)
    for e in range(c.E):
        s, t = int(off[e]), int(off[e + 1])
        r_ab[s:t], r_h[s:t], r_yp[s:t], r_hq[s:t], r_hs[s:t] = oracle.ffn_fwd_rows_mx(
            xp[s:t], inp["W1"][e], inp["W2"][e])
    assert_close("ab", f64(ab)[:n], r_ab)
    assert_close("h", f64(h)[:n], r_h)
    assert_close("yp", f64(yp)[:n], r_yp)
    eq, sf_eq = code_agreement(np_i(hq)[:n], r_hq, hs, r_hs)
    assert eq >= 0.99 and sf_eq >= 0.99, (eq, sf_eq)
    # h's codes where both sides quantised the same bf16 value must be identical
    same_h = f64(h)[:n] == r_h
    same = same_h & np.repeat(hs == r_hs, 32, axis=1)
    np.testing.assert_array_equal(np_i(hq)[:n][same], r_hq[same])


@pytest.mark.parametrize("name", ["small", "many", "pair"])
def test_layer_fwd_mx_then_bf16_backward(name):
    c = CASES[name]
    inp = gen_inputs_host(c)
    cfg = mx_cfg(c)
    g = {k: dev(v) for k, v in inp.items()}
    layer = tde.MoELayer(cfg)
    wq = layer.quantize_weights(g["W1"], g["W2"])
    y = layer.forward_mx(g["logits"], g["x"], wq)
    gr = layer.backward(g["logits"], g["x"], g["dy"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    fo = oracle.layer_fwd(c, inp, mx=True)
    bo = oracle.layer_bwd(c, inp, fo)
    assert_close("y", f64(y), fo["y"])
    assert_close("dx", f64(gr["dx"]), bo["dx"])
    assert_close("dlogits", f64(gr["dlogits"]), bo["dlogits"])
    for e in range(c.E):
        if fo["route"]["kept"][e]:
            assert_close(f"dW1[{e}]", f64(gr["dW1"][e]), bo["dW1"][e])
            assert_close(f"dW2[{e}]", f64(gr["dW2"][e]), bo["dW2"][e])
    # and the MXFP8 forward is close to, but not the same as, the bf16 one
    y16 = tde.MoELayer(cfg_c(c)).forward(g["logits"], g["x"], g["W1"], g["W2"])
    diff = np.linalg.norm(f64(y) - f64(y16)) / np.linalg.norm(f64(y16))
    assert 1e-4 < diff < 0.1, diff


WGRAD_EDGES = MoEConfig("mx_wg_edges", T=1, d=256, E=10, k=1, f=256)
# segment sizes around the 32-row quantisation blocks and the 128-row K blocks, an empty
# expert and one long segment
WGRAD_EDGE_SIZES = [0, 1, 31, 32, 33, 127, 128, 129, 300, 600]


@pytest.mark.parametrize("name,level", [(n, 1) for n in CASES] + [(n, 2) for n in CASES] +
                         [("wg_edges", 2)])
def test_grouped_ffn_bwd_mx_against_oracle(name, level):
    """The data gradients on MXFP8 operands (dyp and dab quantised along their contraction
    axes, the weights' transposes from the blob); the weight gradients bf16 (level 1) or on
    operands quantised along each segment's tokens (level 2)."""
    if name == "wg_edges":
        sizes = WGRAD_EDGE_SIZES
        c = WGRAD_EDGES.replace(T=sum(sizes), E=len(sizes))
        inp = gen_inputs_host(c)
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        n = int(off[-1])
        o = {"offsets": off, "src_tok": np.arange(c.T, dtype=np.int32)}
    else:
        c = CASES[name]
        inp, o, n = route_and_inputs(c)
    cfg = mx_cfg(c, level)
    ws = new_ws(cfg)
    R = c.T * c.k
    off = o["offsets"]
    xp = inp["x"][o["src_tok"][:n]]
    ab = np.empty((n, 2 * c.f)); h = np.empty((n, c.f))
    for e in range(c.E):
        s_, t_ = int(off[e]), int(off[e + 1])
        ab[s_:t_], h[s_:t_], _, _, _ = oracle.ffn_fwd_rows_mx(xp[s_:t_], inp["W1"][e],
                                                              inp["W2"][e])
    from workloads import gen_rows_bf16
    dyp = gen_rows_bf16("dyp_mxb", R, c.d)

    def rows_bf16(a, cols):
        t = torch.full((R, cols), float("nan"), dtype=torch.bfloat16)
        t[:n] = torch.from_numpy(np.asarray(a)).to(torch.bfloat16)
        return t.cuda()

    nbytes, _ = tde.moe_mx_weights_size(cfg)
    wq = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    tde.moe_mx_quantize_weights(cfg, dev(inp["W1"]), dev(inp["W2"]), wq)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    xp_t = rows_bf16(oracle.layer._f64(xp), c.d)
    dab = torch.empty((R, 2 * c.f), **bf); dxp = torch.empty((R, c.d), **bf)
    dW1 = torch.full((c.E, 2 * c.f, c.d), 7.0, **bf)
    dW2 = torch.full((c.E, c.d, c.f), 7.0, **bf)
    tde.moe_grouped_ffn_bwd_mx(cfg, dev(dyp), xp_t, dev(off), wq, rows_bf16(ab, 2 * c.f),
                               rows_bf16(h, c.f), dab, dxp, dW1, dW2, ws)
    torch.cuda.synchronize()
    assert tde.moe_status(ws) == (0, 0)
    dyp64 = oracle.layer._f64(dyp)
    r_dab = np.empty((n, 2 * c.f)); r_dxp = np.empty((n, c.d))
    g1, g2 = f64(dW1), f64(dW2)
    dab_gpu = f64(dab[:n])
    for e in range(c.E):
        s_, t_ = int(off[e]), int(off[e + 1])
        r_dab[s_:t_], r_dxp[s_:t_], _, _ = oracle.ffn_bwd_rows_mx(dyp64[s_:t_], ab[s_:t_],
                                                                  inp["W1"][e], inp["W2"][e])
        args = (oracle.layer._f64(xp[s_:t_]), h[s_:t_], dyp64[s_:t_], r_dab[s_:t_], c.d, c.f)
        w1, w2 = oracle.layer.ffn_wgrad_rows(*args)
        if t_ == s_:
            assert (g1[e] == 0).all() and (g2[e] == 0).all()
            continue
        if level == 2:
            # both sides quantise the same bf16 dab: the GPU's own (it may differ from the
            # oracle's by one bf16 step at a few elements, which an E4M3 code step of 1/8
            # would amplify); dab itself is checked against the oracle below
            m1, m2 = oracle.ffn_wgrad_rows_mx(args[0], args[1], args[2], dab_gpu[s_:t_],
                                              c.d, c.f)
            assert_mx_wgrad(f"dW1[{e}]", g1[e], oracle.bf16(m1), oracle.bf16(w1))
            assert_mx_wgrad(f"dW2[{e}]", g2[e], oracle.bf16(m2), oracle.bf16(w2))
        else:
            assert_close(f"dW1[{e}]", g1[e], oracle.bf16(w1))
            assert_close(f"dW2[{e}]", g2[e], oracle.bf16(w2))
    assert_close("dab", f64(dab[:n]), r_dab)
    # dxp from the GPU's own dab (the FC1 data-gradient quantises it along 2f): the oracle's
    # steps composed on the same bf16 input, so an E4M3 code flip from a one-step bf16
    # difference in dab cannot show up as an error here; dxp against the oracle's own chain
    # stays within the rel-L2 tolerance
    Q = lambda m: oracle.mx_quantize_rows(np.ascontiguousarray(m))[2]
    r_dxp_same = np.empty((n, c.d))
    for e in range(c.E):
        s_, t_ = int(off[e]), int(off[e + 1])
        if t_ > s_:
            W1t = oracle.layer._f64(inp["W1"][e]).T            # [d, 2f], quantised along 2f
            r_dxp_same[s_:t_] = oracle.bf16(Q(dab_gpu[s_:t_]) @ Q(W1t).T)
    assert_close("dxp", f64(dxp[:n]), r_dxp_same)
    assert stats(f64(dxp[:n]), r_dxp)["rel_l2"] <= 1e-2


@pytest.mark.parametrize("name,level", [("small", 1), ("many", 1), ("pair", 1), ("fine", 1),
                                        ("k_eq_E", 1), ("pair", 2), ("fine", 2), ("k_eq_E", 2)])
def test_layer_mx_forward_and_backward(name, level):
    c = CASES[name]
    inp = gen_inputs_host(c)
    cfg = mx_cfg(c, level)
    g = {k: dev(v) for k, v in inp.items()}
    layer = tde.MoELayer(cfg)
    wq = layer.quantize_weights(g["W1"], g["W2"])
    y = layer.forward_mx(g["logits"], g["x"], wq)
    gr = layer.backward_mx(g["logits"], g["x"], g["dy"], wq)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    fo = oracle.layer_fwd(c, inp, mx=True)
    bo = oracle.layer_bwd(c, inp, fo, mx=True, mx_wgrad=level == 2)
    assert_close("y", f64(y), fo["y"])
    assert_close("dx", f64(gr["dx"]), bo["dx"])
    assert_close("dlogits", f64(gr["dlogits"]), bo["dlogits"])
    plain = oracle.layer_bwd(c, inp, fo, mx=True) if level == 2 else None
    for e in range(c.E):
        if fo["route"]["kept"][e]:
            if level == 2:
                assert_layer_mx_wgrad(f"dW1[{e}]", f64(gr["dW1"][e]), bo["dW1"][e],
                                      plain["dW1"][e])
                assert_layer_mx_wgrad(f"dW2[{e}]", f64(gr["dW2"][e]), bo["dW2"][e],
                                      plain["dW2"][e])
            else:
                assert_close(f"dW1[{e}]", f64(gr["dW1"][e]), bo["dW1"][e])
                assert_close(f"dW2[{e}]", f64(gr["dW2"][e]), bo["dW2"][e])


@pytest.mark.parametrize("name,level", [("mixtral", 1), ("qwen3", 1), ("dsv3", 1),
                                        ("capacity", 1), ("mixtral", 2), ("capacity", 2)])
def test_layer_mx_full_size_sampled(name, level):
    """The benchmark's MXFP8 configuration at full size (CTA pairs where the benchmark takes
    them; forward and data gradients in MXFP8, with level 2 the weight gradients too): y,
    dx and dlogits of sampled tokens and sampled weight-gradient entries against the
    oracle's exact restriction."""
    from workloads import CONFIGS, gen_inputs_device
    c = CONFIGS[name]
    g = gen_inputs_device(c, "cuda")
    cfg = mx_cfg(c, level)
    layer = tde.MoELayer(cfg)
    wq = layer.quantize_weights(g["W1"], g["W2"])
    y = layer.forward_mx(g["logits"], g["x"], wq, g.get("W1s"), g.get("W2s"))
    gr = layer.backward_mx(g["logits"], g["x"], g["dy"], wq, g.get("W1s"), g.get("W2s"))
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    src = oracle.TorchSource(g)
    rng = np.random.default_rng(1)
    toks = rng.choice(c.T, size=256, replace=False)
    kept = oracle.route(c, src.logits)["kept"]
    nz = np.nonzero(kept)[0]
    experts = sorted({int(np.argmax(kept)), int(nz[np.argmin(kept[nz])]), 0} & set(nz.tolist()))
    wcols = np.sort(rng.choice(c.f, size=16, replace=False))
    wrows = np.sort(rng.choice(c.d, size=64, replace=False))
    s = oracle.layer_sampled(c, src, toks, experts, wcols, wrows, mx=True, mx_bwd=True,
                             mx_wgrad=level == 2)
    tk = torch.as_tensor(s["tokens"]).cuda()
    assert_close("y", f64(y[tk]), s["y"])
    assert_close("dx", f64(gr["dx"][tk]), s["dx"])
    assert_close("dlogits", f64(gr["dlogits"][tk]), s["dlogits"])
    p0 = (oracle.layer_sampled(c, src, toks[:1], experts, wcols, wrows, mx=True, mx_bwd=True)
          if level == 2 else None)
    for e in experts:
        wc = torch.as_tensor(wcols).cuda(); wr = torch.as_tensor(wrows).cuda()
        got = [f64(gr["dW1"][e][wc][:, wr]), f64(gr["dW1"][e][wc + c.f][:, wr]),
               f64(gr["dW2"][e][wr][:, wc])]
        ref = [s["dW1"][e][0], s["dW1"][e][1], s["dW2"][e]]
        for nm, g_, r_, i in zip(("dW1 gate", "dW1 up", "dW2"), got, ref, range(3)):
            if level == 2:
                plain = p0["dW1"][e][i] if i < 2 else p0["dW2"][e]
                assert_layer_mx_wgrad(f"{nm}[{e}]", g_, r_, plain)
            else:
                assert_close(f"{nm}[{e}]", g_, r_)
