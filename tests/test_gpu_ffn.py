"""GPU parity of the grouped SwiGLU FFN (the tcgen05 grouped GEMMs) against the oracle's
per-expert rows: FC1 + SwiGLU epilogue, FC2, FC2 data-gradient + SwiGLU backward,
FC1 data-gradient and the two variable-K weight gradients.  Shapes span several M, N
and K tiles with ragged segment ends, an empty expert, N tails narrower than a tile,
and buffer rows past offsets[E] poisoned with NaN (they must not leak into anything)."""

import numpy as np
import pytest
import torch

import oracle
import token_dispatch_expert_gb300 as tde
from gpu_util import assert_close, cfg_c, dev, f64, new_ws
from test_gpu_fuzz import draw_config, draw_pair_config
from workloads import CONFIGS, MoEConfig, gen_bf16, gen_inputs_host, gen_logits, gen_rows_bf16

pytestmark = pytest.mark.gpu

NAN_BF16 = np.uint16(0x7FC0)

CASES = {
    "tiny": CONFIGS["tiny"],
    "ragged": MoEConfig("ragged", T=512, d=256, E=4, k=2, f=384, zipf_s=1.2),
    "tails_empty": MoEConfig("tails_empty", T=700, d=320, E=5, k=2, f=192, cap_factor=0.9,
                             zipf_s=1.0),
    "single": MoEConfig("single", T=300, d=128, E=1, k=1, f=256),
    "deepK": MoEConfig("deepK", T=256, d=1024, E=3, k=1, f=640),
}
# seeded random shapes (the layer fuzz's drawers, routing variants off): three on the
# one-CTA path, three on the CTA-pair path
for _i in range(3):
    CASES[f"rand{_i}"] = draw_config(100 + _i).replace(
        select_bias=None, drop_negative=False, drop_by_score=False, recompute=False)
    CASES[f"randpair{_i}"] = draw_pair_config(100 + _i).replace(drop_by_score=False,
                                                               recompute=False)


def setup(c):
    inp = gen_inputs_host(c)
    logits = gen_logits(c)
    if c.name == "tails_empty":
        logits[:, 4] = -1e30            # expert 4 never selected: an empty segment
    o = oracle.route(c, logits)
    n = int(o["offsets"][-1])
    R = c.T * c.k
    xp = np.full((R, c.d), NAN_BF16, np.uint16)
    xp[:n] = inp["x"][o["src_tok"][:n]]
    return inp, o, n, xp


@pytest.mark.parametrize("name", list(CASES))
def test_grouped_ffn_fwd(name):
    c = CASES[name]
    inp, o, n, xp = setup(c)
    R = c.T * c.k
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    ab = torch.empty((R, 2 * c.f), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((R, c.f), dtype=torch.bfloat16, device="cuda")
    yp = torch.empty((R, c.d), dtype=torch.bfloat16, device="cuda")
    tde.moe_grouped_ffn(cfg, dev(xp), dev(o["offsets"]), dev(inp["W1"]), dev(inp["W2"]), ab, h,
                        yp, ws)
    off = o["offsets"]
    r_ab = np.empty((n, 2 * c.f)); r_h = np.empty((n, c.f)); r_yp = np.empty((n, c.d))
    for e in range(c.E):
        s, t = int(off[e]), int(off[e + 1])
        r_ab[s:t], r_h[s:t], r_yp[s:t] = oracle.ffn_fwd_rows(xp[s:t], inp["W1"][e], inp["W2"][e])
    assert_close("ab", f64(ab)[:n], r_ab)
    assert_close("h", f64(h)[:n], r_h)
    assert_close("yp", f64(yp)[:n], r_yp)
    assert tde.moe_status(ws) == (0, 0)


@pytest.mark.parametrize("name", list(CASES))
def test_grouped_ffn_bwd(name):
    c = CASES[name]
    inp, o, n, xp = setup(c)
    R = c.T * c.k
    off = o["offsets"]
    # the backward's saved inputs come from the oracle's forward (rounded to bf16)
    ab = np.empty((n, 2 * c.f)); h = np.empty((n, c.f))
    for e in range(c.E):
        s, t = int(off[e]), int(off[e + 1])
        ab[s:t], h[s:t], _ = oracle.ffn_fwd_rows(xp[s:t], inp["W1"][e], inp["W2"][e])
    dyp = gen_rows_bf16("dyp", R, c.d)
    dyp[n:] = NAN_BF16

    def bits(a, rows, cols):
        t = torch.full((rows, cols), float("nan"), dtype=torch.bfloat16)
        t[:n] = torch.from_numpy(a).to(torch.bfloat16)   # exact: a holds bf16 values
        return t.cuda()

    cfg = cfg_c(c)
    ws = new_ws(cfg)
    dab = torch.empty((R, 2 * c.f), dtype=torch.bfloat16, device="cuda")
    dxp = torch.empty((R, c.d), dtype=torch.bfloat16, device="cuda")
    dW1 = torch.full((c.E, 2 * c.f, c.d), 7.0, dtype=torch.bfloat16, device="cuda")
    dW2 = torch.full((c.E, c.d, c.f), 7.0, dtype=torch.bfloat16, device="cuda")
    tde.moe_grouped_ffn_bwd(cfg, dev(dyp), dev(xp), dev(off), dev(inp["W1"]), dev(inp["W2"]),
                            bits(ab, R, 2 * c.f), bits(h, R, c.f), dab, dxp, dW1, dW2, ws)
    r_dab = np.empty((n, 2 * c.f)); r_dxp = np.empty((n, c.d))
    r_dW1 = np.zeros((c.E, 2 * c.f, c.d)); r_dW2 = np.zeros((c.E, c.d, c.f))
    for e in range(c.E):
        s, t = int(off[e]), int(off[e + 1])
        r_dab[s:t], r_dxp[s:t] = oracle.ffn_bwd_rows(dyp[s:t], ab[s:t], inp["W1"][e],
                                                     inp["W2"][e])
        r_dW1[e], r_dW2[e] = oracle.layer.ffn_wgrad_rows(
            oracle.layer._f64(xp[s:t]), h[s:t], oracle.layer._f64(dyp[s:t]), r_dab[s:t], c.d, c.f)
    assert_close("dab", f64(dab)[:n], r_dab)
    assert_close("dxp", f64(dxp)[:n], r_dxp)
    g1, g2 = f64(dW1), f64(dW2)
    for e in range(c.E):
        if off[e + 1] == off[e]:
            assert (g1[e] == 0).all() and (g2[e] == 0).all(), "empty expert must get zero dW"
            continue
        assert_close(f"dW1[{e}]", g1[e], oracle.bf16(r_dW1[e]))
        assert_close(f"dW2[{e}]", g2[e], oracle.bf16(r_dW2[e]))
    assert tde.moe_status(ws) == (0, 0)


EDGE_CASES = {
    # an empty segment, one row, segment ends 1, 64, 127, 128, 129 and 255 rows into a
    # 256-row tile, segments of several tiles, and an N tail (f = 192)
    "edges": ([1, 64, 127, 128, 129, 255, 300, 600, 0, 385], 256, 192),
    # the swap-AB tail tiles (a segment's last tile with at most 160 rows): N = rows rounded
    # up to 32 at 31 / 32 / 33 rows, the largest tail (160), the smallest ordinary last tile
    # (161), a full last tile (256), tails after full tiles (416 = 256 + 160, 417), and N
    # tails in FC1 (f = 320: the last FC1 tile holds 64 valid columns, all in the first CTA)
    # and in FC2 / FC1 data-gradient (d = 384)
    "tail_edges": ([31, 32, 33, 160, 161, 256, 416, 417, 2, 700], 384, 320),
    # a long segment whose last M tile is a 64-row swap-AB tail tile, taken by CTA pairs
    # that go on to ordinary FC1 tiles right after it: the up warp hands its transposed
    # block to the gate warp and must not restage an ordinary tile into it before the gate
    # warp has read it (once seen as corrupted b, h on the tail rows)
    "long_tail": ([40000, 1000], 256, 512),
}


@pytest.mark.parametrize("name", list(EDGE_CASES))
def test_grouped_ffn_segment_edges(name):
    """Segment sizes chosen to hit the tile cases of the CTA-pair path."""
    sizes, d, f = EDGE_CASES[name]
    E = len(sizes)
    n = sum(sizes)
    c = MoEConfig(name, T=n, d=d, E=E, k=1, f=f)
    assert n / E >= 192          # average rows per group: the pair path is taken
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    inp = gen_inputs_host(c)
    xp = inp["x"]
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    R = c.T * c.k
    ab = torch.empty((R, 2 * c.f), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((R, c.f), dtype=torch.bfloat16, device="cuda")
    yp = torch.empty((R, c.d), dtype=torch.bfloat16, device="cuda")
    tde.moe_grouped_ffn(cfg, dev(xp), dev(off), dev(inp["W1"]), dev(inp["W2"]), ab, h, yp, ws)
    r_ab = np.empty((n, 2 * c.f)); r_h = np.empty((n, c.f)); r_yp = np.empty((n, c.d))
    for e in range(E):
        s, t = int(off[e]), int(off[e + 1])
        r_ab[s:t], r_h[s:t], r_yp[s:t] = oracle.ffn_fwd_rows(xp[s:t], inp["W1"][e], inp["W2"][e])
    assert_close("ab", f64(ab), r_ab)
    assert_close("h", f64(h), r_h)
    assert_close("yp", f64(yp), r_yp)
    # backward from the oracle's saved tensors
    dyp = gen_rows_bf16("dyp_edges", R, c.d)
    dab = torch.empty((R, 2 * c.f), dtype=torch.bfloat16, device="cuda")
    dxp = torch.empty((R, c.d), dtype=torch.bfloat16, device="cuda")
    dW1 = torch.full((E, 2 * c.f, c.d), 7.0, dtype=torch.bfloat16, device="cuda")
    dW2 = torch.full((E, c.d, c.f), 7.0, dtype=torch.bfloat16, device="cuda")
    tde.moe_grouped_ffn_bwd(cfg, dev(dyp), dev(xp), dev(off), dev(inp["W1"]), dev(inp["W2"]),
                            torch.from_numpy(r_ab).to(torch.bfloat16).cuda(),
                            torch.from_numpy(r_h).to(torch.bfloat16).cuda(), dab, dxp, dW1, dW2,
                            ws)
    r_dab = np.empty((n, 2 * c.f)); r_dxp = np.empty((n, c.d))
    g1, g2 = f64(dW1), f64(dW2)
    for e in range(E):
        s, t = int(off[e]), int(off[e + 1])
        r_dab[s:t], r_dxp[s:t] = oracle.ffn_bwd_rows(dyp[s:t], r_ab[s:t], inp["W1"][e],
                                                     inp["W2"][e])
        w1, w2 = oracle.layer.ffn_wgrad_rows(oracle.layer._f64(xp[s:t]), r_h[s:t],
                                             oracle.layer._f64(dyp[s:t]), r_dab[s:t], c.d, c.f)
        if t == s:
            assert (g1[e] == 0).all() and (g2[e] == 0).all()
        else:
            assert_close(f"dW1[{e}]", g1[e], oracle.bf16(w1))
            assert_close(f"dW2[{e}]", g2[e], oracle.bf16(w2))
    assert_close("dab", f64(dab), r_dab)
    assert_close("dxp", f64(dxp), r_dxp)
    assert tde.moe_status(ws) == (0, 0)


@pytest.mark.parametrize("name", list(CASES) + ["edges"])
def test_gather_fused_ffn_against_oracle(name):
    """The permute folded into FC1's operand loads (and into the FC1 weight gradient's):
    every output is compared with the oracle's per-expert rows on the gathered tokens
    (ab, h, yp; dab, dxp, dW1, dW2), and must also equal the unfused path bit for bit (the
    gathered rows are the same bf16 values the permute would have written)."""
    if name == "edges":
        sizes = [1, 64, 127, 128, 129, 255, 300, 600, 0, 385]
        c = MoEConfig("edges_g", T=sum(sizes), d=320, E=len(sizes), k=1, f=192)
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        # a scrambled token order: row p of the buffer reads token perm[p]
        perm = np.random.default_rng(5).permutation(c.T).astype(np.int32)
        inp = gen_inputs_host(c)
        src_tok, n = perm, c.T
    else:
        c = CASES[name]
        inp, o, n, _ = setup(c)
        off, src_tok = o["offsets"], o["src_tok"]
    R = c.T * c.k
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    x, W1, W2 = dev(inp["x"]), dev(inp["W1"]), dev(inp["W2"])
    d_off, d_src = dev(off), dev(src_tok)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    xp = torch.full((R, c.d), float("nan"), **bf)
    tde.moe_permute(cfg, x, d_src, d_off, xp, ws)
    out_u = [torch.full(s, float("nan"), **bf) for s in [(R, 2 * c.f), (R, c.f), (R, c.d)]]
    out_g = [torch.full(s, float("nan"), **bf) for s in [(R, 2 * c.f), (R, c.f), (R, c.d)]]
    tde.moe_grouped_ffn(cfg, xp, d_off, W1, W2, *out_u, ws)
    tde.moe_grouped_ffn_gather(cfg, x, d_src, d_off, W1, W2, *out_g, ws)
    torch.cuda.synchronize()
    # the oracle on the rows the gather reads: xp[p] = x[src_tok[p]], built on the host
    xp_h = inp["x"][src_tok[:n]]
    r_ab = np.empty((n, 2 * c.f)); r_h = np.empty((n, c.f)); r_yp = np.empty((n, c.d))
    for e in range(c.E):
        s0, t0 = int(off[e]), int(off[e + 1])
        r_ab[s0:t0], r_h[s0:t0], r_yp[s0:t0] = oracle.ffn_fwd_rows(xp_h[s0:t0], inp["W1"][e],
                                                                   inp["W2"][e])
    for a, b, r, nm in zip(out_u, out_g, (r_ab, r_h, r_yp), ("ab", "h", "yp")):
        assert_close(f"gather {nm}", f64(b)[:n], r)
        assert torch.equal(a[:n], b[:n]), nm
    # backward from the oracle's saved ab, h (bf16 values), on both paths
    dyp_h = gen_rows_bf16("dyp_g", R, c.d)
    dyp = dev(dyp_h)
    ab = torch.full((R, 2 * c.f), float("nan"), **bf)
    h = torch.full((R, c.f), float("nan"), **bf)
    ab[:n] = torch.from_numpy(r_ab).to(torch.bfloat16).cuda()
    h[:n] = torch.from_numpy(r_h).to(torch.bfloat16).cuda()

    def bwd(fn, src):
        dab = torch.empty((R, 2 * c.f), **bf)
        dxp = torch.empty((R, c.d), **bf)
        dW1 = torch.full((c.E, 2 * c.f, c.d), 7.0, **bf)
        dW2 = torch.full((c.E, c.d, c.f), 7.0, **bf)
        fn(cfg, dyp, *src, d_off, W1, W2, ab, h, dab, dxp, dW1, dW2, ws)
        torch.cuda.synchronize()
        return dab, dxp, dW1, dW2

    u = bwd(tde.moe_grouped_ffn_bwd, (xp,))
    g = bwd(tde.moe_grouped_ffn_bwd_gather, (x, d_src))
    for a, b, nm in zip(u, g, ("dab", "dxp", "dW1", "dW2")):
        if nm in ("dab", "dxp"):
            a, b = a[:n], b[:n]
        assert torch.equal(a, b), nm
    r_dab = np.empty((n, 2 * c.f)); r_dxp = np.empty((n, c.d))
    g1, g2 = f64(g[2]), f64(g[3])
    for e in range(c.E):
        s0, t0 = int(off[e]), int(off[e + 1])
        r_dab[s0:t0], r_dxp[s0:t0] = oracle.ffn_bwd_rows(dyp_h[s0:t0], r_ab[s0:t0],
                                                         inp["W1"][e], inp["W2"][e])
        if t0 == s0:
            assert (g1[e] == 0).all() and (g2[e] == 0).all(), "empty expert must get zero dW"
            continue
        w1, w2 = oracle.layer.ffn_wgrad_rows(oracle.layer._f64(xp_h[s0:t0]), r_h[s0:t0],
                                             oracle.layer._f64(dyp_h[s0:t0]), r_dab[s0:t0],
                                             c.d, c.f)
        assert_close(f"gather dW1[{e}]", g1[e], oracle.bf16(w1))
        assert_close(f"gather dW2[{e}]", g2[e], oracle.bf16(w2))
    assert_close("gather dab", f64(g[0])[:n], r_dab)
    assert_close("gather dxp", f64(g[1])[:n], r_dxp)
    assert tde.moe_status(ws) == (0, 0)


@pytest.mark.parametrize("name", list(CASES) + ["edges"])
def test_dispatch_fused_fc2_dgrad_against_oracle(name):
    """The dispatch of dy fused into the FC2 data-gradient: its rows are dy[src_tok[p]] and
    dh is scaled by the slot's gate weight in the epilogue (w * dy is never rounded to bf16),
    so dab and dxp are compared with the oracle's exact-product variant; dW2 still contracts
    the stored bf16(w * dy) rows, dW1 the fused dab.  Covers ragged segments, an empty
    expert, the swap-AB tail tiles and a scrambled token order."""
    if name == "edges":
        sizes = [1, 64, 127, 128, 129, 255, 300, 600, 0, 385]
        c = MoEConfig("edges_d", T=sum(sizes), d=320, E=len(sizes), k=1, f=192)
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        perm = np.random.default_rng(7).permutation(c.T).astype(np.int32)
        inp = gen_inputs_host(c)
        src_tok, src_slot, n = perm, perm.copy(), c.T      # k = 1: slot = token
        topk_w = np.random.default_rng(8).uniform(0.05, 1.0, c.T).astype(np.float32)
    else:
        c = CASES[name]
        inp, o, n, _ = setup(c)
        off, src_tok, src_slot = o["offsets"], o["src_tok"], o["src_slot"]
        topk_w = o["topk_w"].reshape(-1).astype(np.float32)
    R = c.T * c.k
    xp_h = inp["x"][src_tok[:n]]
    w_rows = topk_w[src_slot[:n]].astype(np.float64)
    dy64 = oracle.layer._f64(inp["dy"])
    # the forward's saved tensors and the stored dyp rows, from the oracle
    r_ab = np.empty((n, 2 * c.f)); r_h = np.empty((n, c.f))
    for e in range(c.E):
        s0, t0 = int(off[e]), int(off[e + 1])
        r_ab[s0:t0], r_h[s0:t0], _ = oracle.ffn_fwd_rows(xp_h[s0:t0], inp["W1"][e], inp["W2"][e])
    dyp_h = oracle.bf16(dy64[src_tok[:n]] * w_rows[:, None])
    bf = dict(dtype=torch.bfloat16, device="cuda")

    def rows(a, cols):
        t = torch.full((R, cols), float("nan"), **bf)
        t[:n] = torch.from_numpy(a).to(torch.bfloat16).cuda()
        return t

    cfg = cfg_c(c)
    ws = new_ws(cfg)
    slots = np.full(R, -1, np.int32); slots[:n] = src_slot[:n]
    toks = np.full(R, -1, np.int32); toks[:n] = src_tok[:n]
    dab = torch.empty((R, 2 * c.f), **bf)
    dxp = torch.empty((R, c.d), **bf)
    dW1 = torch.full((c.E, 2 * c.f, c.d), 7.0, **bf)
    dW2 = torch.full((c.E, c.d, c.f), 7.0, **bf)
    tde.moe_grouped_ffn_bwd_dispatch(cfg, dev(inp["dy"]), dev(topk_w), dev(toks), dev(slots),
                                     rows(dyp_h, c.d), rows(oracle.layer._f64(xp_h), c.d),
                                     dev(off), dev(inp["W1"]), dev(inp["W2"]),
                                     rows(r_ab, 2 * c.f), rows(r_h, c.f), dab, dxp, dW1, dW2, ws)
    torch.cuda.synchronize()
    r_dab = np.empty((n, 2 * c.f)); r_dxp = np.empty((n, c.d))
    g1, g2 = f64(dW1), f64(dW2)
    for e in range(c.E):
        s0, t0 = int(off[e]), int(off[e + 1])
        r_dab[s0:t0], r_dxp[s0:t0] = oracle.ffn_bwd_rows_dispatch(
            inp["dy"][src_tok[s0:t0]], w_rows[s0:t0], r_ab[s0:t0], inp["W1"][e], inp["W2"][e])
        if t0 == s0:
            assert (g1[e] == 0).all() and (g2[e] == 0).all(), "empty expert must get zero dW"
            continue
        w1, w2 = oracle.layer.ffn_wgrad_rows(oracle.layer._f64(xp_h[s0:t0]), r_h[s0:t0],
                                             dyp_h[s0:t0], r_dab[s0:t0], c.d, c.f)
        assert_close(f"dispatch dW1[{e}]", g1[e], oracle.bf16(w1))
        assert_close(f"dispatch dW2[{e}]", g2[e], oracle.bf16(w2))
    assert_close("dispatch dab", f64(dab)[:n], r_dab)
    assert_close("dispatch dxp", f64(dxp)[:n], r_dxp)
    assert tde.moe_status(ws) == (0, 0)


def test_gather_flags_bad_source_rows():
    """An out-of-range source row is flagged (MOE_DEVERR_BAD_INDEX) and row 0 read instead;
    nothing outside x is touched."""
    c = MoEConfig("badg", T=256, d=128, E=2, k=1, f=128)
    inp = gen_inputs_host(c)
    cfg = cfg_c(c)
    ws = new_ws(cfg)
    off = dev(np.array([0, 100, 256], np.int32))
    src = np.arange(256, dtype=np.int32)
    src[17] = 256            # one past the end
    src[200] = -3
    bf = dict(dtype=torch.bfloat16, device="cuda")
    ab, h, yp = (torch.empty(s, **bf) for s in [(256, 256), (256, 128), (256, 128)])
    tde.moe_grouped_ffn_gather(cfg, dev(inp["x"]), dev(src), off, dev(inp["W1"]), dev(inp["W2"]),
                               ab, h, yp, ws)
    st, flags = tde.moe_status(ws)
    assert flags & tde.DEVERR["BAD_INDEX"]
