"""GPU parity of the whole layer (moe_layer_fwd + moe_layer_bwd) against the oracle.

Small and mid shapes: every output compared in full (y, dx, dW1, dW2, dlogits, the
shared expert's grads, and the saved routing bit-exact).  The five workload shapes at
full size, in the configuration the benchmark times: routing bit-exact in full; y, dx
and dlogits on 256 sampled tokens; weight-gradient entries of three whole experts (the
most loaded, the least loaded non-empty one and expert 0) on sampled rows/columns --
each sampled value is the oracle's exact definition restricted to that output."""

import numpy as np
import pytest
import torch

import oracle
import token_dispatch_expert_gb300 as tde
from gpu_util import assert_close, cfg_c, dev, f64, np_i
from workloads import CONFIGS, MoEConfig, gen_inputs_device, gen_inputs_host, gen_logits

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": CONFIGS["tiny"],
    "tiny_cap": CONFIGS["tiny"].replace(name="tiny_cap", cap_factor=0.5),
    "mid": MoEConfig("mid", T=1024, d=512, E=8, k=2, f=512, zipf_s=1.1),
    "mid_sig_shared": MoEConfig("mid_sig_shared", T=768, d=384, E=16, k=4, f=256, fs=256,
                                gate="sigmoid", route_scale=2.5, cap_factor=1.0, zipf_s=1.2),
    # 600 = 2 x 256 + 88 rows: the shared expert's last M tile is a swap-AB tail tile
    "shared_tail": MoEConfig("shared_tail", T=600, d=256, E=4, k=2, f=320, fs=192,
                             gate="sigmoid", route_scale=2.5, zipf_s=1.0),
    # degenerate routings: every token to every expert (k = E), a single token, and a
    # capacity of 6 rows per expert (most assignments dropped)
    "k_eq_E": MoEConfig("k_eq_E", T=200, d=128, E=4, k=4, f=128),
    "T1": MoEConfig("T1_layer", T=1, d=128, E=4, k=2, f=128),
    "cap_tiny": MoEConfig("cap_tiny", T=256, d=128, E=8, k=2, f=128, cap_factor=0.1,
                          zipf_s=1.2),
    # extreme skew: every token to the same expert (1100 rows = 4 whole M tiles and a
    # 76-row tail tile; the seven other experts empty), and every token to the same two
    # experts of sixteen, with a shared expert
    "one_hot": MoEConfig("one_hot", T=1100, d=256, E=8, k=1, f=256, zipf_s=1.0,
                         zipf_alpha=20.0),
    "two_hot_shared": MoEConfig("two_hot", T=700, d=256, E=16, k=2, f=192, fs=128,
                                gate="sigmoid", route_scale=2.5, zipf_s=1.0, zipf_alpha=20.0),
    # the edges of the shape limits: a single expert (k = 1; 300 rows = one whole M tile and
    # a 44-row tail tile), the smallest dims (d = f = 64: one K block, one 64-column N
    # tile), the largest expert count (E = 256, the group limit, with k = 8: about 16 rows
    # per expert, one-CTA tiles, some experts empty), and dims that are odd multiples of 64
    # on CTA pairs (d = 192: three K blocks; f = 448: a half-filled last N tile)
    "E1": MoEConfig("E1", T=300, d=128, E=1, k=1, f=128),
    "min_dims": MoEConfig("min_dims", T=129, d=64, E=4, k=2, f=64),
    "E256": MoEConfig("E256", T=512, d=128, E=256, k=8, f=64, zipf_s=1.1),
    "odd64": MoEConfig("odd64", T=1024, d=192, E=4, k=2, f=448, zipf_s=1.0),
}

ROUTE_KEYS = ["topk_idx", "counts", "kept", "offsets", "dest_row", "src_tok", "src_slot",
              "drop_mask"]


def run_layer(c, g):
    cfg = cfg_c(c)
    layer = tde.MoELayer(cfg)
    y = layer.forward(g["logits"], g["x"], g["W1"], g["W2"], g.get("W1s"), g.get("W2s"))
    grads = layer.backward(g["logits"], g["x"], g["dy"], g["W1"], g["W2"], g.get("W1s"),
                           g.get("W2s"))
    torch.cuda.synchronize()
    return layer, y, grads


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small_full_compare(name):
    c = SMALL[name]
    inp = gen_inputs_host(c)
    g = {k: dev(v) for k, v in inp.items()}
    layer, y, gr = run_layer(c, g)
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
    if c.fs:
        assert_close("dW1s", f64(gr["dW1s"]), bo["dW1s"])
        assert_close("dW2s", f64(gr["dW2s"]), bo["dW2s"])


def test_layer_twice_is_bitwise_deterministic():
    c = SMALL["mid_sig_shared"]
    g = {k: dev(v) for k, v in gen_inputs_host(c).items()}
    _, y1, g1 = run_layer(c, g)
    _, y2, g2 = run_layer(c, g)
    assert torch.equal(y1, y2)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


# a long token axis with narrow experts: 262144 kept rows, about a thousand M tiles per
# launch and a few hundred tiles per CTA pair, and a row count past 2^17 in every offset
LONG = MoEConfig("long_tokens", T=131072, d=256, E=16, k=2, f=512, zipf_s=1.1)


@pytest.mark.parametrize("name", ["mixtral", "qwen3", "dsv3", "capacity", "long_tokens"])
def test_layer_full_size_sampled(name):
    check_layer_sampled(LONG if name == "long_tokens" else CONFIGS[name])


def check_layer_sampled(c):
    """The layer at a size the oracle cannot evaluate in full: routing in full; y, dx and
    dlogits on 256 sampled tokens (plus dropped ones under a capacity); 16 x 64 entries of
    the weight gradients of three experts (the most loaded, the least loaded non-empty one,
    expert 0) and of the shared expert."""
    g = gen_inputs_device(c, "cuda")
    layer, y, gr = run_layer(c, g)
    assert layer.status() == (0, 0)
    src = oracle.TorchSource(g)
    logits = src.logits
    o_r = oracle.route(c, logits)
    v = layer.views()
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(np_i(v[key]), o_r[key], err_msg=key)
    rng = np.random.default_rng(0)
    toks = rng.choice(c.T, size=256, replace=False)
    if c.capacity:   # make sure some sampled tokens have dropped slots
        dropped = np.nonzero(o_r["drop_mask"].any(1))[0]
        toks = np.unique(np.concatenate([toks, dropped[:8]]))
    kept = o_r["kept"]
    nz = np.nonzero(kept)[0]
    experts = sorted({int(np.argmax(kept)), int(nz[np.argmin(kept[nz])]), 0})
    wcols = np.sort(rng.choice(min(c.f, c.fs) if c.fs else c.f, size=16, replace=False))
    wrows = np.sort(rng.choice(c.d, size=64, replace=False))
    s = oracle.layer_sampled(c, src, toks, experts, wcols, wrows)
    tk = s["tokens"]
    assert_close("y", f64(y[torch.as_tensor(tk).cuda()]), s["y"])
    assert_close("dx", f64(gr["dx"][torch.as_tensor(tk).cuda()]), s["dx"])
    assert_close("dlogits", f64(gr["dlogits"][torch.as_tensor(tk).cuda()]), s["dlogits"])
    dW1 = gr["dW1"]; dW2 = gr["dW2"]
    for e in experts:
        if kept[e] == 0:
            continue
        gate = f64(dW1[e][torch.as_tensor(wcols).cuda()][:, torch.as_tensor(wrows).cuda()])
        up = f64(dW1[e][torch.as_tensor(wcols + c.f).cuda()][:, torch.as_tensor(wrows).cuda()])
        w2 = f64(dW2[e][torch.as_tensor(wrows).cuda()][:, torch.as_tensor(wcols).cuda()])
        assert_close(f"dW1 gate[{e}]", gate, s["dW1"][e][0])
        assert_close(f"dW1 up[{e}]", up, s["dW1"][e][1])
        assert_close(f"dW2[{e}]", w2, s["dW2"][e])
    if c.fs:
        wc = torch.as_tensor(wcols).cuda(); wr = torch.as_tensor(wrows).cuda()
        assert_close("dW1s gate", f64(gr["dW1s"][wc][:, wr]), s["dW1s"][0])
        assert_close("dW1s up", f64(gr["dW1s"][wc + c.fs][:, wr]), s["dW1s"][1])
        assert_close("dW2s", f64(gr["dW2s"][wr][:, wc]), s["dW2s"])
