"""Seeded random layer configurations, compared with the oracle in full (every output).

Each case draws the shape (T, d, f, E, k, a shared expert or none), the gate, a capacity
or none, a Zipf skew or none and the routing variants (selection-only bias, negative-score
dropping, dropping by score, FC1 recompute) from a fixed seed, within the library's limits
and small enough for the float64 oracle to finish in seconds.  The fixed cases elsewhere
pin the known edges; these look for combinations nobody listed."""

import numpy as np
import pytest
import torch

import oracle
import token_dispatch_expert_gb300 as tde
from gpu_util import assert_close, dev, f64, np_i, record, stats
from test_gpu_layer import ROUTE_KEYS, check_layer_sampled, run_layer
from test_gpu_mxfp8 import assert_layer_mx_wgrad, mx_cfg
from workloads import MoEConfig, gen_inputs_host

pytestmark = pytest.mark.gpu

N_CASES = 64
N_PAIR_CASES = 40


def draw_config(i: int) -> MoEConfig:
    rng = np.random.default_rng(1000 + i)
    E = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 32, 64, 100, 256]))
    k = int(rng.integers(1, min(8, E) + 1))
    d = int(rng.choice([64, 128, 192, 256, 384, 512]))
    f = int(rng.choice([64, 128, 192, 256, 320, 448, 512, 640]))
    fs = int(rng.choice([64, 128, 192])) if rng.random() < 0.3 else 0
    # tokens: mostly a sizeable fraction of a cap that keeps the oracle's work around 1e9
    # flops, sometimes a handful (log-uniform)
    cap_t = max(2, min(3000, int(1.5e9 / (12 * k * d * f + (12 * d * fs if fs else 0)))))
    if rng.random() < 0.2:
        T = max(1, int(np.exp(rng.uniform(0, np.log(cap_t)))))
    else:
        T = max(1, int(rng.uniform(0.25, 1.0) * cap_t))
    sigmoid = rng.random() < 0.35
    cap = float(rng.uniform(0.3, 1.5)) if rng.random() < 0.4 else None
    zipf = float(rng.uniform(0.8, 1.6)) if rng.random() < 0.7 else None
    alpha = float(rng.uniform(0.5, 3.0))
    bias = (tuple(float(v) for v in rng.normal(0, 0.7, E)) if rng.random() < 0.15 else None)
    drop_neg = bool(rng.random() < 0.1)
    by_score = bool(cap is not None and rng.random() < 0.4)
    recompute = bool(rng.random() < 0.15)
    return MoEConfig(f"fuzz{i}", T=T, d=d, E=E, k=k, f=f, fs=fs,
                     gate="sigmoid" if sigmoid else "softmax",
                     route_scale=2.5 if sigmoid else 1.0, cap_factor=cap, zipf_s=zipf,
                     zipf_alpha=alpha, select_bias=bias, drop_negative=drop_neg,
                     drop_by_score=by_score, recompute=recompute)


def draw_pair_config(i: int) -> MoEConfig:
    """Few experts and many rows each, so the CTA-pair tiles, their swap-AB tail tiles and
    long segments are exercised (at least 192 rows per expert on average)."""
    rng = np.random.default_rng(2000 + i)
    E = int(rng.choice([1, 2, 3, 4, 5, 6, 8]))
    k = int(rng.integers(1, min(4, E) + 1))
    d = int(rng.choice([64, 128, 192, 256]))
    f = int(rng.choice([64, 128, 192, 256, 320, 384]))
    fs = int(rng.choice([64, 128])) if rng.random() < 0.25 else 0
    lo = (192 * E + k - 1) // k
    hi = max(lo + 1, min(12000, int(2e9 / (12 * k * d * f + (12 * d * fs if fs else 0)))))
    T = int(rng.integers(lo, hi + 1))
    sigmoid = rng.random() < 0.3
    cap = float(rng.uniform(0.8, 1.5)) if rng.random() < 0.3 else None
    zipf = float(rng.uniform(0.5, 1.3)) if rng.random() < 0.5 else None
    return MoEConfig(f"fuzzpair{i}", T=T, d=d, E=E, k=k, f=f, fs=fs,
                     gate="sigmoid" if sigmoid else "softmax",
                     route_scale=2.5 if sigmoid else 1.0, cap_factor=cap, zipf_s=zipf,
                     zipf_alpha=float(rng.uniform(0.3, 1.0)),
                     drop_by_score=bool(cap is not None and rng.random() < 0.4),
                     recompute=bool(rng.random() < 0.15))


def test_draws_are_within_the_limits():
    for c in [draw_config(i) for i in range(N_CASES)] + [draw_pair_config(i)
                                                         for i in range(N_PAIR_CASES)]:
        assert 1 <= c.k <= min(8, c.E) and c.E <= 256 and c.d % 64 == 0 and c.f % 64 == 0


@pytest.mark.parametrize("i", [f"any{i}" for i in range(N_CASES)] +
                         [f"pair{i}" for i in range(N_PAIR_CASES)])
def test_layer_random_config_full_compare(i):
    c = draw_config(int(i[3:])) if i.startswith("any") else draw_pair_config(int(i[4:]))
    inp = gen_inputs_host(c)
    g = {k: dev(v) for k, v in inp.items()}
    layer, y, gr = run_layer(c, g)
    assert layer.status() == (0, 0), c
    fo = oracle.layer_fwd(c, inp)
    bo = oracle.layer_bwd(c, inp, fo)
    v = layer.views()
    for key in ROUTE_KEYS:
        if key in v:
            np.testing.assert_array_equal(np_i(v[key]), fo["route"][key], err_msg=f"{key} {c}")
    assert_close("y", f64(y), fo["y"])
    assert_close("dx", f64(gr["dx"]), bo["dx"])
    assert_close("dlogits", f64(gr["dlogits"]), bo["dlogits"])
    for e in range(c.E):
        if fo["route"]["kept"][e] == 0:
            assert (f64(gr["dW1"][e]) == 0).all() and (f64(gr["dW2"][e]) == 0).all()
            continue
        assert_close(f"dW1[{e}]", f64(gr["dW1"][e]), bo["dW1"][e])
        assert_close(f"dW2[{e}]", f64(gr["dW2"][e]), bo["dW2"][e])
    if c.fs:
        assert_close("dW1s", f64(gr["dW1s"]), bo["dW1s"])
        assert_close("dW2s", f64(gr["dW2s"]), bo["dW2s"])


N_MX_CASES = 40


def draw_mx_config(i: int):
    """The MXFP8 layer (routed forward and data gradients, with level 2 the weight
    gradients too): d, f multiples of 128, one-CTA and CTA-pair segment lengths."""
    rng = np.random.default_rng(3000 + i)
    E = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
    k = int(rng.integers(1, min(4, E) + 1))
    d = int(rng.choice([128, 256, 384]))
    f = int(rng.choice([128, 256, 384, 512]))
    fs = int(rng.choice([128, 256])) if rng.random() < 0.25 else 0
    cap_t = max(2, min(6000, int(1.5e9 / (12 * k * d * f + (12 * d * fs if fs else 0)))))
    T = max(1, int(rng.uniform(0.1, 1.0) * cap_t))
    sigmoid = rng.random() < 0.3
    cap = float(rng.uniform(0.6, 1.5)) if rng.random() < 0.3 else None
    zipf = float(rng.uniform(0.6, 1.4)) if rng.random() < 0.5 else None
    level = int(rng.choice([1, 2]))
    c = MoEConfig(f"fuzzmx{i}", T=T, d=d, E=E, k=k, f=f, fs=fs,
                  gate="sigmoid" if sigmoid else "softmax",
                  route_scale=2.5 if sigmoid else 1.0, cap_factor=cap, zipf_s=zipf)
    return c, level


@pytest.mark.parametrize("i", range(N_MX_CASES))
def test_mx_layer_random_config(i):
    c, level = draw_mx_config(i)
    inp = gen_inputs_host(c)
    g = {k: dev(v) for k, v in inp.items()}
    layer = tde.MoELayer(mx_cfg(c, level))
    wq = layer.quantize_weights(g["W1"], g["W2"])
    y = layer.forward_mx(g["logits"], g["x"], wq, g.get("W1s"), g.get("W2s"))
    gr = layer.backward_mx(g["logits"], g["x"], g["dy"], wq, g.get("W1s"), g.get("W2s"))
    torch.cuda.synchronize()
    assert layer.status() == (0, 0), (c, level)
    fo = oracle.layer_fwd(c, inp, mx=True)
    bo = oracle.layer_bwd(c, inp, fo, mx=True, mx_wgrad=level == 2)
    plain = oracle.layer_bwd(c, inp, fo, mx=True) if level == 2 else None
    # y and dx pass through E4M3 codes that each side takes from its own bf16 h and dab;
    # where those differ by one bf16 step at a block's largest element the whole block's
    # scale can move, so these two take the layer-level MXFP8 bound (rel-L2 1e-2, every
    # entry within 0.1 of rms + |o|); dlogits does not pass through a quantisation
    for name, got, ref in (("y", y, fo["y"]), ("dx", gr["dx"], bo["dx"])):
        st = stats(f64(got), ref)
        record(name, st)
        assert st["rel_l2"] <= 1e-2 and st["max_scaled"] <= 0.1, (name, st)
    assert_close("dlogits", f64(gr["dlogits"]), bo["dlogits"])
    for e in range(c.E):
        if fo["route"]["kept"][e] == 0:
            continue
        if level == 2:
            assert_layer_mx_wgrad(f"dW1[{e}]", f64(gr["dW1"][e]), bo["dW1"][e], plain["dW1"][e])
            assert_layer_mx_wgrad(f"dW2[{e}]", f64(gr["dW2"][e]), bo["dW2"][e], plain["dW2"][e])
        else:
            assert_close(f"dW1[{e}]", f64(gr["dW1"][e]), bo["dW1"][e])
            assert_close(f"dW2[{e}]", f64(gr["dW2"][e]), bo["dW2"][e])
    if c.fs:
        assert_close("dW1s", f64(gr["dW1s"]), bo["dW1s"])
        assert_close("dW2s", f64(gr["dW2s"]), bo["dW2s"])


N_BIG_CASES = 8


def draw_big_config(i: int) -> MoEConfig:
    """Large shapes, checked on sampled outputs: tens of thousands of tokens, widths up to
    4096, up to 256 experts, many tiles per CTA and long or very uneven segments."""
    rng = np.random.default_rng(4000 + i)
    E = int(rng.choice([2, 4, 8, 16, 32, 64, 128, 256]))
    k = int(rng.integers(1, min(8, E) + 1))
    d = int(rng.choice([512, 1024, 2048, 4096]))
    f = int(rng.choice([256, 512, 768, 1024, 1408, 2048]))
    fs = int(rng.choice([512, 1024])) if rng.random() < 0.25 else 0
    T = int(rng.choice([4096, 8192, 16384, 32768, 65536]))
    while T * k * max(d, f) * 6 > (40 << 30) or E * 3 * d * f * 2 > (8 << 30):
        T //= 2                                  # keep the device footprint to a few GB
    sigmoid = rng.random() < 0.3
    cap = float(rng.uniform(0.7, 1.5)) if rng.random() < 0.35 else None
    zipf = float(rng.uniform(0.6, 1.6)) if rng.random() < 0.7 else None
    return MoEConfig(f"fuzzbig{i}", T=T, d=d, E=E, k=k, f=f, fs=fs,
                     gate="sigmoid" if sigmoid else "softmax",
                     route_scale=2.5 if sigmoid else 1.0, cap_factor=cap, zipf_s=zipf,
                     zipf_alpha=float(rng.uniform(0.3, 2.0)),
                     drop_by_score=bool(cap is not None and rng.random() < 0.4))


@pytest.mark.parametrize("i", range(N_BIG_CASES))
def test_layer_random_large_config_sampled(i):
    check_layer_sampled(draw_big_config(i))


N_ROUTE_CASES = 200


def draw_route_config(i: int):
    """Routing alone (bit-exact): any token count up to 2^17, any expert count up to 256,
    k up to 8, the gates, capacities, skews, ties and the routing variants.  Returns the
    configuration and its logits; a third of the cases quantise the logits to a coarse grid
    so that ties between experts and between tokens are common."""
    rng = np.random.default_rng(5000 + i)
    E = int(rng.integers(1, 257))
    k = int(rng.integers(1, min(8, E) + 1))
    T = int(np.exp(rng.uniform(0, np.log(1 << 17))))
    sigmoid = rng.random() < 0.3
    cap = float(rng.uniform(0.1, 2.0)) if rng.random() < 0.5 else None
    c = MoEConfig(f"fuzzroute{i}", T=max(1, T), d=64, E=E, k=k, f=64,
                  gate="sigmoid" if sigmoid else "softmax",
                  route_scale=2.5 if sigmoid else 1.0, cap_factor=cap,
                  zipf_s=float(rng.uniform(0.5, 2.0)) if rng.random() < 0.6 else None,
                  zipf_alpha=float(rng.uniform(0.3, 3.0)),
                  select_bias=(tuple(float(v) for v in np.round(rng.normal(0, 1, E), 2))
                               if rng.random() < 0.25 else None),
                  drop_negative=bool(rng.random() < 0.2),
                  drop_by_score=bool(cap is not None and rng.random() < 0.5))
    from workloads import gen_logits
    logits = gen_logits(c)
    if rng.random() < 0.33:
        logits = np.round(logits * 2.0) / 2.0          # a half-unit grid: many exact ties
    return c, logits.astype(np.float32)


@pytest.mark.parametrize("i", range(N_ROUTE_CASES))
def test_route_random_config_bit_exact(i):
    from gpu_util import run_route
    c, logits = draw_route_config(i)
    r, ws = run_route(c, dev(logits))
    o = oracle.route(c, logits)
    for key in ROUTE_KEYS:
        np.testing.assert_array_equal(np_i(r[key]), o[key], err_msg=f"{key} {c}")
    w = np_i(r["topk_w"]).astype(np.float64)
    np.testing.assert_allclose(w, o["topk_w"], rtol=2.0 ** -20, atol=1e-30)
    assert tde.moe_status(ws) == (0, 0)

