"""Pins of the oracle's backward pass.

CPU only.  Two independent references, both on the exact (unrounded) layer:
  * torch float64 autograd through the dense masked formulation (tests/dense_ref.py);
  * central finite differences of L = sum(y * dy) evaluated with the oracle's own
    forward, which checks the backward formulas (combine/gate backward, SwiGLU
    backward, the two data-gradient products and the variable-K weight gradients)
    against the forward alone.
Tokens whose k-th and (k+1)-th logits are closer than 10 eps are skipped for the
logit derivatives, because the selection would flip inside the difference stencil.
"""

import math

import numpy as np
import pytest

import oracle
from dense_ref import dense_grads
from workloads import MoEConfig, bf16_bits_to_f64, gen_inputs_host

CFGS = {
    "softmax": MoEConfig("g_soft", T=40, d=64, E=6, k=2, f=64),
    "softmax_cap": MoEConfig("g_cap", T=48, d=64, E=4, k=2, f=64, cap_factor=0.5, zipf_s=1.5),
    "sigmoid_shared": MoEConfig("g_sig", T=36, d=64, E=5, k=3, f=64, fs=64, gate="sigmoid",
                                route_scale=2.5, cap_factor=0.8, zipf_s=1.2),
    # one score carries almost all the weight (a 14-logit gap between the two selected
    # experts): the gate gradient is a tiny difference of nearly equal terms
    "sigmoid_dominant": MoEConfig("g_dom", T=32, d=64, E=6, k=2, f=64, gate="sigmoid",
                                  route_scale=2.5, zipf_s=1.0, zipf_alpha=20.0),
    "softmax_dominant": MoEConfig("g_sdom", T=32, d=64, E=6, k=2, f=64, zipf_s=1.0,
                                  zipf_alpha=20.0),
}


def f64_inputs(cfg):
    inp = gen_inputs_host(cfg)
    out = {"logits": inp["logits"]}
    for n, v in inp.items():
        if n != "logits":
            out[n] = bf16_bits_to_f64(v)
    return out


def oracle_grads(cfg, inp):
    f = oracle.layer_fwd(cfg, inp, rnd=False)
    b = oracle.layer_bwd(cfg, inp, f, rnd=False)
    return f, b


@pytest.mark.parametrize("name", list(CFGS))
def test_backward_equals_autograd_of_dense_layer(name):
    cfg = CFGS[name]
    inp = f64_inputs(cfg)
    f, b = oracle_grads(cfg, inp)
    y_ref, g = dense_grads(cfg, inp)
    np.testing.assert_allclose(f["y"], y_ref.numpy(), rtol=1e-11, atol=1e-13)
    pairs = [("dx", "x"), ("dW1", "W1"), ("dW2", "W2"), ("dlogits", "logits")]
    if cfg.fs:
        pairs += [("dW1s", "W1s"), ("dW2s", "W2s")]
    for ours, leaf in pairs:
        ref = g[leaf].numpy()
        scale = np.abs(ref).max()
        np.testing.assert_allclose(b[ours], ref, rtol=1e-9, atol=1e-11 * scale, err_msg=ours)


def _loss(cfg, inp):
    y = oracle.layer_fwd(cfg, inp, rnd=False)["y"]
    return float((y * inp["dy"]).sum())


@pytest.mark.parametrize("name", list(CFGS))
def test_backward_equals_finite_differences(name):
    cfg = CFGS[name]
    inp = f64_inputs(cfg)
    _, b = oracle_grads(cfg, inp)
    rng = np.random.default_rng(7)
    eps = 1e-4
    checks = []
    for leaf, grad in [("x", "dx"), ("W1", "dW1"), ("W2", "dW2")] + \
            ([("W1s", "dW1s"), ("W2s", "dW2s")] if cfg.fs else []):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, s)) for s in inp[leaf].shape)
            checks.append((leaf, grad, idx))
    # logits: pick tokens with a clear gap between the k-th and (k+1)-th logits
    lg = inp["logits"].astype(np.float64)
    srt = -np.sort(-lg, axis=-1)
    ok = np.nonzero(srt[:, cfg.k - 1] - srt[:, cfg.k] > 10 * eps)[0]
    for t in rng.choice(ok, size=min(8, len(ok)), replace=False):
        for e in range(cfg.E):
            checks.append(("logits", "dlogits", (int(t), e)))
    for leaf, grad, idx in checks:
        p = {n: (v.copy() if n == leaf else v) for n, v in inp.items()}
        base = p[leaf][idx]
        if leaf == "logits":
            # perturb in float32 (the layer's logit dtype); use the realised step
            up = np.float32(base + eps); dn = np.float32(base - eps)
            p[leaf][idx] = up; lp = _loss(cfg, p)
            p[leaf][idx] = dn; lm = _loss(cfg, p)
            fd = (lp - lm) / (float(up) - float(dn))
            tol = 2e-4 * max(1.0, abs(fd))
        else:
            p[leaf][idx] = base + eps; lp = _loss(cfg, p)
            p[leaf][idx] = base - eps; lm = _loss(cfg, p)
            fd = (lp - lm) / (2 * eps)
            tol = 1e-6 * max(1.0, abs(fd))
        assert abs(fd - b[grad][idx]) <= tol, (leaf, idx, fd, b[grad][idx])


@pytest.mark.parametrize("gate", ["softmax", "sigmoid"])
def test_two_expert_gate_gradient_closed_form(gate):
    """k = 2 closed forms, derived by hand, with g_j = <dy, yp_j>:
    softmax, w_0 = 1 / (1 + exp(l_1 - l_0)):  dl_0 = -dl_1 = w_0 w_1 (g_0 - g_1);
    sigmoid, w_j = s sigma_j / S, S = sigma_0 + sigma_1:
        dl_0 = s sigma_0 (1 - sigma_0) sigma_1 (g_0 - g_1) / S^2, and symmetrically."""
    scale = 2.5 if gate == "sigmoid" else 1.0
    cfg = MoEConfig("cf_" + gate, T=24, d=8, E=4, k=2, f=8, gate=gate, route_scale=scale)
    lg = np.random.default_rng(3).standard_normal((cfg.T, cfg.E)).astype(np.float32) * 3
    r = oracle.route(cfg, lg)
    rng = np.random.default_rng(4)
    yp = rng.standard_normal((cfg.T * cfg.k, cfg.d))
    dy = rng.standard_normal((cfg.T, cfg.d))
    _, dl = oracle.combine_bwd(cfg, lg, r, dy, yp, rnd=False)
    for t in range(cfg.T):
        e0, e1 = r["topk_idx"][t]
        g0, g1 = (float(dy[t] @ yp[r["dest_row"][t, j]]) for j in range(2))
        l0, l1 = float(lg[t, e0]), float(lg[t, e1])
        if gate == "softmax":
            w0 = 1.0 / (1.0 + math.exp(l1 - l0))
            d0 = w0 * (1.0 - w0) * (g0 - g1)
            d1 = -d0
        else:
            s0, s1 = 1.0 / (1.0 + math.exp(-l0)), 1.0 / (1.0 + math.exp(-l1))
            S = s0 + s1
            d0 = scale * s0 * (1.0 - s0) * s1 * (g0 - g1) / S ** 2
            d1 = scale * s1 * (1.0 - s1) * s0 * (g1 - g0) / S ** 2
        others = [e for e in range(cfg.E) if e not in (e0, e1)]
        np.testing.assert_allclose([dl[t, e0], dl[t, e1]], [d0, d1], rtol=1e-12, atol=1e-15)
        assert (dl[t, others] == 0).all()


@pytest.mark.parametrize("gate", ["softmax", "sigmoid"])
def test_single_expert_gate_gradient_is_zero(gate):
    """k = 1: both gates renormalise over the one selected expert, so its weight is the
    constant 1 (softmax) or `scale` (sigmoid) and every logit's gradient is exactly 0."""
    scale = 2.5 if gate == "sigmoid" else 1.0
    cfg = MoEConfig("k1_" + gate, T=64, d=8, E=6, k=1, f=8, gate=gate, route_scale=scale)
    lg = np.random.default_rng(5).standard_normal((cfg.T, cfg.E)).astype(np.float32) * 3
    r = oracle.route(cfg, lg)
    np.testing.assert_array_equal(r["topk_w"], np.full((cfg.T, 1), scale))
    rng = np.random.default_rng(6)
    yp = rng.standard_normal((cfg.T, cfg.d))
    dy = rng.standard_normal((cfg.T, cfg.d))
    _, dl = oracle.combine_bwd(cfg, lg, r, dy, yp, rnd=False)
    assert (dl == 0).all()

