"""A second, independent formulation of the MoE layer for pinning the oracle.

Instead of routing rows through a permuted buffer, it evaluates EVERY expert on
EVERY token with dense torch float64 matmuls and masks the result:

    y = sum_e keep[t,e] * w[t,e] * FFN_e(x[t])  (+ FFN_shared(x[t]))

Selection uses numpy's lexsort (key: logit descending, expert id ascending); the
capacity rule keeps the first `cap` tokens (in token order) of each expert, or with
drop-by-score the `cap` with the largest logit (lexsort again); the
gate weights come from torch.softmax over all E experts renormalised over the
selected ones, or from torch.sigmoid normalised over the selected ones.  Gradients
come from torch autograd.  Nothing here is shared with oracle/ (no import, no helper).
"""

import numpy as np
import torch

from workloads import bf16_bits_to_f64


def as_t(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = bf16_bits_to_f64(a)
    return torch.tensor(np.asarray(a, np.float64), dtype=torch.float64)


def selection(logits: np.ndarray, k: int) -> np.ndarray:
    T, E = logits.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -logits.astype(np.float64)), axis=-1)
    return order[:, :k]


def keep_mask(sel: np.ndarray, E: int, cap: int, eligible=None, score=None) -> tuple:
    """mask: selected; keep: selected, eligible and within the first `cap` eligible tokens
    of the expert in token order -- or, given `score` [T, E], within the `cap` eligible
    tokens of the expert with the largest score (ties: lower token first)."""
    T, k = sel.shape
    mask = np.zeros((T, E), np.int64)
    np.put_along_axis(mask, sel, 1, axis=-1)
    elig = mask if eligible is None else mask * eligible
    rank = np.cumsum(elig, axis=0) - 1
    keep = elig.copy()
    if cap > 0 and score is None:
        keep = elig * (rank < cap)
    elif cap > 0:
        for e in range(E):
            toks = np.flatnonzero(elig[:, e])
            if toks.size > cap:
                best = toks[np.lexsort((toks, -score[toks, e].astype(np.float64)))[:cap]]
                keep[:, e] = 0
                keep[best, e] = 1
    return mask, keep


def _round(t, rnd):
    if not rnd:
        return t
    return t.to(torch.bfloat16).to(torch.float64)


def swiglu(x, W1, W2, rnd=False):
    f = W1.shape[0] // 2
    a = _round(x @ W1[:f].T, rnd)
    b = _round(x @ W1[f:].T, rnd)
    h = _round(torch.nn.functional.silu(a) * b, rnd)
    return _round(h @ W2.T, rnd)


def dense_layer(cfg, inp: dict, rnd=False, requires_grad=False):
    """Returns (y, leaves) where leaves maps input names to leaf tensors."""
    lg_np = np.asarray(inp["logits"], np.float32)
    key = lg_np
    if getattr(cfg, "select_bias", None) is not None:
        key = (lg_np + np.asarray(cfg.select_bias, np.float32)[None, :]).astype(np.float32)
    sel = selection(key, cfg.k)
    eligible = (lg_np >= 0).astype(np.int64) if getattr(cfg, "drop_negative", False) else None
    score = lg_np if getattr(cfg, "drop_by_score", False) else None
    mask, keep = keep_mask(sel, cfg.E, cfg.capacity, eligible, score)
    leaves = {n: as_t(inp[n]) for n in ("x", "W1", "W2", "W1s", "W2s") if n in inp}
    leaves["logits"] = torch.tensor(lg_np.astype(np.float64))
    if requires_grad:
        for v in leaves.values():
            v.requires_grad_(True)
    lg = leaves["logits"]
    m = torch.tensor(mask, dtype=torch.float64)
    kp = torch.tensor(keep, dtype=torch.float64)
    if cfg.gate == "softmax":
        p = torch.softmax(lg, dim=-1) * m
        w = p / p.sum(-1, keepdim=True)
    else:
        s = torch.sigmoid(lg) * m
        w = cfg.route_scale * s / s.sum(-1, keepdim=True)
    x = leaves["x"]
    y = torch.zeros_like(x)
    for e in range(cfg.E):
        ye = swiglu(x, leaves["W1"][e], leaves["W2"][e], rnd)
        y = y + (w[:, e] * kp[:, e])[:, None] * ye
    if cfg.fs:
        y = y + swiglu(x, leaves["W1s"], leaves["W2s"], rnd)
    return _round(y, rnd), leaves


def dense_grads(cfg, inp: dict):
    y, leaves = dense_layer(cfg, inp, rnd=False, requires_grad=True)
    dy = as_t(inp["dy"])
    (y * dy).sum().backward()
    return y.detach(), {n: v.grad for n, v in leaves.items()}
