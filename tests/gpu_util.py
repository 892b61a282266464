"""Helpers for the GPU parity tests: device copies of the seeded inputs, conversion of
results to float64, and the tolerance checks.

Tolerance (bf16 outputs and gradients with fp32 accumulation, compared against the
oracle's float64 result with the same bf16 rounding points):
    rel-L2 = ||g - o||_2 / ||o||_2                  <= 1e-2
    max_i |g_i - o_i| / (rms(o) + |o_i|)            <= 2e-2
The second form is the max-abs bound of 2e-2 taken on the tensor's own scale; dividing
by rms(o) + |o_i| keeps a one-ulp bf16 rounding difference on a large element (which
any correct bf16 kernel may show) inside the bound while still bounding the error of
every small element by 2e-2 * rms.

Every comparison also records, for the report printed at the end of the run
(tests/conftest.py): the raw max |g - o|, max |g - o| / rms(o) (the max-abs bound read on
the tensor's RMS alone), and how many elements differ from the oracle by more than one
bf16 ulp of the oracle's value (ulp(o) = 2^(floor(log2 |o|) - 7), 2^-133 at zero).
"""

import numpy as np
import torch

import token_dispatch_expert_gb300 as tde
from workloads import bf16_bits_to_f64

REL_L2_TOL = 1e-2
MAX_TOL = 2e-2


def cfg_c(c):
    bias = None
    if getattr(c, "select_bias", None) is not None:
        bias = torch.tensor(np.asarray(c.select_bias, np.float32), device="cuda")
    return tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs, c.gate, c.route_scale, c.capacity,
                           select_bias=bias, drop_negative=getattr(c, "drop_negative", False),
                           recompute=getattr(c, "recompute", False),
                           drop_by_score=getattr(c, "drop_by_score", False))


def dev(a, device="cuda"):
    """numpy -> torch on the device; uint16 bf16 bit patterns become bfloat16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        if t.dtype == np.uint16:
            return bf16_bits_to_f64(t)
        return t.astype(np.float64)
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def np_i(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_ulp(o) -> np.ndarray:
    """One bf16 unit in the last place at each value of o (8 significant bits): 2^(e - 7)
    for 2^e <= |o| < 2^(e+1), floored at the smallest bf16 subnormal 2^-133."""
    o = np.abs(np.asarray(o, np.float64))
    _, ex = np.frexp(o)                      # o = m * 2^ex, m in [0.5, 1)
    return np.where(o < 2.0 ** -126, 2.0 ** -133, np.ldexp(1.0, ex - 8))


def stats(g, o):
    g = np.asarray(g, np.float64); o = np.asarray(o, np.float64)
    if not o.size:
        return {"rel_l2": 0.0, "max_scaled": 0.0, "max_abs": 0.0, "max_over_rms": 0.0,
                "n_gt_1ulp": 0, "n": 0}
    diff = np.abs(g - o)
    nrm = np.linalg.norm(o)
    rel = float(np.linalg.norm(g - o) / nrm) if nrm > 0 else float(np.linalg.norm(g - o))
    rms = float(np.sqrt(np.mean(o * o)))
    mx = float((diff / (rms + np.abs(o) + 1e-30)).max())
    return {"rel_l2": rel, "max_scaled": mx, "max_abs": float(diff.max()),
            "max_over_rms": float(diff.max() / rms) if rms > 0 else float(diff.max()),
            "n_gt_1ulp": int((diff > bf16_ulp(o)).sum()), "n": int(o.size)}


# (test id, tensor name, stats) of every comparison in this process, for the end-of-run
# report; the test id is set by an autouse fixture in conftest.py
RECORDS = []
CURRENT_TEST = ["?"]


def record(name, s):
    RECORDS.append((CURRENT_TEST[0], name, s))


def assert_close(name, g, o, rel_tol=REL_L2_TOL, max_tol=MAX_TOL):
    s = stats(g, o)
    record(name, s)
    assert np.isfinite(np.asarray(g, np.float64)).all(), f"{name}: non-finite values"
    assert s["rel_l2"] <= rel_tol and s["max_scaled"] <= max_tol, f"{name}: {s}"
    return s


def alloc_route(c, device="cuda"):
    T, E, k = c.T, c.E, c.k
    i32 = dict(dtype=torch.int32, device=device)
    return {
        "topk_idx": torch.empty((T, k), **i32),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device=device),
        "counts": torch.empty(E, **i32), "kept": torch.empty(E, **i32),
        "offsets": torch.empty(E + 1, **i32), "dest_row": torch.empty((T, k), **i32),
        "src_tok": torch.empty(T * k, **i32), "src_slot": torch.empty(T * k, **i32),
        "drop_mask": torch.empty((T, k), dtype=torch.uint8, device=device),
    }


def new_ws(cfg, device="cuda"):
    ws_b, _ = tde.moe_workspace_size(cfg)
    ws = torch.empty(ws_b, dtype=torch.uint8, device=device)
    tde.moe_ws_init(ws)
    return ws


def run_route(c, logits_dev, ws=None):
    cfg = cfg_c(c)
    if ws is None:
        ws = new_ws(cfg)
    r = alloc_route(c)
    tde.moe_route(cfg, logits_dev, r["topk_idx"], r["topk_w"], r["counts"], r["kept"],
                  r["offsets"], r["dest_row"], r["src_tok"], r["src_slot"], r["drop_mask"], ws)
    return r, ws
