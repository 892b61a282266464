"""Composition of the oracle's C steps into the whole MoE layer (fwd and bwd).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every array here is float64
(bf16 inputs are widened exactly); `rnd=True` rounds to bf16 wherever the GPU path
stores a bf16 tensor, `rnd=False` keeps the exact double result.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from workloads import bf16_bits_to_f64

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

GATE = {"softmax": 0, "sigmoid": 1}


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (-O2, OpenMP) into oracle/_build/."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        os.makedirs(_LIB_DIR, exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.orc_threads.argtypes = []
        lib.orc_threads.restype = i32
        lib.orc_bf16.argtypes = [f64]
        lib.orc_bf16.restype = f64
        lib.orc_round_bf16_array.argtypes = [P, i64]
        lib.orc_route.argtypes = [i64, i32, i32, i32, f64, i64, P, P, i32, i32, P, P, P, P, P,
                                  P, P, P, P]
        lib.orc_route.restype = i64
        lib.orc_permute.argtypes = [i64, i32, P, P, P]
        lib.orc_ffn_fwd_rows.argtypes = [i64, i32, i32, P, P, P, i32, P, P, P]
        lib.orc_e4m3.argtypes = [f64]
        lib.orc_e4m3.restype = f64
        lib.orc_e4m3_code.argtypes = [f64]
        lib.orc_e4m3_code.restype = ctypes.c_uint8
        lib.orc_mx_quantize_rows.argtypes = [i64, i32, P, P, P, P]
        lib.orc_ffn_fwd_rows_mx.argtypes = [i64, i32, i32, P, P, P, P, P, P, P, P]
        lib.orc_ffn_bwd_rows_mx.argtypes = [i64, i32, i32, P, P, P, P, P, P, P, P]
        lib.orc_ffn_bwd_rows.argtypes = [i64, i32, i32, P, P, P, P, i32, P, P]
        lib.orc_ffn_wgrad_rows.argtypes = [i64, i32, i32, P, P, P, P, P, P]
        lib.orc_combine.argtypes = [i64, P, i32, i32, P, P, P, P, P, i32, P]
        lib.orc_combine_bwd.argtypes = [i64, P, i32, i32, i32, i32, f64, P, P, P, P, P, P, P,
                                        i32, P, P]
        lib.orc_unpermute_reduce.argtypes = [i64, P, i32, i32, P, P, P, P, i32, P]
        _lib = lib
    return _lib


def threads() -> int:
    """Threads the C oracle's parallel loops run on (OpenMP's current maximum)."""
    return int(_load().orc_threads())


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16(a) -> np.ndarray:
    """Round a float64 array to bf16 values (kept as float64)."""
    out = _c(a, np.float64).copy()
    _load().orc_round_bf16_array(_p(out), out.size)
    return out


def _f64(a) -> np.ndarray:
    """Widen bf16 bit patterns (uint16/int16) exactly; pass float arrays through."""
    a = np.asarray(a)
    if a.dtype in (np.uint16, np.int16):
        return bf16_bits_to_f64(a.view(np.uint16))
    return _c(a, np.float64)


# --------------------------------------------------------------------------- route
def route(cfg, logits: np.ndarray) -> dict:
    """Top-k selection, gate weights, histogram, capacity, scan and PFT side arrays."""
    lib = _load()
    T, E, k = cfg.T, cfg.E, cfg.k
    lg = _c(logits, np.float32)
    assert lg.shape == (T, E)
    r = {
        "topk_idx": np.empty((T, k), np.int32),
        "topk_w": np.empty((T, k), np.float64),
        "counts": np.empty(E, np.int32),
        "kept": np.empty(E, np.int32),
        "offsets": np.empty(E + 1, np.int32),
        "dest_row": np.empty((T, k), np.int32),
        "src_tok": np.empty(T * k, np.int32),
        "src_slot": np.empty(T * k, np.int32),
        "drop_mask": np.empty((T, k), np.uint8),
    }
    bias = getattr(cfg, "select_bias", None)
    bias_a = None if bias is None else _c(bias, np.float32)
    nan = lib.orc_route(T, E, k, GATE[cfg.gate], float(cfg.route_scale), int(cfg.capacity),
                        _p(lg), _p(bias_a), int(getattr(cfg, "drop_negative", False)),
                        int(getattr(cfg, "drop_by_score", False)), _p(r["topk_idx"]), _p(r["topk_w"]), _p(r["counts"]),
                        _p(r["kept"]), _p(r["offsets"]), _p(r["dest_row"]), _p(r["src_tok"]),
                        _p(r["src_slot"]), _p(r["drop_mask"]))
    r["nan_logits"] = int(nan)
    r["drops"] = int(r["drop_mask"].sum())
    return r


# --------------------------------------------------------------------------- steps
def ffn_fwd_rows(xr, W1e, W2e, rnd=True):
    lib = _load()
    xr, W1e, W2e = _f64(xr), _f64(W1e), _f64(W2e)
    n, d = xr.shape
    f = W1e.shape[0] // 2
    ab = np.empty((n, 2 * f)); h = np.empty((n, f)); yp = np.empty((n, d))
    if n:
        lib.orc_ffn_fwd_rows(n, d, f, _p(xr), _p(W1e), _p(W2e), int(rnd), _p(ab), _p(h), _p(yp))
    return ab, h, yp


def e4m3(v: float) -> float:
    """Round to the nearest FP8 E4M3 value (ties to even), saturating at +-448."""
    return float(_load().orc_e4m3(float(v)))


def e4m3_code(q: float) -> int:
    return int(_load().orc_e4m3_code(float(q)))


def mx_quantize_rows(v):
    """MXFP8 of each row of v [rows, cols] in blocks of 32: (E4M3 codes uint8 [rows, cols],
    E8M0 scale codes uint8 [rows, cols/32], dequantised float64 [rows, cols])."""
    v = _f64(v)
    rows, cols = v.shape
    assert cols % 32 == 0
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty((rows, cols // 32), np.uint8)
    deq = np.empty((rows, cols))
    if rows:
        _load().orc_mx_quantize_rows(rows, cols, _p(v), _p(codes), _p(scales), _p(deq))
    return codes, scales, deq


def mx_quantize_cols(v):
    """MXFP8 of each column of v [rows, cols] in blocks of 32 consecutive rows from row 0;
    a short last block is quantised as if zero-padded to 32 rows (zeros never raise the
    block maximum).  Returns the dequantised float64 [rows, cols]: the weight-gradient
    operands quantised along the tokens of one expert segment."""
    v = _f64(v)
    rows, cols = v.shape
    if rows == 0:
        return np.zeros((0, cols))
    rp = -(-rows // 32) * 32
    t = np.zeros((cols, rp))
    t[:, :rows] = v.T
    return np.ascontiguousarray(mx_quantize_rows(t)[2][:, :rows].T)


def ffn_wgrad_rows_mx(xr, h, dyp, dab, d, f):
    """The expert's weight gradients on MXFP8 operands quantised along its tokens:
    dW1 = Q(dab)^T Q(xr), dW2 = Q(dyp)^T Q(h), each Q in 32-row blocks from the segment's
    first row (mx_quantize_cols); float64 accumulation."""
    if xr is None or xr.shape[0] == 0:
        return np.zeros((2 * f, d)), np.zeros((d, f))
    return ffn_wgrad_rows(mx_quantize_cols(xr), mx_quantize_cols(h), mx_quantize_cols(dyp),
                          mx_quantize_cols(dab), d, f)


def ffn_fwd_rows_mx(xr, W1e, W2e):
    """The expert FFN forward on MXFP8 operands: (ab, h, yp, h codes, h scales)."""
    lib = _load()
    xr, W1e, W2e = _f64(xr), _f64(W1e), _f64(W2e)
    n, d = xr.shape
    f = W1e.shape[0] // 2
    ab = np.empty((n, 2 * f)); h = np.empty((n, f)); yp = np.empty((n, d))
    hc = np.empty((n, f), np.uint8); hs = np.empty((n, f // 32), np.uint8)
    if n:
        lib.orc_ffn_fwd_rows_mx(n, d, f, _p(xr), _p(W1e), _p(W2e), _p(ab), _p(h), _p(yp),
                                _p(hc), _p(hs))
    return ab, h, yp, hc, hs


def ffn_bwd_rows_mx(dyp, ab, W1e, W2e):
    """The expert FFN's data gradients on MXFP8 operands: (dab, dxp, dab codes, dab scales)."""
    lib = _load()
    dyp, ab, W1e, W2e = _f64(dyp), _f64(ab), _f64(W1e), _f64(W2e)
    n, d = dyp.shape
    f = W1e.shape[0] // 2
    dab = np.empty((n, 2 * f)); dxr = np.empty((n, d))
    dc = np.empty((n, 2 * f), np.uint8); ds = np.empty((n, 2 * f // 32), np.uint8)
    if n:
        lib.orc_ffn_bwd_rows_mx(n, d, f, _p(dyp), _p(ab), _p(W1e), _p(W2e), _p(dab), _p(dxr),
                                _p(dc), _p(ds))
    return dab, dxr, dc, ds


def ffn_bwd_rows(dyp, ab, W1e, W2e, rnd=True):
    lib = _load()
    dyp, ab, W1e, W2e = _f64(dyp), _f64(ab), _f64(W1e), _f64(W2e)
    n, d = dyp.shape
    f = W1e.shape[0] // 2
    dab = np.empty((n, 2 * f)); dxr = np.empty((n, d))
    if n:
        lib.orc_ffn_bwd_rows(n, d, f, _p(dyp), _p(ab), _p(W1e), _p(W2e), int(rnd), _p(dab),
                             _p(dxr))
    return dab, dxr


def ffn_bwd_rows_dispatch(dy_rows, w, ab, W1e, W2e):
    """The expert's data gradients when the dispatch of dy is fused into the FC2
    data-gradient (Primus MoE blog, MegaMoE section): each row's upstream gradient is its
    token's dy row times the slot's gate weight, taken exactly (w * dy in float64, with no
    bf16 rounding of the product), so dh = w (dy W2e); da, db and dxp then follow as in
    ffn_bwd_rows, rounded where the GPU path stores them."""
    g = _f64(dy_rows) * np.asarray(w, np.float64)[:, None]
    return ffn_bwd_rows(g, ab, W1e, W2e)


def ffn_wgrad_rows(xr, h, dyp, dab, d, f):
    lib = _load()
    dW1 = np.zeros((2 * f, d)); dW2 = np.zeros((d, f))
    n = 0 if xr is None else xr.shape[0]
    if n:
        lib.orc_ffn_wgrad_rows(n, d, f, _p(_f64(xr)), _p(_f64(h)), _p(_f64(dyp)), _p(_f64(dab)),
                               _p(dW1), _p(dW2))
    return dW1, dW2


def permute(cfg, r, x) -> np.ndarray:
    """xp[p] = x[src_tok[p]] for the rows the routing kept (a plain copy)."""
    n_rows = int(r["offsets"][-1])
    x = _f64(x)
    xp = np.empty((n_rows, cfg.d))
    _load().orc_permute(n_rows, cfg.d, _p(_c(r["src_tok"], np.int32)), _p(x), _p(xp))
    return xp


def combine(cfg, dest_row, topk_w, yp, ys=None, toks=None, yp_row_of=None, rnd=True):
    lib = _load()
    d, k = cfg.d, cfg.k
    toks_a = None if toks is None else _c(toks, np.int64)
    n_tok = cfg.T if toks is None else len(toks_a)
    y = np.empty((n_tok, d))
    lib.orc_combine(n_tok, _p(toks_a), k, d, _p(_c(dest_row, np.int32)), _p(_c(topk_w, np.float64)),
                    _p(_f64(yp)), _p(None if yp_row_of is None else _c(yp_row_of, np.int64)),
                    _p(None if ys is None else _f64(ys)), int(rnd), _p(y))
    return y


def combine_bwd(cfg, logits, r, dy, yp, toks=None, yp_row_of=None, n_rows=None, rnd=True):
    """Returns (dyp [n_rows, d], dlogits [n_tok, E]); dyp rows not touched stay 0."""
    lib = _load()
    d, k, E = cfg.d, cfg.k, cfg.E
    toks_a = None if toks is None else _c(toks, np.int64)
    n_tok = cfg.T if toks is None else len(toks_a)
    yp = _f64(yp)
    if n_rows is None:
        n_rows = yp.shape[0]
    dyp = np.zeros((n_rows, d))
    dl = np.empty((n_tok, E))
    lib.orc_combine_bwd(n_tok, _p(toks_a), E, k, d, GATE[cfg.gate], float(cfg.route_scale),
                        _p(_c(logits, np.float32)), _p(_c(r["topk_idx"], np.int32)),
                        _p(_c(r["topk_w"], np.float64)), _p(_c(r["dest_row"], np.int32)),
                        _p(_f64(dy)), _p(yp),
                        _p(None if yp_row_of is None else _c(yp_row_of, np.int64)), int(rnd),
                        _p(dyp), _p(dl))
    return dyp, dl


def unpermute_reduce(cfg, dest_row, dxp, dxs=None, toks=None, row_of=None, rnd=True):
    lib = _load()
    d, k = cfg.d, cfg.k
    toks_a = None if toks is None else _c(toks, np.int64)
    n_tok = cfg.T if toks is None else len(toks_a)
    dx = np.empty((n_tok, d))
    lib.orc_unpermute_reduce(n_tok, _p(toks_a), k, d, _p(_c(dest_row, np.int32)), _p(_f64(dxp)),
                             _p(None if row_of is None else _c(row_of, np.int64)),
                             _p(None if dxs is None else _f64(dxs)), int(rnd), _p(dx))
    return dx


# --------------------------------------------------------------------------- full layer
def layer_fwd(cfg, inp: dict, rnd: bool = True, r: dict | None = None, mx: bool = False) -> dict:
    """Whole forward on the host, every token and every expert.

    inp holds logits (f32 [T,E]) and x, W1, W2 (+ W1s, W2s) as bf16 bits or float64.
    mx: the routed experts' GEMMs on MXFP8 operands (ffn_fwd_rows_mx); the shared expert
    stays bf16 (the MXFP8 recipe covers the routed-expert grouped GEMMs)."""
    if r is None:
        r = route(cfg, inp["logits"])
    x = _f64(inp["x"])
    W1 = _f64(inp["W1"]); W2 = _f64(inp["W2"])
    off = r["offsets"]
    n_rows = int(off[-1])
    xp = np.empty((n_rows, cfg.d))
    _load().orc_permute(n_rows, cfg.d, _p(r["src_tok"]), _p(x), _p(xp))
    ab = np.empty((n_rows, 2 * cfg.f)); h = np.empty((n_rows, cfg.f)); yp = np.empty((n_rows, cfg.d))
    hq = np.zeros((n_rows, cfg.f), np.uint8) if mx else None
    hs = np.zeros((n_rows, cfg.f // 32), np.uint8) if mx else None
    for e in range(cfg.E):
        s, t = int(off[e]), int(off[e + 1])
        if mx:
            ab[s:t], h[s:t], yp[s:t], hq[s:t], hs[s:t] = ffn_fwd_rows_mx(xp[s:t], W1[e], W2[e])
        else:
            ab[s:t], h[s:t], yp[s:t] = ffn_fwd_rows(xp[s:t], W1[e], W2[e], rnd)
    out = dict(route=r, xp=xp, ab=ab, h=h, yp=yp)
    if mx:
        out["hq"], out["h_sf"] = hq, hs
    ys = None
    if cfg.fs:
        out["ab_s"], out["h_s"], ys = ffn_fwd_rows(x, inp["W1s"], inp["W2s"], rnd)
        out["ys"] = ys
    out["y"] = combine(cfg, r["dest_row"], r["topk_w"], yp, ys, rnd=rnd)
    return out


def layer_bwd(cfg, inp: dict, fwd: dict, rnd: bool = True, mx: bool = False,
              mx_wgrad: bool = False) -> dict:
    """Whole backward on the host given the forward's saved tensors and inp['dy'].
    mx: the routed experts' data-gradient GEMMs on MXFP8 operands (ffn_bwd_rows_mx);
    mx_wgrad: their weight gradients too, on operands quantised along each segment's tokens
    (ffn_wgrad_rows_mx).  The shared expert stays bf16."""
    r = fwd["route"]
    off = r["offsets"]
    x = _f64(inp["x"]); dy = _f64(inp["dy"])
    W1 = _f64(inp["W1"]); W2 = _f64(inp["W2"])
    dyp, dlogits = combine_bwd(cfg, inp["logits"], r, dy, fwd["yp"], rnd=rnd)
    n_rows = int(off[-1])
    dab = np.empty((n_rows, 2 * cfg.f)); dxp = np.empty((n_rows, cfg.d))
    dW1 = np.zeros((cfg.E, 2 * cfg.f, cfg.d)); dW2 = np.zeros((cfg.E, cfg.d, cfg.f))
    for e in range(cfg.E):
        s, t = int(off[e]), int(off[e + 1])
        if mx:
            dab[s:t], dxp[s:t], _, _ = ffn_bwd_rows_mx(dyp[s:t], fwd["ab"][s:t], W1[e], W2[e])
        else:
            dab[s:t], dxp[s:t] = ffn_bwd_rows(dyp[s:t], fwd["ab"][s:t], W1[e], W2[e], rnd)
        wg = ffn_wgrad_rows_mx if mx_wgrad else ffn_wgrad_rows
        dW1[e], dW2[e] = wg(fwd["xp"][s:t], fwd["h"][s:t], dyp[s:t], dab[s:t], cfg.d, cfg.f)
    out = dict(dyp=dyp, dlogits=dlogits, dab=dab, dxp=dxp)
    dxs = None
    if cfg.fs:
        dab_s, dxs = ffn_bwd_rows(dy, fwd["ab_s"], inp["W1s"], inp["W2s"], rnd)
        dW1s, dW2s = ffn_wgrad_rows(x, fwd["h_s"], dy, dab_s, cfg.d, cfg.fs)
        out.update(dab_s=dab_s, dx_s=dxs, dW1s=bf16(dW1s) if rnd else dW1s,
                   dW2s=bf16(dW2s) if rnd else dW2s)
    out["dx"] = unpermute_reduce(cfg, r["dest_row"], dxp, dxs, rnd=rnd)
    out["dW1"] = bf16(dW1) if rnd else dW1
    out["dW2"] = bf16(dW2) if rnd else dW2
    return out


# --------------------------------------------------------------------------- sampled layer
class HostSource:
    """Input access for the sampled evaluation when the inputs live in host arrays."""

    def __init__(self, inp: dict):
        self.inp = inp
        self.logits = np.asarray(inp["logits"], np.float32)

    def rows(self, name, idx):
        return _f64(np.asarray(self.inp[name])[np.asarray(idx, np.int64)])

    def expert(self, name, e):
        return _f64(np.asarray(self.inp[name])[e])

    def whole(self, name):
        return _f64(self.inp[name])


class TorchSource:
    """Input access when the inputs are torch tensors (host copies of slices only).

    The tensors are the seeded synthetic inputs, never results of the GPU path."""

    def __init__(self, inp: dict):
        self.inp = inp
        self.logits = inp["logits"].detach().cpu().numpy().astype(np.float32)

    @staticmethod
    def _np(t):
        import torch
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            return bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
        return t.double().numpy()

    def rows(self, name, idx):
        import torch
        return self._np(self.inp[name][torch.as_tensor(np.asarray(idx, np.int64)).to(
            self.inp[name].device)])

    def expert(self, name, e):
        return self._np(self.inp[name][e])

    def whole(self, name):
        return self._np(self.inp[name])


def layer_sampled(cfg, src, tokens, experts=(), wcols=None, wrows=None, rnd=True,
                  mx: bool = False, mx_bwd: bool = False, mx_wgrad: bool = False) -> dict:
    """The exact layer restricted to a subset of outputs (for configurations too big
    to evaluate in full on the host):

      y, dx, dlogits         for the tokens in `tokens`;
      dW1, dW2 entries       for experts in `experts`, f-columns `wcols` and
                             d-rows `wrows`:  dW2[e][wrows][:, wcols],
                             dW1[e][wcols][:, wrows] (gate) and dW1[e][f+wcols][:, wrows] (up);
      dW1s, dW2s entries     likewise for the shared expert, if any.

    Every value is computed from the inputs alone through the same steps as the full
    layer; only the rows/columns that the requested outputs depend on are evaluated.
    mx: the routed experts' forward on MXFP8 operands (as layer_fwd(mx=True)); mx_bwd:
    their data-gradient GEMMs too (as layer_bwd(mx=True)); mx_wgrad: their weight
    gradients too (as layer_bwd(mx_wgrad=True)).  The restriction stays exact because
    every MX block lies inside one token row, one row of a weight (or of its transpose), or
    one column of an expert segment's rows."""
    r = route(cfg, src.logits)
    k, d, f = cfg.k, cfg.d, cfg.f
    toks = np.unique(np.asarray(tokens, np.int64))
    dest = r["dest_row"]
    rows = np.unique(dest[toks].reshape(-1))
    rows = rows[rows >= 0]
    row_of = np.full(cfg.T * k, -1, np.int64)
    row_of[rows] = np.arange(len(rows))
    n = len(rows)
    yp = np.empty((n, d)); dxp = np.empty((n, d))
    xp = src.rows("x", r["src_tok"][rows])
    # dyp rows straight from their definition w * dy[t] (the same values combine_bwd writes)
    slots = r["src_slot"][rows]
    dyp = src.rows("dy", slots // k) * r["topk_w"].reshape(-1)[slots][:, None]
    if rnd:
        dyp = bf16(dyp)
    off = r["offsets"]
    eid = np.searchsorted(off, rows, side="right") - 1   # expert of each row
    for e in np.unique(eid):           # each expert's weights are fetched once
        sel = np.nonzero(eid == e)[0]
        W1e, W2e = src.expert("W1", int(e)), src.expert("W2", int(e))
        if mx:
            ab, _, yp[sel], _, _ = ffn_fwd_rows_mx(xp[sel], W1e, W2e)
        else:
            ab, _, yp[sel] = ffn_fwd_rows(xp[sel], W1e, W2e, rnd)
        if mx_bwd:
            _, dxp[sel], _, _ = ffn_bwd_rows_mx(dyp[sel], ab, W1e, W2e)
        else:
            _, dxp[sel] = ffn_bwd_rows(dyp[sel], ab, W1e, W2e, rnd)
        del W1e, W2e
    out = {"route": r, "tokens": toks}
    ys = dxs = None
    x_t = src.rows("x", toks)
    dy_t = src.rows("dy", toks)
    if cfg.fs:
        W1s, W2s = src.whole("W1s"), src.whole("W2s")
        ab_s, h_s, ys = ffn_fwd_rows(x_t, W1s, W2s, rnd)
        _, dxs = ffn_bwd_rows(dy_t, ab_s, W1s, W2s, rnd)
    out["y"] = combine(cfg, dest, r["topk_w"], yp, ys, toks=toks, yp_row_of=row_of, rnd=rnd)
    _, dl = combine_bwd(cfg, src.logits, r, dy_t, yp, toks=toks, yp_row_of=row_of, rnd=rnd)
    out["dlogits"] = dl
    out["dx"] = unpermute_reduce(cfg, dest, dxp, dxs, toks=toks, row_of=row_of, rnd=rnd)

    # weight-gradient entries of whole experts (every row of the expert contributes)
    if len(experts):
        wcols = np.asarray(wcols, np.int64)
        wrows = np.asarray(wrows, np.int64)
        dW1 = {}; dW2 = {}
        W1cols = np.concatenate([wcols, f + wcols])
        for e in experts:
            e = int(e)
            s, t = int(off[e]), int(off[e + 1])
            W1e = src.expert("W1", e); W2e = src.expert("W2", e)
            slots = r["src_slot"][s:t]
            tk = slots // k
            xr = src.rows("x", tk)
            w = r["topk_w"].reshape(-1)[slots]
            dyp_e = src.rows("dy", tk) * w[:, None]
            if rnd:
                dyp_e = bf16(dyp_e)
            g1, g2 = _wgrad_cols(xr, dyp_e, W1e, W2e, wcols, wrows, rnd, mx=mx, mx_bwd=mx_bwd,
                                 mx_wgrad=mx_wgrad)
            dW1[e] = g1; dW2[e] = g2
        out["dW1"] = dW1; out["dW2"] = dW2
        out["wcols"] = wcols; out["wrows"] = wrows
        if cfg.fs:
            xs = src.whole("x"); dys = src.whole("dy")
            out["dW1s"], out["dW2s"] = _wgrad_cols(xs, dys, src.whole("W1s"), src.whole("W2s"),
                                                   wcols, wrows, rnd)
    return out


def _wgrad_cols(xr, dyp, W1e, W2e, cols, drows, rnd, mx=False, mx_bwd=False, mx_wgrad=False):
    """dW2[drows][:, cols] and dW1[[cols, f+cols]][:, drows] of one expert from all its rows,
    evaluating only the FFN columns `cols` (exact: a, b, h, dh, da, db of column c depend
    on column c alone).  Uses the oracle's row steps on the column-restricted weights.
    mx: a and b from MXFP8 operands (x rows and W1 rows are whole MX rows), h from them."""
    f = W1e.shape[0] // 2
    W1c = np.concatenate([W1e[cols], W1e[f + cols]])       # [2m, d]  (gate cols, up cols)
    W2c = np.ascontiguousarray(W2e[:, cols])                # [d, m]
    if mx:
        m = len(cols)
        ab = bf16(mx_quantize_rows(xr)[2] @ mx_quantize_rows(W1c)[2].T)
        a, b = ab[:, :m], ab[:, m:]
        h = bf16(a / (1.0 + np.exp(-a)) * b)
    else:
        ab, h, _ = ffn_fwd_rows(xr, W1c, W2c, rnd)          # ab = [a_cols | b_cols]
    if mx_bwd:
        # dh from MXFP8 dyp (along d) and W2^T rows of these columns (along d), then the
        # SwiGLU backward; only dab (bf16) enters the weight gradients
        dh = mx_quantize_rows(dyp)[2] @ mx_quantize_rows(np.ascontiguousarray(W2c.T))[2].T
        a, b = ab[:, :len(cols)], ab[:, len(cols):]
        sg = 1.0 / (1.0 + np.exp(-a))
        dab = np.concatenate([bf16(dh * b * (sg * (1.0 + a * (1.0 - sg)))),
                              bf16(dh * (a * sg))], axis=1)
    else:
        dab, _ = ffn_bwd_rows(dyp, ab, W1c, W2c, rnd)       # [da_cols | db_cols]
    m = len(cols)
    if mx_wgrad:   # operands quantised per column along the segment's rows
        dW2 = mx_quantize_cols(dyp[:, drows]).T @ mx_quantize_cols(h)
        dW1 = mx_quantize_cols(dab).T @ mx_quantize_cols(xr[:, drows])
    else:
        dW2 = (dyp[:, drows].T @ h)                          # [len(drows), m]
        dW1 = (dab.T @ xr[:, drows])                         # [2m, len(drows)]
    if rnd:
        dW2 = bf16(dW2); dW1 = bf16(dW1)
    return dW1.reshape(2, m, len(drows)), dW2
