"""GB300-native single-GPU Mixture-of-Experts layer.

Python binding of the C ABI in include/moe.h: every function here has the name of the
C entry point it calls and only marshals arguments (torch tensors -> device pointers,
the current CUDA stream -> cudaStream_t).  Every step of the layer runs in the CUDA
kernels of libmoe_gb300.so; there is no Python or CPU fallback -- if the library is
missing, every call raises.

PyTorch is used for device memory and streams only.
"""

from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH, build  # noqa: F401

__all__ = [
    "MoEConfigC", "MoEError", "make_config", "lib",
    "moe_capacity_from_factor", "moe_workspace_size", "moe_ctx_offsets", "moe_ws_init",
    "moe_route", "moe_route_noalloc", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_combine_bwd",
    "moe_grouped_ffn_bwd", "moe_unpermute_reduce", "moe_layer_fwd", "moe_layer_bwd",
    "moe_grouped_ffn_gather", "moe_grouped_ffn_bwd_gather", "moe_grouped_ffn_bwd_dispatch",
    "moe_mx_weights_size", "moe_mx_quantize_weights", "moe_mx_act_scales_size",
    "moe_mx_permute_quant", "moe_grouped_ffn_mx", "moe_grouped_ffn_bwd_mx", "moe_layer_fwd_mx",
    "moe_layer_bwd_mx",
    "moe_status", "moe_status_string", "moe_selftest_wait_timeout", "moe_gemm_clock_trace",
    "moe_gemm_clock_read", "ctx_views", "MoELayer", "CTX_FIELDS",
]

GATES = {"softmax": 0, "sigmoid": 1}
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_DEVICE_FLAG", 5: "MOE_ERR_TIMEOUT"}
DEVERR = {"NAN_LOGIT": 0x1, "BAD_INDEX": 0x2, "TIMEOUT": 0x4, "BAD_OFFSETS": 0x8}
CTX_FIELDS = ["topk_idx", "topk_w", "counts", "kept", "offsets", "dest_row", "src_tok",
              "src_slot", "drop_mask", "xp", "ab", "h", "yp", "ab_s", "h_s", "ys"]


class MoEConfigC(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("ffn", ctypes.c_int32), ("ffn_shared", ctypes.c_int32),
                ("gate", ctypes.c_int32), ("route_scale", ctypes.c_float),
                ("capacity", ctypes.c_int32), ("select_bias", ctypes.c_void_p),
                ("drop_negative", ctypes.c_int32), ("recompute", ctypes.c_int32),
                ("drop_by_score", ctypes.c_int32), ("mxfp8", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(token_dispatch_expert_gb300.build() or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        cfgp = ctypes.POINTER(MoEConfigC)
        sig = {
            "moe_capacity_from_factor": ([I64, I32, I32, ctypes.c_double], I32),
            "moe_workspace_size": ([cfgp, ctypes.POINTER(ctypes.c_size_t),
                                    ctypes.POINTER(ctypes.c_size_t)], I32),
            "moe_ctx_offsets": ([cfgp, ctypes.POINTER(ctypes.c_size_t)], I32),
            "moe_ws_init": ([P, P], I32),
            "moe_route": ([cfgp] + [P] * 12, I32),
            "moe_route_noalloc": ([cfgp] + [P] * 12, I32),
            "moe_permute": ([cfgp] + [P] * 6, I32),
            "moe_grouped_ffn": ([cfgp] + [P] * 9, I32),
            "moe_grouped_ffn_gather": ([cfgp] + [P] * 10, I32),
            "moe_grouped_ffn_bwd_gather": ([cfgp] + [P] * 14, I32),
            "moe_grouped_ffn_bwd_dispatch": ([cfgp] + [P] * 17, I32),
            "moe_combine": ([cfgp] + [P] * 7, I32),
            "moe_combine_bwd": ([cfgp] + [P] * 10, I32),
            "moe_grouped_ffn_bwd": ([cfgp] + [P] * 13, I32),
            "moe_unpermute_reduce": ([cfgp] + [P] * 6, I32),
            "moe_layer_fwd": ([cfgp] + [P] * 10, I32),
            "moe_mx_weights_size": ([cfgp, ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_size_t)], I32),
            "moe_mx_quantize_weights": ([cfgp] + [P] * 4, I32),
            "moe_mx_act_scales_size": ([cfgp, I32, ctypes.POINTER(ctypes.c_size_t)], I32),
            "moe_mx_permute_quant": ([cfgp] + [P] * 8, I32),
            "moe_grouped_ffn_mx": ([cfgp] + [P] * 11, I32),
            "moe_layer_fwd_mx": ([cfgp] + [P] * 9, I32),
            "moe_grouped_ffn_bwd_mx": ([cfgp] + [P] * 12, I32),
            "moe_layer_bwd_mx": ([cfgp] + [P] * 15, I32),
            "moe_layer_bwd": ([cfgp] + [P] * 16, I32),
            "moe_status": ([P, P, ctypes.POINTER(ctypes.c_int32)], I32),
            "moe_gemm_clock_trace": ([I32], I32),
            "moe_gemm_clock_read": ([ctypes.POINTER(ctypes.c_uint64)] * 3, I32),
            "moe_selftest_wait_timeout": ([P, I64, P], I32),
            "moe_status_string": ([I32], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def make_config(T, d, E, k, ffn, ffn_shared=0, gate="softmax", route_scale=1.0,
                capacity=0, select_bias=None, drop_negative=False,
                recompute=False, drop_by_score=False, mxfp8=False) -> MoEConfigC:
    """select_bias: a float32 device tensor [E] (kept alive by the returned config) or None.
    mxfp8: 0 / False (bf16), 1 / True (routed forward and data gradients in MXFP8) or 2 (and
    the weight gradients)."""
    cfg = MoEConfigC(int(T), int(d), int(E), int(k), int(ffn), int(ffn_shared),
                     GATES[gate] if isinstance(gate, str) else int(gate), float(route_scale),
                     int(capacity), _p(select_bias), int(bool(drop_negative)),
                     int(bool(recompute)), int(bool(drop_by_score)), int(mxfp8))
    cfg._keep = select_bias
    return cfg


def _p(t):
    """Device pointer of a tensor (or an int address); None -> NULL.  The C calls take
    dense row-major device buffers: a host tensor or a strided view is refused here rather
    than handed to a kernel as a pointer."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got strides {tuple(t.stride())}")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != 0:
        raise MoEError(status, where)


def _cfg(cfg):
    return ctypes.byref(cfg)


# --------------------------------------------------------------------------- host helpers
def moe_capacity_from_factor(T, k, E, c) -> int:
    return lib().moe_capacity_from_factor(int(T), int(k), int(E), float(c))


def moe_workspace_size(cfg):
    ws, ctx = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(_cfg(cfg), ctypes.byref(ws), ctypes.byref(ctx)),
           "moe_workspace_size")
    return ws.value, ctx.value


def moe_ctx_offsets(cfg):
    arr = (ctypes.c_size_t * len(CTX_FIELDS))()
    _check(lib().moe_ctx_offsets(_cfg(cfg), arr), "moe_ctx_offsets")
    return list(arr)


def moe_status_string(s) -> str:
    return lib().moe_status_string(int(s)).decode()


# --------------------------------------------------------------------------- device calls
def moe_ws_init(ws, stream=None):
    _check(lib().moe_ws_init(_p(ws), _s(stream)), "moe_ws_init")


def moe_route(cfg, logits, topk_idx, topk_w, counts, kept, offsets, dest_row, src_tok, src_slot,
              drop_mask, ws, stream=None):
    _check(lib().moe_route(_cfg(cfg), _p(logits), _p(topk_idx), _p(topk_w), _p(counts), _p(kept),
                           _p(offsets), _p(dest_row), _p(src_tok), _p(src_slot), _p(drop_mask),
                           _p(ws), _s(stream)), "moe_route")


def moe_route_noalloc(cfg, logits, topk_idx, topk_w, counts, kept, offsets, dest_row, src_tok,
                      src_slot, drop_mask, dev_flags=None, stream=None):
    """moe_route without a workspace, for callers that cannot allocate device memory
    (see include/moe.h); dev_flags is an optional device int32 for the error bits."""
    _check(lib().moe_route_noalloc(_cfg(cfg), _p(logits), _p(topk_idx), _p(topk_w), _p(counts),
                                   _p(kept), _p(offsets), _p(dest_row), _p(src_tok),
                                   _p(src_slot), _p(drop_mask), _p(dev_flags), _s(stream)),
           "moe_route_noalloc")


def moe_permute(cfg, x, src_tok, offsets, xp, ws, stream=None):
    _check(lib().moe_permute(_cfg(cfg), _p(x), _p(src_tok), _p(offsets), _p(xp), _p(ws),
                             _s(stream)), "moe_permute")


def moe_grouped_ffn(cfg, xp, offsets, W1, W2, ab, h, yp, ws, stream=None):
    _check(lib().moe_grouped_ffn(_cfg(cfg), _p(xp), _p(offsets), _p(W1), _p(W2), _p(ab), _p(h),
                                 _p(yp), _p(ws), _s(stream)), "moe_grouped_ffn")


def moe_combine(cfg, yp, dest_row, topk_w, ys, y, ws, stream=None):
    _check(lib().moe_combine(_cfg(cfg), _p(yp), _p(dest_row), _p(topk_w), _p(ys), _p(y), _p(ws),
                             _s(stream)), "moe_combine")


def moe_combine_bwd(cfg, dy, yp, logits, topk_idx, topk_w, dest_row, dyp, dlogits, ws,
                    stream=None):
    _check(lib().moe_combine_bwd(_cfg(cfg), _p(dy), _p(yp), _p(logits), _p(topk_idx), _p(topk_w),
                                 _p(dest_row), _p(dyp), _p(dlogits), _p(ws), _s(stream)),
           "moe_combine_bwd")


def moe_grouped_ffn_gather(cfg, x, src_tok, offsets, W1, W2, ab, h, yp, ws, stream=None):
    _check(lib().moe_grouped_ffn_gather(_cfg(cfg), _p(x), _p(src_tok), _p(offsets), _p(W1),
                                        _p(W2), _p(ab), _p(h), _p(yp), _p(ws), _s(stream)),
           "moe_grouped_ffn_gather")


def moe_grouped_ffn_bwd_gather(cfg, dyp, x, src_tok, offsets, W1, W2, ab, h, dab, dxp, dW1, dW2,
                               ws, stream=None):
    _check(lib().moe_grouped_ffn_bwd_gather(_cfg(cfg), _p(dyp), _p(x), _p(src_tok), _p(offsets),
                                            _p(W1), _p(W2), _p(ab), _p(h), _p(dab), _p(dxp),
                                            _p(dW1), _p(dW2), _p(ws), _s(stream)),
           "moe_grouped_ffn_bwd_gather")


def moe_grouped_ffn_bwd_dispatch(cfg, dy, topk_w, src_tok, src_slot, dyp, xp, offsets, W1, W2,
                                 ab, h, dab, dxp, dW1, dW2, ws, stream=None):
    """moe_grouped_ffn_bwd with the FC2 data-gradient reading dy through src_tok and scaling
    by the slot's gate weight (see include/moe.h)."""
    _check(lib().moe_grouped_ffn_bwd_dispatch(_cfg(cfg), _p(dy), _p(topk_w), _p(src_tok),
                                              _p(src_slot), _p(dyp), _p(xp), _p(offsets),
                                              _p(W1), _p(W2), _p(ab), _p(h), _p(dab), _p(dxp),
                                              _p(dW1), _p(dW2), _p(ws), _s(stream)),
           "moe_grouped_ffn_bwd_dispatch")


def moe_mx_weights_size(cfg):
    """(bytes, offsets of the MXFP8 blob's parts: W1 codes, W1 scales, W2 codes, W2 scales,
    W2^T codes, W2^T scales, W1^T codes, W1^T scales)."""
    b = ctypes.c_size_t(0)
    offs = (ctypes.c_size_t * 8)()
    _check(lib().moe_mx_weights_size(_cfg(cfg), ctypes.byref(b), offs), "moe_mx_weights_size")
    return b.value, [o for o in offs]


def moe_mx_act_scales_size(cfg, K) -> int:
    b = ctypes.c_size_t(0)
    _check(lib().moe_mx_act_scales_size(_cfg(cfg), int(K), ctypes.byref(b)),
           "moe_mx_act_scales_size")
    return b.value


def moe_mx_quantize_weights(cfg, W1, W2, wq, stream=None):
    _check(lib().moe_mx_quantize_weights(_cfg(cfg), _p(W1), _p(W2), _p(wq), _s(stream)),
           "moe_mx_quantize_weights")


def moe_mx_permute_quant(cfg, x, src_tok, offsets, xp, xq, x_sf, ws, stream=None):
    _check(lib().moe_mx_permute_quant(_cfg(cfg), _p(x), _p(src_tok), _p(offsets), _p(xp),
                                      _p(xq), _p(x_sf), _p(ws), _s(stream)),
           "moe_mx_permute_quant")


def moe_grouped_ffn_mx(cfg, xq, x_sf, offsets, wq, ab, h, hq, h_sf, yp, ws, stream=None):
    _check(lib().moe_grouped_ffn_mx(_cfg(cfg), _p(xq), _p(x_sf), _p(offsets), _p(wq), _p(ab),
                                    _p(h), _p(hq), _p(h_sf), _p(yp), _p(ws), _s(stream)),
           "moe_grouped_ffn_mx")


def moe_layer_fwd_mx(cfg, logits, x, wq, W1s, W2s, y, ctx, ws, stream=None):
    _check(lib().moe_layer_fwd_mx(_cfg(cfg), _p(logits), _p(x), _p(wq), _p(W1s), _p(W2s), _p(y),
                                  _p(ctx), _p(ws), _s(stream)), "moe_layer_fwd_mx")


def moe_grouped_ffn_bwd_mx(cfg, dyp, xp, offsets, wq, ab, h, dab, dxp, dW1, dW2, ws,
                           stream=None):
    _check(lib().moe_grouped_ffn_bwd_mx(_cfg(cfg), _p(dyp), _p(xp), _p(offsets), _p(wq), _p(ab),
                                        _p(h), _p(dab), _p(dxp), _p(dW1), _p(dW2), _p(ws),
                                        _s(stream)), "moe_grouped_ffn_bwd_mx")


def moe_layer_bwd_mx(cfg, ctx, logits, x, dy, wq, W1s, W2s, dx, dW1, dW2, dW1s, dW2s, dlogits,
                     ws, stream=None):
    _check(lib().moe_layer_bwd_mx(_cfg(cfg), _p(ctx), _p(logits), _p(x), _p(dy), _p(wq),
                                  _p(W1s), _p(W2s), _p(dx), _p(dW1), _p(dW2), _p(dW1s), _p(dW2s),
                                  _p(dlogits), _p(ws), _s(stream)), "moe_layer_bwd_mx")


def moe_grouped_ffn_bwd(cfg, dyp, xp, offsets, W1, W2, ab, h, dab, dxp, dW1, dW2, ws,
                        stream=None):
    _check(lib().moe_grouped_ffn_bwd(_cfg(cfg), _p(dyp), _p(xp), _p(offsets), _p(W1), _p(W2),
                                     _p(ab), _p(h), _p(dab), _p(dxp), _p(dW1), _p(dW2), _p(ws),
                                     _s(stream)), "moe_grouped_ffn_bwd")


def moe_unpermute_reduce(cfg, dxp, dest_row, dxs, dx, ws, stream=None):
    _check(lib().moe_unpermute_reduce(_cfg(cfg), _p(dxp), _p(dest_row), _p(dxs), _p(dx), _p(ws),
                                      _s(stream)), "moe_unpermute_reduce")


def moe_layer_fwd(cfg, logits, x, W1, W2, W1s, W2s, y, ctx, ws, stream=None):
    _check(lib().moe_layer_fwd(_cfg(cfg), _p(logits), _p(x), _p(W1), _p(W2), _p(W1s), _p(W2s),
                               _p(y), _p(ctx), _p(ws), _s(stream)), "moe_layer_fwd")


def moe_layer_bwd(cfg, ctx, logits, x, dy, W1, W2, W1s, W2s, dx, dW1, dW2, dW1s, dW2s, dlogits,
                  ws, stream=None):
    _check(lib().moe_layer_bwd(_cfg(cfg), _p(ctx), _p(logits), _p(x), _p(dy), _p(W1), _p(W2),
                               _p(W1s), _p(W2s), _p(dx), _p(dW1), _p(dW2), _p(dW1s), _p(dW2s),
                               _p(dlogits), _p(ws), _s(stream)), "moe_layer_bwd")


def moe_selftest_wait_timeout(ws, budget_cycles, stream=None):
    """Enqueue a bounded wait that is never satisfied (see include/moe.h)."""
    _check(lib().moe_selftest_wait_timeout(_p(ws), int(budget_cycles), _s(stream)),
           "moe_selftest_wait_timeout")


def moe_gemm_clock_trace(enable):
    """Turn the grouped GEMMs' clock tracing on (zeroing its sums) or off (keeping them)."""
    _check(lib().moe_gemm_clock_trace(1 if enable else 0), "moe_gemm_clock_trace")


def moe_gemm_clock_read():
    """The traced sums: (SM cycles, nanoseconds, loops) of the GEMM tile loops."""
    c, n, k = ctypes.c_uint64(0), ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(lib().moe_gemm_clock_read(ctypes.byref(c), ctypes.byref(n), ctypes.byref(k)),
           "moe_gemm_clock_read")
    return c.value, n.value, k.value


def moe_status(ws, stream=None):
    """Synchronise the stream and read + clear the device error word: (status, flags)."""
    flags = ctypes.c_int32(0)
    s = lib().moe_status(_p(ws), _s(stream), ctypes.byref(flags))
    return s, flags.value


# --------------------------------------------------------------------------- conveniences
def ctx_views(cfg, ctx):
    """Typed torch views of the saved tensors inside a forward context buffer."""
    import torch
    off = moe_ctx_offsets(cfg)
    T, k, E, d, f, fs = cfg.T, cfg.k, cfg.E, cfg.d, cfg.ffn, cfg.ffn_shared
    R = T * k
    spec = {
        "topk_idx": (torch.int32, (T, k)), "topk_w": (torch.float32, (T, k)),
        "counts": (torch.int32, (E,)), "kept": (torch.int32, (E,)),
        "offsets": (torch.int32, (E + 1,)), "dest_row": (torch.int32, (T, k)),
        "src_tok": (torch.int32, (R,)), "src_slot": (torch.int32, (R,)),
        "drop_mask": (torch.uint8, (T, k)), "xp": (torch.bfloat16, (R, d)),
        "ab": (torch.bfloat16, (R, 2 * f)), "h": (torch.bfloat16, (R, f)),
        "yp": (torch.bfloat16, (R, d)), "ab_s": (torch.bfloat16, (T, 2 * fs)),
        "h_s": (torch.bfloat16, (T, fs)), "ys": (torch.bfloat16, (T, d if fs else 0)),
    }
    if cfg.recompute:   # FC1's outputs are not kept in ctx
        for name, cols in (("ab", 2 * f), ("h", f), ("ab_s", 2 * fs), ("h_s", fs)):
            spec[name] = (torch.bfloat16, (0, cols))
    out = {}
    for i, name in enumerate(CTX_FIELDS):
        dt, shape = spec[name]
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dt).element_size()
        out[name] = ctx[off[i]: off[i] + nbytes].view(dt).view(shape)
    return out


class MoELayer:
    """Owns the workspace and forward context (torch device buffers) of one layer shape
    and calls moe_layer_fwd / moe_layer_bwd on them."""

    def __init__(self, cfg: MoEConfigC, device="cuda"):
        import torch
        self.cfg = cfg
        ws_b, ctx_b = moe_workspace_size(cfg)
        self.ws = torch.empty(ws_b, dtype=torch.uint8, device=device)
        self.ctx = torch.empty(ctx_b, dtype=torch.uint8, device=device)
        moe_ws_init(self.ws)

    def views(self):
        return ctx_views(self.cfg, self.ctx)

    def forward(self, logits, x, W1, W2, W1s=None, W2s=None, y=None, stream=None):
        import torch
        if y is None:
            y = torch.empty_like(x)
        moe_layer_fwd(self.cfg, logits, x, W1, W2, W1s, W2s, y, self.ctx, self.ws, stream)
        return y

    def quantize_weights(self, W1, W2, stream=None):
        """MXFP8 blob of the routed weights (cache it while W1, W2 are unchanged)."""
        import torch
        nbytes, _ = moe_mx_weights_size(self.cfg)
        wq = torch.empty(nbytes, dtype=torch.uint8, device=W1.device)
        moe_mx_quantize_weights(self.cfg, W1, W2, wq, stream)
        return wq

    def forward_mx(self, logits, x, wq, W1s=None, W2s=None, y=None, stream=None):
        """Forward with the routed experts in MXFP8 (config made with mxfp8=1 or 2); the
        bf16 backward() may follow it, or backward_mx()."""
        import torch
        if y is None:
            y = torch.empty_like(x)
        moe_layer_fwd_mx(self.cfg, logits, x, wq, W1s, W2s, y, self.ctx, self.ws, stream)
        return y

    def backward_mx(self, logits, x, dy, wq, W1s=None, W2s=None, out=None, stream=None):
        """Backward with the data-gradient GEMMs in MXFP8 (after forward_mx), and with
        mxfp8=2 the routed weight gradients too; `out` as in backward(); the
        weight-gradient shapes come from the config."""
        import torch
        c = self.cfg
        if out is None:
            bf = dict(dtype=torch.bfloat16, device=x.device)
            out = {"dx": torch.empty_like(x),
                   "dW1": torch.empty((c.E, 2 * c.ffn, c.d), **bf),
                   "dW2": torch.empty((c.E, c.d, c.ffn), **bf),
                   "dlogits": torch.empty_like(logits)}
            if c.ffn_shared:
                out["dW1s"] = torch.empty_like(W1s)
                out["dW2s"] = torch.empty_like(W2s)
        moe_layer_bwd_mx(c, self.ctx, logits, x, dy, wq, W1s, W2s, out["dx"], out["dW1"],
                         out["dW2"], out.get("dW1s"), out.get("dW2s"), out["dlogits"], self.ws,
                         stream)
        return out

    def backward(self, logits, x, dy, W1, W2, W1s=None, W2s=None, out=None, stream=None):
        import torch
        if out is None:
            out = {"dx": torch.empty_like(x), "dW1": torch.empty_like(W1),
                   "dW2": torch.empty_like(W2),
                   "dlogits": torch.empty_like(logits)}
            if self.cfg.ffn_shared:
                out["dW1s"] = torch.empty_like(W1s)
                out["dW2s"] = torch.empty_like(W2s)
        moe_layer_bwd(self.cfg, self.ctx, logits, x, dy, W1, W2, W1s, W2s, out["dx"], out["dW1"],
                      out["dW2"], out.get("dW1s"), out.get("dW2s"), out["dlogits"], self.ws,
                      stream)
        return out

    def status(self, stream=None):
        return moe_status(self.ws, stream)
