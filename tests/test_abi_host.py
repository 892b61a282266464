"""The C-ABI library builds for sm_103a, loads, exports every entry point that
include/moe.h declares, and its host-only logic (capacity, sizes, validation, status
names) behaves as documented.  CPU only: nothing here launches a kernel."""

import ctypes
import os
import re

import pytest

import token_dispatch_expert_gb300 as tde
from workloads import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    tde.build()
    return tde.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n


def test_binding_names_match_the_header():
    for n in declared_symbols():
        assert hasattr(tde, n), n
        assert n in tde.__all__, n


def cfg_of(c):
    return tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs, c.gate, c.route_scale, c.capacity,
                           recompute=c.recompute)


def test_capacity_from_factor(L):
    assert tde.moe_capacity_from_factor(16384, 6, 64, 1.25) == 1920
    assert tde.moe_capacity_from_factor(256, 2, 8, 0.5) == 32
    assert tde.moe_capacity_from_factor(5, 2, 4, 0.8) == 2
    assert tde.moe_capacity_from_factor(100, 2, 8, 0.0) == 0
    assert tde.moe_capacity_from_factor(0, 2, 8, 1.0) == -1
    for c in CONFIGS.values():
        if c.cap_factor:
            assert tde.moe_capacity_from_factor(c.T, c.k, c.E, c.cap_factor) == c.capacity


def test_workspace_and_ctx_layout(L):
    for c in CONFIGS.values():
        cfg = cfg_of(c)
        ws, ctx = tde.moe_workspace_size(cfg)
        off = tde.moe_ctx_offsets(cfg)
        assert all(o % 256 == 0 for o in off)
        assert off == sorted(off)
        R = c.T * c.k
        # the saved activations alone: xp, ab, h, yp
        assert ctx >= R * (c.d + 2 * c.f + c.f + c.d) * 2
        assert ws >= 256
        # recompute moves ab and h (and the shared expert's) out of ctx into ws
        rc = cfg_of(c.replace(recompute=True))
        ws_r, ctx_r = tde.moe_workspace_size(rc)
        moved = (R * 3 * c.f + c.T * 3 * c.fs) * 2
        assert ctx - ctx_r >= moved
        assert ws_r - ws >= moved
        # drop by score (with a capacity) needs one word per assignment more in ws
        bs = tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs, c.gate, c.route_scale,
                             c.capacity or 1, drop_by_score=True)
        plain = tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs, c.gate, c.route_scale,
                                c.capacity or 1)
        assert tde.moe_workspace_size(bs)[0] - tde.moe_workspace_size(plain)[0] >= R * 4
        # MXFP8 weight gradients: the four along-token quantised operands (codes + scales)
        if c.d % 128 == 0 and c.f % 128 == 0:
            mx = [tde.moe_workspace_size(tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs,
                                                         c.gate, c.route_scale, c.capacity,
                                                         mxfp8=m))[0] for m in (0, 1, 2)]
            kcap = 128 * ((R + 127) // 128 + c.E)
            assert mx[1] > mx[0]
            assert mx[2] - mx[1] >= (2 * c.d + 3 * c.f) * kcap


@pytest.mark.parametrize("bad,status", [
    (dict(k=9, E=16), 2),          # k > 8 unsupported
    (dict(E=300, k=2), 2),         # E > 256
    (dict(d=100), 2),              # d % 64
    (dict(ffn=96), 2),             # f % 64
    (dict(k=5, E=4), 1),           # k > E invalid
    (dict(T=0), 1),
    (dict(gate=7), 1),
    (dict(capacity=-1), 1),
    (dict(drop_negative=2), 1),
    (dict(recompute=-1), 1),
    (dict(select_bias=2), 1),      # not 4-byte aligned
    (dict(drop_by_score=3), 1),
    (dict(mxfp8=3), 1),
    (dict(mxfp8=-1), 1),
    (dict(mxfp8=2, d=192), 2),     # MXFP8 needs d, ffn multiples of 128
])
def test_invalid_configs_rejected_before_launch(L, bad, status):
    base = dict(T=64, d=128, E=8, k=2, ffn=128, ffn_shared=0, gate=0, route_scale=1.0,
                capacity=0)
    base.update(bad)
    cfg = tde.MoEConfigC(**base)
    ws, ctx = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(ws), ctypes.byref(ctx)) == status
    # a device call with the bad config returns the same status with nothing enqueued
    assert L.moe_permute(ctypes.byref(cfg), 16, 16, 16, 16, 16, None) == status


def test_null_and_misaligned_pointers_rejected(L):
    cfg = cfg_of(CONFIGS["tiny"])
    assert L.moe_permute(ctypes.byref(cfg), None, 16, 16, 16, 16, None) == 1
    assert L.moe_permute(ctypes.byref(cfg), 8, 16, 16, 16, 16, None) == 1   # not 16B aligned
    assert L.moe_route(ctypes.byref(cfg), *([None] * 11), None) == 1
    assert L.moe_layer_fwd(ctypes.byref(cfg), *([None] * 9), None) == 1
    # the shared expert's weights are required when ffn_shared > 0
    c = CONFIGS["dsv3"]
    cfg = cfg_of(c)
    assert L.moe_layer_fwd(ctypes.byref(cfg), 16, 16, 16, 16, None, None, 16, 16, 16,
                           None) == 1


def test_status_strings(L):
    for s, name in tde.STATUS.items():
        assert tde.moe_status_string(s) == name
    assert tde.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_binding_refuses_host_and_strided_tensors():
    """The binding hands kernels raw pointers: a host tensor or a non-contiguous view is
    refused before any call."""
    import torch
    with pytest.raises(ValueError, match="CUDA"):
        tde._p(torch.zeros(4))
    assert tde._p(None) is None and tde._p(1234) == 1234


def test_noalloc_route_refusals_before_any_device_call(L):
    """moe_route_noalloc validates its arguments and the size of its fixed scratch on the
    host: null or misaligned pointers and shapes whose routing scratch exceeds the array
    are refused before anything touches a device."""
    def cfg(T, E, k, cap=0, by_score=False):
        return tde.make_config(T, 64, E, k, 64, capacity=cap, drop_by_score=by_score)

    ok = [16] * 10
    c = cfg(64, 8, 2)
    assert L.moe_route_noalloc(ctypes.byref(c), *([None] * 10), None, None) == 1
    assert L.moe_route_noalloc(ctypes.byref(c), 8, *ok[1:], None, None) == 1    # misaligned
    assert L.moe_route_noalloc(ctypes.byref(c), *ok, 18, None) == 1             # flags word
    # plain routing: ceil(T/32) * E * 4 bytes; T = 32768 more than E = 256 allows
    assert L.moe_route_noalloc(ctypes.byref(cfg(32769, 256, 8)), *ok, None, None) == 2
    # drop by score adds (E+1)*4 and T*k*4 bytes (each rounded up to 256): with E = 64 and
    # k = 8 the 1 MiB array holds T = 26200 and not one token more
    assert L.moe_route_noalloc(ctypes.byref(cfg(26201, 64, 8, 1, True)), *ok, None, None) == 2
    # the same shape routed by token order needs only the histogram: not refused for size
    # (with a device present this would launch, so it is only called where there is none)
    import torch
    if not torch.cuda.is_available():
        for c2 in (cfg(26201, 64, 8, 1, False), cfg(26200, 64, 8, 1, True),
                   cfg(32768, 256, 8)):
            assert L.moe_route_noalloc(ctypes.byref(c2), *ok, None, None) == 3   # no device


def test_dispatch_fused_backward_refusals(L):
    """moe_grouped_ffn_bwd_dispatch checks its configuration and every pointer on the host
    (null or not 16-byte aligned: MOE_ERR_INVALID_ARG) before anything is enqueued."""
    cfg = cfg_of(CONFIGS["tiny"])
    ok = [16] * 16
    assert L.moe_grouped_ffn_bwd_dispatch(ctypes.byref(cfg), *([None] * 16), None) == 1
    for i in range(16):
        bad = list(ok)
        bad[i] = None if i % 2 else 24          # null, or 8 bytes off a 16-byte boundary
        assert L.moe_grouped_ffn_bwd_dispatch(ctypes.byref(cfg), *bad, None) == 1, i
    big = tde.MoEConfigC(T=64, d=100, E=8, k=2, ffn=128, ffn_shared=0, gate=0,
                         route_scale=1.0, capacity=0)
    assert L.moe_grouped_ffn_bwd_dispatch(ctypes.byref(big), *ok, None) == 2   # d % 64


def test_gemm_clock_read_refuses_null_pointers(L):
    """Refused before any device call, so it runs without a GPU."""
    c = ctypes.c_uint64(0)
    assert L.moe_gemm_clock_read(None, ctypes.byref(c), ctypes.byref(c)) == 1
    assert L.moe_gemm_clock_read(ctypes.byref(c), None, ctypes.byref(c)) == 1
    assert L.moe_gemm_clock_read(ctypes.byref(c), ctypes.byref(c), None) == 1
