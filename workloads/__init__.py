"""Seeded synthetic inputs for the MoE layer, shared by the oracle side and the GPU side.

This module only draws random numbers and lays them out; it contains none of the
layer's arithmetic (no routing, no gating, no FFN).  Both the CPU oracle tests and
the CUDA parity tests / benchmark take their inputs from here, so that the two sides
see bit-identical data.

Input recipe (shapes stand in for the models named on the pages: Mixtral,
Qwen3-30B-A3B, DeepSeek-V3, and the X-MoE capacity setting c = 1.25):

* x  ~ N(0, 1), rounded to bf16, shape [T, d]
* dy ~ N(0, 1), rounded to bf16, shape [T, d] (upstream gradient of the layer output)
* router logits ~ N(0, 1) fp32, shape [T, E], plus a per-expert Zipf bias for the
  skewed configurations: draw a seeded permutation r_e of 1..E and add
  bias_e = -alpha * s * ln(r_e), i.e. the log of a Zipf(s) pmf scaled by alpha, so the
  softmax mass of expert e is proportional to r_e^(-alpha*s).
* expert weights ~ N(0, 0.02), rounded to bf16: W1 [E, 2f, d] (rows 0..f-1 gate,
  f..2f-1 up, nn.Linear (out, in) layout), W2 [E, d, f]; the shared expert adds
  W1s [2fs, d] and W2s [d, fs].

Every tensor has its own generator, seeded from (seed, configuration name, tensor
name).  Small configurations are drawn on the host with numpy's PCG64; the large
ones draw x / dy / weights with a seeded torch CUDA generator (tens of GB of
weights would take minutes on the host), and the host copies of any slice the
oracle needs are taken from those device tensors.
"""

from __future__ import annotations

import dataclasses
import math
import zlib

import numpy as np


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    d: int          # model width
    E: int          # routed experts
    k: int          # experts per token
    f: int          # routed expert SwiGLU width
    fs: int = 0     # shared expert SwiGLU width (0 = no shared expert)
    gate: str = "softmax"      # "softmax" (renormalised over the top-k) or "sigmoid"
    route_scale: float = 1.0   # 2.5 for the DeepSeek-V3-style sigmoid gate
    cap_factor: float | None = None   # capacity factor c; None = unlimited
    zipf_s: float | None = None       # Zipf exponent of the expert bias (None = no bias)
    zipf_alpha: float = 1.0           # scale of the Zipf bias
    # routing variants
    select_bias: tuple | None = None  # per-expert bias added to the logits for selection only
    drop_negative: bool = False       # drop assignments whose raw logit is negative
    drop_by_score: bool = False       # on overflow keep the best-scored, not the earliest
    recompute: bool = False           # backward recomputes FC1 instead of saving ab, h

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def capacity(self) -> int:
        """Per-expert capacity floor(c*T*k/E); 0 means unlimited."""
        if self.cap_factor is None:
            return 0
        # exact rational arithmetic so that e.g. 1.25*16384*6/64 = 1920 exactly
        from fractions import Fraction
        c = Fraction(self.cap_factor).limit_denominator(1 << 20)
        return int(math.floor(c * self.T * self.k / self.E))

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    # Tiny MoE layer (small case the oracle finishes in seconds)
    "tiny": MoEConfig("tiny", T=256, d=128, E=8, k=2, f=256),
    # Mixtral-style layer, near-uniform load
    "mixtral": MoEConfig("mixtral", T=4096, d=4096, E=8, k=2, f=14336),
    # Qwen3-30B-A3B-style fine-grained layer, Zipf(1.1) bias x 0.5
    "qwen3": MoEConfig("qwen3", T=8192, d=2048, E=128, k=8, f=768, zipf_s=1.1, zipf_alpha=0.5),
    # DeepSeek-V3-style layer: sigmoid gate x 2.5 + one shared expert, Zipf(1.2) bias
    "dsv3": MoEConfig("dsv3", T=4096, d=7168, E=256, k=8, f=2048, fs=2048, gate="sigmoid",
                      route_scale=2.5, zipf_s=1.2, zipf_alpha=1.0),
    # X-MoE-style capacity-dropping layer, c = 1.25, Zipf(1.5) bias
    "capacity": MoEConfig("capacity", T=16384, d=4096, E=64, k=6, f=1408, cap_factor=1.25,
                          zipf_s=1.5, zipf_alpha=1.0),
}


# Smaller shapes with the same per-expert GEMM shapes, for profiler captures that must
# stay within a few GB of device memory: Mixtral's expert (d=4096, f=14336, ~1024 rows
# per expert) with 2 experts and top-1; Qwen3's (d=2048, f=768, ~512 rows per expert,
# the same Zipf skew) with a quarter of the tokens and experts.
PROFILE_CONFIGS = {
    "mixtral_e2": MoEConfig("mixtral_e2", T=2048, d=4096, E=2, k=1, f=14336),
    "qwen3_e32": MoEConfig("qwen3_e32", T=2048, d=2048, E=32, k=8, f=768, zipf_s=1.1,
                           zipf_alpha=0.5),
}


def _seed(seed: int, cfg_name: str, tensor: str) -> int:
    return (seed * 1_000_003 + zlib.crc32(f"{cfg_name}/{tensor}".encode())) & 0x7FFFFFFF


def _rng(seed: int, cfg_name: str, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(_seed(seed, cfg_name, tensor)))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even) and return the raw
    uint16 bit patterns.  Inputs here are finite draws from a normal distribution: the
    largest finite pattern plus 0x8000 still fits in 32 bits, so the sum cannot wrap."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bit patterns to float64."""
    u = (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).astype(np.float64)


def gen_select_bias(cfg: MoEConfig, scale: float = 1.0, seed: int = 0) -> tuple:
    """A per-expert selection bias (as a balancing controller would hold): N(0, scale^2)."""
    z = _rng(seed, cfg.name, "select_bias").standard_normal(cfg.E, dtype=np.float32) * scale
    return tuple(float(v) for v in z.astype(np.float32))


def zipf_bias(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    """Per-expert logit bias -alpha*s*ln(r_e) for a seeded permutation r of 1..E."""
    if cfg.zipf_s is None:
        return np.zeros(cfg.E, dtype=np.float64)
    r = _rng(seed, cfg.name, "zipf_rank").permutation(cfg.E) + 1
    return -cfg.zipf_alpha * cfg.zipf_s * np.log(r.astype(np.float64))


def gen_logits(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    """Router logits [T, E] float32: N(0, 1) plus the Zipf bias (added before routing)."""
    z = _rng(seed, cfg.name, "logits").standard_normal((cfg.T, cfg.E), dtype=np.float32)
    b = zipf_bias(cfg, seed).astype(np.float32)
    return np.ascontiguousarray(z + b[None, :], dtype=np.float32)


def gen_bf16(cfg: MoEConfig, tensor: str, shape, std: float = 1.0, seed: int = 0) -> np.ndarray:
    """Host draw of N(0, std^2) rounded to bf16; returns uint16 bit patterns."""
    z = _rng(seed, cfg.name, tensor).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return f32_to_bf16_bits(z)


WEIGHT_STD = 0.02


def weight_shapes(cfg: MoEConfig) -> dict:
    s = {"W1": (cfg.E, 2 * cfg.f, cfg.d), "W2": (cfg.E, cfg.d, cfg.f)}
    if cfg.fs:
        s["W1s"] = (2 * cfg.fs, cfg.d)
        s["W2s"] = (cfg.d, cfg.fs)
    return s


def gen_inputs_host(cfg: MoEConfig, seed: int = 0) -> dict:
    """All inputs of one fwd+bwd step on the host (small configurations).

    Returns numpy arrays: logits f32 [T,E]; x, dy, W1, W2 (and W1s, W2s) as uint16
    bf16 bit patterns."""
    out = {
        "logits": gen_logits(cfg, seed),
        "x": gen_bf16(cfg, "x", (cfg.T, cfg.d), 1.0, seed),
        "dy": gen_bf16(cfg, "dy", (cfg.T, cfg.d), 1.0, seed),
    }
    for name, shape in weight_shapes(cfg).items():
        out[name] = gen_bf16(cfg, name, shape, WEIGHT_STD, seed)
    return out


def gen_inputs_device(cfg: MoEConfig, device, seed: int = 0, chunk_elems: int = 1 << 28) -> dict:
    """All inputs of one step as torch tensors on `device` (large configurations).

    logits come from the host generator (small); x, dy and the weights are drawn with a
    seeded torch generator on the device, in chunks so the fp32 temporaries stay small."""
    import torch

    out = {"logits": torch.from_numpy(gen_logits(cfg, seed)).to(device)}

    def draw(tensor, shape, std):
        g = torch.Generator(device=device)
        g.manual_seed(_seed(seed, cfg.name, tensor))
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = t.view(-1)
        n = flat.numel()
        for s in range(0, n, chunk_elems):
            e = min(n, s + chunk_elems)
            z = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
            if std != 1.0:
                z.mul_(std)
            flat[s:e].copy_(z)
        return t

    out["x"] = draw("x", (cfg.T, cfg.d), 1.0)
    out["dy"] = draw("dy", (cfg.T, cfg.d), 1.0)
    for name, shape in weight_shapes(cfg).items():
        out[name] = draw(name, shape, WEIGHT_STD)
    return out


def gen_rows_bf16(name: str, rows: int, cols: int, seed: int = 0, std: float = 1.0) -> np.ndarray:
    """Stand-alone N(0, std^2) bf16 matrix (e.g. a synthetic expert-output buffer yp
    for testing the combine step on its own)."""
    z = np.random.Generator(np.random.PCG64(_seed(seed, "rows", name))).standard_normal(
        (rows, cols), dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return f32_to_bf16_bits(z)
