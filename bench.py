"""Benchmark of the single-GPU MoE layer (forward + backward) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one forward + backward of the MoE layer over one batch of T tokens:
route -> permute -> grouped FC1/SwiGLU/FC2 -> (shared expert) -> combine, then
combine/gate backward -> FC2 data-grad + SwiGLU backward -> FC2 weight-grad ->
FC1 data-grad -> FC1 weight-grad -> un-permute reduce.  The headline workload is the
Mixtral-style layer (T=4096, d=4096, E=8, top-2, f=14336) on synthetic seeded inputs;
the same line carries a `workloads` block with the tiny, Qwen3-, DeepSeek-V3- and
capacity-shaped layers measured the same way, and an `mxfp8` block with the Mixtral layer
on MXFP8 operands.  The metric is tokens/s of the whole step; the dominant kernel (the
tcgen05 grouped GEMM, six launches per step) is reported against its roofline.

Timing: `steps` steps are captured into one CUDA graph and replayed once after the
warm-up; each phase boundary is an event-record node on a side branch that waits for the
kernels before it, so the kernels keep their own chain (and their dependent-launch overlap)
while the events time them.  `value`, the per-phase split, the GEMM time and the clocks all
come from that one replay, so the GEMM time is a part of the step it divides; a replay of a
one-step graph without events and an eager loop are reported beside it.

With N > 1 (torchrun) every rank runs an independent replica of the layer (the path
does not shard: replicas only); the reported value is the sum over ranks, the time
the max over ranks.

--impl reference times the CPU oracle (the plain double-precision C reference of the
layer) on the host cores: routing, permute, combine, its backward and the reduce in
full, the expert FFN on a sample of rows, extrapolated to the whole layer.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# DRAM bytes per bf16 grouped-GEMM launch (average over the six launches of a step), from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of a profiling shape with
# the same per-expert GEMMs and 1/4 of the experts and of the rows -- every operand and
# result scales with those -- times 4: `mixtral_e2` for the Mixtral layer, `qwen3_e32` for
# the Qwen3 layer.  Valid for the grouped-GEMM kernel as it stands (late dependent-launch
# release, clock trace, the FC1 tail-tile hand-off wait, the per-CTA tile table, the
# epilogues that read a chunk's row pieces first and compute its rows without branches,
# the evict-first weight-gradient stores); emptied whenever the kernel changes, until the
# capture is taken again.
GEMM_TRAFFIC_PER_LAUNCH = {
    "mixtral": (4 * (658.5 + 340.6 + 491.2 + 248.1 + 671.1 + 540.5) / 6 * 1e6, "mixtral_e2"),
    "qwen3": (4 * (326.0 + 162.7 + 243.3 + 137.4 + 300.5 + 256.3) / 6 * 1e6, "qwen3_e32"),
}

# the extra workloads measured beside the headline, each in its own block of the line
EXTRA_WORKLOADS = ["tiny", "qwen3", "dsv3", "capacity"]


def gemm_algorithmic_bytes(c, rows_kept: int) -> float:
    """Each expert's weights read (or weight gradient written) once per GEMM, each
    activation row read / written once: the six launches of a step."""
    d, f, R = c.d, c.f, rows_kept
    W1, W2 = c.E * 2 * f * d * 2, c.E * d * f * 2
    xp, ab, h = R * d * 2, R * 2 * f * 2, R * f * 2
    b = (W1 + xp + ab + h) + (W2 + h + xp) + (W2 + xp + 2 * ab) + (xp + h + W2) + \
        (W1 + ab + xp) + (ab + xp + W1)
    return float(b)


def gemm_phases(c, rows_kept: int):
    """(flops, algorithmic bytes) of each of the six grouped-GEMM launches of a step, the
    shared expert's (T rows, one group) added to the matching launch."""
    def six(E, rows, d, f):
        W1, W2 = E * 2 * f * d * 2, E * d * f * 2
        xp, ab, h = rows * d * 2, rows * 2 * f * 2, rows * f * 2
        F = rows * d * f
        return [(4.0 * F, W1 + xp + ab + h),        # FC1 + SwiGLU
                (2.0 * F, W2 + h + xp),             # FC2
                (2.0 * F, W2 + xp + 2 * ab),        # FC2 dgrad + SwiGLU bwd
                (2.0 * F, xp + h + W2),             # dW2
                (4.0 * F, W1 + ab + xp),            # FC1 dgrad
                (4.0 * F, ab + xp + W1)]            # dW1
    ph = six(c.E, rows_kept, c.d, c.f)
    if c.fs:
        ph = [(a + x, b + y) for (a, b), (x, y) in zip(ph, six(1, c.T, c.d, c.fs))]
    return ph


def gemm_flops(c, rows_kept: int) -> float:
    """Algorithmic flops of the six grouped-GEMM launches: 18*d*f per kept row, plus the
    shared expert's 18*d*fs per token."""
    return 18.0 * c.d * c.f * rows_kept + (18.0 * c.d * c.fs * c.T if c.fs else 0.0)


def memory_bytes(c, rows_kept: int) -> dict:
    """Algorithmic bytes of the HBM-bound steps: each source row read once, each
    destination row written once, index arrays counted."""
    T, d, k, E, Rk = c.T, c.d, c.k, c.E, rows_kept
    return {
        "permute": (T + Rk) * d * 2 + Rk * 4,
        "combine": (Rk + T + (T if c.fs else 0)) * d * 2 + T * k * 8,
        "combine_bwd": (T + 2 * Rk) * d * 2 + T * E * 4 + T * k * 12,
        "unpermute_reduce": (Rk + T + (T if c.fs else 0)) * d * 2 + T * k * 4,
    }


def choose_peak(peaks: dict, clk: dict, gemm_mhz=None):
    """The bf16 tensor peak that applies to a timed region: the burst figure (measured with
    the SM clock at its maximum) when the GEMMs ran at the maximum clock, the sustained
    figure (measured under the power cap) when they ran lower.  The clock is the one the
    GEMM kernels measured over their own tile loops (`gemm_mhz`, moe_gemm_clock_trace)
    when given, else the median of the nvidia-smi samples in the region."""
    burst = float(peaks["bf16_tflops"])
    sus = float(peaks.get("bf16_tflops_sustained", burst))
    mx = clk.get("sm_max_mhz") or peaks.get("sm_max_mhz")
    if gemm_mhz is not None:
        med, what = gemm_mhz, "SM clock of the GEMMs' tile loops (clock64 / %globaltimer)"
    else:
        med, what = clk.get("sm_mhz"), "median SM clock of the nvidia-smi samples"
    if med is None or not mx:
        return sus, "sustained", "bf16_tflops_sustained (no SM clock measured in the region)"
    if med >= 0.95 * mx:
        return burst, "burst", (f"bf16_tflops (burst): {what} {med:.0f} MHz of "
                                f"{mx:.0f} max in the timed region")
    return sus, "sustained", (f"bf16_tflops_sustained: {what} {med:.0f} MHz, below "
                              f"0.95 x {mx:.0f} max, in the timed region")


def gemm_clock_summary(sums):
    """moe_gemm_clock_read()'s (cycles, ns, loops) as the SM clock of the GEMM tile loops."""
    cycles, ns, loops = sums
    if not loops or not ns:
        return None
    return {"sm_mhz": round(cycles / ns * 1e3, 1), "loops": loops,
            "source": "clock64 cycles over %globaltimer nanoseconds of every grouped-GEMM "
                      "CTA's tile loop in the timed run (moe_gemm_clock_trace)"}


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms), each stamped with the host time it arrived, so
    that the clocks of any timed window can be summarised."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []      # (host time, sm MHz, max MHz, power W, set of reasons)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                pw = float(parts[3])
            except ValueError:
                pw = None
            rs = {n for n, v in zip(self.REASONS, parts[5:9]) if v.lower() in ("active", "1")}
            self.samples.append((time.time(), sm, mx, pw, rs))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def window(self, t0: float, t1: float, pad: float = 0.06) -> dict:
        """Summary of the samples that arrived in [t0, t1 + pad] (the reader stamps a sample
        slightly after it was taken); the nearest sample if none did."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sel = [s for s in self.samples if t0 <= s[0] <= t1 + pad]
        if not sel and self.samples:
            mid = 0.5 * (t0 + t1)
            sel = [min(self.samples, key=lambda s: abs(s[0] - mid))]
        sm = sorted(s[1] for s in sel)
        reasons = set()
        for s in sel:
            reasons |= s[4]
        pw = [s[3] for s in sel if s[3] is not None]
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": sel[-1][2] if sel else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sel)}


# --------------------------------------------------------------------------- dist
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(world, value: float, op) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    device = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(world, value: float) -> float:
    import torch.distributed as dist
    return _reduce(world, value, dist.ReduceOp.MAX) if world > 1 else value


def sum_over_ranks(world, value: float) -> float:
    import torch.distributed as dist
    return _reduce(world, value, dist.ReduceOp.SUM) if world > 1 else value


def replica_throughput(world, tokens_local: float, ms_local: float):
    """Whole-job throughput of independent replicas: all ranks' tokens over the slowest
    rank's time.  Returns (tokens_total, ms_max, tokens_per_s)."""
    ms_max = max_over_ranks(world, ms_local)
    tokens_total = sum_over_ranks(world, tokens_local)
    return tokens_total, ms_max, tokens_total / (ms_max / 1e3)


# --------------------------------------------------------------------------- oracle timing
class OracleTimer:
    """Times the CPU oracle (float64 C, OpenMP) on one workload.

    Routing, permute, combine, the combine / gate backward and the un-permute reduce run in
    full, on every token.  The expert FFN (forward, data gradients and weight gradients) is
    timed on one expert's rows: the oracle's row loops run one row per thread, so a sample
    of n rows costs about a + b*n for n a multiple of the thread count, a being the fixed
    cost of one expert (its weight-gradient buffers) and b the cost of a row.  Two samples
    (one and two rows per thread) give a and b; the FFN of the whole layer is then
    sum over experts of (a + b * kept_e), plus the shared expert's T rows.  When that
    estimate fits the time budget, every expert's FFN is timed in full instead and nothing
    is extrapolated.

    The oracle is timed as it stands (float64, the same build the tests use): it is not
    tuned for speed.  Inputs come from the host generators; the combine and reduce are fed
    the permuted tokens as their expert rows (their values do not change the work)."""

    def __init__(self, c):
        import numpy as np
        import oracle
        from workloads import WEIGHT_STD, gen_bf16, gen_logits

        oracle.build()
        self.c = c
        self.np = np
        self.threads = oracle.threads()
        self.logits = gen_logits(c)
        self.x = oracle.layer._f64(gen_bf16(c, "x", (c.T, c.d)))
        self.dy = oracle.layer._f64(gen_bf16(c, "dy", (c.T, c.d)))
        self.r = oracle.route(c, self.logits)            # sizes the rest (untimed)
        self.kept = [int(v) for v in self.r["kept"]]
        self.rows = int(self.r["offsets"][-1])
        self.e_s = int(np.argmax(self.r["kept"]))         # the FFN sample's expert
        self.W1e = oracle.layer._f64(gen_bf16(c, "W1[sample]", (2 * c.f, c.d), WEIGHT_STD))
        self.W2e = oracle.layer._f64(gen_bf16(c, "W2[sample]", (c.d, c.f), WEIGHT_STD))
        self.full_W = None

    def parts(self) -> dict:
        """Seconds of each step the oracle runs on every token."""
        import oracle
        c, r = self.c, self.r
        t = {}
        t0 = time.perf_counter()
        oracle.route(c, self.logits)
        t["route"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        xp = oracle.permute(c, r, self.x)
        t["permute"] = time.perf_counter() - t0
        ys = self.x if c.fs else None
        t0 = time.perf_counter()
        oracle.combine(c, r["dest_row"], r["topk_w"], xp, ys)
        t["combine"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.combine_bwd(c, self.logits, r, self.dy, xp)
        t["combine_bwd"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.unpermute_reduce(c, r["dest_row"], xp, ys)
        t["unpermute_reduce"] = time.perf_counter() - t0
        self._xp = xp
        return t

    def ffn(self, rows, W1e, W2e) -> float:
        """Seconds of the expert FFN forward + backward (data and weight gradients) on the
        given rows of one expert."""
        import oracle
        n = rows.shape[0]
        dyp = self.dy[: n]
        t0 = time.perf_counter()
        ab, h, _ = oracle.ffn_fwd_rows(rows, W1e, W2e)
        dab, _ = oracle.ffn_bwd_rows(dyp, ab, W1e, W2e)
        oracle.layer.ffn_wgrad_rows(rows, h, dyp, dab, self.c.d, W1e.shape[0] // 2)
        return time.perf_counter() - t0

    def _sample_rows(self, n):
        s = int(self.r["offsets"][self.e_s])
        if n <= self.kept[self.e_s]:
            return self._xp[s:s + n]
        return self.x[self.np.arange(n) % self.c.T]      # more rows than the expert holds

    def fit(self):
        """a, b of the FFN cost model from samples of one and three rows per thread."""
        n1, n2 = self.threads, 3 * self.threads
        t1 = self.ffn(self._sample_rows(n1), self.W1e, self.W2e)
        t2 = self.ffn(self._sample_rows(n2), self.W1e, self.W2e)
        b = max((t2 - t1) / (n2 - n1), 1e-9)
        a = max(t1 - b * n1, 0.0)
        return a, b, [(n1, t1), (n2, t2)]

    def measure(self, budget_s: float, a_fixed: float | None = None) -> dict:
        """One timing of the oracle on the workload.  With a_fixed (the per-expert fixed
        cost from an earlier fit) only one FFN sample is timed and gives b."""
        c = self.c
        parts = self.parts()
        if a_fixed is None:
            a, b, samples = self.fit()
        else:
            n1 = self.threads
            t1 = self.ffn(self._sample_rows(n1), self.W1e, self.W2e)
            a, b, samples = a_fixed, max((t1 - a_fixed) / n1, 1e-9), [(n1, t1)]
        fs_scale = (c.fs / c.f) if c.fs else 0.0
        est = sum(a + b * n for n in self.kept if n) + \
            ((a + b * c.T) * fs_scale if c.fs else 0.0)
        extrapolated = True
        ffn_s = est
        if est <= budget_s:
            ffn_s = self.ffn_full()
            extrapolated = False
        total = sum(parts.values()) + ffn_s
        return {"seconds_per_step": total, "tokens_per_s": c.T / total,
                "extrapolated": extrapolated, "parts_s": parts, "ffn_s": ffn_s,
                "ffn_fit": {"a_s": a, "b_s_per_row": b, "samples": [list(x) for x in samples]},
                "rows_kept": self.rows}

    def ffn_full(self) -> float:
        """Every expert's FFN (and the shared expert's) timed on its own rows."""
        import oracle
        from workloads import WEIGHT_STD, gen_bf16, weight_shapes
        c = self.c
        if self.full_W is None:
            self.full_W = {n: oracle.layer._f64(gen_bf16(c, n, s, WEIGHT_STD))
                           for n, s in weight_shapes(c).items()}
        W = self.full_W
        off = self.r["offsets"]
        t = 0.0
        for e in range(c.E):
            s0, s1 = int(off[e]), int(off[e + 1])
            if s1 > s0:
                t += self.ffn(self._xp[s0:s1], W["W1"][e], W["W2"][e])
        if c.fs:
            t += self.ffn(self.x, W["W1s"], W["W2s"])
        return t

    def describe(self, m: dict) -> str:
        c = self.c
        fit = m["ffn_fit"]
        if not m["extrapolated"]:
            return (f"route, permute, combine, combine backward, reduce and every expert's "
                    f"FFN fwd+bwd on all {c.T} tokens (float64 C oracle, OpenMP)")
        ns = " and ".join(str(x[0]) for x in fit["samples"])
        return (f"route, permute, combine, combine backward and reduce timed on all {c.T} "
                f"tokens; the expert FFN fwd+bwd timed on {ns} rows of expert {self.e_s} and "
                f"extrapolated to the {m['rows_kept']} kept rows of {c.E} experts"
                + (" and the shared expert" if c.fs else "")
                + " as sum_e (a + b * rows_e) (float64 C oracle, OpenMP)")


# --------------------------------------------------------------------------- one workload
class Workload:
    """Device buffers and the step of one workload: the layer's calls in order, with an
    optional event recorded at each phase boundary (on the current stream)."""

    def __init__(self, c, dev, seed=0, mxfp8=0, fuse_gather=False, mx_cache_weights=True,
                 fuse_dispatch_bwd=False):
        import torch

        import token_dispatch_expert_gb300 as tde
        from workloads import gen_inputs_device

        self.c, self.dev, self.mxfp8 = c, dev, mxfp8
        self.fuse_gather, self.mx_cache = fuse_gather, mx_cache_weights
        self.fuse_dispatch_bwd = fuse_dispatch_bwd
        self.tde = tde
        bias_t = (torch.tensor(c.select_bias, dtype=torch.float32, device=dev)
                  if c.select_bias is not None else None)
        self.cfg = tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs, c.gate, c.route_scale,
                                   c.capacity, select_bias=bias_t,
                                   drop_negative=c.drop_negative, recompute=c.recompute,
                                   drop_by_score=c.drop_by_score, mxfp8=mxfp8)
        g = self.g = gen_inputs_device(c, dev, seed=seed)
        self.side = torch.cuda.Stream(device=dev)   # where the phase events are recorded
        R = c.T * c.k
        ws_b, ctx_b = tde.moe_workspace_size(self.cfg)
        self.ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
        self.ctx = torch.empty(ctx_b, dtype=torch.uint8, device=dev)
        tde.moe_ws_init(self.ws)
        self.v = tde.ctx_views(self.cfg, self.ctx)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((c.T, c.d), **bf)
        self.dyp = torch.empty((R, c.d), **bf)
        self.dab = torch.empty((R, 2 * c.f), **bf)
        self.dxp = torch.empty((R, c.d), **bf)
        self.dx = torch.empty((c.T, c.d), **bf)
        self.dW1 = torch.empty_like(g["W1"])
        self.dW2 = torch.empty_like(g["W2"])
        self.dl = torch.empty((c.T, c.E), dtype=torch.float32, device=dev)
        self.shared = None
        if c.fs:
            # the shared expert as a one-group grouped FFN over all T tokens
            s_cfg = tde.make_config(c.T, c.d, 1, 1, c.fs)
            s_off = torch.tensor([0, c.T], dtype=torch.int32, device=dev)
            self.shared = dict(cfg=s_cfg, off=s_off, ab=torch.empty((c.T, 2 * c.fs), **bf),
                               h=torch.empty((c.T, c.fs), **bf), ys=torch.empty((c.T, c.d), **bf),
                               dab=torch.empty((c.T, 2 * c.fs), **bf),
                               dx=torch.empty((c.T, c.d), **bf),
                               dW1=torch.empty_like(g["W1s"]), dW2=torch.empty_like(g["W2s"]))
        self.phases = ["route", "permute", "ffn_fwd", "combine", "combine_bwd", "ffn_bwd",
                       "unpermute_reduce"]
        if c.recompute:
            # FC1 is recomputed inside the backward: the step runs through the two
            # whole-layer calls, timed as two phases
            self.phases = ["layer_fwd", "layer_bwd"]
        self.mxb = None
        if mxfp8:
            nbytes, _ = tde.moe_mx_weights_size(self.cfg)
            self.wq = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            u8 = dict(dtype=torch.uint8, device=dev)
            # the activation scales are atoms tiled by 128 rows per expert segment: sized
            # by the library, not by rows x K/32
            self.mxb = dict(xq=torch.empty((R, c.d), **u8),
                            xs=torch.empty(tde.moe_mx_act_scales_size(self.cfg, c.d), **u8),
                            hq=torch.empty((R, c.f), **u8),
                            hs=torch.empty(tde.moe_mx_act_scales_size(self.cfg, c.f), **u8))
            if mx_cache_weights:
                # weight-quantisation caching: the blob is made once, as when one optimizer
                # step's weights serve many micro-batches
                tde.moe_mx_quantize_weights(self.cfg, g["W1"], g["W2"], self.wq)
            else:
                self.phases = ["mx_weight_quant"] + self.phases

    def join_marks(self):
        """The current stream waits for the side stream the phase events are recorded on."""
        import torch
        torch.cuda.current_stream().wait_stream(self.side)

    # route 3, permute 1, FC1+FC2 2, combine 1, combine-bwd 1, backward GEMMs 4 plus the two
    # per-segment map preparations, reduce 1; the shared expert 2 + 4
    def launches_per_step(self) -> int:
        c = self.c
        n = 3 + 1 + 2 + 1 + 1 + 6 + 1 + (6 if self.shared else 0)
        if self.fuse_gather:
            n -= 1
        if c.recompute:
            n += 1 + (1 if self.shared else 0)          # the recomputed FC1
        if c.drop_by_score and c.capacity > 0:
            n += 2                                      # score scatter + select
        if self.mxfp8:
            n += 1                                      # dyp quantised for the data gradients
        if self.mxfp8 == 2:
            n += 2                                      # 4 along-token quantisations replace
            #                                             the 2 per-segment map preparations
        if self.mxfp8 and not self.mx_cache:
            n += 4                                      # the four weight-quantisation kernels
        return n

    def step(self, ev=None):
        """One forward + backward.  ev: len(phases) + 1 events marking the phase boundaries
        (or None).  Each is recorded on a side stream that first waits for the work enqueued
        so far: the event completes when the kernels before it have, while the next kernel
        still depends on the previous kernel alone, so its dependent-launch overlap and the
        step's kernel-to-kernel chain are what they are without the events.  The caller
        joins the side stream (`join_marks`) before the work after the step needs it."""
        import torch
        tde, c, g, v, ws = self.tde, self.c, self.g, self.v, self.ws
        shared = self.shared
        n_mark = [0]

        def mark():
            if ev is not None:
                self.side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(self.side):
                    ev[n_mark[0]].record()
            n_mark[0] += 1

        mark()
        if c.recompute:
            outs = {"dx": self.dx, "dW1": self.dW1, "dW2": self.dW2, "dlogits": self.dl}
            tde.moe_layer_fwd(self.cfg, g["logits"], g["x"], g["W1"], g["W2"], g.get("W1s"),
                              g.get("W2s"), self.y, self.ctx, ws)
            mark()
            tde.moe_layer_bwd(self.cfg, self.ctx, g["logits"], g["x"], g["dy"], g["W1"],
                              g["W2"], g.get("W1s"), g.get("W2s"), self.dx, self.dW1, self.dW2,
                              shared["dW1"] if shared else None,
                              shared["dW2"] if shared else None, self.dl, ws)
            mark()
            return
        if self.mxfp8 and not self.mx_cache:
            tde.moe_mx_quantize_weights(self.cfg, g["W1"], g["W2"], self.wq)
            mark()
        tde.moe_route(self.cfg, g["logits"], v["topk_idx"], v["topk_w"], v["counts"], v["kept"],
                      v["offsets"], v["dest_row"], v["src_tok"], v["src_slot"], v["drop_mask"],
                      ws)
        mark()
        if self.mxfp8:         # permute + quantise (bf16 xp kept for the backward)
            m = self.mxb
            tde.moe_mx_permute_quant(self.cfg, g["x"], v["src_tok"], v["offsets"], v["xp"],
                                     m["xq"], m["xs"], ws)
            mark()
            tde.moe_grouped_ffn_mx(self.cfg, m["xq"], m["xs"], v["offsets"], self.wq, v["ab"],
                                   v["h"], m["hq"], m["hs"], v["yp"], ws)
        elif self.fuse_gather:   # the permute folded into FC1's loads: no xp
            mark()
            tde.moe_grouped_ffn_gather(self.cfg, g["x"], v["src_tok"], v["offsets"], g["W1"],
                                       g["W2"], v["ab"], v["h"], v["yp"], ws)
        else:
            tde.moe_permute(self.cfg, g["x"], v["src_tok"], v["offsets"], v["xp"], ws)
            mark()
            tde.moe_grouped_ffn(self.cfg, v["xp"], v["offsets"], g["W1"], g["W2"], v["ab"],
                                v["h"], v["yp"], ws)
        if shared:
            tde.moe_grouped_ffn(shared["cfg"], g["x"], shared["off"], g["W1s"], g["W2s"],
                                shared["ab"], shared["h"], shared["ys"], ws)
        mark()
        tde.moe_combine(self.cfg, v["yp"], v["dest_row"], v["topk_w"],
                        shared["ys"] if shared else None, self.y, ws)
        mark()
        tde.moe_combine_bwd(self.cfg, g["dy"], v["yp"], g["logits"], v["topk_idx"],
                            v["topk_w"], v["dest_row"], self.dyp, self.dl, ws)
        mark()
        if self.mxfp8:   # the data-gradient GEMMs on MXFP8 operands (level 2: the weight
            #              gradients too, else bf16)
            tde.moe_grouped_ffn_bwd_mx(self.cfg, self.dyp, v["xp"], v["offsets"], self.wq,
                                       v["ab"], v["h"], self.dab, self.dxp, self.dW1, self.dW2,
                                       ws)
        elif self.fuse_dispatch_bwd:   # the FC2 data-gradient reads dy through src_tok
            tde.moe_grouped_ffn_bwd_dispatch(self.cfg, g["dy"], v["topk_w"], v["src_tok"],
                                             v["src_slot"], self.dyp, v["xp"], v["offsets"],
                                             g["W1"], g["W2"], v["ab"], v["h"], self.dab,
                                             self.dxp, self.dW1, self.dW2, ws)
        elif self.fuse_gather:
            tde.moe_grouped_ffn_bwd_gather(self.cfg, self.dyp, g["x"], v["src_tok"],
                                           v["offsets"], g["W1"], g["W2"], v["ab"], v["h"],
                                           self.dab, self.dxp, self.dW1, self.dW2, ws)
        else:
            tde.moe_grouped_ffn_bwd(self.cfg, self.dyp, v["xp"], v["offsets"], g["W1"],
                                    g["W2"], v["ab"], v["h"], self.dab, self.dxp, self.dW1,
                                    self.dW2, ws)
        if shared:
            tde.moe_grouped_ffn_bwd(shared["cfg"], g["dy"], g["x"], shared["off"], g["W1s"],
                                    g["W2s"], shared["ab"], shared["h"], shared["dab"],
                                    shared["dx"], shared["dW1"], shared["dW2"], ws)
        mark()
        tde.moe_unpermute_reduce(self.cfg, self.dxp, v["dest_row"],
                                 shared["dx"] if shared else None, self.dx, ws)
        mark()

    def e2e(self, steps: int, warmup: int, world: int):
        """End to end through the public whole-layer API with host buffers in pinned memory,
        the way a training loop streams them: every step copies its inputs (logits, x, dy)
        host -> device and its results (y, dx, dlogits) device -> host, on one copy stream
        per direction, double-buffered so that step i+1's inputs and step i's results move
        while the GPU computes.  All copies fall inside the timed region.
        Returns (ms for `steps` steps, h2d bytes per step, d2h bytes per step)."""
        import torch
        tde, c, g, dev = self.tde, self.c, self.g, self.dev
        stream = torch.cuda.current_stream(dev)
        layer = tde.MoELayer(self.cfg, device=dev)
        h_logits = g["logits"].cpu().pin_memory()
        h_x = g["x"].cpu().pin_memory()
        h_dy = g["dy"].cpu().pin_memory()
        h_y = torch.empty((c.T, c.d), dtype=torch.bfloat16).pin_memory()
        h_dx = torch.empty((c.T, c.d), dtype=torch.bfloat16).pin_memory()
        h_dl = torch.empty((c.T, c.E), dtype=torch.float32).pin_memory()
        shared = self.shared
        bufs = []
        for b in range(2):
            o = {"dx": torch.empty_like(self.dx), "dW1": self.dW1, "dW2": self.dW2,
                 "dlogits": torch.empty_like(self.dl)}
            if shared:
                o["dW1s"] = shared["dW1"]; o["dW2s"] = shared["dW2"]
            bufs.append({"logits": torch.empty_like(g["logits"]), "x": torch.empty_like(g["x"]),
                         "dy": torch.empty_like(g["dy"]), "y": torch.empty_like(self.y),
                         "out": o})
        in_stream = torch.cuda.Stream(device=dev)
        out_stream = torch.cuda.Stream(device=dev)
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "done", "copied")}

        def copy_in(b):
            with torch.cuda.stream(in_stream):
                bufs[b]["logits"].copy_(h_logits, non_blocking=True)
                bufs[b]["x"].copy_(h_x, non_blocking=True)
                bufs[b]["dy"].copy_(h_dy, non_blocking=True)
                ev["in"][b].record(in_stream)

        def run(n):
            copy_in(0)
            for i in range(n):
                b = i & 1
                B = bufs[b]
                stream.wait_event(ev["in"][b])
                if i >= 2:
                    stream.wait_event(ev["copied"][b])   # step i-2's results are on the host
                if self.mxfp8:
                    if not self.mx_cache:
                        tde.moe_mx_quantize_weights(self.cfg, g["W1"], g["W2"], self.wq)
                    layer.forward_mx(B["logits"], B["x"], self.wq, g.get("W1s"), g.get("W2s"),
                                     y=B["y"])
                    layer.backward_mx(B["logits"], B["x"], B["dy"], self.wq, g.get("W1s"),
                                      g.get("W2s"), out=B["out"])
                else:
                    layer.forward(B["logits"], B["x"], g["W1"], g["W2"], g.get("W1s"),
                                  g.get("W2s"), y=B["y"])
                    layer.backward(B["logits"], B["x"], B["dy"], g["W1"], g["W2"],
                                   g.get("W1s"), g.get("W2s"), out=B["out"])
                ev["done"][b].record(stream)
                if i + 1 < n:
                    if i >= 1:   # buffer 1-b was last read by step i-1
                        in_stream.wait_event(ev["done"][1 - b])
                    copy_in(1 - b)
                with torch.cuda.stream(out_stream):
                    out_stream.wait_event(ev["done"][b])
                    h_y.copy_(B["y"], non_blocking=True)
                    h_dx.copy_(B["out"]["dx"], non_blocking=True)
                    h_dl.copy_(B["out"]["dlogits"], non_blocking=True)
                    ev["copied"][b].record(out_stream)
            stream.wait_event(ev["copied"][(n - 1) & 1])

        run(max(1, warmup))
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(steps)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        st, fl = layer.status()
        if st != 0:
            raise RuntimeError(f"device status after the e2e loop: {st} {fl:#x}")
        h2d = h_logits.numel() * 4 + h_x.numel() * 2 + h_dy.numel() * 2
        d2h = h_y.numel() * 2 + h_dx.numel() * 2 + h_dl.numel() * 4
        return e0.elapsed_time(e1), h2d, d2h


def graph_phase_times(wl, steps: int):
    """Per-phase device times inside a CUDA-graph replay: `steps` steps captured into one
    graph whose phase boundaries are event-record nodes on side branches (each waits for
    the kernels before it; the kernels keep their own chain, see Workload.step), replayed
    once to warm up and once timed.  Returns (phase ms per step, total ms per step) or None
    when event-record nodes are not available."""
    import torch
    P = len(wl.phases)
    try:
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(P + 1)]
               for _ in range(steps)]
    except TypeError:
        return None
    try:
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph):
            for i in range(steps):
                wl.step(evs[i])
            wl.join_marks()
        gph.replay()
        torch.cuda.synchronize()
        gph.replay()
        torch.cuda.synchronize()
        phase = {ph: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps
                 for j, ph in enumerate(wl.phases)}
        total = evs[0][0].elapsed_time(evs[-1][-1]) / steps
    except RuntimeError:
        return None
    del gph
    return phase, total


def measure(c, args, dev, world, rank, clocks, peaks, peak_src, mxfp8=0, e2e=True,
            fuse_gather=False, mx_cache=True, fuse_dispatch_bwd=False) -> dict:
    """Times one workload (see the module docstring) and returns its results."""
    import torch

    wl = Workload(c, dev, seed=rank, mxfp8=mxfp8, fuse_gather=fuse_gather,
                  mx_cache_weights=mx_cache, fuse_dispatch_bwd=fuse_dispatch_bwd)
    tde = wl.tde
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    st, fl = tde.moe_status(wl.ws)
    if st != 0:
        raise RuntimeError(f"{c.name}: device status after warm-up: "
                           f"{tde.moe_status_string(st)} {fl:#x}")
    rows_kept = int(wl.v["offsets"][-1].item())
    counts = wl.v["counts"].cpu().tolist()
    kept = wl.v["kept"].cpu().tolist()

    barrier(world)
    torch.cuda.synchronize()
    # 1. the timed replay: `value`, the per-phase split and the GEMM time (first after the
    #    warm-up, so every workload is timed at the same point of its run), with the GEMMs'
    #    clock traced over it
    tde.moe_gemm_clock_trace(True)
    w0 = time.time()
    pg = None if args.no_graph else graph_phase_times(wl, args.steps)
    w_pg = time.time()
    gemm_clock = None
    if pg is not None:
        torch.cuda.synchronize()
        tde.moe_gemm_clock_trace(False)
        gemm_clock = gemm_clock_summary(tde.moe_gemm_clock_read())
    # 2. a one-step graph without phase events, replayed `steps` times (reported beside)
    graph_ms = None
    g0w = g1w = None
    if not args.no_graph:
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph):
            wl.step()
        gph.replay()
        torch.cuda.synchronize()
        barrier(world)
        g0w = time.time()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            gph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        g1w = time.time()
        graph_ms = g0.elapsed_time(g1)
        del gph
    # 3. eager launches with events at the phase boundaries (reported beside the graph
    #    figure; their phase split is the fallback when graph event nodes are unavailable)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    eager_events = []
    for _ in range(args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(wl.phases) + 1)]
        wl.step(ev)
        eager_events.append(ev)
    wl.join_marks()
    t_end.record(stream)
    torch.cuda.synchronize()
    eager_ms = t_start.elapsed_time(t_end)
    w1 = time.time()
    if pg is None:   # the eager loop is the timed run: its GEMMs' clock
        tde.moe_gemm_clock_trace(False)
        gemm_clock = gemm_clock_summary(tde.moe_gemm_clock_read())
    barrier(world)
    st, fl = tde.moe_status(wl.ws)
    if st != 0:
        raise RuntimeError(f"{c.name}: device status after timing: "
                           f"{tde.moe_status_string(st)} {fl:#x}")
    eager_phase = {ph: sum(ev[i].elapsed_time(ev[i + 1]) for ev in eager_events) / args.steps
                   for i, ph in enumerate(wl.phases)}
    if pg is not None:
        phase_ms, phase_total = pg
        phase_src = ("CUDA-graph replay of the timed steps with an event-record node on a "
                     "side branch at each phase boundary")
        total_ms = phase_total * args.steps
    else:
        phase_ms, phase_total = eager_phase, eager_ms / args.steps
        phase_src = "eager launches with CUDA events at the phase boundaries"
        total_ms = graph_ms if graph_ms is not None else eager_ms
    tokens_total, total_ms_max, value = replica_throughput(world, float(c.T * args.steps),
                                                           total_ms)
    ms_per_step = total_ms_max / args.steps
    # clocks: of the run the GEMM time comes from (the phase graph, else the eager loop),
    # of the plain replay (`value`), and of the whole timed region
    clk_all = clocks.window(w0, w1)
    clk = clocks.window(w0, w_pg) if pg is not None else clk_all
    clk_graph = clk if pg is not None else (clocks.window(g0w, g1w) if g0w is not None
                                             else clk_all)

    res = {"workload": describe(c, mxfp8, fuse_gather, mx_cache)
                       + (" dispatch(dy)-fused-FC2-dgrad" if fuse_dispatch_bwd else ""),
           "tokens_per_step": c.T,
           "tokens_per_s": round(value, 1), "ms_per_step": round(ms_per_step, 4),
           "eager_ms_per_step": round(eager_ms / args.steps, 4),
           "graph_no_events_ms_per_step": (round(graph_ms / args.steps, 4)
                                            if graph_ms is not None else None),
           "rows_kept": rows_kept, "dropped": c.T * c.k - rows_kept,
           "phase_ms": {k: round(v, 4) for k, v in phase_ms.items()},
           "phase_ms_total": round(phase_total, 4), "phase_timing": phase_src,
           "launches_per_step": wl.launches_per_step(), "clocks": clk_all,
           "_tokens_total": tokens_total, "_clk_graph": clk_graph}
    if c.capacity:
        res["capacity"] = c.capacity
        res["load_histogram"] = {"counts": counts, "kept": kept}
    elif c.E <= 64:
        res["load_histogram"] = {"counts": counts}
    else:
        res["load"] = {"max": max(counts), "min": min(counts),
                       "mean": round(sum(counts) / len(counts), 1)}

    # ---- roofline of the grouped GEMMs
    if c.recompute:
        gemm_ms = phase_total      # the GEMMs are not separable from the two layer calls
    else:
        gemm_ms = phase_ms["ffn_fwd"] + phase_ms["ffn_bwd"]
    res["roofline"] = gemm_roofline(c, rows_kept, gemm_ms, peaks, peak_src, clk, mxfp8,
                                    gemm_clock)
    # ---- row movers against HBM (device times inside the replay)
    hbm = float(peaks["hbm_gbs"])
    mem = {}
    for ph, b in memory_bytes(c, rows_kept).items():
        if ph not in phase_ms:
            continue
        gbs = b / (phase_ms[ph] * 1e-3) / 1e9
        mem[ph] = {"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3),
                   "us": round(phase_ms[ph] * 1e3, 2), "bytes": b}
    mem["route_us"] = round(phase_ms.get("route", 0.0) * 1e3, 2)
    mem["note"] = (f"hbm_gbs {hbm} of {peak_src}; times from the {phase_src}: an interval "
                   f"runs from the completion of the phase before to this phase's completion")
    res["memory_kernels"] = mem
    if e2e and not args.no_e2e and not c.recompute:
        e_ms, h2d, d2h = wl.e2e(args.steps, args.warmup, world)
        e_ms = max_over_ranks(world, e_ms)
        res["e2e"] = {"value": round(tokens_total / (e_ms / 1e3), 1), "unit": "tokens/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def describe(c, mxfp8=0, fuse_gather=False, mx_cache=True) -> str:
    return (f"{c.name}: T={c.T} d={c.d} E={c.E} top-{c.k} {c.gate} f={c.f}"
            + (f" shared fs={c.fs}" if c.fs else "")
            + (f" capacity {c.capacity}" if c.capacity else "")
            + (" select-bias" if c.select_bias is not None else "")
            + (" drop-negative" if c.drop_negative else "")
            + (" drop-by-score" if c.drop_by_score else "")
            + (" recompute-FC1" if c.recompute else "")
            + (" gather-fused" if fuse_gather else "")
            + (" MXFP8 fwd+dgrad" if mxfp8 else "")
            + (" MXFP8 wgrad" if mxfp8 == 2 else "")
            + (" cached-weight-quant" if mxfp8 and mx_cache else ""))


def gemm_roofline(c, rows_kept, gemm_ms, peaks, peak_src, clk, mxfp8, gemm_clock=None) -> dict:
    """The grouped GEMMs of one step against their roofline.  bf16: each of the six
    launches takes at least the larger of its tensor time and its HBM time; where the HBM
    terms dominate (weight streaming) the GEMMs are graded on HBM bandwidth."""
    flops = gemm_flops(c, rows_kept)
    if c.recompute:   # FC1 again in the backward: 4*d*f per kept row (+ shared per token)
        flops += 4.0 * c.d * c.f * rows_kept + (4.0 * c.d * c.fs * c.T if c.fs else 0.0)
    gemm_s = gemm_ms / 1e3
    achieved = flops / gemm_s / 1e12
    peak, which, why = choose_peak(peaks, clk,
                                   gemm_clock["sm_mhz"] if gemm_clock else None)
    burst = float(peaks["bf16_tflops"])
    sus = float(peaks.get("bf16_tflops_sustained", burst))
    hbm = float(peaks["hbm_gbs"])
    out = {"kernel": ("whole step: GEMM flops incl. the recomputed FC1 over the step time"
                      if c.recompute else
                      "grouped_gemm (tcgen05; FC1, FC2, 2 dgrad, 2 wgrad per step)"
                      if not mxfp8 else
                      "grouped GEMMs: block-scaled MXFP8 (routed fwd + dgrad"
                      + (" + wgrad" if mxfp8 == 2 else "") + ") and bf16 (the rest)"),
           "gemm_flops_per_step": flops, "gemm_ms_per_step": round(gemm_ms, 4),
           "gemm_clock": gemm_clock}
    if mxfp8:
        # routed FC1 + FC2 and the two data gradients (12 d f per row), at level 2 the two
        # weight gradients (6 d f) too, run at the E4M3 rate; no E4M3 peak is measured here,
        # so it is taken as 2x the measured bf16 one (the nominal dense ratio 4.5 / 2.25)
        mx_fl = (18.0 if mxfp8 == 2 else 12.0) * c.d * c.f * rows_kept
        ideal = mx_fl / (2 * peak * 1e12) + (flops - mx_fl) / (peak * 1e12)
        pk = flops / ideal / 1e12
        out.update({"bound": "tensor", "achieved": round(achieved, 1), "peak": round(pk, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / pk, 4),
                    "peak_source": (f"flop-weighted: the MXFP8 GEMMs at 2x and the rest at 1x "
                                    f"of {why} ({peak_src}); the 2x E4M3 rate is the nominal "
                                    f"ratio, not a measured peak")})
        return out
    phases = gemm_phases(c, rows_kept)
    t_tensor = sum(fl / (peak * 1e12) for fl, _ in phases)
    t_hbm = sum(by / (hbm * 1e9) for _, by in phases)
    t_roof = sum(max(fl / (peak * 1e12), by / (hbm * 1e9)) for fl, by in phases)
    gbytes = sum(by for _, by in phases)
    per_launch = {"roofline_ms": round(t_roof * 1e3, 4),
                  "frac_of_roofline": round(t_roof / gemm_s, 4),
                  "tensor_ms": round(t_tensor * 1e3, 4), "hbm_ms": round(t_hbm * 1e3, 4)}
    if t_hbm > t_tensor:
        gbs = gbytes / gemm_s / 1e9
        out.update({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4),
                    "peak_source": f"hbm_gbs of {peak_src}",
                    "bytes_note": "algorithmic GEMM bytes (weights once per launch, activation "
                                  "rows once) over the GEMM time",
                    "tensor_achieved_tflops": round(achieved, 1),
                    "tensor_frac": round(achieved / peak, 4)})
    else:
        out.update({"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "peak_source": f"{why} ({peak_src})"})
    out.update({"peak_choice": which, "frac_of_burst": round(achieved / burst, 4),
                "frac_of_sustained": round(achieved / sus, 4), "per_launch_roofline": per_launch,
                "algorithmic_bytes_per_launch": round(gbytes / 6)})
    tr = GEMM_TRAFFIC_PER_LAUNCH.get(c.name) if not c.recompute else None
    out["traffic"] = tr[0] if tr else None
    out["traffic_note"] = (f"DRAM bytes per launch, average of the 6 GEMM launches (ncu on the "
                           f"{tr[1]} shape x4)" if tr else
                           "no ncu capture of this configuration's GEMMs")
    return out


# --------------------------------------------------------------------------- ours
def bench_ours(args, world, rank, local):
    import torch

    import token_dispatch_expert_gb300 as tde
    from workloads import CONFIGS, PROFILE_CONFIGS, gen_select_bias

    c = CONFIGS.get(args.config) or PROFILE_CONFIGS[args.config]
    if args.select_bias:
        c = c.replace(select_bias=gen_select_bias(c, args.select_bias))
    c = c.replace(drop_negative=args.drop_negative, recompute=args.recompute,
                  drop_by_score=args.drop_by_score)
    variant = (args.select_bias or args.drop_negative or args.recompute or args.drop_by_score
               or args.fuse_gather or args.mxfp8 or args.fuse_dispatch_bwd)
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    tde.lib()
    peaks, peak_src = load_peaks()
    clocks = ClockSampler(local)
    clocks.start()
    try:
        mx_level = (2 if args.mx_wgrad else 1) if args.mxfp8 else 0
        head = measure(c, args, dev, world, rank, clocks, peaks, peak_src, mxfp8=mx_level,
                       fuse_gather=args.fuse_gather, mx_cache=args.mx_cache_weights,
                       fuse_dispatch_bwd=args.fuse_dispatch_bwd)
        extra = {}
        if args.workloads == "auto":
            names = [] if variant or args.config != "mixtral" else EXTRA_WORKLOADS
        elif args.workloads == "none":
            names = []
        else:
            names = [n for n in args.workloads.split(",") if n]
        for n in names:
            r = measure(CONFIGS[n], args, dev, world, rank, clocks, peaks, peak_src)
            r.pop("_tokens_total"); r.pop("_clk_graph")
            extra[n] = r
        mx_block = None
        if not args.no_mx and not variant and args.config == "mixtral" and \
                args.workloads != "none":
            # the headline layer and the capacity layer, each with MXFP8 forward and data
            # gradients (level 1) and with MXFP8 weight gradients too (level 2)
            mx_block = {}
            for mc_name, mc_cfg in (("mixtral", c), ("capacity", CONFIGS["capacity"])):
                for lvl in (1, 2):
                    r = measure(mc_cfg, args, dev, world, rank, clocks, peaks, peak_src,
                                mxfp8=lvl)
                    r.pop("_tokens_total"); r.pop("_clk_graph")
                    key = "fwd_dgrad" if lvl == 1 else "fwd_dgrad_wgrad"
                    mx_block[key if mc_name == "mixtral" else f"{mc_name}_{key}"] = r
    finally:
        clocks.stop()

    clk = head["_clk_graph"]
    line = {
        "metric": "MoE layer fwd+bwd tokens/s on 1 GB300",
        "value": head["tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": (("mxfp8 (routed fwd + dgrad + wgrad) + bf16 shared" if args.mx_wgrad else
                   "mxfp8 (routed fwd + dgrad) + bf16") if args.mxfp8 else "bf16"),
        "data": "synthetic (seeded N(0,1) tokens/logits, N(0,0.02) bf16 weights)",
        "config": {"workload": head["workload"], "tokens_per_step": c.T,
                   "rows_kept": head["rows_kept"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": (f"no flush: each step's GEMMs alone stream "
                          f"{sum(b for _, b in gemm_phases(c, head['rows_kept'])) / 1e9:.1f} "
                          f"GB of weights, gradients and activations (L2 is 129 MB)")},
        "roofline": head["roofline"],
        "timing": ("`steps` steps captured as one CUDA graph with an event-record node on a "
                   "side branch at each phase boundary (the kernels keep their own chain), "
                   "replayed once on the launching stream: value, phase split, GEMM time and "
                   "clocks from that replay" if not args.no_graph else
                   "eager launches between CUDA events on the launching stream"),
        "eager_ms_per_step": head["eager_ms_per_step"],
        "graph_no_events_ms_per_step": head["graph_no_events_ms_per_step"],
        "e2e": head.get("e2e"),
        "permute_gbs": head["memory_kernels"].get("permute", {}).get("GB/s"),
        "memory_kernels": head["memory_kernels"],
        "phase_ms": head["phase_ms"],
        "phase_ms_total": head["phase_ms_total"],
        "gpu_launches": head["launches_per_step"] * args.steps,
        "clocks": clk,
        "workloads": extra or None,
        "mxfp8": mx_block,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ot = OracleTimer(c)
        m = ot.measure(args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(m["tokens_per_s"], 4), "unit": "tokens/s",
                                "cores": ot.threads, "kind": "oracle",
                                "extrapolated": m["extrapolated"],
                                "seconds_per_step": round(m["seconds_per_step"], 2),
                                "sample": ot.describe(m),
                                "parts_s": {k: round(v, 3) for k, v in m["parts_s"].items()},
                                "ffn_s": round(m["ffn_s"], 2),
                                "ffn_fit": m["ffn_fit"]}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def bench_reference(args, world, rank, local):
    """The CPU oracle timed on the host cores (rank 0 only): each step times routing,
    permute, combine, the combine backward and the reduce on every token and the expert FFN
    on its row samples, and extrapolates the FFN to the whole layer."""
    from workloads import CONFIGS
    if rank != 0:
        return None
    c = CONFIGS[args.config]
    ot = OracleTimer(c)
    budget = max(2.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    # the per-expert fixed cost is fitted once; each step then times one FFN sample
    first = ot.measure(budget)
    a = first["ffn_fit"]["a_s"] if first["extrapolated"] else None
    for _ in range(max(0, args.warmup - 1)):
        ot.measure(budget, a)
    ms = [ot.measure(budget, a) for _ in range(args.steps)]
    ms.sort(key=lambda m: m["seconds_per_step"])
    m = ms[len(ms) // 2]
    value = m["tokens_per_s"]
    return {
        "impl": "reference",
        "metric": "MoE layer fwd+bwd tokens/s on 1 GB300",
        "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(m["seconds_per_step"] * 1e3, 1),
        "ms_per_step_extrapolated": m["extrapolated"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": describe(c), "tokens_per_step": c.T},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": ot.threads,
                         "kind": "oracle", "extrapolated": m["extrapolated"],
                         "sample": "each step: " + ot.describe(m)
                                   + "; the median step is reported"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="mixtral")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="time budget of the oracle's expert FFN in the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the eager launches instead of a CUDA-graph replay of the step")
    ap.add_argument("--workloads", default="auto",
                    help="extra workloads measured beside the headline: auto (tiny, qwen3, "
                         "dsv3, capacity for the default Mixtral run), none, or a comma list")
    ap.add_argument("--no-mx", action="store_true", help="skip the MXFP8 block")
    ap.add_argument("--select-bias", type=float, default=0.0,
                    help="std of a seeded per-expert selection-only bias (0: none)")
    ap.add_argument("--drop-negative", action="store_true",
                    help="drop selections whose raw logit is negative")
    ap.add_argument("--fuse-gather", action="store_true",
                    help="fold the permute into the FC1 and dW1 operand loads")
    ap.add_argument("--fuse-dispatch-bwd", action="store_true",
                    help="the FC2 data-gradient reads dy through src_tok, scaled by the gate "
                         "weight in its epilogue")
    ap.add_argument("--mxfp8", action="store_true",
                    help="routed experts' forward and data-gradient GEMMs on MXFP8 operands "
                         "(weight gradients bf16)")
    ap.add_argument("--mx-wgrad", action="store_true",
                    help="with --mxfp8: the weight gradients on MXFP8 operands too, quantised "
                         "along each expert segment's tokens")
    ap.add_argument("--mx-cache-weights", action="store_true",
                    help="with --mxfp8: quantise the weights once, outside the timed steps")
    ap.add_argument("--drop-by-score", action="store_true",
                    help="an expert over capacity keeps its best-scored assignments")
    ap.add_argument("--recompute", action="store_true",
                    help="backward recomputes FC1 instead of saving its outputs")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = bench_reference(args, world, rank, local)
    else:
        line = bench_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
