"""Benchmark of the single-GPU MoE layer (forward + backward) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one forward + backward of the MoE layer over one batch of T tokens:
route -> permute -> grouped FC1/SwiGLU/FC2 -> (shared expert) -> combine, then
combine/gate backward -> FC2 data-grad + SwiGLU backward -> FC2 weight-grad ->
FC1 data-grad -> FC1 weight-grad -> un-permute reduce.  The default workload is the
Mixtral-style layer (T=4096, d=4096, E=8, top-2, f=14336) on synthetic seeded
inputs.  The metric is tokens/s of the whole step; the dominant kernel (the tcgen05
grouped GEMM, six launches per step) is also reported against the measured bf16
tensor peak.

With N > 1 (torchrun) every rank runs an independent replica of the layer (the path
does not shard: replicas only); the reported value is the sum over ranks, the time
the max over ranks.

--impl reference times the CPU oracle (the plain double-precision C reference of the
layer) on the host cores, on a bounded sample of the same workload.
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
# the Qwen3 layer.  Valid for the grouped-GEMM kernel as of the transposed-epilogue version;
# set to None when the kernel changes.
GEMM_TRAFFIC_PER_LAUNCH = {
    "mixtral": (4 * (658.7 + 340.1 + 490.5 + 252.5 + 671.2 + 544.8) / 6 * 1e6, "mixtral_e2"),
    "qwen3": (4 * (325.9 + 163.5 + 242.9 + 143.4 + 300.6 + 261.7) / 6 * 1e6, "qwen3_e32"),
}


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


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

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
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


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
    """The CPU oracle's full forward + backward (routing, expert FFN with both weight
    gradients, combine, all in float64) on the first t tokens of the workload, with the
    workload's d, f, E, k, gate and capacity rule.  Inputs come from the host generators
    and are built once.

    Workloads whose float64 weights and weight gradients for all E experts exceed
    MEM_BUDGET (DeepSeek-V3: about 90 GB) run the sample on the experts its tokens route
    to: the logits restricted to those experts' columns (kept in expert order) select the
    same top-k with the same gate weights, because both gates (softmax renormalised over
    the top-k, sigmoid normalised over the selected) depend only on the selected logits.
    Their weights are drawn per expert from the same N(0, 0.02^2) bf16 distribution."""

    MEM_BUDGET = 32 << 30

    def __init__(self, c):
        import oracle
        from workloads import WEIGHT_STD, gen_bf16, gen_logits, weight_shapes

        oracle.build()
        self.c = c
        self.threads = oracle.threads()     # what its OpenMP loops run on
        self.logits = gen_logits(c)
        self.x = gen_bf16(c, "x", (c.T, c.d))
        self.dy = gen_bf16(c, "dy", (c.T, c.d))
        per_expert = 2 * 3 * c.d * c.f * 8          # weights + weight gradients, float64
        self.restrict = c.cap_factor is None and c.E * per_expert > self.MEM_BUDGET
        self.max_experts = max(c.k, self.MEM_BUDGET // per_expert)
        self.W = {}
        self._expert_w = {}
        for n, shape in weight_shapes(c).items():
            if self.restrict and n in ("W1", "W2"):
                continue
            self.W[n] = oracle.layer._f64(gen_bf16(c, n, shape, WEIGHT_STD))

    def _experts(self, t: int):
        import numpy as np
        import oracle
        r = oracle.route(self.c.replace(T=t), self.logits[:t])
        return np.unique(r["topk_idx"])

    def _inputs(self, t: int):
        import numpy as np
        import oracle
        from workloads import WEIGHT_STD, gen_bf16
        c = self.c
        inp = {"logits": self.logits[:t], "x": self.x[:t], "dy": self.dy[:t]}
        inp.update(self.W)
        if not self.restrict:
            return c.replace(T=t), inp
        used = self._experts(t)
        for e in used:
            if e not in self._expert_w:
                self._expert_w[e] = tuple(
                    oracle.layer._f64(gen_bf16(c, f"{n}[{e}]", shape, WEIGHT_STD))
                    for n, shape in (("W1", (2 * c.f, c.d)), ("W2", (c.d, c.f))))
        inp["logits"] = np.ascontiguousarray(self.logits[:t][:, used])
        inp["W1"] = np.stack([self._expert_w[e][0] for e in used])
        inp["W2"] = np.stack([self._expert_w[e][1] for e in used])
        sub = c.replace(T=t, E=len(used))
        if getattr(c, "select_bias", None) is not None:
            sub = sub.replace(select_bias=np.ascontiguousarray(c.select_bias[used]))
        return sub, inp

    def run(self, t: int) -> float:
        import oracle
        sub, inp = self._inputs(t)
        t0 = time.perf_counter()
        fo = oracle.layer_fwd(sub, inp)
        oracle.layer_bwd(sub, inp, fo)
        return time.perf_counter() - t0

    def max_tokens(self) -> int:
        """The largest sample whose experts fit MEM_BUDGET (all T when unrestricted)."""
        if not self.restrict:
            return self.c.T
        t = 1
        while t < self.c.T and len(self._experts(t + 1)) <= self.max_experts:
            t += 1
        return t

    def calibrate(self, budget_s: float) -> int:
        """Token count whose run takes about budget_s seconds: fit time = a + b*t from two
        probes (the weight-gradient buffers give the oracle a cost independent of t)."""
        t_max = self.max_tokens()
        t1, t2 = min(2, t_max), min(6, t_max)
        if t2 <= t1:
            return t_max
        d1, d2 = self.run(t1), self.run(t2)
        b = max((d2 - d1) / (t2 - t1), 1e-6)
        a = max(d1 - b * t1, 0.0)
        t = int((budget_s - a) / b) if budget_s > a else t2
        return int(min(t_max, max(t2, t)))


# --------------------------------------------------------------------------- ours
def bench_ours(args, world, rank, local):
    import numpy as np
    import torch

    import token_dispatch_expert_gb300 as tde
    from workloads import CONFIGS, PROFILE_CONFIGS, gen_inputs_device, gen_select_bias

    c = CONFIGS.get(args.config) or PROFILE_CONFIGS[args.config]
    if args.select_bias:
        c = c.replace(select_bias=gen_select_bias(c, args.select_bias))
    c = c.replace(drop_negative=args.drop_negative, recompute=args.recompute,
                  drop_by_score=args.drop_by_score)
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    tde.lib()
    bias_t = (torch.tensor(c.select_bias, dtype=torch.float32, device=dev)
              if c.select_bias is not None else None)
    cfg = tde.make_config(c.T, c.d, c.E, c.k, c.f, c.fs, c.gate, c.route_scale, c.capacity,
                          select_bias=bias_t, drop_negative=c.drop_negative,
                          recompute=c.recompute, drop_by_score=c.drop_by_score,
                          mxfp8=(2 if args.mx_wgrad else 1) if args.mxfp8 else 0)
    g = gen_inputs_device(c, dev, seed=rank)
    R = c.T * c.k
    ws_b, ctx_b = tde.moe_workspace_size(cfg)
    ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
    ctx = torch.empty(ctx_b, dtype=torch.uint8, device=dev)
    tde.moe_ws_init(ws)
    v = tde.ctx_views(cfg, ctx)
    bf = dict(dtype=torch.bfloat16, device=dev)
    y = torch.empty((c.T, c.d), **bf)
    dyp = torch.empty((R, c.d), **bf)
    dab = torch.empty((R, 2 * c.f), **bf)
    dxp = torch.empty((R, c.d), **bf)
    dx = torch.empty((c.T, c.d), **bf)
    dW1 = torch.empty_like(g["W1"])
    dW2 = torch.empty_like(g["W2"])
    dl = torch.empty((c.T, c.E), dtype=torch.float32, device=dev)
    shared = None
    if c.fs:
        # the shared expert as a one-group grouped FFN over all T tokens
        s_cfg = tde.make_config(c.T, c.d, 1, 1, c.fs)
        s_off = torch.tensor([0, c.T], dtype=torch.int32, device=dev)
        shared = dict(cfg=s_cfg, off=s_off, ab=torch.empty((c.T, 2 * c.fs), **bf),
                      h=torch.empty((c.T, c.fs), **bf), ys=torch.empty((c.T, c.d), **bf),
                      dab=torch.empty((c.T, 2 * c.fs), **bf), dx=torch.empty((c.T, c.d), **bf),
                      dW1=torch.empty_like(g["W1s"]), dW2=torch.empty_like(g["W2s"]))
    stream = torch.cuda.current_stream(dev)
    PHASES = ["route", "permute", "ffn_fwd", "combine", "combine_bwd", "ffn_bwd",
              "unpermute_reduce"]
    if c.recompute:
        # FC1 is recomputed inside the backward: the step runs through the two whole-layer
        # calls, timed as two phases
        PHASES = ["layer_fwd", "layer_bwd"]
        l_outs = {"dx": dx, "dW1": dW1, "dW2": dW2, "dlogits": dl}
        if shared:
            l_outs["dW1s"] = shared["dW1"]; l_outs["dW2s"] = shared["dW2"]

    def step_layer(ev):
        if ev is not None:
            ev[0].record(stream)
        tde.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W2"], g.get("W1s"),
                          g.get("W2s"), y, ctx, ws)
        if ev is not None:
            ev[1].record(stream)
        tde.moe_layer_bwd(cfg, ctx, g["logits"], g["x"], g["dy"], g["W1"], g["W2"],
                          g.get("W1s"), g.get("W2s"), dx, dW1, dW2, l_outs.get("dW1s"),
                          l_outs.get("dW2s"), dl, ws)
        if ev is not None:
            ev[2].record(stream)

    if args.mxfp8:
        # the routed experts' forward in MXFP8; the weights are re-quantised every step
        # (the conservative case: no reuse across micro-batches), timed as their own phase
        PHASES = ["mx_weight_quant"] + PHASES
        nbytes, _ = tde.moe_mx_weights_size(cfg)
        wq = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        u8 = dict(dtype=torch.uint8, device=dev)
        # the activation scales are atoms tiled by 128 rows per expert segment: sized by
        # the library, not by rows x K/32
        mxb = dict(xq=torch.empty((R, c.d), **u8),
                   xs=torch.empty(tde.moe_mx_act_scales_size(cfg, c.d), **u8),
                   hq=torch.empty((R, c.f), **u8),
                   hs=torch.empty(tde.moe_mx_act_scales_size(cfg, c.f), **u8))
        if args.mx_cache_weights:
            # weight-quantisation caching: the blob is made once, as when one optimizer
            # step's weights serve many micro-batches
            tde.moe_mx_quantize_weights(cfg, g["W1"], g["W2"], wq)

    def step(ev):
        if c.recompute:
            return step_layer(ev)
        # ev: len(PHASES) + 1 events recorded at the phase boundaries (or None)
        n_mark = [0]

        def mark():
            if ev is not None:
                ev[n_mark[0]].record(stream)
            n_mark[0] += 1
        mark()
        if args.mxfp8:
            if not args.mx_cache_weights:
                tde.moe_mx_quantize_weights(cfg, g["W1"], g["W2"], wq)
            mark()
        tde.moe_route(cfg, g["logits"], v["topk_idx"], v["topk_w"], v["counts"], v["kept"],
                      v["offsets"], v["dest_row"], v["src_tok"], v["src_slot"], v["drop_mask"],
                      ws)
        mark()
        if args.mxfp8:         # permute + quantise (bf16 xp kept for the backward)
            tde.moe_mx_permute_quant(cfg, g["x"], v["src_tok"], v["offsets"], v["xp"],
                                     mxb["xq"], mxb["xs"], ws)
            mark()
            tde.moe_grouped_ffn_mx(cfg, mxb["xq"], mxb["xs"], v["offsets"], wq, v["ab"], v["h"],
                                   mxb["hq"], mxb["hs"], v["yp"], ws)
        elif args.fuse_gather:   # the permute folded into FC1's loads: no xp
            mark()
            tde.moe_grouped_ffn_gather(cfg, g["x"], v["src_tok"], v["offsets"], g["W1"],
                                       g["W2"], v["ab"], v["h"], v["yp"], ws)
        else:
            tde.moe_permute(cfg, g["x"], v["src_tok"], v["offsets"], v["xp"], ws)
            mark()
            tde.moe_grouped_ffn(cfg, v["xp"], v["offsets"], g["W1"], g["W2"], v["ab"], v["h"],
                                v["yp"], ws)
        if shared:
            tde.moe_grouped_ffn(shared["cfg"], g["x"], shared["off"], g["W1s"], g["W2s"],
                                shared["ab"], shared["h"], shared["ys"], ws)
        mark()
        tde.moe_combine(cfg, v["yp"], v["dest_row"], v["topk_w"],
                        shared["ys"] if shared else None, y, ws)
        mark()
        tde.moe_combine_bwd(cfg, g["dy"], v["yp"], g["logits"], v["topk_idx"], v["topk_w"],
                            v["dest_row"], dyp, dl, ws)
        mark()
        if args.mxfp8:   # the data-gradient GEMMs on MXFP8 operands (with --mx-wgrad the
            #              weight gradients too, else bf16)
            tde.moe_grouped_ffn_bwd_mx(cfg, dyp, v["xp"], v["offsets"], wq, v["ab"], v["h"], dab,
                                       dxp, dW1, dW2, ws)
        elif args.fuse_gather:
            tde.moe_grouped_ffn_bwd_gather(cfg, dyp, g["x"], v["src_tok"], v["offsets"], g["W1"],
                                           g["W2"], v["ab"], v["h"], dab, dxp, dW1, dW2, ws)
        else:
            tde.moe_grouped_ffn_bwd(cfg, dyp, v["xp"], v["offsets"], g["W1"], g["W2"], v["ab"],
                                    v["h"], dab, dxp, dW1, dW2, ws)
        if shared:
            tde.moe_grouped_ffn_bwd(shared["cfg"], g["dy"], g["x"], shared["off"], g["W1s"],
                                    g["W2s"], shared["ab"], shared["h"], shared["dab"],
                                    shared["dx"], shared["dW1"], shared["dW2"], ws)
        mark()
        tde.moe_unpermute_reduce(cfg, dxp, v["dest_row"], shared["dx"] if shared else None,
                                 dx, ws)
        mark()

    # route 3, permute 1, FC1+FC2 2, combine 1, combine-bwd 1, backward GEMMs 4 plus the two
    # per-segment map preparations, reduce 1; the shared expert 2 + 4
    launches_per_step = 3 + 1 + 2 + 1 + 1 + 6 + 1 + (6 if shared else 0)
    if args.fuse_gather:
        launches_per_step -= 1
    if c.recompute:
        launches_per_step += 1 + (1 if shared else 0)   # the recomputed FC1
    if c.drop_by_score and c.capacity > 0:
        launches_per_step += 2                          # score scatter + select
    if args.mxfp8:
        launches_per_step += 1                          # dyp quantised for the data gradients
    if args.mxfp8 and args.mx_wgrad:
        launches_per_step += 2                          # 4 along-token quantisations replace
        #                                                 the 2 per-segment map preparations
    if args.mxfp8 and not args.mx_cache_weights:
        launches_per_step += 4                          # the four weight-quantisation kernels
    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    st, fl = tde.moe_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {tde.moe_status_string(st)} {fl:#x}")
    rows_kept = int(v["offsets"][-1].item())

    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    step_events = []
    for i in range(args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(PHASES) + 1)]
        step(ev)   # events are read back after the loop (no host sync inside it)
        step_events.append(ev)
    t_end.record(stream)
    torch.cuda.synchronize()
    eager_ms = t_start.elapsed_time(t_end)
    graph_ms = None
    if not args.no_graph:
        # the same step captured once as a CUDA graph and replayed: the kernels and their
        # order are identical, only the host launch gaps between them go away
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph):
            step(None)
        gph.replay()
        torch.cuda.synchronize()
        barrier(world)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for i in range(args.steps):
            gph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1)
    barrier(world)
    clk = clocks.stop()
    total_ms = graph_ms if graph_ms is not None else eager_ms
    phase_ms = {ph: 0.0 for ph in PHASES}
    for ev in step_events:
        for i, ph in enumerate(PHASES):
            phase_ms[ph] += ev[i].elapsed_time(ev[i + 1]) / args.steps
    if c.recompute:   # the GEMMs are not separable from the rest of the two layer calls
        gemm_ms = eager_ms
    else:
        gemm_ms = (phase_ms["ffn_fwd"] + phase_ms["ffn_bwd"]) * args.steps
    st, fl = tde.moe_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after timing: {tde.moe_status_string(st)} {fl:#x}")

    tokens_total, total_ms_max, value = replica_throughput(world, float(c.T * args.steps),
                                                           total_ms)
    ms_per_step = total_ms_max / args.steps

    e2e_value = None
    h2d = d2h = 0
    if not args.no_e2e:
        # End to end through the public whole-layer API with host buffers in pinned memory,
        # the way a training loop streams them: every step copies its inputs (logits, x,
        # dy) host -> device and its results (y, dx, dlogits) device -> host, on a copy
        # stream, double-buffered so that step i+1's inputs and step i's results move
        # while the GPU computes.  All copies fall inside the timed region.
        layer = tde.MoELayer(cfg, device=dev)
        h_logits = g["logits"].cpu().pin_memory()
        h_x = g["x"].cpu().pin_memory()
        h_dy = g["dy"].cpu().pin_memory()
        h_y = torch.empty((c.T, c.d), dtype=torch.bfloat16).pin_memory()
        h_dx = torch.empty((c.T, c.d), dtype=torch.bfloat16).pin_memory()
        h_dl = torch.empty((c.T, c.E), dtype=torch.float32).pin_memory()
        bufs = []
        for b in range(2):
            o = {"dx": torch.empty_like(dx), "dW1": dW1, "dW2": dW2,
                 "dlogits": torch.empty_like(dl)}
            if shared:
                o["dW1s"] = shared["dW1"]; o["dW2s"] = shared["dW2"]
            bufs.append({"logits": torch.empty_like(g["logits"]), "x": torch.empty_like(g["x"]),
                         "dy": torch.empty_like(g["dy"]), "y": torch.empty_like(y), "out": o})
        # one copy stream per direction: a step's inputs come in while the previous step's
        # results go out (the two directions have their own copy engines)
        in_stream = torch.cuda.Stream(device=dev)
        out_stream = torch.cuda.Stream(device=dev)
        ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "done", "copied")}

        def copy_in(b):
            with torch.cuda.stream(in_stream):
                bufs[b]["logits"].copy_(h_logits, non_blocking=True)
                bufs[b]["x"].copy_(h_x, non_blocking=True)
                bufs[b]["dy"].copy_(h_dy, non_blocking=True)
                ev["in"][b].record(in_stream)

        def e2e_run(n):
            copy_in(0)
            for i in range(n):
                b = i & 1
                B = bufs[b]
                stream.wait_event(ev["in"][b])
                if i >= 2:
                    stream.wait_event(ev["copied"][b])   # step i-2's results are on the host
                if args.mxfp8:
                    if not args.mx_cache_weights:
                        tde.moe_mx_quantize_weights(cfg, g["W1"], g["W2"], wq)
                    layer.forward_mx(B["logits"], B["x"], wq, g.get("W1s"), g.get("W2s"),
                                     y=B["y"])
                    layer.backward_mx(B["logits"], B["x"], B["dy"], wq, g.get("W1s"),
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

        e2e_run(max(1, args.warmup))
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(world, e0.elapsed_time(e1))
        e2e_value = tokens_total / (e2e_ms / 1e3)
        h2d = h_logits.numel() * 4 + h_x.numel() * 2 + h_dy.numel() * 2
        d2h = h_y.numel() * 2 + h_dx.numel() * 2 + h_dl.numel() * 4

    peaks, peak_src = load_peaks()
    flops = gemm_flops(c, rows_kept)
    if c.recompute:   # FC1 again in the backward: 4*d*f per kept row (+ shared per token)
        flops += 4.0 * c.d * c.f * rows_kept + (4.0 * c.d * c.fs * c.T if c.fs else 0.0)
    gemm_s_per_step = gemm_ms / args.steps / 1e3
    achieved = flops / gemm_s_per_step / 1e12
    # the GEMMs run inside a continuous loop of steps (the power cap engages): the sustained
    # measured peak is the denominator; the burst fraction is reported beside it
    peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    burst = float(peaks["bf16_tflops"])
    mx_line = None
    if args.mxfp8:
        # the forward's routed GEMMs run at the E4M3 rate: 2x the measured bf16 peak (the
        # nominal dense ratio 4.5 / 2.25 PFLOP/s).  The step's ideal GEMM time is the sum of
        # the forward (at that rate) and everything else (bf16); the peak reported is the
        # flop rate that ideal time stands for.
        # routed FC1 + FC2 (6 d f per row) and the two data gradients (6 d f per row) run at
        # the E4M3 rate, with --mx-wgrad the two weight gradients (6 d f per row) too; the
        # rest (bf16 weight gradients, the shared expert) at the bf16 rate
        fwd_mx = (18.0 if args.mx_wgrad else 12.0) * c.d * c.f * rows_kept
        ideal_s = fwd_mx / (2 * peak * 1e12) + (flops - fwd_mx) / (peak * 1e12)
        ideal_b = fwd_mx / (2 * burst * 1e12) + (flops - fwd_mx) / (burst * 1e12)
        # (the ffn_fwd phase also holds the bf16 shared expert when there is one)
        mx_line = {"ffn_fwd_tflops": None if c.fs else
                   round(6.0 * c.d * c.f * rows_kept / (phase_ms["ffn_fwd"] * 1e-3) / 1e12,
                         1),
                   "fp8_peak_sustained": 2 * peak, "fp8_peak_burst": 2 * burst,
                   "weight_quant_ms": round(phase_ms["mx_weight_quant"], 4),
                   "note": ("weights quantised once before timing (cached)"
                            if args.mx_cache_weights else
                            "weights re-quantised every step (included in value)")}
        peak = round(flops / ideal_s / 1e12, 1)
        burst = round(flops / ideal_b / 1e12, 1)
    # per-launch roofline (bf16): each GEMM launch takes at least the larger of its tensor
    # time and its HBM time; where the HBM terms dominate (weight streaming, e.g. 256 small
    # experts) the GEMMs are graded on HBM bandwidth instead of the tensor peak
    roof = None
    if not args.mxfp8 and not c.recompute:
        hbm_peak = float(peaks["hbm_gbs"])
        phases = gemm_phases(c, rows_kept)
        t_tensor = sum(fl / (peak * 1e12) for fl, _ in phases)
        t_hbm = sum(by / (hbm_peak * 1e9) for _, by in phases)
        t_roof = sum(max(fl / (peak * 1e12), by / (hbm_peak * 1e9)) for fl, by in phases)
        gbytes = sum(by for _, by in phases)
        roof = {"roofline_ms": round(t_roof * 1e3, 4),
                "frac_of_roofline": round(t_roof / gemm_s_per_step, 4),
                "tensor_ms": round(t_tensor * 1e3, 4), "hbm_ms": round(t_hbm * 1e3, 4),
                "hbm_bound": t_hbm > t_tensor, "gemm_bytes": gbytes,
                "gemm_gbs": round(gbytes / gemm_s_per_step / 1e9, 1)}
    # measured DRAM traffic of the bf16 grouped GEMMs (the MXFP8 and recompute runs launch
    # other kernels, which have no capture here)
    traffic = (GEMM_TRAFFIC_PER_LAUNCH.get(c.name) if not args.mxfp8 and not c.recompute
               else None)
    # algorithmic bytes of the HBM-bound steps (each source row read once, each
    # destination row written once, index arrays counted)
    T_, d_, k_, E_ = c.T, c.d, c.k, c.E
    Rk = rows_kept
    mem_bytes = {
        "permute": (T_ + Rk) * d_ * 2 + Rk * 4,
        "combine": (Rk + T_ + (T_ if c.fs else 0)) * d_ * 2 + T_ * k_ * 8,
        "combine_bwd": (T_ + 2 * Rk) * d_ * 2 + T_ * E_ * 4 + T_ * k_ * 12,
        "unpermute_reduce": (Rk + T_ + (T_ if c.fs else 0)) * d_ * 2 + T_ * k_ * 4,
    }
    hbm = float(peaks["hbm_gbs"])
    mem = {}
    for ph, b in mem_bytes.items():
        if ph not in phase_ms:
            continue
        gbs = b / (phase_ms[ph] * 1e-3) / 1e9
        mem[ph] = {"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3),
                   "us": round(phase_ms[ph] * 1e3, 2), "bytes": b}
    line = {
        "metric": "MoE layer fwd+bwd tokens/s on 1 GB300",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": (("mxfp8 (routed fwd + dgrad + wgrad) + bf16 shared" if args.mx_wgrad else
                   "mxfp8 (routed fwd + dgrad) + bf16") if args.mxfp8 else "bf16"),
        "data": "synthetic (seeded N(0,1) tokens/logits, N(0,0.02) bf16 weights)",
        "config": {"workload": f"{c.name}: T={c.T} d={c.d} E={c.E} top-{c.k} "
                               f"{c.gate} f={c.f}" + (f" shared fs={c.fs}" if c.fs else "")
                               + (f" capacity {c.capacity}" if c.capacity else "")
                               + (f" select-bias N(0,{args.select_bias}^2)"
                                  if args.select_bias else "")
                               + (" drop-negative" if c.drop_negative else "")
                               + (" drop-by-score" if c.drop_by_score else "")
                               + (" recompute-FC1" if c.recompute else "")
                               + (" MXFP8-forward" if args.mxfp8 else "")
                               + (" MXFP8-wgrad" if args.mxfp8 and args.mx_wgrad else "")
                               + (" cached-weight-quant" if args.mxfp8 and args.mx_cache_weights
                                  else ""),
                   "tokens_per_step": c.T, "rows_kept": rows_kept,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": (f"no flush: each step's GEMMs alone stream "
                          f"{sum(b for _, b in gemm_phases(c, rows_kept)) / 1e9:.1f} GB of "
                          f"weights, gradients and activations (L2 is 129 MB)")},
        "roofline": {"kernel": ("whole step, GEMM flops incl. the recomputed FC1 over the "
                                "step time" if c.recompute else
                                "grouped_gemm (tcgen05; FC1, FC2, 2 dgrad, 2 wgrad per step)"),
                     **({"bound": "hbm", "achieved": roof["gemm_gbs"],
                         "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": round(roof["gemm_gbs"] / float(peaks["hbm_gbs"]), 4),
                         "bytes_note": "algorithmic GEMM bytes (weights once per launch, "
                                       "activation rows once) over the GEMM time; "
                                       f"hbm_gbs of {peak_src}",
                         "tensor_achieved_tflops": round(achieved, 1),
                         "tensor_frac": round(achieved / peak, 4)}
                        if roof is not None and roof["hbm_bound"] else
                        {"bound": "tensor", "achieved": round(achieved, 1),
                         "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4)}),
                     "frac_of_burst": round(achieved / burst, 4),
                     **({} if roof is None else {
                         "per_launch_roofline": {k2: v2 for k2, v2 in roof.items()
                                                 if k2 not in ("gemm_bytes",)}}),
                     "peak_source": (f"bf16_tflops_sustained of {peak_src} (kernel timed "
                                     f"inside a continuous step loop); burst {burst}"
                                     if not args.mxfp8 else
                                     f"flop-weighted: routed FC1, FC2, data gradients"
                                     f"{' and weight gradients' if args.mx_wgrad else ''} at "
                                     f"2x, the rest at 1x bf16_tflops_sustained of "
                                     f"{peak_src}; burst {burst}"),
                     "traffic": traffic[0] if traffic else None,
                     "traffic_note": (f"DRAM bytes per launch, average of the 6 GEMM launches "
                                      f"(ncu on the {traffic[1]} shape x4)" if traffic else
                                      "no ncu capture of this configuration's GEMMs"),
                     "algorithmic_bytes_per_launch": round(
                         gemm_algorithmic_bytes(c, rows_kept) / 6),
                     "gemm_ms_per_step": round(gemm_ms / args.steps, 4),
                     "gemm_share_of_step": round(gemm_ms / eager_ms, 4)},
        "timing": ("one step captured as a CUDA graph, replayed `steps` times between CUDA "
                   "events on the launching stream" if graph_ms is not None else
                   "eager launches between CUDA events on the launching stream"),
        "eager_ms_per_step": round(eager_ms / args.steps, 4),
        "mxfp8": mx_line,
        "e2e": None if e2e_value is None else {
            "value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h},
        "permute_gbs": mem["permute"]["GB/s"] if "permute" in mem else None,
        "memory_kernels": dict(mem, hbm_peak_gbs=hbm,
                               note=f"hbm_gbs of {peak_src}; CUDA events per phase, live"),
        "phase_ms": {k2: round(v2, 4) for k2, v2 in phase_ms.items()},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ot = OracleTimer(c)
        t = ot.calibrate(args.cpu_seconds)
        dt = ot.run(t)
        rate = t / dt
        line["cpu_baseline"] = {"value": round(rate, 3), "unit": "tokens/s", "cores": ot.threads,
                                "kind": "oracle",
                                "sample": f"full fwd+bwd of the first {t} tokens of the "
                                          f"workload ({dt:.1f} s, float64 C oracle, OpenMP)"
                                          + (", on the experts they route to"
                                             if ot.restrict else "")}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


def bench_reference(args, world, rank, local):
    """The CPU oracle timed on the host cores (rank 0 only)."""
    from workloads import CONFIGS
    if rank != 0:
        return None
    c = CONFIGS[args.config]
    ot = OracleTimer(c)
    # size each step so that warm-up + steps end within a few minutes
    budget = max(2.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    t = ot.calibrate(budget)
    for _ in range(args.warmup):
        ot.run(t)
    times = [ot.run(t) for _ in range(args.steps)]
    sec_per_token = sorted(times)[len(times) // 2] / t
    value = 1.0 / sec_per_token
    thr = ot.threads
    return {
        "impl": "reference",
        "metric": "MoE layer fwd+bwd tokens/s on 1 GB300",
        "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec_per_token * c.T * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{c.name}: T={c.T} d={c.d} E={c.E} top-{c.k} f={c.f}",
                   "tokens_per_step": c.T},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": thr,
                         "kind": "oracle",
                         "sample": f"each step: full fwd+bwd of the first {t} tokens"
                                   + (", on the experts they route to" if ot.restrict else "")},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="mixtral")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the eager launches instead of a CUDA-graph replay of the step")
    ap.add_argument("--select-bias", type=float, default=0.0,
                    help="std of a seeded per-expert selection-only bias (0: none)")
    ap.add_argument("--drop-negative", action="store_true",
                    help="drop selections whose raw logit is negative")
    ap.add_argument("--fuse-gather", action="store_true",
                    help="fold the permute into the FC1 and dW1 operand loads")
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
