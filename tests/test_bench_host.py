"""Host-side logic of bench.py: the per-launch GEMM flops and bytes, the choice of the
tensor peak from the sampled clocks, the clock window summary, and the CPU baseline's
oracle timing (in full where it fits, extrapolated from row samples otherwise)."""

import numpy as np
import pytest

import bench
import oracle
from workloads import CONFIGS, MoEConfig, gen_logits


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "capacity"])
def test_gemm_phases_sum_to_the_step_totals(name):
    c = CONFIGS[name]
    rows = c.T * c.k
    ph = bench.gemm_phases(c, rows)
    assert len(ph) == 6
    assert sum(f for f, _ in ph) == pytest.approx(bench.gemm_flops(c, rows), rel=1e-12)
    if not c.fs:
        assert sum(b for _, b in ph) == pytest.approx(bench.gemm_algorithmic_bytes(c, rows),
                                                      rel=1e-12)
    # FC1 and the FC1 data-gradient and weight-gradient carry 4 d f per row, the rest 2 d f
    F = rows * c.d * c.f + (c.T * c.d * c.fs if c.fs else 0)
    assert [round(f / F) for f, _ in ph] == [4, 2, 2, 2, 4, 4]


def test_peak_follows_the_sampled_clock():
    peaks = {"bf16_tflops": 1928.4, "bf16_tflops_sustained": 1716.7, "sm_max_mhz": 2070.0}
    assert bench.choose_peak(peaks, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[:2] == \
        (1928.4, "burst")
    assert bench.choose_peak(peaks, {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0})[1] == "burst"
    assert bench.choose_peak(peaks, {"sm_mhz": 1600.0, "sm_max_mhz": 2070.0})[:2] == \
        (1716.7, "sustained")
    assert bench.choose_peak(peaks, {"sm_mhz": None, "sm_max_mhz": None})[1] == "sustained"


def test_peak_follows_the_gemm_kernels_own_clock():
    """The clock the GEMM tile loops measured overrides the nvidia-smi median."""
    peaks = {"bf16_tflops": 1928.4, "bf16_tflops_sustained": 1716.7, "sm_max_mhz": 2070.0}
    smi = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}
    assert bench.choose_peak(peaks, smi, gemm_mhz=1709.0)[:2] == (1716.7, "sustained")
    assert bench.choose_peak(peaks, smi, gemm_mhz=2050.0)[:2] == (1928.4, "burst")
    assert "tile loops" in bench.choose_peak(peaks, smi, gemm_mhz=1709.0)[2]
    assert bench.choose_peak(peaks, {"sm_mhz": 1600.0, "sm_max_mhz": 2070.0},
                             gemm_mhz=2070.0)[1] == "burst"


def test_gemm_clock_summary():
    g = bench.gemm_clock_summary((3_400_000_000, 2_000_000_000, 152))
    assert g["sm_mhz"] == 1700.0 and g["loops"] == 152
    assert bench.gemm_clock_summary((0, 0, 0)) is None


def test_clock_window_summary():
    cs = bench.ClockSampler(0)
    cs.proc = object()           # as if nvidia-smi were running
    cs.samples = [(10.0, 2070.0, 2070.0, 500.0, set()),
                  (10.05, 1900.0, 2070.0, 900.0, {"sw_power_cap"}),
                  (10.1, 2000.0, 2070.0, 800.0, set()),
                  (20.0, 1000.0, 2070.0, 100.0, {"hw_slowdown"})]
    w = cs.window(10.0, 10.1)
    assert w["samples"] == 3 and w["sm_mhz"] == 2000.0 and w["reasons"] == ["sw_power_cap"]
    assert w["power_w_max"] == 900.0
    # no sample inside: the nearest one stands in
    w = cs.window(19.0, 19.5)
    assert w["samples"] == 1 and w["sm_mhz"] == 1000.0


def test_oracle_timer_full_and_extrapolated():
    """Where the estimate fits the budget every expert's FFN is timed (nothing
    extrapolated); with no budget the FFN is extrapolated from the row samples as
    sum_e (a + b * rows_e)."""
    c = CONFIGS["tiny"]
    ot = bench.OracleTimer(c)
    m = ot.measure(60.0)
    assert not m["extrapolated"]
    assert m["rows_kept"] == c.T * c.k
    assert set(m["parts_s"]) == {"route", "permute", "combine", "combine_bwd",
                                 "unpermute_reduce"}
    assert m["tokens_per_s"] == pytest.approx(c.T / m["seconds_per_step"])
    m = ot.measure(0.0)
    assert m["extrapolated"]
    a, b = m["ffn_fit"]["a_s"], m["ffn_fit"]["b_s_per_row"]
    assert m["ffn_s"] == pytest.approx(sum(a + b * n for n in ot.kept if n))
    assert "extrapolated" in ot.describe(m)
    # one sample with the fixed cost given
    m2 = ot.measure(0.0, a_fixed=a)
    assert m2["extrapolated"] and len(m2["ffn_fit"]["samples"]) == 1


@pytest.mark.parametrize("name", sorted(bench.GEMM_TRAFFIC_PER_LAUNCH))
def test_measured_traffic_is_near_the_algorithmic_bytes(name):
    """Each stored DRAM figure names a profiling shape with the same per-expert GEMMs at a
    quarter of the rows and experts, and lies near the workload's algorithmic bytes per
    launch (ncu counts writes still held in L2 at the launch's end as not yet written)."""
    from workloads import PROFILE_CONFIGS
    traffic, shape = bench.GEMM_TRAFFIC_PER_LAUNCH[name]
    c, p = CONFIGS[name], PROFILE_CONFIGS[shape]
    assert (p.d, p.f) == (c.d, c.f)
    assert p.T * p.k * 4 == c.T * c.k and p.E * 4 == c.E
    alg = bench.gemm_algorithmic_bytes(c, c.T * c.k) / 6
    assert 0.8 * alg < traffic < 1.1 * alg


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reference_lines(cmd, env_threads):
    import json, os, subprocess, sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {**os.environ, "OMP_NUM_THREADS": str(env_threads)}
    out = subprocess.run([sys.executable, *cmd], cwd=root, capture_output=True, text=True,
                         timeout=900, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    return [json.loads(l) for l in out.stdout.splitlines() if l.startswith("{")]


def _check_reference_line(d, n_gpus, threads):
    assert d["impl"] == "reference" and d["n_gpus"] == n_gpus
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] == threads
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_prints_one_line():
    """`bench.py --impl reference` times the oracle on the host (no GPU needed) and prints
    one JSON line whose core count is the threads the oracle actually ran on."""
    lines = _reference_lines(["bench.py", "--impl", "reference", "--config", "tiny",
                              "--steps", "1", "--warmup", "3"], 2)
    assert len(lines) == 1
    _check_reference_line(lines[0], 1, 2)


def test_reference_arm_under_two_ranks():
    """Launched as two ranks, rank 0 alone runs and prints; the other rank exits 0."""
    lines = _reference_lines(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node",
                              "2", "--master-addr", "127.0.0.1", "--master-port",
                              str(_free_port()), "bench.py", "--impl", "reference", "--gpus",
                              "2", "--config", "tiny", "--steps", "1", "--warmup", "3"], 1)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2, 1)
