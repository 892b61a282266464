"""Host-side arithmetic of bench.py: the per-launch GEMM flops and bytes, and the exactness
of the CPU baseline's expert restriction (routing a token sample over only the experts it
selects gives the same choices and gate weights)."""

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


@pytest.mark.parametrize("gate,scale", [("softmax", 1.0), ("sigmoid", 2.5)])
def test_expert_restriction_keeps_choices_and_weights(gate, scale):
    c = MoEConfig("restrict", T=48, d=64, E=40, k=6, f=64, gate=gate, route_scale=scale,
                  zipf_s=1.2)
    lg = gen_logits(c)
    full = oracle.route(c, lg)
    used = np.unique(full["topk_idx"])
    assert len(used) < c.E
    sub = oracle.route(c.replace(E=len(used)), np.ascontiguousarray(lg[:, used]))
    np.testing.assert_array_equal(used[sub["topk_idx"]], full["topk_idx"])
    np.testing.assert_array_equal(sub["topk_w"], full["topk_w"])


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
