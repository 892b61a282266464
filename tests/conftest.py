import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session", autouse=True)
def _oracle_built():
    import oracle
    oracle.build()
    yield


@pytest.fixture(autouse=True)
def _name_the_comparisons(request):
    """Tag every GPU-vs-oracle comparison with the test that made it (for the report)."""
    gu = sys.modules.get("gpu_util")
    if gu is not None:
        gu.CURRENT_TEST[0] = request.node.nodeid.split("::", 1)[-1]
    yield


def pytest_terminal_summary(terminalreporter):
    """Parity report: per test, the worst of its GPU-vs-oracle comparisons -- rel-L2, the
    scaled max bound the tests assert, max |g - o| / rms(o), the raw max |g - o| -- and how
    many compared elements differ by more than one bf16 ulp of the oracle's value."""
    gu = sys.modules.get("gpu_util")
    if gu is None or not gu.RECORDS:
        return
    tr = terminalreporter
    tr.section("GPU vs oracle parity (bf16 / fp32 outputs)")
    tr.write_line(f"{'test':<58} {'tensors':>7} {'rel_l2':>9} {'max_scl':>9} {'max/rms':>9} "
                  f"{'max_abs':>9} {'>1ulp':>9} {'of':>11}")
    by_test = {}
    for test, name, s in gu.RECORDS:
        by_test.setdefault(test, []).append((name, s))
    tot_bad = tot_n = 0
    for test, recs in by_test.items():
        ss = [s for _, s in recs]
        bad = sum(s["n_gt_1ulp"] for s in ss)
        n = sum(s["n"] for s in ss)
        tot_bad += bad; tot_n += n
        tr.write_line(f"{test[:58]:<58} {len(ss):>7} {max(s['rel_l2'] for s in ss):>9.2e} "
                      f"{max(s['max_scaled'] for s in ss):>9.2e} "
                      f"{max(s['max_over_rms'] for s in ss):>9.2e} "
                      f"{max(s['max_abs'] for s in ss):>9.2e} {bad:>9} {n:>11}")
    worst = sorted(gu.RECORDS, key=lambda r: -r[2]["max_over_rms"])[:12]
    tr.write_line("largest max |g - o| / rms(o):")
    for test, name, s in worst:
        tr.write_line(f"  {test[:50]:<50} {name[:18]:<18} max/rms {s['max_over_rms']:.3e} "
                      f"max_scl {s['max_scaled']:.3e} rel_l2 {s['rel_l2']:.2e} "
                      f">1ulp {s['n_gt_1ulp']}/{s['n']}")
    tr.write_line(f"total: {len(gu.RECORDS)} comparisons, {tot_bad} of {tot_n} elements "
                  f"({tot_bad / max(tot_n, 1):.2e}) more than 1 bf16 ulp from the oracle")
