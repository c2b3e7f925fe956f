"""Host-side pieces of bench.py that need no GPU: the oracle's timed sample and the
kernel-source hash that keeps a traffic capture valid."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402
from workloads import host_bits  # noqa: E402


def _host(w):
    return {"q": host_bits(w.q), "k_pool": host_bits(w.k_pool), "v_pool": host_bits(w.v_pool),
            "k_new": host_bits(w.k_new), "v_new": host_bits(w.v_new)}


def test_oracle_sample_spreads_rows_and_keeps_its_budget():
    """The sample takes rows spread over the whole batch (not a prefix, whose rows see
    the fewest keys), writes their own new tokens, stops on its time budget and copies
    the pools once per process."""
    w = workloads.make(1)
    host = _host(w)
    orc = oracle.default()
    t0 = time.perf_counter()
    v, sample, el = bench.oracle_step_sample(w, orc, host, 2, budget_s=0.3)
    assert v > 0 and 0.3 <= el < 5.0 and time.perf_counter() - t0 < 30.0
    assert f"spread evenly over all {w.total_q}" in sample
    kp = host["_kp"]
    bench.oracle_step_sample(w, orc, host, 2, budget_s=0.05)
    assert host["_kp"] is kp                      # the working pools are made once


def test_kernel_hash_ignores_comments_only():
    code = 'int f(int x) { return x + 1; }  // one\n'
    assert bench._code_only(code) == bench._code_only('/* a */ int f(int x)\n{ return x + 1; }\n')
    assert bench._code_only(code) != bench._code_only(code.replace("+ 1", "+ 2"))
    assert bench._code_only('const char* s = "// not a comment";') == \
        'const char* s = "// not a comment";'
