"""Failure detection on the GPU without a fault: every pipeline wait of the attention
kernels is bounded, and a wait that runs out makes the kernel record PA_DEVERR_TIMEOUT
and return instead of hanging. These tests shorten the bound (plan option
wait_limit_ns) so that the waits run out, check that each kernel reports the timeout
through the device error word, and that the same process then computes the batch
correctly with the default bound (the context stays usable). The kernels run in a child
process (tests/wait_timeout_case.py), so that this test process's CUDA context is never
at stake; collected second to last."""
import json
import os
import subprocess
import sys

import pytest
import torch

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_short_wait_bound_reports_timeout_and_context_stays_usable():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gu.lib()  # built before the child starts
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "wait_timeout_case.py")],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, f"child failed:\n{r.stdout[-2000:]}\n{r.stderr[-4000:]}"
    res = json.loads(r.stdout.strip().splitlines()[-1])
    for name, x in res.items():
        # every call with the short bound ran out somewhere and said so
        assert all(c == 5 for c in x["short_bound_errors"]), (name, x)
        # then the same batch with the default bound: no error, oracle parity
        assert x["error_after"] == 0, (name, x)
        assert x["finite"], (name, x)
        assert x["max_abs"] <= gu.ATOL_MAX and x["mean_abs"] <= gu.ATOL_MEAN, (name, x)
