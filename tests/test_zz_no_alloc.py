"""pa_attention_static: the attention entry point that allocates nothing.

Some callers cannot allocate device memory for a workspace: a serving engine
that reserved nearly all HBM for its KV-cache pool at start-up (a later
cudaMalloc can fail), a loop that must not pay cudaMalloc's device-wide
synchronization, or a plain C caller with no allocator of its own. For them the
library keeps a fixed scratch array in its device image. These tests call that
entry point through the C ABI and compare it with pa_attention, which takes a
caller workspace. The file is collected last so that a failure here does not
hide the rest of the suite.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gu.lib()


def _inputs(w, dev="cuda"):
    return dict(q=w.q.to(dev), k_pool=w.k_pool.to(dev), v_pool=w.v_pool.to(dev),
                block_table=torch.from_numpy(w.block_table).to(dev),
                context_lens=torch.from_numpy(w.context_lens).to(dev),
                query_lens=torch.from_numpy(w.query_lens).to(dev))


def test_static_workspace_matches_caller_workspace_on_two_calls(pa):
    # two different batches back to back: the second call runs on whatever the first left
    # in the shared array; the first batch is split so partial results go through it too
    batches = [
        (workloads.make(1), dict(max_chunk_tokens=64)),
        (workloads.make_custom([900, 33, 2500, 1], [1, 17, 3, 1], Hq=16, Hkv=4, D=128,
                               block_size=32, seed=404), dict()),
    ]
    for w, kw in batches:
        x = _inputs(w)
        plan = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size,
                       w.max_blocks, **kw)
        assert plan.workspace_bytes <= pa.STATIC_WORKSPACE_BYTES
        ref = pa.pa_attention(plan, **x)
        got = pa.pa_attention_static(plan, **x)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error(reset=True) == 0
        # the same plan and kernels on the same inputs: only the scratch's address
        # differs, so the outputs must agree bit for bit (stale tables or partials left
        # in the shared array by the previous call would show here)
        assert torch.equal(got, ref)
        if kw:
            assert plan.stats()["n_split_groups"] > 0


def test_static_workspace_rejects_oversized_plan(pa):
    # about 320k work items: the plan tables alone exceed the fixed array
    n = 5000
    plan = pa.Plan([1] * n, [1] * n, 64, 64, 64, 16, 1)
    assert plan.workspace_bytes > pa.STATIC_WORKSPACE_BYTES
    dev = "cuda"
    q = torch.zeros(n, 64, 64, dtype=torch.bfloat16, device=dev)
    kp = torch.zeros(2, 16, 64, 64, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(n, 1, dtype=torch.int32, device=dev)
    lens = torch.ones(n, dtype=torch.int32, device=dev)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_attention_static(plan, q, kp, kp, bt, lens, lens)
    assert e.value.status == 2
