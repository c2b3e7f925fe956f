"""Child process of tests/test_zy_wait_timeout.py: makes the bounded pipeline waits of
each attention kernel run out, then checks that the library still computes the right
result. Run in its own process so that the parent's CUDA context is never at stake.

Every kernel bounds each wait of its pipeline (a wait on an mbarrier that a TMA copy,
an MMA or another warp completes). The plan option ``wait_limit_ns`` shortens that bound
to a few nanoseconds, so a wait runs out as soon as its barrier is not already complete:
the kernel records PA_DEVERR_TIMEOUT, waits (with the default one-second bound) for the
copies and MMAs it issued, frees its tensor memory and returns. The test then reads the
error word, clears it and runs the same batch with the default bound.

Prints one JSON line: per kernel, the error word after the short-bound calls, the error
word after the normal call, and the normal call's max / mean abs error against the
oracle.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402
from tests import gpu_util as gu  # noqa: E402

# (name, batch, plan options selecting the kernel)
CASES = [
    ("decode_kernel", dict(context_lens=[2000, 300, 900], query_lens=[1, 3, 2], Hq=4, Hkv=4,
                           D=64, block_size=16, seed=901), dict()),
    ("tcd_kernel", dict(context_lens=[3000, 1500, 700], query_lens=[1, 4, 2], Hq=8, Hkv=2,
                        D=128, block_size=16, seed=902), dict()),
    ("tc_kernel", dict(context_lens=[2000, 700, 1200], query_lens=[20, 30, 25], Hq=8, Hkv=2,
                       D=128, block_size=32, seed=903), dict(tc_pair=-1)),
    ("tc2_kernel", dict(context_lens=[3000, 1800], query_lens=[60, 50], Hq=8, Hkv=2, D=128,
                        block_size=32, seed=904), dict(tc_pair=1)),
    ("split + combine_kernel", dict(context_lens=[6000, 4000], query_lens=[1, 1], Hq=8, Hkv=8,
                                    D=128, block_size=16, seed=905),
     dict(max_chunk_tokens=512)),
]


def main():
    pa = gu.lib()
    dev = "cuda"
    res = {}
    for name, b, kw in CASES:
        w = workloads.make_custom(b["context_lens"], b["query_lens"], Hq=b["Hq"], Hkv=b["Hkv"],
                                  D=b["D"], block_size=b["block_size"], seed=b["seed"],
                                  write_new=False)
        bt = torch.from_numpy(w.block_table).to(dev)
        cl = torch.from_numpy(w.context_lens).to(dev)
        ql = torch.from_numpy(w.query_lens).to(dev)
        q, kp, vp = w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev)
        pa.pa_get_device_error(reset=True)
        short = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size,
                        w.max_blocks, wait_limit_ns=1, **kw)
        st = short.stats()
        codes = []
        for _ in range(3):
            pa.pa_attention(short, q, kp, vp, bt, cl, ql)
            torch.cuda.synchronize()
            codes.append(pa.pa_get_device_error(reset=True))
        plan = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size,
                       w.max_blocks, **kw)
        out = pa.pa_attention(plan, q, kp, vp, bt, cl, ql)
        torch.cuda.synchronize()
        after = pa.pa_get_device_error(reset=True)
        ref = gu.oracle_step(w)
        got = out.float().cpu().numpy()
        mx, mn = gu.attn_errors(got, gu.oracle_rows(w, ref))
        res[name] = {"short_bound_errors": codes, "error_after": after, "max_abs": mx,
                     "mean_abs": mn, "finite": bool(np.isfinite(got).all()),
                     "plan": {k: st[k] for k in ("n_dec_items", "n_tc_items", "n_tc_pair_items",
                                                 "n_tc_decode_items", "n_split_groups")}}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
