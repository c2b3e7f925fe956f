"""Helpers shared by the GPU parity tests: run one step of the hot path through the
C ABI, run the same step through the oracle, compare."""
import os

import numpy as np
import torch

import oracle
from tests.oracle_checks import f64, u16

ATOL_MAX = 5e-3     # attention: max abs error against the fp64 oracle
ATOL_MEAN = 5e-4    # attention: mean abs error


def lib():
    from paged_kv_cache_02_gb300 import _build
    _build.build()
    import paged_kv_cache_02_gb300 as pa
    return pa


def gpu_step(pa, w, dev="cuda", out_dtype=torch.float32, fused=False, **plan_kw):
    """slot mapping -> copy-on-write copies -> KV write -> attention, all through libpa
    (``fused``: the KV write and the attention in one pa_attention_write call)."""
    bt = torch.from_numpy(w.block_table).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    ql = torch.from_numpy(w.query_lens).to(dev)
    kp, vp = w.k_pool.to(dev).clone(), w.v_pool.to(dev).clone()
    sid = torch.from_numpy(w.new_seq).to(dev)
    pos = torch.from_numpy(w.new_pos).to(dev)
    slots = pa.pa_slot_mapping(bt, w.num_blocks, w.block_size, sid, pos)
    if len(w.cow_src):
        pa.pa_copy_blocks(kp, vp, torch.from_numpy(w.cow_src).to(dev),
                          torch.from_numpy(w.cow_dst).to(dev))
    plan = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size, w.max_blocks,
                   **plan_kw)
    if fused:
        # the step's new tokens are its query tokens, in q's row order
        assert len(w.new_seq) == w.total_q
        out = pa.pa_attention_write(plan, w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev), slots,
                                    kp, vp, bt, cl, ql, out_dtype=out_dtype)
    else:
        pa.pa_write_kv(w.k_new.to(dev), w.v_new.to(dev), slots, kp, vp)
        out = pa.pa_attention(plan, w.q.to(dev), kp, vp, bt, cl, ql, out_dtype=out_dtype)
    err = pa.pa_get_device_error(reset=True)
    return dict(slots=slots.cpu().numpy(), k_pool=kp, v_pool=vp, out=out, err=err, plan=plan)


def oracle_step(w, orc=None):
    """The same step through the oracle, on host copies of the inputs."""
    orc = orc or oracle.default()
    kp, vp = u16(w.k_pool), u16(w.v_pool)
    slots = orc.slot_mapping(w.block_table, w.num_blocks, w.block_size, w.new_seq, w.new_pos)
    if len(w.cow_src):
        orc.copy_blocks(kp, vp, w.cow_src, w.cow_dst)
    orc.write_kv(u16(w.k_new), u16(w.v_new), slots, kp, vp)
    return dict(slots=slots, k_pool=kp, v_pool=vp)


def oracle_threads():
    return max(1, os.cpu_count() or 1)


def oracle_rows(w, ref, rows=None, orc=None):
    orc = orc or oracle.default()
    if "q_bits" not in ref:
        ref["q_bits"] = u16(w.q)
    return orc.attention(ref["q_bits"], ref["k_pool"], ref["v_pool"], w.block_table,
                         w.context_lens, w.query_lens, rows=rows, n_threads=oracle_threads())


def pools_equal(gpu_pool: torch.Tensor, ref_pool: np.ndarray) -> bool:
    return np.array_equal(u16(gpu_pool), ref_pool)


def attn_errors(got: np.ndarray, want: np.ndarray):
    d = np.abs(got.astype(np.float64) - want)
    return float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0


def assert_attention_close(got, want, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    mx, mn = attn_errors(got, want)
    assert mx <= ATOL_MAX and mn <= ATOL_MEAN, f"{what}: max abs {mx:.3g}, mean abs {mn:.3g}"
    return mx, mn


def compare_all_rows(got_out, w, ref, what, chunk=4096):
    """Every query row of ``got_out`` (device or host tensor [T, Hq, D]) against the
    oracle, in chunks of rows so that host memory stays bounded; returns (max abs, mean
    abs, rows) over all rows and asserts the attention tolerance. When the environment
    names a report file (PA_PARITY_REPORT), one JSON line per call is appended to it."""
    import json
    import time
    T = w.total_q
    got = got_out.float().cpu().numpy()
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    mx, tot, n = 0.0, 0.0, 0
    t0 = time.perf_counter()
    orc = oracle.default()
    for r0 in range(0, T, chunk):
        rows = np.arange(r0, min(T, r0 + chunk), dtype=np.int64)
        want = oracle_rows(w, ref, rows, orc=orc)
        d = np.abs(got[rows].astype(np.float64) - want)
        mx = max(mx, float(d.max()))
        tot += float(d.sum())
        n += d.size
    mean = tot / max(1, n)
    dt = time.perf_counter() - t0
    path = os.environ.get("PA_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, "rows": T, "values": n, "max_abs": mx,
                                "mean_abs": mean, "oracle_s": dt,
                                "threads": oracle_threads()}) + "\n")
    assert mx <= ATOL_MAX and mean <= ATOL_MEAN, f"{what}: max abs {mx:.3g}, mean abs {mean:.3g}"
    return mx, mean, T


def sample_rows(w, n, seed):
    """Seeded sample of query rows, always including the first and last row of every
    row group and of the longest sequence."""
    T = w.total_q
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    pref = np.concatenate([[0], np.cumsum(w.query_lens)])
    longest = int(np.argmax(w.context_lens))
    if w.query_lens[longest] > 0:
        rows.update({int(pref[longest]), int(pref[longest + 1] - 1)})
    rows.update({0, T - 1})
    return np.array(sorted(rows), dtype=np.int64)
