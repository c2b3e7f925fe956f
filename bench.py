"""Benchmark of the paged-attention hot path on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one batch: slot mapping, the
copy-on-write block copies (when the batch has any), the KV write of the step's
new tokens, and paged attention over the block tables (CUDA-core decode items,
tensor-core items, the split-KV combine). Inputs are resident in HBM when the
timed region starts; the KV pools (several GB) are larger than L2, so no flush
is needed between steps. The default workload is the largest one, the
Pensieve-style unified batch with the Llama-2-13B attention shape (Hq=Hkv=40,
D=128, block size 32): 64 multi-turn conversations, each a new prompt of 32-512
tokens over a 512-3072-token history split into two sub-requests that share
blocks, plus 128 decode sequences (about 48.6k query rows over 436k KV tokens).
The key ``configs`` times the attention kernels of every other workload and of
the mixed batches' prefill and decode sub-batches, each against its roofline.

Prints ONE JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle on
the host cores instead (a deliberately plain program, the baseline arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged attn tokens/s and achieved HBM GB/s / TC util vs roofline (1×GB300)"
UNIT = "tokens/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {"decode": ["pa_dec.cu", "pa_ptx.cuh", "pa_internal.h"],
                  "tc": ["pa_tc.cu", "pa_tc.cuh", "pa_ptx.cuh", "pa_internal.h"],
                  "tc2": ["pa_tc2.cu", "pa_tc.cuh", "pa_ptx.cuh", "pa_internal.h"],
                  "tcd": ["pa_tcd.cu", "pa_tc.cuh", "pa_ptx.cuh", "pa_internal.h"]}
# kernel symbol of each (for the launch-list summaries)
KERNEL_NAMES = {"decode": "decode_kernel", "tc": "tc_kernel", "tc2": "tc2_kernel",
                "tcd": "tcd_kernel"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def _code_only(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed: what the
    compiler sees, so that editing a comment does not change a kernel's hash."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                                  # string or character literal
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernels) -> str:
    """sha256 of the code (comments and whitespace aside) of the sources of the listed
    kernels (a name or a list), each file once."""
    if isinstance(kernels, str):
        kernels = [kernels]
    files = sorted({f for k in kernels for f in KERNEL_SOURCES[k]})
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_02_gb300", "csrc", f),
                  encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "_source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while running (read-only query)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = [s for t, s in self.samples if t0 <= t <= t1] or [s for _, s in self.samples]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ distributed plumbing

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle (CPU) arm

def oracle_step_sample(w, orc, host, n_threads, budget_s=10.0, max_passes=1000):
    """Times the oracle on bounded passes over the same workload: slot mapping, copies,
    KV write and attention for R query rows spread evenly over the whole batch (so the
    sample has the batch's mix of context lengths). Returns (rows/s, sample, seconds)."""
    import numpy as np
    T = w.total_q
    # cost of each row (visible keys x heads) for sizing a pass to about budget / 3
    pref = np.concatenate([[0], np.cumsum(w.query_lens)])
    seq_of_row = np.repeat(np.arange(w.num_seqs), w.query_lens)
    pos = w.context_lens[seq_of_row] - w.query_lens[seq_of_row] + (np.arange(T) - pref[seq_of_row])
    cost = (pos + 1).astype(np.float64) * w.Hq * w.D * 2  # MACs per row
    spread = lambda r: np.unique(np.linspace(0, T - 1, max(1, min(T, r))).astype(np.int64))
    key = ("_macs_per_s", n_threads)                      # measured once per process
    if key not in host:
        probe_rows = spread(16)
        t_probe = time.perf_counter()
        orc.attention(host["q"], host["k_pool"], host["v_pool"], w.block_table,
                      w.context_lens, w.query_lens, rows=probe_rows, n_threads=n_threads)
        dt_probe = max(1e-6, time.perf_counter() - t_probe)
        host[key] = max(1e6, cost[probe_rows].sum() / dt_probe)
    macs_per_s = host[key]
    rows = spread(int(macs_per_s * budget_s / 3.0 / cost.mean()) + 1)
    R = len(rows)
    # working copies of the pools, made once per process (a pass writes into them)
    if "_kp" not in host:
        host["_kp"], host["_vp"] = host["k_pool"].copy(), host["v_pool"].copy()
    kp, vp = host["_kp"], host["_vp"]
    # the write in proportion: when the new tokens are the query rows (one new token per
    # query token, in the same order), a pass writes the new tokens of its rows only
    tok = rows if len(w.new_seq) == T else np.arange(len(w.new_seq))
    done_rows = 0
    passes = 0
    t0 = time.perf_counter()
    while True:
        slots = orc.slot_mapping(w.block_table, w.num_blocks, w.block_size, w.new_seq[tok],
                                 w.new_pos[tok])
        if len(w.cow_src):
            orc.copy_blocks(kp, vp, w.cow_src, w.cow_dst)
        orc.write_kv(host["k_new"][tok], host["v_new"][tok], slots, kp, vp)
        orc.attention(host["q"], kp, vp, w.block_table, w.context_lens, w.query_lens,
                      rows=None if R == T else rows, n_threads=n_threads)
        done_rows += R
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or passes >= max_passes:
            break
    sample = (f"{passes} pass(es) of slot mapping + KV write + attention of {R} query rows "
              f"spread evenly over all {T} (and their {len(tok)} new tokens) of {w.name}, "
              f"{el:.1f} s on {n_threads} threads")
    return done_rows / el, sample, el


def run_reference(args, w, cfg_name):
    import numpy as np
    import oracle
    from workloads import host_bits as u16
    orc = oracle.default()
    host = {"q": u16(w.q), "k_pool": u16(w.k_pool), "v_pool": u16(w.v_pool),
            "k_new": u16(w.k_new), "v_new": u16(w.v_new)}
    n_threads = os.cpu_count() or 1
    # about 150 s for the whole run whatever --steps and --warmup are: each step is at
    # least one pass (about 0.1 s on the GPU machine's 16 cores), so with the default 1,000
    # steps a step is one pass
    budget = max(0.01, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_step_sample(w, orc, host, n_threads, budget_s=min(budget, 2.0), max_passes=1)
    vals, samples, total = [], [], 0.0
    for _ in range(args.steps):
        v, s, el = oracle_step_sample(w, orc, host, n_threads, budget_s=budget)
        vals.append(v)
        samples.append(s)
        total += el
    value = float(np.median(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * w.total_q / value, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg_name,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_threads, "kind": "oracle",
                         "sample": samples[0]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def run_gpu(args, w, cfg_name, rank, local, world):
    import numpy as np
    import torch
    import paged_kv_cache_02_gb300 as pa

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    # ---- device-resident inputs
    bt = torch.from_numpy(w.block_table).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    ql = torch.from_numpy(w.query_lens).to(dev)
    sid = torch.from_numpy(w.new_seq).to(dev)
    pos = torch.from_numpy(w.new_pos).to(dev)
    src = torch.from_numpy(w.cow_src).to(dev)
    dst = torch.from_numpy(w.cow_dst).to(dev)
    q, kn, vn = w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev)
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    slots = torch.empty(len(w.new_seq), dtype=torch.int64, device=dev)
    out_dtype = torch.bfloat16 if args.out == "bf16" else torch.float32
    out = torch.empty(q.shape, dtype=out_dtype, device=dev)
    plan_kw = dict(tc_min_rows=args.tc_min_rows, max_chunk_tokens=args.max_chunk,
                   tc_pair=args.tc_pair)
    plan = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size, w.max_blocks,
                   **plan_kw)
    st = plan.stats()
    ws = plan.workspace(dev)
    n_pairs = len(w.cow_src)

    ev = {k: [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
          for k in ("a", "b", "c", "d", "f", "e")}

    def step(i=None, fused=None):
        fused = args.fused if fused is None else fused
        if i is not None:
            ev["a"][i].record(stream)
        pa.pa_slot_mapping(bt, w.num_blocks, w.block_size, sid, pos, out=slots)
        if i is not None:
            ev["b"][i].record(stream)
        if n_pairs:
            pa.pa_copy_blocks(kp, vp, src, dst)
        if i is not None:
            ev["c"][i].record(stream)
        if not fused:
            pa.pa_write_kv(kn, vn, slots, kp, vp)
        if i is not None:
            ev["d"][i].record(stream)
        # the plan's tables go up once per step (a model would share them across its
        # layers), then the attention kernels
        pa.pa_plan_upload(plan, ws)
        if i is not None:
            ev["f"][i].record(stream)
        if not fused:
            pa.pa_attention_planned(plan, q, kp, vp, bt, cl, ql, ws, out=out)
        else:
            # the KV write of the decode rows inside the key-major kernel, the other rows'
            # write kernel first (the step's new tokens are its query tokens)
            pa.pa_attention_write(plan, q, kn, vn, slots, kp, vp, bt, cl, ql, out=out,
                                  workspace=ws, planned=True)
        if i is not None:
            ev["e"][i].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    err = pa.pa_get_device_error(reset=True)
    if err:
        raise RuntimeError(f"device error {pa.DEVERR.get(err, err)} during warm-up")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)  # the sampler's first line
    barrier(world)
    torch.cuda.synchronize(dev)
    start_ev = torch.cuda.Event(enable_timing=True)
    end_ev = torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    start_ev.record(stream)
    for i in range(args.steps):
        step(i)
    end_ev.record(stream)
    torch.cuda.synchronize(dev)
    h1 = time.perf_counter()
    barrier(world)
    clocks.stop()
    elapsed_ms = start_ev.elapsed_time(end_ev)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    per = {k: float(np.mean([ev[a][i].elapsed_time(ev[b][i]) for i in range(args.steps)]))
           for k, (a, b) in {"slot_mapping": ("a", "b"), "copy_blocks": ("b", "c"),
                             "write_kv": ("c", "d"), "attention": ("d", "e"),
                             "plan_upload": ("d", "f"), "attention_kernels": ("f", "e")}.items()}
    if args.fused:
        per["write_kv"] = "inside the attention call (fused): the decode rows in the " \
                          "key-major kernel, the other rows in one write kernel first"
    err = pa.pa_get_device_error(reset=True)
    if err:
        raise RuntimeError(f"device error {pa.DEVERR.get(err, err)} in the timed region")

    # the other form of the step (fused KV write + attention, or the two calls), timed the
    # same way for comparison; not part of `value`
    n_alt = max(3, min(args.steps, 50))
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        step(fused=not args.fused)
    torch.cuda.synchronize(dev)
    a_ev.record(stream)
    for _ in range(n_alt):
        step(fused=not args.fused)
    b_ev.record(stream)
    torch.cuda.synchronize(dev)
    err = pa.pa_get_device_error(reset=True)
    if err:
        raise RuntimeError(f"device error {pa.DEVERR.get(err, err)} timing the other step form")
    alt_ms = a_ev.elapsed_time(b_ev) / n_alt
    alt_step = {"path": ("pa_write_kv + pa_attention_planned" if args.fused else
                         "pa_attention_write_planned (fused KV write + attention)"),
                "ms_per_step": alt_ms, "tokens_per_s": w.total_q / (alt_ms / 1000.0),
                "steps": n_alt}

    T = w.total_q
    value = T * args.steps * world / (elapsed_ms / 1000.0)
    n_tc1 = st["n_tc_items"] - st["n_tc_pair_items"] - st["n_tc_decode_items"]
    st_write = 1 if (not args.fused or st["n_tc_decode_items"] == 0 or
                     plan_fused_rows(w) < T) else 0
    launches_per_step = 1 + (1 if n_pairs else 0) + st_write + (1 if st["n_dec_items"] else 0) + \
        (1 if n_tc1 else 0) + (1 if st["n_tc_pair_items"] else 0) + \
        (1 if st["n_tc_decode_items"] else 0) + (1 if st["n_split_groups"] else 0)

    # ---- roofline of the dominant kernel (paged attention)
    peaks = measured_peaks()
    kv_b, q_b, o_b = w.kv_bytes(), w.q_bytes(), T * w.Hq * w.D * out.element_size()
    flops = w.flops()
    # the roofline is that of the attention kernels: timed here on their own (one planned
    # call per timed call, tables uploaded once), since the step's call also holds the
    # write kernel of the non-decode rows
    attn_ms, _ = time_attention(w, dev, **plan_kw)
    attn_s = attn_ms / 1000.0
    hbm_peak = float(peaks["hbm_gbs"])
    tc_peak = float(peaks.get("bf16_tflops", 1900.0))
    t_hbm = (kv_b + q_b) / (hbm_peak * 1e9)
    t_tc = flops / (tc_peak * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    # the attention call runs one kernel when the plan holds one kind of item; its
    # committed DRAM counters apply while that kernel's sources are unchanged
    n_tcd, n_tc2 = st["n_tc_decode_items"], st["n_tc_pair_items"]
    n_tc1 = st["n_tc_items"] - n_tcd - n_tc2
    kinds = {k: n for k, n in (("decode", st["n_dec_items"]), ("tc", n_tc1), ("tc2", n_tc2),
                               ("tcd", n_tcd)) if n}
    # DRAM bytes of the call's attention kernels per call, from the committed capture,
    # while those kernels' sources hash to the captured ones
    traffic = None
    if kinds and not st["n_split_groups"] and os.path.exists(PROFILE_TRAFFIC):
        with open(PROFILE_TRAFFIC) as f:
            prof = json.load(f)
        entry = prof.get(args.config_key)
        if entry and sorted(entry.get("kernels", [])) == sorted(kinds) and \
                entry.get("kernel_hash") == kernel_source_hash(sorted(kinds)):
            traffic = entry.get("dram_bytes_per_launch")
    if bound == "hbm":
        achieved = (kv_b + q_b) / attn_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic,
                "peak_source": f"{peaks['_source']} hbm_gbs",
                "kernels": [KERNEL_NAMES[k] for k in kinds]}
    else:
        achieved = flops / attn_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved / tc_peak, "traffic": traffic,
                "peak_source": f"{peaks['_source']} bf16_tflops",
                "kernels": [KERNEL_NAMES[k] for k in kinds]}

    # ---- end to end through the public API, host buffers in pinned memory
    pin = lambda t: t.cpu().pin_memory()
    h_in = [pin(w.q), pin(w.k_new), pin(w.v_new), pin(bt), pin(cl), pin(ql), pin(sid), pin(pos),
            pin(src), pin(dst)]
    depth = 3                               # steps in flight
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(depth)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    # sets of device buffers: step i uses set i % depth
    d_sets = [[torch.empty_like(t, device=dev) for t in h_in] for _ in range(depth)]
    d_outs = [out] + [torch.empty_like(out) for _ in range(depth - 1)]
    # each buffer set has its own plan workspace (the step's plan tables go up with the
    # step's inputs)
    ws_sets = [plan.workspace(dev) for _ in range(depth)]
    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)
    free_ev = [None] * depth

    # Several steps in flight, as a serving loop runs them: the host builds step i's plan
    # and enqueues its work while the GPU still works on the steps before, then waits for
    # step i - depth + 1 to finish (its output is in host memory by then). Step i's
    # inputs go up on a copy stream and its output comes back on another, so that they
    # overlap the kernels of the neighbouring steps; events order the reuse of each
    # buffer set (the copies into set i % depth wait until step i - depth has read it
    # and its output is home).
    # The step's plan tables go up on the copy stream too, ahead of its inputs: uploaded
    # by the attention call on the compute stream, they would queue on the copy engine
    # behind the next step's inputs and hold the kernels back. Every step still copies
    # all of its own inputs in and its whole output out.
    inflight = []

    def e2e_step(i):
        k = i % depth
        dset, d_out, h_out, ws_k = d_sets[k], d_outs[k], h_outs[k], ws_sets[k]
        p2 = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size, w.max_blocks,
                     **plan_kw)
        if p2.workspace_bytes > ws_k.numel():
            raise RuntimeError("plan workspace grew between steps")
        if free_ev[k] is not None:
            s_h2d.wait_event(free_ev[k])
        with torch.cuda.stream(s_h2d):
            pa.pa_plan_upload(p2, ws_k)
            for hb, db in zip(h_in, dset):
                db.copy_(hb, non_blocking=True)
        in_ev = torch.cuda.Event()
        in_ev.record(s_h2d)
        dq, dkn, dvn, dbt, dcl, dql, dsid, dpos, dsrc, ddst = dset
        stream.wait_event(in_ev)
        pa.pa_slot_mapping(dbt, w.num_blocks, w.block_size, dsid, dpos, out=slots)
        if n_pairs:
            pa.pa_copy_blocks(kp, vp, dsrc, ddst)
        pa.pa_write_kv(dkn, dvn, slots, kp, vp)
        pa.pa_attention_planned(p2, dq, kp, vp, dbt, dcl, dql, ws_k, out=d_out)
        comp_ev = torch.cuda.Event()
        comp_ev.record(stream)
        s_d2h.wait_event(comp_ev)
        with torch.cuda.stream(s_d2h):
            h_out.copy_(d_out, non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_d2h)
        free_ev[k] = done
        inflight.append((done, p2))
        if len(inflight) > depth - 1:
            ev0, p0 = inflight.pop(0)
            ev0.synchronize()
            p0.close()

    def e2e_drain():
        while inflight:
            ev0, p0 = inflight.pop(0)
            ev0.synchronize()
            p0.close()

    for i in range(min(3, args.warmup)):
        e2e_step(i)
    e2e_drain()
    # at least 120 steps (about 1 s): the host link's occasional 20-50 ms stalls then
    # move the figure little
    e2e_steps = max(120, min(args.steps, 200))
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_drain()
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = T * e2e_steps * world / e2e_s
    err = pa.pa_get_device_error(reset=True)
    if err:
        raise RuntimeError(f"device error {pa.DEVERR.get(err, err)} in the end-to-end run")

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg_name,
        "out_dtype": args.out,
        "step_path": ("pa_attention_write_planned (fused KV write + attention)" if args.fused
                      else "pa_write_kv + pa_attention_planned"),
        "other_step_form": alt_step,
        "attention_kernels_ms": attn_ms,
        "roofline": roof,
        "hbm_gbs_attention": (kv_b + q_b) / attn_s / 1e9,
        "tc_tflops_attention": flops / attn_s / 1e12,
        "per_call_ms": per,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "includes": "H2D of the step's inputs from pinned memory, host plan build "
                            "and upload of its work tables (not counted in h2d_bytes: under "
                            "1 MB), slot mapping, copies, KV write, attention, D2H of the "
                            f"output; {depth} steps in flight (the host prepares step i "
                            "while the GPU runs the steps before), H2D (tables first) and "
                            "D2H on their own streams"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(h0, h1),
        "plan": {k: st[k] for k in ("n_dec_items", "n_tc_items", "n_split_groups", "chunk_tokens")},
        "bytes": {"kv": kv_b, "q": q_b, "o_write": o_b}, "flops": flops,
    }
    if rank == 0:
        if not args.no_configs:
            line["configs"] = configs_sweep(args, w, dev)
        line["swap"] = swap_measure(w, dev)
        line["block_manager"] = block_manager_host(w)
        line["cpu_baseline"] = cpu_baseline(args, w)
        print(json.dumps(line), flush=True)


def plan_fused_rows(w):
    """Query rows whose sequence has at most 16 packed rows per KV head (q * Hq / Hkv <=
    16): the rows the fused call writes inside the key-major kernel (D = 128, block size
    >= 8, Hq / Hkv dividing 16)."""
    g = w.Hq // w.Hkv
    if w.D != 128 or w.block_size < 8 or 16 % g:
        return 0
    q = w.query_lens.astype(int)
    return int(q[q * g <= 16].sum())


def roofline_entry(w, ms, peaks, out_bytes_per_elem=4):
    """Roofline of one attention call: the slower of K/V + Q bytes at the measured HBM
    bandwidth and the causal FLOPs at the measured bf16 tensor rate."""
    kv_b, q_b, flops = w.kv_bytes(), w.q_bytes(), w.flops()
    hbm, tc = float(peaks["hbm_gbs"]), float(peaks.get("bf16_tflops", 1900.0))
    s = ms / 1000.0
    t_hbm, t_tc = (kv_b + q_b) / (hbm * 1e9), flops / (tc * 1e12)
    gbs, tfs = (kv_b + q_b) / s / 1e9, flops / s / 1e12
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return {"bound": bound,
            "achieved": gbs if bound == "hbm" else tfs,
            "peak": hbm if bound == "hbm" else tc,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": max(t_hbm, t_tc) / s,
            "frac_hbm": t_hbm / s, "frac_tc": t_tc / s,
            "gbs": gbs, "tflops": tfs, "ms": ms,
            "t_hbm_ms": t_hbm * 1e3, "t_tc_ms": t_tc * 1e3,
            "tokens_per_s": w.total_q / s,
            "total_q": w.total_q, "kv_tokens": int(w.context_lens.sum())}


def time_attention(w, dev, reps=30, warmup=5, **plan_kw):
    """CUDA-event time of the attention kernels of one planned call (tables uploaded once
    before the timed calls), averaged over ``reps`` back-to-back calls; also the plan's
    kernels. Inputs resident in HBM; their pools exceed L2 except config 1's."""
    import torch
    import paged_kv_cache_02_gb300 as pa
    bt = torch.from_numpy(w.block_table).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    ql = torch.from_numpy(w.query_lens).to(dev)
    q = w.q.to(dev)
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    plan = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size, w.max_blocks,
                   **plan_kw)
    ws = plan.workspace(dev)
    pa.pa_plan_upload(plan, ws)
    for _ in range(warmup):
        pa.pa_attention_planned(plan, q, kp, vp, bt, cl, ql, ws, out=out)
    stream = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(reps):
        pa.pa_attention_planned(plan, q, kp, vp, bt, cl, ql, ws, out=out)
    b.record(stream)
    b.synchronize()
    err = pa.pa_get_device_error(reset=True)
    if err:
        raise RuntimeError(f"device error {pa.DEVERR.get(err, err)} timing {w.name}")
    st = plan.stats()
    n_tc1 = st["n_tc_items"] - st["n_tc_pair_items"] - st["n_tc_decode_items"]
    kernels = [n for n, c in (("decode_kernel", st["n_dec_items"]),
                              ("tcd_kernel", st["n_tc_decode_items"]),
                              ("tc2_kernel", st["n_tc_pair_items"]), ("tc_kernel", n_tc1),
                              ("combine_kernel", st["n_split_groups"])) if c]
    plan.close()
    return a.elapsed_time(b) / reps, kernels


def configs_sweep(args, w_head, dev):
    """Attention kernels of every config and of the mixed batches' prefill and decode
    sub-batches, each with its roofline (the spec bars: decode-dominated batches
    against HBM, prefill-dominated ones against the tensor cores)."""
    import gc
    import torch
    import workloads
    peaks = measured_peaks()
    res = {}

    def add(key, w, bar=None):
        ms, kernels = time_attention(w, dev)
        e = roofline_entry(w, ms, peaks)
        e["kernels"] = kernels
        if bar:
            # any one of the listed (roofline, fraction) alternatives meets the bar
            e["bar"] = [f"{kind} >= {thr}" for kind, thr in bar]
            e["bar_met"] = any(e["frac_hbm" if kind == "hbm" else "frac_tc"] >= thr
                               for kind, thr in bar)
        res[key] = e
        log(f"configs: {key}: {ms:.4f} ms, frac {e['frac']:.3f} ({e['bound']})")

    head = args.config
    for cfg in [1, 2, 3, 4, 5, "5cow"]:
        key = f"cfg{cfg}"
        w = w_head if str(cfg) == str(head) and not args.subset and not args.contiguous \
            and args.block_size is None else workloads.make(cfg, device=dev)
        bar = {2: [("hbm", 0.70)], 5: [("hbm", 0.70)], "5cow": [("hbm", 0.70)]}.get(cfg)
        add(key, w, bar)
        if cfg in (3, 4):
            # config 3's prefill sub-batch is HBM-bound (its K/V bytes outweigh its FLOPs
            # at machine balance), so its binding roofline at 0.70 is accepted too
            add(f"{key}_prefill", w.subset(w.groups["prefill_seqs"]),
                [("tensor", 0.50), ("hbm", 0.70)] if cfg == 3 else [("tensor", 0.50)])
            add(f"{key}_decode", w.subset(w.groups["decode_seqs"]), [("hbm", 0.70)])
        if w is not w_head:
            del w
            gc.collect()
            torch.cuda.empty_cache()
    # Pensieve's kernel microbenchmark (Fig. 12): the multi-token kernels on the
    # prefill sub-batches with paged blocks against the same draw with every sequence's
    # blocks consecutive, each kernel forced in turn
    pvc = {}
    for cfg in (3, 4):
        wp = w_head if str(cfg) == str(head) and not args.subset and not args.contiguous \
            and args.block_size is None else workloads.make(cfg, device=dev)
        wc = workloads.make(cfg, device=dev, contiguous=True)
        for kern, pair in (("tc_kernel", -1), ("tc2_kernel", 1)):
            a_ms, _ = time_attention(wp.subset(wp.groups["prefill_seqs"]), dev, tc_pair=pair)
            b_ms, _ = time_attention(wc.subset(wc.groups["prefill_seqs"]), dev, tc_pair=pair)
            pvc[f"cfg{cfg}_prefill_{kern}"] = {"paged_ms": a_ms, "contiguous_ms": b_ms,
                                               "paged_over_contiguous": a_ms / b_ms}
            log(f"paged vs contiguous: cfg{cfg} prefill {kern}: {a_ms:.4f} / {b_ms:.4f} ms")
        del wc
        if wp is not w_head:
            del wp
        gc.collect()
        torch.cuda.empty_cache()
    res["paged_vs_contiguous"] = pvc
    res["_note"] = ("attention kernels of one planned call (tables uploaded once), CUDA "
                    "events over 30 calls after 5 warm-up calls; frac = roofline time / "
                    "measured; bar: decode-dominated >= 0.70 of HBM, prefill-dominated >= "
                    "0.50 of the tensor roofline (config 3's prefill is HBM-bound: its "
                    "binding roofline is accepted too)")
    return res


def swap_measure(w, dev, reps=20):
    """pa_swap_blocks bandwidth at this workload's block shape: n scattered blocks of
    both pools out to page-locked host pools and back in, CUDA-event timed, beside one
    contiguous copy-engine transfer of the same bytes (pinned host -> device)."""
    import torch
    import paged_kv_cache_02_gb300 as pa
    nb = int(w.k_pool.shape[0])
    n = max(1, min(512, nb // 2))
    shape = tuple(w.k_pool.shape[1:])
    kh = torch.empty((n,) + shape, dtype=torch.bfloat16).pin_memory()
    vh = torch.empty((n,) + shape, dtype=torch.bfloat16).pin_memory()
    g = torch.Generator().manual_seed(7)
    src = torch.randperm(nb, generator=g)[:n].to(torch.int32).to(dev)
    dst = torch.randperm(n, generator=g).to(torch.int32).to(dev)
    nbytes = 2 * n * kh[0].numel() * 2
    flat = torch.empty(nbytes // 2, dtype=torch.bfloat16).pin_memory()
    flat_d = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / reps / 1e3

    t_out = timed(lambda: pa.pa_swap_blocks(w.k_pool, w.v_pool, kh, vh, src, dst, "out"))
    t_in = timed(lambda: pa.pa_swap_blocks(w.k_pool, w.v_pool, kh, vh, dst, src, "in"))
    t_ce = timed(lambda: flat_d.copy_(flat, non_blocking=True))
    err = pa.pa_get_device_error()
    return {"blocks": n, "bytes_per_call": nbytes, "out_gbs": nbytes / t_out / 1e9,
            "in_gbs": nbytes / t_in / 1e9, "copy_engine_h2d_gbs": nbytes / t_ce / 1e9,
            "device_error": err,
            "note": "scattered block ids both sides; copy engine = one contiguous pinned copy"}


def block_manager_host(w, steps=32):
    """Host cost of the KV block manager (pa_bm_*) at this workload's scale: the
    sequences' histories are appended once, then each timed step appends one token to
    every sequence (slots and the copy-on-write decision) and exports all block-table
    rows and context lengths, as a decode step of a serving loop would."""
    import ctypes as C
    import numpy as np
    import paged_kv_cache_02_gb300 as pa
    B = int(w.block_size)
    N = len(w.context_lens)
    L = np.asarray(w.context_lens, np.int64)
    hist = np.maximum(L - np.asarray(w.query_lens, np.int64), 0).astype(np.int32)
    # every history held unshared (the manager's pool, not the workload's, is sized for
    # that: a shared-prefix workload's pool is smaller), plus room for the timed steps
    nb = int(sum(-(-int(x) // B) for x in hist)) + N * (-(-steps // B) + 1)
    mb = int(max(-(-(int(x) + steps) // B) for x in hist)) + 1
    bm = pa.BlockManager(nb, B)
    ids = np.arange(N, dtype=np.int64)
    for s in range(N):
        bm.add(s)
    bm.append_batch(ids.tolist(), hist.tolist())
    lib = pa.library()
    ones = np.ones(N, np.int32)
    slots = np.zeros(N, np.int64)
    src = np.zeros(N, np.int32)
    dst = np.zeros(N, np.int32)
    bt = np.zeros((N, mb), np.int32)
    cl = np.zeros(N, np.int32)
    n_cow = C.c_int32(0)
    t0 = time.perf_counter()
    for _ in range(steps):
        st = lib.pa_bm_append(bm._h, ids.ctypes.data, ones.ctypes.data, N, slots.ctypes.data,
                              src.ctypes.data, dst.ctypes.data, C.byref(n_cow))
        st |= lib.pa_bm_tables(bm._h, ids.ctypes.data, N, mb, bt.ctypes.data, cl.ctypes.data)
        if st:
            return {"error": int(st)}
    dt = time.perf_counter() - t0
    bm.close()
    return {"us_per_step": dt / steps * 1e6, "seqs": N, "steps": steps,
            "includes": "one token appended to every sequence (slots, copy-on-write decision) "
                        "and every block-table row and context length exported, host only"}


def cpu_baseline(args, w):
    if args.no_cpu_baseline:
        return None
    import oracle
    from workloads import host_bits as u16
    orc = oracle.default()
    host = {"q": u16(w.q), "k_pool": u16(w.k_pool), "v_pool": u16(w.v_pool),
            "k_new": u16(w.k_new), "v_new": u16(w.v_new)}
    n = os.cpu_count() or 1
    v, sample, _ = oracle_step_sample(w, orc, host, n, budget_s=args.cpu_budget)
    v1, sample1, _ = oracle_step_sample(w, orc, host, 1, budget_s=max(1.0, args.cpu_budget / 4))
    return {"value": v, "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample,
            "one_core": {"value": v1, "unit": UNIT, "sample": sample1}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="3",
                    help="workload: 1..5 or 5cow (default 3, the Pensieve-style mixed batch)")
    ap.add_argument("--fused", action="store_true",
                    help="time the step as the fused call (pa_attention_write_planned) instead "
                         "of pa_write_kv + pa_attention_planned; the other form is reported "
                         "beside it either way")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config attention sweep (key 'configs')")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tc-min-rows", type=int, default=0,
                    help="plan option: rows from which items use the tensor cores (0 = default)")
    ap.add_argument("--out", choices=["f32", "bf16"], default="f32",
                    help="attention output dtype")
    ap.add_argument("--tc-pair", type=int, default=0,
                    help="plan option: 0 = automatic (default), 1 = 256-row tensor-core items, "
                         "-1 = 128-row only")
    ap.add_argument("--max-chunk", type=int, default=0,
                    help="plan option: split-KV chunk length (0 = automatic)")
    ap.add_argument("--subset", choices=["prefill", "decode"], default=None,
                    help="run only the prefill or decode sequences of a mixed batch (3, 4)")
    ap.add_argument("--max-seqs", type=int, default=None,
                    help="keep only the first N sequences (config 2) or N conversations + 2N decodes (config 3), for profiler captures")
    ap.add_argument("--block-size", type=int, default=None,
                    help="block-size sweep: config 2 or 4 with another block size")
    ap.add_argument("--contiguous", action="store_true",
                    help="config 2, 3 or 4 with each sequence's blocks consecutive")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.config_key = f"cfg{args.config}"
    rank, local, world = dist_setup(args.gpus)

    import workloads
    cfg = args.config if args.config == "5cow" else int(args.config)

    if args.impl == "reference":
        if rank != 0:
            return
        w = workloads.make(cfg, device="cpu" if cfg == 1 else "cuda")
        run_reference(args, w, cfg_dict(w, cfg))
        return

    import torch
    torch.cuda.set_device(local)
    w = workloads.make(cfg, device=f"cuda:{local}", max_seqs=args.max_seqs,
                       block_size=args.block_size, contiguous=args.contiguous)
    if args.block_size is not None:
        args.config_key += f"_B{args.block_size}"
    if args.contiguous:
        args.config_key += "_contiguous"
    if args.subset:
        w = w.subset(w.groups[f"{args.subset}_seqs"])
        args.config_key += f"_{args.subset}"
    run_gpu(args, w, cfg_dict(w, cfg, args.subset), rank, local, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cfg_dict(w, cfg, subset=None):
    tag = f" ({subset} sequences only)" if subset else ""
    return {"workload": f"config {cfg}: {w.name}{tag}", "num_seqs": w.num_seqs, "total_q": w.total_q,
            "kv_tokens": int(w.context_lens.sum()), "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
            "block_size": w.block_size, "num_blocks": w.num_blocks,
            "cow_pairs": int(len(w.cow_src)), "new_tokens": int(len(w.new_seq)),
            "l2": "no flush: the K/V pools read each step are larger than the 129 MB L2",
            "parallelism": "replicas only (one independent batch per GPU)"}


if __name__ == "__main__":
    main()
