"""CPU-side checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, and its host logic (argument checks, the plan) behaves. No kernel runs."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_02_gb300 import _build
    _build.build()
    import paged_kv_cache_02_gb300 as pa
    return pa


def declared_entry_points():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(pa_[a-z0-9_]+)\s*\(",
                                src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for must in ("pa_write_kv", "pa_copy_blocks", "pa_attention", "pa_plan_create",
                 "pa_plan_destroy", "pa_status_string", "pa_slot_mapping", "pa_plan_upload",
                 "pa_attention_planned", "pa_bm_create", "pa_bm_append", "pa_bm_fork",
                 "pa_bm_free", "pa_bm_tables"):
        assert must in names, names


def test_library_exports_every_declared_symbol(pa):
    lib = pa.library()
    for name in declared_entry_points():
        assert hasattr(lib, name), f"libpa.so does not export {name}"


def test_status_strings_and_version(pa):
    lib = pa.library()
    for s in range(8):
        assert lib.pa_status_string(s) != b"unknown status"
    assert lib.pa_status_string(99) == b"unknown status"
    assert "sm_103a" in pa.version()


def plan(pa, L, q, Hq=4, Hkv=4, D=64, B=16, **kw):
    mb = max(1, max((-(-l // B) for l in L), default=1))
    return pa.Plan(L, q, Hq, Hkv, D, B, mb, **kw)


@pytest.mark.parametrize("bad,status", [
    (dict(L=[5], q=[6]), 3),                      # query longer than context
    (dict(L=[5], q=[-1]), 3),
    (dict(Hq=6, Hkv=4), 2),                        # heads not a multiple
    (dict(D=96), 4),                               # head dim not built
    (dict(B=12), 4),                               # block size not a power of two
    (dict(wait_limit_ns=-5), 1),                   # a negative wait bound
])
def test_plan_rejects(pa, bad, status):
    args = dict(L=[5, 9], q=[1, 2], Hq=4, Hkv=4, D=64, B=16)
    args.update(bad)
    L, q = args.pop("L"), args.pop("q")
    if len(L) != len(q):
        L = L[:len(q)]
    with pytest.raises(pa.PagedAttentionError) as e:
        plan(pa, L, q, **args)
    assert e.value.status == status


def test_plan_options_reserved_must_be_zero(pa):
    import ctypes as C
    from paged_kv_cache_02_gb300 import _binding as b
    opts = b._Options(0, 0, 0, 0, 0, 1000)
    opts.reserved[1] = 7
    cl = (C.c_int32 * 1)(9)
    ql = (C.c_int32 * 1)(1)
    h, ws = C.c_void_p(), C.c_size_t(0)
    assert b._lib().pa_plan_create(cl, ql, 1, 4, 4, 64, 16, 1, C.byref(opts), C.byref(h),
                                   C.byref(ws)) == 1
    opts.reserved[1] = 0
    assert b._lib().pa_plan_create(cl, ql, 1, 4, 4, 64, 16, 1, C.byref(opts), C.byref(h),
                                   C.byref(ws)) == 0
    assert b._lib().pa_plan_destroy(h) == 0


def test_plan_rejects_short_table(pa):
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.Plan([40], [1], 4, 4, 64, 16, 2)
    assert e.value.status == 3


def _coverage(items, L, q, g, Hkv):
    """Every (seq, kv head, row) covered by exactly one row range; for each the key
    chunks partition [0, last visible key] without overlap."""
    seen = {}
    for path, s, kvh, rb, rc, kb, ke, part, q0 in items:
        for r in range(rb, rb + rc):
            seen.setdefault((s, kvh, r), []).append((kb, ke, part))
    for s in range(len(L)):
        for kvh in range(Hkv):
            for r in range(q[s] * g):
                assert (s, kvh, r) in seen, (s, kvh, r)
                ranges = sorted(seen[(s, kvh, r)])
                assert ranges[0][0] == 0
                for (a0, a1, _), (b0, b1, _) in zip(ranges, ranges[1:]):
                    assert a1 == b0
                t = r // g
                assert ranges[-1][1] >= L[s] - q[s] + t + 1
                assert ranges[-1][1] <= L[s]
                if len(ranges) == 1:
                    assert ranges[0][2] == -1
                else:
                    assert all(p >= 0 for _, _, p in ranges)
    assert len(seen) == sum(qq * g * Hkv for qq in q)


@pytest.mark.parametrize("chunk", [0, 128, 256])
def test_plan_covers_every_row_and_key(pa, chunk):
    L = [7, 33, 64, 100, 0, 513, 2048]
    q = [1, 1, 7, 17, 0, 40, 1]
    for Hq, Hkv in ((4, 4), (8, 2), (16, 1)):
        p = plan(pa, L, q, Hq=Hq, Hkv=Hkv, max_chunk_tokens=chunk)
        items = p.items()
        _coverage(items, L, q, Hq // Hkv, Hkv)
        st = p.stats()
        assert st["total_q"] == sum(q) and st["kv_tokens"] == sum(L)
        assert st["n_dec_items"] + st["n_tc_items"] == len(items)
        assert st["workspace_bytes"] >= 256
        if chunk:
            assert st["chunk_tokens"] == chunk
            assert all(ke - kb <= chunk for *_, kb, ke, _, _ in items)
        # partial rows are distinct
        parts = [(pt + i) for (_, _, _, _, rc, _, _, pt, _) in items if pt >= 0 for i in range(rc)]
        assert len(parts) == len(set(parts)) == st["n_partials"]
        # q_row0 = prefix sum of query lens
        pref = np.concatenate([[0], np.cumsum(q)])
        for it in items:
            assert it[8] == pref[it[1]]


def test_plan_pair_tiles(pa):
    """With tc_pair=1 tensor-core rows go in 256-row items (two 128-row tiles); rows that
    do not fill a whole item form the sequence's first item, a 128-row item when at most
    128 rows are left over; tc_pair=-1 keeps 128-row items only."""
    L = [300, 1000, 700, 129, 2000]
    q = [300, 40, 33, 129, 1]
    g, Hkv = 8, 2
    p = plan(pa, L, q, Hq=g * Hkv, Hkv=Hkv, D=128, max_chunk_tokens=256, tc_pair=1)
    items = p.items()
    _coverage(items, L, q, g, Hkv)
    rows_by_path = {}
    for path, s, kvh, rb, rc, *_ in items:
        rows_by_path.setdefault(int(path), []).append((int(s), int(rc)))
    assert all(rc <= 128 for _, rc in rows_by_path.get(1, []))
    assert all(128 < rc <= 256 for _, rc in rows_by_path[2])
    assert p.stats()["n_tc_pair_items"] == len(rows_by_path[2])
    # 300 tokens x 8 heads = 2400 rows = 9 x 256 + 96
    assert sorted(rc for s, rc in set((s, rc) for s, rc in rows_by_path[2] if s == 0)) == [256]
    # the leading partial item: rows [0, 96) of sequence 0 (2400 = 96 + 9 x 256), each
    # KV head, one-tile path, over keys up to the last of its 12 tokens
    lead = [it for it in items if it[1] == 0 and it[3] == 0]
    assert len(lead) > 0 and all(it[0] == 1 and it[4] == 96 for it in lead)
    assert max(it[6] for it in lead) == L[0] - q[0] + 96 // g
    p1 = plan(pa, L, q, Hq=g * Hkv, Hkv=Hkv, D=128, max_chunk_tokens=256, tc_pair=-1)
    items1 = p1.items()
    _coverage(items1, L, q, g, Hkv)
    assert 2 not in set(items1[:, 0].tolist())
    assert p1.stats()["n_tc_pair_items"] == 0


def test_plan_partial_tile_first_reads_fewer_keys(pa):
    """The partial row tile of a sequence comes first: every other tile is whole, and the
    keys the items read (summed over items) are n (T - r) fewer than with the partial tile
    last (n whole tiles of T rows, r rows over; g = 1)."""
    L, q = [800, 2300, 300], [800, 300, 300]      # a recomputed context, a new prompt
    for pair, T in ((1, 256), (-1, 128)):
        p = plan(pa, L, q, Hq=4, Hkv=4, D=128, tc_pair=pair)
        items = p.items()
        _coverage(items, L, q, 1, 4)
        for s in range(3):
            mine = sorted(set((int(it[3]), int(it[4])) for it in items
                              if it[1] == s and it[2] == 0))
            r = q[s] % T
            assert mine[0] == (0, r if r else T)
            assert all(rc == T for _, rc in mine[1:])
            keys = sum(int(it[6]) - int(it[5]) for it in items if it[1] == s and it[2] == 0)
            n = q[s] // T
            # partial tile last: tiles end at T, 2T, ..., nT, then q
            last = sum(L[s] - q[s] + T * k for k in range(1, n + 1)) + (L[s] if r else 0)
            assert keys == last - (n * (T - r) if r else 0)


def _tc_intensity(L, q, g, Hkv, D=128):
    """FLOPs per byte of the multi-token tensor-core work (rows > 16): Q K^T and P V over
    the causally visible keys, against K and V read once per (sequence, KV head), Q in
    bf16 and the output in fp32."""
    flops = byts = 0.0
    for l, n in zip(L, q):
        if n * g <= 16:
            continue
        visible = sum(l - n + t + 1 for t in range(n))
        flops += 4.0 * D * g * Hkv * visible
        byts += 4.0 * D * Hkv * l + 6.0 * D * g * Hkv * n
    return flops / byts


def test_plan_pair_automatic(pa):
    """By default 256-row items are used only when the multi-token work is memory-bound:
    FLOPs per byte of K/V, Q and output below the machine balance of 280."""
    g, Hkv = 1, 8
    # short prompts over long histories: little work per K/V byte
    L_lo, q_lo = [3000, 2500, 2800], [200, 180, 250]
    # long prompts packed 8 heads per KV head: much work per K/V byte
    L_hi, q_hi = [1500, 1200, 1800], [256, 200, 240]
    assert _tc_intensity(L_lo, q_lo, g, Hkv) < 280
    assert _tc_intensity(L_hi, q_hi, 8, Hkv) > 280
    lo = plan(pa, L_lo, q_lo, Hq=g * Hkv, Hkv=Hkv, D=128)
    hi = plan(pa, L_hi, q_hi, Hq=8 * Hkv, Hkv=Hkv, D=128)
    assert lo.stats()["n_tc_pair_items"] > 0
    assert hi.stats()["n_tc_pair_items"] == 0 and hi.stats()["n_tc_items"] > 0
    # the explicit settings override the choice either way
    assert plan(pa, L_hi, q_hi, Hq=8 * Hkv, Hkv=Hkv, D=128,
                tc_pair=1).stats()["n_tc_pair_items"] > 0
    assert plan(pa, L_lo, q_lo, Hq=g * Hkv, Hkv=Hkv, D=128,
                tc_pair=-1).stats()["n_tc_pair_items"] == 0


def test_plan_decode_items(pa):
    """A (sequence, KV head) pair with at most 16 tensor-core rows becomes one item of
    path 3 (keys on the 128-row side) when Hq / Hkv divides 16; tc_decode=-1 disables it."""
    L = [300, 1000, 700, 40, 2000]
    q = [1, 2, 3, 40, 1]
    for g in (1, 2, 4, 8, 16):
        Hkv = 2
        p = plan(pa, L, q, Hq=g * Hkv, Hkv=Hkv, D=128, max_chunk_tokens=256, tc_min_rows=1)
        items = p.items()
        _coverage(items, L, q, g, Hkv)
        for path, s, kvh, rb, rc, *_ in items:
            if q[s] * g <= 16:
                assert path == 3 and rb == 0 and rc == q[s] * g
            else:
                assert path in (1, 2)
        st = p.stats()
        assert st["n_tc_decode_items"] == sum(1 for it in items if it[0] == 3)
        p1 = plan(pa, L, q, Hq=g * Hkv, Hkv=Hkv, D=128, tc_min_rows=1, tc_decode=-1)
        assert 3 not in set(p1.items()[:, 0].tolist())
    # g = 3 does not divide 16: no such items
    p3 = plan(pa, L, q, Hq=6, Hkv=2, D=128, tc_min_rows=1)
    assert p3.stats()["n_tc_decode_items"] == 0


def test_plan_orders_longest_first(pa):
    L = list(range(100, 2100, 50))
    p = plan(pa, L, [1] * len(L), num_sms=1000)    # one round of the walk
    lens = [ke - kb for *_, kb, ke, _, _ in p.items()]
    assert lens == sorted(lens, reverse=True)


def test_plan_snake_rounds(pa):
    """Longest first, every other round of G = num_sms items reversed: CTA c (which walks
    items c, c + G, ...) gets the c-th longest of round 0, the c-th shortest of round 1."""
    L = [100 + 37 * i for i in range(10)]
    p = plan(pa, L, [1] * len(L), Hq=1, Hkv=1, num_sms=4, max_chunk_tokens=4096)
    lens = [int(ke - kb) for *_, kb, ke, _, _ in p.items()]
    desc = sorted(lens, reverse=True)
    assert lens == desc[0:4] + desc[4:8][::-1] + desc[8:10]
    loads = [sum(lens[c::4]) for c in range(4)]
    plain = [sum(desc[c::4]) for c in range(4)]
    assert max(loads) - min(loads) <= max(plain) - min(plain)


def test_plan_auto_split_fills_the_gpu(pa):
    # one very long decode: 8 KV heads x 100k keys must be split into many chunks
    p = pa.Plan([100_000], [1], 8, 8, 128, 16, 100_000 // 16 + 1, num_sms=152)
    st = p.stats()
    assert st["n_split_groups"] == 8
    assert st["n_dec_items"] + st["n_tc_items"] >= 152
    # a large decode batch needs no split
    L = [1000 + 3 * i for i in range(256)]
    p2 = pa.Plan(L, [1] * 256, 40, 40, 128, 16, 200, num_sms=152)
    assert p2.stats()["n_split_groups"] == 0


def test_empty_batch(pa):
    p = pa.Plan([0, 0], [0, 0], 4, 4, 64, 16, 1)
    assert p.stats()["total_q"] == 0 and len(p.items()) == 0


def test_plan_upload_checks_arguments_before_enqueuing(pa):
    """pa_plan_upload rejects a missing, short or misaligned workspace synchronously,
    before any copy is enqueued (so these checks run without a GPU)."""
    import ctypes as C
    lib = pa.library()
    p = pa.Plan([300, 40], [20, 1], 8, 2, 128, 16, 32, num_sms=152)
    need = p.workspace_bytes
    assert lib.pa_plan_upload(None, C.c_void_p(4096), need, None) == 1     # no plan
    assert lib.pa_plan_upload(p._h, None, need, None) == 1                  # no workspace
    assert lib.pa_plan_upload(p._h, C.c_void_p(4096), need - 1, None) == 2  # too small
    assert lib.pa_plan_upload(p._h, C.c_void_p(4096 + 16), need, None) == 4  # misaligned
    empty = pa.Plan([0], [0], 8, 2, 128, 16, 1)
    assert lib.pa_plan_upload(empty._h, None, 0, None) == 0                 # nothing to do
