"""KV block manager: the oracle's pins, and the library's manager against them and
against the oracle (host code only: no GPU)."""
import ctypes as C

import numpy as np
import pytest

from oracle.block_manager import BlockManager, OutOfBlocks
from tests import bm_checks as bc


def oracle_factory(mutation=0):
    return lambda nb, B, order, nhb=0: BlockManager(nb, B, free_order=order, mutation=mutation,
                                                     num_host_blocks=nhb)


@pytest.mark.parametrize("check", bc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle_factory())


MUTANTS = {1: "copy keeps the shared count", 2: "shared block written in place",
           3: "offset off by one", 4: "freed blocks lost", 5: "fork not counted",
           6: "swap copies shared blocks twice", 7: "swap keeps source references"}


@pytest.mark.parametrize("mutation", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_oracle_planted_mistake_is_caught(mutation):
    caught = []
    for check in bc.ALL_CHECKS:
        try:
            check(oracle_factory(mutation))
        except (AssertionError, OutOfBlocks, IndexError, KeyError):
            caught.append(check.__name__)
    assert caught, f"mutation {MUTANTS[mutation]} passed every pin"


def test_oracle_rejects_bad_calls():
    bm = BlockManager(8, 4)
    bm.add(1)
    with pytest.raises(KeyError):
        bm.add(1)
    with pytest.raises(KeyError):
        bm.append(2, 1)
    with pytest.raises(KeyError):
        bm.fork(2, 3)
    with pytest.raises(ValueError):
        bm.append_batch([1, 1], [1, 1])
    with pytest.raises(ValueError):
        bm.append(1, -1)
    with pytest.raises(ValueError):
        BlockManager(4, 4, free_order=[0, 1, 2, 2])


# ---------------------------------------------------------------- the library's manager

@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_02_gb300 import _build
    _build.build()
    import paged_kv_cache_02_gb300 as pa
    return pa


def library_factory(pa):
    return lambda nb, B, order, nhb=0: pa.BlockManager(nb, B, free_order=order,
                                                        num_host_blocks=nhb)


@pytest.mark.parametrize("check", bc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_library_pin(pa, check):
    """The library's manager passes the same pins as the oracle."""
    check(library_factory(pa))


@pytest.mark.parametrize("seed,nb,B", [(11, 48, 4), (12, 20, 16), (13, 300, 2), (14, 16, 8)])
def test_library_matches_oracle(pa, seed, nb, B):
    """Same operations, same decisions: every slot, copy, table and count equal."""
    ops = bc.random_ops(seed, n_ops=400)
    lib, orc = pa.BlockManager(nb, B), BlockManager(nb, B)
    log_lib, log_orc = [], []
    live_lib = bc.run_ops(lib, ops, nb, B, log_lib)
    live_orc = bc.run_ops(orc, ops, nb, B, log_orc)
    assert log_lib == log_orc
    assert any(e != ("full",) and e[1] for e in log_orc), "no copy-on-write exercised"
    assert ("full",) in log_orc or nb > 100
    assert sorted(live_lib) == sorted(live_orc)
    for s in live_orc:
        assert lib.table(s) == orc.table(s) and lib.filled(s) == orc.filled(s)
    assert [lib.refcount(b) for b in range(nb)] == [orc.refcount(b) for b in range(nb)]
    assert lib.num_free() == orc.num_free()


@pytest.mark.parametrize("seed,nb,nhb,B", [(21, 40, 24, 4), (22, 30, 60, 8), (25, 64, 8, 2)])
def test_library_matches_oracle_with_swaps(pa, seed, nb, nhb, B):
    """Histories with swaps out and in: the same pairs, tables, counts, residency."""
    ops = bc.random_ops(seed, n_ops=400, swaps=True)
    lib = pa.BlockManager(nb, B, num_host_blocks=nhb)
    orc = BlockManager(nb, B, num_host_blocks=nhb)
    log_lib, log_orc = [], []
    live = bc.run_ops(lib, ops, nb, B, log_lib, num_host_blocks=nhb)
    bc.run_ops(orc, ops, nb, B, log_orc, num_host_blocks=nhb)
    assert log_lib == log_orc
    assert any(e[0] == "swap_in" and e[1] for e in log_orc), "no swap-in exercised"
    for s in live:
        assert lib.table(s) == orc.table(s) and lib.is_on_host(s) == orc.is_on_host(s)
    assert [lib.host_refcount(b) for b in range(nhb)] == [orc.host_refcount(b)
                                                          for b in range(nhb)]
    assert lib.num_free_host() == orc.num_free_host() and lib.num_free() == orc.num_free()


def test_library_tables_for_attention(pa):
    """pa_bm_tables rows feed the attention calls: padded with -1, lengths = tokens."""
    bm = pa.BlockManager(32, 4, free_order=list(range(31, -1, -1)))
    for s, n in ((0, 7), (1, 4), (2, 0)):
        bm.add(s)
        bm.append(s, n)
    bm.fork(0, 3)
    bt, cl = bm.tables([3, 1, 2, 0], 3)
    assert bt.tolist() == [[31, 30, -1], [29, -1, -1], [-1, -1, -1], [31, 30, -1]]
    assert cl.tolist() == [7, 4, 0, 7]
    with pytest.raises(pa.PagedAttentionError):
        bm.tables([0], 1)                   # 2 blocks do not fit in 1 column


def test_library_rejects_bad_calls(pa):
    bm = pa.BlockManager(8, 4)
    bm.add(1)
    with pytest.raises(KeyError):
        bm.add(1)
    with pytest.raises(KeyError):
        bm.append(2, 1)
    with pytest.raises(KeyError):
        bm.fork(2, 3)
    with pytest.raises(KeyError):
        bm.free_seq(5)
    with pytest.raises(ValueError):
        bm.append_batch([1, 1], [1, 1])
    with pytest.raises(ValueError):
        bm.append(1, -1)
    lib = pa.library()
    h = C.c_void_p()
    bad = np.array([0, 1, 1, 3], np.int32)
    assert lib.pa_bm_create(4, 4, bad.ctypes.data, C.byref(h)) == 1
    assert lib.pa_bm_create(0, 4, None, C.byref(h)) == 1
    n = C.c_int32(0)
    # a duplicate id inside one step is refused by the library itself too
    ids = np.array([1, 1], np.int64)
    cnt = np.array([1, 1], np.int32)
    slots = np.zeros(2, np.int64)
    src = np.zeros(2, np.int32)
    assert lib.pa_bm_append(bm._h, ids.ctypes.data, cnt.ctypes.data, 2, slots.ctypes.data,
                            src.ctypes.data, src.ctypes.data, C.byref(n)) == 1
    assert lib.pa_bm_refcount(bm._h, 8, C.byref(n)) == 3


@pytest.mark.parametrize("impl", ["oracle", "library"])
def test_config5cow_copies_are_the_managers(pa, impl):
    """The fork step of config 5cow (32 prompts of 1032 tokens x 8 samples, block size
    16) replayed through a block manager: prompt, fork to 8 samples, one decode token
    each in sample order. The manager's copies, tables and slots equal the workload's,
    so the harness's copy list is the manager's decision (vLLM post, 2.1)."""
    import workloads
    w = workloads.make("5cow")
    B, nb = w.block_size, int(w.k_pool.shape[0])
    P, S, prompt = 32, 8, 1032
    n_shared = -(-prompt // B)
    bt = w.block_table
    order = []
    for p in range(P):
        order += bt[p * S + S - 1, :n_shared].tolist()        # the last sample keeps them
        order += w.cow_dst[p * (S - 1):(p + 1) * (S - 1)].tolist()
    rest = sorted(set(range(nb)) - set(order))
    bm = (BlockManager(nb, B, free_order=order + rest) if impl == "oracle"
          else pa.BlockManager(nb, B, free_order=order + rest))
    copies, slots = [], []
    for p in range(P):
        bm.add((p, 0))
        bm.append((p, 0), prompt)
        for s in range(1, S):
            bm.fork((p, 0), (p, s))
        sl, cp = bm.append_batch([(p, s) for s in range(S)], [1] * S)
        slots += sl
        copies += cp
    assert copies == list(zip(w.cow_src.tolist(), w.cow_dst.tolist()))
    for i in range(P * S):
        t = bm.table((i // S, i % S))
        assert t == bt[i, :len(t)].tolist()
    pos = np.asarray(w.context_lens, np.int64) - 1
    want = [int(bt[i, pos[i] // B]) * B + int(pos[i] % B) for i in range(P * S)]
    assert slots == want


@pytest.mark.parametrize("impl", ["oracle", "library"])
def test_edge_cases(pa, impl):
    make = oracle_factory() if impl == "oracle" else library_factory(pa)
    bm = make(8, 4, None)
    bm.add(0)
    assert bm.append(0, 0) == ([], []) and bm.table(0) == [] and bm.filled(0) == 0
    bm.fork(0, 1)                                  # fork of an empty request
    s0, c0 = bm.append(0, 2)
    s1, c1 = bm.append(1, 2)
    assert c0 == c1 == [] and bm.table(0) != bm.table(1) and bm.num_free() == 6
    bm.free_seq(1)
    bm.add(1)                                      # an id can be reused after free
    assert bm.table(1) == [] and bm.num_free() == 7
    bm.append(0, 2)                                # fills block of 0 exactly (4 tokens)
    bm.fork(0, 2)
    s, c = bm.append(2, 1)                         # full shared block: new block, no copy
    assert c == [] and len(bm.table(2)) == 2 and bm.table(2)[0] == bm.table(0)[0]
    assert bm.refcount(bm.table(0)[0]) == 2
    # block size 1: every token takes a block; forks never need a copy
    one = make(6, 1, None)
    one.add("x"); one.append("x", 3); one.fork("x", "y")
    assert one.append_batch(["x", "y"], [1, 1])[1] == []
    assert one.num_free() == 1


def test_swap_roundtrip_moves_the_right_blocks(pa):
    """The library's swap pairs drive a model copy (the oracle's block swap) on numpy
    pools; the same scenario runs on the GPU with pa_swap_blocks in test_swap_gpu."""
    from oracle.swap import swap_blocks
    rng = np.random.default_rng(3)
    kd = rng.integers(0, 2**16, (16, 4, 2, 8), dtype=np.uint16)
    vd = rng.integers(0, 2**16, (16, 4, 2, 8), dtype=np.uint16)
    kh = np.zeros((12, 4, 2, 8), np.uint16)
    vh = np.zeros_like(kh)
    bm = pa.BlockManager(16, 4, num_host_blocks=12)

    def gather(table):
        return np.concatenate([kd[table], vd[table]])

    def scribble(blocks):
        kd[blocks] = 7
        vd[blocks] = 9

    def move(pairs, direction):
        src = [a for a, _ in pairs]
        dst = [b for _, b in pairs]
        if direction == "out":
            swap_blocks(kd, vd, kh, vh, src, dst)
        else:
            swap_blocks(kh, vh, kd, vd, src, dst)

    bc.swap_roundtrip(bm, gather, scribble, move)
