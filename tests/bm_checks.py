"""Pins for a KV block manager (the oracle's, and the same checks for the library's).

Each ``check_*`` takes a factory ``make(num_blocks, block_size, free_order,
num_host_blocks=0)`` that returns an object with the oracle's interface (add, fork,
free_seq, append, append_batch, swap_out, swap_in, table, filled, num_free,
refcount, host_refcount, num_free_host, is_on_host) and raises AssertionError when
the manager disagrees with something that does not come from the manager itself:

* the vLLM post's worked example ("1. overall architecture": slots, #filled, the
  third block) and its copy-on-write example ("2.1 parallel sampling"), stored in
  ``tests/golden``;
* the property a KV manager exists for, checked by brute force: after any seeded
  sequence of add / fork / append / free, replaying the returned writes and block
  copies on a model pool (one token id per slot) lets every live sequence read back
  exactly its own tokens at every position;
* bookkeeping invariants: a block's count equals the number of block-table entries
  naming it, free and referenced blocks partition the pool, a table has
  ceil(L / B) entries;
* all-or-nothing on an exhausted pool;
* swapping (vLLM post, "3. scheduling and preemption"): after any seeded history
  with swaps out and in, every request reads back its tokens from the pool it lives
  in, and blocks shared by requests swapped together stay shared.
"""
import json
import os
import random

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _order_first(first, num_blocks):
    return list(first) + [b for b in range(num_blocks) if b not in first]


def check_worked_example(make):
    g = _golden("worked_example_slots.json")
    B, bt = g["block_size"], g["block_table"]
    bm = make(16, B, _order_first(bt, 16))
    bm.add("req")
    for step in g["steps"]:
        slots, copies = bm.append("req", len(step["positions"]))
        assert copies == [], step["what"]
        assert slots == step["slots"], (step["what"], slots, step["slots"])
        table = bm.table("req")
        # #filled of the request's last block, as the block table records it
        last = str(table[-1])
        assert bm.filled("req") == step["filled_after"][last], step["what"]
    assert bm.table("req") == bt


def check_cow_example(make):
    g = _golden("cow_example.json")
    B = g["block_size"]
    first = g["tables_before"]["A1"] + [c[1] for c in g["copies"]]
    bm = make(16, B, _order_first(first, 16))
    bm.add("A1")
    bm.append("A1", g["prompt_len"])
    bm.fork("A1", "A2")
    assert bm.table("A1") == g["tables_before"]["A1"] and bm.table("A2") == g["tables_before"]["A2"]
    for b, c in g["refcount_before"].items():
        assert bm.refcount(int(b)) == c, ("before", b)
    all_copies = []
    for wr in g["writes"]:
        slots, copies = bm.append(wr["sample"], 1)
        assert slots == [wr["slot"]], (wr, slots)
        all_copies += [list(c) for c in copies]
    assert all_copies == g["copies"], all_copies
    for name, t in g["tables_after"].items():
        assert bm.table(name) == t, name
    for b, c in g["refcount_after"].items():
        assert bm.refcount(int(b)) == c, ("after", b)


def _invariants(bm, model, num_blocks, B, host=None, num_host_blocks=0):
    refs = [0] * num_blocks
    hrefs = [0] * num_host_blocks
    for s in model:
        t = bm.table(s)
        assert len(t) == -(-len(model[s]) // B), ("table length", s)
        on_host = host is not None and s in host
        for b in t:
            if on_host:
                hrefs[b] += 1
            else:
                refs[b] += 1
    for b in range(num_blocks):
        assert bm.refcount(b) == refs[b], ("refcount", b, bm.refcount(b), refs[b])
    used = sum(1 for r in refs if r > 0)
    assert bm.num_free() + used == num_blocks, ("free + used", bm.num_free(), used)
    if num_host_blocks:
        for b in range(num_host_blocks):
            assert bm.host_refcount(b) == hrefs[b], ("host refcount", b)
        hused = sum(1 for r in hrefs if r > 0)
        assert bm.num_free_host() + hused == num_host_blocks, "host free + used"


def random_ops(seed, n_ops=300, swaps=False):
    """Seeded operation list: ("add", s), ("fork", parent, child), ("append", [(s, n)]),
    ("free", s), and with ``swaps`` ("swap_out", [s...]) / ("swap_in", [s...]), over at
    most 12 live sequences. Operations that do not apply when replayed (an append to a
    swapped-out request, ...) are dropped by ``run_ops``."""
    rng = random.Random(seed)
    ops, live, nxt = [], [], 0
    for _ in range(n_ops):
        r = rng.random()
        if swaps and live and rng.random() < 0.2:
            k = rng.randint(1, min(3, len(live)))
            ops.append((rng.choice(["swap_out", "swap_in"]), rng.sample(live, k)))
            continue
        if not live or (r < 0.15 and len(live) < 12):
            ops.append(("add", nxt)); live.append(nxt); nxt += 1
        elif r < 0.30 and len(live) < 12:
            p = rng.choice(live)
            ops.append(("fork", p, nxt)); live.append(nxt); nxt += 1
        elif r < 0.40 and len(live) > 1:
            s = rng.choice(live)
            ops.append(("free", s)); live.remove(s)
        else:
            k = rng.randint(1, len(live))
            batch = rng.sample(live, k)
            ops.append(("append", [(s, rng.choice([1, 1, 1, 2, 3, 5, 9, 17])) for s in batch]))
    return ops


def _is_full(e):
    return "block" in str(e).lower() or "space" in str(e).lower()


def run_ops(bm, ops, num_blocks, B, log=None, num_host_blocks=0):
    """Replays ops on bm and on model pools (device and host); checks every read-back and
    invariant. Appends and swaps that a pool cannot hold must raise and change nothing."""
    pool = [None] * (num_blocks * B)       # token id held by each device slot
    hpool = [None] * (num_host_blocks * B)  # and by each host slot
    model = {}                              # sequence -> its token ids by position
    host = set()                            # sequences swapped out
    tok = 0

    def snapshot():
        return ({s: bm.table(s) for s in model}, bm.num_free(),
                bm.num_free_host() if num_host_blocks else 0)

    for op in ops:
        if op[0] == "add":
            bm.add(op[1]); model[op[1]] = []
        elif op[0] == "fork":
            if op[1] not in model or op[1] in host:    # a swapped-out parent: dropped
                continue
            bm.fork(op[1], op[2]); model[op[2]] = list(model[op[1]])
        elif op[0] == "free":
            if op[1] not in model:
                continue
            bm.free_seq(op[1]); del model[op[1]]; host.discard(op[1])
        elif op[0] in ("swap_out", "swap_in"):
            out = op[0] == "swap_out"
            seqs = [s for s in op[1] if s in model and (s in host) != out]
            if not seqs:
                continue
            before = snapshot()
            try:
                pairs = bm.swap_out(seqs) if out else bm.swap_in(seqs)
            except Exception as e:
                if not _is_full(e):
                    raise
                assert snapshot() == before, "swap not atomic"
                if log is not None:
                    log.append(("full",))
                continue
            src_pool, dst_pool = (pool, hpool) if out else (hpool, pool)
            for a, b in pairs:                  # copies read before any block is reused
                dst_pool[b * B:(b + 1) * B] = src_pool[a * B:(a + 1) * B]
            for s in seqs:
                (host.add if out else host.discard)(s)
            if log is not None:
                log.append((op[0], tuple(map(tuple, pairs))))
        else:
            batch = [(s, n) for s, n in op[1] if s in model and s not in host]
            if not batch:
                continue
            seqs = [s for s, _ in batch]
            ns = [n for _, n in batch]
            before = snapshot()
            try:
                slots, copies = bm.append_batch(seqs, ns)
            except Exception as e:   # pool exhausted: nothing may have changed
                if not _is_full(e):
                    raise
                assert snapshot() == before, "not atomic"
                if log is not None:
                    log.append(("full",))
                continue
            for src, dst in copies:             # copies happen before the writes
                pool[dst * B:(dst + 1) * B] = pool[src * B:(src + 1) * B]
            k = 0
            for s, n in zip(seqs, ns):
                for _ in range(n):
                    pool[slots[k]] = tok
                    model[s].append(tok)
                    tok += 1; k += 1
            assert k == len(slots)
            if log is not None:
                log.append((tuple(slots), tuple(map(tuple, copies))))
        for s, toks in model.items():
            t = bm.table(s)
            src = hpool if s in host else pool
            for p, want in enumerate(toks):
                got = src[t[p // B] * B + p % B]
                assert got == want, ("read-back", s, p, got, want)
            if num_host_blocks:
                assert bm.is_on_host(s) == (s in host), ("residency", s)
        _invariants(bm, model, num_blocks, B, host, num_host_blocks)
    return model


def check_random_histories(make):
    for seed, (nb, B) in enumerate([(64, 4), (40, 16), (200, 1), (24, 8)]):
        run_ops(make(nb, B, None), random_ops(seed), nb, B)


def check_swap_histories(make):
    """Seeded histories with swaps out and in: after every operation each request
    reads back its own tokens from the pool it lives in (vLLM post, 3, swapping)."""
    for seed, (nb, nhb, B) in enumerate([(40, 24, 4), (30, 60, 8), (64, 8, 2)]):
        run_ops(make(nb, B, None, nhb), random_ops(100 + seed, swaps=True), nb, B,
                num_host_blocks=nhb)


def check_swap_keeps_sharing(make):
    """Two samples sharing a prompt swap out together: each shared block is copied
    once and stays shared in the host pool; back in, they share again."""
    bm = make(12, 4, None, 12)
    bm.add("A1")
    bm.append("A1", 7)                         # blocks 0, 1
    bm.fork("A1", "A2")
    bm.append("A1", 1)                         # copy 1 -> 2, A1 [0, 2], A2 [0, 1]
    pairs = bm.swap_out(["A1", "A2"])
    assert pairs == [(0, 0), (2, 1), (1, 2)], pairs
    assert bm.table("A1") == [0, 1] and bm.table("A2") == [0, 2]
    assert bm.host_refcount(0) == 2 and bm.num_free() == 12 and bm.num_free_host() == 9
    back = bm.swap_in(["A2"])                  # only A2 returns: host block 0 stays for A1
    assert back == [(0, 3), (2, 4)], back
    assert bm.host_refcount(0) == 1 and bm.refcount(3) == 1 and bm.num_free_host() == 10


def check_exhaustion_is_atomic(make):
    bm = make(4, 4, None)
    bm.add(0); bm.add(1)
    bm.append(0, 6)                          # blocks 0, 1
    bm.fork(0, 2)
    failed = False
    try:
        bm.append_batch([1, 2], [9, 1])      # 3 new blocks + 1 copy > 2 free
    except Exception:
        failed = True
    assert failed, "an append beyond the pool must fail"
    assert bm.table(1) == [] and bm.table(2) == [0, 1] and bm.num_free() == 2
    slots, copies = bm.append(2, 1)          # one copy of the shared partial block
    assert copies == [(1, 2)] and slots == [2 * 4 + 2]


ALL_CHECKS = [check_worked_example, check_cow_example, check_random_histories,
              check_exhaustion_is_atomic, check_swap_histories, check_swap_keeps_sharing]


def swap_roundtrip(bm, gather, scribble, move):
    """A request and its fork swapped out, their device blocks overwritten, both swapped
    back in to other blocks: they read back what they held, through their new tables.

    gather(table) -> copy of those device blocks; scribble(blocks) overwrites device
    blocks; move(pairs, direction) copies blocks ("out": device -> host, "in": back)."""
    bm.add("A")
    bm.append("A", 30)
    bm.add("B")
    bm.append("B", 20)
    bm.fork("A", "C")
    bm.append("C", 1)                            # copy-on-write of A's partial block
    want = {s: gather(bm.table(s)) for s in ("A", "C")}
    keep_b = gather(bm.table("B"))
    # (the copy of C's partial block is the caller's: it moved with pa_copy_blocks or
    # here simply with the pool contents of the shared block, which equal both tables')
    distinct = set(bm.table("A")) | set(bm.table("C"))
    out = bm.swap_out(["A", "C"])
    assert sorted(d for d, _ in out) == sorted(distinct), out   # shared blocks once
    move(out, "out")
    freed = [d for d, _ in out]
    scribble(freed)
    back = bm.swap_in(["C", "A"])
    assert len(back) == len(distinct) and all(bm.refcount(d) > 0 for _, d in back)
    move(back, "in")
    for s in ("A", "C"):
        got = gather(bm.table(s))
        assert got == want[s] if isinstance(got, list) else (got == want[s]).all(), s
    got_b = gather(bm.table("B"))
    assert got_b == keep_b if isinstance(got_b, list) else (got_b == keep_b).all()
