"""Pins for the oracle: checks against what the pages and the mathematics fix.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a value or property that does not come from the oracle
itself: the pages' worked examples, hand-derived closed forms, an independent
contiguous softmax written with numpy matrices, torch's fp64
``scaled_dot_product_attention`` (a library routine), brute-force invariances.
The planted-mistake test runs every check against deliberately broken oracle
builds and requires each one to be caught.
"""
import json
import math
import os

import numpy as np
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (a copy)."""
    return workloads.host_bits(t)


def bf16_bits(x) -> np.ndarray:
    return u16(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64, by widening to float32 bits."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ independent refs

def contiguous_reference(q, K, V, L, ql, scale):
    """Causal softmax attention of one sequence with contiguous K/V, numpy matrices.

    q [ql, Hq, D], K/V [L, Hkv, D] float64. The mask keeps key j for query row i
    when j <= L - ql + i (the rows are the last ql tokens), written with np.tril.
    """
    Hq, Hkv = q.shape[1], K.shape[1]
    g = Hq // Hkv
    Kr = np.repeat(K, g, axis=1)          # query head h reads KV head h // g
    Vr = np.repeat(V, g, axis=1)
    S = np.einsum("qhd,khd->hqk", q, Kr) * scale
    keep = np.tril(np.ones((ql, L), dtype=bool), k=L - ql)
    S = np.where(keep[None], S, -np.inf)
    S = S - S.max(axis=-1, keepdims=True)
    P = np.exp(S)
    P /= P.sum(axis=-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", P, Vr)


def sdpa_reference(q, K, V, L, ql, scale):
    """Same thing through torch's fp64 scaled_dot_product_attention with an explicit mask."""
    Hq, Hkv = q.shape[1], K.shape[1]
    g = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)                       # [Hq, ql, D]
    kt = torch.from_numpy(K).repeat_interleave(g, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(V).repeat_interleave(g, dim=1).permute(1, 0, 2)
    rows = torch.arange(ql)[:, None] + (L - ql)
    mask = torch.arange(L)[None, :] <= rows
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()


def identity_layout(w):
    """Re-lay a workload so every sequence owns consecutive physical blocks 0,1,2,...

    Returns (k_pool, v_pool, block_table, bases) with pools as uint16 arrays;
    sequence s's K is then literally k_pool[base:base+n].reshape(-1, Hkv, D)[:L].
    Built from per-token gathers of the original table's slots.
    """
    B = w.block_size
    kp, vp = u16(w.k_pool), u16(w.v_pool)
    need = [-(-int(L) // B) for L in w.context_lens]
    total = max(1, sum(need))
    nk = np.zeros((total, B) + kp.shape[2:], np.uint16)
    nv = np.zeros_like(nk)
    bt = np.full((w.num_seqs, max(1, max(need) if need else 1)), -1, np.int32)
    bases, off = [], 0
    for s, n in enumerate(need):
        bt[s, :n] = np.arange(off, off + n)
        for j in range(n):
            nk[off + j] = kp[w.block_table[s, j]]
            nv[off + j] = vp[w.block_table[s, j]]
        bases.append(off)
        off += n
    return nk, nv, bt, bases


def _check_close(a, b, tol, what):
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs diff {err} > {tol}"


# ------------------------------------------------------------ checks

def check_bf16_decode(orc):
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x7F80: math.inf, 0x8000: -0.0}
    for bits, want in cases.items():
        got = orc.bf16_to_double(bits)
        assert got == want, f"bf16 0x{bits:04x}: {got} != {want}"


def check_worked_example_slots(orc):
    g = _golden("worked_example_slots.json")
    B = g["block_size"]
    bt = np.array([g["block_table"]], np.int32)
    for step in g["steps"]:
        pos = np.array(step["positions"], np.int32)
        got = orc.slot_mapping(bt, 8, B, np.zeros(len(pos), np.int32), pos)
        assert got.tolist() == step["slots"], f"{step['what']}: {got.tolist()} != {step['slots']}"


def check_worked_example_write_then_attend(orc):
    """Prefill 7 tokens, two decode steps; after each step every row equals contiguous attention."""
    g = _golden("worked_example_slots.json")
    B, Hkv, D, Hq = g["block_size"], 2, 8, 4
    bt = np.array([g["block_table"]], np.int32)
    nb = 8
    gen = torch.Generator().manual_seed(7)
    kp = bf16_bits(torch.randn(nb, B, Hkv, D, generator=gen))
    vp = bf16_bits(torch.randn(nb, B, Hkv, D, generator=gen))
    K_all = bf16_bits(torch.randn(9, Hkv, D, generator=gen))
    V_all = bf16_bits(torch.randn(9, Hkv, D, generator=gen))
    Q_all = bf16_bits(torch.randn(9, Hq, D, generator=gen))
    L = 0
    for step in g["steps"]:
        pos = np.array(step["positions"], np.int32)
        slots = orc.slot_mapping(bt, nb, B, np.zeros(len(pos), np.int32), pos)
        orc.write_kv(K_all[pos], V_all[pos], slots, kp, vp)
        L = int(pos[-1]) + 1
        ql = len(pos)
        # the written bytes sit exactly where the page puts them
        for p, sl in zip(pos, step["slots"]):
            assert np.array_equal(kp.reshape(-1, Hkv, D)[sl], K_all[p])
            assert np.array_equal(vp.reshape(-1, Hkv, D)[sl], V_all[p])
        got = orc.attention(Q_all[pos], kp, vp, bt, [L], [ql])
        ref = contiguous_reference(f64(Q_all[pos]), f64(K_all[:L]), f64(V_all[:L]), L, ql,
                                   1 / math.sqrt(D))
        _check_close(got, ref, 1e-12, step["what"])
    # filled counts: #filled of the last block = L - B * (ceil(L / B) - 1)
    assert L - B * (-(-L // B) - 1) == 1


def check_cow_example(orc):
    g = _golden("cow_example.json")
    B, Hkv, D, nb = g["block_size"], 1, 4, 8
    gen = torch.Generator().manual_seed(11)
    kp = bf16_bits(torch.randn(nb, B, Hkv, D, generator=gen))
    vp = bf16_bits(torch.randn(nb, B, Hkv, D, generator=gen))
    before_k, before_v = kp.copy(), vp.copy()
    new_k = bf16_bits(torch.randn(2, Hkv, D, generator=gen))
    new_v = bf16_bits(torch.randn(2, Hkv, D, generator=gen))
    src = [c[0] for c in g["copies"]]
    dst = [c[1] for c in g["copies"]]
    orc.copy_blocks(kp, vp, src, dst)
    assert np.array_equal(kp[3], before_k[1]) and np.array_equal(vp[3], before_v[1])
    names = ["A1", "A2"]
    bt = np.array([g["tables_after"][n] + [-1] for n in names], np.int32)
    pos = np.array([w["position"] for w in g["writes"]], np.int32)
    seq = np.array([names.index(w["sample"]) for w in g["writes"]], np.int32)
    slots = orc.slot_mapping(bt, nb, B, seq, pos)
    assert slots.tolist() == [w["slot"] for w in g["writes"]], slots
    orc.write_kv(new_k, new_v, slots, kp, vp)
    flat_k = kp.reshape(-1, Hkv, D)
    assert np.array_equal(flat_k[15], new_k[0]) and np.array_equal(flat_k[7], new_k[1])
    # block 3 = old block 1 with A1's token in its last slot; block 7 untouched
    assert np.array_equal(kp[3, :3], before_k[1, :3]) and np.array_equal(kp[1, :3], before_k[1, :3])
    assert np.array_equal(kp[7], before_k[7]) and np.array_equal(vp[7], before_v[7])
    untouched = [b for b in range(nb) if b not in (1, 3)]
    assert np.array_equal(kp[untouched], before_k[untouched])
    assert np.array_equal(vp[3, 3], new_v[0]) and np.array_equal(vp[1, 3], new_v[1])


def check_closed_forms(orc):
    g = _golden("closed_forms.json")
    for case in g["cases"]:
        Hq, Hkv, D, B = case["Hq"], case["Hkv"], case["D"], case["block_size"]
        L, ql = case["context_lens"][0], case["query_lens"][0]
        k = np.asarray(case["k"], np.float32).reshape(L, Hkv, D)
        v = np.asarray(case["v"], np.float32).reshape(L, Hkv, D)
        q = np.asarray(case["q"], np.float32).reshape(ql, Hq, D)
        nblk = -(-L // B)
        # scatter the context into a permuted pool so the table is exercised too
        nb = nblk + 3
        perm = np.random.default_rng(5).permutation(nb)[:nblk].astype(np.int32)
        kp = np.zeros((nb, B, Hkv, D), np.float32)
        vp = np.zeros_like(kp)
        for t in range(L):
            kp[perm[t // B], t % B] = k[t]
            vp[perm[t // B], t % B] = v[t]
        scale = 0.0 if case["scale"] is None else case["scale"]
        got = orc.attention(bf16_bits(q), bf16_bits(kp), bf16_bits(vp), perm[None], [L], [ql],
                            scale=scale)
        want = np.asarray(case["expected"], np.float64).reshape(ql, Hq, D)
        _check_close(got, want, 1e-12, case["name"])


def _small_batches():
    yield workloads.make(1)
    yield workloads.make_custom([5, 1, 16, 17, 40, 0, 3], [5, 1, 3, 17, 1, 0, 2], Hq=6, Hkv=2, D=8,
                                block_size=4, seed=3)
    yield workloads.make_custom([33, 9, 64], [2, 9, 1], Hq=8, Hkv=1, D=16, block_size=8, seed=4)


def check_against_contiguous(orc):
    """Identity block table: each sequence's K/V is a plain reshape of consecutive blocks."""
    for w in _small_batches():
        kp, vp, bt, bases = identity_layout(w)
        q = u16(w.q)
        got = orc.attention(q, kp, vp, bt, w.context_lens, w.query_lens)
        r0 = 0
        for s in range(w.num_seqs):
            L, ql = int(w.context_lens[s]), int(w.query_lens[s])
            if ql == 0:
                continue
            n = -(-L // w.block_size)
            K = f64(kp[bases[s]:bases[s] + n].reshape(-1, w.Hkv, w.D)[:L])
            V = f64(vp[bases[s]:bases[s] + n].reshape(-1, w.Hkv, w.D)[:L])
            scale = 1 / math.sqrt(w.D)
            ref = contiguous_reference(f64(q[r0:r0 + ql]), K, V, L, ql, scale)
            ref2 = sdpa_reference(f64(q[r0:r0 + ql]), K, V, L, ql, scale)
            _check_close(got[r0:r0 + ql], ref, 1e-12, f"{w.name} seq {s} vs numpy")
            _check_close(got[r0:r0 + ql], ref2, 1e-12, f"{w.name} seq {s} vs torch sdpa")
            r0 += ql


def check_permutation_invariance(orc):
    """Only the mapping matters: relabelling physical blocks leaves outputs bit-identical."""
    for w in _small_batches():
        kp, vp = u16(w.k_pool), u16(w.v_pool)
        base = orc.attention(u16(w.q), kp, vp, w.block_table, w.context_lens, w.query_lens)
        perm = np.random.default_rng(w.seed + 1).permutation(w.num_blocks)
        kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
        kp2[perm], vp2[perm] = kp, vp
        bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
        got = orc.attention(u16(w.q), kp2, vp2, bt2, w.context_lens, w.query_lens)
        assert np.array_equal(base, got), f"{w.name}: permuting physical ids changed the result"


def check_block_size_invariance(orc):
    """The same logical K/V laid out with B in {1,2,4,8,16,32} gives bit-identical outputs."""
    w = workloads.make_custom([37, 12, 1, 64], [3, 12, 1, 2], Hq=4, Hkv=2, D=8, block_size=4,
                              seed=9)
    kp, vp = u16(w.k_pool), u16(w.v_pool)
    ref = None
    for B in (1, 2, 4, 8, 16, 32):
        need = [-(-int(L) // B) for L in w.context_lens]
        nb = sum(need) + 2
        perm = np.random.default_rng(B).permutation(nb)
        nk = np.zeros((nb, B, w.Hkv, w.D), np.uint16)
        nv = np.zeros_like(nk)
        bt = np.full((w.num_seqs, max(need)), -1, np.int32)
        off = 0
        for s, n in enumerate(need):
            bt[s, :n] = perm[off:off + n]
            off += n
            for t in range(int(w.context_lens[s])):
                src = w.block_table[s, t // w.block_size], t % w.block_size
                nk[bt[s, t // B], t % B] = kp[src]
                nv[bt[s, t // B], t % B] = vp[src]
        got = orc.attention(u16(w.q), nk, nv, bt, w.context_lens, w.query_lens)
        if ref is None:
            ref = got
        assert np.array_equal(ref, got), f"block size {B} changed the result"


def check_blockwise_form(orc):
    """Token form and block form of the definition agree."""
    for w in _small_batches():
        a = orc.attention(u16(w.q), u16(w.k_pool), u16(w.v_pool), w.block_table, w.context_lens,
                          w.query_lens)
        b = orc.attention_blockwise(u16(w.q), u16(w.k_pool), u16(w.v_pool), w.block_table,
                                    w.context_lens, w.query_lens)
        _check_close(a, b, 1e-12, f"{w.name}: block form")


def check_subrequests(orc):
    """Pensieve's dropped-token handling (Fig. 8): sub-request A (leading r tokens attend to
    themselves) and B (new prompt attends to the whole context) reproduce the matching rows
    of one request whose queries are every token of the context."""
    L, r, qn = 45, 8, 11
    Hq, Hkv, D, B = 4, 2, 8, 4
    full = workloads.make_custom([L], [L], Hq=Hq, Hkv=Hkv, D=D, block_size=B, seed=21)
    kp, vp, q = u16(full.k_pool), u16(full.v_pool), u16(full.q)
    one = orc.attention(q, kp, vp, full.block_table, [L], [L])
    bt2 = np.concatenate([full.block_table, full.block_table])
    q2 = np.concatenate([q[:r], q[L - qn:]])
    two = orc.attention(q2, kp, vp, bt2, [r, L], [r, qn])
    assert np.array_equal(two[:r], one[:r]), "sub-request A rows differ"
    assert np.array_equal(two[r:], one[L - qn:]), "sub-request B rows differ"


def check_special_cases(orc):
    """All visible V rows equal -> o is that row; all K zero -> o is the mean of visible V."""
    w = workloads.make_custom([9, 20], [2, 3], Hq=2, Hkv=1, D=4, block_size=4, seed=31)
    kp, vp = u16(w.k_pool), u16(w.v_pool)
    row = bf16_bits([0.5, -1.25, 3.0, 0.0])
    vp_eq = np.broadcast_to(row, vp.shape).copy()
    got = orc.attention(u16(w.q), kp, vp_eq, w.block_table, w.context_lens, w.query_lens)
    _check_close(got, np.broadcast_to(f64(row), got.shape), 1e-14, "equal V rows give that row")
    kz = np.zeros_like(kp)
    got = orc.attention(u16(w.q), kz, vp, w.block_table, w.context_lens, w.query_lens)
    r0 = 0
    for s in range(w.num_seqs):
        L, ql = int(w.context_lens[s]), int(w.query_lens[s])
        for i in range(ql):
            p = L - ql + i
            toks = [f64(vp[w.block_table[s, t // 4], t % 4, 0]) for t in range(p + 1)]
            _check_close(got[r0 + i, 0], np.mean(toks, axis=0), 1e-12, "uniform weights")
        r0 += ql


def check_garbage_is_masked(orc):
    """NaN in slots past each context (tail of the last block, unused blocks) changes nothing."""
    w = workloads.make_custom([9, 20, 3], [2, 3, 3], Hq=2, Hkv=2, D=4, block_size=8, seed=41)
    kp, vp = u16(w.k_pool), u16(w.v_pool)
    base = orc.attention(u16(w.q), kp, vp, w.block_table, w.context_lens, w.query_lens)
    kn, vn = kp.copy(), vp.copy()
    used = np.zeros((w.num_blocks, w.block_size), bool)
    for s in range(w.num_seqs):
        for t in range(int(w.context_lens[s])):
            used[w.block_table[s, t // 8], t % 8] = True
    kn[~used] = 0x7FC0
    vn[~used] = 0x7FC0
    got = orc.attention(u16(w.q), kn, vn, w.block_table, w.context_lens, w.query_lens)
    assert np.array_equal(base, got)


ALL_CHECKS = [check_bf16_decode, check_worked_example_slots, check_worked_example_write_then_attend,
              check_cow_example, check_closed_forms, check_against_contiguous,
              check_permutation_invariance, check_block_size_invariance, check_blockwise_form,
              check_subrequests, check_special_cases, check_garbage_is_masked]
