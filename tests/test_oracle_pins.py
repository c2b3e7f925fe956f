"""CPU-only pins of the fp64 oracle (no GPU, no CUDA library)."""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import workloads
from oracle import build as obuild
from tests import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(orc, check):
    check(orc)


def test_rows_subset_and_threads_match(orc):
    w = workloads.make(1)
    q, kp, vp = oc.u16(w.q), oc.u16(w.k_pool), oc.u16(w.v_pool)
    full = orc.attention(q, kp, vp, w.block_table, w.context_lens, w.query_lens)
    thr = orc.attention(q, kp, vp, w.block_table, w.context_lens, w.query_lens, n_threads=4)
    assert np.array_equal(full, thr)
    rows = np.array([25, 0, 9, 3], np.int64)
    sub = orc.attention(q, kp, vp, w.block_table, w.context_lens, w.query_lens, rows=rows)
    assert np.array_equal(sub, full[rows])


@pytest.mark.parametrize("bad", ["q_gt_L", "heads", "block_id", "table_short", "total_q"])
def test_attention_rejects_invalid(orc, bad):
    w = workloads.make_custom([9, 20], [2, 3], Hq=4, Hkv=2, D=8, block_size=4, seed=1)
    q, kp, vp = oc.u16(w.q), oc.u16(w.k_pool), oc.u16(w.v_pool)
    bt, L, ql = w.block_table.copy(), w.context_lens.copy(), w.query_lens.copy()
    if bad == "q_gt_L":
        ql = np.array([10, 3], np.int32); L = np.array([9, 20], np.int32)
        q = np.zeros((13, 4, 8), np.uint16)
    elif bad == "heads":
        q = np.zeros((5, 3, 8), np.uint16)
    elif bad == "block_id":
        bt[1, 2] = w.num_blocks
    elif bad == "table_short":
        L = np.array([9, 20 + 4 * bt.shape[1]], np.int32)
    elif bad == "total_q":
        q = q[:4]
    with pytest.raises(oracle.OracleError):
        orc.attention(q, kp, vp, bt, L, ql)


def test_write_rejects_duplicates_and_range(orc):
    kp = np.zeros((4, 2, 1, 2), np.uint16); vp = kp.copy()
    kn = np.ones((2, 1, 2), np.uint16); vn = kn.copy()
    with pytest.raises(oracle.OracleError):
        orc.write_kv(kn, vn, [3, 3], kp, vp)
    with pytest.raises(oracle.OracleError):
        orc.write_kv(kn, vn, [0, 8], kp, vp)
    assert not kp.any(), "a rejected write must leave the pool untouched"
    orc.write_kv(kn, vn, [-1, 5], kp, vp)
    assert kp.reshape(8, 2)[5].tolist() == [1, 1] and kp.sum() == 2


def test_copy_rejects_bad_pairs(orc):
    kp = np.zeros((4, 2, 1, 2), np.uint16); vp = kp.copy()
    for src, dst in ([[0, 1], [2, 2]], [[0, 1], [1, 2]], [[0], [4]]):
        with pytest.raises(oracle.OracleError):
            orc.copy_blocks(kp, vp, src, dst)


def test_bytes_formula_matches_page_example():
    """vLLM wiki note, problem/motivation: OPT-13B keeps about 800 KB of KV per token
    (40 layers, hidden 5120 = 40 heads x 128, fp16). One layer of the decode workload has
    the same head shape, so 40 layers x its per-token K+V bytes must be 819,200 B."""
    w = workloads.make_custom([1], [1], Hq=40, Hkv=40, D=128, block_size=16, seed=0)
    per_token_layer = w.kv_bytes() // int(w.context_lens.sum())
    assert per_token_layer * 40 == 819_200
    assert abs(819_200 / 1024 - 800) < 1.0


def test_flop_count_brute_force():
    w = workloads.make_custom([7, 33, 5, 12], [1, 4, 5, 0], Hq=2, Hkv=1, D=4, block_size=4, seed=2)
    pairs = 0
    for L, ql in zip(w.context_lens, w.query_lens):
        for i in range(int(ql)):
            pairs += int(L) - int(ql) + i + 1
    assert w.flops() == 4 * w.Hq * w.D * pairs


MUTANTS = {1: "scale 1/D", 2: "top-left mask", 3: "interleaved GQA map", 4: "diagonal dropped",
           5: "slot ignores the table", 6: "COW copies only K", 7: "no causal mask",
           8: "V written from K"}


@pytest.mark.parametrize("mutation", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_planted_mistake_is_caught(mutation):
    """Every planted mistake in the oracle must fail at least one pin."""
    with tempfile.TemporaryDirectory() as d:
        path = obuild.build(os.path.join(d, f"liboracle_m{mutation}.so"), mutation=mutation)
        bad = oracle.Oracle(path)
        caught = []
        for check in oc.ALL_CHECKS:
            try:
                check(bad)
            except (AssertionError, oracle.OracleError):
                caught.append(check.__name__)
        assert caught, f"mutation {MUTANTS[mutation]} passed every pin"


def test_swap_oracle_agrees_with_copy_blocks(orc):
    """A swap from pool A to pool B is the oracle's copy_blocks (the C implementation)
    on the stacked pool [B; A] with A's ids shifted; and a swap out then in restores."""
    from oracle.swap import swap_blocks
    rng = np.random.default_rng(5)
    shape = (6, 4, 2, 8)
    A_k, A_v = (rng.integers(0, 2**16, (9,) + shape[1:], dtype=np.uint16) for _ in range(2))
    B_k, B_v = (rng.integers(0, 2**16, shape, dtype=np.uint16) for _ in range(2))
    src, dst = np.array([8, 0, 3, 3], np.int32), np.array([5, 1, 0, 2], np.int32)
    stk_k, stk_v = np.concatenate([B_k, A_k]), np.concatenate([B_v, A_v])
    orc.copy_blocks(stk_k, stk_v, src + len(B_k), dst)
    swap_blocks(A_k, A_v, B_k, B_v, src, dst)
    assert np.array_equal(B_k, stk_k[:len(B_k)]) and np.array_equal(B_v, stk_v[:len(B_v)])
    back_k, back_v = np.zeros_like(A_k), np.zeros_like(A_v)
    swap_blocks(B_k, B_v, back_k, back_v, dst[:3], src[:3])
    for s in src[:3]:
        assert np.array_equal(back_k[s], A_k[s]) and np.array_equal(back_v[s], A_v[s])
    with pytest.raises(ValueError):
        swap_blocks(A_k, A_v, B_k, B_v, [0, 1], [2, 2])
    with pytest.raises(ValueError):
        swap_blocks(A_k, A_v, B_k, B_v, [9], [0])
