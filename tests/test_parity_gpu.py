"""GPU parity of the hot path (through the C ABI) against the fp64 oracle.

Writes, copies and slot mappings must be bit-exact; attention must be within
max abs 5e-3 and mean abs 5e-4 of the oracle (bf16 inputs, fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util as gu
from tests.oracle_checks import f64, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gu.lib()


def full_check(pa, w, **plan_kw):
    got = gu.gpu_step(pa, w, **plan_kw)
    ref = gu.oracle_step(w)
    assert got["err"] == 0, f"device error {pa.DEVERR.get(got['err'])}"
    assert np.array_equal(got["slots"], ref["slots"]), "slot mapping differs"
    assert gu.pools_equal(got["k_pool"], ref["k_pool"]), "K pool differs after write/copy"
    assert gu.pools_equal(got["v_pool"], ref["v_pool"]), "V pool differs after write/copy"
    want = gu.oracle_rows(w, ref)
    out = got["out"].float().cpu().numpy()
    return gu.assert_attention_close(out, want, w.name), got, want


def test_config1_tiny_mixed(pa):
    full_check(pa, workloads.make(1))


@pytest.mark.parametrize("chunk", [64, 128])
def test_config1_forced_split(pa, chunk):
    w = workloads.make(1) if chunk == 64 else workloads.make_custom(
        [7, 130, 300, 1000], [1, 20, 3, 1], Hq=8, Hkv=2, D=128, block_size=16, seed=chunk)
    (_, _), got, want = full_check(pa, w, max_chunk_tokens=chunk)
    assert got["plan"].stats()["n_split_groups"] > 0
    base = gu.gpu_step(pa, w)["out"]
    assert torch.allclose(got["out"], base, atol=gu.ATOL_MAX, rtol=0)


CASES = []
for B in (8, 16, 32):
    for D in (64, 128):
        for Hq, Hkv in ((4, 4), (8, 2), (8, 1)):
            CASES.append((B, D, Hq, Hkv))
CASES += [(16, 128, 12, 4), (32, 128, 64, 4), (16, 64, 12, 4)]


@pytest.mark.parametrize("B,D,Hq,Hkv", CASES)
def test_ragged_fuzz(pa, B, D, Hq, Hkv):
    rng = np.random.default_rng(B * 1000 + D * 10 + Hq + Hkv)
    n = 7
    L = rng.integers(0, 300, size=n)
    L[0] = 0
    L[1] = 1
    q = np.array([rng.integers(0, min(l, 40) + 1) for l in L])
    q[2] = min(L[2], 1)
    w = workloads.make_custom(L, q, Hq=Hq, Hkv=Hkv, D=D, block_size=B, seed=int(rng.integers(1e6)))
    full_check(pa, w)
    full_check(pa, w, max_chunk_tokens=64)


@pytest.mark.parametrize("B", [1, 4, 64, 128, 256])
def test_block_size_extremes(pa, B):
    w = workloads.make_custom([3, 200, 517, 64], [3, 1, 9, 64], Hq=8, Hkv=2, D=128, block_size=B,
                              seed=B)
    full_check(pa, w)


def test_long_context_split(pa):
    w = workloads.make_custom([40000, 1], [1, 1], Hq=8, Hkv=8, D=128, block_size=16, seed=77)
    got = gu.gpu_step(pa, w)
    assert got["plan"].stats()["n_split_groups"] > 0
    ref = gu.oracle_step(w)
    gu.assert_attention_close(got["out"].cpu().numpy(), gu.oracle_rows(w, ref), "40k context")


@pytest.mark.parametrize("g", [1, 4, 8])
def test_tensor_core_and_cuda_core_paths_agree(pa, g):
    """Decode is multi-token attention with q = 1 (Pensieve, unified batching): forcing every
    item onto the tensor-core tiles or onto the CUDA-core path gives the same result."""
    w = workloads.make_custom([1, 17, 130, 300, 700], [1, 17, 1, 37, 5], Hq=4 * g, Hkv=4, D=128,
                              block_size=16, seed=100 + g)
    (_, _), tc_run, want = full_check(pa, w, tc_min_rows=1)
    assert tc_run["plan"].stats()["n_dec_items"] == 0
    (_, _), dec_run, _ = full_check(pa, w, tc_min_rows=-1)
    assert dec_run["plan"].stats()["n_tc_items"] == 0
    assert torch.allclose(tc_run["out"], dec_run["out"], atol=gu.ATOL_MAX, rtol=0)


def test_tensor_core_tiny_first(pa):
    """Smallest tensor-core case (one 128-row tile, one key tile)."""
    w = workloads.make_custom([40], [20], Hq=8, Hkv=8, D=128, block_size=16, seed=9)
    (_, _), got, _ = full_check(pa, w, tc_min_rows=1)
    assert got["plan"].stats()["n_tc_items"] > 0


PAIR_CASES = [
    # (g, block_size, chunk): ragged row counts around the 128 / 256 tile edges
    (1, 16, 0), (1, 32, 128), (8, 32, 0), (8, 8, 256), (4, 256, 0), (16, 64, 192),
]


@pytest.mark.parametrize("g,B,chunk", PAIR_CASES)
def test_tensor_core_pair_tiles(pa, g, B, chunk):
    """Items of 129..256 rows run as two 128-row tiles sharing every K/V tile; the result
    matches the oracle and the one-tile kernel."""
    rows = [129, 200, 256, 257, 384, 511, 64]
    q = [max(1, -(-r // g)) for r in rows]
    L = [qq + extra for qq, extra in zip(q, [0, 37, 300, 5, 900, 128, 700])]
    w = workloads.make_custom(L, q, Hq=2 * g, Hkv=2, D=128, block_size=B, seed=300 + g + B)
    kw = dict(max_chunk_tokens=chunk) if chunk else {}
    (_, _), pair_run, want = full_check(pa, w, tc_pair=1, **kw)
    assert pair_run["plan"].stats()["n_tc_pair_items"] > 0
    (_, _), one_run, _ = full_check(pa, w, tc_pair=-1, **kw)
    assert one_run["plan"].stats()["n_tc_pair_items"] == 0
    assert torch.allclose(pair_run["out"], one_run["out"], atol=gu.ATOL_MAX, rtol=0)


@pytest.mark.parametrize("chunk", [0, 64])
def test_tensor_core_pair_half_tile_tails(pa, chunk):
    """The two-tile kernel takes each 128-key tile as two 64-key score halves: key ranges
    ending at 64 and 65 keys into the last tile (its second half has no key, or one), and
    with 64-key split chunks every item's only tile has an empty second half."""
    w = workloads.make_custom([320, 321, 448, 257], [256, 256, 256, 200], Hq=2, Hkv=2, D=128,
                              block_size=16, seed=77)
    kw = dict(max_chunk_tokens=chunk) if chunk else {}
    (_, _), got, _ = full_check(pa, w, tc_pair=1, **kw)
    assert got["plan"].stats()["n_tc_pair_items"] > 0
    if chunk:
        assert got["plan"].stats()["n_split_groups"] > 0


@pytest.mark.parametrize("g", [8, 64, 128])
def test_tensor_core_pair_bf16_and_wide_groups(pa, g):
    """Two-tile items with bf16 output (the epilogue's tensor stores in bf16) and with
    64 or 128 query heads per KV head (a warp's 32 rows are heads of one token)."""
    q = [max(1, 300 // g) + 1, max(1, 129 // g) + 1, 1]
    L = [qq + extra for qq, extra in zip(q, [400, 33, 17])]
    w = workloads.make_custom(L, q, Hq=g, Hkv=1, D=128, block_size=32, seed=900 + g)
    want = gu.oracle_rows(w, gu.oracle_step(w))
    got = gu.gpu_step(pa, w, tc_pair=1)
    assert got["plan"].stats()["n_tc_pair_items"] > 0
    gu.assert_attention_close(got["out"].cpu().numpy(), want, f"g={g} fp32")
    got16 = gu.gpu_step(pa, w, out_dtype=torch.bfloat16, tc_pair=1)
    d = np.abs(got16["out"].float().cpu().numpy() - want)
    # bf16 rounding of outputs of magnitude up to a few units: half an ulp is <= 2^-8 * |o|
    bound = np.abs(want) * 2.0 ** -8 + gu.ATOL_MAX
    assert np.all(d <= bound), float((d - bound).max())


@pytest.mark.parametrize("g", [1, 8, 64, 128])
def test_tensor_core_one_tile_bf16_and_wide_groups(pa, g):
    """One-tile items only (tc_pair=-1): fp32 and bf16 outputs (the epilogue's tensor
    stores in both layouts), 1 to 128 query heads per KV head, full and partial 128-row
    tiles over several key tiles."""
    q = [max(1, 384 // g), max(1, 200 // g) + 1, max(1, 129 // g), 1]
    L = [qq + extra for qq, extra in zip(q, [500, 77, 260, 40])]
    w = workloads.make_custom(L, q, Hq=g, Hkv=1, D=128, block_size=32, seed=700 + g)
    want = gu.oracle_rows(w, gu.oracle_step(w))
    got = gu.gpu_step(pa, w, tc_pair=-1)
    st = got["plan"].stats()
    assert st["n_tc_pair_items"] == 0 and st["n_tc_items"] > st["n_tc_decode_items"]
    gu.assert_attention_close(got["out"].cpu().numpy(), want, f"g={g} fp32")
    got16 = gu.gpu_step(pa, w, out_dtype=torch.bfloat16, tc_pair=-1)
    d = np.abs(got16["out"].float().cpu().numpy() - want)
    bound = np.abs(want) * 2.0 ** -8 + gu.ATOL_MAX
    assert np.all(d <= bound), float((d - bound).max())


def test_tensor_core_pair_single_tile_items(pa):
    """Many consecutive two-tile items of one key tile each: every item's last S follows
    its first, so the next item's Q can land while the softmax warps still finish the
    previous item; they must take each item's description from its own barrier."""
    n = 600
    rng = np.random.default_rng(31)
    q = [32] * n
    L = [int(x) for x in rng.integers(32, 129, size=n)]
    w = workloads.make_custom(L, q, Hq=8, Hkv=1, D=128, block_size=16, seed=32,
                              write_new=False)
    got = gu.gpu_step(pa, w, tc_pair=1)
    assert got["err"] == 0, pa.DEVERR.get(got["err"])
    assert got["plan"].stats()["n_tc_pair_items"] == n
    rows = gu.sample_rows(w, 400, seed=33)
    want = gu.oracle_rows(w, gu.oracle_step(w), rows=rows)
    gu.assert_attention_close(got["out"].cpu().numpy()[rows], want, "single-tile items")


def test_tensor_core_pair_tiny_first(pa):
    """Smallest two-tile case: 129 rows, one key tile."""
    w = workloads.make_custom([129], [129], Hq=1, Hkv=1, D=128, block_size=16, seed=11)
    (_, _), got, _ = full_check(pa, w, tc_pair=1)
    assert got["plan"].stats()["n_tc_pair_items"] == 1


DECODE_CASES = [
    # (g, block_size, chunk): items of at most 16 rows, keys on the 128-row side
    (1, 16, 0), (2, 32, 0), (4, 16, 128), (8, 8, 0), (8, 256, 64), (16, 64, 0),
]


@pytest.mark.parametrize("g,B,chunk", DECODE_CASES)
def test_tensor_core_decode_items(pa, g, B, chunk):
    """Decode-like items (q x g <= 16 rows) on the key-major tensor-core kernel: ragged
    contexts around the 16- and 128-key edges, oracle and the other paths agree."""
    q = [1, 1, 1, 1, max(1, 16 // g), 1, max(1, 8 // g)]
    L = [1, 15, 128, 129, 300, 1000, 2049]
    w = workloads.make_custom(L, q, Hq=2 * g, Hkv=2, D=128, block_size=B, seed=500 + g + B)
    kw = dict(tc_min_rows=1)
    if chunk:
        kw["max_chunk_tokens"] = chunk
    (_, _), run, want = full_check(pa, w, **kw)
    assert run["plan"].stats()["n_tc_decode_items"] > 0
    (_, _), other, _ = full_check(pa, w, tc_decode=-1, **kw)
    assert other["plan"].stats()["n_tc_decode_items"] == 0
    assert torch.allclose(run["out"], other["out"], atol=gu.ATOL_MAX, rtol=0)


def test_tensor_core_decode_row_counts(pa):
    """Every row count 1..16 (the kernel runs the 1-, 2-, 4-, 8- or 16-row variant)."""
    q = list(range(1, 17))
    L = [q_ + 37 * i + 5 for i, q_ in enumerate(q)]
    w = workloads.make_custom(L, q, Hq=2, Hkv=2, D=128, block_size=16, seed=707)
    (_, _), got, _ = full_check(pa, w)
    items = got["plan"].items()
    assert sorted(set(items[items[:, 0] == 3][:, 4].tolist())) == q


def test_tensor_core_decode_tiny_first(pa):
    """Smallest key-major case: one row, one key."""
    w = workloads.make_custom([1], [1], Hq=1, Hkv=1, D=128, block_size=16, seed=13)
    (_, _), got, _ = full_check(pa, w, tc_min_rows=1)
    assert got["plan"].stats()["n_tc_decode_items"] == 1


def test_tensor_core_decode_nan_tail_and_bf16(pa):
    """Slots past each context hold NaN; the block tail inside the last 16-key step must
    not reach the output. bf16 output too."""
    w = workloads.make_custom([9, 20, 3, 130, 1001], [1, 1, 1, 1, 1], Hq=8, Hkv=2, D=128,
                              block_size=32, seed=15)
    used = np.zeros((w.num_blocks, w.block_size), bool)
    for s_, l_ in enumerate(w.context_lens):
        for t_ in range(int(l_)):
            used[w.block_table[s_, t_ // w.block_size], t_ % w.block_size] = True
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    w.k_pool[torch.from_numpy(~used)] = nan
    w.v_pool[torch.from_numpy(~used)] = nan
    got = gu.gpu_step(pa, w, tc_min_rows=1)
    assert got["plan"].stats()["n_tc_decode_items"] > 0
    want = gu.oracle_rows(w, gu.oracle_step(w))
    gu.assert_attention_close(got["out"].cpu().numpy(), want, "nan tail")
    got16 = gu.gpu_step(pa, w, out_dtype=torch.bfloat16, tc_min_rows=1)
    d = np.abs(got16["out"].float().cpu().numpy() - want)
    assert np.all(np.isfinite(d)) and d.max() <= 2e-2


def _growing_scores(w, slope=1.0 / 96, seed=5):
    """Rewrites a batch so that every query row's scores grow along the keys: K at
    position p is c(p) = p * slope on every dimension (plus small noise) and query rows
    are a_r on every dimension with a_r alternating between 1 and 1/20 by token. With
    D = 128 a row with a_r = 1 gains about 16 * 128 * slope in log2 units per 128 keys,
    so the kernels' lazy O rescale (when the running maximum grows by more than 2^8)
    fires on nearly every key tile for those rows and never for the others, in the
    same warps."""
    g = torch.Generator().manual_seed(seed)
    D = w.D
    kp = w.k_pool.float()
    for s, L in enumerate(w.context_lens):
        for p in range(int(L)):
            phys = int(w.block_table[s, p // w.block_size])
            kp[phys, p % w.block_size] = p * slope + 0.05 * torch.randn(w.Hkv, D, generator=g)
    w.k_pool = kp.to(torch.bfloat16)
    q = torch.empty(w.q.shape)
    tok = 0
    for n in w.query_lens:
        for t in range(int(n)):
            q[tok + t] = 1.0 if t % 2 == 0 else 0.05
        tok += int(n)
    w.q = q.to(torch.bfloat16)
    return w


NO_SPLIT = 1 << 14   # a chunk longer than every key range: no split-KV items


@pytest.mark.parametrize("kw", [{}, {"max_chunk_tokens": NO_SPLIT},
                                {"tc_pair": 1, "max_chunk_tokens": NO_SPLIT},
                                {"tc_pair": -1, "max_chunk_tokens": NO_SPLIT},
                                {"tc_min_rows": -1, "max_chunk_tokens": NO_SPLIT},
                                {"tc_decode": -1}, {"max_chunk_tokens": 192}])
def test_lazy_rescale_on_growing_scores(pa, kw):
    """Scores that keep growing along the keys force the online softmax to move its
    reference maximum tile after tile (the O rescale in TMEM, or in registers on the
    CUDA cores) in every kernel: key-major (q = 1, 3), one-tile (q = 40 or remainders),
    two-tile (q = 300 x 4 heads) and split items; checked against the oracle."""
    w = workloads.make_custom([900, 333, 700, 1100, 260], [1, 3, 40, 300, 2], Hq=8, Hkv=2,
                              D=128, block_size=16, seed=55, write_new=False)
    w = _growing_scores(w)
    want = gu.oracle_rows(w, gu.oracle_step(w))
    got = gu.gpu_step(pa, w, **kw)
    assert got["err"] == 0, pa.DEVERR.get(got["err"])
    gu.assert_attention_close(got["out"].cpu().numpy(), want, f"growing scores {kw}")


def test_unused_slots_hold_nan(pa):
    """Slots past each context (tail of the last block, unused blocks) hold NaN: no effect."""
    w = workloads.make_custom([9, 20, 3, 130], [2, 3, 3, 1], Hq=4, Hkv=2, D=128, block_size=16,
                              seed=5)
    used = np.zeros((w.num_blocks, w.block_size), bool)
    for s in range(w.num_seqs):
        for t in range(int(w.context_lens[s])):
            used[w.block_table[s, t // 16], t % 16] = True
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    mask = torch.from_numpy(~used)
    w.k_pool[mask] = nan
    w.v_pool[mask] = nan
    (_, _), got, _ = full_check(pa, w)
    assert torch.isfinite(got["out"]).all()


def test_permuted_physical_ids_bit_identical(pa):
    w = workloads.make_custom([77, 300, 5], [5, 1, 5], Hq=8, Hkv=2, D=128, block_size=16, seed=8)
    a = gu.gpu_step(pa, w)["out"]
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    inv = torch.from_numpy(np.argsort(perm))
    w.k_pool = w.k_pool[inv].contiguous()
    w.v_pool = w.v_pool[inv].contiguous()
    w.block_table = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    b = gu.gpu_step(pa, w)["out"]
    assert torch.equal(a, b)


def test_subrequests_match_single_request(pa):
    """Pensieve Fig. 8: sub-requests A (leading tokens on themselves) and B (new prompt on
    the whole context) reproduce the matching rows of one full causal request."""
    L, r, qn = 300, 64, 45
    full = workloads.make_custom([L], [L], Hq=8, Hkv=8, D=128, block_size=32, seed=12,
                                 write_new=False)
    two_w = workloads.make_custom([r, L], [r, qn], Hq=8, Hkv=8, D=128, block_size=32, seed=12,
                                  write_new=False)
    two_w.block_table = np.concatenate([full.block_table, full.block_table])
    two_w.k_pool, two_w.v_pool, two_w.num_blocks = full.k_pool, full.v_pool, full.num_blocks
    two_w.q = torch.cat([full.q[:r], full.q[L - qn:]])
    want = gu.oracle_rows(full, gu.oracle_step(full))
    for kw in ({}, {"tc_pair": 1}, {"tc_pair": -1}):
        one = gu.gpu_step(pa, full, **kw)["out"]
        two = gu.gpu_step(pa, two_w, **kw)["out"]
        gu.assert_attention_close(one.cpu().numpy(), want, "one request")
        gu.assert_attention_close(two[:r].cpu().numpy(), want[:r], "sub-request A")
        gu.assert_attention_close(two[r:].cpu().numpy(), want[L - qn:], "sub-request B")
    # With 128-row tiles only, every row takes the same arithmetic in both batches (the
    # same key tiles, the same exponentials); the rows only land in different work
    # items, so the two agree far inside the oracle tolerance. (With 256-row items the
    # full request's rows run in the two-tile kernel, whose per-row arithmetic differs
    # from the one-tile kernel's, and then only the oracle comparison above applies.)
    d_a = float((two[:r] - one[:r]).abs().max())
    d_b = float((two[r:] - one[L - qn:]).abs().max())
    assert d_a <= 2e-4 and d_b <= 2e-4, (d_a, d_b)


def test_plan_upload_serves_several_calls(pa):
    """One pa_plan_upload serves several pa_attention_planned calls, as a model's layers
    share a step's plan: each call equals pa_attention on the same inputs bit for bit,
    with a mix of key-major, one-tile, two-tile and split items."""
    w = workloads.make_custom([300, 130, 40, 1000, 700], [40, 20, 1, 3, 200], Hq=8, Hkv=2,
                              D=128, block_size=16, seed=77, write_new=False)
    dev = "cuda"
    bt = torch.from_numpy(w.block_table).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    ql = torch.from_numpy(w.query_lens).to(dev)
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    plan = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size, w.max_blocks,
                   tc_pair=1, max_chunk_tokens=256)
    st = plan.stats()
    assert st["n_tc_pair_items"] and st["n_tc_decode_items"] and st["n_split_groups"]
    g = torch.Generator().manual_seed(78)
    qs = [w.q.to(dev)] + [torch.randn(w.q.shape, generator=g).to(torch.bfloat16).to(dev)
                          for _ in range(2)]
    want = [pa.pa_attention(plan, q, kp, vp, bt, cl, ql) for q in qs]
    ws = plan.workspace(dev)
    pa.pa_plan_upload(plan, ws)
    got = [pa.pa_attention_planned(plan, q, kp, vp, bt, cl, ql, ws) for q in qs]
    assert pa.pa_get_device_error(reset=True) == 0
    for a, b in zip(got, want):
        assert torch.equal(a, b)
    ref = gu.oracle_rows(w, gu.oracle_step(w))
    gu.assert_attention_close(got[0].cpu().numpy(), ref, "planned call")


def test_plan_tables_outlive_early_destroy(pa):
    """Destroyed plans hand their pinned table buffers to later plans only once the
    uploads from them have completed: plans created, launched and destroyed while the
    stream is still busy (so every upload is still queued) and replaced by new plans
    with other tables all give the results of plans run one at a time."""
    dev = "cuda"
    ws_ = [workloads.make_custom([300 + 40 * i, 90 + i, 1000 - 30 * i], [1 + i, 20 + 3 * i, 2],
                                 Hq=8, Hkv=2, D=128, block_size=16, seed=500 + i,
                                 write_new=False) for i in range(6)]
    # device inputs first: a copy from pageable memory would wait for the busy stream
    dev_in = [(torch.from_numpy(w.block_table).to(dev), torch.from_numpy(w.context_lens).to(dev),
               torch.from_numpy(w.query_lens).to(dev), w.q.to(dev), w.k_pool.to(dev),
               w.v_pool.to(dev)) for w in ws_]
    torch.cuda.synchronize()

    def run(w, t):
        bt, cl, ql, q, kp, vp = t
        plan = pa.Plan(w.context_lens, w.query_lens, w.Hq, w.Hkv, w.D, w.block_size,
                       w.max_blocks)
        out = pa.pa_attention(plan, q, kp, vp, bt, cl, ql)
        plan.close()
        return out
    want = []
    for w, t in zip(ws_, dev_in):
        want.append(run(w, t))
        torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)       # keep the stream busy: the uploads below queue up
    got = [run(w, t) for w, t in zip(ws_, dev_in)]
    torch.cuda.synchronize()
    assert pa.pa_get_device_error(reset=True) == 0
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_bf16_output(pa):
    w = workloads.make(1)
    got = gu.gpu_step(pa, w, out_dtype=torch.bfloat16)
    want = gu.oracle_rows(w, gu.oracle_step(w))
    out = got["out"].float().cpu().numpy()
    # within one bf16 rounding of the oracle plus the attention tolerance
    assert np.all(np.abs(out - want) <= np.abs(want) * 2.0 ** -8 + gu.ATOL_MAX)


def test_empty_batch_and_zero_queries(pa):
    w = workloads.make_custom([0, 5, 0], [0, 0, 0], Hq=4, Hkv=4, D=64, block_size=16, seed=1)
    got = gu.gpu_step(pa, w)
    assert got["out"].numel() == 0 and got["err"] == 0


def test_bad_block_id_is_reported_not_faulted(pa):
    """A block id past the pool is skipped by the kernel and reported in the error word."""
    w = workloads.make_custom([40, 40], [1, 1], Hq=4, Hkv=4, D=64, block_size=16, seed=3,
                              write_new=False)
    good = w.block_table.copy()
    w.block_table[1, 1] = w.num_blocks + 5
    got = gu.gpu_step(pa, w)
    assert got["err"] == 2
    # the healthy sequence is still right
    w.block_table = good
    want = gu.oracle_rows(w, gu.oracle_step(w), rows=np.array([0]))
    gu.assert_attention_close(got["out"].cpu().numpy()[:1], want, "healthy row")


def test_write_kv_skip_and_range(pa):
    dev = "cuda"
    kp = torch.zeros(4, 2, 1, 8, dtype=torch.bfloat16, device=dev)
    vp = kp.clone()
    kn = torch.ones(3, 1, 8, dtype=torch.bfloat16, device=dev)
    vn = kn * 2
    slots = torch.tensor([-1, 5, 99], dtype=torch.int64, device=dev)
    pa.pa_write_kv(kn, vn, slots, kp, vp)
    assert pa.pa_get_device_error(reset=True) == 1
    flat = kp.view(8, 8).float().cpu()
    assert flat[5].eq(1).all() and flat.sum() == 8
    assert vp.view(8, 8)[5].float().eq(2).all()


def test_cow_config_copies_bit_exact(pa):
    """Config 5cow (the fork step): 224 copy-on-write block copies, then the KV write,
    bit-exact on both whole pools; attention compared with the oracle on every row."""
    w = workloads.make("5cow", device="cuda")
    got = gu.gpu_step(pa, w)
    ref = gu.oracle_step(w)
    assert got["err"] == 0
    assert np.array_equal(got["slots"], ref["slots"])
    assert gu.pools_equal(got["k_pool"], ref["k_pool"])
    assert gu.pools_equal(got["v_pool"], ref["v_pool"])
    gu.compare_all_rows(got["out"], w, ref, w.name)


@pytest.mark.parametrize("config", [2, 3, 4, 5])
def test_full_size_configs(pa, config):
    """The bench's workloads at full size, in the plan the bench times: slot maps and
    both whole pools bit-exact, and attention compared with the fp64 oracle on EVERY
    query row and head (config 3: about 48.6k rows x 40 heads), so that every work item
    of every kernel -- every persistent CTA round and barrier phase -- is checked."""
    w = workloads.make(config, device="cuda")
    got = gu.gpu_step(pa, w)
    assert got["err"] == 0
    ref = gu.oracle_step(w)
    assert np.array_equal(got["slots"], ref["slots"])
    assert gu.pools_equal(got["k_pool"], ref["k_pool"])
    assert gu.pools_equal(got["v_pool"], ref["v_pool"])
    del got["k_pool"], got["v_pool"]
    gu.compare_all_rows(got["out"], w, ref, w.name)


FUSED_CASES = {
    "config1": lambda: workloads.make(1),
    # decode rows of g = 4 with split keys: the new tokens straddle 64-key chunk
    # boundaries, so several chunk items of one (sequence, KV head) each write theirs
    "split_straddle": lambda: workloads.make_custom([190, 257, 66, 1000, 4], [3, 4, 2, 1, 4],
                                                    Hq=16, Hkv=4, D=128, block_size=16,
                                                    seed=611),
    # decode rows beside one-tile and two-tile rows: the write kernel skips the rows the
    # key-major kernel writes
    "mixed_paths": lambda: workloads.make_custom([300, 700, 40, 900, 129], [1, 200, 40, 2, 100],
                                                 Hq=8, Hkv=2, D=128, block_size=32, seed=612),
}


@pytest.mark.parametrize("case", list(FUSED_CASES))
def test_fused_write_attention(pa, case):
    """pa_attention_write = pa_write_kv + pa_attention: both whole pools bit-exact against
    the oracle's write, every attention row within tolerance, the output bit-identical to
    the unfused pair of calls, and the same with split keys forced."""
    w = FUSED_CASES[case]()
    for kw in (dict(), dict(max_chunk_tokens=64)):
        got = gu.gpu_step(pa, w, fused=True, **kw)
        ref = gu.oracle_step(w)
        assert got["err"] == 0, f"device error {pa.DEVERR.get(got['err'])}"
        assert gu.pools_equal(got["k_pool"], ref["k_pool"]), "K pool differs after the write"
        assert gu.pools_equal(got["v_pool"], ref["v_pool"]), "V pool differs after the write"
        gu.compare_all_rows(got["out"], w, ref, f"fused {case} {kw}")
        base = gu.gpu_step(pa, w, **kw)
        assert torch.equal(got["out"], base["out"])
    if case != "config1":
        assert got["plan"].stats()["n_tc_decode_items"] > 0


@pytest.mark.parametrize("config", [2, 3, "5cow"])
def test_fused_write_attention_full_size(pa, config):
    """The fused call on the full-size decode, mixed and copy-on-write batches: pools
    bit-exact, every row against the oracle."""
    w = workloads.make(config, device="cuda")
    got = gu.gpu_step(pa, w, fused=True)
    assert got["err"] == 0
    ref = gu.oracle_step(w)
    assert gu.pools_equal(got["k_pool"], ref["k_pool"])
    assert gu.pools_equal(got["v_pool"], ref["v_pool"])
    del got["k_pool"], got["v_pool"]
    gu.compare_all_rows(got["out"], w, ref, f"fused {w.name}")
