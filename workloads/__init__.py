"""Seeded synthetic workloads for the paged-attention hot path.

This module only draws inputs: sequence lengths, block placement (block
tables), the positions of the step's new tokens, copy-on-write pairs and bf16
values. It holds none of the attention, slot or copy arithmetic; the library
and the oracle each compute those from what is drawn here.

Shapes follow the chat workloads the pages describe (ShareGPT-like multi-turn
conversations for Pensieve, OPT-13B / Llama-2 attention shapes, vLLM's
parallel sampling). No dataset is read: every length and value is drawn from
a seeded generator (``torch.Generator().manual_seed(1000 + config)``, used for
lengths, then placement, then values, in that order).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = ["Workload", "make", "make_custom", "host_bits", "CONFIG_NAMES", "CONFIG_IDS"]

CONFIG_NAMES = {
    1: "tiny mixed batch: 4 seqs, Hq=Hkv=4, D=64, B=16",
    2: "decode-only, OPT-13B attention shape: 256 seqs x q=1, Hq=Hkv=40, D=128, B=16",
    3: "Pensieve unified multi-turn, Llama-2-13B shape: 64 conversations as 2 sub-requests each "
       "+ 128 decode, Hq=Hkv=40, D=128, B=32",
    4: "GQA, Llama-2-70B layer shape: 128 seqs, Hq=64, Hkv=8, D=128, B=32",
    5: "shared-prefix parallel sampling: 32 prompts x 8 samples, Hq=32, Hkv=8, D=128, B=16",
    "5cow": "shared-prefix fork step with copy-on-write: 32 prompts x 8 samples, 1032-token "
            "prompts, Hq=32, Hkv=8, D=128, B=16",
}
CONFIG_IDS = [1, 2, 3, 4, 5, "5cow"]


@dataclass
class Workload:
    name: str
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray          # int32 [N]
    query_lens: np.ndarray            # int32 [N]
    block_table: np.ndarray           # int32 [N, max_blocks]; -1 past each sequence's blocks
    new_seq: np.ndarray               # int32 [n_new]: block-table row of each new token
    new_pos: np.ndarray               # int32 [n_new]: its absolute position in that sequence
    cow_src: np.ndarray               # int32 [P]: copy-on-write source blocks for this step
    cow_dst: np.ndarray               # int32 [P]: their destinations
    q: torch.Tensor                   # bf16 [T, Hq, D]
    k_pool: torch.Tensor              # bf16 [num_blocks, B, Hkv, D], state before the step
    v_pool: torch.Tensor
    k_new: torch.Tensor               # bf16 [n_new, Hkv, D]
    v_new: torch.Tensor
    seed: int = 0
    groups: dict = field(default_factory=dict)   # named row groups (e.g. decode / prefill)

    @property
    def num_seqs(self) -> int:
        return int(len(self.context_lens))

    @property
    def total_q(self) -> int:
        return int(self.query_lens.sum())

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def subset(self, seqs) -> "Workload":
        """The sub-batch of the listed sequences (same pools, same values, same blocks)."""
        seqs = np.asarray(sorted(int(x) for x in seqs), dtype=np.int64)
        pref = np.concatenate([[0], np.cumsum(self.query_lens.astype(np.int64))])
        rows = np.concatenate([np.arange(pref[s], pref[s + 1]) for s in seqs]) if len(seqs) else \
            np.zeros(0, np.int64)
        remap = {int(s): i for i, s in enumerate(seqs)}
        keep = np.array([int(s) in remap for s in self.new_seq], dtype=bool)
        idx = torch.from_numpy(np.nonzero(keep)[0])
        return Workload(name=self.name, Hq=self.Hq, Hkv=self.Hkv, D=self.D,
                        block_size=self.block_size, num_blocks=self.num_blocks,
                        context_lens=self.context_lens[seqs], query_lens=self.query_lens[seqs],
                        block_table=self.block_table[seqs],
                        new_seq=np.array([remap[int(s)] for s in self.new_seq[keep]], np.int32),
                        new_pos=self.new_pos[keep], cow_src=self.cow_src, cow_dst=self.cow_dst,
                        q=self.q[torch.from_numpy(rows).to(self.q.device)],
                        k_pool=self.k_pool, v_pool=self.v_pool,
                        k_new=self.k_new[idx.to(self.k_new.device)],
                        v_new=self.v_new[idx.to(self.v_new.device)], seed=self.seed, groups={})

    def kv_bytes(self) -> int:
        """K and V bytes one attention pass reads: sum over sequences of L * 2 * Hkv * D * 2."""
        return int(self.context_lens.astype(np.int64).sum()) * 2 * self.Hkv * self.D * 2

    def q_bytes(self) -> int:
        return self.total_q * self.Hq * self.D * 2

    def flops(self) -> int:
        """4 * Hq * D per visible (query, key) pair; a row at position p sees p + 1 keys."""
        L = self.context_lens.astype(np.int64)
        q = self.query_lens.astype(np.int64)
        pairs = int((q * (L - q) + q * (q + 1) // 2).sum())
        return 4 * self.Hq * self.D * pairs


# ----------------------------------------------------------------- helpers

def host_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor as a host array of its uint16 bit patterns (a copy): the form in
    which the CPU-side consumers of these inputs take bf16 values."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _cdiv(a, b):
    return -(-a // b)


def _randint(g, lo, hi, n):
    """n integers uniform in [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (n,), generator=g).numpy().astype(np.int64)


def _values(seed: int, device, shapes, scales):
    """bf16 N(0,1) * scale tensors, drawn in order from one generator on ``device``.

    Large tensors are drawn in slices along their first dimension so that the
    float32 staging buffer stays small.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    out = []
    for shape, scale in zip(shapes, scales):
        t = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        if t.numel():
            rows_per = max(1, (1 << 26) // max(1, t[0].numel()))
            for i in range(0, shape[0], rows_per):
                sl = t[i:i + rows_per]
                x = torch.randn(sl.shape, generator=g, device=dev, dtype=torch.float32)
                if scale != 1.0:
                    x.mul_(scale)
                sl.copy_(x)
        out.append(t)
    return out


def _place(g, need_per_seq, num_blocks, max_blocks, region=None):
    """Assign each sequence its blocks from a seeded permutation of the pool.

    ``region`` optionally restricts the permutation to a range of block ids.
    Returns the block table (padding -1).
    """
    lo, hi = (0, num_blocks) if region is None else region
    perm = (torch.randperm(hi - lo, generator=g) + lo).numpy().astype(np.int32)
    bt = np.full((len(need_per_seq), max_blocks), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(need_per_seq):
        bt[s, :n] = perm[off:off + n]
        off += n
    assert off <= hi - lo
    return bt


def _finish(name, seed, Hq, Hkv, D, B, nb, L, ql, bt, new_seq, new_pos, device,
            q_scale=1.0, cow=None, groups=None):
    L = np.asarray(L, dtype=np.int32)
    ql = np.asarray(ql, dtype=np.int32)
    T = int(ql.sum())
    n_new = len(new_seq)
    q, kp, vp, kn, vn = _values(
        seed, device,
        [(T, Hq, D), (nb, B, Hkv, D), (nb, B, Hkv, D), (n_new, Hkv, D), (n_new, Hkv, D)],
        [q_scale, 1.0, 1.0, 1.0, 1.0])
    src, dst = (np.zeros(0, np.int32), np.zeros(0, np.int32)) if cow is None else cow
    return Workload(name=name, Hq=Hq, Hkv=Hkv, D=D, block_size=B, num_blocks=nb,
                    context_lens=L, query_lens=ql, block_table=bt,
                    new_seq=np.asarray(new_seq, np.int32), new_pos=np.asarray(new_pos, np.int32),
                    cow_src=np.asarray(src, np.int32), cow_dst=np.asarray(dst, np.int32),
                    q=q, k_pool=kp, v_pool=vp, k_new=kn, v_new=vn, seed=seed,
                    groups=groups or {})


def _last_tokens(L, ql):
    """(sequence, position) of the last ql[s] tokens of every sequence."""
    seqs, pos = [], []
    for s, (l, q) in enumerate(zip(L, ql)):
        seqs += [s] * int(q)
        pos += list(range(int(l) - int(q), int(l)))
    return seqs, pos


# ----------------------------------------------------------------- configs

def make_custom(context_lens, query_lens, Hq, Hkv, D, block_size, seed=0, device="cpu",
                pool_factor=1.2, num_blocks=None, q_scale=1.0, write_new=True):
    """A ragged batch with the given lengths; blocks placed by a seeded permutation.

    The new tokens of the step are the last query_len tokens of every sequence
    (written before attention when ``write_new``).
    """
    g = torch.Generator().manual_seed(int(seed))
    L = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    need = [_cdiv(int(l), block_size) for l in L]
    max_blocks = max(1, max(need) if len(need) else 1)
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * max(1, sum(need)))))
    bt = _place(g, need, num_blocks, max_blocks)
    seqs, pos = _last_tokens(L, ql) if write_new else ([], [])
    return _finish(f"custom(seed={seed})", int(seed), Hq, Hkv, D, block_size, num_blocks, L, ql,
                   bt, seqs, pos, device, q_scale=q_scale)


def _cfg1(device):
    seed = 1001
    g = torch.Generator().manual_seed(seed)
    L, ql = [7, 33, 64, 100], [1, 1, 7, 17]
    B, nb = 16, 64
    need = [_cdiv(l, B) for l in L]
    bt = _place(g, need, nb, max(need))
    seqs, pos = _last_tokens(L, ql)
    return _finish(CONFIG_NAMES[1], seed, 4, 4, 64, B, nb, L, ql, bt, seqs, pos, device)


def _cfg2(device, max_seqs=None, block_size=None, contiguous=False):
    """Decode-only batch. ``block_size`` and ``contiguous`` give the block-size sweep's
    variants of the same draw (same lengths and values): another block size, or each
    sequence's blocks at consecutive physical ids instead of a seeded permutation."""
    seed = 1002
    g = torch.Generator().manual_seed(seed)
    N, B, H, D = 256, 16, 40, 128
    if block_size is not None:
        B = int(block_size)
    L = _randint(g, 128, 2048, N)
    if max_seqs is not None:
        N, L = min(N, max_seqs), L[:max_seqs]
    ql = np.ones(N, np.int64)
    need = [_cdiv(int(l), B) for l in L]
    nb = int(math.ceil(1.2 * sum(need)))
    bt = _place(g, need, nb, max(need))
    name = CONFIG_NAMES[2]
    if block_size is not None and B != 16:
        name = name.replace("B=16", f"B={B}")
    if contiguous:
        off = 0
        for s, n in enumerate(need):
            bt[s, :n] = np.arange(off, off + n, dtype=np.int32)
            off += n
        name += ", contiguous blocks"
    seqs, pos = _last_tokens(L, ql)
    return _finish(name, seed, H, H, D, B, nb, L, ql, bt, seqs, pos, device,
                   q_scale=1.0 / math.sqrt(D))


def _cfg3(device, contiguous=False, max_seqs=None):
    """64 conversations (history + new turn) as two sub-requests each, plus 128 decodes.

    Conversation c has ``hist`` cached tokens and ``qn`` new prompt tokens. Its
    leading ``r = 32 k`` tokens (k uniform in [1, hist // 64]) were dropped and
    are recomputed this step; tokens [r, hist) were swapped back in. The
    leading and new-turn blocks come from pool region 0, the swapped-in middle
    from region 1. Sub-request A: context r, query r (the leading tokens attend
    to themselves). Sub-request B: context hist + qn, query qn (the new prompt
    attends to the whole context). Both rows of the block table list the same
    physical blocks for the shared part. ``contiguous``: the same draw with each
    conversation's (and decode sequence's) blocks at consecutive physical ids, for the
    paged-against-contiguous comparison of the multi-token kernels.
    """
    seed = 1003
    g = torch.Generator().manual_seed(seed)
    Hq = Hkv = 40
    D, B, C, ND = 128, 32, 64, 128
    hist = _randint(g, 512, 3072, C)
    qn = _randint(g, 32, 512, C)
    kk = np.array([int(_randint(g, 1, int(h) // 64, 1)[0]) for h in hist], dtype=np.int64)
    r = 32 * kk
    Ld = _randint(g, 256, 4096, ND)
    if max_seqs is not None:
        # the first max_seqs conversations and 2 * max_seqs decode sequences of the same
        # length draw (the block placement is drawn for the smaller pool)
        C, ND = min(C, int(max_seqs)), min(ND, 2 * int(max_seqs))
        hist, qn, kk, Ld = hist[:C], qn[:C], kk[:C], Ld[:ND]
        r = 32 * kk
    # block needs per region
    full = hist + qn
    nblk = [_cdiv(int(x), B) for x in full]
    lead_blk = [int(x) // B for x in r]                  # r is a multiple of 32 = B
    tail_first = [int(h) // B for h in hist]             # block holding token hist (if any)
    mid_blk = [tf - lb for tf, lb in zip(tail_first, lead_blk)]
    new_blk = [nb_ - tf for nb_, tf in zip(nblk, tail_first)]
    dec_blk = [_cdiv(int(x), B) for x in Ld]
    need0 = sum(lead_blk) + sum(new_blk) + sum(dec_blk)
    need1 = sum(mid_blk)
    n0, n1 = int(math.ceil(1.2 * need0)), int(math.ceil(1.2 * need1))
    nb = n0 + n1
    perm0 = (torch.randperm(n0, generator=g)).numpy().astype(np.int32)
    perm1 = (torch.randperm(n1, generator=g) + n0).numpy().astype(np.int32)
    max_blocks = max(max(nblk), max(dec_blk))
    rows_L, rows_q, bt_rows = [], [], []
    o0 = o1 = 0
    conv_tables = []
    for c in range(C):
        row = np.full(max_blocks, -1, np.int32)
        lb, mb, nwb = lead_blk[c], mid_blk[c], new_blk[c]
        row[:lb] = perm0[o0:o0 + lb]; o0 += lb
        row[lb:lb + mb] = perm1[o1:o1 + mb]; o1 += mb
        row[lb + mb:lb + mb + nwb] = perm0[o0:o0 + nwb]; o0 += nwb
        conv_tables.append(row)
    dec_tables = []
    for s in range(ND):
        row = np.full(max_blocks, -1, np.int32)
        row[:dec_blk[s]] = perm0[o0:o0 + dec_blk[s]]; o0 += dec_blk[s]
        dec_tables.append(row)
    if contiguous:
        off = 0
        for row in conv_tables + dec_tables:
            n = int((row >= 0).sum())
            row[:n] = np.arange(off, off + n, dtype=np.int32)
            off += n
        assert off <= nb
    new_seq, new_pos = [], []
    for c in range(C):
        # sub-request A: the recomputed leading tokens
        a = len(rows_L)
        rows_L.append(int(r[c])); rows_q.append(int(r[c])); bt_rows.append(conv_tables[c])
        # sub-request B: the new prompt over the whole context
        b = len(rows_L)
        rows_L.append(int(full[c])); rows_q.append(int(qn[c])); bt_rows.append(conv_tables[c])
        new_seq += [a] * int(r[c]); new_pos += list(range(int(r[c])))
        new_seq += [b] * int(qn[c]); new_pos += list(range(int(hist[c]), int(full[c])))
    n_conv_rows = len(rows_L)
    for s in range(ND):
        i = len(rows_L)
        rows_L.append(int(Ld[s])); rows_q.append(1); bt_rows.append(dec_tables[s])
        new_seq.append(i); new_pos.append(int(Ld[s]) - 1)
    bt = np.stack(bt_rows).astype(np.int32)
    groups = {"prefill_seqs": list(range(n_conv_rows)),
              "decode_seqs": list(range(n_conv_rows, len(rows_L)))}
    name = CONFIG_NAMES[3] + (", contiguous blocks" if contiguous else "")
    return _finish(name, seed, Hq, Hkv, D, B, nb, rows_L, rows_q, bt, new_seq,
                   new_pos, device, groups=groups)


def _cfg4(device, block_size=None, contiguous=False):
    """GQA batch. ``block_size`` and ``contiguous`` give the same draw with another block
    size or with each sequence's blocks at consecutive physical ids."""
    seed = 1004
    g = torch.Generator().manual_seed(seed)
    N, Hq, Hkv, D, B = 128, 64, 8, 128, 32
    if block_size is not None:
        B = int(block_size)
    z = torch.randn(N, generator=g, dtype=torch.float64).numpy()
    L = np.minimum(np.rint(np.exp(math.log(1500.0) + 0.5 * z)).astype(np.int64), 4096)
    is_prefill = torch.rand(N, generator=g, dtype=torch.float64).numpy() >= 0.7
    qlen_draw = _randint(g, 16, 256, N)
    ql = np.where(is_prefill, qlen_draw, 1).astype(np.int64)
    L = np.maximum(L, ql)
    need = [_cdiv(int(l), B) for l in L]
    nb = int(math.ceil(1.1 * sum(need)))
    bt = _place(g, need, nb, max(need))
    name = CONFIG_NAMES[4]
    if B != 32:
        name = name.replace("B=32", f"B={B}")
    if contiguous:
        off = 0
        for s, n in enumerate(need):
            bt[s, :n] = np.arange(off, off + n, dtype=np.int32)
            off += n
        name += ", contiguous blocks"
    seqs, pos = _last_tokens(L, ql)
    groups = {"prefill_seqs": [int(i) for i in np.nonzero(ql > 1)[0]],
              "decode_seqs": [int(i) for i in np.nonzero(ql == 1)[0]]}
    return _finish(name, seed, Hq, Hkv, D, B, nb, L, ql, bt, seqs, pos, device,
                   groups=groups)


def _cfg5(device, cow: bool):
    """Parallel sampling over a shared prompt (vLLM post, "2.1 parallel sampling").

    Main step: 1024-token prompts (64 full blocks, shared by the 8 samples of a
    group); sample s already holds d_s ~ U{0..256} private tokens and decodes
    one more (context 1025 + d_s). With no partial shared block nothing needs a
    copy, so the step's copy list is empty.

    Fork step (``cow``): 1032-token prompts (64 full blocks + one shared block
    holding 8 tokens), every sample decodes its first token at position 1032.
    In each group the first seven writers get a fresh block copied from the
    shared partial block and the last writes into the original (refcount 1 by
    then), which gives 7 * 32 = 224 copies.
    """
    seed = 1005 if not cow else 1006
    g = torch.Generator().manual_seed(seed)
    P, S, Hq, Hkv, D, B = 32, 8, 32, 8, 128, 16
    prompt = 1032 if cow else 1024
    n_shared = _cdiv(prompt, B)
    d = np.zeros(P * S, np.int64) if cow else _randint(g, 0, 256, P * S)
    L = prompt + d + 1
    priv = [_cdiv(int(l), B) - n_shared for l in L]       # private blocks per sample
    if cow:
        priv = [1] * (P * S)                               # room for a copy of the partial block
    need = P * n_shared + sum(priv)
    nb = int(math.ceil(1.2 * need))
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int32)
    max_blocks = max(_cdiv(int(l), B) for l in L)
    bt = np.full((P * S, max_blocks), -1, np.int32)
    off = 0
    src, dst = [], []
    for p in range(P):
        shared = perm[off:off + n_shared]; off += n_shared
        for s in range(S):
            i = p * S + s
            bt[i, :n_shared] = shared
            mine = perm[off:off + priv[i]]; off += priv[i]
            if cow:
                if s < S - 1:       # refcount > 1 when this sample writes: copy, then remap
                    src.append(int(shared[-1])); dst.append(int(mine[0]))
                    bt[i, n_shared - 1] = mine[0]
            else:
                bt[i, n_shared:n_shared + priv[i]] = mine
    ql = np.ones(P * S, np.int64)
    seqs, pos = _last_tokens(L, ql)
    name = CONFIG_NAMES["5cow" if cow else 5]
    return _finish(name, seed, Hq, Hkv, D, B, nb, L, ql, bt, seqs, pos, device,
                   cow=(np.array(src, np.int32), np.array(dst, np.int32)))


def make(config, device="cpu", max_seqs=None, block_size=None, contiguous=False) -> Workload:
    """Workload for config 1..5 or "5cow", values drawn on ``device``.

    ``max_seqs`` keeps only the first sequences of the decode-only batch (config 2), or
    the first conversations and twice as many decode sequences of config 3: the same
    length draw, smaller, for profiler captures that must stay small. ``block_size``
    (configs 2 and 4) and ``contiguous`` (configs 2, 3 and 4) give the block-size sweep's
    and the paged-against-contiguous comparison's variants of the same draw.
    """
    if block_size is not None and config not in (2, "2", 4, "4"):
        raise ValueError("block_size variants exist for configs 2 and 4 only")
    if contiguous and config not in (2, "2", 3, "3", 4, "4"):
        raise ValueError("contiguous variants exist for configs 2, 3 and 4 only")
    if config in (1, "1"):
        return _cfg1(device)
    if config in (2, "2"):
        return _cfg2(device, max_seqs, block_size, contiguous)
    if config in (3, "3"):
        return _cfg3(device, contiguous, max_seqs)
    if config in (4, "4"):
        return _cfg4(device, block_size, contiguous)
    if config in (5, "5"):
        return _cfg5(device, cow=False)
    if config == "5cow":
        return _cfg5(device, cow=True)
    raise ValueError(f"unknown config {config!r}")
