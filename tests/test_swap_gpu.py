"""GPU parity of pa_swap_blocks (device pools <-> page-locked host pools) against the
oracle's block swap: bit-exact, whole pools compared (untouched blocks included)."""
import numpy as np
import pytest
import torch

from oracle.swap import swap_blocks
from tests import gpu_util as gu
from tests.oracle_checks import u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gu.lib()


def _pools(n, shape, seed, device=None, pin=False):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn((n,) + shape, generator=g).to(torch.bfloat16)
    v = torch.randn((n,) + shape, generator=g).to(torch.bfloat16)
    if pin:
        return k.pin_memory(), v.pin_memory()
    return (k.to(device), v.to(device)) if device else (k, v)


@pytest.mark.parametrize("B,Hkv,D", [(16, 40, 128), (32, 8, 128), (16, 4, 64)])
def test_swap_out_and_in_bit_exact(pa, B, Hkv, D):
    dev = "cuda"
    pa.pa_get_device_error()                              # start from a clear error word
    nb, nhb = 300, 200
    kd, vd = _pools(nb, (B, Hkv, D), 1, device=dev)
    kh, vh = _pools(nhb, (B, Hkv, D), 2, pin=True)
    rng = np.random.default_rng(B + D)
    src = rng.choice(nb, 150, replace=False).astype(np.int32)
    dst = rng.choice(nhb, 150, replace=False).astype(np.int32)
    want_k, want_v = u16(kh), u16(vh)
    swap_blocks(u16(kd), u16(vd), want_k, want_v, src, dst)
    pa.pa_swap_blocks(kd, vd, kh, vh, torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev),
                      "out")
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert np.array_equal(u16(kh), want_k) and np.array_equal(u16(vh), want_v)
    # back in: host blocks -> other device blocks (a restore into fresh slots)
    src2 = dst[:100]
    dst2 = rng.choice(nb, 100, replace=False).astype(np.int32)
    want_kd, want_vd = u16(kd), u16(vd)
    swap_blocks(u16(kh), u16(vh), want_kd, want_vd, src2, dst2)
    pa.pa_swap_blocks(kd, vd, kh, vh, torch.from_numpy(src2).to(dev),
                      torch.from_numpy(dst2).to(dev), "in")
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert np.array_equal(u16(kd), want_kd) and np.array_equal(u16(vd), want_vd)


def test_swap_rejects_pageable_host_memory_and_skips_bad_ids(pa):
    dev = "cuda"
    pa.pa_get_device_error()
    kd, vd = _pools(8, (16, 2, 64), 3, device=dev)
    kh, vh = _pools(8, (16, 2, 64), 4)                  # pageable: refused on the host
    ids = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_swap_blocks(kd, vd, kh, vh, ids, ids, "out")
    kh, vh = kh.pin_memory(), vh.pin_memory()
    before_k, before_v = u16(kh), u16(vh)
    bad_src = torch.tensor([0, 8], dtype=torch.int32, device=dev)   # 8 is outside the pool
    dst = torch.tensor([5, 6], dtype=torch.int32, device=dev)
    pa.pa_swap_blocks(kd, vd, kh, vh, bad_src, dst, "out")
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 2                 # block id out of range, recorded
    want_k, want_v = before_k.copy(), before_v.copy()
    want_k[5], want_v[5] = u16(kd)[0], u16(vd)[0]          # the valid pair still moved
    assert np.array_equal(u16(kh), want_k) and np.array_equal(u16(vh), want_v)


def test_block_manager_drives_swaps(pa):
    """The block manager's swap pairs moved by pa_swap_blocks: requests swapped out, their
    device blocks overwritten, swapped back in to other blocks, read back intact."""
    from tests import bm_checks as bc
    dev = "cuda"
    pa.pa_get_device_error()
    kd, vd = _pools(16, (4, 2, 64), 5, device=dev)
    kh, vh = _pools(12, (4, 2, 64), 6, pin=True)
    bm = pa.BlockManager(16, 4, num_host_blocks=12)

    def gather(table):
        t = torch.tensor(table, dtype=torch.long, device=dev)
        return torch.cat([kd[t], vd[t]]).cpu()

    def scribble(blocks):
        t = torch.tensor(blocks, dtype=torch.long, device=dev)
        kd[t] = 7.0
        vd[t] = 9.0

    def move(pairs, direction):
        src = torch.tensor([a for a, _ in pairs], dtype=torch.int32, device=dev)
        dst = torch.tensor([b for _, b in pairs], dtype=torch.int32, device=dev)
        pa.pa_swap_blocks(kd, vd, kh, vh, src, dst, direction)
        torch.cuda.synchronize()

    bc.swap_roundtrip(bm, gather, scribble, move)
    assert pa.pa_get_device_error() == 0
