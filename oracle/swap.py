"""Block swaps between two pools (device <-> host), in plain Python.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

vLLM post (devpress), "3. scheduling and preemption": when the GPU's blocks run
out, the blocks of evicted requests are copied to CPU memory and copied back when
the requests resume; Pensieve summary, ahead-of-time swapping of KV tokens to the
CPU cache and their restore. Pair i copies whole block src[i] of one pool (K and V)
into block dst[i] of the other; destinations must be distinct (the copies would
race otherwise), every id inside its pool.
"""
import numpy as np


def swap_blocks(k_from, v_from, k_to, v_to, src, dst) -> None:
    """k_from, v_from [n_from, B, Hkv, D]; k_to, v_to [n_to, B, Hkv, D] (same dtype),
    modified in place."""
    src = [int(x) for x in np.asarray(src).reshape(-1)]
    dst = [int(x) for x in np.asarray(dst).reshape(-1)]
    if len(src) != len(dst):
        raise ValueError("src and dst need the same length")
    if len(set(dst)) != len(dst):
        raise ValueError("destinations must be distinct")
    n_from, n_to = k_from.shape[0], k_to.shape[0]
    for s, d in zip(src, dst):
        if not (0 <= s < n_from and 0 <= d < n_to):
            raise ValueError(f"block pair ({s}, {d}) outside the pools")
    for s, d in zip(src, dst):
        k_to[d] = k_from[s]
        v_to[d] = v_from[s]
