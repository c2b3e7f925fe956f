// pa_kv.cu -- cache maintenance kernels: slot mapping, KV write, copy-on-write block copy,
// block swaps between the device pools and page-locked host pools.
//
// vLLM post (devpress), "1. overall architecture": token position p of a
// sequence lives in slot block_table[p / B] * B + p % B of the pool, a pool row
// being the Hkv * D values of one token. vLLM wiki note, "kernel layer": the
// new tokens' K/V are scattered into their slots (fused reshape + block write)
// and whole blocks are copied for copy-on-write (batched block copy; vLLM post,
// "2.1 parallel sampling"). Swapping (vLLM post, "3. scheduling and preemption":
// evicted blocks are copied to CPU memory and back; Pensieve summary, ahead-of-time
// swapping of KV tokens to the CPU cache and their restore) moves whole blocks between
// the device pools and host pools of the same layout.
//
// All are bandwidth-bound byte movers: 16-byte vector accesses, a grid sized to
// a multiple of the SM count, every index range-checked (a bad index is
// skipped and recorded in the device error word, never dereferenced).
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

__global__ void slot_mapping_kernel(const int32_t* __restrict__ bt, int32_t num_seqs,
                                    int32_t max_blocks, int32_t block_size, int32_t num_blocks,
                                    const int32_t* __restrict__ seq_ids,
                                    const int32_t* __restrict__ positions, int64_t n,
                                    int64_t* __restrict__ slots, int* err) {
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int32_t s = seq_ids[t];
    const int32_t p = positions[t];
    int64_t slot = -1;
    if (p >= 0) {
      const int32_t logical = p / block_size;
      if (s < 0 || s >= num_seqs || logical >= max_blocks) {
        record_error(err, PA_DEVERR_TABLE_RANGE);
      } else {
        const int32_t phys = bt[(int64_t)s * max_blocks + logical];
        if (phys < 0 || phys >= num_blocks)
          record_error(err, PA_DEVERR_BLOCK_RANGE);
        else
          slot = (int64_t)phys * block_size + (p - logical * block_size);
      }
    }
    slots[t] = slot;
  }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

// Moves token rows of 16-byte vectors: one warp per row at a time, the row's slot read
// once, then the row's vectors spread over the lanes (512 contiguous bytes per warp
// access), kCopyUnroll loads of K and of V in flight per lane before their stores.
// Source rows are contiguous; the destination row comes from the slot list. Rows whose
// entry in `skip` (optional, one byte per row) is non-zero are left to another kernel.
__global__ void __launch_bounds__(kCopyThreads) write_kv_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slots, int64_t n_rows, int vec_per_row,
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int64_t n_slots,
    const uint8_t* __restrict__ skip, int* err) {
  constexpr int kWarps = kCopyThreads / 32;
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = (int64_t)gridDim.x * kWarps;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < n_rows;
       row += n_warps) {
    if (skip && __ldg(skip + row)) continue;
    const int64_t slot = __ldg(slots + row);
    if (slot < 0) continue;
    if (slot >= n_slots) {
      if (lane == 0) record_error(err, PA_DEVERR_SLOT_RANGE);
      continue;
    }
    const uint4* ks = k_new + row * vec_per_row;
    const uint4* vs = v_new + row * vec_per_row;
    uint4* kd = k_pool + slot * vec_per_row;
    uint4* vd = v_pool + slot * vec_per_row;
    for (int c0 = 0; c0 < vec_per_row; c0 += 32 * kCopyUnroll) {
      uint4 kv[kCopyUnroll], vv[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < vec_per_row) {
          kv[u] = __ldcs(ks + c);
          vv[u] = __ldcs(vs + c);
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < vec_per_row) {
          kd[c] = kv[u];
          vd[c] = vv[u];
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ src,
    const int32_t* __restrict__ dst, int64_t n_vec, int64_t vec_per_block, int32_t num_blocks,
    int* err) {
  const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
  for (int64_t base = blockIdx.x * (int64_t)kCopyThreads + threadIdx.x; base < n_vec;
       base += stride * kCopyUnroll) {
    uint4 kv[kCopyUnroll], vv[kCopyUnroll];
    int64_t to[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = base + u * stride;
      to[u] = -1;
      if (i < n_vec) {
        const int64_t pair = i / vec_per_block;
        const int64_t off = i - pair * vec_per_block;
        const int32_t s = __ldg(src + pair), d = __ldg(dst + pair);
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
          record_error(err, PA_DEVERR_BLOCK_RANGE);
        } else {
          to[u] = (int64_t)d * vec_per_block + off;
          const int64_t from = (int64_t)s * vec_per_block + off;
          kv[u] = k_pool[from];
          vv[u] = v_pool[from];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      if (to[u] >= 0) {
        k_pool[to[u]] = kv[u];
        v_pool[to[u]] = vv[u];
      }
    }
  }
}

// Moves whole blocks from one pool to another (device <-> page-locked host memory,
// the host side through its device mapping): vector i is 16-byte chunk
// i % vec_per_block of pair i / vec_per_block; K and V move in the same thread.
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(
    const uint4* __restrict__ k_from, const uint4* __restrict__ v_from, uint4* __restrict__ k_to,
    uint4* __restrict__ v_to, const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
    int64_t n_vec, int64_t vec_per_block, int32_t n_from, int32_t n_to, int* err) {
  const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
  for (int64_t base = blockIdx.x * (int64_t)kCopyThreads + threadIdx.x; base < n_vec;
       base += stride * kCopyUnroll) {
    uint4 kv[kCopyUnroll], vv[kCopyUnroll];
    int64_t to[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t i = base + u * stride;
      to[u] = -1;
      if (i < n_vec) {
        const int64_t pair = i / vec_per_block;
        const int64_t off = i - pair * vec_per_block;
        const int32_t s = __ldg(src + pair), d = __ldg(dst + pair);
        if (s < 0 || s >= n_from || d < 0 || d >= n_to) {
          record_error(err, PA_DEVERR_BLOCK_RANGE);
        } else {
          to[u] = (int64_t)d * vec_per_block + off;
          const int64_t from = (int64_t)s * vec_per_block + off;
          kv[u] = __ldcs(k_from + from);
          vv[u] = __ldcs(v_from + from);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      if (to[u] >= 0) {
        __stcs(k_to + to[u], kv[u]);
        __stcs(v_to + to[u], vv[u]);
      }
    }
  }
}

int copy_grid(int64_t n_vec) {
  int sms = sm_count();  // of the current device
  if (sms <= 0) sms = 1;
  const int64_t want = (n_vec + (int64_t)kCopyThreads * kCopyUnroll - 1) /
                       ((int64_t)kCopyThreads * kCopyUnroll);
  const int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread CTAs per SM
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_slot_mapping(const int32_t* bt, int32_t num_seqs, int32_t max_blocks,
                                int32_t block_size, int32_t num_blocks, const int32_t* seq_ids,
                                const int32_t* positions, int64_t n, int64_t* slots, int* err,
                                cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  slot_mapping_kernel<<<(int)blocks, 256, 0, s>>>(bt, num_seqs, max_blocks, block_size,
                                                  num_blocks, seq_ids, positions, n, slots, err);
  return cudaGetLastError();
}

cudaError_t launch_write_kv(const void* k_new, const void* v_new, const int64_t* slots,
                            int64_t n_new, void* k_pool, void* v_pool, int64_t n_slots,
                            int64_t row_bytes, int* err, cudaStream_t s,
                            const uint8_t* skip) {
  const int64_t vec_per_row = row_bytes / 16;
  if (n_new <= 0 || vec_per_row <= 0) return cudaSuccess;
  if (vec_per_row > INT32_MAX) return cudaErrorInvalidValue;
  // one warp per row; at most 8 resident 256-thread CTAs per SM
  int sms = sm_count();
  if (sms <= 0) sms = 1;
  const int64_t want = (n_new + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  write_kv_kernel<<<grid, kCopyThreads, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, n_new,
      (int)vec_per_row, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), n_slots, skip,
      err);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int32_t* src, const int32_t* dst,
                               int32_t n_pairs, int32_t num_blocks, int64_t block_bytes, int* err,
                               cudaStream_t s) {
  const int64_t vec_per_block = block_bytes / 16;
  const int64_t n_vec = (int64_t)n_pairs * vec_per_block;
  if (n_vec == 0) return cudaSuccess;
  copy_blocks_kernel<<<copy_grid(n_vec), kCopyThreads, 0, s>>>(
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), src, dst, n_vec, vec_per_block,
      num_blocks, err);
  return cudaGetLastError();
}

cudaError_t launch_swap_blocks(const void* k_from, const void* v_from, void* k_to, void* v_to,
                               const int32_t* src, const int32_t* dst, int32_t n_pairs,
                               int32_t n_from, int32_t n_to, int64_t block_bytes, int* err,
                               cudaStream_t s) {
  const int64_t vec_per_block = block_bytes / 16;
  const int64_t n_vec = (int64_t)n_pairs * vec_per_block;
  if (n_vec == 0) return cudaSuccess;
  swap_blocks_kernel<<<copy_grid(n_vec), kCopyThreads, 0, s>>>(
      static_cast<const uint4*>(k_from), static_cast<const uint4*>(v_from),
      static_cast<uint4*>(k_to), static_cast<uint4*>(v_to), src, dst, n_vec, vec_per_block,
      n_from, n_to, err);
  return cudaGetLastError();
}

}  // namespace pa
