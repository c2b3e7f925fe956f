// pa_tc2.cu -- paged multi-token attention, two 128-row query tiles per CTA (tcgen05).
//
// Same computation as pa_tc.cu ("PagedAttention" wiki page, "mathematical
// formulation"; Pensieve summary, multi-token attention with the causal mask
// fused), for items of 129..256 packed rows: two 128-row tiles A and B of the
// same (sequence, KV head) that read the same keys. Every K/V tile that lands in
// shared memory feeds both tiles, so a FLOP costs half the K/V traffic of a
// single tile, and the two tiles form two independent chains
//     S_t(j) = Q_t K_j^T  ->  softmax_t(j)  ->  O_t += P_t(j) V_j
// that keep the tensor core busy while the other chain's softmax runs.
//
// The scores of a chain come in halves of 64 keys, each into the chain's one score
// buffer, and P goes to one of two separate P buffers: the score of the next half
// can then be computed as soon as the softmax has read the current one, while that
// softmax runs and before its P V is issued, instead of after that P V as when P is
// written over the scores. Per half h of a chain:
//     S_t(h) = Q_t K_h^T  ->  softmax_t(h)  ->  O_t += P_t(h) V_h
// with S_t(h + 1) issued once softmax_t(h) has loaded S_t(h), and P_t(h) written
// once the P V of half h - 2 (the previous user of its P buffer) is done.
//
// Warps (12, one persistent CTA per SM):
//   0        TMA producer: both tiles' Q rows once per item (single buffer);
//            K and V tiles of 128 keys gathered per block piece into two
//            2-stage rings with their own barriers, so that K_{j+2} is loaded
//            as soon as both chains have multiplied by both halves of K_j.
//   1        score issuer of both chains (operands in shared memory only).
//   2, 3     P V issuer of chain A / B (P from TMEM): each issues into its own
//            chain's accumulator only.
//   4-7      softmax of chain A, 8-11 softmax of chain B: one thread per row
//            (its TMEM lane) reads its 64 scores of a half with one TMEM load,
//            writes P to the half's P buffer as bf16 pairs and rescales O in TMEM
//            only when the running maximum grows by more than 2^8. The epilogue
//            stages O through shared memory so that every global store writes
//            whole 64-byte row pieces.
// TMEM columns of chain t: S_t at 128 t + [0, 64), its P buffers at 128 t + [64, 96)
// and 128 t + [96, 128), O_t at 256 + 128 t + [0, 128). TMEM loads/stores and
// whole-warp waits are always warp-uniform; every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"

namespace pa {
namespace {

constexpr int kKeys = 128;              // keys per tile
constexpr int kD = 128;
constexpr int kStages = 2;
constexpr int kThreads2 = 384;          // 12 warps
constexpr int kHalfKeys = 64;           // keys per score half
constexpr int kHalf = 128 * 128;        // 128 rows x 64 elements, swizzled (16 KB)
constexpr int kSoftmaxWarps = 8;
constexpr int kStageCols = 16;          // epilogue staging: 32 rows x 16 fp32 per warp
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, kHalfKeys, false);
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(128, kD, true);

__host__ __device__ constexpr uint32_t s_col(int t) { return (uint32_t)t * 128u; }
__host__ __device__ constexpr uint32_t p_col(int t, int b) {
  return (uint32_t)t * 128u + 64u + (uint32_t)b * 32u;
}
__host__ __device__ constexpr uint32_t o_col(int t) { return 256u + (uint32_t)t * 128u; }

struct Tc2Smem {
  uint8_t q[2][2][kHalf];               // [tile A/B][D half]
  uint8_t k[kStages][2][kHalf];         // [stage][D half], rows = keys
  uint8_t v[kStages][2][kHalf];
  float stage[kSoftmaxWarps][32 * kStageCols];
  int bt_cache[2][kBtCache];
  Item info[3];                         // item k and its lengths, by k % 3 (written by the
  int info_L[3], info_ql[3];            // producer before item k's Q load, published by
  uint64_t info_full[3];                // info_full[k % 3])
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t q_full, q_free;
  uint64_t s_full[2], s_free[2];        // [chain]: score of a half done / read by the softmax
  uint64_t p_full[2][2];                // [chain][P buffer]: P of a half written
  uint64_t o_done[2][2];                // [chain][P buffer]: the P V that read it is done
  uint64_t o_free[2];                   // [chain]: the epilogue read O
  uint64_t drain[3];
  uint32_t tmem_base;
  int k_issued[kStages], k_consumed[kStages];
  int v_issued[kStages], v_consumed[kStages];
  int q_issued, q_consumed;
  int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t ph(int n, int ring) { return (uint32_t)(n / ring) & 1u; }

__device__ __forceinline__ int tiles_of(const Item& x) {
  return (x.kv_end - x.kv_begin + kKeys - 1) / kKeys;
}

// The work items of a CTA: items c + i G, i < cnt (c = blockIdx.x, G = gridDim.x), a
// round-robin walk of the longest-first list. CTAs then work on items of similar
// length at the same time, and the row tiles of one (sequence, KV head) -- which read
// the same keys -- sit next to each other in that list: their K/V reads meet in L2.
struct ItemWalk {
  int c, G, cnt;
  __device__ __forceinline__ int at(int s) const { return c + s * G; }
};

__device__ __forceinline__ ItemWalk item_walk(int n_items) {
  ItemWalk w;
  w.c = blockIdx.x;
  w.G = gridDim.x;
  w.cnt = w.c < n_items ? (n_items - w.c + w.G - 1) / w.G : 0;
  return w;
}

template <bool kSW>
__global__ void __launch_bounds__(kThreads2, 1)
    tc2_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ CUtensorMap omap, const Item* __restrict__ items,
               int n_items, int box_t) {
  extern __shared__ uint8_t smem_raw[];
  Tc2Smem& sm = *reinterpret_cast<Tc2Smem*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ItemWalk W = item_walk(n_items);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);    // the score issuer, after both chains' last half
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 2);    // both chains' P V issuers
      sm.k_issued[s] = sm.k_consumed[s] = 0;
      sm.v_issued[s] = sm.v_consumed[s] = 0;
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_free, 1);          // the score issuer, after the item's last score
    for (int i = 0; i < 3; ++i) mbar_init(&sm.info_full[i], 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.s_free[t], 128);
      for (int b = 0; b < 2; ++b) {
        mbar_init(&sm.p_full[t][b], 128);
        mbar_init(&sm.o_done[t][b], 1);
      }
      mbar_init(&sm.o_free[t], 128);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&sm.drain[i], 1);
    sm.q_issued = 0;
    sm.q_consumed = 0;
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      prefetch_tensormap(&qmap);
    }
    const int pieces = kKeys / box_t;
    const uint32_t piece_bytes = (uint32_t)box_t * 128u;
    int n = 0, k = 0;
    bool ok = true;
    int nb[kBtPerLane];
    Item item_next{};
    if (W.cnt > 0) {
      const Item f = items[W.at(0)];
      bt_prefetch(a.block_table + (int64_t)f.seq * a.max_blocks, a.max_blocks,
                  bt_window(f.kv_begin, f.kv_end, a.block_size), lane, nb);
      bt_store(sm.bt_cache[0], nb, lane);
      if (W.cnt > 1) item_next = items[W.at(1)];
    }
    __syncwarp();
    for (int sidx = 0; sidx < W.cnt && ok; ++sidx, ++k) {
      const Item item = items[W.at(sidx)];
      const BtWindow win = bt_window(item.kv_begin, item.kv_end, a.block_size);
      const int* cache = sm.bt_cache[k & 1];
      const bool has_next = sidx + 1 < W.cnt;
      Item item_after{};
      if (has_next) {
        bt_prefetch(a.block_table + (int64_t)item_next.seq * a.max_blocks, a.max_blocks,
                    bt_window(item_next.kv_begin, item_next.kv_end, a.block_size), lane, nb);
        if (sidx + 2 < W.cnt) item_after = items[W.at(sidx + 2)];
      }
      // both tiles' Q rows. The buffer is free once both chains issued the item's last
      // S: q_free then completed phase k - 1. It cannot be further ahead, since phase k
      // needs the Q load below.
      if (k > 0) {
        ok = mbar_wait_warp(&sm.q_free, (uint32_t)(k - 1) & 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
      }
      if (lane == 0) {
        // the item's description for the softmax warps (the arrive releases the writes)
        sm.info[k % 3] = item;
        sm.info_L[k % 3] = __ldg(a.context_lens + item.seq);
        sm.info_ql[k % 3] = __ldg(a.query_lens + item.seq);
        mbar_arrive(&sm.info_full[k % 3]);
        mbar_arrive_expect_tx(&sm.q_full, 4u * kHalf);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int tok = item.q_row0 + (item.row_begin + 128 * t) / a.g;
          tma_load_3d(&sm.q[t][0][0], &qmap, &sm.q_full, 0, item.kv_head * a.g, tok);
          tma_load_3d(&sm.q[t][1][0], &qmap, &sm.q_full, 64, item.kv_head * a.g, tok);
        }
        sm.q_issued += 1;
      }
      __syncwarp();
      const int32_t* bt = a.block_table + (int64_t)item.seq * a.max_blocks;
      for (int t0 = item.kv_begin; t0 < item.kv_end; t0 += kKeys, ++n) {
        const int st = n % kStages;
        bool valid = false;
        int tok = 0;
        if (lane < pieces) {
          const int j0 = t0 + lane * box_t;
          if (j0 < item.kv_end) {
            const int lb = j0 / a.block_size;
            const int phys = bt_lookup(cache, win, bt, a.max_blocks, lb);
            if (phys == -2) {
              record_error(a.err, PA_DEVERR_TABLE_RANGE);
            } else if (phys < 0 || phys >= a.num_blocks) {
              record_error(a.err, PA_DEVERR_BLOCK_RANGE);
            } else {
              valid = true;
              tok = phys * a.block_size + (j0 - lb * a.block_size);
            }
          }
        }
        const uint32_t tile_bytes = __popc(__ballot_sync(0xffffffffu, valid)) * piece_bytes * 2u;
        const uint32_t row_off = (uint32_t)lane * box_t * 128u;
        // K_n: its stage is free once both chains' S of tile n - 2 completed
        ok = mbar_wait_warp(&sm.k_empty[st], ph(n, kStages) ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&sm.k_full[st], tile_bytes);
        __syncwarp();
        if (valid) {
          tma_load_3d(&sm.k[st][0][row_off], &kmap, &sm.k_full[st], 0, item.kv_head, tok);
          tma_load_3d(&sm.k[st][1][row_off], &kmap, &sm.k_full[st], 64, item.kv_head, tok);
        }
        if (lane == 0) sm.k_issued[st] += 1;
        // V_n: free once both chains' P V of tile n - 2 completed
        ok = mbar_wait_warp(&sm.v_empty[st], ph(n, kStages) ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&sm.v_full[st], tile_bytes);
        __syncwarp();
        if (valid) {
          tma_load_3d(&sm.v[st][0][row_off], &vmap, &sm.v_full[st], 0, item.kv_head, tok);
          tma_load_3d(&sm.v[st][1][row_off], &vmap, &sm.v_full[st], 64, item.kv_head, tok);
        }
        if (lane == 0) sm.v_issued[st] += 1;
      }
      if (has_next) {
        bt_store(sm.bt_cache[(k + 1) & 1], nb, lane);
        item_next = item_after;
      }
      __syncwarp();
    }
    if (!ok) sm.abort_flag = 1;
  } else if (warp == 1) {
    // ------------------------------------------------------------ score issuer
    // Per half h (two per K tile, counted over the CTA's items) and chain t: once
    // softmax t has loaded S_t(h - 1) (s_free), S_t(h) = Q_t K_h^T into the chain's score
    // buffer. Both operands are in shared memory.
    // Phase bounds: s_free[t](h) needs s_full[t](h), committed here after the wait for
    // s_free[t](h - 1); k_full of tile n + 2 needs k_empty of tile n and q_full of item
    // k + 1 needs q_free of item k, both committed here after this thread's waits.
    if (lane == 0) {
      bool ok = true;
      int n = 0, h = 0;                           // tile, half of the CTA
      for (int sidx = 0; sidx < W.cnt && ok; ++sidx) {
        const Item it = items[W.at(sidx)];
        const int nt = tiles_of(it);
        if (!mbar_wait(&sm.q_full, (uint32_t)sidx & 1u, a.err, wait_bound<kSW>(a))) { ok = false; break; }
        sm.q_consumed += 1;
        for (int j = 0; j < nt && ok; ++j, ++n) {
          const int st = n % kStages;
          if (!mbar_wait(&sm.k_full[st], ph(n, kStages), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          sm.k_consumed[st] += 1;
          const uint64_t kd0 = tc::smem_desc_sw128(smem_addr(&sm.k[st][0][0]), 16, 1024);
          for (int hk = 0; hk < 2 && ok; ++hk, ++h) {
            // keys 64 hk .. 64 hk + 63 of the tile: rows 64 hk .. of both D halves
            const uint64_t kd = kd0 + (uint64_t)((hk * kHalfKeys * 128) >> 4);
            for (int t = 0; t < 2; ++t) {
              if (h > 0 &&
                  !mbar_wait(&sm.s_free[t], (uint32_t)(h - 1) & 1u, a.err, wait_bound<kSW>(a))) {
                ok = false;
                break;
              }
              tc::fence_after_sync();
              // 8 steps of 16 dims; step kk starts (kk / 4) D halves and (kk % 4) 32-byte
              // chunks into both operands
              const uint64_t qd = tc::smem_desc_sw128(smem_addr(&sm.q[t][0][0]), 16, 1024);
              tc::mma_bf16_c<false>(tmem + s_col(t), qd, kd, kIdescS);
#pragma unroll
              for (int kk = 1; kk < kD / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
                tc::mma_bf16_c<true>(tmem + s_col(t), qd + off, kd + off, kIdescS);
              }
              tc::commit(&sm.s_full[t]);
            }
          }
          if (!ok) break;
          tc::commit(&sm.k_empty[st]);
          if (j + 1 == nt) tc::commit(&sm.q_free);  // the item's last score
        }
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain[0]);
      mbar_wait(&sm.drain[0], 0, a.err);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ P V issuer of chain t
    // Per half h: O_t += P_t(h) V_h once softmax t wrote P_t(h) into P buffer h % 2;
    // P from TMEM, V from shared memory. This thread issues into O_t only.
    // Phase bounds: p_full[t][b] of the next use of buffer b needs o_done[t][b] of this
    // use, committed here after the wait for this use; v_full of tile n + 2 needs
    // v_empty of tile n from both chains' issuers; o_free[t] of item k + 1 needs the
    // first P V of item k + 1.
    const int t = warp - 2;
    if (lane == 0) {
      bool ok = true;
      int n = 0, h = 0;                           // tile, half of the CTA
      for (int sidx = 0; sidx < W.cnt && ok; ++sidx) {
        const Item it = items[W.at(sidx)];
        const int nt = tiles_of(it);
        for (int j = 0; j < nt && ok; ++j, ++n) {
          const int st = n % kStages;
          if (!mbar_wait(&sm.v_full[st], ph(n, kStages), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          if (t == 0) sm.v_consumed[st] += 1;
          // Keys of the tile in the item's range, rounded up to the 16-key step of P V:
          // only those V rows are read. At the item's last tile the rows between the
          // range's end and that step hold whatever the block tail holds: zero them (at
          // most 15 rows) so that 0 * (non-finite) never reaches O. Both chains write
          // the same zeros, each before its own P V.
          const int key0 = it.kv_begin + j * kKeys;
          const int valid = min(kKeys, it.kv_end - key0);
          const int kk_end = (valid + 15) >> 4;
          if (valid < kk_end * 16) {
            for (int r = valid; r < kk_end * 16; ++r) {
              uint4* v0 = reinterpret_cast<uint4*>(&sm.v[st][0][r * 128]);
              uint4* v1 = reinterpret_cast<uint4*>(&sm.v[st][1][r * 128]);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                v0[q] = make_uint4(0, 0, 0, 0);
                v1[q] = make_uint4(0, 0, 0, 0);
              }
            }
            tc::fence_async_shared();
          }
          // at an item's first tile, O_t must have been read out by the previous item's
          // epilogue
          if (j == 0 &&
              !mbar_wait(&sm.o_free[t], ((uint32_t)sidx & 1u) ^ 1u, a.err, wait_bound<kSW>(a))) {
            ok = false;
            break;
          }
          // V as the MN-major B operand: step kk covers keys 16 kk .. 16 kk + 15 (rows
          // of 128 bytes), the two D halves are kHalf apart
          const uint64_t vd = tc::smem_desc_sw128(smem_addr(&sm.v[st][0][0]), kHalf, 1024);
          for (int hk = 0; hk < 2 && ok; ++hk, ++h) {
            const int b = h & 1;
            if (!mbar_wait(&sm.p_full[t][b], (uint32_t)(h >> 1) & 1u, a.err, wait_bound<kSW>(a))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
              const int kk = 4 * hk + kq;           // 16-key step of the tile
              const uint32_t pa = tmem + p_col(t, b) + (uint32_t)kq * 8u;
              const uint64_t vk = vd + (uint64_t)((kk * 16 * 128) >> 4);
              if (kk == 0) {
                if (j > 0)
                  tc::mma_bf16_ts_c<true>(tmem + o_col(t), pa, vk, kIdescO);
                else
                  tc::mma_bf16_ts_c<false>(tmem + o_col(t), pa, vk, kIdescO);
              } else if (kk < kk_end) {
                tc::mma_bf16_ts_c<true>(tmem + o_col(t), pa, vk, kIdescO);
              }
            }
            tc::commit(&sm.o_done[t][b]);
          }
          if (!ok) break;
          tc::commit(&sm.v_empty[st]);
        }
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain[1 + t]);
      mbar_wait(&sm.drain[1 + t], 0, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax of chain t
    // One thread per row (its TMEM lane): the 64 scores of a half are read from TMEM
    // with one load, so no other thread needs the row's maximum or sum. The score
    // buffer is released right after that load; P goes to the half's P buffer.
    // Phase bounds: s_full[t](h + 1) needs s_free[t](h), on which these threads arrive
    // after their wait for s_full[t](h); o_done[t][b] of the next use of buffer b needs
    // p_full[t][b] of that use, written here after the wait for this use; v_full of tile
    // n + 2 needs this chain's P V of tile n. So no barrier is ever two phases ahead of
    // a wait here.
    const int t = (warp - 4) >> 2;                // 0 = tile A (warps 4-7), 1 = tile B
    const int quad = warp & 3;
    const int row = quad * 32 + lane;             // row within the tile = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    float* stg = sm.stage[warp - 4];
    int h = 0;                                    // half of the CTA
    bool ok = true;
    for (int sidx = 0, k = 0; sidx < W.cnt && ok; ++sidx, ++k) {
      // The producer published the item's description in slot k % 3 before its Q load.
      // The slot (and its barrier's next phase) is rewritten for item k + 3 only after
      // every score of item k + 2, and the first of those needs this chain's load of
      // item k + 1's last score: the slot stays valid through this item's epilogue, and
      // the barrier is never two phases ahead of this wait.
      if (!mbar_wait_warp(&sm.info_full[k % 3], ph(k, 3), a.err, wait_bound<kSW>(a))) { ok = false; break; }
      const Item& info = sm.info[k % 3];
      const int kv_begin = info.kv_begin, kv_end = info.kv_end, row_count = info.row_count;
      int lim = -1;                               // causal limit of this row (-1: not a row)
      {
        const int L = sm.info_L[k % 3], ql = sm.info_ql[k % 3];
        if (kv_end > L || info.row_begin + row_count > ql * a.g)
          record_error(a.err, PA_DEVERR_LENS);
        if (t * 128 + row < row_count)
          lim = min(kv_end - 1, L - ql + (info.row_begin + t * 128 + row) / a.g);
      }
      const int nt = (kv_end - kv_begin + kKeys - 1) / kKeys;
      const int trow = t * 128 + row;             // row within the item
      const bool warp_live = t * 128 + quad * 32 < row_count;
      float m_used = -INFINITY, l = 0.f;
      for (int hs = 0; hs < 2 * nt; ++hs, ++h) {
        const int b = h & 1;
        if (!mbar_wait_warp(&sm.s_full[t], (uint32_t)h & 1u, a.err, wait_bound<kSW>(a))) { ok = false; break; }
        tc::fence_after_sync();
        const int key0 = kv_begin + hs * kHalfKeys;
        float s[kHalfKeys];
        if (warp_live) tc::tmem_ld64(t_lane + s_col(t), s);
        // the score buffer may take the next half's score
        tc::fence_before_sync();
        mbar_arrive(&sm.s_free[t]);
        float pk[4][8];                           // P as bf16 pairs, 8 columns per 16 keys
        if (warp_live) {
          if (key0 + kHalfKeys - 1 > lim) {
#pragma unroll
            for (int i = 0; i < kHalfKeys; ++i)
              if (key0 + i > lim) s[i] = -INFINITY;
          }
          // running maximum of the raw scores (the scale is positive)
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < kHalfKeys / 2; ++i) m4[i & 3] = fmax3(m4[i & 3], s[2 * i], s[2 * i + 1]);
          const float m_new =
              fmaxf(m_used, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2);
          if (m_used == -INFINITY) m_used = m_new;
          // O_t is rescaled by 2^(m_used - m_new) only when the maximum grew by more
          // than 2^8; otherwise P keeps the older (smaller) maximum as its reference.
          const bool need = m_new > m_used + kRescaleLog2;
          const bool warp_rescale = __any_sync(0xffffffffu, need);
          const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
          if (need) {
            l *= alpha;
            m_used = m_new;
          }
          if (warp_rescale) {
            // O_t must be idle: the P V of half h - 1 (of this item: the first half of an
            // item never rescales) is done. tcgen05.ld / st are warp-collective, so the
            // warp rescales together (factor 1 for rows that need none).
            if (!mbar_wait_warp(&sm.o_done[t][(h - 1) & 1], (uint32_t)((h - 1) >> 1) & 1u, a.err,
                                wait_bound<kSW>(a))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
#pragma unroll 1
            for (int c8 = 0; c8 < kD / 16; ++c8) {
              float o[16];
              const uint32_t addr = t_lane + o_col(t) + (uint32_t)c8 * 16u;
              tc::tmem_ld16(addr, o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= alpha;
              tc::tmem_st16(addr, o);
            }
          }
          // P = 2^(scale * s - m) as bf16 pairs: keys 16 c .. 16 c + 15 go to columns
          // 8 c .. 8 c + 7 of the P buffer; a masked score is -inf and gives exactly 0
          const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
          const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
          const uint64_t nm2 = f2_pack(neg_m, neg_m);
          uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2) {
              const int i = c * 8 + i2;
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sc2, nm2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
              pk[c][i2] = __uint_as_float(pack_bf16(p0, p1));
            }
          }
          float sa, sb;
          f2_unpack(f2_add(sum2[0], sum2[1]), sa, sb);
          l += sa + sb;
        } else {
          // rows past the item: zero P, so that no stale bits reach the tensor core
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2) pk[c][i2] = 0.f;
        }
        // the P buffer is free once the P V of half h - 2 is done
        if (!mbar_wait_warp(&sm.o_done[t][b], ((uint32_t)(h >> 1) & 1u) ^ 1u, a.err, wait_bound<kSW>(a))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        __syncwarp();  // tcgen05.st is .sync.aligned: reconverge after the per-row work
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_st8(t_lane + p_col(t, b) + (uint32_t)c * 8u, pk[c]);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        mbar_arrive(&sm.p_full[t][b]);
      }
      if (!ok) break;
      // ---- epilogue: the chain's last P V (o_done of its buffer is at most one phase
      // ahead: the next use of that buffer needs this chain's P of the next item)
      if (!mbar_wait_warp(&sm.o_done[t][(h - 1) & 1], (uint32_t)((h - 1) >> 1) & 1u, a.err,
                          wait_bound<kSW>(a))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // A warp whose 32 rows all belong to the item (and go to the output, not to
      // split partials) hands O / l to the TMA: it writes 16-column pieces of its rows
      // into its staging buffer in the output box's layout (packed row-major, which is
      // tokens x heads x columns) and one lane issues an asynchronous tensor store, so
      // the warp moves on while the bytes drain. Other warps store rows themselves.
      const int rho0 = info.row_begin + t * 128 + quad * 32;
      const bool whole = info.part < 0 && t * 128 + quad * 32 + 32 <= row_count;
      if (whole) {
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const int c1 = info.kv_head * a.g + rho0 % a.g;
        const int c2 = info.q_row0 + rho0 / a.g;
#pragma unroll 1
        for (int c4 = 0; c4 < kD / 32; ++c4) {
          float o[32];
          __syncwarp();  // tcgen05.ld is .sync.aligned: reconverge after the single-lane store
          tc::tmem_ld32(t_lane + o_col(t) + (uint32_t)c4 * 32u, o);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // the previous store has read the staging buffer
            if (lane == 0) bulk_wait_read();
            __syncwarp();
            // rows of 16 columns swizzled as the tensor map says (fp32: 16-byte chunk c
            // of row r at c ^ ((r / 2) % 4); bf16: at c ^ ((r / 4) % 2)): the eight
            // lanes of each quarter-warp write to distinct banks
            if (a.out_bf16) {
              uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(stg) + lane * 32);
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                uint4 w;
                w.x = pack_bf16(o[hh * 16 + 8 * i + 0] * inv, o[hh * 16 + 8 * i + 1] * inv);
                w.y = pack_bf16(o[hh * 16 + 8 * i + 2] * inv, o[hh * 16 + 8 * i + 3] * inv);
                w.z = pack_bf16(o[hh * 16 + 8 * i + 4] * inv, o[hh * 16 + 8 * i + 5] * inv);
                w.w = pack_bf16(o[hh * 16 + 8 * i + 6] * inv, o[hh * 16 + 8 * i + 7] * inv);
                d[i ^ ((lane >> 2) & 1)] = w;
              }
            } else {
              float4* d = reinterpret_cast<float4*>(stg + lane * kStageCols);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d[i ^ ((lane >> 1) & 3)] =
                    make_float4(o[hh * 16 + 4 * i] * inv, o[hh * 16 + 4 * i + 1] * inv,
                                o[hh * 16 + 4 * i + 2] * inv, o[hh * 16 + 4 * i + 3] * inv);
            }
            tc::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&omap, stg, c4 * 32 + hh * 16, c1, c2);
              bulk_commit();
            }
          }
        }
      } else if (warp_live) {
        // destination of this lane's row (nullptr: not a row of the item)
        char* dst_row = nullptr;
        float inv = 1.f;
        const int part = info.part;
        if (trow < row_count) {
          if (part < 0) {
            inv = (l > 0.f) ? 1.f / l : 0.f;
            const int rho = info.row_begin + trow;
            const int qt = rho / a.g;
            const int h = info.kv_head * a.g + (rho - qt * a.g);
            const int64_t off = ((int64_t)(info.q_row0 + qt) * a.Hq + h) * kD;
            dst_row = reinterpret_cast<char*>(a.out) + off * (a.out_bf16 ? 2 : 4);
          } else {
            const int64_t prow = (int64_t)part + trow;
            dst_row = reinterpret_cast<char*>(a.part_acc + prow * kD);
            a.part_ml[prow * 2 + 0] = m_used;
            a.part_ml[prow * 2 + 1] = l;
          }
        }
        const bool bf = a.out_bf16 && part < 0;
        // the staging buffer may still feed an earlier tensor store of this warp
        if (lane == 0) bulk_wait_read();
        __syncwarp();
#pragma unroll 1
        for (int c4 = 0; c4 < kD / 32; ++c4) {
          float o[32];
          tc::tmem_ld32(t_lane + o_col(t) + (uint32_t)c4 * 32u, o);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // this lane's 16 values -> staging row `lane`; 16-byte chunk cj sits at
            // position cj ^ ((row / 2) % 4), which keeps both the row-wise writes and
            // the column-wise reads below free of bank conflicts
#pragma unroll
            for (int cj = 0; cj < 4; ++cj) {
              const int pos = cj ^ ((lane >> 1) & 3);
              reinterpret_cast<float4*>(stg + lane * kStageCols)[pos] =
                  make_float4(o[hh * 16 + 4 * cj] * inv, o[hh * 16 + 4 * cj + 1] * inv,
                              o[hh * 16 + 4 * cj + 2] * inv, o[hh * 16 + 4 * cj + 3] * inv);
            }
            __syncwarp();
            // 8 rows x 64 bytes per store instruction: lane -> row 8 qq + lane / 4,
            // 16-byte chunk lane % 4
            const int col0 = c4 * 32 + hh * 16 + (lane & 3) * 4;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const int r = qq * 8 + (lane >> 2);
              char* d = reinterpret_cast<char*>(__shfl_sync(
                  0xffffffffu, reinterpret_cast<unsigned long long>(dst_row), r));
              const float4 v = reinterpret_cast<const float4*>(
                  stg + r * kStageCols)[(lane & 3) ^ ((r >> 1) & 3)];
              if (d) {
                if (bf) {
                  uint2 w;
                  w.x = pack_bf16(v.x, v.y);
                  w.y = pack_bf16(v.z, v.w);
                  *reinterpret_cast<uint2*>(d + col0 * 2) = w;
                } else {
                  *reinterpret_cast<float4*>(d + col0 * 4) = v;
                }
              }
            }
            __syncwarp();
          }
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&sm.o_free[t]);
    }
    // every tensor store of this warp has landed before the CTA exits
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (!ok) sm.abort_flag = 1;
  }
  tc::fence_before_sync();
  __syncthreads();
  // After an abort, give copies still in flight a bounded time to land.
  if (sm.abort_flag && threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    for (int s = 0; s < kStages; ++s) {
      if (sm.k_issued[s] > sm.k_consumed[s]) {
        const uint32_t parity = (uint32_t)(sm.k_issued[s] - 1) & 1u;
        while (!mbar_try_wait(smem_addr(&sm.k_full[s]), parity))
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
      if (sm.v_issued[s] > sm.v_consumed[s]) {
        const uint32_t parity = (uint32_t)(sm.v_issued[s] - 1) & 1u;
        while (!mbar_try_wait(smem_addr(&sm.v_full[s]), parity))
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
    if (sm.q_issued > sm.q_consumed) {
      const uint32_t parity = (uint32_t)(sm.q_issued - 1) & 1u;
      while (!mbar_try_wait(smem_addr(&sm.q_full), parity))
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  pdl_wait();  // exit only after the kernel this one may overlap has completed
}

}  // namespace

int tc2_smem_bytes() { return (int)sizeof(Tc2Smem) + 1024; }

cudaError_t launch_tc2(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const CUtensorMap& qmap, const CUtensorMap& omap, const Item* items,
                       int32_t n_items, int box_t, int grid, cudaStream_t s, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  const int smem = tc2_smem_bytes();
  auto* k = a.wait_ns == kWaitLimitNsHost ? tc2_kernel<false> : tc2_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_kernel(k, grid, kThreads2, smem, s, pdl, a, kmap, vmap, qmap, omap, items,
                    n_items, box_t);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
