// pa_tc3.cu -- paged multi-token attention on tcgen05, one 128-row query tile per item,
// three TMEM score buffers.
//
// Same computation as pa_tc.cu and pa_tc2.cu ("PagedAttention" wiki page, "mathematical
// formulation"; Pensieve summary, multi-token attention with the causal mask fused): for
// an item of at most 128 packed rows (query tokens x the query heads of one KV head), the
// two matrix products S = Q K^T and O += P V per 128-key tile, with an online softmax
// between them and the causal limit applied to the scores, over a context reached
// through the block table.
//
// Why a third kernel: in the one-tile and two-tile kernels the score of tile n + 2 (or
// n + 1) goes into the TMEM columns whose P the P V of tile n still reads, so a query
// tile's chain score -> softmax -> P V -> next score is serial, and measured, about 4,300
// cycles per tile against 1,024 of tensor work. Here the softmax keeps one running
// maximum per row (one thread per row reads its whole 128-key score row, as in the
// two-tile kernel), so one O accumulator suffices, and the TMEM holds three score
// buffers beside it: the score of tile n + 3 waits only for the P V of tile n, while the
// softmax works on tiles n + 1 and n + 2. The softmax then runs back to back, and the
// tensor core interleaves the products of three tiles.
//
// Warps (7, one persistent CTA per SM):
//   0     TMA producer: the item's 128 Q rows (one buffer, loaded once every score of the
//         previous item is done), K tiles into a 2-stage ring, V tiles into a 3-stage
//         ring, each gathered per block piece through the block table.
//   1     score issuer: S_n = Q K_n^T (M = N = 128) into buffer n % 3 once the P V of
//         tile n - 3 has released it.
//   2     P V issuer: O += P_n V_n per key half as soon as that half of P_n is written.
//   3-6   softmax: warp w owns TMEM lane quadrant w % 4 (32 rows), one thread per row;
//         P goes back over the scores as bf16 pairs; O is rescaled in TMEM only when a
//         row's maximum grows by more than 2^8 (after the previous P V is done); the
//         epilogue stages O / l through shared memory for TMA stores.
// TMEM: score buffers [0, 128), [128, 256), [256, 384); O [384, 512). Every TMEM load or
// store is issued by a warp on its own lane quadrant (warp % 4) under a warp-uniform
// condition, after reconvergence; every wait is bounded.
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

constexpr int kRows = kTcRows;          // 128 rows per tile (M)
constexpr int kKeys = 128;              // keys per tile
constexpr int kD = 128;
constexpr int kSBuf = 3;                // TMEM score buffers
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr int kThreads3 = 224;          // 7 warps
constexpr int kHalf = 128 * 128;        // 128 rows x 64 elements, swizzled (16 KB)
constexpr int kSoftmaxWarps = 4;
constexpr int kStageCols = 16;          // epilogue staging: 32 rows x 16 fp32 per warp
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 384;

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kKeys, false);  // Q K^T, both K-major
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD, true);      // P V, V MN-major

__host__ __device__ constexpr uint32_t s_col(int b) { return (uint32_t)b * 128u; }

struct Tc3Smem {
  uint8_t q[2][kHalf];                  // [D half], 128 rows
  uint8_t k[kKStages][2][kHalf];        // [stage][D half], rows = keys
  uint8_t v[kVStages][2][kHalf];
  float stage[kSoftmaxWarps][32 * kStageCols];
  int bt_cache[2][kBtCache];            // block ids of the producer, by item parity
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t q_full, q_free;
  uint64_t s_full[kSBuf], s_free[kSBuf];
  uint64_t p_full[kSBuf][2];            // [score buffer][key half]: that half of P written
  uint64_t o_done[2];                   // [tile parity]: the P V of that tile is done
  uint64_t o_free;                      // the epilogue has read O
  uint64_t drain[2];
  uint32_t tmem_base;
  int k_issued[kKStages], k_consumed[kKStages];
  int v_issued[kVStages], v_consumed[kVStages];
  int q_issued, q_consumed;
  int abort_flag;
};
static_assert(sizeof(Tc3Smem) + 1024 <= 227 * 1024, "shared memory of the three-buffer kernel");

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

template <bool kSW>
__global__ void __launch_bounds__(kThreads3, 1)
    tc3_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ CUtensorMap omap, const Item* __restrict__ items,
               int n_items, int box_t) {
  extern __shared__ uint8_t smem_raw[];
  Tc3Smem& sm = *reinterpret_cast<Tc3Smem*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      sm.k_issued[s] = sm.k_consumed[s] = 0;
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
      sm.v_issued[s] = sm.v_consumed[s] = 0;
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_free, 1);
    for (int b = 0; b < kSBuf; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 1);
      mbar_init(&sm.p_full[b][0], kSoftmaxWarps * 32);
      mbar_init(&sm.p_full[b][1], kSoftmaxWarps * 32);
    }
    mbar_init(&sm.o_done[0], 1);
    mbar_init(&sm.o_done[1], 1);
    mbar_init(&sm.o_free, kSoftmaxWarps * 32);
    mbar_init(&sm.drain[0], 1);
    mbar_init(&sm.drain[1], 1);
    sm.q_issued = sm.q_consumed = 0;
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
    // Phase bounds: q_free of item k needs the item's last score, which needs its Q
    // load (q_full) from here; k_empty of tile n + kKStages needs the score of tile n,
    // v_empty of tile n + kVStages the P V of tile n, which need this warp's loads of
    // tile n. So no barrier is ever two phases ahead of a wait here.
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      prefetch_tensormap(&qmap);
    }
    const int pieces = kKeys / box_t;                     // <= 16
    const uint32_t piece_bytes = (uint32_t)box_t * 128u;  // one D half of one piece
    int n = 0, k = 0;
    bool ok = true;
    int nb[kBtPerLane];
    Item item_next{};
    if ((int)blockIdx.x < n_items) {
      const Item f = items[blockIdx.x];
      bt_prefetch(a.block_table + (int64_t)f.seq * a.max_blocks, a.max_blocks,
                  bt_window(f.kv_begin, f.kv_end, a.block_size), lane, nb);
      bt_store(sm.bt_cache[0], nb, lane);
      if ((int)blockIdx.x + G < n_items) item_next = items[blockIdx.x + G];
    }
    __syncwarp();
    for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
      const Item item = items[it];
      const BtWindow win = bt_window(item.kv_begin, item.kv_end, a.block_size);
      const int* cache = sm.bt_cache[k & 1];
      const bool has_next = it + G < n_items;
      Item item_after{};
      if (has_next) {
        bt_prefetch(a.block_table + (int64_t)item_next.seq * a.max_blocks, a.max_blocks,
                    bt_window(item_next.kv_begin, item_next.kv_end, a.block_size), lane, nb);
        if (it + 2 * G < n_items) item_after = items[it + 2 * G];
      }
      // the item's 128 Q rows once every score of the previous item is done
      if (k > 0) {
        ok = mbar_wait_warp(&sm.q_free, (uint32_t)(k - 1) & 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full, 2u * kHalf);
        const int tok = item.q_row0 + item.row_begin / a.g;
        tma_load_3d(&sm.q[0][0], &qmap, &sm.q_full, 0, item.kv_head * a.g, tok);
        tma_load_3d(&sm.q[1][0], &qmap, &sm.q_full, 64, item.kv_head * a.g, tok);
        sm.q_issued += 1;
      }
      __syncwarp();
      const int32_t* bt = a.block_table + (int64_t)item.seq * a.max_blocks;
      for (int t0 = item.kv_begin; t0 < item.kv_end; t0 += kKeys, ++n) {
        const int sk = n % kKStages, sv = n % kVStages;
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
        // K_n: its stage is free once the score of tile n - kKStages is done
        ok = mbar_wait_warp(&sm.k_empty[sk], ph(n, kKStages) ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&sm.k_full[sk], tile_bytes);
        __syncwarp();
        if (valid) {
          tma_load_3d(&sm.k[sk][0][row_off], &kmap, &sm.k_full[sk], 0, item.kv_head, tok);
          tma_load_3d(&sm.k[sk][1][row_off], &kmap, &sm.k_full[sk], 64, item.kv_head, tok);
        }
        if (lane == 0) sm.k_issued[sk] += 1;
        // V_n: its stage is free once the P V of tile n - kVStages is done
        ok = mbar_wait_warp(&sm.v_empty[sv], ph(n, kVStages) ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&sm.v_full[sv], tile_bytes);
        __syncwarp();
        if (valid) {
          tma_load_3d(&sm.v[sv][0][row_off], &vmap, &sm.v_full[sv], 0, item.kv_head, tok);
          tma_load_3d(&sm.v[sv][1][row_off], &vmap, &sm.v_full[sv], 64, item.kv_head, tok);
        }
        if (lane == 0) sm.v_issued[sv] += 1;
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
    // Phase bounds: q_full of item k + 1 needs q_free(k), committed here; k_full of tile
    // n + kKStages needs k_empty(n), committed here; s_free[b] of tile n + 3 needs the
    // P V of tile n + 3, which needs s_full(n + 3) from here.
    if (lane == 0) {
      int n = 0, k = 0;
      bool ok = true;
      int nt_next = (int)blockIdx.x < n_items ? tiles_of(items[blockIdx.x]) : 0;
      for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
        const int nt = nt_next;
        if (it + G < n_items) nt_next = tiles_of(items[it + G]);
        if (!mbar_wait(&sm.q_full, (uint32_t)k & 1u, a.err, wait_bound<kSW>(a))) { ok = false; break; }
        sm.q_consumed += 1;
        tc::fence_after_sync();
        const uint64_t qd = tc::smem_desc_sw128(smem_addr(&sm.q[0][0]), 16, 1024);
        for (int j = 0; j < nt; ++j, ++n) {
          const int sk = n % kKStages, b = n % kSBuf;
          if (!mbar_wait(&sm.k_full[sk], ph(n, kKStages), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          sm.k_consumed[sk] += 1;
          // buffer b's last reader, the P V of tile n - 3, is done
          if (!mbar_wait(&sm.s_free[b], ph(n, kSBuf) ^ 1u, a.err, wait_bound<kSW>(a))) { ok = false; break; }
          tc::fence_after_sync();
          // S = Q K^T: 8 steps of 16 dims; step kk starts (kk / 4) D halves and
          // (kk % 4) 32-byte chunks into both operands
          const uint64_t kd = tc::smem_desc_sw128(smem_addr(&sm.k[sk][0][0]), 16, 1024);
          tc::mma_bf16_c<false>(tmem + s_col(b), qd, kd, kIdescS);
#pragma unroll
          for (int kk = 1; kk < kD / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
            tc::mma_bf16_c<true>(tmem + s_col(b), qd + off, kd + off, kIdescS);
          }
          tc::commit(&sm.s_full[b]);
          tc::commit(&sm.k_empty[sk]);
        }
        if (ok) tc::commit(&sm.q_free);  // the item's last score issued: Q may be reloaded
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain[0]);
      mbar_wait(&sm.drain[0], 0, a.err);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ P V issuer
    // Phase bounds: p_full[b][h] of tile n + 3 needs s_full(n + 3), which needs s_free
    // from the P V of tile n, committed here; v_full of tile n + kVStages needs v_empty(n),
    // committed here; o_free of item k + 1 needs the P V of item k + 1.
    if (lane == 0) {
      int n = 0, k = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
        const Item item = items[it];
        const int nt = tiles_of(item);
        for (int j = 0; j < nt; ++j, ++n) {
          const int sv = n % kVStages, b = n % kSBuf;
          if (!mbar_wait(&sm.v_full[sv], ph(n, kVStages), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          sm.v_consumed[sv] += 1;
          // at an item's first tile, O must have been read out by the previous item's
          // epilogue
          if (j == 0 &&
              !mbar_wait(&sm.o_free, ((uint32_t)k & 1u) ^ 1u, a.err, wait_bound<kSW>(a))) {
            ok = false;
            break;
          }
          // Keys of the tile in the item's range, rounded up to the 16-key step of P V:
          // only those V rows are read. At the item's last tile the rows between the
          // range's end and that step hold whatever the block tail holds: zero them (at
          // most 15) so that 0 * (non-finite) never reaches O.
          const int valid = min(kKeys, item.kv_end - (item.kv_begin + j * kKeys));
          const int kk_end = (valid + 15) >> 4;
          if (valid < kk_end * 16) {
            for (int r = valid; r < kk_end * 16; ++r) {
              uint4* v0 = reinterpret_cast<uint4*>(&sm.v[sv][0][r * 128]);
              uint4* v1 = reinterpret_cast<uint4*>(&sm.v[sv][1][r * 128]);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                v0[q] = make_uint4(0, 0, 0, 0);
                v1[q] = make_uint4(0, 0, 0, 0);
              }
            }
            tc::fence_async_shared();
          }
          // V as the MN-major B operand: step kk covers keys 16 kk .. 16 kk + 15 (rows of
          // 128 bytes), the two D halves kHalf apart. P (bf16 pairs) sits over the first
          // 64 columns of the scores: keys 16 kk .. at columns 8 kk ..
          const uint64_t vd = tc::smem_desc_sw128(smem_addr(&sm.v[sv][0][0]), kHalf, 1024);
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {
            if (!mbar_wait(&sm.p_full[b][hk], ph(n, kSBuf), a.err, wait_bound<kSW>(a))) { ok = false; break; }
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 4 * hk; kk < 4 * hk + 4; ++kk) {
              const uint32_t pa = tmem + s_col(b) + (uint32_t)kk * 8u;
              const uint64_t vk = vd + (uint64_t)((kk * 16 * 128) >> 4);
              if (kk == 0) {
                if (j > 0)
                  tc::mma_bf16_ts_c<true>(tmem + kColO, pa, vk, kIdescO);
                else
                  tc::mma_bf16_ts_c<false>(tmem + kColO, pa, vk, kIdescO);
              } else if (kk < kk_end) {
                tc::mma_bf16_ts_c<true>(tmem + kColO, pa, vk, kIdescO);
              }
            }
          }
          if (!ok) break;
          tc::commit(&sm.o_done[n & 1]);
          tc::commit(&sm.s_free[b]);
          tc::commit(&sm.v_empty[sv]);
        }
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain[1]);
      mbar_wait(&sm.drain[1], 0, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    // One thread per row (its TMEM lane): the whole 128-key score row is read with one
    // TMEM load, so no other thread needs the row's maximum or sum. P goes back over the
    // scores 8 columns at a time and is handed to the P V issuer in two key halves.
    // Phase bounds: s_full[b] of tile n + 3 needs s_free from the P V of tile n, which
    // needs p_full(n) from here; o_done[x] of tile n + 1 needs p_full(n + 1) from here,
    // and s_full(n) implies that the P V of tile n - 3 and every product issued before it
    // are done, so a wait for the P V of tile n - 1 (rescale) is never two phases off;
    // the epilogue waits for tile n - 2 first (implied done up to n - 4 by s_full(n - 1))
    // and then for tile n - 1.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;             // tile row = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    float* stg = sm.stage[warp - 3];
    int n = 0;                                    // tile of the CTA
    bool ok = true;
    // items two ahead, their lengths one ahead (the length loads need the sequence index)
    Item item_next{}, item_next2{};
    int L_next = 0, ql_next = 0;
    if ((int)blockIdx.x < n_items) {
      item_next = items[blockIdx.x];
      L_next = __ldg(a.context_lens + item_next.seq);
      ql_next = __ldg(a.query_lens + item_next.seq);
      if ((int)blockIdx.x + G < n_items) item_next2 = items[blockIdx.x + G];
    }
    for (int it = blockIdx.x; it < n_items && ok; it += G) {
      const Item info = item_next;
      const int L = L_next, ql = ql_next;
      if (it + G < n_items) {
        item_next = item_next2;
        L_next = __ldg(a.context_lens + item_next.seq);
        ql_next = __ldg(a.query_lens + item_next.seq);
        if (it + 2 * G < n_items) item_next2 = items[it + 2 * G];
      }
      const int kv_begin = info.kv_begin, kv_end = info.kv_end, row_count = info.row_count;
      if (kv_end > L || info.row_begin + row_count > ql * a.g) record_error(a.err, PA_DEVERR_LENS);
      // causal limit of this row (-1: not a row of the item)
      const int lim = row < row_count ? min(kv_end - 1, L - ql + (info.row_begin + row) / a.g) : -1;
      const int nt = (kv_end - kv_begin + kKeys - 1) / kKeys;
      const bool warp_live = quad * 32 < row_count;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j, ++n) {
        const int b = n % kSBuf;
        if (!mbar_wait_warp(&sm.s_full[b], ph(n, kSBuf), a.err, wait_bound<kSW>(a))) { ok = false; break; }
        tc::fence_after_sync();
        const int key0 = kv_begin + j * kKeys;
        const uint32_t s_addr = t_lane + s_col(b);
        if (warp_live) {
          const bool masked = key0 + kKeys - 1 > lim;
          float s[128];
          tc::tmem_ld128(s_addr, s);
          if (masked) {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (key0 + i > lim) s[i] = -INFINITY;
          }
          // running maximum of the raw scores (the scale is positive)
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < 64; ++i) m4[i & 3] = fmax3(m4[i & 3], s[2 * i], s[2 * i + 1]);
          const float m_new =
              fmaxf(m_used, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2);
          if (m_used == -INFINITY) m_used = m_new;
          // O is rescaled by 2^(m_used - m_new) only when the maximum grew by more than
          // 2^8; otherwise P keeps the older (smaller) maximum as its reference.
          const bool need = m_new > m_used + kRescaleLog2;
          const bool warp_rescale = __any_sync(0xffffffffu, need);
          const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
          if (need) {
            l *= alpha;
            m_used = m_new;
          }
          // P = 2^(scale * s - m) as bf16 pairs: keys 16 c .. 16 c + 15 go to columns
          // 8 c .. 8 c + 7; a masked score is -inf and gives exactly 0
          const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
          const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
          const uint64_t nm2 = f2_pack(neg_m, neg_m);
          uint64_t sum2[2] = {0ull, 0ull};
          __syncwarp();  // tcgen05.st is .sync.aligned: reconverge after the per-row update
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float pk[8];
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2) {
              const int i = c * 8 + i2;
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sc2, nm2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
              pk[i2] = __uint_as_float(pack_bf16(p0, p1));
            }
            tc::tmem_st8(s_addr + (uint32_t)c * 8u, pk);
            if (c == 3 && warp_rescale) {
              // O must be idle: the P V of the previous tile (same item: a rescale needs
              // an earlier tile) may still run. The P V of this tile waits for p_full,
              // arrived below. 16 columns at a time; tcgen05.ld / st are warp-collective,
              // so the warp rescales together (factor 1 for rows that need none).
              if (!mbar_wait_warp(&sm.o_done[(n - 1) & 1], ph(n - 1, 2), a.err,
                                  wait_bound<kSW>(a))) {
                ok = false;
              }
              tc::fence_after_sync();
              if (ok) {
#pragma unroll 1
                for (int c8 = 0; c8 < kD / 16; ++c8) {
                  float o[16];
                  const uint32_t addr = t_lane + kColO + (uint32_t)c8 * 16u;
                  tc::tmem_ld16(addr, o);
#pragma unroll
                  for (int i = 0; i < 16; ++i) o[i] *= alpha;
                  tc::tmem_st16(addr, o);
                }
              }
            }
            if ((c & 3) == 3) {
              // keys 64 (c / 4) .. + 63 are in TMEM: that half's P V may start
              tc::tmem_wait_st();
              tc::fence_before_sync();
              mbar_arrive(&sm.p_full[b][c >> 2]);
            }
          }
          float sa, sb;
          f2_unpack(f2_add(sum2[0], sum2[1]), sa, sb);
          l += sa + sb;
          if (!ok) break;
        } else {
          // rows past the item: zero P, so that no stale bits reach the tensor core
          float z[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) z[i] = 0.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tc::tmem_st16(s_addr + (uint32_t)c * 16u, z);
            if (c & 1) {
              tc::tmem_wait_st();
              tc::fence_before_sync();
              mbar_arrive(&sm.p_full[b][c >> 1]);
            }
          }
        }
      }
      if (!ok) break;
      // ---- epilogue: the item's last P V, and the one before it first (see the phase
      // bounds above)
      if (n >= 2 &&
          !mbar_wait_warp(&sm.o_done[(n - 2) & 1], ph(n - 2, 2), a.err, wait_bound<kSW>(a))) {
        ok = false;
        break;
      }
      if (!mbar_wait_warp(&sm.o_done[(n - 1) & 1], ph(n - 1, 2), a.err, wait_bound<kSW>(a))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // A warp whose 32 rows all belong to the item (and go to the output, not to split
      // partials) hands O / l to the TMA: it writes 16-column pieces of its rows into its
      // staging buffer in the output box's layout (packed row-major: tokens x heads x
      // columns) and one lane issues an asynchronous tensor store. Other warps store
      // rows themselves.
      const int rho0 = info.row_begin + quad * 32;
      const bool whole = info.part < 0 && quad * 32 + 32 <= row_count;
      if (whole) {
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const int c1 = info.kv_head * a.g + rho0 % a.g;
        const int c2 = info.q_row0 + rho0 / a.g;
#pragma unroll 1
        for (int c4 = 0; c4 < kD / 32; ++c4) {
          float o[32];
          __syncwarp();  // tcgen05.ld is .sync.aligned: reconverge after the single-lane store
          tc::tmem_ld32(t_lane + kColO + (uint32_t)c4 * 32u, o);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // the previous store has read the staging buffer
            if (lane == 0) bulk_wait_read();
            __syncwarp();
            // rows of 16 columns swizzled as the tensor map says (fp32: 16-byte chunk c of
            // row r at c ^ ((r / 2) % 4); bf16: at c ^ ((r / 4) % 2)): the eight lanes of
            // each quarter-warp write to distinct banks
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
        if (row < row_count) {
          if (part < 0) {
            inv = (l > 0.f) ? 1.f / l : 0.f;
            const int rho = info.row_begin + row;
            const int qt = rho / a.g;
            const int h = info.kv_head * a.g + (rho - qt * a.g);
            const int64_t off = ((int64_t)(info.q_row0 + qt) * a.Hq + h) * kD;
            dst_row = reinterpret_cast<char*>(a.out) + off * (a.out_bf16 ? 2 : 4);
          } else {
            const int64_t prow = (int64_t)part + row;
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
          tc::tmem_ld32(t_lane + kColO + (uint32_t)c4 * 32u, o);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // this lane's 16 values -> staging row `lane`; 16-byte chunk cj sits at
            // position cj ^ ((row / 2) % 4), free of bank conflicts both ways
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
      mbar_arrive(&sm.o_free);
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
    for (int s = 0; s < kKStages; ++s) {
      if (sm.k_issued[s] > sm.k_consumed[s]) {
        const uint32_t parity = (uint32_t)(sm.k_issued[s] - 1) & 1u;
        while (!mbar_try_wait(smem_addr(&sm.k_full[s]), parity))
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
    for (int s = 0; s < kVStages; ++s) {
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

int tc3_smem_bytes() { return (int)sizeof(Tc3Smem) + 1024; }

cudaError_t launch_tc3(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const CUtensorMap& qmap, const CUtensorMap& omap, const Item* items,
                       int32_t n_items, int box_t, int grid, cudaStream_t s, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  const int smem = tc3_smem_bytes();
  auto* k = a.wait_ns == kWaitLimitNsHost ? tc3_kernel<false> : tc3_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_kernel(k, grid, kThreads3, smem, s, pdl, a, kmap, vmap, qmap, omap, items, n_items,
                    box_t);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
