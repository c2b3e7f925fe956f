// pa_tc.cu -- paged multi-token attention on the 5th-generation tensor cores (tcgen05),
// one 128-row query tile per item.
//
// What it computes: the same exact causal attention as the decode kernel
// ("PagedAttention" wiki page, "mathematical formulation"), for items whose rows
// (query tokens x the query heads of one KV head) fill a 128-row tile. Pensieve
// summary, multi-token attention: with many query tokens per request the work is two
// matrix-matrix products (S = Q K^T, O = P V) over a KV context that lives in
// non-contiguous blocks, with the causal mask fused so that the score matrix is never
// written to memory.
//
// How (GB300): one persistent CTA per SM, warp-specialised, 12 warps.
//   warps 0, 3 TMA producers: warp 0 loads the item's 128 Q rows (one 3-D box per
//              D half; the next item's Q loads while the current item's last tiles
//              and epilogue run) and, per 128-key tile, K into a 2-stage ring; warp 3
//              loads V into a 3-stage ring (a V tile is consumed one softmax later
//              than its K tile). Each gathers a tile per block piece straight from the
//              physical blocks named by the block table, 128-byte swizzled, with its
//              own barriers, so that a K tile never waits behind a V slot that the
//              P V products still hold. Block ids come from a shared-memory cache per
//              producer, filled one item ahead.
//   warp 1     issues S_j = Q K_j^T (M = N = 128) into TMEM buffer j % 2, so S_{j+1}
//              is computed while the softmax works on S_j.
//   warp 2     issues O_h += P_{j,h} V_{j,h} for the two key halves h of the tile
//              (keys 64 h .. 64 h + 63) into two accumulators O_0, O_1, each as soon
//              as its half of P is in TMEM. One thread alone cannot issue both
//              products as fast as the tensor core executes them.
//   warps 4-11 softmax: warp w owns TMEM lane quadrant w % 4 (32 rows) and key half
//              h = (w - 4) / 4 of every tile; one thread per row runs its own online
//              softmax over the keys of its half (log2 domain, lazy rescale of O_h
//              when its maximum grows by more than 2^8), so two warps share each
//              quadrant's work and no thread needs another's maximum or sum until the
//              item's end, where the two halves' (m, l, O) of a row are merged. P_h is
//              written back over that half's scores as bf16 pairs. The epilogue writes
//              16-column pieces of a warp's 32 rows into a staging buffer in the output
//              box's layout and one lane issues an asynchronous TMA store (warps with
//              rows past the item store rows themselves).
// TMEM columns: S double buffer [0, 256), O_0 [256, 384), O_1 [384, 512). TMEM
// loads/stores and whole-warp waits are always warp-uniform; every wait is bounded.
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
constexpr int kKeys = 128;              // keys per tile (N of S, K of P V)
constexpr int kD = 128;                 // head dim of this kernel
constexpr int kKStages = 2;             // K ring
constexpr int kVStages = 3;             // V ring: a V tile is needed a softmax later than K
constexpr int kQBuf = 1;                // Q buffers (the next item's Q loads under the
                                        // current item's last softmax and epilogue)
constexpr int kSoftmaxWarps = 8;
constexpr int kThreadsTc = (4 + kSoftmaxWarps) * 32;
constexpr int kHalf = 128 * 128;        // 128 rows x 64 elements, swizzled (16 KB)
constexpr int kStageCols = 16;          // epilogue staging: 32 rows x 16 fp32 per warp
constexpr float kRescaleLog2 = 8.f;     // O_h is rescaled once its max grows by > 2^8
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kKeys, false);  // Q K^T, both K-major
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD, true);      // P V, V is MN-major

__host__ __device__ constexpr uint32_t s_col(int b) { return (uint32_t)b * 128u; }
__host__ __device__ constexpr uint32_t o_col(int h) { return 256u + (uint32_t)h * 128u; }

struct TcSmem {
  uint8_t q[kQBuf][2][kHalf];           // [buffer][D half]
  uint8_t k[kKStages][2][kHalf];        // [stage][D half], rows = keys
  uint8_t v[kVStages][2][kHalf];        // [stage][D half], rows = keys
  float stage[kSoftmaxWarps][32 * kStageCols];
  float xm[2][2][kRows], xl[2][2][kRows];  // [item parity][key half][row]: (m, l) at the end
  int bt_cache[2][2][kBtCache];         // [K / V producer][item parity]: block ids
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t q_full[kQBuf], q_free[kQBuf];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2][2];                // [S buffer][key half]: P of that half written
  uint64_t o_done[2][2];                // [key half][tile parity]: P V of that half done
  uint64_t o_free;                      // the epilogue has read O_0 and O_1
  uint64_t xbar[4];                     // per lane quadrant: its two softmax warps met
  uint64_t drain[2];
  uint32_t tmem_base;
  int k_issued[kKStages], k_consumed[kKStages];
  int v_issued[kVStages], v_consumed[kVStages];
  int q_issued[kQBuf], q_consumed[kQBuf];
  int abort_flag;
};
static_assert(sizeof(TcSmem) + 1024 <= 227 * 1024, "shared memory of the one-tile kernel");

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

// TMA producer of K (kIsK, also the item's Q) or of V. Phase bounds: q_free[b] of
// item k + kQBuf needs q_full(k + kQBuf) from here; the ring's empty barrier of tile
// n + R (R stages) needs its full barrier of tile n + R from here. So no barrier is
// ever two phases ahead of the waits below.
template <bool kIsK, bool kSW>
__device__ __forceinline__ void produce(TcSmem& sm, const AttnArgs& a, const CUtensorMap& map,
                                        const CUtensorMap& qmap, const Item* __restrict__ items,
                                        int n_items, int box_t, int lane) {
  const int G = gridDim.x;
  constexpr int kStages = kIsK ? kKStages : kVStages;
  uint64_t* full = kIsK ? sm.k_full : sm.v_full;
  uint64_t* empty = kIsK ? sm.k_empty : sm.v_empty;
  uint8_t(*ring)[2][kHalf] = kIsK ? sm.k : sm.v;
  int* issued = kIsK ? sm.k_issued : sm.v_issued;
  int(*bt_cache)[kBtCache] = sm.bt_cache[kIsK ? 0 : 1];
  if (lane == 0) {
    prefetch_tensormap(&map);
    if (kIsK) prefetch_tensormap(&qmap);
  }
  const int pieces = kKeys / box_t;                     // <= 16
  const uint32_t piece_bytes = (uint32_t)box_t * 128u;  // one D half of one piece
  int n = 0, k = 0;                                     // tile / item counters of the CTA
  bool ok = true;
  // block ids are staged one item ahead: registers -> shared cache at the switch
  int nb[kBtPerLane];
  Item item_next{};
  if ((int)blockIdx.x < n_items) {
    const Item f = items[blockIdx.x];
    bt_prefetch(a.block_table + (int64_t)f.seq * a.max_blocks, a.max_blocks,
                bt_window(f.kv_begin, f.kv_end, a.block_size), lane, nb);
    bt_store(bt_cache[0], nb, lane);
    if ((int)blockIdx.x + G < n_items) item_next = items[blockIdx.x + G];
  }
  __syncwarp();
  for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
    const Item item = items[it];
    const BtWindow win = bt_window(item.kv_begin, item.kv_end, a.block_size);
    const int* cache = bt_cache[k & 1];
    const bool has_next = it + G < n_items;
    Item item_after{};
    if (has_next) {
      bt_prefetch(a.block_table + (int64_t)item_next.seq * a.max_blocks, a.max_blocks,
                  bt_window(item_next.kv_begin, item_next.kv_end, a.block_size), lane, nb);
      if (it + 2 * G < n_items) item_after = items[it + 2 * G];
    }
    if (kIsK) {
      // the item's 128 Q rows: tokens x the g heads of its KV head, one box per D half
      const int qb = k % kQBuf;
      ok = mbar_wait_warp(&sm.q_free[qb], ph(k, kQBuf) ^ 1u, a.err, wait_bound<kSW>(a));
      if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full[qb], 2u * kHalf);
        const int tok = item.q_row0 + item.row_begin / a.g;
        tma_load_3d(&sm.q[qb][0][0], &qmap, &sm.q_full[qb], 0, item.kv_head * a.g, tok);
        tma_load_3d(&sm.q[qb][1][0], &qmap, &sm.q_full[qb], 64, item.kv_head * a.g, tok);
        sm.q_issued[qb] += 1;
      }
      __syncwarp();
    }
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
            if (kIsK) record_error(a.err, PA_DEVERR_TABLE_RANGE);
          } else if (phys < 0 || phys >= a.num_blocks) {
            if (kIsK) record_error(a.err, PA_DEVERR_BLOCK_RANGE);
          } else {
            valid = true;
            tok = phys * a.block_size + (j0 - lb * a.block_size);
          }
        }
      }
      const uint32_t tile_bytes = __popc(__ballot_sync(0xffffffffu, valid)) * piece_bytes * 2u;
      // K_n is free once S of tile n - 2 completed, V_n once both halves' P V of it did
      ok = mbar_wait_warp(&empty[st], ph(n, kStages) ^ 1u, a.err, wait_bound<kSW>(a));
      if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
      if (lane == 0) mbar_arrive_expect_tx(&full[st], tile_bytes);
      __syncwarp();
      if (valid) {
        const uint32_t row_off = (uint32_t)lane * box_t * 128u;
        tma_load_3d(&ring[st][0][row_off], &map, &full[st], 0, item.kv_head, tok);
        tma_load_3d(&ring[st][1][row_off], &map, &full[st], 64, item.kv_head, tok);
      }
      if (lane == 0) issued[st] += 1;
    }
    if (has_next) {
      bt_store(bt_cache[(k + 1) & 1], nb, lane);
      item_next = item_after;
    }
    __syncwarp();
  }
  if (!ok) sm.abort_flag = 1;
}

template <bool kSW>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
              const __grid_constant__ CUtensorMap omap, const Item* __restrict__ items,
              int n_items, int box_t) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(align1024(smem_raw));
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
    for (int b = 0; b < kQBuf; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_free[b], 1);
      sm.q_issued[b] = sm.q_consumed[b] = 0;
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 1);
      mbar_init(&sm.p_full[b][0], kRows);
      mbar_init(&sm.p_full[b][1], kRows);
      mbar_init(&sm.o_done[0][b], 1);
      mbar_init(&sm.o_done[1][b], 1);
      mbar_init(&sm.drain[b], 1);
    }
    mbar_init(&sm.o_free, kSoftmaxWarps * 32);
    for (int qd = 0; qd < 4; ++qd) mbar_init(&sm.xbar[qd], 64);
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
    produce<true, kSW>(sm, a, kmap, qmap, items, n_items, box_t, lane);
  } else if (warp == 3) {
    produce<false, kSW>(sm, a, vmap, qmap, items, n_items, box_t, lane);
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // Phase bounds: q_full of item k + kQBuf needs q_free(k), committed here; k_full of
    // tile n + 2 needs k_empty(n), committed here; s_free of tile n + 2 needs the P V
    // of tile n + 2, which needs s_full(n + 2) from here.
    if (lane == 0) {
      int n = 0, k = 0;
      bool ok = true;
      int nt_next = (int)blockIdx.x < n_items ? tiles_of(items[blockIdx.x]) : 0;
      for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
        const int nt = nt_next;
        if (it + G < n_items) nt_next = tiles_of(items[it + G]);
        const int qb = k % kQBuf;
        if (!mbar_wait(&sm.q_full[qb], ph(k, kQBuf), a.err, wait_bound<kSW>(a))) { ok = false; break; }
        sm.q_consumed[qb] += 1;
        tc::fence_after_sync();
        const uint64_t qd = tc::smem_desc_sw128(smem_addr(&sm.q[qb][0][0]), 16, 1024);
        for (int j = 0; j < nt; ++j, ++n) {
          const int st = n % kKStages;
          const int b = n & 1;
          if (!mbar_wait(&sm.k_full[st], ph(n, kKStages), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          sm.k_consumed[st] += 1;
          // the buffer's last readers, both halves' P V of tile n - 2, are done
          if (!mbar_wait(&sm.s_free[b], ph(n, 2) ^ 1u, a.err, wait_bound<kSW>(a))) { ok = false; break; }
          tc::fence_after_sync();
          // S = Q K^T: 8 steps of 16 dims; step kk starts (kk / 4) D halves and
          // (kk % 4) 32-byte chunks into both operands
          const uint64_t kd = tc::smem_desc_sw128(smem_addr(&sm.k[st][0][0]), 16, 1024);
          tc::mma_bf16_c<false>(tmem + s_col(b), qd, kd, kIdescS);
#pragma unroll
          for (int kk = 1; kk < kD / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
            tc::mma_bf16_c<true>(tmem + s_col(b), qd + off, kd + off, kIdescS);
          }
          tc::commit(&sm.s_full[b]);
          tc::commit(&sm.k_empty[st]);
        }
        if (ok) tc::commit(&sm.q_free[qb]);  // the item's last S issued: Q may be reloaded
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain[0]);
      mbar_wait(&sm.drain[0], 0, a.err);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ P V issuer
    // Phase bounds: p_full[b][h] of tile n + 2 needs s_full(n + 2), which needs
    // s_free(n), committed here after the P V of tile n; v_full of tile n + kVStages
    // needs v_empty(n), committed here; o_free of item k + 1 needs the P V of item k + 1.
    if (lane == 0) {
      int n = 0, k = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
        const Item item = items[it];
        const int nt = tiles_of(item);
        bool o_init0 = false, o_init1 = false;  // O_h written in this item
        for (int j = 0; j < nt; ++j, ++n) {
          const int st = n % kVStages;
          const int b = n & 1;
          if (!mbar_wait(&sm.v_full[st], ph(n, kVStages), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          sm.v_consumed[st] += 1;
          // at an item's first tile, O_0 and O_1 must have been read out by the previous
          // item's epilogue
          if (j == 0 && !mbar_wait(&sm.o_free, ((uint32_t)k & 1u) ^ 1u, a.err, wait_bound<kSW>(a))) {
            ok = false;
            break;
          }
          // Keys of the tile in the item's range, rounded up to the 16-key step of P V:
          // only those V rows are read. At the item's last tile the rows between the
          // range's end and that step hold whatever the block tail holds: zero them
          // (at most 15 rows) so that 0 * (non-finite) never reaches O.
          const int valid = min(kKeys, item.kv_end - (item.kv_begin + j * kKeys));
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
          // V as the MN-major B operand: step kk covers keys 16 kk .. 16 kk + 15 (rows
          // of 128 bytes), the two D halves are kHalf apart. P_h (bf16 pairs) sits over
          // the first 32 columns of that key half's scores.
          const uint64_t vd = tc::smem_desc_sw128(smem_addr(&sm.v[st][0][0]), kHalf, 1024);
          // half 0: keys 0..63 of the tile
          if (!mbar_wait(&sm.p_full[b][0], ph(n, 2), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          tc::fence_after_sync();
          {
            const uint32_t pa = tmem + s_col(b);
            if (o_init0)
              tc::mma_bf16_ts_c<true>(tmem + o_col(0), pa, vd, kIdescO);
            else
              tc::mma_bf16_ts_c<false>(tmem + o_col(0), pa, vd, kIdescO);
            o_init0 = true;
#pragma unroll
            for (int kq = 1; kq < 4; ++kq)
              if (kq < kk_end)
                tc::mma_bf16_ts_c<true>(tmem + o_col(0), pa + (uint32_t)kq * 8u,
                                        vd + (uint64_t)((kq * 16 * 128) >> 4), kIdescO);
          }
          tc::commit(&sm.o_done[0][b]);
          // half 1: keys 64..127 of the tile
          if (!mbar_wait(&sm.p_full[b][1], ph(n, 2), a.err, wait_bound<kSW>(a))) { ok = false; break; }
          tc::fence_after_sync();
          if (kk_end > 4) {
            const uint32_t pa = tmem + s_col(b) + 64u;
            const uint64_t vd1 = vd + (uint64_t)((4 * 16 * 128) >> 4);
            if (o_init1)
              tc::mma_bf16_ts_c<true>(tmem + o_col(1), pa, vd1, kIdescO);
            else
              tc::mma_bf16_ts_c<false>(tmem + o_col(1), pa, vd1, kIdescO);
            o_init1 = true;
#pragma unroll
            for (int kq = 1; kq < 4; ++kq)
              if (4 + kq < kk_end)
                tc::mma_bf16_ts_c<true>(tmem + o_col(1), pa + (uint32_t)kq * 8u,
                                        vd1 + (uint64_t)((kq * 16 * 128) >> 4), kIdescO);
          }
          tc::commit(&sm.o_done[1][b]);
          tc::commit(&sm.s_free[b]);
          tc::commit(&sm.v_empty[st]);
        }
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain[1]);
      mbar_wait(&sm.drain[1], 0, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    // Warp w: lane quadrant quad = w % 4 (rows 32 quad ..), key half h = (w - 4) / 4.
    // Phase bounds: s_full of tile n + 2 needs s_free(n), i.e. both halves' P V(n),
    // which need p_full(n) from here; o_done[h][b] of tile n + 2 needs p_full(n + 2)
    // from here, and s_full(n) implies that P V(n - 2) and everything before it are
    // done, so the waits for P V(n - 1) are never two phases off. xbar[quad] completes
    // only with both warps of the quadrant, and the (m, l) exchange buffers alternate
    // by item: a warp can be at most one item ahead of its partner (the next item's
    // third tile needs the partner's P of that item).
    const int quad = warp & 3;
    const int h = (warp - 4) >> 2;
    const int row = quad * 32 + lane;             // tile row = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    float* stg = sm.stage[warp - 4];
    int n = 0, k = 0;
    bool ok = true;
    // Items are read two ahead and their lengths one ahead: the length loads need the
    // item's sequence index, so with one stage they would wait for the item load
    // itself right at the item switch.
    Item item_next{}, item_next2{};
    int L_next = 0, ql_next = 0;
    if ((int)blockIdx.x < n_items) {
      item_next = items[blockIdx.x];
      L_next = __ldg(a.context_lens + item_next.seq);
      ql_next = __ldg(a.query_lens + item_next.seq);
      if ((int)blockIdx.x + G < n_items) item_next2 = items[blockIdx.x + G];
    }
    for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
      const Item item = item_next;
      const int L = L_next, ql = ql_next;
      if (it + G < n_items) {
        item_next = item_next2;
        L_next = __ldg(a.context_lens + item_next.seq);
        ql_next = __ldg(a.query_lens + item_next.seq);
        if (it + 2 * G < n_items) item_next2 = items[it + 2 * G];
      }
      if (item.kv_end > L || item.row_begin + item.row_count > ql * a.g)
        record_error(a.err, PA_DEVERR_LENS);
      const int nt = tiles_of(item);
      const bool live = row < item.row_count;
      const bool warp_live = quad * 32 < item.row_count;
      // this row's last visible key (causal, bottom-right aligned), -1 past the item
      const int lim = live ? min(item.kv_end - 1, L - ql + (item.row_begin + row) / a.g) : -1;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j, ++n) {
        const int b = n & 1;
        if (!mbar_wait_warp(&sm.s_full[b], ph(n, 2), a.err, wait_bound<kSW>(a))) { ok = false; break; }
        tc::fence_after_sync();
        const int k0 = item.kv_begin + j * kKeys + 64 * h;   // first key of this half
        const uint32_t s_addr = t_lane + s_col(b) + (uint32_t)(64 * h);
        if (warp_live) {
          float s[64];
          tc::tmem_ld64(s_addr, s);
          if (k0 + 63 > lim) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (k0 + i > lim) s[i] = -INFINITY;
          }
          // running maximum of this half's raw scores (the scale is positive)
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < 32; ++i) m4[i & 3] = fmax3(m4[i & 3], s[2 * i], s[2 * i + 1]);
          const float m_new =
              fmaxf(m_used, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2);
          // nothing accumulated yet: adopt the new maximum
          if (m_used == -INFINITY) m_used = m_new;
          // O_h is rescaled by 2^(m_used - m_new) only when the maximum grew by more
          // than 2^8; otherwise P keeps the older (smaller) maximum as its reference.
          const bool need = m_new > m_used + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            // O_h must be idle: the previous tile's P V of this half may still run
            if (!mbar_wait_warp(&sm.o_done[h][(n - 1) & 1], ph(n - 1, 2), a.err, wait_bound<kSW>(a))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
            // tcgen05.ld / st are warp-collective: the warp rescales together (factor 1
            // for rows that need none), 16 columns at a time
#pragma unroll 1
            for (int c8 = 0; c8 < kD / 16; ++c8) {
              float o[16];
              const uint32_t addr = t_lane + o_col(h) + (uint32_t)c8 * 16u;
              tc::tmem_ld16(addr, o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= alpha;
              tc::tmem_st16(addr, o);
            }
            if (need) {
              l *= alpha;
              m_used = m_new;
            }
          }
          // P = 2^(scale * s - m) as bf16 pairs over this half's first 32 columns; a
          // masked score is -inf and gives exactly 0
          const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
          const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
          const uint64_t nm2 = f2_pack(neg_m, neg_m);
          uint64_t sum2[2] = {0ull, 0ull};
          __syncwarp();  // tcgen05.st is .sync.aligned: reconverge after the per-row update
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float pk[16];
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              const int i = c * 16 + i2;
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sc2, nm2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
              pk[i2] = __uint_as_float(pack_bf16(p0, p1));
            }
            tc::tmem_st16(s_addr + (uint32_t)c * 16u, pk);
          }
          float sa, sb;
          f2_unpack(f2_add(sum2[0], sum2[1]), sa, sb);
          l += sa + sb;
        } else {
          // rows past the item: zero P, so that no stale bits reach the tensor core
          float z[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) z[i] = 0.f;
          tc::tmem_st16(s_addr, z);
          tc::tmem_st16(s_addr + 16u, z);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        mbar_arrive(&sm.p_full[b][h]);
      }
      if (!ok) break;
      // ---- epilogue: merge the two halves of each row, then O / l. This warp writes
      // output columns 64 h .. 64 h + 63 of its 32 rows.
      const int xb = k & 1;
      sm.xm[xb][h][row] = m_used;
      sm.xl[xb][h][row] = l;
      mbar_arrive(&sm.xbar[quad]);
      if (!mbar_wait_warp(&sm.xbar[quad], (uint32_t)k & 1u, a.err, wait_bound<kSW>(a))) { ok = false; break; }
      // both halves' last P V (each at most one phase ahead of this wait: see above)
      if (!mbar_wait_warp(&sm.o_done[0][(n - 1) & 1], ph(n - 1, 2), a.err, wait_bound<kSW>(a)) ||
          !mbar_wait_warp(&sm.o_done[1][(n - 1) & 1], ph(n - 1, 2), a.err, wait_bound<kSW>(a))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (warp_live) {
        const float m0 = sm.xm[xb][0][row], m1 = sm.xm[xb][1][row];
        const float l0 = sm.xl[xb][0][row], l1 = sm.xl[xb][1][row];
        const float mm = fmaxf(m0, m1);
        // a half without a visible key of this row has l = 0 and an O_h that is not
        // part of the sum (it may not even have been written in this item)
        const float w0 = l0 > 0.f ? fast_exp2(m0 - mm) : 0.f;
        const float w1 = l1 > 0.f ? fast_exp2(m1 - mm) : 0.f;
        const float lt = l0 * w0 + l1 * w1;
        const int rho0 = item.row_begin + quad * 32;
        const bool whole = item.part < 0 && quad * 32 + 32 <= item.row_count;
        char* dst_row = nullptr;                  // this lane's row (nullptr: not stored)
        float inv = 1.f;
        if (item.part < 0) {
          inv = (lt > 0.f) ? 1.f / lt : 0.f;
          if (!whole && live) {
            const int rho = item.row_begin + row;
            const int qt = rho / a.g;
            const int hd = item.kv_head * a.g + (rho - qt * a.g);
            const int64_t off = ((int64_t)(item.q_row0 + qt) * a.Hq + hd) * kD;
            dst_row = reinterpret_cast<char*>(a.out) + off * (a.out_bf16 ? 2 : 4);
          }
        } else if (live) {
          const int64_t prow = (int64_t)item.part + row;
          dst_row = reinterpret_cast<char*>(a.part_acc + prow * kD);
          if (h == 0) {
            a.part_ml[prow * 2 + 0] = mm;
            a.part_ml[prow * 2 + 1] = lt;
          }
        }
        const float f0 = w0 * inv, f1 = w1 * inv;
        const bool bf = a.out_bf16 && item.part < 0;
        const int c1 = item.kv_head * a.g + rho0 % a.g;
        const int c2 = item.q_row0 + rho0 / a.g;
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          // 16 output columns 64 h + 16 c4 ..: (w0 O_0 + w1 O_1) / l
          const int col = 64 * h + 16 * c4;
          float o0[16], o1[16], o[16];
          // tcgen05.ld is .sync.aligned: reconverge after the per-row setup and after
          // the previous piece's single-lane store
          __syncwarp();
          tc::tmem_ld16(t_lane + o_col(0) + (uint32_t)col, o0);
          tc::tmem_ld16(t_lane + o_col(1) + (uint32_t)col, o1);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o[i] = (w0 > 0.f ? o0[i] * f0 : 0.f) + (w1 > 0.f ? o1[i] * f1 : 0.f);
          // the previous tensor store of this warp has read the staging buffer
          if (lane == 0) bulk_wait_read();
          __syncwarp();
          if (whole) {
            // the output box's layout: row-major rows (tokens x heads) of 16 columns,
            // swizzled as the tensor map says (fp32: 16-byte chunk c of row r at
            // c ^ ((r / 2) % 4); bf16: at c ^ ((r / 4) % 2)), so that the eight lanes of
            // each quarter-warp write to distinct banks
            if (a.out_bf16) {
              uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(stg) + lane * 32);
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                uint4 w;
                w.x = pack_bf16(o[8 * i + 0], o[8 * i + 1]);
                w.y = pack_bf16(o[8 * i + 2], o[8 * i + 3]);
                w.z = pack_bf16(o[8 * i + 4], o[8 * i + 5]);
                w.w = pack_bf16(o[8 * i + 6], o[8 * i + 7]);
                d[i ^ ((lane >> 2) & 1)] = w;
              }
            } else {
              float4* d = reinterpret_cast<float4*>(stg + lane * kStageCols);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d[i ^ ((lane >> 1) & 3)] =
                    make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
            tc::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&omap, stg, col, c1, c2);
              bulk_commit();
            }
          } else {
            // this lane's 16 values -> staging row `lane`; 16-byte chunk cj sits at
            // position cj ^ ((row / 2) % 4), free of bank conflicts both ways
#pragma unroll
            for (int cj = 0; cj < 4; ++cj) {
              const int pos = cj ^ ((lane >> 1) & 3);
              reinterpret_cast<float4*>(stg + lane * kStageCols)[pos] =
                  make_float4(o[4 * cj], o[4 * cj + 1], o[4 * cj + 2], o[4 * cj + 3]);
            }
            __syncwarp();
            // 8 rows x 64 bytes per store instruction: lane -> row 8 qq + lane / 4,
            // 16-byte chunk lane % 4
            const int colw = col + (lane & 3) * 4;
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
                  *reinterpret_cast<uint2*>(d + colw * 2) = w;
                } else {
                  *reinterpret_cast<float4*>(d + colw * 4) = v;
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
    for (int b = 0; b < kQBuf; ++b) {
      if (sm.q_issued[b] > sm.q_consumed[b]) {
        const uint32_t parity = (uint32_t)(sm.q_issued[b] - 1) & 1u;
        while (!mbar_try_wait(smem_addr(&sm.q_full[b]), parity))
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  pdl_wait();  // exit only after the kernel this one may overlap has completed
}

}  // namespace

int tc_smem_bytes() { return (int)sizeof(TcSmem) + 1024; }

cudaError_t launch_tc(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      const CUtensorMap& qmap, const CUtensorMap& omap, const Item* items,
                      int32_t n_items, int box_t, int grid, cudaStream_t s, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  const int smem = tc_smem_bytes();
  auto* k = a.wait_ns == kWaitLimitNsHost ? tc_kernel<false> : tc_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_kernel(k, grid, kThreadsTc, smem, s, pdl, a, kmap, vmap, qmap, omap, items,
                    n_items, box_t);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
