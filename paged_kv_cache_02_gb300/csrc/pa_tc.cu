// pa_tc.cu -- paged multi-token attention on the 5th-generation tensor cores (tcgen05).
//
// What it computes: the same exact causal attention as the decode kernel
// ("PagedAttention" wiki page, "mathematical formulation"), for items whose
// rows (query tokens x the query heads of one KV head) fill a 128-row tile.
// Pensieve summary, multi-token attention: with many query tokens per request
// the work is two matrix-matrix products (S = Q K^T, O = P V) over a KV
// context that lives in non-contiguous blocks, with the causal mask fused so
// that the score matrix is never written to memory.
//
// How (GB300): one persistent CTA per SM, warp-specialised, 7 warps.
//   warp 0     TMA producer: the item's 128 Q rows (one 3-D box per D half,
//              double-buffered across items) and, per 128-key tile, one 3-D
//              TMA copy per (block piece, D half, K or V) straight from the
//              physical blocks named by the block table, 128-byte swizzled,
//              into a 2-stage ring. Block ids come from a shared-memory cache
//              filled one item ahead.
//   warp 1     issues S_j = Q K_j^T (tcgen05.mma, both operands in shared
//              memory, M = N = 128) into TMEM buffer j % 2.
//   warp 2     issues O += P_j V_j with P_j read from TMEM (the softmax writes
//              it over S_j as bf16) and V_j from shared memory. Two issuing
//              warps keep the tensor core fed: one thread alone cannot issue
//              these instructions as fast as they execute.
//   warps 3-6  one thread per row (its TMEM lane): mask (causal, bottom-right
//              aligned), online softmax in the log2 domain, P to TMEM,
//              O rescaled in TMEM only when the running maximum grows by more
//              than 2^8, output O / l. Warps whose rows all lie past the item's
//              rows skip the arithmetic.
// TMEM columns: S/P double buffer [0, 256), O [256, 384). Every wait is bounded.
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
constexpr int kStagesTc = 2;
constexpr int kThreadsTc = 224;
constexpr int kHalf = 128 * 128;        // 128 rows x 64 elements, swizzled (16 KB)
constexpr float kRescaleLog2 = 8.f;     // O is rescaled once the max grows by > 2^8
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;        // first column of O

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kKeys, false);  // Q K^T, both K-major
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD, true);      // P V, V is MN-major

struct TcSmem {
  uint8_t q[2][2][kHalf];               // [buffer][D half]
  uint8_t k[kStagesTc][2][kHalf];       // [stage][D half], rows = keys
  uint8_t v[kStagesTc][2][kHalf];       // [stage][D half], rows = keys
  int bt_cache[2][kBtCache];            // block ids of the current and the next item
  uint64_t kv_full[kStagesTc];
  uint64_t kv_empty[kStagesTc];
  uint64_t q_full[2], q_free[2];
  uint64_t s_full[2], s_free[2], p_full[2];
  uint64_t o_done[2];                   // P V of tiles with this parity done (one barrier per
                                        // parity, so a waiter is never two phases behind)
  uint64_t o_free, drain[2];
  uint32_t tmem_base;
  int issued[kStagesTc];
  int consumed[kStagesTc];
  int q_issued[2];
  int q_consumed[2];
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

__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
              const Item* __restrict__ items, int n_items, int box_t) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesTc; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
      sm.issued[s] = 0;
      sm.consumed[s] = 0;
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_free[b], 1);
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 1);
      mbar_init(&sm.p_full[b], kRows);
      mbar_init(&sm.drain[b], 1);
      sm.q_issued[b] = 0;
      sm.q_consumed[b] = 0;
    }
    mbar_init(&sm.o_done[0], 1);
    mbar_init(&sm.o_done[1], 1);
    mbar_init(&sm.o_free, kRows);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Phase bounds: q_free[b] of item k + 2 needs q_full(k + 2) from here, and
    // kv_empty of tile n + 2 needs kv_full(n + 2) from here, so neither barrier is
    // ever two phases ahead of the wait below.
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      prefetch_tensormap(&qmap);
    }
    const int pieces = kKeys / box_t;                     // <= 16
    const uint32_t piece_bytes = (uint32_t)box_t * 128u;  // one D half of one piece
    int n = 0, k = 0;                                     // global tile / item counters
    bool ok = true;
    // block ids are staged one item ahead: registers -> shared cache at the switch
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
      // the item's 128 Q rows: tokens x the g heads of its KV head, one box per D half
      {
        const int qb = k & 1;
        ok = mbar_wait_warp(&sm.q_free[qb], ph(k, 2) ^ 1u, a.err);
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
        const int st = n % kStagesTc;
        ok = mbar_wait_warp(&sm.kv_empty[st], ph(n, kStagesTc) ^ 1u, a.err);
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
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
        const uint32_t cnt = __popc(__ballot_sync(0xffffffffu, valid));
        if (lane == 0) mbar_arrive_expect_tx(&sm.kv_full[st], cnt * piece_bytes * 4u);
        __syncwarp();
        if (valid) {
          const uint32_t row_off = (uint32_t)lane * box_t * 128u;
          tma_load_3d(&sm.k[st][0][row_off], &kmap, &sm.kv_full[st], 0, item.kv_head, tok);
          tma_load_3d(&sm.k[st][1][row_off], &kmap, &sm.kv_full[st], 64, item.kv_head, tok);
          tma_load_3d(&sm.v[st][0][row_off], &vmap, &sm.kv_full[st], 0, item.kv_head, tok);
          tma_load_3d(&sm.v[st][1][row_off], &vmap, &sm.kv_full[st], 64, item.kv_head, tok);
        }
        if (lane == 0) sm.issued[st] += 1;
      }
      if (has_next) {
        bt_store(sm.bt_cache[(k + 1) & 1], nb, lane);
        item_next = item_after;
      }
      __syncwarp();
    }
    if (!ok) sm.abort_flag = 1;
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // Phase bounds: q_full of item k + 2 needs q_free(k), committed here; kv_full of
    // tile n + 2 needs kv_empty(n), i.e. P V(n), which needs s_full(n) from here;
    // s_free of tile n + 2 needs S(n + 2) from here.
    if (lane == 0) {
      int n = 0, k = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
        const int nt = tiles_of(items[it]);
        const int qb = k & 1;
        if (!mbar_wait(&sm.q_full[qb], ph(k, 2), a.err)) { ok = false; break; }
        sm.q_consumed[qb] += 1;
        tc::fence_after_sync();
        const uint64_t qd = tc::smem_desc_sw128(smem_addr(&sm.q[qb][0][0]), 16, 1024);
        for (int j = 0; j < nt; ++j, ++n) {
          const int st = n % kStagesTc;
          const int b = n & 1;
          if (!mbar_wait(&sm.kv_full[st], ph(n, kStagesTc), a.err)) { ok = false; break; }
          sm.consumed[st] += 1;
          if (!mbar_wait(&sm.s_free[b], ph(n, 2) ^ 1u, a.err)) { ok = false; break; }
          tc::fence_after_sync();
          // S = Q K^T: 8 steps of 16 dims; step kk starts (kk / 4) D halves and
          // (kk % 4) 32-byte chunks into both operands
          const uint64_t kd = tc::smem_desc_sw128(smem_addr(&sm.k[st][0][0]), 16, 1024);
          tc::mma_bf16_c<false>(tmem + (uint32_t)b * kKeys, qd, kd, kIdescS);
#pragma unroll
          for (int kk = 1; kk < kD / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
            tc::mma_bf16_c<true>(tmem + (uint32_t)b * kKeys, qd + off, kd + off, kIdescS);
          }
          tc::commit(&sm.s_full[b]);
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
    // Phase bounds: p_full of tile n + 2 needs s_full(n + 2), which needs s_free(n)
    // committed here; o_free of item k + 1 needs the P V of item k + 1 from here.
    if (lane == 0) {
      int n = 0, k = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
        const int nt = tiles_of(items[it]);
        for (int j = 0; j < nt; ++j, ++n) {
          const int st = n % kStagesTc;
          const int b = n & 1;
          if (!mbar_wait(&sm.p_full[b], ph(n, 2), a.err)) { ok = false; break; }
          if (j == 0 && !mbar_wait(&sm.o_free, ((uint32_t)k & 1u) ^ 1u, a.err)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          // V as the MN-major B operand: step kk covers keys 16 kk .. 16 kk + 15 (rows
          // of 128 bytes), the two D halves are kHalf apart
          const uint64_t vd = tc::smem_desc_sw128(smem_addr(&sm.v[st][0][0]), kHalf, 1024);
          const uint32_t pa = tmem + (uint32_t)b * kKeys;
          if (j > 0)
            tc::mma_bf16_ts_c<true>(tmem + kTmemO, pa, vd, kIdescO);
          else
            tc::mma_bf16_ts_c<false>(tmem + kTmemO, pa, vd, kIdescO);
#pragma unroll
          for (int kk = 1; kk < kKeys / 16; ++kk) {
            tc::mma_bf16_ts_c<true>(tmem + kTmemO, pa + (uint32_t)kk * 8u,
                                    vd + (uint64_t)((kk * 16 * 128) >> 4), kIdescO);
          }
          tc::commit(&sm.o_done[b]);
          tc::commit(&sm.kv_empty[st]);
          tc::commit(&sm.s_free[b]);
        }
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain[1]);
      mbar_wait(&sm.drain[1], 0, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    // Phase bounds: s_full of tile n + 2 needs s_free(n), i.e. P V(n), which needs
    // p_full(n) from here; o_done[b] completes one phase per P V of tiles of parity
    // b, and P V(n + 1) needs p_full(n + 1) from here, so the waits for P V(n - 1)
    // (rescale) and for the item's last P V (epilogue) are never two phases behind.
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;             // tile row = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    int n = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += G) {
      const Item item = items[it];
      const int nt = tiles_of(item);
      const bool live = row < item.row_count;
      const bool warp_live = quad * 32 < item.row_count;
      int t = 0, h = 0, lim = -1;
      if (live) {
        const int rho = item.row_begin + row;
        t = rho / a.g;
        h = item.kv_head * a.g + (rho - t * a.g);
        const int L = __ldg(a.context_lens + item.seq);
        const int ql = __ldg(a.query_lens + item.seq);
        lim = min(item.kv_end - 1, L - ql + t);
        if (item.kv_end > L || item.row_begin + item.row_count > ql * a.g)
          record_error(a.err, PA_DEVERR_LENS);
      }
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j, ++n) {
        const int b = n & 1;
        if (!mbar_wait_warp(&sm.s_full[b], ph(n, 2), a.err)) { ok = false; break; }
        tc::fence_after_sync();
        const int key0 = item.kv_begin + j * kKeys;
        if (warp_live) {
          float s[kKeys];
          {
            float s0[64], s1[64];
            tc::tmem_ld64(t_lane + (uint32_t)b * kKeys, s0);
            tc::tmem_ld64(t_lane + (uint32_t)b * kKeys + 64u, s1);
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              s[i] = s0[i];
              s[64 + i] = s1[i];
            }
          }
          // running max of the raw scores (the scale is positive, so it commutes with
          // max); only a tile that crosses this row's causal limit needs the mask
          if (key0 + kKeys - 1 > lim) {
#pragma unroll
            for (int c = 0; c < kKeys; ++c) s[c] = (key0 + c <= lim) ? s[c] : -INFINITY;
          }
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
          for (int c = 8; c < kKeys; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
          const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          const float m_new = fmaxf(m_used, mx * a.scale_log2);
          // nothing accumulated yet: O holds only zero rows, adopt the new maximum
          if (m_used == -INFINITY) m_used = m_new;
          // tcgen05.ld / st are warp-collective: the whole warp rescales when any of
          // its rows needs it, the others with factor 1
          const bool need = m_new > m_used + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            // the previous P V must be done before O is rescaled
            if (!mbar_wait_warp(&sm.o_done[(n - 1) & 1], ph(n - 1, 2), a.err)) { ok = false; break; }
            tc::fence_after_sync();
            const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll 1
            for (int c4 = 0; c4 < kD / 32; ++c4) {
              float o[32];
              const uint32_t addr = t_lane + kTmemO + (uint32_t)c4 * 32u;
              tc::tmem_ld32(addr, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tc::tmem_st32(addr, o);
            }
            if (need) {
              l *= alpha;
              m_used = m_new;
            }
          }
          // P = 2^(scale * s - m) as bf16 pairs over the S columns: the A operand of P V.
          // A masked score is -inf and gives exactly 0.
          const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
          float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            float pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float p0 = fast_exp2(fmaf(s[h2 * 64 + 2 * c], a.scale_log2, neg_m));
              const float p1 = fast_exp2(fmaf(s[h2 * 64 + 2 * c + 1], a.scale_log2, neg_m));
              sum8[c & 7] += p0 + p1;
              pk[c] = __uint_as_float(pack_bf16(p0, p1));
            }
            tc::tmem_st32(t_lane + (uint32_t)b * kKeys + (uint32_t)h2 * 32u, pk);
          }
          tc::tmem_wait_st();
          l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
               ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        } else {
          // rows past the item: zero P, so that no stale bits reach the tensor core
          float z[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) z[c] = 0.f;
          tc::tmem_st32(t_lane + (uint32_t)b * kKeys, z);
          tc::tmem_st32(t_lane + (uint32_t)b * kKeys + 32u, z);
          tc::tmem_wait_st();
        }
        // keys past the item's range hold whatever the block tail holds: zero those
        // V rows so that 0 * (non-finite) never reaches the accumulator
        if (key0 + row >= item.kv_end) {
          const int st = n % kStagesTc;
          uint4* v0 = reinterpret_cast<uint4*>(&sm.v[st][0][row * 128]);
          uint4* v1 = reinterpret_cast<uint4*>(&sm.v[st][1][row * 128]);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v0[i] = make_uint4(0, 0, 0, 0);
            v1[i] = make_uint4(0, 0, 0, 0);
          }
          tc::fence_async_shared();
        }
        tc::fence_before_sync();
        mbar_arrive(&sm.p_full[b]);
      }
      if (!ok) break;
      // ---- epilogue: O / l
      if (!mbar_wait_warp(&sm.o_done[(n - 1) & 1], ph(n - 1, 2), a.err)) { ok = false; break; }
      tc::fence_after_sync();
      // tcgen05.ld is warp-collective: every lane of a live warp reads its row of O,
      // only rows of the item are stored
      if (warp_live) {
        float* out_f = nullptr;
        __nv_bfloat16* out_h = nullptr;
        float inv = 1.f;
        if (live) {
          if (item.part < 0) {
            inv = (l > 0.f) ? 1.f / l : 0.f;
            const int64_t off = ((int64_t)(item.q_row0 + t) * a.Hq + h) * kD;
            if (a.out_bf16)
              out_h = reinterpret_cast<__nv_bfloat16*>(a.out) + off;
            else
              out_f = reinterpret_cast<float*>(a.out) + off;
          } else {
            const int64_t prow = (int64_t)item.part + row;
            out_f = a.part_acc + prow * kD;
            a.part_ml[prow * 2 + 0] = m_used;
            a.part_ml[prow * 2 + 1] = l;
          }
        }
#pragma unroll 1
        for (int c4 = 0; c4 < kD / 32; ++c4) {
          float o[32];
          tc::tmem_ld32(t_lane + kTmemO + (uint32_t)c4 * 32u, o);
          if (out_f) {
            float4* dst = reinterpret_cast<float4*>(out_f + c4 * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                   o[4 * i + 3] * inv);
          } else if (out_h) {
            uint4* dst = reinterpret_cast<uint4*>(out_h + c4 * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = pack_bf16(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
              w.y = pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
              w.z = pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
              w.w = pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
              dst[i] = w;
            }
          }
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&sm.o_free);
    }
    if (!ok) sm.abort_flag = 1;
  }

  tc::fence_before_sync();
  __syncthreads();
  // After an abort, give copies still in flight a bounded time to land.
  if (sm.abort_flag && threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    for (int s = 0; s < kStagesTc; ++s) {
      if (sm.issued[s] > sm.consumed[s]) {
        const uint32_t parity = (uint32_t)(sm.issued[s] - 1) & 1u;
        while (!mbar_try_wait(smem_addr(&sm.kv_full[s]), parity))
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
    for (int b = 0; b < 2; ++b) {
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
}

}  // namespace

int tc_smem_bytes() { return (int)sizeof(TcSmem) + 1024; }

cudaError_t launch_tc(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      const CUtensorMap& qmap, const Item* items, int32_t n_items, int box_t,
                      int grid, cudaStream_t s) {
  if (n_items <= 0) return cudaSuccess;
  const int smem = tc_smem_bytes();
  cudaError_t e =
      cudaFuncSetAttribute(tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  tc_kernel<<<grid, kThreadsTc, smem, s>>>(a, kmap, vmap, qmap, items, n_items, box_t);
  return cudaGetLastError();
}

}  // namespace pa
