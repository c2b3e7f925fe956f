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
// How (GB300): one persistent CTA per SM, warp-specialised.
//   warp 0     TMA producer: per 128-key tile, one 3-D TMA copy per (block
//              piece, D half, K or V) straight from the physical blocks named by
//              the block table, 128-byte swizzled, into a 2-stage ring.
//   warp 1     allocates TMEM and issues tcgen05.mma from one thread:
//              S(j+1) = Q K_{j+1}^T is issued before O += P_j V_j so the tensor
//              core computes the next scores while the softmax runs.
//   warps 2-5  one thread per row (its TMEM lane): load the Q rows into
//              shared memory, read S from TMEM, mask (causal, bottom-right
//              aligned), online softmax in the log2 domain, write P (bf16,
//              swizzled) for the next MMA, rescale O in TMEM only when the
//              running maximum grows by more than 2^8, and write the output.
// TMEM columns: S double buffer [0,256), O [256,384). Every wait is bounded.
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

constexpr int kRows = kTcRows;        // 128 rows per tile (M)
constexpr int kKeys = 128;            // keys per tile (N of S, K of P V)
constexpr int kD = 128;               // head dim of this kernel
constexpr int kStagesTc = 2;
constexpr int kThreadsTc = 192;
constexpr int kHalf = kRows * 128;    // bytes of one 128-row x 64-element swizzled sub-tile
constexpr float kRescaleLog2 = 8.f;   // O is rescaled once the max grows by > 2^8
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kKeys, false);  // Q K^T, both K-major
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD, true);      // P V, V is MN-major

struct TcSmem {
  uint8_t q[2][kHalf];                  // Q rows, D halves
  uint8_t k[kStagesTc][2][kHalf];       // K tile, D halves
  uint8_t v[kStagesTc][2][kHalf];       // V tile, D halves (rows = keys)
  uint8_t p[2][kHalf];                  // P tile, key halves
  uint64_t kv_full[kStagesTc];
  uint64_t kv_empty[kStagesTc];
  uint64_t q_full, s_full[2], s_free[2], p_full, o_done, o_free, drain;
  uint32_t tmem_base;
  int issued[kStagesTc];
  int consumed[kStagesTc];
  int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap, const Item* __restrict__ items,
              int n_items, int box_t) {
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
    mbar_init(&sm.q_full, kRows);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], kRows);
    }
    mbar_init(&sm.p_full, kRows);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.o_free, kRows);
    mbar_init(&sm.drain, 1);
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
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int pieces = kKeys / box_t;                  // <= 16
    const uint32_t piece_bytes = (uint32_t)box_t * 128u;  // one D half of one piece
    int n = 0;                                         // global tile counter
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += G) {
      const Item item = items[it];
      const int32_t* bt = a.block_table + (int64_t)item.seq * a.max_blocks;
      for (int t0 = item.kv_begin; t0 < item.kv_end; t0 += kKeys, ++n) {
        const int st = n & 1;
        const uint32_t ph = (uint32_t)(n >> 1) & 1u;
        ok = mbar_wait(&sm.kv_empty[st], ph ^ 1u, a.err);
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        bool valid = false;
        int tok = 0;
        if (lane < pieces) {
          const int j0 = t0 + lane * box_t;
          if (j0 < item.kv_end) {
            const int lb = j0 / a.block_size;
            if (lb >= a.max_blocks) {
              record_error(a.err, PA_DEVERR_TABLE_RANGE);
            } else {
              const int phys = __ldg(bt + lb);
              if (phys < 0 || phys >= a.num_blocks) {
                record_error(a.err, PA_DEVERR_BLOCK_RANGE);
              } else {
                valid = true;
                tok = phys * a.block_size + (j0 - lb * a.block_size);
              }
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
    }
    if (!ok) sm.abort_flag = 1;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_addr(&sm.q[0][0]);
      const uint32_t p_addr = smem_addr(&sm.p[0][0]);
      int nS = 0, nP = 0, item_idx = 0;
      bool ok = true;
      // S(tile nS) = Q K^T into TMEM buffer nS % 2
      auto issue_s = [&]() -> bool {
        const int st = nS & 1;
        if (!mbar_wait(&sm.kv_full[st], (uint32_t)(nS >> 1) & 1u, a.err)) return false;
        sm.consumed[st] += 1;
        if (!mbar_wait(&sm.s_free[st], ((uint32_t)(nS >> 1) & 1u) ^ 1u, a.err)) return false;
        tc::fence_after_sync();
        const uint32_t k_addr = smem_addr(&sm.k[st][0][0]);
        const uint32_t d_tmem = tmem + (uint32_t)st * kKeys;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u;
          tc::mma_bf16(d_tmem, tc::smem_desc_sw128(q_addr + off, 16, 1024),
                       tc::smem_desc_sw128(k_addr + off, 16, 1024), kIdescS, kk > 0);
        }
        tc::commit(&sm.s_full[st]);
        ++nS;
        return true;
      };
      for (int it = blockIdx.x; it < n_items && ok; it += G, ++item_idx) {
        const Item item = items[it];
        const int nt = (item.kv_end - item.kv_begin + kKeys - 1) / kKeys;
        if (!mbar_wait(&sm.q_full, (uint32_t)item_idx & 1u, a.err)) { ok = false; break; }
        tc::fence_after_sync();
        if (!issue_s()) { ok = false; break; }
        for (int j = 0; j < nt; ++j) {
          if (j + 1 < nt && !issue_s()) { ok = false; break; }
          // O += P_j V_j
          if (!mbar_wait(&sm.p_full, (uint32_t)nP & 1u, a.err)) { ok = false; break; }
          if (j == 0 && !mbar_wait(&sm.o_free, ((uint32_t)item_idx & 1u) ^ 1u, a.err)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const int st = nP & 1;
          const uint32_t v_addr = smem_addr(&sm.v[st][0][0]);
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            const uint32_t a_off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u;
            const uint32_t b_off = (uint32_t)kk * 16u * 128u;
            tc::mma_bf16(tmem + 2u * kKeys, tc::smem_desc_sw128(p_addr + a_off, 16, 1024),
                         tc::smem_desc_sw128(v_addr + b_off, kHalf, 1024), kIdescO,
                         (j > 0) || (kk > 0));
          }
          tc::commit(&sm.o_done);
          tc::commit(&sm.kv_empty[st]);
          ++nP;
        }
      }
      if (!ok) sm.abort_flag = 1;
      // every MMA this thread issued has finished before the CTA moves on
      tc::commit(&sm.drain);
      mbar_wait(&sm.drain, 0, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;             // tile row = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    int n = 0, item_idx = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += G, ++item_idx) {
      const Item item = items[it];
      const int nt = (item.kv_end - item.kv_begin + kKeys - 1) / kKeys;
      const bool live = row < item.row_count;
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
      // ---- this row of Q into the swizzled Q tile (zeros for rows past the item)
      {
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + ((int64_t)(item.q_row0 + t) * a.Hq + h) * kD);
        uint4 vals[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) vals[j] = live ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          *reinterpret_cast<uint4*>(&sm.q[j >> 3][tc::sw128_offset(row, j & 7)]) = vals[j];
        tc::fence_async_shared();
        mbar_arrive(&sm.q_full);
      }
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j, ++n) {
        const int b = n & 1;
        if (!mbar_wait(&sm.s_full[b], (uint32_t)(n >> 1) & 1u, a.err)) { ok = false; break; }
        tc::fence_after_sync();
        float s[kKeys];
#pragma unroll
        for (int c4 = 0; c4 < kKeys / 32; ++c4) {
          float tmp[32];
          tc::tmem_ld32(t_lane + (uint32_t)b * kKeys + (uint32_t)c4 * 32u, tmp);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c4 * 32 + i] = tmp[i];
        }
        tc::fence_before_sync();
        mbar_arrive(&sm.s_free[b]);
        // mask and scale; running max
        const int key0 = item.kv_begin + j * kKeys;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          s[c] = (key0 + c <= lim) ? s[c] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
        const float m_new = fmaxf(m_used, mx);
        if (j > 0) {
          // P V of the previous tile must be done before O or P are touched
          if (!mbar_wait(&sm.o_done, (uint32_t)(n - 1) & 1u, a.err)) { ok = false; break; }
          tc::fence_after_sync();
        }
        if (m_used == -INFINITY) {
          m_used = m_new;  // nothing accumulated yet: O holds only zero rows
        } else if (m_new > m_used + kRescaleLog2) {
          const float alpha = fast_exp2(m_used - m_new);
#pragma unroll
          for (int c4 = 0; c4 < kD / 32; ++c4) {
            float o[32];
            const uint32_t addr = t_lane + 2u * kKeys + (uint32_t)c4 * 32u;
            tc::tmem_ld32(addr, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tc::tmem_st32(addr, o);
          }
          tc::tmem_wait_st();
          l *= alpha;
          m_used = m_new;
        }
        // P = 2^(s - m) in bf16, written as the swizzled A operand of the next MMA
        float sum = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < kKeys / 8; ++c8) {
          float p[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float x = s[c8 * 8 + i];
            p[i] = (x == -INFINITY) ? 0.f : fast_exp2(x - m_used);
          }
          uint4 w;
          w.x = pack_bf16(p[0], p[1]);
          w.y = pack_bf16(p[2], p[3]);
          w.z = pack_bf16(p[4], p[5]);
          w.w = pack_bf16(p[6], p[7]);
          // the normaliser sums the rounded weights the tensor core multiplies
          sum += bf16lo(w.x) + bf16hi(w.x) + bf16lo(w.y) + bf16hi(w.y) + bf16lo(w.z) +
                 bf16hi(w.z) + bf16lo(w.w) + bf16hi(w.w);
          *reinterpret_cast<uint4*>(&sm.p[c8 >> 3][tc::sw128_offset(row, c8 & 7)]) = w;
        }
        l += sum;
        // keys past the item's range hold whatever the block tail holds: zero those
        // V rows so that 0 * (non-finite) never reaches the accumulator
        if (key0 + row >= item.kv_end) {
          const int st = n & 1;
          uint4* v0 = reinterpret_cast<uint4*>(&sm.v[st][0][row * 128]);
          uint4* v1 = reinterpret_cast<uint4*>(&sm.v[st][1][row * 128]);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v0[i] = make_uint4(0, 0, 0, 0);
            v1[i] = make_uint4(0, 0, 0, 0);
          }
        }
        tc::fence_async_shared();
        tc::fence_before_sync();
        mbar_arrive(&sm.p_full);
      }
      if (!ok) break;
      // ---- epilogue: O / l
      if (!mbar_wait(&sm.o_done, (uint32_t)(n - 1) & 1u, a.err)) { ok = false; break; }
      tc::fence_after_sync();
      float o[kD];
#pragma unroll
      for (int c4 = 0; c4 < kD / 32; ++c4) {
        float tmp[32];
        tc::tmem_ld32(t_lane + 2u * kKeys + (uint32_t)c4 * 32u, tmp);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c4 * 32 + i] = tmp[i];
      }
      tc::fence_before_sync();
      mbar_arrive(&sm.o_free);
      if (live) {
        if (item.part < 0) {
          const float inv = (l > 0.f) ? 1.f / l : 0.f;
          const int64_t off = ((int64_t)(item.q_row0 + t) * a.Hq + h) * kD;
          if (a.out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off);
#pragma unroll
            for (int c8 = 0; c8 < kD / 8; ++c8) {
              uint4 w;
              w.x = pack_bf16(o[c8 * 8 + 0] * inv, o[c8 * 8 + 1] * inv);
              w.y = pack_bf16(o[c8 * 8 + 2] * inv, o[c8 * 8 + 3] * inv);
              w.z = pack_bf16(o[c8 * 8 + 4] * inv, o[c8 * 8 + 5] * inv);
              w.w = pack_bf16(o[c8 * 8 + 6] * inv, o[c8 * 8 + 7] * inv);
              dst[c8] = w;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off);
#pragma unroll
            for (int c4 = 0; c4 < kD / 4; ++c4)
              dst[c4] = make_float4(o[c4 * 4] * inv, o[c4 * 4 + 1] * inv, o[c4 * 4 + 2] * inv,
                                    o[c4 * 4 + 3] * inv);
          }
        } else {
          const int64_t prow = (int64_t)item.part + row;
          float4* dst = reinterpret_cast<float4*>(a.part_acc + prow * kD);
#pragma unroll
          for (int c4 = 0; c4 < kD / 4; ++c4)
            dst[c4] = make_float4(o[c4 * 4], o[c4 * 4 + 1], o[c4 * 4 + 2], o[c4 * 4 + 3]);
          a.part_ml[prow * 2 + 0] = m_used;
          a.part_ml[prow * 2 + 1] = l;
        }
      }
    }
    if (!ok) sm.abort_flag = 1;
  }

  tc::fence_before_sync();
  __syncthreads();
  // After an abort, give copies still in flight a bounded time to land.
  if (sm.abort_flag && threadIdx.x == 0) {
    for (int s = 0; s < kStagesTc; ++s) {
      if (sm.issued[s] > sm.consumed[s]) {
        const uint32_t parity = (uint32_t)(sm.issued[s] - 1) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_addr(&sm.kv_full[s]), parity))
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
                      const Item* items, int32_t n_items, int box_t, int grid, cudaStream_t s) {
  if (n_items <= 0) return cudaSuccess;
  const int smem = tc_smem_bytes();
  cudaError_t e =
      cudaFuncSetAttribute(tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  tc_kernel<<<grid, kThreadsTc, smem, s>>>(a, kmap, vmap, items, n_items, box_t);
  return cudaGetLastError();
}

}  // namespace pa
