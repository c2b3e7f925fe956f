// pa_dec.cu -- paged attention on CUDA cores for items with few rows (decode and
// short multi-token queries), plus the split-KV combine pass.
//
// What it computes: "PagedAttention" wiki page, "mathematical formulation" --
// o_i = sum_{j<=i} softmax_j(q_i.k_j / sqrt(d)) v_j, evaluated one K/V block at a
// time (the block form); the keys of a sequence are reached only through its
// block table (vLLM post, "1. overall architecture"). Several query rows share
// one pass over the keys: the query heads of one KV head (GQA packing) and, for
// multi-token items, several query tokens, each with its own causal limit
// (Pensieve summary, multi-token attention with the causal mask fused).
//
// How (GB300): one persistent CTA per SM walks a static round-robin list of
// items. Warp 8 is a producer: for every 64-key stage it reads the block ids
// and issues one 3-D TMA copy per (block piece, K or V) into a 4-stage
// shared-memory ring guarded by mbarriers, running ahead across item
// boundaries. Warps 0-7 consume: QK^T with each 16-byte K chunk loaded once and
// reused for every row, scores reduced across the lanes of a token with a
// reduce-scatter of shuffles, an online softmax in the log2 domain (one warp
// per row), then P.V with the rescale folded in. Memory traffic is the
// algorithmic minimum: every K/V byte of an item's key range is read once.
// Long key ranges are split by the plan; split items write (m, l, acc) partials
// that combine_kernel merges exactly (the normaliser of the softmax rewritten
// as a sum over chunks).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kStages = 4;
constexpr int kCWarps = 8;                       // consumer warps
constexpr int kCThreads = kCWarps * 32;          // consumer threads
constexpr int kThreads = kCThreads + 32;         // + one producer warp
constexpr int kSPad = kKeyTile + 4;              // score row stride (bank spread)
constexpr int kConsumerBar = 1;                  // named barrier id of the consumers

template <int D, int RM>
struct DecSmem {
  uint16_t k[kStages][kKeyTile][D];
  uint16_t v[kStages][kKeyTile][D];
  float s[RM][kSPad];           // scores of the stage, log2 domain
  float p[kKeyTile][RM];        // probabilities, key-major
  float red[kCWarps][RM][D];    // end-of-item reduction of the P.V partial sums
  float alpha[RM];
  float m[RM];
  float l[RM];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int issued[kStages];    // TMA phases issued per stage (producer)
  int consumed[kStages];  // phases the consumers have waited for
  int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Sum across the CH lanes of a token group, scattering rows: afterwards lane
// holds the full score of row `row` (RM <= CH).
template <int N, int OFF, int RM>
struct ReduceScatter {
  __device__ __forceinline__ static void run(float (&v)[RM], int lane, int& row) {
    if constexpr (OFF > 0) {
      if constexpr (N > 1) {
        constexpr int H = N / 2;
        const bool up = (lane & OFF) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = up ? v[i] : v[i + H];
          const float keep = up ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
        }
        row += up ? H : 0;
        ReduceScatter<H, OFF / 2, RM>::run(v, lane, row);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
        ReduceScatter<1, OFF / 2, RM>::run(v, lane, row);
      }
    }
  }
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// All consumer threads agree on `ok` (AND) at a named barrier.
__device__ __forceinline__ bool consumers_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(kConsumerBar), "n"(kCThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
  f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
  f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

template <int D, int RM>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const Item* __restrict__ items,
                  int n_items, int box_t) {
  constexpr int CH = D / 8;                     // 16-byte chunks per key row
  constexpr int TPW = 32 / CH;                  // keys per warp step
  constexpr int QK_STEPS = kKeyTile / (kCWarps * TPW);
  constexpr int PV_STEPS = kKeyTile / (kCWarps * TPW);
  static_assert(RM <= CH, "rows per item must not exceed the lanes of a key");
  static_assert(QK_STEPS * kCWarps * TPW == kKeyTile, "tile split");

  extern __shared__ uint8_t smem_raw[];
  DecSmem<D, RM>& sm = *reinterpret_cast<DecSmem<D, RM>*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCWarps);
      sm.issued[s] = 0;
      sm.consumed[s] = 0;
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kCWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int pieces = kKeyTile / box_t;
    const uint32_t piece_bytes = (uint32_t)box_t * D * 2u;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const Item item = items[it];
      const int L = __ldg(a.context_lens + item.seq);
      const int kv_end = min(item.kv_end, L);
      const int32_t* bt = a.block_table + (int64_t)item.seq * a.max_blocks;
      for (int t0 = item.kv_begin; t0 < kv_end; t0 += kKeyTile) {
        ok = mbar_wait(&sm.empty[stage], phase ^ 1u, a.err);
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        // pieces lane and lane + 32 of this stage (a stage has at most 64 pieces)
        auto locate = [&](int pc, int& tok) -> bool {
          if (pc >= pieces) return false;
          const int j0 = t0 + pc * box_t;
          if (j0 >= kv_end) return false;
          const int lb = j0 / a.block_size;
          if (lb >= a.max_blocks) {
            record_error(a.err, PA_DEVERR_TABLE_RANGE);
            return false;
          }
          const int phys = __ldg(bt + lb);
          if (phys < 0 || phys >= a.num_blocks) {
            record_error(a.err, PA_DEVERR_BLOCK_RANGE);
            return false;
          }
          tok = phys * a.block_size + (j0 - lb * a.block_size);
          return true;
        };
        int tok0 = 0, tok1 = 0;
        const bool v0 = locate(lane, tok0);
        const bool v1 = locate(lane + 32, tok1);
        const uint32_t n_pieces = __popc(__ballot_sync(0xffffffffu, v0)) +
                                  __popc(__ballot_sync(0xffffffffu, v1));
        // one arrive carrying every byte of the stage, before any copy is issued
        if (lane == 0) mbar_arrive_expect_tx(&sm.full[stage], n_pieces * piece_bytes * 2u);
        __syncwarp();
        if (v0) {
          tma_load_3d(&sm.k[stage][lane * box_t][0], &kmap, &sm.full[stage], 0, item.kv_head, tok0);
          tma_load_3d(&sm.v[stage][lane * box_t][0], &vmap, &sm.full[stage], 0, item.kv_head, tok0);
        }
        if (v1) {
          tma_load_3d(&sm.k[stage][(lane + 32) * box_t][0], &kmap, &sm.full[stage], 0,
                      item.kv_head, tok1);
          tma_load_3d(&sm.v[stage][(lane + 32) * box_t][0], &vmap, &sm.full[stage], 0,
                      item.kv_head, tok1);
        }
        if (lane == 0) sm.issued[stage] += 1;
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) sm.abort_flag = 1;
  } else {
    // ------------------------------------------------------------ consumers
    const int c = lane % CH;   // 16-byte chunk of the key row this lane owns
    const int tl = lane / CH;  // key within the warp step
    int stage = 0;
    uint32_t phase = 0;
    bool alive = true;
    for (int it = blockIdx.x; it < n_items && alive; it += gridDim.x) {
      const Item item = items[it];
      const int L = __ldg(a.context_lens + item.seq);
      const int ql = __ldg(a.query_lens + item.seq);
      const int kv_end = min(item.kv_end, L);
      const int nrows = item.row_count;
      if (threadIdx.x == 0 && item.row_begin + nrows > ql * a.g)
        record_error(a.err, PA_DEVERR_LENS);

      // this lane's chunk of every row's query, pre-scaled into the log2 domain
      float qv[RM][8];
#pragma unroll
      for (int r = 0; r < RM; ++r) {
        if (r < nrows) {
          const int rho = item.row_begin + r;
          const int t = rho / a.g;
          const int h = item.kv_head * a.g + (rho - t * a.g);
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(
                                    a.q + ((int64_t)(item.q_row0 + t) * a.Hq + h) * D) + c);
          unpack8(w, qv[r]);
#pragma unroll
          for (int e = 0; e < 8; ++e) qv[r][e] *= a.scale_log2;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) qv[r][e] = 0.f;
        }
      }
      // causal limit of the row this warp runs the softmax for
      int my_lim = -1;
      if (warp < RM && warp < nrows) {
        const int t = (item.row_begin + warp) / a.g;
        my_lim = min(kv_end - 1, L - ql + t);
      }
      float m_run = -INFINITY, l_run = 0.f;
      float acc[RM][8];
#pragma unroll
      for (int r = 0; r < RM; ++r)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;

      for (int t0 = item.kv_begin; t0 < kv_end; t0 += kKeyTile) {
        const bool got = mbar_wait(&sm.full[stage], phase, a.err);
        // ---- S = Q K^T for the stage's 64 keys
        const uint16_t* Ks = &sm.k[stage][0][0];
#pragma unroll
        for (int i = 0; i < QK_STEPS; ++i) {
          const int tok = warp * (kKeyTile / kCWarps) + i * TPW + tl;
          float kf[8];
          unpack8(*reinterpret_cast<const uint4*>(Ks + tok * D + c * 8), kf);
          float part[RM];
#pragma unroll
          for (int r = 0; r < RM; ++r) {
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) x = fmaf(qv[r][e], kf[e], x);
            part[r] = x;
          }
          int row = 0;
          ReduceScatter<RM, CH / 2, RM>::run(part, lane, row);
          if ((c & (CH / RM - 1)) == 0) sm.s[row][tok] = part[0];
        }
        if (!consumers_all(got)) { alive = false; break; }
        if (threadIdx.x == 0) sm.consumed[stage] += 1;
        // ---- online softmax, one warp per row
        if (warp < RM) {
          const int j0 = t0 + lane, j1 = t0 + lane + 32;
          const float s0 = (j0 <= my_lim) ? sm.s[warp][lane] : -INFINITY;
          const float s1 = (j1 <= my_lim) ? sm.s[warp][lane + 32] : -INFINITY;
          const float m_new = fmaxf(m_run, warp_max(fmaxf(s0, s1)));
          const float alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
          const float p0 = (j0 <= my_lim) ? fast_exp2(s0 - m_new) : 0.f;
          const float p1 = (j1 <= my_lim) ? fast_exp2(s1 - m_new) : 0.f;
          l_run = l_run * alpha + warp_sum(p0 + p1);
          m_run = m_new;
          sm.p[lane][warp] = p0;
          sm.p[lane + 32][warp] = p1;
          if (lane == 0) sm.alpha[warp] = alpha;
        }
        named_bar_sync(kConsumerBar, kCThreads);
        // ---- O = alpha * O + P V
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          const float al = sm.alpha[r];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[r][e] *= al;
        }
        const uint16_t* Vs = &sm.v[stage][0][0];
#pragma unroll
        for (int i = 0; i < PV_STEPS; ++i) {
          const int tok = i * (kCWarps * TPW) + warp * TPW + tl;
          if (t0 + tok < kv_end) {
            float vf[8];
            unpack8(*reinterpret_cast<const uint4*>(Vs + tok * D + c * 8), vf);
            float pr[RM];
#pragma unroll
            for (int r = 0; r < RM; ++r) pr[r] = sm.p[tok][r];
#pragma unroll
            for (int r = 0; r < RM; ++r)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pr[r], vf[e], acc[r][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!alive) break;

      // ---- epilogue: sum the P.V partials of all keys of the warp, then of all warps
#pragma unroll
      for (int off = CH; off < 32; off <<= 1)
#pragma unroll
        for (int r = 0; r < RM; ++r)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], off);
      if (tl == 0) {
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          float4* dst = reinterpret_cast<float4*>(&sm.red[warp][r][c * 8]);
          dst[0] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
          dst[1] = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
        }
      }
      if (warp < RM && lane == 0) {
        sm.m[warp] = m_run;
        sm.l[warp] = l_run;
      }
      named_bar_sync(kConsumerBar, kCThreads);
      for (int idx = threadIdx.x; idx < nrows * D; idx += kCThreads) {
        const int r = idx / D, d = idx - r * D;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) o += sm.red[w][r][d];
        if (item.part < 0) {
          const int rho = item.row_begin + r;
          const int t = rho / a.g;
          const int h = item.kv_head * a.g + (rho - t * a.g);
          const int64_t off = ((int64_t)(item.q_row0 + t) * a.Hq + h) * D + d;
          const float l = sm.l[r];
          o = (l > 0.f) ? o / l : 0.f;
          if (a.out_bf16)
            reinterpret_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(o);
          else
            reinterpret_cast<float*>(a.out)[off] = o;
        } else {
          const int64_t prow = (int64_t)item.part + r;
          a.part_acc[prow * D + d] = o;
          if (d == 0) {
            a.part_ml[prow * 2 + 0] = sm.m[r];
            a.part_ml[prow * 2 + 1] = sm.l[r];
          }
        }
      }
      named_bar_sync(kConsumerBar, kCThreads);
    }
    if (!alive && threadIdx.x == 0) sm.abort_flag = 1;
  }
  __syncthreads();
  // After an abort, give copies still in flight a bounded time to land
  // before the CTA's shared memory is released.
  if (sm.abort_flag && threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      if (sm.issued[s] > sm.consumed[s]) {
        const uint32_t parity = (uint32_t)(sm.issued[s] - 1) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_addr(&sm.full[s]), parity))
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  }
}

// Merges the key chunks of split rows: m* = max m_c, l* = sum_c l_c 2^(m_c - m*),
// o = sum_c acc_c 2^(m_c - m*) / l*.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnArgs a,
                                                      const SplitGroup* __restrict__ groups) {
  constexpr int PER = D / 32;
  const SplitGroup gp = groups[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < gp.row_count; r += 8) {
    float mstar = -INFINITY;
    for (int c = 0; c < gp.n_parts; ++c) {
      const int64_t prow = (int64_t)gp.part_begin + (int64_t)c * gp.row_count + r;
      mstar = fmaxf(mstar, a.part_ml[prow * 2]);
    }
    float o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = 0.f;
    float lsum = 0.f;
    for (int c = 0; c < gp.n_parts; ++c) {
      const int64_t prow = (int64_t)gp.part_begin + (int64_t)c * gp.row_count + r;
      const float mc = a.part_ml[prow * 2];
      if (mc == -INFINITY) continue;
      const float w = fast_exp2(mc - mstar);
      lsum += w * a.part_ml[prow * 2 + 1];
      const float* src = a.part_acc + prow * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] = fmaf(w, src[e], o[e]);
    }
    const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
    const int rho = gp.row_begin + r;
    const int t = rho / a.g;
    const int h = gp.kv_head * a.g + (rho - t * a.g);
    const int64_t off = ((int64_t)(gp.q_row0 + t) * a.Hq + h) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      if (a.out_bf16)
        reinterpret_cast<__nv_bfloat16*>(a.out)[off + e] = __float2bfloat16_rn(o[e] * inv);
      else
        reinterpret_cast<float*>(a.out)[off + e] = o[e] * inv;
    }
  }
}

template <int D, int RM>
cudaError_t launch_dec_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const Item* items, int32_t n_items, int box_t, int grid,
                         cudaStream_t s) {
  const int smem = (int)sizeof(DecSmem<D, RM>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, RM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_kernel<D, RM><<<grid, kThreads, smem, s>>>(a, kmap, vmap, items, n_items, box_t);
  return cudaGetLastError();
}

template <int D>
constexpr int dec_smem(int rows_max) {
  return rows_max <= 1   ? (int)sizeof(DecSmem<D, 1>) + 1024
         : rows_max <= 2 ? (int)sizeof(DecSmem<D, 2>) + 1024
         : rows_max <= 4 ? (int)sizeof(DecSmem<D, 4>) + 1024
                         : (int)sizeof(DecSmem<D, 8>) + 1024;
}

}  // namespace

int decode_smem_bytes(int D, int rows_max) {
  return D == 128 ? dec_smem<128>(rows_max) : dec_smem<64>(rows_max);
}

cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const Item* items, int32_t n_items, int D, int rows_max, int box_t,
                          int grid, cudaStream_t s) {
  if (n_items <= 0) return cudaSuccess;
  if (D == 128) {
    if (rows_max <= 1) return launch_dec_t<128, 1>(a, kmap, vmap, items, n_items, box_t, grid, s);
    if (rows_max <= 2) return launch_dec_t<128, 2>(a, kmap, vmap, items, n_items, box_t, grid, s);
    if (rows_max <= 4) return launch_dec_t<128, 4>(a, kmap, vmap, items, n_items, box_t, grid, s);
    return launch_dec_t<128, 8>(a, kmap, vmap, items, n_items, box_t, grid, s);
  }
  if (rows_max <= 1) return launch_dec_t<64, 1>(a, kmap, vmap, items, n_items, box_t, grid, s);
  if (rows_max <= 2) return launch_dec_t<64, 2>(a, kmap, vmap, items, n_items, box_t, grid, s);
  if (rows_max <= 4) return launch_dec_t<64, 4>(a, kmap, vmap, items, n_items, box_t, grid, s);
  return launch_dec_t<64, 8>(a, kmap, vmap, items, n_items, box_t, grid, s);
}

cudaError_t launch_combine(const AttnArgs& a, const SplitGroup* groups, int32_t n_groups, int D,
                           cudaStream_t s) {
  if (n_groups <= 0) return cudaSuccess;
  if (D == 128)
    combine_kernel<128><<<n_groups, 256, 0, s>>>(a, groups);
  else
    combine_kernel<64><<<n_groups, 256, 0, s>>>(a, groups);
  return cudaGetLastError();
}

}  // namespace pa
