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
// items. Warp 8 is the producer: for every 64-key stage it issues one 3-D TMA
// copy per (block piece, K or V) into a shared-memory ring guarded by
// mbarriers, and on an item's first stage also the item's query rows (1-D bulk
// copies). An item's block ids are loaded while the previous item is being
// issued and kept in shared memory, so no global load sits between a free
// stage and its copies. Warps 0-7 consume, each on its own 8-key slice of every stage and
// with its own online softmax (an exact split of the keys inside the CTA): no
// CTA-wide barrier is needed per stage. QK^T loads every 16-byte K chunk once
// and uses it for all rows; the per-key sums are reduce-scattered with
// shuffles; P.V folds the rescale in. At the end of an item the eight warp
// partials (m, l, acc) are merged with the log-sum-exp rule. Every K/V byte of
// an item's key range is read from HBM once. Long key ranges are split by the
// plan; split items write (m, l, acc) partials that combine_kernel merges.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kCWarps = 8;                       // consumer warps
constexpr int kCThreads = kCWarps * 32;          // consumer threads
constexpr int kThreads = kCThreads + 32;         // + one producer warp
constexpr int kSlice = kKeyTile / kCWarps;       // keys per warp per stage (8)
constexpr int kConsumerBar = 1;                  // named barrier id of the consumers

// Pipeline depth from the shared-memory budget (stages of 64 keys).
template <int D, int RM>
constexpr int dec_stages() {
  return D == 64 ? 8 : (RM <= 2 ? 6 : 5);
}

template <int D, int RM>
struct DecSmem {
  static constexpr int S = dec_stages<D, RM>();
  uint16_t k[S][kKeyTile][D];
  uint16_t v[S][kKeyTile][D];
  uint16_t q[S][RM][D];              // the item's query rows, carried by its first stage
  float s[kCWarps][RM][kSlice];      // per-warp scores of the slice (log2 domain)
  float p[kCWarps][kSlice][RM];      // per-warp probabilities, key-major
  float alpha[kCWarps][RM];          // per-warp rescale factors of the stage
  float red[kCWarps][RM][D];         // end-of-item partial sums of the warps
  float red_m[kCWarps][RM];
  float red_l[kCWarps][RM];
  float wgt[kCWarps][RM];            // merge weights 2^(m_w - m)
  float inv_l[RM];
  float m_fin[RM];
  float l_fin[RM];
  uint64_t full[S];
  uint64_t empty[S];
  int bt_cache[2][kBtCache];  // block ids of the producer's current and next item
  int issued[S];    // copy phases issued per stage (producer)
  int consumed[S];  // phases the consumers have waited for
  int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Sum across the CH lanes of a key group, scattering rows: afterwards the lane
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

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
  f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
  f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

// 1-D bulk copy global -> shared, completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

template <int D, int RM, bool kSW>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const Item* __restrict__ items,
                  int n_items, int box_t) {
  using Smem = DecSmem<D, RM>;
  constexpr int S = Smem::S;
  constexpr int CH = D / 8;                     // 16-byte chunks per key row
  constexpr int TPW = 32 / CH;                  // keys per warp step
  constexpr int STEPS = kSlice / TPW;           // warp steps per slice
  static_assert(RM <= CH, "rows per item must not exceed the lanes of a key");
  static_assert(STEPS * TPW == kSlice, "slice split");

  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCWarps);
      sm.issued[s] = 0;
      sm.consumed[s] = 0;
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == kCWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int pieces = kKeyTile / box_t;           // <= 64
    const uint32_t piece_bytes = (uint32_t)box_t * D * 2u;
    const int G = gridDim.x;
    int stage = 0;
    uint32_t phase = 0;
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
    int k = 0;
    for (int it = blockIdx.x; it < n_items && ok; it += G, ++k) {
      const Item cur = items[it];
      const BtWindow win = bt_window(cur.kv_begin, cur.kv_end, a.block_size);
      const int* cache = sm.bt_cache[k & 1];
      const int32_t* bt = a.block_table + (int64_t)cur.seq * a.max_blocks;
      const bool has_next = it + G < n_items;
      Item item_after{};
      if (has_next) {
        bt_prefetch(a.block_table + (int64_t)item_next.seq * a.max_blocks, a.max_blocks,
                    bt_window(item_next.kv_begin, item_next.kv_end, a.block_size), lane, nb);
        if (it + 2 * G < n_items) item_after = items[it + 2 * G];
      }
      for (int t0 = cur.kv_begin; t0 < cur.kv_end; t0 += kKeyTile) {
        ok = mbar_wait_warp(&sm.empty[stage], phase ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        // pieces lane and lane + 32 of this stage (a stage has at most 64 pieces)
        auto locate = [&](int pc, int& tok) -> bool {
          if (pc >= pieces) return false;
          const int j0 = t0 + pc * box_t;
          if (j0 >= cur.kv_end) return false;
          const int lb = j0 / a.block_size;
          const int ph = bt_lookup(cache, win, bt, a.max_blocks, lb);
          if (ph == -2) { record_error(a.err, PA_DEVERR_TABLE_RANGE); return false; }
          if (ph < 0 || ph >= a.num_blocks) { record_error(a.err, PA_DEVERR_BLOCK_RANGE); return false; }
          tok = ph * a.block_size + (j0 - lb * a.block_size);
          return true;
        };
        int tok0 = 0, tok1 = 0;
        const bool v0 = locate(lane, tok0);
        const bool v1 = locate(lane + 32, tok1);
        uint32_t bytes = (__popc(__ballot_sync(0xffffffffu, v0)) +
                          __popc(__ballot_sync(0xffffffffu, v1))) * piece_bytes * 2u;
        // the item's query rows ride on its first stage: one copy per query token
        const bool first = (t0 == cur.kv_begin);
        int qt_first = 0, n_qtok = 0;
        if (first) {
          qt_first = cur.row_begin / a.g;
          n_qtok = (cur.row_begin + cur.row_count - 1) / a.g - qt_first + 1;
          bytes += (uint32_t)cur.row_count * D * 2u;
        }
        // one arrive carrying every byte of the stage, before any copy is issued
        if (lane == 0) mbar_arrive_expect_tx(&sm.full[stage], bytes);
        __syncwarp();
        if (v0) {
          tma_load_3d(&sm.k[stage][lane * box_t][0], &kmap, &sm.full[stage], 0, cur.kv_head, tok0);
          tma_load_3d(&sm.v[stage][lane * box_t][0], &vmap, &sm.full[stage], 0, cur.kv_head, tok0);
        }
        if (v1) {
          tma_load_3d(&sm.k[stage][(lane + 32) * box_t][0], &kmap, &sm.full[stage], 0,
                      cur.kv_head, tok1);
          tma_load_3d(&sm.v[stage][(lane + 32) * box_t][0], &vmap, &sm.full[stage], 0,
                      cur.kv_head, tok1);
        }
        if (first && lane < n_qtok) {
          const int t = qt_first + lane;
          const int h_lo = max(cur.row_begin, t * a.g) - t * a.g;
          const int h_hi = min(cur.row_begin + cur.row_count, (t + 1) * a.g) - t * a.g;
          const uint16_t* src =
              a.q + ((int64_t)(cur.q_row0 + t) * a.Hq + (int64_t)cur.kv_head * a.g + h_lo) * D;
          bulk_load(&sm.q[stage][t * a.g + h_lo - cur.row_begin][0], src,
                    (uint32_t)(h_hi - h_lo) * D * 2u, &sm.full[stage]);
        }
        if (lane == 0) sm.issued[stage] += 1;
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (has_next) {
        bt_store(sm.bt_cache[(k + 1) & 1], nb, lane);
        item_next = item_after;
      }
      __syncwarp();
    }
    if (!ok) sm.abort_flag = 1;
  } else {
    // ------------------------------------------------------------ consumers
    const int c = lane % CH;   // 16-byte chunk of the key row this lane owns
    const int tl = lane / CH;  // key within the warp step
    // softmax lanes: (row, key) pairs of the warp's slice
    constexpr int PPL = (RM * kSlice + 31) / 32;   // pairs per lane (1 or 2)
    constexpr int LPR = kSlice / PPL;              // lanes per row
    const int sm_row = lane / LPR;                 // row this lane runs the softmax for
    const int sm_key = (lane % LPR) * PPL;         // first slice key of its pair(s)
    int stage = 0;
    uint32_t phase = 0;
    bool alive = true;
    const int G = gridDim.x;
    // items and their sequences' lengths are fetched one item ahead
    Item item{}, nitem{};
    int L = 0, ql = 0;
    if ((int)blockIdx.x < n_items) {
      item = items[blockIdx.x];
      L = __ldg(a.context_lens + item.seq);
      ql = __ldg(a.query_lens + item.seq);
    }
    if ((int)blockIdx.x + G < n_items) nitem = items[blockIdx.x + G];
    for (int it = blockIdx.x; it < n_items && alive; it += G) {
      Item nn{};
      int nL = 0, nql = 0;
      if (it + 2 * G < n_items) nn = items[it + 2 * G];
      if (it + G < n_items) {
        nL = __ldg(a.context_lens + nitem.seq);
        nql = __ldg(a.query_lens + nitem.seq);
      }
      const int kv_end = item.kv_end;
      const int nrows = item.row_count;
      int lim = -1;   // last key the softmax row of this lane may see
      if (sm_row < RM && sm_row < nrows) {
        const int t = (item.row_begin + sm_row) / a.g;
        lim = min(kv_end - 1, L - ql + t);
        if (warp == 0 && lane == 0 && (item.kv_end > L || item.row_begin + nrows > ql * a.g))
          record_error(a.err, PA_DEVERR_LENS);
      }
      float qv[RM][8];
      float m_run = -INFINITY, l_run = 0.f;
      float acc[RM][8];
#pragma unroll
      for (int r = 0; r < RM; ++r)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;

      for (int t0 = item.kv_begin; t0 < kv_end; t0 += kKeyTile) {
        const bool got = mbar_wait_warp(&sm.full[stage], phase, a.err, wait_bound<kSW>(a));
        if (!got) { alive = false; break; }
        if (warp == 0 && lane == 0) sm.consumed[stage] += 1;
        if (t0 == item.kv_begin) {
          // query rows of the item (arrived with this stage), pre-scaled to the log2 domain
#pragma unroll
          for (int r = 0; r < RM; ++r) {
            if (r < nrows) {
              unpack8(*reinterpret_cast<const uint4*>(&sm.q[stage][r][c * 8]), qv[r]);
#pragma unroll
              for (int e = 0; e < 8; ++e) qv[r][e] *= a.scale_log2;
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) qv[r][e] = 0.f;
            }
          }
        }
        // ---- S = Q K^T on this warp's 8 keys
        const uint16_t* Ks = &sm.k[stage][warp * kSlice][0];
#pragma unroll
        for (int i = 0; i < STEPS; ++i) {
          const int key = i * TPW + tl;
          float kf[8];
          unpack8(*reinterpret_cast<const uint4*>(Ks + key * D + c * 8), kf);
          float part[RM];
#pragma unroll
          for (int r = 0; r < RM; ++r) {
            float x0 = qv[r][0] * kf[0], x1 = qv[r][1] * kf[1];
            x0 = fmaf(qv[r][2], kf[2], x0); x1 = fmaf(qv[r][3], kf[3], x1);
            x0 = fmaf(qv[r][4], kf[4], x0); x1 = fmaf(qv[r][5], kf[5], x1);
            x0 = fmaf(qv[r][6], kf[6], x0); x1 = fmaf(qv[r][7], kf[7], x1);
            part[r] = x0 + x1;
          }
          int row = 0;
          ReduceScatter<RM, CH / 2, RM>::run(part, lane, row);
          if ((c & (CH / RM - 1)) == 0) sm.s[warp][row][key] = part[0];
        }
        __syncwarp();
        // ---- online softmax of the warp's slice: lanes own (row, key) pairs
        {
          const int kbase = t0 + warp * kSlice + sm_key;
          float sv[PPL], pv[PPL];
          float mx = -INFINITY;
#pragma unroll
          for (int u = 0; u < PPL; ++u) {
            const bool ok_key = (sm_row < RM) && (kbase + u <= lim);
            sv[u] = ok_key ? sm.s[warp][sm_row][sm_key + u] : -INFINITY;
            mx = fmaxf(mx, sv[u]);
          }
#pragma unroll
          for (int o = LPR / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const float m_new = fmaxf(m_run, mx);
          const float alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
          float sum = 0.f;
#pragma unroll
          for (int u = 0; u < PPL; ++u) {
            pv[u] = (sv[u] == -INFINITY) ? 0.f : fast_exp2(sv[u] - m_new);
            sum += pv[u];
          }
#pragma unroll
          for (int o = LPR / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          l_run = l_run * alpha + sum;
          m_run = m_new;
          if (sm_row < RM) {
#pragma unroll
            for (int u = 0; u < PPL; ++u) sm.p[warp][sm_key + u][sm_row] = pv[u];
            if (lane % LPR == 0) sm.alpha[warp][sm_row] = alpha;
          }
        }
        __syncwarp();
        // ---- acc = alpha * acc + P V on the warp's 8 keys
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          const float al = sm.alpha[warp][r];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[r][e] *= al;
        }
        const uint16_t* Vs = &sm.v[stage][warp * kSlice][0];
#pragma unroll
        for (int i = 0; i < STEPS; ++i) {
          const int key = i * TPW + tl;
          if (t0 + warp * kSlice + key < kv_end) {
            float vf[8];
            unpack8(*reinterpret_cast<const uint4*>(Vs + key * D + c * 8), vf);
            float pr[RM];
#pragma unroll
            for (int r = 0; r < RM; ++r) pr[r] = sm.p[warp][key][r];
#pragma unroll
            for (int r = 0; r < RM; ++r)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pr[r], vf[e], acc[r][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      // the whole consumer group agrees before touching the shared merge buffers
      {
        uint32_t all_ok;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred q, %2, %3, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(all_ok)
            : "r"((uint32_t)alive), "n"(kConsumerBar), "n"(kCThreads)
            : "memory");
        if (!all_ok) { alive = false; break; }
      }

      // ---- merge: keys of the warp (lanes of a chunk), then the eight warps
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
      if (sm_row < RM && lane % LPR == 0) {
        sm.red_m[warp][sm_row] = m_run;
        sm.red_l[warp][sm_row] = l_run;
      }
      named_bar_sync(kConsumerBar, kCThreads);
      if (threadIdx.x < RM) {
        const int r = threadIdx.x;
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) m = fmaxf(m, sm.red_m[w][r]);
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) {
          const float mw = sm.red_m[w][r];
          const float wg = (mw == -INFINITY) ? 0.f : fast_exp2(mw - m);
          sm.wgt[w][r] = wg;
          l += wg * sm.red_l[w][r];
        }
        sm.m_fin[r] = m;
        sm.l_fin[r] = l;
        sm.inv_l[r] = (l > 0.f) ? 1.f / l : 0.f;
      }
      named_bar_sync(kConsumerBar, kCThreads);
      for (int idx = threadIdx.x; idx < nrows * D; idx += kCThreads) {
        const int r = idx / D, d = idx - r * D;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) o = fmaf(sm.wgt[w][r], sm.red[w][r][d], o);
        if (item.part < 0) {
          const int rho = item.row_begin + r;
          const int t = rho / a.g;
          const int h = item.kv_head * a.g + (rho - t * a.g);
          const int64_t off = ((int64_t)(item.q_row0 + t) * a.Hq + h) * D + d;
          o *= sm.inv_l[r];
          if (a.out_bf16)
            reinterpret_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(o);
          else
            reinterpret_cast<float*>(a.out)[off] = o;
        } else {
          const int64_t prow = (int64_t)item.part + r;
          a.part_acc[prow * D + d] = o;
          if (d == 0) {
            a.part_ml[prow * 2 + 0] = sm.m_fin[r];
            a.part_ml[prow * 2 + 1] = sm.l_fin[r];
          }
        }
      }
      named_bar_sync(kConsumerBar, kCThreads);
      item = nitem;
      L = nL;
      ql = nql;
      nitem = nn;
    }
    if (!alive && threadIdx.x == 0) sm.abort_flag = 1;
  }
  __syncthreads();
  // After an abort, give copies still in flight a bounded time to land
  // before the CTA's shared memory is released.
  if (sm.abort_flag && threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      if (sm.issued[s] > sm.consumed[s]) {
        const uint32_t parity = (uint32_t)(sm.issued[s] - 1) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_addr(&sm.full[s]), parity))
          if (global_timer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  }
  pdl_wait();  // exit only after the kernel this one may overlap has completed
}

// Merges the key chunks of split rows: m* = max m_c, l* = sum_c l_c 2^(m_c - m*),
// o = sum_c acc_c 2^(m_c - m*) / l*.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnArgs a,
                                                      const SplitGroup* __restrict__ groups) {
  constexpr int PER = D / 32;
  // the partials of every attention kernel of the call: each of those waits for its
  // predecessor before it exits, so the completion of the last implies all of them
  pdl_wait();
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
                         cudaStream_t s, bool pdl) {
  const int smem = (int)sizeof(DecSmem<D, RM>) + 1024;
  auto* k = a.wait_ns == kWaitLimitNsHost ? decode_kernel<D, RM, false>
                                          : decode_kernel<D, RM, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_kernel(k, grid, kThreads, smem, s, pdl, a, kmap, vmap, items, n_items, box_t);
  if (e != cudaSuccess) return e;
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
                          int grid, cudaStream_t s, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  if (D == 128) {
    if (rows_max <= 1) return launch_dec_t<128, 1>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
    if (rows_max <= 2) return launch_dec_t<128, 2>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
    if (rows_max <= 4) return launch_dec_t<128, 4>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
    return launch_dec_t<128, 8>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
  }
  if (rows_max <= 1) return launch_dec_t<64, 1>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
  if (rows_max <= 2) return launch_dec_t<64, 2>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
  if (rows_max <= 4) return launch_dec_t<64, 4>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
  return launch_dec_t<64, 8>(a, kmap, vmap, items, n_items, box_t, grid, s, pdl);
}

cudaError_t launch_combine(const AttnArgs& a, const SplitGroup* groups, int32_t n_groups, int D,
                           cudaStream_t s, bool pdl) {
  if (n_groups <= 0) return cudaSuccess;
  cudaError_t e = D == 128 ? launch_kernel(combine_kernel<128>, n_groups, 256, 0, s, pdl, a, groups)
                           : launch_kernel(combine_kernel<64>, n_groups, 256, 0, s, pdl, a, groups);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
