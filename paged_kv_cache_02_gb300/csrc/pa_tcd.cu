// pa_tcd.cu -- paged attention for items of at most 16 query rows on the tensor cores.
//
// Same computation as the other attention kernels ("PagedAttention" wiki page,
// "mathematical formulation": softmax of q.k / sqrt(D) over the context, weighted
// sum of v, the keys reached block by block through the block table), for decode-
// like items: one (sequence, KV head) with at most 16 packed rows (query tokens x
// the g query heads of the KV head; GQA packing). A 128-row tile would leave most
// of its rows empty, so this kernel puts the KEYS on the 128-row side:
//     S^T = K Q^T      M = 128 keys,  N = 16 rows, K = D
//     O^T += V^T P^T   M = D = 128,   N = 16 rows, K = 128 keys
// With keys on TMEM lanes, a thread owns one key of the tile: its 16 row scores
// come from one TMEM load, the row maxima and sums are reductions across lanes,
// and the output comes back with one thread per head dimension, so every row is
// stored by 128 consecutive threads.
//
// Warps (6, one persistent CTA per SM):
//   0     TMA producer: the item's 16 query rows (double-buffered across items),
//         K and V tiles of 128 keys into two 3-stage rings with their own barriers
//         (a K stage is free once its S^T is done); one 5-D copy per block piece
//         and tile brings both D halves of the piece's keys.
//   1     MMA issuer: issues whichever of the next S^T (up to two tiles ahead)
//         and the next P V is ready, so neither waits behind the other's data.
//   2-5   softmax: thread = key of the tile (TMEM lane), then = head dimension for
//         the O rescale and the epilogue. P^T goes to shared memory (bf16, the
//         K-major B operand of the second product).
// TMEM: S^T double buffer in columns [0, 32), O^T in [32, 48). Every wait is
// bounded; TMEM loads / stores and whole-warp waits are warp-uniform.
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

constexpr int kKeys = 128;              // keys per tile (M of S^T, K of P V)
constexpr int kD = 128;                 // head dim (M of O^T)
constexpr int kN = kTcdRows;            // query rows per item (N), 16
constexpr int kStages = 3;
constexpr int kThreadsD = 192;
constexpr int kHalf = 128 * 128;        // 128 rows x 64 elements, swizzled (16 KB)
// A K or V tile is 16 groups of 8 keys, 2 KB each: [D half][8 rows x 128 B], every half
// one 128-byte swizzle atom. A block piece is then a run of whole groups, which one TMA
// copy of a 5-D box fills with both D halves (a box of box_t tokens x 256 bytes instead
// of two of 128 bytes per token: twice the bytes per copy, half the copies).
constexpr int kGroup = 2048;            // 8 keys, both D halves
constexpr int kGroupHalf = 1024;        // one D half of a group
constexpr int kQHalf = kN * 128;        // 16 rows x 64 elements (2 KB)
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kColO = 32;

// S^T: A = K tile (K-major), B = Q (K-major). O^T: A = V^T (the V tile read MN-major),
// B = P^T (K-major).
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, kN, false);
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(128, kN, false) | (1u << 15);

struct TcdSmem {
  uint8_t k[kStages][2 * kHalf];        // [stage][group of 8 keys][D half][8 rows]
  uint8_t v[kStages][2 * kHalf];
  uint8_t q[2][2][kQHalf];              // [item parity][D half], 16 rows
  uint8_t p[2][2][kQHalf];              // P^T [tile parity][key half], 16 rows x 64 keys
  float4 red[2][4][kN / 4];             // cross-warp partial maxima / sums [parity][warp][row]
  int bt_cache[2][kBtCache];
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t q_full[2], q_free[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_free[2];
  uint64_t o_tile[2];                   // P V of tiles of this parity done
  uint64_t o_free;                      // the epilogue read O^T
  uint64_t xbar;                        // the 4 softmax warps met (128 arrivals)
  uint64_t drain;
  uint32_t tmem_base;
  int k_issued[kStages], k_consumed[kStages];
  int v_issued[kStages], v_consumed[kStages];
  int q_issued[2], q_consumed[2];
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

// Reduces v[0..NR) over the 32 lanes of the warp with op (max or sum). The first
// log2(NR) steps halve the rows a lane carries (exchanging the other half with the
// lane `o` away), the rest combine whole values; afterwards lane L holds in v[0] the
// result for row (L >> (5 - log2 NR)) & (NR - 1), and the lanes whose low 5 - log2 NR
// bits are zero are the writers (one per row).
template <int NR, bool MAX>
__device__ __forceinline__ void warp_reduce_rows(float (&v)[NR], int lane) {
#pragma unroll
  for (int o = 16, w = NR / 2; w >= 1; o >>= 1, w >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < NR / 2; ++i) {
      if (i < w) {
        const float keep = hi ? v[i + w] : v[i];
        const float give = hi ? v[i] : v[i + w];
        const float got = __shfl_xor_sync(0xffffffffu, give, o);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
    }
  }
#pragma unroll
  for (int o = 32 / NR / 2; o >= 1; o >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], o);
    v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
  }
}

template <int NR>
__device__ __forceinline__ constexpr int log2i() {
  return NR >= 16 ? 4 : NR >= 8 ? 3 : NR >= 4 ? 2 : NR >= 2 ? 1 : 0;
}

// The four warps' partials of rows 0..NR-1 (vector loads, all issued before use),
// combined with op.
template <int NR, bool MAX>
__device__ __forceinline__ void combine4(const float4 (&red)[4][kN / 4], float (&out)[NR]) {
  constexpr int V = (NR + 3) / 4;
  float4 w[4][V];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int c = 0; c < V; ++c) w[q][c] = red[q][c];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 f = w[q][r >> 2];
      e[q] = (r & 3) == 0 ? f.x : (r & 3) == 1 ? f.y : (r & 3) == 2 ? f.z : f.w;
    }
    out[r] = MAX ? fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3])) : (e[0] + e[1]) + (e[2] + e[3]);
  }
}

template <int NR>
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, float (&v)[NR]) {
  if constexpr (NR == 16)
    tc::tmem_ld16(taddr, v);
  else
    tc::tmem_ld_n<NR>(taddr, v);
}

template <int NR>
__device__ __forceinline__ void tmem_st_rows(uint32_t taddr, const float (&v)[NR]) {
  if constexpr (NR == 16)
    tc::tmem_st16(taddr, v);
  else
    tc::tmem_st_n<NR>(taddr, v);
}

// State of one softmax thread across items.
struct SoftmaxThread {
  uint32_t t_lane;  // TMEM address of this warp's lane quadrant
  int quad, lane;
  int kl;           // key in the tile (S^T, P^T) / head dimension (O^T)
  uint32_t x;       // meetings of the four softmax warps so far
  int n;            // tiles of the CTA so far
};

// Meets the other softmax warps: red[x % 2][quad][*] written before, read after.
template <bool kSW>
__device__ __forceinline__ bool meet(TcdSmem& sm, SoftmaxThread& th, const AttnArgs& a) {
  tc::fence_before_sync();
  mbar_arrive(&sm.xbar);
  const bool r = mbar_wait_warp(&sm.xbar, th.x & 1u, a.err, wait_bound<kSW>(a));
  ++th.x;
  tc::fence_after_sync();
  return r;
}

// One item on the softmax warps, for items of at most NR rows: only the first NR
// columns of S^T, P^T and O^T are touched (the others feed output rows that are
// never stored). Returns false if a bounded wait ran out.
template <int NR, bool kSW>
__device__ bool softmax_item(TcdSmem& sm, const AttnArgs& a, const Item& item, int L, int ql,
                             SoftmaxThread& th) {
  constexpr int H = (NR + 1) / 2;            // P^T rows written by the even lane of a pair
  const int nt = tiles_of(item);
  // causal limit of each row (-1: not a row of the item)
  int lim[NR];
  float m_used[NR], l_part[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    lim[r] = r < item.row_count ? min(item.kv_end - 1, L - ql + (item.row_begin + r) / a.g) : -1;
    m_used[r] = -INFINITY;
    l_part[r] = 0.f;
  }
  for (int j = 0; j < nt; ++j, ++th.n) {
    const int n = th.n;
    const int b = n & 1;
    const int key = item.kv_begin + j * kKeys + th.kl;
    // ---- scores of this thread's key for the rows; the buffer is free again after
    float s[NR];
    if (!mbar_wait_warp(&sm.s_full[b], ph(n, 2), a.err, wait_bound<kSW>(a))) return false;
    tc::fence_after_sync();
    tmem_ld_rows<NR>(th.t_lane + (uint32_t)b * kN, s);
    tc::fence_before_sync();
    mbar_arrive(&sm.s_free[b]);
    // causal mask (keys past the range fail it too); a masked score is -inf
#pragma unroll
    for (int r = 0; r < NR; ++r)
      if (key > lim[r]) s[r] = -INFINITY;
    // ---- row maxima over the tile's 128 keys
    {
      float v[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) v[r] = s[r];
      warp_reduce_rows<NR, true>(v, th.lane);
      constexpr int sh = 5 - log2i<NR>();
      if ((th.lane & ((1 << sh) - 1)) == 0)
        reinterpret_cast<float*>(sm.red[th.x & 1][th.quad])[(th.lane >> sh) & (NR - 1)] = v[0];
    }
    const uint32_t xb = th.x & 1;
    if (!meet<kSW>(sm, th, a)) return false;
    float mt[NR];
    combine4<NR, true>(sm.red[xb], mt);
    float alpha[NR];
    bool any_rescale = false;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float m_new = fmaxf(m_used[r], mt[r] * a.scale_log2);
      alpha[r] = 1.f;
      if (m_used[r] == -INFINITY) {
        m_used[r] = m_new;                      // nothing accumulated yet
      } else if (m_new > m_used[r] + kRescaleLog2) {
        alpha[r] = fast_exp2(m_used[r] - m_new);
        m_used[r] = m_new;
        any_rescale = true;
      }
    }
    // every thread saw the same maxima: the decision is uniform across the warps
    if (any_rescale) {
      // O^T must be idle: wait for the previous tile's P V
      if (!mbar_wait_warp(&sm.o_tile[(n - 1) & 1], ph(n - 1, 2), a.err, wait_bound<kSW>(a))) return false;
      tc::fence_after_sync();
      float o[NR];
      tmem_ld_rows<NR>(th.t_lane + kColO, o);
#pragma unroll
      for (int r = 0; r < NR; ++r) o[r] *= alpha[r];
      tmem_st_rows<NR>(th.t_lane + kColO, o);
      tc::tmem_wait_st();
#pragma unroll
      for (int r = 0; r < NR; ++r) l_part[r] *= alpha[r];
    }
    // ---- P^T = 2^(scale s - m): bf16 pairs of neighbouring keys, one row each
    float p[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float neg_m = (m_used[r] == -INFINITY) ? 0.f : -m_used[r];
      p[r] = fast_exp2(fmaf(s[r], a.scale_log2, neg_m));
      l_part[r] += p[r];
    }
    // P^T buffer b is free once the P V of tile n - 2 is done
    if (!mbar_wait_warp(&sm.p_free[b], ph(n, 2) ^ 1u, a.err, wait_bound<kSW>(a))) return false;
    {
      // the even lane of a pair writes rows 0..H-1 for keys (kl, kl + 1), the odd lane
      // rows H..NR-1; K-major, 128-byte swizzle: row r, key k at key half k / 64,
      // 16-byte chunk (k % 64) / 8 ^ (r % 8)
      const bool odd = th.lane & 1;
      const int k0 = th.kl & ~1;
      uint8_t* pb = &sm.p[b][k0 >> 6][0];
      const int kh = k0 & 63;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float give = odd ? p[i] : (H + i < NR ? p[H + i] : 0.f);
        const float got = __shfl_xor_sync(0xffffffffu, give, 1);
        const int r = odd ? H + i : i;
        if (r < NR) {
          const uint32_t w = odd ? pack_bf16(got, p[(H + i) < NR ? H + i : 0])
                                 : pack_bf16(p[i], got);
          const int off = r * 128 + ((((kh >> 3) ^ (r & 7))) << 4) + (kh & 7) * 2;
          *reinterpret_cast<uint32_t*>(pb + off) = w;
        }
      }
    }
    tc::fence_async_shared();
    tc::fence_before_sync();
    mbar_arrive(&sm.p_full[b]);
  }
  // ---- epilogue: row sums across the 128 key positions, then O^T / l with one thread
  // per head dimension (row r of the output is 128 consecutive threads)
  {
    float v[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) v[r] = l_part[r];
    warp_reduce_rows<NR, false>(v, th.lane);
    constexpr int sh = 5 - log2i<NR>();
    if ((th.lane & ((1 << sh) - 1)) == 0)
      reinterpret_cast<float*>(sm.red[th.x & 1][th.quad])[(th.lane >> sh) & (NR - 1)] = v[0];
  }
  const uint32_t xb = th.x & 1;
  if (!meet<kSW>(sm, th, a)) return false;
  float l_row[NR];
  combine4<NR, false>(sm.red[xb], l_row);
  // the item's last P V (its phase is at most one ahead: see the phase bounds)
  const int n_last = th.n - 1;
  if (!mbar_wait_warp(&sm.o_tile[n_last & 1], ph(n_last, 2), a.err, wait_bound<kSW>(a))) return false;
  tc::fence_after_sync();
  float o[NR];
  tmem_ld_rows<NR>(th.t_lane + kColO, o);
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (r < item.row_count) {
      const int rho = item.row_begin + r;
      const int qt = rho / a.g;
      if (item.part < 0) {
        const int h = item.kv_head * a.g + (rho - qt * a.g);
        const int64_t off = ((int64_t)(item.q_row0 + qt) * a.Hq + h) * kD + th.kl;
        const float val = (l_row[r] > 0.f) ? o[r] / l_row[r] : 0.f;
        if (a.out_bf16)
          reinterpret_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(val);
        else
          reinterpret_cast<float*>(a.out)[off] = val;
      } else {
        const int64_t prow = (int64_t)item.part + r;
        a.part_acc[prow * kD + th.kl] = o[r];
        if (th.kl == 0) {
          a.part_ml[prow * 2 + 0] = m_used[r];
          a.part_ml[prow * 2 + 1] = l_row[r];
        }
      }
    }
  }
  tc::fence_before_sync();
  mbar_arrive(&sm.o_free);
  return true;
}

template <bool kSW>
__global__ void __launch_bounds__(kThreadsD, 1)
    tcd_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
               const Item* __restrict__ items, int n_items, int box_t) {
  extern __shared__ uint8_t smem_raw[];
  TcdSmem& sm = *reinterpret_cast<TcdSmem*>(align1024(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
      sm.k_issued[s] = sm.k_consumed[s] = 0;
      sm.v_issued[s] = sm.v_consumed[s] = 0;
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_free[b], 1);
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 128);
      mbar_init(&sm.p_full[b], 128);
      mbar_init(&sm.p_free[b], 1);
      mbar_init(&sm.o_tile[b], 1);
      sm.q_issued[b] = 0;
      sm.q_consumed[b] = 0;
    }
    mbar_init(&sm.o_free, 128);
    mbar_init(&sm.xbar, 128);
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
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      prefetch_tensormap(&qmap);
    }
    const int pieces = kKeys / box_t;
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
      // the item's 16 query rows: tokens x the g heads of its KV head, one box per D
      // half. Buffer k % 2 is free once the issuer issued every S^T of item k - 2.
      {
        const int qb = k & 1;
        ok = mbar_wait_warp(&sm.q_free[qb], ph(k, 2) ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.q_full[qb], 2u * kQHalf);
          const int tok = item.q_row0 + item.row_begin / a.g;
          tma_load_3d(&sm.q[qb][0][0], &qmap, &sm.q_full[qb], 0, item.kv_head * a.g, tok);
          tma_load_3d(&sm.q[qb][1][0], &qmap, &sm.q_full[qb], 64, item.kv_head * a.g, tok);
          sm.q_issued[qb] += 1;
        }
        __syncwarp();
      }
      // Fused KV write (vLLM-SOSP23 note, kernel layer: the new tokens' reshape and block
      // write fused with the attention that reads them): the item's new tokens -- the
      // sequence's query tokens whose positions fall in its key range -- are copied to
      // their slots for this KV head, 16-byte vectors spread over the lanes. They are
      // read only by this item (no other item of the call covers these positions of
      // this KV head), so ordering the copies before the TMA loads of the tile that
      // holds them is enough: a proxy fence by every writing lane, then the warp
      // barrier, before that tile is issued.
      int first_new = item.kv_end;               // first position this item wrote
      if (a.k_new != nullptr) {
        const int L = __ldg(a.context_lens + item.seq);
        const int ql = __ldg(a.query_lens + item.seq);
        const int p0 = max(item.kv_begin, L - ql), p1 = min(item.kv_end, L);
        if (p0 < p1) {
          first_new = p0;
          const int64_t vec_row = (int64_t)a.Hkv * (kD / 8);   // 16-byte vectors per token
          const int64_t head_off = (int64_t)item.kv_head * (kD / 8);
          const int64_t row0 = (int64_t)item.q_row0 + (p0 - (L - ql));
          for (int v = lane; v < (p1 - p0) * (kD / 8); v += 32) {
            const int64_t row = row0 + v / (kD / 8);
            const int c = v % (kD / 8);
            const int64_t slot = __ldg(a.slots + row);
            if (slot >= a.n_slots) {
              record_error(a.err, PA_DEVERR_SLOT_RANGE);
            } else if (slot >= 0) {
              const int64_t from = row * vec_row + head_off + c;
              const int64_t to = slot * vec_row + head_off + c;
              const uint4 kx = __ldg(a.k_new + from), vx = __ldg(a.v_new + from);
              a.k_pool[to] = kx;
              a.v_pool[to] = vx;
            }
          }
        }
      }
      bool fence_due = first_new < item.kv_end;
      const int32_t* bt = a.block_table + (int64_t)item.seq * a.max_blocks;
      for (int t0 = item.kv_begin; t0 < item.kv_end; t0 += kKeys, ++n) {
        const int st = n % kStages;
        if (fence_due && t0 + kKeys > first_new) {
          // the generic-proxy copies above, before the async-proxy (TMA) reads below
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __syncwarp();
          fence_due = false;
        }
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
        const uint32_t piece_off = (uint32_t)lane * box_t * 256u;  // whole groups
        // K_n: its stage is free once S^T of tile n - 3 is done
        ok = mbar_wait_warp(&sm.k_empty[st], ph(n, kStages) ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&sm.k_full[st], tile_bytes);
        __syncwarp();
        if (valid)
          tma_load_5d(&sm.k[st][piece_off], &kmap, &sm.k_full[st], 0, 0, 0, tok >> 3, item.kv_head);
        if (lane == 0) sm.k_issued[st] += 1;
        // V_n: free once P V of tile n - 3 is done
        ok = mbar_wait_warp(&sm.v_empty[st], ph(n, kStages) ^ 1u, a.err, wait_bound<kSW>(a));
        if (!ok || *(volatile int*)&sm.abort_flag) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&sm.v_full[st], tile_bytes);
        __syncwarp();
        if (valid)
          tma_load_5d(&sm.v[st][piece_off], &vmap, &sm.v_full[st], 0, 0, 0, tok >> 3, item.kv_head);
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
    // ------------------------------------------------------------ MMA issuer
    // An event loop over two cursors: the next S^T (at most two tiles ahead of P V, one
    // per S^T buffer) and the next P V, each issued as soon as its barriers show it is
    // ready. Phase bounds: k_full / v_full of tile n + 3 need S^T / P V of tile n;
    // s_free / p_full of tile n + 2 need the softmax of tile n + 2, which needs
    // s_full(n + 2) from here; q_full of item k + 2 needs q_free(k) from here; o_free
    // of item k + 1 needs the P V of item k + 1. So every check below looks at the
    // phase it means.
    if (lane == 0) {
      bool ok = true;
      // S^T cursor: item index it_s, the CTA's k_s-th item, its tile j_s, CTA tile n_s
      // (each cursor holds its next item already loaded, so that an item switch does
      // not wait for a global load)
      int it_s = blockIdx.x, k_s = 0, j_s = 0, n_s = 0;
      int nt_s = it_s < n_items ? tiles_of(items[it_s]) : 0;
      int nt_s_next = it_s + G < n_items ? tiles_of(items[it_s + G]) : 0;
      uint64_t qd = 0;
      // P V cursor
      int it_p = blockIdx.x, k_p = 0, j_p = 0, n_p = 0;
      Item item_p = it_p < n_items ? items[it_p] : Item{};
      Item item_p_next = it_p + G < n_items ? items[it_p + G] : Item{};
      int nt_p = it_p < n_items ? tiles_of(item_p) : 0;
      uint64_t t_idle = global_timer_ns();
      while (it_p < n_items) {
        bool progress = false;
        if (it_s < n_items && n_s < n_p + 2) {
          const int st = n_s % kStages;
          const int b = n_s & 1;
          if ((j_s > 0 || mbar_try_wait(smem_addr(&sm.q_full[k_s & 1]), ph(k_s, 2))) &&
              mbar_try_wait(smem_addr(&sm.k_full[st]), ph(n_s, kStages)) &&
              mbar_try_wait(smem_addr(&sm.s_free[b]), ph(n_s, 2) ^ 1u)) {
            if (j_s == 0) {
              sm.q_consumed[k_s & 1] += 1;
              qd = tc::smem_desc_sw128(smem_addr(&sm.q[k_s & 1][0][0]), 16, 1024);
            }
            sm.k_consumed[st] += 1;
            tc::fence_after_sync();
            // S^T = K Q^T: 8 steps of 16 dims; step kk starts (kk % 4) 32-byte chunks into
            // D half kk / 4 of both operands (K's 8-row groups are kGroup apart, its
            // halves kGroupHalf; Q's halves kQHalf)
            const uint64_t kd = tc::smem_desc_sw128(smem_addr(&sm.k[st][0]), 16, kGroup);
            tc::mma_bf16_c<false>(tmem + (uint32_t)b * kN, kd, qd, kIdescS);
#pragma unroll
            for (int kk = 1; kk < kD / 16; ++kk) {
              const uint64_t ko = (uint64_t)(((kk >> 2) * kGroupHalf + (kk & 3) * 32) >> 4);
              const uint64_t qo = (uint64_t)(((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4);
              tc::mma_bf16_c<true>(tmem + (uint32_t)b * kN, kd + ko, qd + qo, kIdescS);
            }
            tc::commit(&sm.s_full[b]);
            tc::commit(&sm.k_empty[st]);
            if (j_s + 1 == nt_s) tc::commit(&sm.q_free[k_s & 1]);  // the item's last S^T
            ++n_s;
            if (++j_s == nt_s) {
              j_s = 0;
              ++k_s;
              it_s += G;
              nt_s = nt_s_next;
              nt_s_next = it_s + G < n_items ? tiles_of(items[it_s + G]) : 0;
            }
            progress = true;
          }
        }
        if (n_p < n_s) {
          const int st = n_p % kStages;
          const int b = n_p & 1;
          // at an item's first tile, O^T must have been read out by the previous epilogue
          if (mbar_try_wait(smem_addr(&sm.p_full[b]), ph(n_p, 2)) &&
              (j_p > 0 || mbar_try_wait(smem_addr(&sm.o_free), ((uint32_t)k_p & 1u) ^ 1u)) &&
              mbar_try_wait(smem_addr(&sm.v_full[st]), ph(n_p, kStages))) {
            sm.v_consumed[st] += 1;
            // Keys of the tile in the item's range, rounded up to the 16-key step: only
            // those V rows are read. At the item's last tile, the rows between the
            // range's end and that step hold whatever the block tail holds: zero them (at
            // most 15) so that 0 * (non-finite) never reaches O.
            const int key0 = item_p.kv_begin + j_p * kKeys;
            const int valid = min(kKeys, item_p.kv_end - key0);
            const int kk_end = (valid + 15) >> 4;
            if (valid < kk_end * 16) {
              for (int r = valid; r < kk_end * 16; ++r) {
                uint4* v0 = reinterpret_cast<uint4*>(&sm.v[st][(r >> 3) * kGroup + (r & 7) * 128]);
                uint4* v1 = v0 + kGroupHalf / 16;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  v0[q] = make_uint4(0, 0, 0, 0);
                  v1[q] = make_uint4(0, 0, 0, 0);
                }
              }
              tc::fence_async_shared();
            }
            tc::fence_after_sync();
            // O^T += V^T P^T: step kk covers keys 16 kk .. 16 kk + 15: two 8-key groups of
            // V (the MN-major A operand: D halves kGroupHalf apart, groups kGroup) and P^T
            // columns (K-major B, key halves kQHalf apart)
            const uint64_t vd =
                tc::smem_desc_sw128(smem_addr(&sm.v[st][0]), kGroupHalf, kGroup);
            const uint64_t pd = tc::smem_desc_sw128(smem_addr(&sm.p[b][0][0]), 16, 1024);
            if (j_p > 0)
              tc::mma_bf16_c<true>(tmem + kColO, vd, pd, kIdescO);
            else
              tc::mma_bf16_c<false>(tmem + kColO, vd, pd, kIdescO);
#pragma unroll
            for (int kk = 1; kk < kKeys / 16; ++kk) {
              if (kk < kk_end) {
                const uint64_t vo = (uint64_t)((kk * 2 * kGroup) >> 4);
                const uint64_t po = (uint64_t)(((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4);
                tc::mma_bf16_c<true>(tmem + kColO, vd + vo, pd + po, kIdescO);
              }
            }
            tc::commit(&sm.v_empty[st]);
            tc::commit(&sm.p_free[b]);
            tc::commit(&sm.o_tile[b]);
            ++n_p;
            if (++j_p == nt_p) {
              j_p = 0;
              ++k_p;
              it_p += G;
              if (it_p < n_items) {
                item_p = item_p_next;
                nt_p = tiles_of(item_p);
                if (it_p + G < n_items) item_p_next = items[it_p + G];
              }
            }
            progress = true;
          }
        }
        if (progress) {
          t_idle = global_timer_ns();
        } else if (global_timer_ns() - t_idle > wait_bound<kSW>(a)) {
          record_error(a.err, PA_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        if (*(volatile int*)&sm.abort_flag) { ok = false; break; }
      }
      if (!ok) sm.abort_flag = 1;
      tc::commit(&sm.drain);
      mbar_wait(&sm.drain, 0, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    // Thread = key of the tile (TMEM lane quad * 32 + lane) for S^T and P^T, and =
    // head dimension for O^T. The four warps meet on an mbarrier of 128 arrivals
    // (bounded wait) to combine their partial row maxima / sums in shared memory;
    // meeting x uses buffer x % 2, and a warp cannot write it again before the other
    // warps passed meeting x + 1, i.e. read meeting x. Each item runs the variant for
    // the smallest of 1, 2, 4, 8, 16 rows that holds it.
    // Phase bounds: s_full(n + 2) needs s_free(n) from here; p_free(n + 2) needs
    // p_full(n + 2); o_tile(n + 1) needs p_full(n + 1); so no barrier is ever two
    // phases ahead of a wait here.
    SoftmaxThread th;
    th.quad = warp & 3;
    th.lane = lane;
    th.kl = th.quad * 32 + lane;
    th.t_lane = tmem + ((uint32_t)(th.quad * 32) << 16);
    th.x = 0;
    th.n = 0;
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
    for (int it = blockIdx.x; it < n_items && ok; it += G) {
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
      const int rc = item.row_count;
      if (rc <= 1)
        ok = softmax_item<1, kSW>(sm, a, item, L, ql, th);
      else if (rc <= 2)
        ok = softmax_item<2, kSW>(sm, a, item, L, ql, th);
      else if (rc <= 4)
        ok = softmax_item<4, kSW>(sm, a, item, L, ql, th);
      else if (rc <= 8)
        ok = softmax_item<8, kSW>(sm, a, item, L, ql, th);
      else
        ok = softmax_item<16, kSW>(sm, a, item, L, ql, th);
    }
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
  pdl_wait();  // exit only after the kernel this one may overlap has completed
}

}  // namespace

int tcd_smem_bytes() { return (int)sizeof(TcdSmem) + 1024; }

cudaError_t launch_tcd(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const CUtensorMap& qmap, const Item* items, int32_t n_items, int box_t,
                       int grid, cudaStream_t s, bool pdl) {
  if (n_items <= 0) return cudaSuccess;
  const int smem = tcd_smem_bytes();
  auto* k = a.wait_ns == kWaitLimitNsHost ? tcd_kernel<false> : tcd_kernel<true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_kernel(k, grid, kThreadsD, smem, s, pdl, a, kmap, vmap, qmap, items, n_items,
                    box_t);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
