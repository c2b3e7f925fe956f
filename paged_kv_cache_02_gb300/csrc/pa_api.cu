// pa_api.cu -- the C ABI: argument checks, the host plan, tensor maps, launches.
//
// The plan is the auxiliary data Pensieve computes on the CPU (Pensieve summary,
// kernel microbenchmark): the batch's (sequence, KV head) pairs cut into work
// items, each item a range of packed rows (query tokens x the query heads of one
// KV head) against a range of keys. Items with many rows go to the tensor-core
// kernel, the rest to the CUDA-core kernel; long key ranges are split so that
// every SM has work (split-KV), and the split rows are merged by a combine pass.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <utility>
#include <atomic>
#include <cmath>
#include <mutex>
#include <new>
#include <vector>

#include "pa_internal.h"

namespace pa {

// ------------------------------------------------------------------ error word
// One word per device (plus spare room), written by kernels with atomicCAS.
__device__ int g_error_word[4];

int* device_error_word() {
  static std::mutex mu;
  static int* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(p);
  }
  return cache[dev];
}

int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (dev < 0 || dev >= 64) return 0;
  int sms = cache[dev].load(std::memory_order_relaxed);
  if (sms > 0) return sms;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// ------------------------------------------------------------------ tensor maps
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

pa_status make_pool_map(CUtensorMap* map, const void* pool, int64_t num_blocks, int block_size,
                        int Hkv, int D, int box_d, int box_t, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)(num_blocks * block_size)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_t};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

pa_status make_pool_map_grouped(CUtensorMap* map, const void* pool, int64_t num_blocks,
                                int block_size, int Hkv, int box_t) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  constexpr int D = 128;
  // dims: 64 elements of a D half, 8 tokens, the 2 D halves, groups of 8 tokens, heads
  cuuint64_t dims[5] = {64u, 8u, 2u, (cuuint64_t)(num_blocks * block_size / 8),
                        (cuuint64_t)Hkv};
  cuuint64_t strides[4] = {(cuuint64_t)Hkv * D * 2, 128u, (cuuint64_t)8 * Hkv * D * 2,
                           (cuuint64_t)D * 2};
  cuuint32_t box[5] = {64u, 8u, 2u, (cuuint32_t)(box_t / 8), 1u};
  cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(pool), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

pa_status make_q_map(CUtensorMap* map, const void* q, int64_t total_q, int Hq, int D, int g,
                     int rows) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)total_q};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)g, (cuuint32_t)(rows / g)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

pa_status make_out_map(CUtensorMap* map, void* out, int64_t total_q, int Hq, int D, int g,
                       bool bf16) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const int es = bf16 ? 2 : 4;
  const int gb = g < 32 ? g : 32;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)total_q};
  cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)Hq * D * es};
  cuuint32_t box[3] = {16u, (cuuint32_t)gb, (cuuint32_t)(32 / gb)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  bf16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

// ====================================================================== plan

struct pa_plan_s {
  int32_t num_seqs, Hq, Hkv, D, block_size, max_blocks, g;
  int64_t total_q;
  int32_t n_dec, n_tc, n_tc2, n_tcd, n_groups;
  int32_t dec_rows_max;
  uint64_t wait_ns;         // bound on each pipeline wait of the kernels
  int64_t n_part_rows;
  int32_t chunk;
  int64_t kv_tokens;
  // workspace layout (byte offsets)
  size_t off_dec, off_tc, off_tc2, off_tcd, off_groups, off_wmask, off_acc, off_ml, ws_bytes;
  int64_t n_fused_rows;     // rows whose K/V the key-major kernel writes in a fused call
  bool wmask;               // the tables hold a per-row byte: 1 = written in that kernel
  size_t table_bytes;       // bytes of the item / group tables (copied each call)
  void* host_tables;        // table image: [dec][tc][tc pair items][groups] at their offsets
  bool host_pinned;
  size_t host_cap;          // bytes of the pinned buffer (>= table_bytes)
  cudaEvent_t upload_ev;    // recorded after each upload of the tables (pinned only)
  bool upload_recorded;
  bool host_reusable;       // every upload is covered by upload_ev
};

namespace {

using pa::Item;
using pa::SplitGroup;

// Pinned host buffers of destroyed plans, kept for the next plans: a serving loop creates
// and destroys a plan every step, and page-locking fresh memory costs more than building
// the plan (about 0.27 ms per allocate + free pair on the GB300's Grace host). A buffer
// is reused only once the last copy from it has completed (its upload event).
struct PinnedBuf {
  void* ptr;
  size_t cap;
  cudaEvent_t ev;
  bool recorded;
};
std::mutex g_pinned_mu;
std::vector<PinnedBuf> g_pinned_free;
constexpr size_t kPinnedCacheMax = 8;

bool pinned_take(size_t bytes, PinnedBuf* out) {
  std::lock_guard<std::mutex> lock(g_pinned_mu);
  int best = -1;
  for (size_t i = 0; i < g_pinned_free.size(); ++i) {
    const PinnedBuf& b = g_pinned_free[i];
    if (b.cap < bytes || (best >= 0 && b.cap >= g_pinned_free[best].cap)) continue;
    if (b.recorded && cudaEventQuery(b.ev) != cudaSuccess) continue;  // copy in flight
    best = (int)i;
  }
  if (best < 0) return false;
  *out = g_pinned_free[best];
  out->recorded = false;
  g_pinned_free.erase(g_pinned_free.begin() + best);
  return true;
}

void pinned_give(const PinnedBuf& b) {
  {
    std::lock_guard<std::mutex> lock(g_pinned_mu);
    if (g_pinned_free.size() < kPinnedCacheMax) {
      g_pinned_free.push_back(b);
      return;
    }
  }
  if (b.recorded) cudaEventSynchronize(b.ev);
  cudaFreeHost(b.ptr);
  if (b.ev) cudaEventDestroy(b.ev);
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int device_sms() { return pa::sm_count(); }

// Kernel a work item runs on (the path number pa_plan_export reports).
enum Path : int { kPathDec = 0, kPathTc = 1, kPathTcPair = 2, kPathTcDecode = 3 };

struct Unit {
  int32_t seq, kvh, row_begin, row_count, keys, q_row0;
  int path;
};

}  // namespace

// The new tokens' K/V of a fused write + attention call (null: attention only).
struct FusedWrite {
  const void* k_new;       // [total_q, Hkv, D] bf16, device
  const void* v_new;
  const int64_t* slots;    // [total_q], device
};

static pa_status attention_impl(pa_plan_t p, void* d_out, pa_dtype out_dtype, const void* d_q,
                                const void* d_k_pool, const void* d_v_pool,
                                const int32_t* d_block_table, const int32_t* d_context_lens,
                                const int32_t* d_query_lens, int32_t num_blocks, float scale,
                                void* d_workspace, size_t workspace_bytes, void* stream,
                                bool upload, const FusedWrite* fw = nullptr);

// Marks the stream position after a copy from the plan's pinned table buffer, so that the
// buffer is handed to a later plan only once the copy has completed.
static pa_status note_upload(pa_plan_t p, cudaStream_t s) {
  if (!p->host_pinned) return PA_OK;
  if (!p->upload_ev &&
      cudaEventCreateWithFlags(&p->upload_ev, cudaEventDisableTiming) != cudaSuccess) {
    p->upload_ev = nullptr;
    p->host_reusable = false;
    return PA_ERR_CUDA;
  }
  if (cudaEventRecord(p->upload_ev, s) != cudaSuccess) {
    p->host_reusable = false;
    return PA_ERR_CUDA;
  }
  p->upload_recorded = true;
  return PA_OK;
}

namespace pa {
// Whole blocks from pool (k_from, v_from) to pool (k_to, v_to), defined in pa_kv.cu:
// either side may be the device mapping of page-locked host memory.
cudaError_t launch_swap_blocks(const void* k_from, const void* v_from, void* k_to, void* v_to,
                               const int32_t* src, const int32_t* dst, int32_t n_pairs,
                               int32_t n_from, int32_t n_to, int64_t block_bytes, int* err,
                               cudaStream_t s);
}  // namespace pa

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_SHAPE: return "inconsistent shapes";
    case PA_ERR_RANGE: return "value out of range";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_TIMEOUT: return "bounded device wait ran out";
    case PA_ERR_NO_SPACE: return "too few free blocks in the pool";
  }
  return "unknown status";
}

const char* pa_version(void) { return "pa 0.1 sm_103a"; }

pa_status pa_get_device_error(int32_t* code, int32_t reset, void* stream) {
  if (!code) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, pa::g_error_word, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
  *code = v;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(pa::g_error_word, &zero, sizeof(int)) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return PA_OK;
}

pa_status pa_slot_mapping(const int32_t* d_block_table, int32_t num_seqs,
                          int32_t max_blocks_per_seq, int32_t block_size, int32_t num_blocks,
                          const int32_t* d_seq_ids, const int32_t* d_positions, int64_t n,
                          int64_t* d_slots, void* stream) {
  if (n < 0 || num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (n == 0) return PA_OK;
  if (!d_block_table || !d_seq_ids || !d_positions || !d_slots) return PA_ERR_INVALID_ARG;
  int* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  cudaError_t e = pa::launch_slot_mapping(d_block_table, num_seqs, max_blocks_per_seq, block_size,
                                          num_blocks, d_seq_ids, d_positions, n, d_slots, err,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_write_kv(const void* d_k_new, const void* d_v_new, const int64_t* d_slot_mapping,
                      int64_t n_new, void* d_k_pool, void* d_v_pool, int32_t num_blocks,
                      int32_t block_size, int32_t Hkv, int32_t D, void* stream) {
  if (n_new < 0 || num_blocks <= 0 || block_size <= 0 || Hkv <= 0 || D <= 0)
    return PA_ERR_INVALID_ARG;
  if (n_new == 0) return PA_OK;
  if (!d_k_new || !d_v_new || !d_slot_mapping || !d_k_pool || !d_v_pool) return PA_ERR_INVALID_ARG;
  if (D % 8) return PA_ERR_UNSUPPORTED;
  for (const void* p : {d_k_new, d_v_new, (const void*)d_k_pool, (const void*)d_v_pool})
    if (reinterpret_cast<uintptr_t>(p) % 16) return PA_ERR_UNSUPPORTED;
  int* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t row_bytes = (int64_t)Hkv * D * 2;
  cudaError_t e = pa::launch_write_kv(d_k_new, d_v_new, d_slot_mapping, n_new, d_k_pool, d_v_pool,
                                      (int64_t)num_blocks * block_size, row_bytes, err,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(void* d_k_pool, void* d_v_pool, const int32_t* d_src,
                         const int32_t* d_dst, int32_t n_pairs, int32_t num_blocks,
                         int32_t block_size, int32_t Hkv, int32_t D, void* stream) {
  if (n_pairs < 0 || num_blocks <= 0 || block_size <= 0 || Hkv <= 0 || D <= 0)
    return PA_ERR_INVALID_ARG;
  if (n_pairs == 0) return PA_OK;
  if (!d_k_pool || !d_v_pool || !d_src || !d_dst) return PA_ERR_INVALID_ARG;
  if (D % 8) return PA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(d_k_pool) % 16 || reinterpret_cast<uintptr_t>(d_v_pool) % 16)
    return PA_ERR_UNSUPPORTED;
  int* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t block_bytes = (int64_t)block_size * Hkv * D * 2;
  cudaError_t e = pa::launch_copy_blocks(d_k_pool, d_v_pool, d_src, d_dst, n_pairs, num_blocks,
                                         block_bytes, err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Device view of `bytes` of page-locked host memory at h: both ends must lie in memory
// that CUDA has mapped (cudaHostAlloc, or cudaHostRegister with mapping), contiguously.
static bool host_device_view(void* h, int64_t bytes, void** d) {
  cudaPointerAttributes a0, a1;
  if (cudaPointerGetAttributes(&a0, h) != cudaSuccess ||
      cudaPointerGetAttributes(&a1, static_cast<char*>(h) + (bytes - 1)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a0.type != cudaMemoryTypeHost || a1.type != cudaMemoryTypeHost || !a0.devicePointer ||
      !a1.devicePointer)
    return false;
  if (static_cast<char*>(a1.devicePointer) - static_cast<char*>(a0.devicePointer) != bytes - 1)
    return false;
  *d = a0.devicePointer;
  return true;
}

pa_status pa_swap_blocks(void* d_k_pool, void* d_v_pool, int32_t num_blocks, void* h_k_pool,
                         void* h_v_pool, int32_t num_host_blocks, const int32_t* d_src,
                         const int32_t* d_dst, int32_t n_pairs, int32_t block_size, int32_t Hkv,
                         int32_t D, int32_t direction, void* stream) {
  if (n_pairs < 0 || num_blocks <= 0 || num_host_blocks <= 0 || block_size <= 0 || Hkv <= 0 ||
      D <= 0 || (direction != PA_SWAP_OUT && direction != PA_SWAP_IN))
    return PA_ERR_INVALID_ARG;
  if (n_pairs == 0) return PA_OK;
  if (!d_k_pool || !d_v_pool || !h_k_pool || !h_v_pool || !d_src || !d_dst)
    return PA_ERR_INVALID_ARG;
  if (D % 8) return PA_ERR_UNSUPPORTED;
  for (const void* ptr : {(const void*)d_k_pool, (const void*)d_v_pool, (const void*)h_k_pool,
                          (const void*)h_v_pool})
    if (reinterpret_cast<uintptr_t>(ptr) % 16) return PA_ERR_UNSUPPORTED;
  const int64_t block_bytes = (int64_t)block_size * Hkv * D * 2;
  void* hk = nullptr;
  void* hv = nullptr;
  if (!host_device_view(h_k_pool, (int64_t)num_host_blocks * block_bytes, &hk) ||
      !host_device_view(h_v_pool, (int64_t)num_host_blocks * block_bytes, &hv))
    return PA_ERR_INVALID_ARG;
  int* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      direction == PA_SWAP_OUT
          ? pa::launch_swap_blocks(d_k_pool, d_v_pool, hk, hv, d_src, d_dst, n_pairs,
                                   num_blocks, num_host_blocks, block_bytes, err, s)
          : pa::launch_swap_blocks(hk, hv, d_k_pool, d_v_pool, d_src, d_dst, n_pairs,
                                   num_host_blocks, num_blocks, block_bytes, err, s);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_plan_create(const int32_t* h_context_lens, const int32_t* h_query_lens,
                         int32_t num_seqs, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t block_size, int32_t max_blocks_per_seq,
                         const pa_plan_options* opts, pa_plan_t* out, size_t* workspace_bytes) {
  if (!out || !workspace_bytes) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!h_context_lens || !h_query_lens)) return PA_ERR_INVALID_ARG;
  if (Hq % Hkv) return PA_ERR_SHAPE;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(block_size) || block_size > 256) return PA_ERR_UNSUPPORTED;
  pa_plan_options o;
  memset(&o, 0, sizeof o);
  if (opts) {
    o = *opts;
    for (int i = 0; i < 2; ++i)
      if (o.reserved[i]) return PA_ERR_INVALID_ARG;
    if (o.wait_limit_ns < 0) return PA_ERR_INVALID_ARG;
  }
  const int g = Hq / Hkv;
  int64_t total_q = 0, kv_tokens = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t L = h_context_lens[s], q = h_query_lens[s];
    if (L < 0 || q < 0 || q > L) return PA_ERR_RANGE;
    if (((int64_t)L + block_size - 1) / block_size > max_blocks_per_seq) return PA_ERR_RANGE;
    total_q += q;
    kv_tokens += L;
  }
  if (total_q * Hq > INT32_MAX || (int64_t)Hq * g > INT32_MAX) return PA_ERR_UNSUPPORTED;

  int sms = o.num_sms > 0 ? o.num_sms : device_sms();
  if (sms <= 0) sms = 152;
  // Tensor-core tiles: D = 128, blocks of at least 8 tokens (one swizzle atom per piece) and
  // g dividing the 128-row tile (a tile is whole tokens x the g heads of one KV head).
  const bool tc_enabled = (D == 128) && (block_size >= 8) && (pa::kTcRows % g == 0) &&
                          o.tc_min_rows >= 0;
  const bool pair_enabled = tc_enabled && o.tc_pair >= 0;
  // (sequence, KV head) pairs with at most 16 rows: keys on the 128-row side
  const bool tcd_enabled = tc_enabled && (pa::kTcdRows % g == 0) && o.tc_decode >= 0;
  // by default every row count goes to the tensor cores when the key-major kernel takes
  // the small ones; otherwise pairs with fewer than kTcMinRowsDefault rows stay on the
  // CUDA cores
  const int tc_min_rows =
      o.tc_min_rows > 0 ? o.tc_min_rows : (tcd_enabled ? 1 : pa::kTcMinRowsDefault);
  // 256-row items (two query tiles sharing every K/V tile) read half the K/V bytes per
  // query row of 128-row items; 128-row items pipeline better (a CTA keeps two score
  // buffers and eight softmax warps for one tile). By default pairs are used when the
  // multi-token tensor-core work of the batch is memory-bound: fewer FLOPs per byte of
  // K/V (read once per sequence and KV head), Q and output than the machine balance.
  bool use_pair = pair_enabled && o.tc_pair > 0;
  if (pair_enabled && o.tc_pair == 0) {
    double flops = 0.0, bytes = 0.0;
    for (int32_t s = 0; s < num_seqs; ++s) {
      const double L = h_context_lens[s], q = h_query_lens[s];
      const int64_t rows = (int64_t)h_query_lens[s] * g;
      if (rows < tc_min_rows || (tcd_enabled && rows <= pa::kTcdRows)) continue;
      // causal: query token t (0-based among the q) sees L - q + t + 1 keys
      const double keys = q * (L - q) + q * (q + 1) / 2;
      flops += 4.0 * D * g * Hkv * keys;                // Q K^T and P V
      bytes += 4.0 * D * Hkv * L + 6.0 * D * Hq * q;    // K + V bf16, Q bf16, O fp32
    }
    use_pair = flops < pa::kTcMachineBalance * bytes;
  }

  // ---- units: (sequence, KV head, row tile). With pairs, tensor-core rows go in tiles
  // of 256 (two 128-row halves sharing every K/V tile), without in tiles of 128. A
  // sequence's rows that do not fill whole tiles form its FIRST tile, not its last: the
  // rows are causal, so the first rows see the fewest keys, and the partial tile (which
  // costs a whole tile's K/V reads and MMAs per key) then runs over the shortest key
  // range. Of n full tiles and r rows left over this reads n (T - r) keys fewer than
  // putting the partial tile last (T the tile's rows; g = 1) -- for a sub-request that
  // recomputes a context's leading tokens, about a third of its keys.
  std::vector<Unit> units;
  std::vector<std::pair<int64_t, int32_t>> fused_runs;  // (first row, rows): key-major seqs
  int64_t n_fused_rows = 0;
  int64_t total_keys = 0;
  int64_t q_row0 = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t L = h_context_lens[s], q = h_query_lens[s];
    if (q > 0) {
      const int64_t rows = (int64_t)q * g;
      const bool tc = tc_enabled && rows >= tc_min_rows;
      if (tc && tcd_enabled && rows <= pa::kTcdRows) {
        fused_runs.push_back({q_row0, q});
        n_fused_rows += q;
      }
      const bool multi = tc && !(tcd_enabled && rows <= pa::kTcdRows);
      const int64_t tile = use_pair ? 2 * pa::kTcRows : pa::kTcRows;
      // rows of the leading partial tile (multiple of g, since tile is)
      const int64_t lead = multi ? rows % tile : 0;
      for (int32_t kvh = 0; kvh < Hkv; ++kvh) {
        for (int64_t rb = 0; rb < rows;) {
          const int64_t left = rows - rb;
          int path, rt;
          if (!tc) {
            path = kPathDec; rt = pa::kDecRows;
          } else if (!multi) {
            path = kPathTcDecode; rt = pa::kTcdRows;
          } else {
            rt = (rb == 0 && lead > 0) ? (int)lead : (int)tile;
            path = rt > pa::kTcRows ? kPathTcPair : kPathTc;
          }
          const int32_t rc = (int32_t)std::min<int64_t>(rt, left);
          const int32_t t_last = (int32_t)((rb + rc - 1) / g);
          const int32_t keys = L - q + t_last + 1;
          units.push_back({s, kvh, (int32_t)rb, rc, keys, (int32_t)q_row0, path});
          total_keys += keys;
          rb += rc;
        }
      }
    }
    q_row0 += q;
  }
  // ---- split-KV chunk length
  int64_t chunk;
  if (o.max_chunk_tokens > 0) {
    chunk = align_up((size_t)o.max_chunk_tokens, pa::kChunkAlign);
  } else {
    // about three items per SM over the whole batch, never below 256 keys
    chunk = std::max<int64_t>(256, align_up((size_t)(total_keys / (3 * (int64_t)sms) + 1),
                                            pa::kChunkAlign));
  }
  std::vector<Item> dec, tc, tc2, tcd;
  std::vector<SplitGroup> groups;
  int64_t part_rows = 0;
  int32_t dec_rows_max = 1;
  bool any_split = false;
  for (const Unit& u : units) {
    const int64_t n_chunks = (u.keys + chunk - 1) / chunk;
    std::vector<Item>& dst = u.path == kPathDec ? dec
                             : u.path == kPathTc ? tc
                             : u.path == kPathTcPair ? tc2
                                                     : tcd;
    if (u.path == kPathDec) dec_rows_max = std::max(dec_rows_max, u.row_count);
    if (n_chunks <= 1) {
      dst.push_back({u.seq, u.kvh, u.row_begin, u.row_count, 0, u.keys, -1, u.q_row0});
    } else {
      any_split = true;
      if (part_rows + n_chunks * u.row_count > INT32_MAX) return PA_ERR_UNSUPPORTED;
      groups.push_back({u.seq, u.kvh, u.row_begin, u.row_count, (int32_t)part_rows,
                        (int32_t)n_chunks, u.q_row0, 0});
      for (int64_t c = 0; c < n_chunks; ++c) {
        const int32_t kb = (int32_t)(c * chunk);
        const int32_t ke = (int32_t)std::min<int64_t>((c + 1) * chunk, u.keys);
        dst.push_back({u.seq, u.kvh, u.row_begin, u.row_count, kb, ke,
                       (int32_t)(part_rows + c * u.row_count), u.q_row0});
      }
      part_rows += n_chunks * u.row_count;
    }
  }
  // Longest key range first, then every other round of G items (G = the kernel's grid,
  // one CTA per SM) reversed: a persistent CTA c walks items c, c + G, c + 2G, ..., so
  // it takes the c-th longest of round 0, the c-th shortest of round 1, and so on (a
  // snake), which evens out the CTAs' totals better than plain round-robin. Items of
  // one round stay together, so CTAs still work on similar items at the same time.
  auto longer = [](const Item& x, const Item& y) {
    return (x.kv_end - x.kv_begin) > (y.kv_end - y.kv_begin);
  };
  auto snake = [&](std::vector<Item>& v) {
    std::stable_sort(v.begin(), v.end(), longer);
    const size_t G = std::min<size_t>(v.size(), (size_t)sms);
    if (G == 0) return;
    for (size_t r0 = G; r0 < v.size(); r0 += 2 * G)
      std::reverse(v.begin() + r0, v.begin() + std::min(v.size(), r0 + G));
  };
  snake(dec);
  snake(tc);
  snake(tc2);
  snake(tcd);

  pa_plan_s* p = new (std::nothrow) pa_plan_s();
  if (!p) return PA_ERR_INVALID_ARG;
  p->num_seqs = num_seqs; p->Hq = Hq; p->Hkv = Hkv; p->D = D; p->block_size = block_size;
  p->max_blocks = max_blocks_per_seq; p->g = g; p->total_q = total_q;
  p->n_dec = (int32_t)dec.size(); p->n_tc = (int32_t)tc.size(); p->n_tc2 = (int32_t)tc2.size();
  p->n_tcd = (int32_t)tcd.size();
  p->n_groups = (int32_t)groups.size();
  p->dec_rows_max = dec_rows_max; p->n_part_rows = part_rows;
  p->wait_ns = o.wait_limit_ns > 0 ? (uint64_t)o.wait_limit_ns : pa::kWaitLimitNsHost;
  p->chunk = any_split ? (int32_t)chunk : 0; p->kv_tokens = kv_tokens;
  size_t off = 0;
  p->off_dec = off; off = align_up(off + dec.size() * sizeof(Item), 256);
  p->off_tc = off; off = align_up(off + tc.size() * sizeof(Item), 256);
  p->off_tc2 = off; off = align_up(off + tc2.size() * sizeof(Item), 256);
  p->off_tcd = off; off = align_up(off + tcd.size() * sizeof(Item), 256);
  p->off_groups = off; off = align_up(off + groups.size() * sizeof(SplitGroup), 256);
  // per-row byte for the fused KV write, needed only when some rows are written by the
  // key-major kernel and some by the write kernel
  p->n_fused_rows = n_fused_rows;
  p->wmask = n_fused_rows > 0 && n_fused_rows < total_q;
  p->off_wmask = off; off = align_up(off + (p->wmask ? (size_t)total_q : 0), 256);
  p->table_bytes = off;
  p->off_acc = off; off = align_up(off + (size_t)part_rows * D * sizeof(float), 256);
  p->off_ml = off; off = align_up(off + (size_t)part_rows * 2 * sizeof(float), 256);
  p->ws_bytes = std::max<size_t>(off, 256);
  p->host_tables = nullptr;
  p->host_pinned = false;
  p->host_cap = 0;
  p->upload_ev = nullptr;
  p->upload_recorded = false;
  p->host_reusable = true;
  if (p->table_bytes > 0) {
    PinnedBuf b;
    if (pinned_take(p->table_bytes, &b)) {
      p->host_tables = b.ptr;
      p->host_cap = b.cap;
      p->upload_ev = b.ev;
      p->host_pinned = true;
    } else if (cudaMallocHost(&p->host_tables, p->table_bytes) == cudaSuccess) {
      p->host_pinned = true;
      p->host_cap = p->table_bytes;
    } else {
      cudaGetLastError();
      p->host_tables = malloc(p->table_bytes);
      if (!p->host_tables) { delete p; return PA_ERR_INVALID_ARG; }
    }
    uint8_t* h = static_cast<uint8_t*>(p->host_tables);
    memset(h, 0, p->table_bytes);
    if (!dec.empty()) memcpy(h + p->off_dec, dec.data(), dec.size() * sizeof(Item));
    if (!tc.empty()) memcpy(h + p->off_tc, tc.data(), tc.size() * sizeof(Item));
    if (!tc2.empty()) memcpy(h + p->off_tc2, tc2.data(), tc2.size() * sizeof(Item));
    if (!tcd.empty()) memcpy(h + p->off_tcd, tcd.data(), tcd.size() * sizeof(Item));
    if (!groups.empty())
      memcpy(h + p->off_groups, groups.data(), groups.size() * sizeof(SplitGroup));
    if (p->wmask)
      for (const auto& r : fused_runs) memset(h + p->off_wmask + r.first, 1, (size_t)r.second);
  }
  *out = p;
  *workspace_bytes = p->ws_bytes;
  return PA_OK;
}

pa_status pa_plan_destroy(pa_plan_t p) {
  if (!p) return PA_OK;
  if (p->host_tables) {
    if (p->host_pinned && p->host_reusable) {
      pinned_give({p->host_tables, p->host_cap, p->upload_ev, p->upload_recorded});
    } else if (p->host_pinned) {
      cudaDeviceSynchronize();  // an upload not covered by the event may be in flight
      cudaFreeHost(p->host_tables);
      if (p->upload_ev) cudaEventDestroy(p->upload_ev);
    } else {
      free(p->host_tables);
    }
  }
  delete p;
  return PA_OK;
}

pa_status pa_plan_get_stats(pa_plan_t p, pa_plan_stats* out) {
  if (!p || !out) return PA_ERR_INVALID_ARG;
  out->total_q = p->total_q;
  out->num_seqs = p->num_seqs;
  out->n_dec_items = p->n_dec;
  out->n_tc_items = p->n_tc + p->n_tc2 + p->n_tcd;
  out->n_tc_pair_items = p->n_tc2;
  out->n_tc_decode_items = p->n_tcd;
  out->n_split_groups = p->n_groups;
  out->n_partials = (int32_t)p->n_part_rows;
  out->chunk_tokens = p->chunk;
  out->kv_tokens = p->kv_tokens;
  out->workspace_bytes = (int64_t)p->ws_bytes;
  return PA_OK;
}

pa_status pa_plan_export(pa_plan_t p, int32_t* h_items, int32_t max_items, int32_t* n_items) {
  if (!p || !n_items || max_items < 0 || (max_items > 0 && !h_items)) return PA_ERR_INVALID_ARG;
  *n_items = p->n_dec + p->n_tc + p->n_tc2 + p->n_tcd;
  const uint8_t* h = static_cast<const uint8_t*>(p->host_tables);
  int32_t k = 0;
  for (int path = 0; path < 4; ++path) {
    const int32_t n = path == kPathDec ? p->n_dec
                      : path == kPathTc ? p->n_tc
                      : path == kPathTcPair ? p->n_tc2
                                            : p->n_tcd;
    const size_t off = path == kPathDec ? p->off_dec
                       : path == kPathTc ? p->off_tc
                       : path == kPathTcPair ? p->off_tc2
                                             : p->off_tcd;
    const Item* it = reinterpret_cast<const Item*>(h + off);
    for (int32_t i = 0; i < n && k < max_items; ++i, ++k) {
      int32_t* r = h_items + (int64_t)k * 9;
      r[0] = path; r[1] = it[i].seq; r[2] = it[i].kv_head; r[3] = it[i].row_begin;
      r[4] = it[i].row_count; r[5] = it[i].kv_begin; r[6] = it[i].kv_end; r[7] = it[i].part;
      r[8] = it[i].q_row0;
    }
  }
  return PA_OK;
}

pa_status pa_plan_upload(pa_plan_t p, void* d_workspace, size_t workspace_bytes,
                         void* stream) {
  if (!p) return PA_ERR_INVALID_ARG;
  if (p->total_q == 0) return PA_OK;
  if (!d_workspace) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < p->ws_bytes) return PA_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256) return PA_ERR_UNSUPPORTED;
  if (p->table_bytes &&
      cudaMemcpyAsync(d_workspace, p->host_tables, p->table_bytes, cudaMemcpyHostToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return note_upload(p, static_cast<cudaStream_t>(stream));
}

pa_status pa_attention(pa_plan_t p, void* d_out, pa_dtype out_dtype, const void* d_q,
                       const void* d_k_pool, const void* d_v_pool, const int32_t* d_block_table,
                       const int32_t* d_context_lens, const int32_t* d_query_lens,
                       int32_t num_blocks, float scale, void* d_workspace,
                       size_t workspace_bytes, void* stream) {
  return attention_impl(p, d_out, out_dtype, d_q, d_k_pool, d_v_pool, d_block_table,
                        d_context_lens, d_query_lens, num_blocks, scale, d_workspace,
                        workspace_bytes, stream, true);
}

pa_status pa_attention_planned(pa_plan_t p, void* d_out, pa_dtype out_dtype, const void* d_q,
                               const void* d_k_pool, const void* d_v_pool,
                               const int32_t* d_block_table, const int32_t* d_context_lens,
                               const int32_t* d_query_lens, int32_t num_blocks, float scale,
                               void* d_workspace, size_t workspace_bytes, void* stream) {
  return attention_impl(p, d_out, out_dtype, d_q, d_k_pool, d_v_pool, d_block_table,
                        d_context_lens, d_query_lens, num_blocks, scale, d_workspace,
                        workspace_bytes, stream, false);
}

pa_status pa_attention_write(pa_plan_t p, void* d_out, pa_dtype out_dtype, const void* d_q,
                             const void* d_k_new, const void* d_v_new,
                             const int64_t* d_slot_mapping, void* d_k_pool, void* d_v_pool,
                             const int32_t* d_block_table, const int32_t* d_context_lens,
                             const int32_t* d_query_lens, int32_t num_blocks, float scale,
                             void* d_workspace, size_t workspace_bytes, void* stream) {
  const FusedWrite fw{d_k_new, d_v_new, d_slot_mapping};
  return attention_impl(p, d_out, out_dtype, d_q, d_k_pool, d_v_pool, d_block_table,
                        d_context_lens, d_query_lens, num_blocks, scale, d_workspace,
                        workspace_bytes, stream, true, &fw);
}

pa_status pa_attention_write_planned(pa_plan_t p, void* d_out, pa_dtype out_dtype,
                                     const void* d_q, const void* d_k_new, const void* d_v_new,
                                     const int64_t* d_slot_mapping, void* d_k_pool,
                                     void* d_v_pool, const int32_t* d_block_table,
                                     const int32_t* d_context_lens,
                                     const int32_t* d_query_lens, int32_t num_blocks,
                                     float scale, void* d_workspace, size_t workspace_bytes,
                                     void* stream) {
  const FusedWrite fw{d_k_new, d_v_new, d_slot_mapping};
  return attention_impl(p, d_out, out_dtype, d_q, d_k_pool, d_v_pool, d_block_table,
                        d_context_lens, d_query_lens, num_blocks, scale, d_workspace,
                        workspace_bytes, stream, false, &fw);
}

}  // extern "C"

// Arguments are checked before anything is enqueued; then the plan's tables are
// uploaded (unless the caller did it with pa_plan_upload) and the kernels launched.
static pa_status attention_impl(pa_plan_t p, void* d_out, pa_dtype out_dtype, const void* d_q,
                                const void* d_k_pool, const void* d_v_pool,
                                const int32_t* d_block_table, const int32_t* d_context_lens,
                                const int32_t* d_query_lens, int32_t num_blocks, float scale,
                                void* d_workspace, size_t workspace_bytes, void* stream,
                                bool upload, const FusedWrite* fw) {
  if (!p) return PA_ERR_INVALID_ARG;
  if (out_dtype != PA_F32 && out_dtype != PA_BF16) return PA_ERR_INVALID_ARG;
  if (num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if ((int64_t)num_blocks * p->block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (p->total_q == 0) return PA_OK;
  if (fw) {
    if (!fw->k_new || !fw->v_new || !fw->slots) return PA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(fw->k_new) % 16 || reinterpret_cast<uintptr_t>(fw->v_new) % 16)
      return PA_ERR_UNSUPPORTED;
  }
  if (!d_out || !d_q || !d_k_pool || !d_v_pool || !d_block_table || !d_context_lens ||
      !d_query_lens || !d_workspace)
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < p->ws_bytes) return PA_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256) return PA_ERR_UNSUPPORTED;
  for (const void* ptr : {d_q, d_k_pool, d_v_pool, (const void*)d_out})
    if (reinterpret_cast<uintptr_t>(ptr) % 16) return PA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = pa::device_error_word();
  if (!err) return PA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  if (upload && p->table_bytes) {
    if (cudaMemcpyAsync(ws, p->host_tables, p->table_bytes, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    const pa_status st = note_upload(p, s);
    if (st != PA_OK) return st;
  }

  pa::AttnArgs a;
  a.q = static_cast<const uint16_t*>(d_q);
  a.out = d_out;
  a.out_bf16 = out_dtype == PA_BF16;
  a.block_table = d_block_table;
  a.context_lens = d_context_lens;
  a.query_lens = d_query_lens;
  a.max_blocks = p->max_blocks;
  a.num_blocks = num_blocks;
  a.block_size = p->block_size;
  a.Hq = p->Hq; a.Hkv = p->Hkv; a.g = p->g;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)p->D);
  a.scale_log2 = sc * 1.4426950408889634f;
  a.part_acc = reinterpret_cast<float*>(ws + p->off_acc);
  a.part_ml = reinterpret_cast<float*>(ws + p->off_ml);
  a.err = err;
  a.wait_ns = p->wait_ns;
  a.k_new = nullptr;
  a.v_new = nullptr;
  a.slots = nullptr;
  a.n_slots = (int64_t)num_blocks * p->block_size;
  a.k_pool = static_cast<uint4*>(const_cast<void*>(d_k_pool));
  a.v_pool = static_cast<uint4*>(const_cast<void*>(d_v_pool));
  if (fw) {
    // rows the key-major kernel does not write go through the write kernel first
    if (p->n_fused_rows < p->total_q) {
      const uint8_t* skip = p->wmask ? ws + p->off_wmask : nullptr;
      cudaError_t e = pa::launch_write_kv(fw->k_new, fw->v_new, fw->slots, p->total_q,
                                          const_cast<void*>(d_k_pool),
                                          const_cast<void*>(d_v_pool), a.n_slots,
                                          (int64_t)p->Hkv * p->D * 2, err, s, skip);
      if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    if (p->n_fused_rows > 0) {
      a.k_new = static_cast<const uint4*>(fw->k_new);
      a.v_new = static_cast<const uint4*>(fw->v_new);
      a.slots = fw->slots;
    }
  }

  // The first attention kernel of the call starts after everything before it in the
  // stream (the table upload, the write kernel); each later one is launched as a
  // programmatic dependent of the one before, so that its CTAs start in that kernel's
  // tail (see launch_kernel).
  bool pdl = false;
  if (p->n_dec > 0) {
    const int box_t = std::min(p->block_size, pa::kKeyTile);
    CUtensorMap kmap, vmap;
    pa_status st = pa::make_pool_map(&kmap, d_k_pool, num_blocks, p->block_size, p->Hkv, p->D,
                                     p->D, box_t, false);
    if (st != PA_OK) return st;
    st = pa::make_pool_map(&vmap, d_v_pool, num_blocks, p->block_size, p->Hkv, p->D, p->D, box_t,
                           false);
    if (st != PA_OK) return st;
    int sms = device_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    const int grid = std::min(p->n_dec, sms);
    cudaError_t e = pa::launch_decode(a, kmap, vmap, reinterpret_cast<const Item*>(ws + p->off_dec),
                                      p->n_dec, p->D, p->dec_rows_max, box_t, grid, s, pdl);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    pdl = true;
  }
  if (p->n_tc + p->n_tc2 + p->n_tcd > 0) {
    const int box_t = std::min(p->block_size, 64);
    CUtensorMap kmap, vmap;
    pa_status st = pa::make_pool_map(&kmap, d_k_pool, num_blocks, p->block_size, p->Hkv, p->D,
                                     64, box_t, true);
    if (st != PA_OK) return st;
    st = pa::make_pool_map(&vmap, d_v_pool, num_blocks, p->block_size, p->Hkv, p->D, 64, box_t,
                           true);
    if (st != PA_OK) return st;
    int sms = device_sms();
    if (sms <= 0) return PA_ERR_CUDA;
    CUtensorMap qmap;
    st = pa::make_q_map(&qmap, d_q, p->total_q, p->Hq, p->D, p->g, pa::kTcRows);
    if (st != PA_OK) return st;
    CUtensorMap omap;
    if (p->n_tc2 + p->n_tc > 0) {
      st = pa::make_out_map(&omap, d_out, p->total_q, p->Hq, p->D, p->g, a.out_bf16 != 0);
      if (st != PA_OK) return st;
    }
    if (p->n_tc2 > 0) {
      const int grid = std::min(p->n_tc2, sms);
      cudaError_t e = pa::launch_tc2(a, kmap, vmap, qmap, omap,
                                     reinterpret_cast<const Item*>(ws + p->off_tc2), p->n_tc2,
                                     box_t, grid, s, pdl);
      if (e != cudaSuccess) return PA_ERR_CUDA;
      pdl = true;
    }
    if (p->n_tc > 0) {
      const int grid = std::min(p->n_tc, sms);
      cudaError_t e = pa::launch_tc(a, kmap, vmap, qmap, omap,
                                    reinterpret_cast<const Item*>(ws + p->off_tc), p->n_tc, box_t,
                                    grid, s, pdl);
      if (e != cudaSuccess) return PA_ERR_CUDA;
      pdl = true;
    }
    // the key-major (decode) items last: measured 0.5-1.7% faster on the mixed
    // configurations than first, the memory-bound decode kernel filling the tail
    // of the multi-token kernels
    if (p->n_tcd > 0) {
      CUtensorMap qmap16, kmap_g, vmap_g;
      st = pa::make_q_map(&qmap16, d_q, p->total_q, p->Hq, p->D, p->g, pa::kTcdRows);
      if (st != PA_OK) return st;
      st = pa::make_pool_map_grouped(&kmap_g, d_k_pool, num_blocks, p->block_size, p->Hkv, box_t);
      if (st != PA_OK) return st;
      st = pa::make_pool_map_grouped(&vmap_g, d_v_pool, num_blocks, p->block_size, p->Hkv, box_t);
      if (st != PA_OK) return st;
      const int grid = std::min(p->n_tcd, sms);
      cudaError_t e = pa::launch_tcd(a, kmap_g, vmap_g, qmap16,
                                     reinterpret_cast<const Item*>(ws + p->off_tcd), p->n_tcd,
                                     box_t, grid, s, pdl);
      if (e != cudaSuccess) return PA_ERR_CUDA;
      pdl = true;
    }
  }
  if (p->n_groups > 0) {
    cudaError_t e = pa::launch_combine(
        a, reinterpret_cast<const SplitGroup*>(ws + p->off_groups), p->n_groups, p->D, s, pdl);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}


// ====================================================================== no-alloc variant
// Scratch for pa_attention_static: a fixed device array instead of a caller
// workspace, for callers that cannot allocate device memory (see pa.h). Its
// name is only a host-side stand-in; kernels get the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) uint8_t g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

namespace {
// Device address of g_static_workspace on the current device, looked up on the
// first call per device with that device current, then cached.
pa_status static_workspace(void** out) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr)
      return PA_ERR_CUDA;
    cache[dev] = ptr;
  }
  *out = cache[dev];
  return PA_OK;
}
}  // namespace

extern "C" pa_status pa_attention_static(pa_plan_t plan, void* d_out, pa_dtype out_dtype,
                                         const void* d_q, const void* d_k_pool,
                                         const void* d_v_pool, const int32_t* d_block_table,
                                         const int32_t* d_context_lens,
                                         const int32_t* d_query_lens, int32_t num_blocks,
                                         float scale, void* stream) {
  if (!plan) return PA_ERR_INVALID_ARG;
  if (plan->ws_bytes > (size_t)PA_STATIC_WORKSPACE_BYTES) return PA_ERR_SHAPE;
  void* ws = nullptr;
  const pa_status st = static_workspace(&ws);
  if (st != PA_OK) return st;
  return pa_attention(plan, d_out, out_dtype, d_q, d_k_pool, d_v_pool, d_block_table,
                      d_context_lens, d_query_lens, num_blocks, scale, ws,
                      (size_t)PA_STATIC_WORKSPACE_BYTES, stream);
}
