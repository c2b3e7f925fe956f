// pa_internal.h -- host-side declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// One unit of attention work: a range of rows of one (sequence, KV head) pair
// against a range of keys. Row rho of the pair is query token rho / g and query
// head kv_head * g + rho % g, g = Hq / Hkv (query heads packed per KV head).
struct Item {
  int32_t seq;
  int32_t kv_head;
  int32_t row_begin;  // first packed row
  int32_t row_count;  // rows in this item
  int32_t kv_begin;   // first key (a multiple of the key tile)
  int32_t kv_end;     // one past the last key any row of the item may see
  int32_t part;       // first partial-result row of this item, -1 = write the output directly
  int32_t q_row0;     // row of the sequence's first query in q / out
};
static_assert(sizeof(Item) == 32, "Item is 32 bytes");

// Rows whose keys were split: merged by the combine kernel.
struct SplitGroup {
  int32_t seq;
  int32_t kv_head;
  int32_t row_begin;
  int32_t row_count;
  int32_t part_begin;  // chunk c, row r of the group is partial row part_begin + c * row_count + r
  int32_t n_parts;     // key chunks
  int32_t q_row0;
  int32_t pad;
};
static_assert(sizeof(SplitGroup) == 32, "SplitGroup is 32 bytes");

constexpr int kDecRows = 8;     // rows a CUDA-core item holds at most
constexpr int kTcRows = 128;    // rows of a tensor-core item (one M tile)
// GB300 machine balance for bf16 attention: dense tensor rate (~1.9 PFLOP/s) over HBM
// bandwidth (~6.8 TB/s), in FLOPs per byte
constexpr double kTcMachineBalance = 280.0;
constexpr int kTcdRows = 16;    // rows of a key-major tensor-core decode item (N)
constexpr int kKeyTile = 64;    // keys per pipeline stage of the decode kernel
constexpr int kChunkAlign = 64;   // split-KV chunk boundaries are multiples of this
constexpr uint64_t kWaitLimitNsHost = 1000000000ull;  // default bound on a pipeline wait

// Common launch arguments of the attention kernels.
struct AttnArgs {
  const uint16_t* q;          // bf16 [total_q, Hq, D]
  void* out;                  // fp32 or bf16 [total_q, Hq, D]
  int32_t out_bf16;
  const int32_t* block_table;
  const int32_t* context_lens;
  const int32_t* query_lens;
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t block_size;
  int32_t Hq, Hkv, g;
  float scale_log2;           // scale * log2(e)
  float* part_acc;            // [n_partial_rows, D]: unnormalised sum of p * v
  float* part_ml;             // [n_partial_rows, 2]: running max (log2 domain) and sum of p
  int* err;                   // device error word
  uint64_t wait_ns;           // bound on each pipeline wait (ns)
  // Fused KV write (null k_new: none). The step's new tokens are its query tokens:
  // k_new / v_new [total_q, Hkv, D] bf16 in q's row order, slots [total_q] the slot of
  // each token's position (-1: skip). The key-major kernel writes the tokens of its
  // items before it reads them.
  const uint4* k_new;
  const uint4* v_new;
  const int64_t* slots;
  int64_t n_slots;            // num_blocks * block_size
  uint4* k_pool;              // the pools, for those writes
  uint4* v_pool;
};

// Launches kernel k on stream s; with pdl, as a programmatic dependent of the
// previous kernel in the stream: its CTAs may start once every CTA of that kernel has
// signalled (griddepcontrol.launch_dependents, at its start), i.e. in the tail of
// that kernel, instead of after its last CTA exits. The attention kernels of one call
// read nothing another one writes (disjoint outputs and partial rows); each waits for
// its predecessor to complete before it exits (griddepcontrol.wait), so a kernel's
// completion still implies that of every kernel before it, and the combine pass waits
// at its start.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), int grid, int block, int smem, cudaStream_t s,
                          bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

// Device address of the error word of the current device (set up once per device).
int* device_error_word();

// Number of SMs of the current device (queried once per device, then cached); 0 if the
// query fails.
int sm_count();

// Builds a 3-D tiled tensor map over a pool viewed as [num_blocks * B][Hkv][D] bf16.
// box = (box_d, 1, box_t); swizzle128 selects the 128-byte swizzle.
// 5-D tiled map over a pool [num_blocks * B][Hkv][128] bf16 whose box is a block piece of
// box_t tokens (a multiple of 8) of one KV head, both D halves, 128-byte swizzled: the box
// lands as box_t / 8 groups of 2 KB, each [D half][8 rows x 128 B], so that one copy per
// piece fills both halves (see the key-major kernel's tile layout).
pa_status make_pool_map_grouped(CUtensorMap* map, const void* pool, int64_t num_blocks,
                                int block_size, int Hkv, int box_t);
pa_status make_pool_map(CUtensorMap* map, const void* pool, int64_t num_blocks, int block_size,
                        int Hkv, int D, int box_d, int box_t, bool swizzle128);

// Launchers (return cudaGetLastError of the launch).
cudaError_t launch_slot_mapping(const int32_t* bt, int32_t num_seqs, int32_t max_blocks,
                                int32_t block_size, int32_t num_blocks, const int32_t* seq_ids,
                                const int32_t* positions, int64_t n, int64_t* slots, int* err,
                                cudaStream_t s);
// skip (optional, device, one byte per row): rows with a non-zero byte are not written
// here (the fused attention call writes them inside the key-major kernel).
cudaError_t launch_write_kv(const void* k_new, const void* v_new, const int64_t* slots,
                            int64_t n_new, void* k_pool, void* v_pool, int64_t n_slots,
                            int64_t row_bytes, int* err, cudaStream_t s,
                            const uint8_t* skip = nullptr);
cudaError_t launch_copy_blocks(void* k_pool, void* v_pool, const int32_t* src, const int32_t* dst,
                               int32_t n_pairs, int32_t num_blocks, int64_t block_bytes, int* err,
                               cudaStream_t s);
cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const Item* items, int32_t n_items, int D, int rows_max, int box_t,
                          int grid, cudaStream_t s, bool pdl = false);
cudaError_t launch_combine(const AttnArgs& a, const SplitGroup* groups, int32_t n_groups, int D,
                           cudaStream_t s, bool pdl = false);
int decode_smem_bytes(int D, int rows_max);
cudaError_t launch_tc(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                      const CUtensorMap& qmap, const CUtensorMap& omap, const Item* items,
                      int32_t n_items, int box_t, int grid, cudaStream_t s, bool pdl = false);
// 3-D tiled map over q viewed as [total_q][Hq][D] bf16 with box (64, g, rows / g), 128-byte
// swizzle: one box is `rows` packed rows (tokens x the g heads of a KV head) of one D half.
pa_status make_q_map(CUtensorMap* map, const void* q, int64_t total_q, int Hq, int D, int g,
                     int rows);
int tc_smem_bytes();
// Items of 129..256 rows: two 128-row tiles per CTA that share every K/V tile.
cudaError_t launch_tc2(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const CUtensorMap& qmap, const CUtensorMap& omap, const Item* items,
                       int32_t n_items, int box_t, int grid, cudaStream_t s, bool pdl = false);
// 3-D tiled map over the output viewed as [total_q][Hq][D] (fp32 or bf16), box (16,
// min(g, 32), 32 / min(g, 32)): one box is 16 columns of the 32 packed rows (tokens x
// heads of one KV head) of a warp. The staging side is swizzled (64-byte rows of fp32
// with the 64-byte pattern, 32-byte rows of bf16 with the 32-byte one) so that a warp
// writes its rows there without bank conflicts.
pa_status make_out_map(CUtensorMap* map, void* out, int64_t total_q, int Hq, int D, int g,
                       bool bf16);
int tc2_smem_bytes();
// Items of at most 16 rows: keys on the 128-row side (S^T = K Q^T, O^T = V^T P^T).
cudaError_t launch_tcd(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const CUtensorMap& qmap, const Item* items, int32_t n_items, int box_t,
                       int grid, cudaStream_t s, bool pdl = false);
int tcd_smem_bytes();
constexpr int kTcMinRowsDefault = 4;   // without the key-major kernel: rows from which the
                                       // tensor cores take a (sequence, KV head) pair

}  // namespace pa
