/*
 * pa.h -- C ABI of libpa: paged multi-token attention over a block-table KV cache.
 *
 * The operations follow the problem as the pages state it:
 *   - vLLM post (devpress), "1. overall architecture": the KV cache is cut
 *     into fixed-size physical blocks of block_size tokens; a sequence's
 *     logical block j lives in physical block block_table[j], so token
 *     position p sits in slot block_table[p / B] * B + p % B.
 *   - vLLM wiki note, "kernel layer": fused reshape + block write, fused
 *     block read + attention, batched block copy.
 *   - vLLM post, "2.1 parallel sampling": copy-on-write copies one whole block.
 *   - "PagedAttention" wiki page, "mathematical formulation": exact causal
 *     softmax attention with scale 1/sqrt(d), token form and block form.
 *   - Pensieve summary, "multi-token attention for non-contiguous cache" and
 *     "unified prefill and generation": every sequence contributes any number
 *     of query tokens, which are the LAST query_len tokens of its context;
 *     decode is query_len == 1; a context split into disjoint segments is
 *     passed as sub-requests (extra rows whose block-table rows repeat the same
 *     physical block ids) without copying.
 *
 * Layouts (row-major, C order):
 *   K pool, V pool   [num_blocks, block_size, Hkv, D]   bf16
 *   q                [total_q, Hq, D]                    bf16, sequences in order;
 *                    sequence s owns rows sum_{s'<s} query_lens[s'] ...
 *   out              [total_q, Hq, D]                    fp32 (PA_F32) or bf16
 *   block_table      [num_seqs, max_blocks_per_seq]      int32 physical block ids
 *   context_lens, query_lens [num_seqs]                  int32; context_len
 *                    counts the step's new tokens (write first, then attend)
 *   query head h reads KV head h / (Hq / Hkv).
 *
 * Conventions:
 *   - Every pointer argument named d_* or documented "device" is a device
 *     pointer owned by the caller; the library never frees or keeps it.
 *     Pointers documented "host" are read during the call only.
 *   - The stream argument is a cudaStream_t passed as void* (NULL = legacy
 *     default stream). Calls are asynchronous on that stream unless stated.
 *   - Argument errors are detected on the host and returned synchronously;
 *     nothing is launched then. Device-side problems (a block id or slot
 *     out of range, a device length that disagrees with the plan, a bounded
 *     wait that ran out) never trap: the kernel skips the access and records
 *     a code in the library's device error word, read by pa_get_device_error.
 *   - No entry point allocates device memory; scratch comes from the
 *     caller's workspace. pa_plan_create allocates host memory only.
 *   - Thread-compatible: distinct plans may be used from distinct threads.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* a null pointer, negative size, inconsistent lengths */
  PA_ERR_SHAPE = 2,        /* sizes that do not fit together */
  PA_ERR_RANGE = 3,        /* a block id, slot or length outside its range */
  PA_ERR_UNSUPPORTED = 4,  /* valid but not built: head dim, alignment, dtype, device */
  PA_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  PA_ERR_TIMEOUT = 6,      /* a bounded device wait ran out */
  PA_ERR_NO_SPACE = 7      /* the block manager's pool has too few free blocks */
} pa_status;

typedef enum { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/* Device error codes stored in the error word (first error wins). */
#define PA_DEVERR_NONE 0
#define PA_DEVERR_SLOT_RANGE 1    /* pa_write_kv: slot >= num_blocks * block_size */
#define PA_DEVERR_BLOCK_RANGE 2   /* a block id outside [0, num_blocks) */
#define PA_DEVERR_TABLE_RANGE 3   /* a position beyond max_blocks_per_seq * block_size */
#define PA_DEVERR_LENS 4          /* device lengths disagree with the plan */
#define PA_DEVERR_TIMEOUT 5       /* a bounded mbarrier wait ran out */

/* Short English text for a status. Never NULL. */
const char* pa_status_string(pa_status s);

/* Library version string, e.g. "pa 0.1 sm_103a". */
const char* pa_version(void);

/* Reads the device error word of the current device after synchronizing
 * `stream`; writes the PA_DEVERR_* code to *code and, when reset != 0,
 * clears it. Returns PA_OK, or PA_ERR_CUDA if the sync or read failed. */
pa_status pa_get_device_error(int32_t* code, int32_t reset, void* stream);

/* Slot of each listed token (vLLM post, "1. overall architecture", worked
 * example): slots[t] = block_table[seq_ids[t]][positions[t] / B] * B
 *                      + positions[t] % B;  positions[t] < 0 gives -1.
 * d_block_table [num_seqs, max_blocks_per_seq] int32, d_seq_ids and
 * d_positions int32 [n], d_slots int64 [n], all device. Out-of-range entries
 * give slot -1 and set the device error word. */
pa_status pa_slot_mapping(const int32_t* d_block_table, int32_t num_seqs,
                          int32_t max_blocks_per_seq, int32_t block_size, int32_t num_blocks,
                          const int32_t* d_seq_ids, const int32_t* d_positions, int64_t n,
                          int64_t* d_slots, void* stream);

/* Scatter the step's new tokens into the cache (vLLM wiki note, "kernel
 * layer": fused reshape + block write; Pensieve: new KV-tokens are stored in
 * their allocated slots before attention). For each t < n_new with
 * slot = d_slot_mapping[t] >= 0: row `slot` of each pool (viewed as
 * [num_blocks * block_size, Hkv, D]) receives token t of d_k_new / d_v_new
 * ([n_new, Hkv, D] bf16). Slot -1 is skipped; a slot past the pool is skipped
 * and recorded (PA_DEVERR_SLOT_RANGE). Slots must be distinct (duplicates
 * race; the result is then one of the writers). Bit-exact copy.
 * Requires D % 8 == 0 and 16-byte aligned pointers (else PA_ERR_UNSUPPORTED). */
pa_status pa_write_kv(const void* d_k_new, const void* d_v_new, const int64_t* d_slot_mapping,
                      int64_t n_new, void* d_k_pool, void* d_v_pool, int32_t num_blocks,
                      int32_t block_size, int32_t Hkv, int32_t D, void* stream);

/* Copy-on-write block copy (vLLM post, "2.1 parallel sampling"): for each
 * pair i < n_pairs, physical block d_src[i] is copied onto d_dst[i] in both
 * pools. d_src, d_dst int32 [n_pairs], device. Destinations must be distinct
 * and disjoint from the sources (else the copies race). Ids outside
 * [0, num_blocks) are skipped and recorded (PA_DEVERR_BLOCK_RANGE).
 * n_pairs == 0 launches nothing. Bit-exact copy. */
pa_status pa_copy_blocks(void* d_k_pool, void* d_v_pool, const int32_t* d_src,
                         const int32_t* d_dst, int32_t n_pairs, int32_t num_blocks,
                         int32_t block_size, int32_t Hkv, int32_t D, void* stream);

/* ---------------------------------------------------------------- plan
 * The plan is the host-side auxiliary data of one batch (Pensieve summary,
 * kernel microbenchmark: the aux data is computed on the CPU). It splits the
 * batch into work items: (sequence, KV head, a range of query rows, a range
 * of keys), picks the CUDA-core decode kernel or the tensor-core tile kernel
 * for each, and splits long key ranges (split-KV) so the GPU fills. A plan
 * depends only on the host lengths and the shapes, so one plan serves every
 * layer of a step. */
typedef struct pa_plan_s* pa_plan_t;

typedef struct {
  int32_t max_chunk_tokens;  /* 0: automatic split-KV; >0: split key ranges into chunks of at
                                most this many tokens (rounded up to 64) */
  int32_t tc_min_rows;       /* 0: default: 1 where the key-major kernel takes pairs of at
                                most 16 rows (tc_decode on, Hq / Hkv dividing 16), else 4;
                                >0: (sequence, KV head) pairs with at least this many rows
                                (query tokens x packed heads) use the tensor cores; <0:
                                never. Tensor-core items need D = 128, block_size >= 8 and
                                Hq / Hkv dividing 128. */
  int32_t num_sms;           /* 0: query the current device */
  int32_t tc_pair;           /* >0: tensor-core rows go in 256-row items (two 128-row tiles
                                per CTA sharing every K/V tile); <0: 128-row items only;
                                0: default (automatic): 256-row items when the batch's
                                multi-token tensor-core work has fewer FLOPs per byte of
                                K/V, Q and output than the GPU's machine balance (280),
                                else 128-row items. Rows that do not fill whole items
                                form a sequence's first item (the rows that see the
                                fewest keys); with 256-row items it is a 128-row item
                                when it has at most 128 rows */
  int32_t tc_decode;         /* 0: default (on): a (sequence, KV head) pair with at most 16
                                tensor-core rows runs with keys on the 128-row side (needs
                                Hq / Hkv dividing 16); <0: never */
  int32_t wait_limit_ns;     /* 0: default: each wait of a kernel's pipeline gives up after
                                about one second; >0: after this many nanoseconds. A wait
                                that runs out records PA_DEVERR_TIMEOUT and the kernel
                                aborts: it waits (with the default bound) for its own copies
                                and MMAs in flight, frees its tensor memory and returns,
                                leaving the outputs undefined. Short limits exist to test
                                that path. */
  int32_t reserved[2];       /* must be zero */
} pa_plan_options;

typedef struct {
  int64_t total_q;           /* sum of query_lens */
  int32_t num_seqs;
  int32_t n_dec_items;       /* CUDA-core items */
  int32_t n_tc_items;        /* tensor-core items (both kinds) */
  int32_t n_split_groups;    /* row groups whose keys were split (need the combine pass) */
  int32_t n_partials;        /* partial results the split items write */
  int32_t chunk_tokens;      /* split chunk length used (0 = no split) */
  int64_t kv_tokens;         /* sum of context_lens (keys read once per KV head) */
  int64_t workspace_bytes;
  int32_t n_tc_pair_items;   /* of which 256-row (two-tile) items */
  int32_t n_tc_decode_items; /* of which items of at most 16 rows (keys on the 128-row side) */
} pa_plan_stats;

/* Build a plan from HOST copies of the lengths. Validates 0 <= query_len <=
 * context_len, ceil(context_len / block_size) <= max_blocks_per_seq,
 * Hq % Hkv == 0, D in {64, 128}, block_size a power of two in [1, 256].
 * On success *out receives the plan and *workspace_bytes the size of the
 * device workspace pa_attention needs (at least 256). opts may be NULL. */
pa_status pa_plan_create(const int32_t* h_context_lens, const int32_t* h_query_lens,
                         int32_t num_seqs, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t block_size, int32_t max_blocks_per_seq,
                         const pa_plan_options* opts, pa_plan_t* out, size_t* workspace_bytes);

/* Frees a plan (NULL is ignored). Safe once no pa_attention that uses it is
 * still being enqueued; kernels already enqueued do not read the plan. */
pa_status pa_plan_destroy(pa_plan_t plan);

pa_status pa_plan_get_stats(pa_plan_t plan, pa_plan_stats* out);

/* Copies the plan's work items to host memory, 9 int32 per item:
 * (path, seq, kv_head, row_begin, row_count, kv_begin, kv_end, part, q_row0),
 * path 0 = CUDA-core kernel, 1 = tensor-core kernel (128-row tile), 2 = tensor-core
 * kernel with two 128-row tiles per item, 3 = tensor-core kernel for items of at most
 * 16 rows (keys on the 128-row side); packed row rho of a
 * (seq, kv_head) pair is query token rho / g and query head kv_head * g + rho % g;
 * part = first partial-result row (-1 = written straight to out); q_row0 = row
 * of the sequence's first query in q. Writes at most max_items items and the
 * total count to *n_items. For inspection and tests; host only. */
pa_status pa_plan_export(pa_plan_t plan, int32_t* h_items, int32_t max_items, int32_t* n_items);

/* Paged multi-token causal attention (PagedAttention wiki page, token and
 * block forms; Pensieve multi-token kernel with the causal mask fused).
 * For every sequence s, query row i < query_lens[s] (absolute position
 * p = context_lens[s] - query_lens[s] + i) and query head h:
 *   out[r, h, :] = sum_{j <= p} softmax_j(scale * q[r,h,:] . k_j) v_j,
 * k_j, v_j read from the pools through d_block_table row s, KV head h/(Hq/Hkv).
 * scale <= 0 selects 1/sqrt(D). The plan must come from the same lengths
 * (device lengths that disagree are recorded as PA_DEVERR_LENS).
 * d_workspace: device buffer of at least the plan's workspace_bytes, 256-byte
 * aligned; its contents need no initialisation and are overwritten.
 * Calls sharing one workspace must not overlap on the GPU.
 * Keys past context_len in a sequence's last block are never used, whatever
 * bits they hold. */
pa_status pa_attention(pa_plan_t plan, void* d_out, pa_dtype out_dtype, const void* d_q,
                       const void* d_k_pool, const void* d_v_pool, const int32_t* d_block_table,
                       const int32_t* d_context_lens, const int32_t* d_query_lens,
                       int32_t num_blocks, float scale, void* d_workspace,
                       size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- one plan, many calls
 * pa_attention = pa_plan_upload + pa_attention_planned. A step's plan is the same for
 * every layer (the lengths and block tables do not change between layers), so a model
 * uploads the plan once per step and launches the kernels once per layer.
 *
 * pa_plan_upload enqueues on `stream` the copy of the plan's work-item tables (pinned
 * host memory, written at plan creation) into the first bytes of d_workspace
 * (workspace_bytes >= the plan's workspace_bytes, 256-byte aligned; else
 * PA_ERR_SHAPE / PA_ERR_UNSUPPORTED). Nothing else in the workspace is touched.
 *
 * pa_attention_planned takes pa_attention's arguments and launches its kernels
 * without the upload: the workspace must hold this plan's tables from a
 * pa_plan_upload (or pa_attention) of this plan ordered before it on the GPU, with no
 * other plan's upload in between. Kernels read the tables and write the split-KV
 * partials behind them, so calls with one plan and workspace must not overlap on the
 * GPU. Argument checks and errors as for pa_attention. */
pa_status pa_plan_upload(pa_plan_t plan, void* d_workspace, size_t workspace_bytes,
                         void* stream);
pa_status pa_attention_planned(pa_plan_t plan, void* d_out, pa_dtype out_dtype,
                               const void* d_q, const void* d_k_pool, const void* d_v_pool,
                               const int32_t* d_block_table, const int32_t* d_context_lens,
                               const int32_t* d_query_lens, int32_t num_blocks, float scale,
                               void* d_workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- fused write + attention
 * The step's KV write and its attention in one call (vLLM-SOSP23 note, "core method",
 * kernel layer: the new tokens' reshape and block write fused with the block read and
 * attention; Pensieve summary, unified prefill and generation: the new tokens' K/V are
 * stored in their slots, then every query attends to its whole context). For the batch
 * shape vLLM and Pensieve run, where a step's new tokens are exactly its query tokens,
 *   pa_attention_write(plan, out, q, k_new, v_new, slot_mapping, ...)
 * has the effect of
 *   pa_write_kv(k_new, v_new, slot_mapping, total_q, ...); pa_attention(plan, out, q, ...)
 * with:
 *   d_k_new, d_v_new  [total_q, Hkv, D] bf16, device, 16-byte aligned: row r is the K/V
 *                     of query row r (same order as q);
 *   d_slot_mapping    int64 [total_q], device: the slot of row r's position, i.e.
 *                     block_table[s][p / B] * B + p % B, or -1 to skip the row's write.
 * Sequences whose rows go to the key-major kernel (at most 16 packed rows per KV head:
 * decode) have their K/V written inside that kernel, just before it loads the tile
 * holding them, so the write costs no launch and no separate pass; the other rows are
 * written by one write kernel launched first. Writes are bit-exact copies. Requirements
 * beyond pa_write_kv's and pa_attention's: a slot that a decode row writes is read in
 * this call only by that row's sequence (what copy-on-write guarantees: a block being
 * written is held by one sequence); Pensieve's sub-requests that read another
 * sub-request's new tokens may share blocks, which is safe here as long as the writing
 * sub-request has more than 16 packed rows per KV head (it then goes through the write
 * kernel), and otherwise needs pa_write_kv + pa_attention. Slot range errors are
 * recorded as PA_DEVERR_SLOT_RANGE, as in pa_write_kv.
 * pa_attention_write_planned is the same without the table upload (see
 * pa_attention_planned); the planned call reads the per-row write flags the upload
 * left in the workspace. */
pa_status pa_attention_write(pa_plan_t plan, void* d_out, pa_dtype out_dtype, const void* d_q,
                             const void* d_k_new, const void* d_v_new,
                             const int64_t* d_slot_mapping, void* d_k_pool, void* d_v_pool,
                             const int32_t* d_block_table, const int32_t* d_context_lens,
                             const int32_t* d_query_lens, int32_t num_blocks, float scale,
                             void* d_workspace, size_t workspace_bytes, void* stream);
pa_status pa_attention_write_planned(pa_plan_t plan, void* d_out, pa_dtype out_dtype,
                                     const void* d_q, const void* d_k_new, const void* d_v_new,
                                     const int64_t* d_slot_mapping, void* d_k_pool,
                                     void* d_v_pool, const int32_t* d_block_table,
                                     const int32_t* d_context_lens,
                                     const int32_t* d_query_lens, int32_t num_blocks,
                                     float scale, void* d_workspace, size_t workspace_bytes,
                                     void* stream);

/* ---------------------------------------------------------------- no-alloc variant
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory for a workspace. A serving engine
 * typically reserves nearly all HBM for its KV-cache pool at start-up, so a
 * later cudaMalloc for scratch can fail, and cudaMalloc also synchronizes the
 * device, which stalls a pipelined decode loop; plain C callers without an
 * allocator of their own are in the same position.
 *
 * pa_attention_static computes exactly what pa_attention computes, but its
 * scratch (the plan's work-item tables and split-KV partial results) lives in
 * a fixed array of PA_STATIC_WORKSPACE_BYTES inside the library's device
 * image, which every GPU that loads the library keeps until the process exits.
 * It allocates nothing and calls no allocating routine. The caller still owns
 * q, out, the pools, block_table and the length arrays.
 *   - A plan whose workspace_bytes exceeds PA_STATIC_WORKSPACE_BYTES is
 *     rejected with PA_ERR_SHAPE before anything is enqueued; use
 *     pa_attention with a caller-provided workspace for such batches.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it for the
 *     life of the process; make that first call before any stream capture.
 *     The cached address belongs to the device's primary context: after
 *     cudaDeviceReset, or when the calling thread runs under another context
 *     of the device, it is stale and this entry point must not be called.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents (nothing in it needs to start at zero: every call writes the
 *     tables and partials it reads). Calls that overlap on the GPU -- on
 *     different streams, or from different threads -- race on it; serialize
 *     them on one stream. */
#define PA_STATIC_WORKSPACE_BYTES (8u << 20)

pa_status pa_attention_static(pa_plan_t plan, void* d_out, pa_dtype out_dtype, const void* d_q,
                              const void* d_k_pool, const void* d_v_pool,
                              const int32_t* d_block_table, const int32_t* d_context_lens,
                              const int32_t* d_query_lens, int32_t num_blocks, float scale,
                              void* stream);

/* Block swaps between the device pools and host pools of the same layout
 * (vLLM post, "3. scheduling and preemption": evicted blocks are copied to CPU
 * memory and copied back when their request resumes; Pensieve summary,
 * ahead-of-time swapping of KV tokens to the CPU cache and their restore).
 * Pair i moves one whole block of both pools:
 *   PA_SWAP_OUT: device block d_src[i] -> host block d_dst[i]
 *   PA_SWAP_IN:  host block d_src[i]   -> device block d_dst[i]
 * d_k_pool, d_v_pool [num_blocks, block_size, Hkv, D] bf16, device;
 * h_k_pool, h_v_pool [num_host_blocks, block_size, Hkv, D] bf16, host memory
 * that CUDA has page-locked and mapped (cudaHostAlloc, or cudaHostRegister with
 * mapping) -- the kernel reads or writes it directly over the CPU-GPU link, so
 * one launch moves any number of scattered blocks; anything else is
 * PA_ERR_INVALID_ARG. d_src, d_dst int32 [n_pairs], device; destinations must
 * be distinct. Asynchronous on `stream`: the host pool must stay allocated
 * until the stream has passed the call. Block ids out of range are skipped
 * and recorded as PA_DEVERR_BLOCK_RANGE. All pools 16-byte aligned, D % 8 == 0
 * (else PA_ERR_UNSUPPORTED). */
#define PA_SWAP_OUT 0
#define PA_SWAP_IN 1
pa_status pa_swap_blocks(void* d_k_pool, void* d_v_pool, int32_t num_blocks, void* h_k_pool,
                         void* h_v_pool, int32_t num_host_blocks, const int32_t* d_src,
                         const int32_t* d_dst, int32_t n_pairs, int32_t block_size, int32_t Hkv,
                         int32_t D, int32_t direction, void* stream);

/* ---------------------------------------------------------------------------
 * Host KV block manager: the physical block allocator, reference counts,
 * fork / append / free and the copy-on-write decision, in host memory only.
 *
 * Follows the vLLM post (devpress), "1. overall architecture" (a request is a
 * list of logical blocks filled left to right; the block table maps them to
 * physical blocks of a pre-cut pool and records how full the last one is; a
 * new physical block is taken only when the last logical block is full; a
 * finished request's blocks are freed) and "2.1 parallel sampling" (a physical
 * block carries a reference count; a request about to write into a block
 * whose count is above one gets a newly taken block into which the shared
 * block is copied, and the shared count drops by one, so the last holder
 * writes in place); the vLLM-SOSP23 note, "core method" (fork / append / free).
 * Pensieve's sub-requests over one context are forks whose block-table rows
 * list the same physical blocks.
 *
 * The manager decides; the caller moves data: the slots an append returns are
 * the slot_mapping of pa_write_kv, its copy pairs are the input of
 * pa_copy_blocks (run before the write), and pa_bm_tables gives the
 * block_table and context_lens rows of pa_plan_create / pa_attention.
 *
 * Free pool: blocks are handed out first in, first out, initially in
 * h_free_order (host, num_blocks distinct ids; NULL = 0, 1, 2, ...); a freed
 * block joins the back of the pool. Sequence ids are caller-chosen int64.
 * Errors: PA_ERR_INVALID_ARG for a null handle or pointer, an unknown or
 * duplicate sequence id, a negative count; PA_ERR_NO_SPACE when an append
 * needs more free blocks than the pool holds -- the manager is then unchanged.
 * A request that is swapped out (below) may only be swapped in or freed.
 * A manager is not thread-safe: use one per thread or lock around calls.
 * --------------------------------------------------------------------------- */
typedef struct pa_bm_s* pa_bm_t;

/* A pool of num_blocks blocks of block_size tokens, all free. */
pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* h_free_order,
                       pa_bm_t* out);
pa_status pa_bm_destroy(pa_bm_t bm);

/* A new request holding no tokens. */
pa_status pa_bm_add(pa_bm_t bm, int64_t seq);

/* A new request `child` sharing every block of `parent` (each count + 1). */
pa_status pa_bm_fork(pa_bm_t bm, int64_t parent, int64_t child);

/* A finished request: each of its blocks loses one reference; blocks left with
 * none return to the free pool, in table order. */
pa_status pa_bm_free(pa_bm_t bm, int64_t seq);

/* One step's new tokens: h_counts[i] tokens for request h_seqs[i] (each listed
 * at most once), at positions L_i .. L_i + h_counts[i] - 1, in the listed order.
 * Writes the slot of every new token to h_slots (int64, sum of counts, request
 * by request, block * block_size + offset) and the copies the write needs
 * first to h_cow_src / h_cow_dst (int32, room for n_seqs pairs; *n_cow pairs
 * written; at most one per request: only a partially filled last block can be
 * shared). All host pointers. All-or-nothing: PA_ERR_NO_SPACE leaves every
 * table and count as it was. */
pa_status pa_bm_append(pa_bm_t bm, const int64_t* h_seqs, const int32_t* h_counts,
                       int32_t n_seqs, int64_t* h_slots, int32_t* h_cow_src,
                       int32_t* h_cow_dst, int32_t* n_cow);

/* Block-table rows and context lengths of the listed requests, for the
 * attention calls: h_block_table [n_seqs, max_blocks] int32 padded with -1
 * (NULL to skip; PA_ERR_SHAPE if a request holds more than max_blocks
 * blocks), h_context_lens [n_seqs] int32 (NULL to skip). Host pointers. */
pa_status pa_bm_tables(pa_bm_t bm, const int64_t* h_seqs, int32_t n_seqs, int32_t max_blocks,
                       int32_t* h_block_table, int32_t* h_context_lens);

/* Tokens held, blocks listed and residency (1: swapped out to the host pool) of
 * one request (any pointer may be NULL); #filled of its last block is
 * len - block_size * (n_blocks - 1). */
pa_status pa_bm_seq_info(pa_bm_t bm, int64_t seq, int64_t* len, int32_t* n_blocks,
                         int32_t* on_host);

/* Swapping (vLLM post, "3. scheduling and preemption": eviction moves all of a
 * request's blocks to CPU memory, managed by a CPU block allocator, and copies
 * them back when the request resumes). pa_bm_set_host_pool gives the manager a
 * host pool of num_host_blocks blocks (once; h_free_order as for the device
 * pool). pa_bm_swap_out moves every listed request (each once, all on the
 * device) to the host pool: each distinct device block they name gets one host
 * block, so blocks they share stay shared; the (device block, host block) copies
 * to make -- with pa_swap_blocks(PA_SWAP_OUT), before the freed device blocks
 * are written again -- go to h_dev / h_host (room for `capacity` pairs;
 * *n_pairs written), in the order the tables name the blocks. Device blocks
 * left without references return to the free pool. pa_bm_swap_in is the
 * reverse for requests on the host (copies with PA_SWAP_IN before they run).
 * A swapped-out request may only be swapped in or freed; its table names host
 * blocks. All-or-nothing: PA_ERR_NO_SPACE when the receiving pool has too few
 * free blocks, PA_ERR_SHAPE when capacity is too small; nothing changes then. */
pa_status pa_bm_set_host_pool(pa_bm_t bm, int32_t num_host_blocks, const int32_t* h_free_order);
pa_status pa_bm_swap_out(pa_bm_t bm, const int64_t* h_seqs, int32_t n_seqs, int32_t* h_dev,
                         int32_t* h_host, int32_t capacity, int32_t* n_pairs);
pa_status pa_bm_swap_in(pa_bm_t bm, const int64_t* h_seqs, int32_t n_seqs, int32_t* h_host,
                        int32_t* h_dev, int32_t capacity, int32_t* n_pairs);
pa_status pa_bm_host_refcount(pa_bm_t bm, int32_t block, int32_t* count);
pa_status pa_bm_host_num_free(pa_bm_t bm, int32_t* n_free);

/* Reference count of one physical block (PA_ERR_RANGE outside the pool). */
pa_status pa_bm_refcount(pa_bm_t bm, int32_t block, int32_t* count);

/* Blocks in the free pool. */
pa_status pa_bm_num_free(pa_bm_t bm, int32_t* n_free);

#ifdef __cplusplus
}
#endif
#endif /* PA_H_ */
