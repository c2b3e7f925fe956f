/*
 * pa_oracle.h -- plain fp64 CPU oracle for paged multi-token attention.
 *
 * TEST INFRASTRUCTURE ONLY. This header and pa_oracle.c state, in the
 * plainest possible C, what the paged KV-cache path computes. Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (web pages on the subject):
 *   - "PagedAttention" (wiki page), section "Mathematical formulation":
 *       token-level causal attention a_ij = exp(q_i.k_j/sqrt(d)) / sum_{t<=i} exp(q_i.k_t/sqrt(d)),
 *       o_i = sum_{j<=i} a_ij v_j; and its block-wise form over K/V blocks of size B.
 *   - vLLM blog post (devpress), section "1. overall architecture", worked example:
 *       logical block j of a sequence lives in physical block block_table[j];
 *       token position p sits in slot block_table[p / B] * B + p % B.
 *   - same post, section "2.1 parallel sampling": copy-on-write copies a whole
 *       physical block to a fresh one.
 *   - "Stateful LLM Serving with Pensieve" summary, "multi-token attention" and
 *       "unified prefill and generation": the query rows of a request are the last
 *       query_len tokens of its context; decode is the query_len == 1 case.
 *
 * Data layout (shared convention with the library, stated independently):
 *   pools  [num_blocks, block_size, Hkv, D]  bf16 bit patterns (uint16)
 *   q      [total_q, Hq, D]                  bf16 bit patterns, sequences in order
 *   out    [rows, Hq, D]                      double
 *   block_table [num_seqs, max_blocks] int32
 *
 * All functions return 0 on success and a negative code on invalid input;
 * oracle_last_error() gives a message.
 */
#ifndef PA_ORACLE_H_
#define PA_ORACLE_H_
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

const char* oracle_last_error(void);

/* bf16 bit pattern -> exact double. */
double oracle_bf16_to_double(uint16_t bits);

/* slots_out[t] = block_table[seq_ids[t]][positions[t] / B] * B + positions[t] % B. */
int oracle_slot_mapping(const int32_t* block_table, int32_t num_seqs, int32_t max_blocks,
                        int32_t block_size, int32_t num_blocks, const int32_t* seq_ids,
                        const int32_t* positions, int64_t n, int64_t* slots_out);

/* For each t with slot_mapping[t] >= 0 copy the Hkv*D values of token t of
 * k_new / v_new into pool slot slot_mapping[t]. Slot -1 means "skip".
 * Duplicate slots or out-of-range slots are rejected before anything is written. */
int oracle_write_kv(const uint16_t* k_new, const uint16_t* v_new, const int64_t* slot_mapping,
                    int64_t n_new, uint16_t* k_pool, uint16_t* v_pool, int32_t num_blocks,
                    int32_t block_size, int32_t Hkv, int32_t D);

/* For each pair i copy physical block src[i] onto dst[i] in both pools.
 * dst ids must be unique and must not appear among the src ids. */
int oracle_copy_blocks(uint16_t* k_pool, uint16_t* v_pool, const int32_t* src, const int32_t* dst,
                       int32_t n_pairs, int32_t num_blocks, int32_t block_size, int32_t Hkv,
                       int32_t D);

/* Exact causal attention over a paged KV cache, fp64.
 * Row r of q belongs to sequence s (rows are grouped by sequence in order,
 * query_lens[s] rows each) and sits at absolute position
 * context_lens[s] - query_lens[s] + i, i = r - (first row of s).
 * Query head h reads KV head h / (Hq / Hkv).
 * If rows != NULL only those n_rows rows are computed and out is
 * [n_rows, Hq, D]; otherwise every row and out is [total_q, Hq, D].
 * scale <= 0 selects 1/sqrt(D). n_threads <= 0 selects 1. */
int oracle_attention(const uint16_t* q, int64_t total_q, int32_t Hq, int32_t D,
                     const uint16_t* k_pool, const uint16_t* v_pool, int32_t num_blocks,
                     int32_t block_size, int32_t Hkv, const int32_t* block_table,
                     int32_t max_blocks, const int32_t* context_lens,
                     const int32_t* query_lens, int32_t num_seqs, double scale,
                     const int64_t* rows, int64_t n_rows, int32_t n_threads, double* out);

/* Block-wise statement of the same attention (PagedAttention page, block form):
 * scores are formed one whole K block at a time, softmax runs over the
 * concatenated block score vectors, the output is the sum over blocks of
 * V_j^T A_ij. Single-threaded; same arguments as oracle_attention. */
int oracle_attention_blockwise(const uint16_t* q, int64_t total_q, int32_t Hq, int32_t D,
                               const uint16_t* k_pool, const uint16_t* v_pool,
                               int32_t num_blocks, int32_t block_size, int32_t Hkv,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* context_lens, const int32_t* query_lens,
                               int32_t num_seqs, double scale, double* out);

#ifdef __cplusplus
}
#endif
#endif
