/*
 * pkv_oracle.h -- plain, slow, obviously correct CPU oracle for attention
 * decode over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this code: only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, helper or
 * constant with the CUDA library.
 *
 * Every floating-point result is computed in binary64 from inputs that are
 * read exactly (bf16 and fp32 values are exactly representable in double).
 *
 * Sources (page titles, sections):
 *   [M5.3]  "M5.3 - KV Memory Layout and Exact Reuse", sections 0x02C, 0x03C-0x03I,
 *           0x04E, 0x0A, 0x0BA, 0x0BB, 0x0BC, 0x0BE, 0x0BI.
 *   [Ch7]   "7. Memory Management and Local Model State", "Logical tokens,
 *           physical blocks" and "Choosing a block size".
 *   [Cache] "Cache Concepts: Prefix Matching vs. Storage" (TokenSpeed), the
 *           slot invariant table[req, pos // P] * P + pos % P with the -1 skip
 *           sentinel, and widening page ids to int64 before multiplying.
 *
 * Cache layout (one layer, separate K and V tensors), row-major, declared
 * axis order [num_blocks, block_size, num_kv_heads, head_dim]: the token-major
 * order of the checked address trace in [M5.3] 0x03F without its layer axis.
 */
#ifndef PKV_ORACLE_H
#define PKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage dtypes understood by the oracle */
enum { PKV_ORACLE_F32 = 0, PKV_ORACLE_BF16 = 1 };

/* status codes */
enum {
  PKV_ORACLE_OK = 0,
  PKV_ORACLE_BAD_ARG = 1,
  PKV_ORACLE_BAD_SLOT = 2,          /* a slot id >= num_blocks * block_size   */
  PKV_ORACLE_BAD_BLOCK = 3,         /* a physical block id outside the pool   */
  /* rejection order of the reference translator, [M5.3] 0x03G / 0x03I      */
  PKV_ORACLE_REJECT_VISIBILITY = 10,/* token outside the request's context    */
  PKV_ORACLE_REJECT_TABLE = 11,     /* logical block beyond the block table   */
  PKV_ORACLE_REJECT_PHYSICAL = 12   /* table entry names no pool block        */
};

/* N = ceil(T / P): block-table references for T tokens, [M5.3] 0x02C. */
int64_t pkv_oracle_num_blocks(int64_t num_tokens, int64_t block_size);

/* valid rows of the last block (0 when T = 0), [M5.3] 0x0A valid_rows. */
int64_t pkv_oracle_tail_rows(int64_t num_tokens, int64_t block_size);

/* slot id = physical slot * P + token offset, [M5.3] 0x03D. */
int64_t pkv_oracle_slot_id(int64_t physical_slot, int64_t block_size,
                           int64_t token_offset);

/* element offset sum_a coord[a] * prod_{b>a} shape[b] of a row-major tensor,
 * [M5.3] 0x03E.  Returns -1 if a coordinate is outside its axis. */
int64_t pkv_oracle_row_major_offset(int rank, const int64_t* shape,
                                    const int64_t* coord);

/* Resolve logical token `token` of one request to (physical block, offset).
 * Checks in the order request visibility -> table bounds -> physical
 * identity ([M5.3] 0x03G, 0x03I) and returns the first failing check. */
int pkv_oracle_resolve(const int32_t* table, int64_t table_len,
                       int64_t context_len, int64_t block_size,
                       int64_t num_pool_blocks, int64_t token,
                       int64_t* block_out, int64_t* offset_out);

/* Slot mapping of logical position `pos` of a request:
 * table[pos / P] * P + pos % P, computed in int64 ([Cache]). */
int64_t pkv_oracle_slot_for_position(const int32_t* table, int64_t block_size,
                                     int64_t pos);

/* The same slot for n (request, position) pairs at once: out[i] is the slot
 * of position positions[i] of the request whose table is row rows[i] of
 * `tables` ([*, table_stride] int32).  A negative row or position, or a
 * position past the table, returns PKV_ORACLE_BAD_ARG. */
int pkv_oracle_slots_for_positions(const int32_t* tables, int64_t table_stride,
                                   const int32_t* rows, const int64_t* positions, int64_t n,
                                   int64_t block_size, int64_t* out);

/* Write new token rows.  Row i (num_kv_heads * head_dim elements of k and of
 * v) goes to slot slots[i]; a negative slot is skipped ([Cache] -1 sentinel).
 * Returns PKV_ORACLE_BAD_SLOT (after writing every valid row) if any slot is
 * >= num_blocks * block_size; such rows are not written. */
int pkv_oracle_kv_append(int dtype, void* k_cache, void* v_cache,
                         int64_t num_blocks, int block_size, int num_kv_heads,
                         int head_dim, const void* k, const void* v,
                         const int64_t* slots, int64_t num_tokens);

/* Copy-on-write block copies: for each pair (src, dst), in order, the whole
 * block src of k_cache and v_cache is copied to block dst ([M5.3] 0x04C,
 * 0x05A).  Returns PKV_ORACLE_BAD_BLOCK if an id is outside the pool; that
 * pair is not copied. */
int pkv_oracle_kv_block_copy(int dtype, void* k_cache, void* v_cache,
                             int64_t num_blocks, int block_size,
                             int num_kv_heads, int head_dim,
                             const int64_t* pairs, int64_t num_pairs);

/* Paged attention decode: one query row per sequence against its full
 * logical history ([M5.3] 0x0A, 0x0BA).  For sequence r and query head h,
 * kv head = h / (num_q_heads / num_kv_heads); the history K_r, V_r is
 * gathered token by token through block_tables[r * max_blocks + t / P];
 * s_t = scale * q . k_t ; m = max s ; out = sum exp(s_t - m) v_t / sum exp(s_t - m);
 * lse = m + log sum exp(s_t - m).  An empty sequence gives out = 0 and
 * lse = -inf.  out: [B, Hq, D] doubles; lse (may be NULL): [B, Hq].
 * q is [B, Hq, D] in the cache dtype.  Uses up to nthreads OpenMP threads
 * over (sequence, head) pairs (nthreads <= 0: one thread). */
int pkv_oracle_paged_decode(int dtype, const void* q, const void* k_cache,
                            const void* v_cache, int64_t num_blocks,
                            int block_size, int num_kv_heads, int head_dim,
                            const int32_t* block_tables, int max_blocks,
                            const int32_t* seq_lens, int num_seqs,
                            int num_q_heads, double scale, double* out,
                            double* lse, int nthreads);

/* Shared-prefix attention by definition ([M5.3] 0x0BC): request r's logical
 * history is the shared prefix blocks followed by its own suffix blocks, so
 * this builds the concatenated block table (prefix_len must be a multiple of
 * the block size) and runs pkv_oracle_paged_decode on it. */
int pkv_oracle_shared_prefix(int dtype, const void* q, const void* k_cache,
                             const void* v_cache, int64_t num_blocks,
                             int block_size, int num_kv_heads, int head_dim,
                             const int32_t* prefix_block_ids,
                             int32_t prefix_len,
                             const int32_t* suffix_block_tables,
                             int max_suffix_blocks,
                             const int32_t* suffix_lens, int num_seqs,
                             int num_q_heads, double scale, double* out,
                             double* lse, int nthreads);

/* Attention over a prefix-tree snapshot by definition ([M5.3] 0x0BB, 0x0BE
 * "reference" schedule): chunk c holds chunk_lens[c] K/V rows, row t in pool
 * block block_ids[chunk_first_id[c] + t / P] at offset t % P, and covers the
 * sequences [chunk_begin[c], chunk_end[c]).  Sequence r's logical history is
 * the concatenation, in array (tree) order, of the rows of every chunk that
 * covers r; one monolithic softmax row runs over it.  The pool is viewed as
 * num_blocks * P blocks of one row each, so each history becomes a table of
 * slot ids for pkv_oracle_paged_decode.  Returns PKV_ORACLE_BAD_ARG for a
 * chunk with len < 1, an empty or out-of-range coverage, or ids outside
 * block_ids; PKV_ORACLE_BAD_BLOCK for a block id outside the pool. */
int pkv_oracle_chunk_tree(int dtype, const void* q, const void* k_cache,
                          const void* v_cache, int64_t num_blocks,
                          int block_size, int num_kv_heads, int head_dim,
                          const int32_t* chunk_first_id,
                          const int32_t* chunk_lens,
                          const int32_t* chunk_begin, const int32_t* chunk_end,
                          int num_chunks, const int32_t* block_ids,
                          int64_t num_block_ids, int num_seqs, int num_q_heads,
                          double scale, double* out, double* lse,
                          int nthreads);

/* ------------------------------------------------------------------------
 * MXFP8 pools: a quantized storage schema ([M5.3] 0x0BB names quantized K/V
 * a cache-ABI field; TokenSpeed's MXFP8 KV keeps scale planes beside the
 * element planes).  Elements are OCP FP8 E4M3 (bias 7, 3 mantissa bits,
 * subnormals, no infinities, 0x7F / 0xFF NaN, largest finite 448); every 32
 * consecutive head_dim elements of one (token, kv head) row share an E8M0
 * scale byte s (the value 2^(s - 127)).  A cache buffer holds the element
 * plane [NB, P, Hkv, D] followed by the scale plane [NB, Hkv, P, D / 32].
 */

/* E4M3 value of a code (NaN codes return NaN). */
double pkv_oracle_e4m3_decode(uint8_t code);

/* E4M3 code of x: round to nearest, ties to even, |x| beyond 448 saturating
 * to 448 (x must not be NaN). */
uint8_t pkv_oracle_e4m3_encode(double x);

/* The same code by searching all finite codes for the nearest value (ties
 * to the even code): slow, for checking pkv_oracle_e4m3_encode. */
uint8_t pkv_oracle_e4m3_encode_exhaustive(double x);

/* Scale byte of a 32-element group with largest magnitude amax: the
 * smallest power of two X = 2^(s - 127) with amax / X <= 448, so that no
 * element saturates; clamped to s in [0, 254]; s = 0 for amax = 0. */
uint8_t pkv_oracle_mx_scale(double amax);

/* Write rows into an MXFP8 pool: for each token i with slot s >= 0, every
 * kv head's D elements of k[i] / v[i] (bf16 bits, or fp32 when
 * in_dtype == PKV_ORACLE_F32) are quantized group by group (scale from the
 * group's largest magnitude, element = E4M3 of x / 2^(s - 127)) into the
 * element and scale planes at that slot.  Returns as pkv_oracle_kv_append. */
int pkv_oracle_kv_append_mxfp8(int in_dtype, uint8_t* k_cache, uint8_t* v_cache,
                               int64_t num_blocks, int block_size,
                               int num_kv_heads, int head_dim, const void* k,
                               const void* v, const int64_t* slots,
                               int64_t num_tokens);

/* Dequantize an MXFP8 pool to fp32 [NB, P, Hkv, D] (exact: an E4M3 value
 * times a power of two within fp32's range for scales from bf16 data). */
int pkv_oracle_mxfp8_to_f32(const uint8_t* cache, int64_t num_blocks,
                            int block_size, int num_kv_heads, int head_dim,
                            float* out);

/* K/V row ledger of a batch ([M5.3] 0x02D, 0x0BI): logical rows are the sum of
 * the requests' context lengths, unique rows the number of distinct
 * (physical block, offset) slots they reference.  Slots are counted in a
 * bitmap of num_blocks * block_size bits. */
int pkv_oracle_row_ledger(const int32_t* block_tables, int max_blocks,
                          const int32_t* seq_lens, int num_seqs,
                          int64_t num_blocks, int block_size,
                          int64_t* logical_rows, int64_t* unique_rows);

/* Split allocator blocks for a kernel ([M5.3] 0x0AC): with P_a = q P_k,
 * allocator block id a becomes the kernel block ids a q, a q + 1, ...,
 * a q + q - 1, in that order; a negative (padding) entry becomes q padding
 * entries (-1).  out receives n * q entries.  Returns PKV_ORACLE_BAD_ARG for
 * q < 1 or an id whose expansion passes INT32_MAX. */
int pkv_oracle_expand_table(const int32_t* table, int64_t n, int32_t q, int32_t* out);

#ifdef __cplusplus
}
#endif
#endif
