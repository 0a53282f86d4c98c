/*
 * pkv_oracle.c -- plain fp64 CPU oracle for paged attention decode.
 *
 * TEST INFRASTRUCTURE ONLY (see pkv_oracle.h).  Deliberately naive: every
 * sequence is gathered token by token through its block table into a
 * contiguous history, then textbook softmax attention runs over it in
 * binary64.  No split-K, no log-sum-exp merging, no tiling.
 */
#include "pkv_oracle.h"

#include <limits.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static size_t elem_bytes(int dtype) {
  return dtype == PKV_ORACLE_BF16 ? 2u : 4u;
}

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double load_elem(int dtype, const void* base, int64_t idx) {
  if (dtype == PKV_ORACLE_BF16) {
    uint16_t h;
    memcpy(&h, (const unsigned char*)base + 2 * idx, 2);
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
  } else {
    float f;
    memcpy(&f, (const unsigned char*)base + 4 * idx, 4);
    return (double)f;
  }
}

int64_t pkv_oracle_num_blocks(int64_t num_tokens, int64_t block_size) {
  if (num_tokens <= 0 || block_size <= 0) return 0;
  return (num_tokens + block_size - 1) / block_size;
}

int64_t pkv_oracle_tail_rows(int64_t num_tokens, int64_t block_size) {
  int64_t n = pkv_oracle_num_blocks(num_tokens, block_size);
  if (n == 0) return 0;
  return num_tokens - (n - 1) * block_size;
}

int64_t pkv_oracle_slot_id(int64_t physical_slot, int64_t block_size,
                           int64_t token_offset) {
  return physical_slot * block_size + token_offset;
}

int64_t pkv_oracle_row_major_offset(int rank, const int64_t* shape,
                                    const int64_t* coord) {
  int64_t off = 0;
  for (int a = 0; a < rank; ++a) {
    if (coord[a] < 0 || coord[a] >= shape[a]) return -1;
    int64_t stride = 1;
    for (int b = a + 1; b < rank; ++b) stride *= shape[b];
    off += coord[a] * stride;
  }
  return off;
}

int pkv_oracle_resolve(const int32_t* table, int64_t table_len,
                       int64_t context_len, int64_t block_size,
                       int64_t num_pool_blocks, int64_t token,
                       int64_t* block_out, int64_t* offset_out) {
  if (block_size <= 0) return PKV_ORACLE_BAD_ARG;
  /* 1. request visibility */
  if (token < 0 || token >= context_len) return PKV_ORACLE_REJECT_VISIBILITY;
  /* 2. table bounds */
  int64_t logical_block = token / block_size;
  int64_t offset = token % block_size;
  if (logical_block >= table_len) return PKV_ORACLE_REJECT_TABLE;
  /* 3. physical identity */
  int64_t physical = (int64_t)table[logical_block];
  if (physical < 0 || physical >= num_pool_blocks)
    return PKV_ORACLE_REJECT_PHYSICAL;
  if (block_out) *block_out = physical;
  if (offset_out) *offset_out = offset;
  return PKV_ORACLE_OK;
}

int64_t pkv_oracle_slot_for_position(const int32_t* table, int64_t block_size,
                                     int64_t pos) {
  int64_t physical = (int64_t)table[pos / block_size];
  return physical * block_size + pos % block_size;
}

int pkv_oracle_kv_append(int dtype, void* k_cache, void* v_cache,
                         int64_t num_blocks, int block_size, int num_kv_heads,
                         int head_dim, const void* k, const void* v,
                         const int64_t* slots, int64_t num_tokens) {
  if (num_tokens < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ORACLE_BAD_ARG;
  const size_t row = (size_t)num_kv_heads * (size_t)head_dim * elem_bytes(dtype);
  const int64_t num_slots = num_blocks * (int64_t)block_size;
  int status = PKV_ORACLE_OK;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t s = slots[i];
    if (s < 0) continue;
    if (s >= num_slots) { status = PKV_ORACLE_BAD_SLOT; continue; }
    memcpy((unsigned char*)k_cache + (size_t)s * row,
           (const unsigned char*)k + (size_t)i * row, row);
    memcpy((unsigned char*)v_cache + (size_t)s * row,
           (const unsigned char*)v + (size_t)i * row, row);
  }
  return status;
}

int pkv_oracle_kv_block_copy(int dtype, void* k_cache, void* v_cache,
                             int64_t num_blocks, int block_size,
                             int num_kv_heads, int head_dim,
                             const int64_t* pairs, int64_t num_pairs) {
  if (num_pairs < 0 || block_size <= 0) return PKV_ORACLE_BAD_ARG;
  const size_t blk = (size_t)block_size * (size_t)num_kv_heads *
                     (size_t)head_dim * elem_bytes(dtype);
  int status = PKV_ORACLE_OK;
  for (int64_t i = 0; i < num_pairs; ++i) {
    int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      status = PKV_ORACLE_BAD_BLOCK;
      continue;
    }
    memmove((unsigned char*)k_cache + (size_t)dst * blk,
            (const unsigned char*)k_cache + (size_t)src * blk, blk);
    memmove((unsigned char*)v_cache + (size_t)dst * blk,
            (const unsigned char*)v_cache + (size_t)src * blk, blk);
  }
  return status;
}

/* Attention for one (sequence, query head) pair over a gathered history. */
static int decode_one(int dtype, const void* q, const void* k_cache,
                      const void* v_cache, int64_t num_blocks, int P, int Hkv,
                      int D, const int32_t* table, int max_blocks, int T,
                      int r, int h, int Hq, double scale, double* o,
                      double* lse_out, double* scores) {
  const int G = Hq / Hkv;
  const int kvh = h / G;
  const int64_t q_base = ((int64_t)r * Hq + h) * D;
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  if (T <= 0) {
    if (lse_out) *lse_out = -INFINITY;
    return PKV_ORACLE_OK;
  }
  /* scores over the request-visible tokens only */
  double m = -INFINITY;
  for (int t = 0; t < T; ++t) {
    int64_t blk, off;
    int st = pkv_oracle_resolve(table, max_blocks, T, P, num_blocks, t, &blk, &off);
    if (st != PKV_ORACLE_OK) return PKV_ORACLE_BAD_BLOCK;
    const int64_t k_base = ((blk * P + off) * Hkv + kvh) * (int64_t)D;
    double dot = 0.0;
    for (int c = 0; c < D; ++c)
      dot += load_elem(dtype, q, q_base + c) * load_elem(dtype, k_cache, k_base + c);
    scores[t] = scale * dot;
    if (scores[t] > m) m = scores[t];
  }
  double denom = 0.0;
  for (int t = 0; t < T; ++t) {
    double p = exp(scores[t] - m);
    denom += p;
    int64_t blk, off;
    pkv_oracle_resolve(table, max_blocks, T, P, num_blocks, t, &blk, &off);
    const int64_t v_base = ((blk * P + off) * Hkv + kvh) * (int64_t)D;
    for (int c = 0; c < D; ++c) o[c] += p * load_elem(dtype, v_cache, v_base + c);
  }
  for (int c = 0; c < D; ++c) o[c] /= denom;
  if (lse_out) *lse_out = m + log(denom);
  return PKV_ORACLE_OK;
}

int pkv_oracle_paged_decode(int dtype, const void* q, const void* k_cache,
                            const void* v_cache, int64_t num_blocks,
                            int block_size, int num_kv_heads, int head_dim,
                            const int32_t* block_tables, int max_blocks,
                            const int32_t* seq_lens, int num_seqs,
                            int num_q_heads, double scale, double* out,
                            double* lse, int nthreads) {
  if (num_seqs < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || max_blocks < 0)
    return PKV_ORACLE_BAD_ARG;
  int max_len = 0;
  for (int r = 0; r < num_seqs; ++r) {
    if (seq_lens[r] < 0) return PKV_ORACLE_BAD_ARG;
    if ((int64_t)seq_lens[r] > (int64_t)max_blocks * block_size)
      return PKV_ORACLE_BAD_ARG;
    if (seq_lens[r] > max_len) max_len = seq_lens[r];
  }
  const int64_t pairs = (int64_t)num_seqs * num_q_heads;
  int status = PKV_ORACLE_OK;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < pairs; ++i) {
      int r = (int)(i / num_q_heads), h = (int)(i % num_q_heads);
      int st = decode_one(dtype, q, k_cache, v_cache, num_blocks, block_size,
                          num_kv_heads, head_dim,
                          block_tables + (int64_t)r * max_blocks, max_blocks,
                          seq_lens[r], r, h, num_q_heads, scale,
                          out + i * head_dim, lse ? lse + i : NULL, scores);
      if (st != PKV_ORACLE_OK) {
#pragma omp critical
        status = st;
      }
    }
    free(scores);
  }
  return status;
}

int pkv_oracle_shared_prefix(int dtype, const void* q, const void* k_cache,
                             const void* v_cache, int64_t num_blocks,
                             int block_size, int num_kv_heads, int head_dim,
                             const int32_t* prefix_block_ids,
                             int32_t prefix_len,
                             const int32_t* suffix_block_tables,
                             int max_suffix_blocks,
                             const int32_t* suffix_lens, int num_seqs,
                             int num_q_heads, double scale, double* out,
                             double* lse, int nthreads) {
  if (block_size <= 0 || prefix_len < 0 || prefix_len % block_size != 0 ||
      max_suffix_blocks < 0 || num_seqs < 0)
    return PKV_ORACLE_BAD_ARG;
  const int npre = prefix_len / block_size;
  const int width = npre + max_suffix_blocks;
  int32_t* tables = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1) *
                                     (size_t)(width > 0 ? width : 1));
  int32_t* lens = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
  for (int r = 0; r < num_seqs; ++r) {
    for (int j = 0; j < npre; ++j) tables[(int64_t)r * width + j] = prefix_block_ids[j];
    for (int j = 0; j < max_suffix_blocks; ++j)
      tables[(int64_t)r * width + npre + j] =
          suffix_block_tables[(int64_t)r * max_suffix_blocks + j];
    lens[r] = prefix_len + suffix_lens[r];
  }
  int st = pkv_oracle_paged_decode(dtype, q, k_cache, v_cache, num_blocks,
                                   block_size, num_kv_heads, head_dim, tables,
                                   width, lens, num_seqs, num_q_heads, scale,
                                   out, lse, nthreads);
  free(tables);
  free(lens);
  return st;
}

int pkv_oracle_chunk_tree(int dtype, const void* q, const void* k_cache,
                          const void* v_cache, int64_t num_blocks,
                          int block_size, int num_kv_heads, int head_dim,
                          const int32_t* chunk_first_id,
                          const int32_t* chunk_lens,
                          const int32_t* chunk_begin, const int32_t* chunk_end,
                          int num_chunks, const int32_t* block_ids,
                          int64_t num_block_ids, int num_seqs, int num_q_heads,
                          double scale, double* out, double* lse,
                          int nthreads) {
  if (block_size <= 0 || num_blocks <= 0 || num_chunks < 0 || num_seqs < 0)
    return PKV_ORACLE_BAD_ARG;
  const int64_t P = block_size;
  for (int c = 0; c < num_chunks; ++c) {
    if (chunk_lens[c] < 1 || chunk_first_id[c] < 0 || chunk_begin[c] < 0 ||
        chunk_begin[c] >= chunk_end[c] || chunk_end[c] > num_seqs)
      return PKV_ORACLE_BAD_ARG;
    if ((int64_t)chunk_first_id[c] + (chunk_lens[c] + P - 1) / P > num_block_ids)
      return PKV_ORACLE_BAD_ARG;
  }
  /* each sequence's history length: the rows of the chunks on its path */
  int32_t* lens = (int32_t*)calloc((size_t)(num_seqs > 0 ? num_seqs : 1), sizeof(int32_t));
  int width = 0;
  for (int r = 0; r < num_seqs; ++r) {
    int64_t T = 0;
    for (int c = 0; c < num_chunks; ++c)
      if (chunk_begin[c] <= r && r < chunk_end[c]) T += chunk_lens[c];
    if (T > INT32_MAX) {
      free(lens);
      return PKV_ORACLE_BAD_ARG;
    }
    lens[r] = (int32_t)T;
    if (lens[r] > width) width = lens[r];
  }
  /* slot table of every history: row t of chunk c is pool slot
   * block * P + t % P, i.e. block (block * P + t % P) of a one-row pool */
  int32_t* slots = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1) *
                                    (size_t)(width > 0 ? width : 1));
  int status = PKV_ORACLE_OK;
  for (int r = 0; r < num_seqs && status == PKV_ORACLE_OK; ++r) {
    int64_t pos = 0;
    for (int c = 0; c < num_chunks && status == PKV_ORACLE_OK; ++c) {
      if (!(chunk_begin[c] <= r && r < chunk_end[c])) continue;
      for (int64_t t = 0; t < chunk_lens[c]; ++t) {
        const int64_t blk = block_ids[chunk_first_id[c] + t / P];
        if (blk < 0 || blk >= num_blocks || blk * P + P - 1 > INT32_MAX) {
          status = PKV_ORACLE_BAD_BLOCK;
          break;
        }
        slots[(int64_t)r * width + pos++] = (int32_t)(blk * P + t % P);
      }
    }
  }
  if (status == PKV_ORACLE_OK)
    status = pkv_oracle_paged_decode(dtype, q, k_cache, v_cache, num_blocks * P, 1,
                                     num_kv_heads, head_dim, slots, width, lens, num_seqs,
                                     num_q_heads, scale, out, lse, nthreads);
  free(slots);
  free(lens);
  return status;
}

int pkv_oracle_row_ledger(const int32_t* block_tables, int max_blocks,
                          const int32_t* seq_lens, int num_seqs,
                          int64_t num_blocks, int block_size,
                          int64_t* logical_rows, int64_t* unique_rows) {
  if (num_blocks <= 0 || block_size <= 0) return PKV_ORACLE_BAD_ARG;
  const int64_t nslots = num_blocks * (int64_t)block_size;
  unsigned char* seen = (unsigned char*)calloc((size_t)(nslots + 7) / 8, 1);
  int64_t logical = 0, unique = 0;
  int status = PKV_ORACLE_OK;
  for (int r = 0; r < num_seqs; ++r) {
    const int32_t* table = block_tables + (int64_t)r * max_blocks;
    for (int64_t t = 0; t < seq_lens[r]; ++t) {
      int64_t blk, off;
      int st = pkv_oracle_resolve(table, max_blocks, seq_lens[r], block_size,
                                  num_blocks, t, &blk, &off);
      if (st != PKV_ORACLE_OK) { status = st; continue; }
      ++logical;
      int64_t s = blk * block_size + off;
      if (!(seen[s >> 3] & (1u << (s & 7)))) {
        seen[s >> 3] |= (unsigned char)(1u << (s & 7));
        ++unique;
      }
    }
  }
  free(seen);
  *logical_rows = logical;
  *unique_rows = unique;
  return status;
}

int pkv_oracle_expand_table(const int32_t* table, int64_t n, int32_t q, int32_t* out) {
  if (q < 1 || n < 0) return PKV_ORACLE_BAD_ARG;
  for (int64_t c = 0; c < n; ++c) {
    const int32_t a = table[c];
    for (int32_t j = 0; j < q; ++j) {
      if (a < 0) {
        out[c * q + j] = -1;
        continue;
      }
      const int64_t k = (int64_t)a * q + j;
      if (k > INT32_MAX) return PKV_ORACLE_BAD_ARG;
      out[c * q + j] = (int32_t)k;
    }
  }
  return PKV_ORACLE_OK;
}
