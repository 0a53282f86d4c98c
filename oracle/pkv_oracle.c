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

int pkv_oracle_slots_for_positions(const int32_t* tables, int64_t table_stride,
                                   const int32_t* rows, const int64_t* positions, int64_t n,
                                   int64_t block_size, int64_t* out) {
  if (n < 0 || table_stride <= 0 || block_size <= 0) return PKV_ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (rows[i] < 0 || positions[i] < 0 || positions[i] / block_size >= table_stride)
      return PKV_ORACLE_BAD_ARG;
    out[i] = pkv_oracle_slot_for_position(tables + (int64_t)rows[i] * table_stride, block_size,
                                          positions[i]);
  }
  return PKV_ORACLE_OK;
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

/* ---------------------------------------------------------------- MXFP8 */

double pkv_oracle_e4m3_decode(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m, -9)               /* m/8 * 2^-6 */
                            : ldexp(8.0 + m, e - 10);             /* (1 + m/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

uint8_t pkv_oracle_e4m3_encode_exhaustive(double x) {
  const uint8_t sign = x < 0 || (x == 0 && signbit(x)) ? 0x80 : 0;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E; /* saturate */
  /* candidates are the finite codes 0..126 in increasing magnitude: find the
   * nearest, ties to the even code (even mantissa) */
  uint8_t best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double d = fabs(pkv_oracle_e4m3_decode((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = (uint8_t)c;
      best_d = d;
    }
  }
  return sign | best;
}

uint8_t pkv_oracle_e4m3_encode(double x) {
  const uint8_t sign = x < 0 || (x == 0 && signbit(x)) ? 0x80 : 0;
  const double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E; /* 448 and beyond: the largest finite */
  if (a < 0.015625) {                 /* below 2^-6: subnormal steps of 2^-9 */
    /* rint rounds to nearest, ties to even (the default mode); 8 steps of
     * 2^-9 is 2^-6, the smallest normal, which is code 8 */
    return sign | (uint8_t)rint(ldexp(a, 9));
  }
  int k;
  frexp(a, &k);                       /* a = f 2^k, f in [0.5, 1) */
  int E = k - 1;                      /* a = s 2^E, s in [1, 2) */
  int q = (int)rint((ldexp(a, -E) - 1.0) * 8.0);  /* 3 mantissa bits, ties to even */
  if (q == 8) {                       /* rounded up to the next power of two */
    q = 0;
    ++E;
  }
  return sign | (uint8_t)(((E + 7) << 3) | q);
}

uint8_t pkv_oracle_mx_scale(double amax) {
  if (!(amax > 0)) return 0;
  /* the smallest e with amax <= 448 * 2^e: a first guess from the binary
   * exponent of amax / 448, settled by exact comparisons (448 * 2^e is exact
   * in binary64) */
  int k;
  frexp(amax / 448.0, &k);
  int e = k;
  while (e > -127 && amax <= ldexp(448.0, e - 1)) --e;
  while (e < 127 && amax > ldexp(448.0, e)) ++e;
  if (e < -127) e = -127;
  return (uint8_t)(e + 127);
}

static double load_in(int in_dtype, const void* base, int64_t idx) {
  return load_elem(in_dtype, base, idx);
}

int pkv_oracle_kv_append_mxfp8(int in_dtype, uint8_t* k_cache, uint8_t* v_cache,
                               int64_t num_blocks, int block_size,
                               int num_kv_heads, int head_dim, const void* k,
                               const void* v, const int64_t* slots,
                               int64_t num_tokens) {
  if (num_tokens < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 32 != 0)
    return PKV_ORACLE_BAD_ARG;
  const int64_t P = block_size, H = num_kv_heads, D = head_dim;
  const int64_t num_slots = num_blocks * P;
  const int64_t plane = num_blocks * P * H * D;
  int status = PKV_ORACLE_OK;
  for (int64_t i = 0; i < num_tokens; ++i) {
    const int64_t s = slots[i];
    if (s < 0) continue;
    if (s >= num_slots) { status = PKV_ORACLE_BAD_SLOT; continue; }
    const int64_t blk = s / P, off = s % P;
    for (int kv = 0; kv < 2; ++kv) {
      const void* src = kv ? v : k;
      uint8_t* cache = kv ? v_cache : k_cache;
      for (int64_t h = 0; h < H; ++h) {
        for (int64_t g = 0; g < D / 32; ++g) {
          const int64_t in0 = (i * H + h) * D + g * 32;
          double amax = 0;
          for (int j = 0; j < 32; ++j) {
            const double x = fabs(load_in(in_dtype, src, in0 + j));
            if (x > amax) amax = x;
          }
          const uint8_t sc = pkv_oracle_mx_scale(amax);
          cache[plane + ((blk * H + h) * P + off) * (D / 32) + g] = sc;
          for (int j = 0; j < 32; ++j) {
            const double x = load_in(in_dtype, src, in0 + j);
            cache[((blk * P + off) * H + h) * D + g * 32 + j] =
                pkv_oracle_e4m3_encode(ldexp(x, 127 - (int)sc));
          }
        }
      }
    }
  }
  return status;
}

int pkv_oracle_mxfp8_to_f32(const uint8_t* cache, int64_t num_blocks,
                            int block_size, int num_kv_heads, int head_dim,
                            float* out) {
  if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim % 32 != 0)
    return PKV_ORACLE_BAD_ARG;
  const int64_t P = block_size, H = num_kv_heads, D = head_dim;
  const int64_t plane = num_blocks * P * H * D;
  for (int64_t b = 0; b < num_blocks; ++b)
    for (int64_t o = 0; o < P; ++o)
      for (int64_t h = 0; h < H; ++h)
        for (int64_t c = 0; c < D; ++c) {
          const int64_t e = ((b * P + o) * H + h) * D + c;
          const int sc = cache[plane + ((b * H + h) * P + o) * (D / 32) + c / 32];
          out[e] = (float)ldexp(pkv_oracle_e4m3_decode(cache[e]), sc - 127);
        }
  return PKV_ORACLE_OK;
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
