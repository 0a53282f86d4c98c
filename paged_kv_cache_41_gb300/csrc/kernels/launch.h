// launch.h -- internal launchers behind the libpkv C ABI (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

namespace pkv {

// Raise a kernel's dynamic shared-memory limit once per device: the attribute
// persists, so later launches that need no more skip the driver call.
struct SmemAttrCache {
  std::mutex mu;
  int set[64] = {};
};

template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kern, int smem, SmemAttrCache& cache) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(cache.mu);
  if (dev >= 0 && dev < 64 && cache.set[dev] >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cache.set[dev] = smem;
  return e;
}

// Launch `kern` so that it may be scheduled while the previous kernel of the
// stream finishes (programmatic dependent launch); the kernel must call
// pdl_wait() before it reads anything an earlier kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k, const void* v,
                             const int64_t* slots, int64_t num_tokens, int64_t num_slots,
                             int64_t row_bytes, unsigned int* err, cudaStream_t stream);

cudaError_t launch_expand_block_tables(const int32_t* in, int64_t n_in, int32_t q, int32_t* out,
                                       unsigned int* err, cudaStream_t stream);

// MXFP8 pools (include/pkv.h): quantize bf16 rows into the element and
// scale planes; plane_bytes = NB * P * Hkv * D, head_dim 64 or 128.
cudaError_t launch_kv_append_mxfp8(void* k_cache, void* v_cache, const void* k, const void* v,
                                   const int64_t* slots, int64_t num_tokens, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_slots,
                                   int64_t plane_bytes, unsigned int* err, cudaStream_t stream);
cudaError_t launch_kv_block_copy(void* k_cache, void* v_cache, const int64_t* pairs,
                                 int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                                 unsigned int* err, cudaStream_t stream);

// Token rows per shared-memory stage of the decode kernel, and the rows of
// one TMA box: a box covers one block, or kStageRows rows of a larger block.
// Block sizes must divide kStageRows or be a multiple of it.
constexpr int kStageRows = 32;
__host__ __device__ constexpr int box_rows_for(int block_size) {
  return block_size < kStageRows ? block_size : kStageRows;
}

// Arguments of the paged decode kernels.
//
// Work list: every (sequence, kv head) segment of ceil(T / kStageRows)
// stages, sequence-major then kv head; S stages in all.  CTA c of C streams
// stages [c w, min((c + 1) w, S)), w = ceil(S / C).  A segment a CTA covers
// whole is written out directly; a segment cut by a CTA boundary leaves one
// record per piece, slot 0 of its CTA for the piece holding the CTA's first
// stage and slot 1 for a last piece that is not also the first.
struct DecodeArgs {
  const void* q;                // [B_q, Hq, D] (bf16 beside an MXFP8 pool)
  const uint8_t* k_scales;      // MXFP8 pools: the scale planes [NB, Hkv, P, D / 32]
  const uint8_t* v_scales;
  const int32_t* q_rows;        // [B] query row of each sequence, or null: row r
  const int32_t* block_tables;  // [B, max_blocks]
  const int32_t* seq_lens;      // [B]
  void* out;                    // [B, Hq, D]
  float* lse_out;               // [B, Hq] natural log, or null
  unsigned int* err;
  int64_t* plan_pre;            // [B + 1] exclusive prefix of work units per sequence (CTA 0 writes)
  float* rec_o;                 // [2C, G, D] normalised piece outputs
  float* rec_lse;               // [2C, G] piece LSEs, base 2
  // States mode (shared prefix): a whole segment writes (O, LSE base 2) to
  // slot st_slot of st_o / st_lse instead of out, and the reduction also
  // merges the st_slot extra states held in slots [0, st_slot).  With out ==
  // nullptr as well (states only), the reduction writes its merge to slot
  // st_slot instead of out.  Plain decode: st_o == nullptr.
  float* st_o;                  // [B, Hq, st_stride, D]
  float* st_lse;                // [B, Hq, st_stride]
  int32_t st_stride;
  int32_t st_slot;
  int64_t num_blocks;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t num_ctas;      // C
  int32_t num_stages;    // shared-memory ring depth
  int32_t stage_units;   // work units of one stage (>= 1) ...
  int32_t piece_units;   // ... and of a piece's fixed cost (>= 0): the split of plan.cuh
  // 1: the length scan of the split (seq_lens in, plan_pre out) and the
  // first batch of stage descriptors (block_tables, q_rows in) run before
  // the wait on the preceding kernel, under its tail.  Set where that kernel
  // is this library's (the prefix kernel, kv_append), which writes none of
  // them, or, for the plain decode, as its interface documents.
  int32_t plan_before_wait;
  float qscale;          // softmax scale * log2(e)
};

// Partial kernel, then the LSE reduction of cut segments, on one stream.
cudaError_t launch_paged_decode(int dtype, int head_dim, int group, const CUtensorMap& tmk,
                                const CUtensorMap& tmv, const DecodeArgs& args,
                                cudaStream_t stream);

// CTAs of one wave of the partial kernel (resident CTAs per SM x SMs).
int decode_resident_ctas(int dtype, int head_dim, int group);

// The LSE reduction of cut segments (and, in states mode, extra states).
cudaError_t launch_decode_reduce(int dtype, int head_dim, const DecodeArgs& args,
                                 cudaStream_t stream);

// Tensor-core decode for eight query heads per kv head (decode_tc.cu): bf16,
// head_dim 128, block sizes dividing 128 or multiples of it.  Stages are
// decode_tc_rows() rows; one CTA per SM.  tmk / tmv: row-group maps (above)
// whose box is min(P, 128) rows of one head, both halves; tmq: a
// 128-byte-swizzled map over q [B, Hq, D] whose box is 64 columns x 8 heads
// x 1 request.  Launches the reduction too.
bool decode_tc_supported(int dtype, int head_dim, int group, int block_size);
// The tensor-core decode over MXFP8 pools (decode_tc_mx.cu): tmk / tmv are
// 4-D uint8 maps over the element planes whose box is 128-byte rows x
// min(P, 128) rows; the scale planes come in args.  Launches the reduction.
bool decode_tc_mx_supported(int dtype, int head_dim, int group, int block_size);
int decode_tc_mx_resident_ctas();
cudaError_t launch_paged_decode_tc_mx(int group, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                      const CUtensorMap& tmq, const DecodeArgs& args,
                                      cudaStream_t stream);
int decode_tc_rows();
int decode_tc_resident_ctas();
cudaError_t launch_paged_decode_tc(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                   const CUtensorMap& tmq, const DecodeArgs& args,
                                   cudaStream_t stream);

// One CTA's work when the prefix kernel runs over a list of chunks (the
// chunk-first phase of a prefix tree): one key split of one chunk against up
// to two 128-row query tiles of the sequences the chunk covers.
struct PrefixItem {
  int32_t ids_off;  // index in prefix_block_ids of the chunk's first block
  int32_t key0;     // first key of the split, counted from the chunk's start
  int32_t nkeys;    // keys in the split (>= 1)
  int32_t req0;     // q row (sequence) of query tile A's first request
  int32_t nreq;     // requests of the pair, <= 2 * 128 / G (tile B iff > 128 / G)
  int32_t st_req0;  // state row of tile A's first request
  int32_t split;    // state slot
  int32_t pad;
};

// Arguments of the shared-prefix tensor-core kernel.  Grid: (key split,
// 128-row query tile pair, kv head) over one prefix, or (item, 1, kv head)
// with an item list.  Its states go to slots [0, num_splits) of
// [rows, Hq, parts_stride] state arrays.
struct PrefixArgs {
  const int32_t* prefix_block_ids;  // [ceil(prefix_len / P)], or every chunk's ids
  const PrefixItem* items;          // [num_items], or null: one prefix over all sequences
  float* part_o;                    // [B, Hq, parts_stride, D]
  float* part_lse;                  // [B, Hq, parts_stride], base 2
  unsigned int* err;
  int64_t num_blocks;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t prefix_len;
  int32_t split_len;     // keys per split, a multiple of 128
  int32_t parts_stride;
  int32_t num_items;
  float qscale;          // softmax scale * log2(e)
  float lse_scale;       // 1: LSE in base 2 (partial states); ln 2: natural log
};

// Arguments of the merge at the end of attention over a prefix tree.
// Sequence r merges states [seq_ptr[r], seq_ptr[r + 1]) of `states`; state
// reference (base, head_stride) names, for query head h, the state at index
// base + h * head_stride of st_o ([.., D] fp32) and st_lse (base 2).
struct TreeMergeArgs {
  const float* st_o;
  const float* st_lse;
  const int32_t* seq_ptr;     // [B + 1]
  const int64_t* states;      // [seq_ptr[B]][2]: (base, head_stride)
  void* out;                  // [B, Hq, D]
  float* lse_out;             // [B, Hq] natural log, or null
  int32_t num_seqs;
  int32_t num_q_heads;
};
cudaError_t launch_tree_merge(int dtype, int head_dim, const TreeMergeArgs& args,
                              cudaStream_t stream);

// Row-group tiles.  The tensor-core kernels stage K and V tiles of bf16 rows
// with the 128-byte swizzle as 8-row atoms interleaved by row group: row r,
// 64-column half h of a tile lies at (r / 8) * (D / 64) KiB + h KiB +
// (r % 8) * 128 B.  A TMA box then brings whole blocks, both halves at once
// (a 16-row block of head_dim 128 is one 4 KiB box instead of two 2 KiB
// ones): the map is 5-D over the pool, (64 columns, 8 rows, D / 64 halves,
// Hkv, NB * P / 8 row groups), and a block's box starts at row group
// block * P / 8 + first row / 8.  K-major operands read it with 8-row groups
// (D / 64) KiB apart; MN-major ones with 64-element halves 1 KiB apart.
constexpr int kRowGroup = 8;

// Query rows per CTA and keys per tile of the prefix kernel.
constexpr int kPrefixRows = 128;
constexpr int kPrefixKeys = 128;

// tmo: the state outputs part_o as a 5-D fp32 tensor (D, parts_stride, G,
// Hkv, num_seqs) with 128-byte swizzle and a box of 32 columns x 1 x G x 1 x
// 128 / G requests.
cudaError_t launch_prefix_attention(int head_dim, int group, int num_splits,
                                    const CUtensorMap& tmq, const CUtensorMap& tmk,
                                    const CUtensorMap& tmv, const CUtensorMap& tmo,
                                    const PrefixArgs& args, cudaStream_t stream);
size_t prefix_smem_bytes(int head_dim, int split_len, int block_size);

// Stage count of the partial kernel's shared-memory ring.
int decode_num_stages(int head_dim, int elem_bytes);

}  // namespace pkv
