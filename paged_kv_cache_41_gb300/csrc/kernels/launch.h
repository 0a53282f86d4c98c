// launch.h -- internal launchers behind the libpkv C ABI (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

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

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k, const void* v,
                             const int64_t* slots, int64_t num_tokens, int64_t num_slots,
                             int64_t row_bytes, unsigned int* err, cudaStream_t stream);

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

// Arguments of the split-K paged decode kernels.
struct DecodeArgs {
  const void* q;                // [B, Hq, D]
  const int32_t* block_tables;  // [B, max_blocks]
  const int32_t* seq_lens;      // [B]
  float* part_o;                // [B, Hq, parts_stride, D] normalised partial outputs
  float* part_lse;              // [B, Hq, parts_stride] partial LSE, base 2
  void* out;                    // [B, Hq, D]
  float* lse_out;               // [B, Hq] natural log, or null
  unsigned int* err;
  int64_t num_blocks;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t blocks_per_part;
  int32_t max_parts;     // partitions per sequence at most (grid.y)
  int32_t part_offset;   // partial slots before the first decode partition
  int32_t parts_stride;  // partial slots per (sequence, head)
  int32_t num_stages;
  float qscale;          // softmax scale * log2(e)
  int32_t direct;        // 1: a single partition per sequence writes out/lse itself
};

// Launch the partial kernel (and the LSE reduction unless args.direct).
cudaError_t launch_paged_decode(int dtype, int head_dim, int group, const CUtensorMap& tmk,
                                const CUtensorMap& tmv, const DecodeArgs& args,
                                cudaStream_t stream);

// LSE reduction over the partial states (also used after the shared prefix).
cudaError_t launch_decode_reduce(int dtype, int head_dim, const DecodeArgs& args,
                                 cudaStream_t stream);

// Arguments of the shared-prefix tensor-core kernel.  Grid: (key split,
// 128-row query tile, kv head).  Its states go to partial slots
// [0, num_splits) of the same workspace layout the decode kernels use.
struct PrefixArgs {
  const int32_t* prefix_block_ids;  // [ceil(prefix_len / P)]
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
  float qscale;          // softmax scale * log2(e)
  float lse_scale;       // 1: LSE in base 2 (partial states); ln 2: natural log
};

// Query rows per CTA and keys per tile of the prefix kernel.
constexpr int kPrefixRows = 128;
constexpr int kPrefixKeys = 128;

cudaError_t launch_prefix_attention(int head_dim, int group, int num_splits,
                                    const CUtensorMap& tmq, const CUtensorMap& tmk,
                                    const CUtensorMap& tmv, const PrefixArgs& args,
                                    cudaStream_t stream);
size_t prefix_smem_bytes(int head_dim, int split_len, int block_size);

// Stage count and dynamic shared memory of the partial kernel.
int decode_num_stages(int block_size, int head_dim, int elem_bytes);
size_t decode_smem_bytes(int block_size, int head_dim, int elem_bytes, int group, int stages);

}  // namespace pkv
