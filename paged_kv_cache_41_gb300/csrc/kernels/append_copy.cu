// append_copy.cu -- K/V append scatter and copy-on-write block copy.
//
// Both are byte copies of whole 16-byte vectors, bit-exact by construction.
//   kv_append: "M5.3 - KV Memory Layout and Exact Reuse" 0x03D (slot id =
//     block * P + offset), 0x04E (append writes row o of the tail block);
//     "Cache Concepts: Prefix Matching vs. Storage" (slot invariant and the -1
//     skip sentinel).  Row i of k/v (Hkv * D elements, contiguous) lands at
//     cache row slot_mapping[i] of the [NB * P, Hkv * D] view of the pool.
//   kv_block_copy: M5.3 0x04C / 0x05A and the fused block-copy kernel of
//     PagedAttention: whole blocks, K and V, for every (src, dst) pair.
//   expand_block_tables: M5.3 0x0AC, allocator blocks of P_a = q P_k rows
//     split into q kernel blocks: id a becomes a q .. a q + q - 1.
#include "common.cuh"
#include "launch.h"

namespace pkv {

// One warp per token row; each lane moves 16-byte vectors of K then of V.
__global__ void __launch_bounds__(256) kv_append_kernel(uint4* __restrict__ kc,
                                                        uint4* __restrict__ vc,
                                                        const uint4* __restrict__ k,
                                                        const uint4* __restrict__ v,
                                                        const int64_t* __restrict__ slots,
                                                        int64_t num_tokens, int64_t num_slots,
                                                        int64_t row_vecs, unsigned int* err) {
  pdl_launch_dependents();  // a decode after this append may be scheduled now
  const int64_t tok = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
  const int lane = threadIdx.x & 31;
  if (tok >= num_tokens) return;
  const int64_t s = slots[tok];
  if (s < 0) return;  // skip sentinel
  if (s >= num_slots) {
    if (lane == 0) atomicOr(err, PKV_DEVERR_SLOT);
    return;
  }
  const uint4* ks = k + tok * row_vecs;
  const uint4* vs = v + tok * row_vecs;
  uint4* kd = kc + s * row_vecs;
  uint4* vd = vc + s * row_vecs;
  for (int64_t i = lane; i < row_vecs; i += 32) {
    uint4 a = __ldg(ks + i);
    uint4 b = __ldg(vs + i);
    kd[i] = a;
    vd[i] = b;
  }
}

cudaError_t launch_kv_append(void* k_cache, void* v_cache, const void* k, const void* v,
                             const int64_t* slots, int64_t num_tokens, int64_t num_slots,
                             int64_t row_bytes, unsigned int* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int warps = 8;
  const int64_t grid = (num_tokens + warps - 1) / warps;
  kv_append_kernel<<<(unsigned)grid, warps * 32, 0, stream>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), static_cast<const uint4*>(k),
      static_cast<const uint4*>(v), slots, num_tokens, num_slots, row_bytes / 16, err);
  return cudaGetLastError();
}

// grid.x = pair, grid.y = 0 (K) / 1 (V), grid.z = chunk of the block.
constexpr int kCopyThreads = 256;
constexpr int kCopyVecsPerThread = 4;

__global__ void __launch_bounds__(kCopyThreads) kv_block_copy_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, const int64_t* __restrict__ pairs,
    int64_t num_blocks, int64_t block_vecs, unsigned int* err) {
  const int64_t src = pairs[2 * (int64_t)blockIdx.x];
  const int64_t dst = pairs[2 * (int64_t)blockIdx.x + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(err, PKV_DEVERR_BLOCK);
    return;
  }
  uint4* base = blockIdx.y == 0 ? kc : vc;
  const uint4* s = base + src * block_vecs;
  uint4* d = base + dst * block_vecs;
  const int64_t chunk = (int64_t)kCopyThreads * kCopyVecsPerThread;
  const int64_t lo = (int64_t)blockIdx.z * chunk;
  uint4 tmp[kCopyVecsPerThread];
#pragma unroll
  for (int j = 0; j < kCopyVecsPerThread; ++j) {
    const int64_t i = lo + j * kCopyThreads + threadIdx.x;
    if (i < block_vecs) tmp[j] = __ldg(s + i);
  }
#pragma unroll
  for (int j = 0; j < kCopyVecsPerThread; ++j) {
    const int64_t i = lo + j * kCopyThreads + threadIdx.x;
    if (i < block_vecs) d[i] = tmp[j];
  }
}

// One thread per output entry: out[i] = in[i / q] * q + i % q, padding kept.
__global__ void __launch_bounds__(256) expand_block_tables_kernel(const int32_t* __restrict__ in,
                                                                  int64_t n_out, int32_t q,
                                                                  int32_t* __restrict__ out,
                                                                  unsigned int* err) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_out) return;
  const int32_t a = __ldg(in + i / q);
  int32_t v = -1;
  if (a >= 0) {
    const int64_t k = (int64_t)a * q + i % q;
    if (k > INT32_MAX) atomicOr(err, PKV_DEVERR_BLOCK);
    else v = (int32_t)k;
  }
  out[i] = v;
}

cudaError_t launch_expand_block_tables(const int32_t* in, int64_t n_in, int32_t q, int32_t* out,
                                       unsigned int* err, cudaStream_t stream) {
  const int64_t n_out = n_in * q;
  if (n_out == 0) return cudaSuccess;
  expand_block_tables_kernel<<<(unsigned)((n_out + 255) / 256), 256, 0, stream>>>(in, n_out, q,
                                                                                 out, err);
  return cudaGetLastError();
}

cudaError_t launch_kv_block_copy(void* k_cache, void* v_cache, const int64_t* pairs,
                                 int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                                 unsigned int* err, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t block_vecs = block_bytes / 16;
  const int64_t chunk = (int64_t)kCopyThreads * kCopyVecsPerThread;
  dim3 grid((unsigned)num_pairs, 2, (unsigned)((block_vecs + chunk - 1) / chunk));
  kv_block_copy_kernel<<<grid, kCopyThreads, 0, stream>>>(static_cast<uint4*>(k_cache),
                                                          static_cast<uint4*>(v_cache), pairs,
                                                          num_blocks, block_vecs, err);
  return cudaGetLastError();
}

}  // namespace pkv
