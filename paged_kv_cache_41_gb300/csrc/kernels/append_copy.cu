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

// MXFP8 append: one warp per (token, kv head) row of D bf16 elements, each
// lane EPL = D / 32 consecutive ones, so a 32-element scale group is 32 / EPL
// lanes.  The group's scale is the smallest power of two X with
// max |x| / X <= 448 (E4M3's largest finite value): for max |x| = (1 + f)
// 2^E (fp32 fields), X = 2^(E - 8), or 2^(E - 7) when 1 + f > 1.75; zero and
// subnormal maxima take the smallest scale.  Elements are x / X (exact: a
// power-of-two multiply) rounded to the nearest E4M3 code, ties to even.
template <int D>
__global__ void __launch_bounds__(256) kv_append_mxfp8_kernel(
    uint8_t* __restrict__ kc, uint8_t* __restrict__ vc, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const int64_t* __restrict__ slots, int64_t num_tokens,
    int num_kv_heads, int block_size, int64_t num_slots, int64_t plane_bytes,
    unsigned int* err) {
  constexpr int EPL = D / 32;          // elements per lane
  constexpr int LPG = 32 / EPL;        // lanes per scale group
  pdl_launch_dependents();
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
  const int lane = threadIdx.x & 31;
  const int H = num_kv_heads, P = block_size;
  if (row >= num_tokens * H) return;
  const int64_t tok = row / H;
  const int h = (int)(row % H);
  const int64_t s = slots[tok];
  if (s < 0) return;  // skip sentinel
  if (s >= num_slots) {
    if (lane == 0 && h == 0) atomicOr(err, PKV_DEVERR_SLOT);
    return;
  }
  const int64_t blk = s / P, off = s % P;
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const __nv_bfloat16* src = (kv ? v : k) + row * D + lane * EPL;
    uint8_t* cache = kv ? vc : kc;
    float x[EPL];
    if constexpr (EPL == 4) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
      x[0] = bf16lo(w.x);
      x[1] = bf16hi(w.x);
      x[2] = bf16lo(w.y);
      x[3] = bf16hi(w.y);
    } else {
      const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(src));
      x[0] = bf16lo(w);
      x[1] = bf16hi(w);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 1; o < LPG; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const uint32_t bits = __float_as_uint(amax);
    const int E = (int)(bits >> 23) - 127;
    int e = E - 8 + ((bits & 0x7fffffu) > 0x600000u ? 1 : 0);
    if ((bits >> 23) == 0 || e < -127) e = -127;  // zero or tiny group
    const uint32_t sbyte = (uint32_t)(e + 127);
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, e in [-127, 126]
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < EPL; i += 2) {
      const __nv_fp8x2_storage_t q2 =
          __nv_cvt_float2_to_fp8x2(make_float2(x[i] * inv, x[i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
      packed |= (uint32_t)q2 << (8 * i);
    }
    uint8_t* dst = cache + ((blk * P + off) * H + h) * D + lane * EPL;
    if constexpr (EPL == 4)
      *reinterpret_cast<uint32_t*>(dst) = packed;
    else
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    if (lane % LPG == 0)
      cache[plane_bytes + ((blk * H + h) * P + off) * (D / 32) + lane / LPG] = (uint8_t)sbyte;
  }
}

cudaError_t launch_kv_append_mxfp8(void* k_cache, void* v_cache, const void* k, const void* v,
                                   const int64_t* slots, int64_t num_tokens, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_slots,
                                   int64_t plane_bytes, unsigned int* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int warps = 8;
  const int64_t rows = num_tokens * num_kv_heads;
  const unsigned grid = (unsigned)((rows + warps - 1) / warps);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  auto* kk = static_cast<const __nv_bfloat16*>(k);
  auto* vv = static_cast<const __nv_bfloat16*>(v);
  if (head_dim == 128)
    kv_append_mxfp8_kernel<128><<<grid, warps * 32, 0, stream>>>(
        kc, vc, kk, vv, slots, num_tokens, num_kv_heads, block_size, num_slots, plane_bytes, err);
  else
    kv_append_mxfp8_kernel<64><<<grid, warps * 32, 0, stream>>>(
        kc, vc, kk, vv, slots, num_tokens, num_kv_heads, block_size, num_slots, plane_bytes, err);
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
