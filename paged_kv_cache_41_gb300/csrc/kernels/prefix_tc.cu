// prefix_tc.cu -- shared-prefix attention on the tcgen05 tensor cores.
//
// What it computes ("M5.3 - KV Memory Layout and Exact Reuse", 0x0BC,
// Hydragen): requests that share one refcounted prefix read the same physical
// K/V blocks, so for each kv head the prefix part of attention is one dense
// contraction of all B*G query rows of that head against the prefix keys,
// instead of B matrix-vector passes over the same bytes.  Each CTA emits, for
// its query rows and its slice of the prefix keys, the state (O_p = u / l,
// LSE_p = m + log2 l) of 0x0BA; the LSE reduction merges those states with
// the paged suffix partitions, so the result equals attention over
// prefix ++ suffix exactly (never an average of normalised outputs).
//
// Design (GB300):
//   * CTA = (key split, 128 query rows, kv head); thread t owns query row t,
//     i.e. TMEM lane t, so the softmax needs no cross-thread reduction;
//   * Q (128 rows x D), K and V tiles (128 keys x D) arrive by TMA with
//     128-byte swizzle, directly in the canonical K-major layout the UMMA
//     descriptors expect; K/V blocks are gathered through the prefix's block
//     ids, keys past the prefix read a zero-filled out-of-range box;
//   * S = Q K^T and O += P V are tcgen05.mma (bf16 in, fp32 accumulate in
//     TMEM); S is double-buffered in TMEM so QK^T of tile j+1 runs while the
//     softmax of tile j does; K and V are double-buffered in shared memory;
//   * P is rounded to bf16 and written in the swizzled K-major layout for the
//     PV MMA; V is consumed MN-major (no transpose);
//   * the exponent base moves only when a row's max grows past 2^8 (exact);
//     the rare rescale of O is a TMEM load/multiply/store of that row.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kHalfBytes = kPrefixRows * 128;  // one 64-column half of a 128-row tile

__host__ __device__ constexpr int prefix_tile_bytes(int head_dim) {
  return (head_dim / 64) * kHalfBytes;
}

}  // namespace

size_t prefix_smem_bytes(int head_dim, int split_len, int block_size) {
  const size_t tiles = (size_t)5 * prefix_tile_bytes(head_dim) + 2 * kHalfBytes;  // Q, K[2], V[2], P
  const size_t ids = ((size_t)split_len / block_size + 2) * sizeof(int);
  return tiles + ((ids + 15) & ~(size_t)15) + 1024;  // +1024: base alignment
}

template <int D, int G>
__global__ void __launch_bounds__(128, 1)
    prefix_attention_kernel(const __grid_constant__ CUtensorMap tmq,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const PrefixArgs a) {
  constexpr int H = D / 64;                  // 64-column halves of a row
  constexpr int RPB = kPrefixRows / G;       // requests per CTA
  constexpr uint32_t kTile = prefix_tile_bytes(D);
  constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kPrefixRows, kPrefixKeys, 0, 0);
  constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kPrefixRows, D, 0, 1);

  const int split = blockIdx.x, mt = blockIdx.y, kvh = blockIdx.z;
  const int P = a.block_size;
  const int PB = prefix_box_rows(P);
  const int key0 = split * a.split_len;
  const int nkeys = min(a.split_len, a.prefix_len - key0);
  if (nkeys <= 0) return;
  const int J = (nkeys + kPrefixKeys - 1) / kPrefixKeys;
  const int id0 = key0 / P;
  const int nid = (key0 + nkeys - 1) / P - id0 + 1;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* qs = sm;
  unsigned char* ks = qs + kTile;          // two stages
  unsigned char* vs = ks + 2 * kTile;      // two stages
  unsigned char* ps = vs + 2 * kTile;      // 128 rows x 128 keys bf16 (two halves)
  int* ids = reinterpret_cast<int*>(ps + 2 * kHalfBytes);
  __shared__ uint64_t qbar, kfull[2], vfull[2], sbar, obar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t == 0) {
    mbar_init(&qbar, 1);
    mbar_init(&kfull[0], 1);
    mbar_init(&kfull[1], 1);
    mbar_init(&vfull[0], 1);
    mbar_init(&vfull[1], 1);
    mbar_init(&sbar, 1);
    mbar_init(&obar, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    abort_flag = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  for (int i = t; i < nid; i += blockDim.x) {
    int b = __ldg(a.prefix_block_ids + id0 + i);
    if (b < 0 || (int64_t)b >= a.num_blocks) {
      atomicOr(a.err, PKV_DEVERR_BLOCK);
      b = (int)a.num_blocks;  // an out-of-range box reads zeros
    }
    ids[i] = b;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tO = tmem + 256;

  // ---- loads and MMA issue (thread 0 only)
  auto load_kv = [&](const CUtensorMap* map, unsigned char* dst, uint64_t* bar, int jt) {
    mbar_arrive_expect_tx(bar, kTile);
    for (int b = 0; b < kPrefixKeys / PB; ++b) {
      const int key = key0 + jt * kPrefixKeys + b * PB;
      int blk = (int)a.num_blocks, row = 0;
      if (key < a.prefix_len) {
        blk = ids[key / P - id0];
        row = key % P;
      }
#pragma unroll
      for (int h = 0; h < H; ++h)
        tma_load_4d(dst + h * kHalfBytes + b * PB * 128, map, h * 64, kvh, row, blk, bar);
    }
  };
  auto issue_qk = [&](int jt) -> bool {
    if (!mbar_wait(&kfull[jt & 1], (jt >> 1) & 1)) return false;
    const uint32_t kb = smem_u32(ks + (jt & 1) * kTile), qb = smem_u32(qs);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
      tc::mma_bf16(tmem + (jt & 1) * 128, tc::smem_desc_sw128(qb + off, 16, 1024),
                   tc::smem_desc_sw128(kb + off, 16, 1024), kIdQK, k > 0 ? 1u : 0u);
    }
    tc::commit(&sbar);
    return true;
  };
  auto issue_pv = [&](int jt) -> bool {
    if (!mbar_wait(&vfull[jt & 1], (jt >> 1) & 1)) return false;
    const uint32_t vb = smem_u32(vs + (jt & 1) * kTile), pb = smem_u32(ps);
#pragma unroll
    for (int k = 0; k < kPrefixKeys / 16; ++k) {
      const uint64_t ad = tc::smem_desc_sw128(pb + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
      // V is MN-major: 64-column d chunks kHalfBytes apart, 8-key groups 1 KiB apart
      const uint64_t bd = tc::smem_desc_sw128(vb + k * 2048, kHalfBytes, 1024);
      tc::mma_bf16(tO, ad, bd, kIdPV, (jt > 0 || k > 0) ? 1u : 0u);
    }
    tc::commit(&obar);
    return true;
  };

  if (t == 0) {
    mbar_arrive_expect_tx(&qbar, kTile);
#pragma unroll
    for (int h = 0; h < H; ++h) tma_load_3d(qs + h * kHalfBytes, &tmq, h * 64, kvh * G, mt * RPB, &qbar);
    load_kv(&tmk, ks, &kfull[0], 0);
    load_kv(&tmv, vs, &vfull[0], 0);
    if (J > 1) {
      load_kv(&tmk, ks + kTile, &kfull[1], 1);
      load_kv(&tmv, vs + kTile, &vfull[1], 1);
    }
    if (!mbar_wait(&qbar, 0) || !issue_qk(0)) {
      atomicOr(a.err, PKV_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  }
  __syncthreads();

  const float c = a.qscale;
  float m_run = -INFINITY, l_run = 0.f;
  bool alive = abort_flag == 0;
  for (int j = 0; j < J && alive; ++j) {
    bool ok = mbar_wait(&sbar, j & 1);
    tc::fence_after_sync();
    if (t == 0 && ok) {
      if (j + 2 < J) load_kv(&tmk, ks + (j & 1) * kTile, &kfull[j & 1], j + 2);
      if (j + 1 < J && !issue_qk(j + 1)) ok = false;
    }
    // ---- scores of this row: S_j * scale * log2 e, keys past the split masked
    float s[kPrefixKeys];
#pragma unroll
    for (int c0 = 0; c0 < kPrefixKeys; c0 += 32) {
      uint32_t r[32];
      tc::tmem_ld32(tmem + (j & 1) * 128 + lane_base + c0, r);
      tc::wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) s[c0 + i] = __uint_as_float(r[i]) * c;
    }
    const int kvalid = nkeys - j * kPrefixKeys;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPrefixKeys; ++i) {
      if (i >= kvalid) s[i] = -INFINITY;
      mx = fmaxf(mx, s[i]);
    }
    const float m_new = fmaxf(m_run, mx);
    const bool need = m_new > m_run + 8.0f;
    const float alpha = need ? exp2f(m_run - m_new) : 1.f;
    if (j > 0) {
      // PV_{j-1} done: O is current, P and V stage (j+1)&1 are free
      if (!mbar_wait(&obar, (j - 1) & 1)) ok = false;
      tc::fence_after_sync();
      if (t == 0 && ok && j + 1 < J) load_kv(&tmv, vs + ((j + 1) & 1) * kTile, &vfull[(j + 1) & 1], j + 1);
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tc::tmem_ld32(tO + lane_base + c0, r);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tc::tmem_st32(tO + lane_base + c0, r);
        }
        tc::wait_st();
      }
    }
    if (need) m_run = m_new;
    l_run *= alpha;
    // ---- P = exp2(s - m) in bf16, swizzled K-major rows for the PV MMA
    float lsum = 0.f;
#pragma unroll
    for (int ch = 0; ch < kPrefixKeys / 8; ++ch) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p0 = exp2f(s[ch * 8 + 2 * i] - m_run);
        const float p1 = exp2f(s[ch * 8 + 2 * i + 1] - m_run);
        lsum += p0 + p1;
        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
        w[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      const int half = ch >> 3, cc = ch & 7;
      uint4* dst = reinterpret_cast<uint4*>(ps + half * kHalfBytes + t * 128 + ((cc ^ (t & 7)) << 4));
      *dst = make_uint4(w[0], w[1], w[2], w[3]);
    }
    l_run += lsum;
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    alive = __syncthreads_and(ok ? 1 : 0) != 0;
    if (t == 0 && alive) {
      tc::fence_after_sync();
      if (!issue_pv(j)) alive = false;
    }
    if (!alive && t == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    alive = __syncthreads_and(alive ? 1 : 0) != 0;
  }

  // ---- epilogue: O / l and the base-2 LSE of this row
  const bool done = __syncthreads_and((alive && mbar_wait(&obar, (J - 1) & 1)) ? 1 : 0) != 0;
  tc::fence_after_sync();
  const int r = mt * RPB + t / G;
  const int g = t % G;
  const bool row_ok = done && r < a.num_seqs;
  if (!done && t == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  const int64_t slot = ((int64_t)r * a.num_q_heads + (int64_t)kvh * G + g) * a.parts_stride + split;
  if (done) {
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t v[32];
      tc::tmem_ld32(tO + lane_base + c0, v);
      tc::wait_ld();
      if (row_ok) {
        float4* dst = reinterpret_cast<float4*>(a.part_o + slot * D + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                               __uint_as_float(v[4 * i + 2]) * inv,
                               __uint_as_float(v[4 * i + 3]) * inv);
      }
    }
  }
  if (row_ok) a.part_lse[slot] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <int D, int G>
static cudaError_t launch_prefix_t(int num_splits, const CUtensorMap& tmq, const CUtensorMap& tmk,
                                   const CUtensorMap& tmv, const PrefixArgs& a,
                                   cudaStream_t stream) {
  const size_t smem = prefix_smem_bytes(D, a.split_len, a.block_size);
  auto kern = prefix_attention_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int m_tiles = (a.num_seqs * G + kPrefixRows - 1) / kPrefixRows;
  dim3 grid((unsigned)num_splits, (unsigned)m_tiles, (unsigned)a.num_kv_heads);
  kern<<<grid, 128, smem, stream>>>(tmq, tmk, tmv, a);
  return cudaGetLastError();
}

template <int D>
static cudaError_t dispatch_prefix_group(int group, int num_splits, const CUtensorMap& tmq,
                                         const CUtensorMap& tmk, const CUtensorMap& tmv,
                                         const PrefixArgs& a, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_prefix_t<D, 1>(num_splits, tmq, tmk, tmv, a, stream);
    case 2: return launch_prefix_t<D, 2>(num_splits, tmq, tmk, tmv, a, stream);
    case 4: return launch_prefix_t<D, 4>(num_splits, tmq, tmk, tmv, a, stream);
    case 8: return launch_prefix_t<D, 8>(num_splits, tmq, tmk, tmv, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefix_attention(int head_dim, int group, int num_splits,
                                    const CUtensorMap& tmq, const CUtensorMap& tmk,
                                    const CUtensorMap& tmv, const PrefixArgs& a,
                                    cudaStream_t stream) {
  return head_dim == 128
             ? dispatch_prefix_group<128>(group, num_splits, tmq, tmk, tmv, a, stream)
             : dispatch_prefix_group<64>(group, num_splits, tmq, tmk, tmv, a, stream);
}

}  // namespace pkv
