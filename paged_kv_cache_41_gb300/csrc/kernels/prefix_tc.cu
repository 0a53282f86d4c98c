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
//     descriptors expect; K/V boxes are gathered through the prefix's block
//     ids, one box per producer lane so a tile's boxes are in flight
//     together; keys past the prefix read a zero-filled out-of-range box;
//   * warp roles: warps 0-3 softmax (one TMEM lane, i.e. query row, per
//     thread), warp 4 issues the MMAs, warps 5 and 6 gather K and V; stages
//     are handed over by mbarriers and tcgen05.commit, never by a CTA-wide
//     barrier;
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
  const size_t ids = 2 * ((size_t)split_len / block_size + 2) * sizeof(int);
  return tiles + ((ids + 15) & ~(size_t)15) + 1024;  // +1024: base alignment
}

template <int D, int G>
__global__ void __launch_bounds__(224, 1)
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
  const int key0 = split * a.split_len;
  const int nkeys = min(a.split_len, a.prefix_len - key0);
  if (nkeys <= 0) return;
  const int J = (nkeys + kPrefixKeys - 1) / kPrefixKeys;
  const int id0 = key0 / P;
  const int nid = (key0 + nkeys - 1) / P - id0 + 1;

  extern __shared__ unsigned char smem_raw[];
  // Align by offsetting the array itself (not through an integer), so the
  // compiler keeps every access in the shared state space.
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* qs = sm;
  unsigned char* ks = qs + kTile;          // two stages
  unsigned char* vs = ks + 2 * kTile;      // two stages
  unsigned char* ps = vs + 2 * kTile;      // 128 rows x 128 keys bf16 (two halves)
  const int nid_cap = a.split_len / P + 2;  // block ids of a split, per producer copy
  int* ids_all = reinterpret_cast<int*>(ps + 2 * kHalfBytes);
  // qbar: Q by TMA; kfull/vfull: a producer warp filled a stage; kfree/vfree:
  // the MMA that read a stage completed; sfull[b]: QK^T into S buffer b done;
  // pfull: the four softmax warps wrote P; ofull: PV done.
  __shared__ uint64_t qbar, kfull[2], vfull[2], kfree[2], vfree[2], sfull[2], pfull, ofull;
  __shared__ uint32_t tmem_base;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t == 0) {
    mbar_init(&qbar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&kfree[i], 1);
      mbar_init(&vfree[i], 1);
      mbar_init(&sfull[i], 1);
    }
    mbar_init(&pfull, 4);
    mbar_init(&ofull, 1);
    fence_barrier_init();
    // Q needs no block ids: start it before anything else
    prefetch_tensormap(&tmq);
    mbar_arrive_expect_tx(&qbar, kTile);
#pragma unroll
    for (int h = 0; h < H; ++h)
      tma_load_3d(qs + h * kHalfBytes, &tmq, h * 64, kvh * G, mt * RPB, &qbar);
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t tO = tmem + 256;

  if (warp == 5 || warp == 6) {
    // ============================================================ producers
    // warp 5 streams Q and K, warp 6 streams V.  A tile is kPrefixKeys / PB
    // blocks x H column halves of TMA boxes (PB rows x 128 B each, 128-byte
    // swizzle); each lane issues its own boxes, so the boxes of a tile are
    // requested in parallel.  A stage is refilled as soon as the MMA that read
    // it has completed; keys past the split read a zero-filled out-of-range
    // box.
    const bool is_k = warp == 5;
    int* ids = ids_all + (is_k ? 0 : nid_cap);  // each producer gathers its own copy
    for (int i = lane; i < nid; i += 32) {
      int b = __ldg(a.prefix_block_ids + id0 + i);
      if (b < 0 || (int64_t)b >= a.num_blocks) {
        if (is_k) atomicOr(a.err, PKV_DEVERR_BLOCK);
        b = -1;  // rows of a bad block are zero-filled
      }
      ids[i] = b;
    }
    __syncwarp();
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    unsigned char* base = is_k ? ks : vs;
    uint64_t* fullb = is_k ? kfull : vfull;
    uint64_t* freeb = is_k ? kfree : vfree;
    const int PB = P < kPrefixKeys ? P : kPrefixKeys;
    const int nbox = (kPrefixKeys / PB) * H;
    if (lane == 0) prefetch_tensormap(map);
    for (int jt = 0; jt < J; ++jt) {
      const int st = jt & 1;
      int ok = 1;
      if (lane == 0 && jt >= 2 && !mbar_wait(&freeb[st], ((jt - 2) >> 1) & 1)) {
        atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        ok = 0;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) mbar_arrive_expect_tx(&fullb[st], kTile);
      __syncwarp();
      for (int bi = lane; bi < nbox; bi += 32) {
        const int b = bi / H, h = bi % H;
        const int key = key0 + jt * kPrefixKeys + b * PB;
        int blk = (int)a.num_blocks, row = 0;  // out of range: zero fill
        if (key < key0 + nkeys && ids[key / P - id0] >= 0) {
          blk = ids[key / P - id0];
          row = key % P;
        }
        tma_load_4d(base + st * kTile + h * kHalfBytes + b * PB * 128, map, h * 64, kvh, row,
                    blk, &fullb[st]);
      }
    }
  } else if (warp == 4) {
    // ============================================================ MMA issue
    if (lane == 0) {
      auto issue_qk = [&](int jt) -> bool {
        if (!mbar_wait(&kfull[jt & 1], (jt >> 1) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t kb = smem_u32(ks + (jt & 1) * kTile), qb = smem_u32(qs);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
          tc::mma_bf16(tmem + (jt & 1) * 128, tc::smem_desc_sw128(qb + off, 16, 1024),
                       tc::smem_desc_sw128(kb + off, 16, 1024), kIdQK, k > 0 ? 1u : 0u);
        }
        tc::commit(&sfull[jt & 1]);
        tc::commit(&kfree[jt & 1]);
        return true;
      };
      auto issue_pv = [&](int jt) -> bool {
        if (!mbar_wait(&vfull[jt & 1], (jt >> 1) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t vb = smem_u32(vs + (jt & 1) * kTile), pb = smem_u32(ps);
#pragma unroll
        for (int k = 0; k < kPrefixKeys / 16; ++k) {
          const uint64_t ad =
              tc::smem_desc_sw128(pb + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
          // V is MN-major: 64-column d chunks kHalfBytes apart, 8-key groups 1 KiB apart
          const uint64_t bd = tc::smem_desc_sw128(vb + k * 2048, kHalfBytes, 1024);
          tc::mma_bf16(tO, ad, bd, kIdPV, (jt > 0 || k > 0) ? 1u : 0u);
        }
        tc::commit(&ofull);
        tc::commit(&vfree[jt & 1]);
        return true;
      };
      bool ok = mbar_wait(&qbar, 0) && issue_qk(0) && (J < 2 || issue_qk(1));
      for (int j = 0; j < J && ok; ++j) {
        // softmax j has read S_j and written P_j
        if (!mbar_wait(&pfull, j & 1)) { ok = false; break; }
        tc::fence_after_sync();
        if (!issue_pv(j)) { ok = false; break; }
        if (j + 2 < J && !issue_qk(j + 2)) { ok = false; break; }
      }
      if (!ok) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    }
  } else {
    // ============================================================ softmax rows
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float c = a.qscale;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < J && ok; ++j) {
      if (!mbar_wait(&sfull[j & 1], (j >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t r[kPrefixKeys];
#pragma unroll
      for (int c0 = 0; c0 < kPrefixKeys; c0 += 32)
        tc::tmem_ld32(tmem + (j & 1) * 128 + lane_base + c0,
                      *reinterpret_cast<uint32_t(*)[32]>(r + c0));
      tc::wait_ld();
      const int kvalid = nkeys - j * kPrefixKeys;
      float s[kPrefixKeys];
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kPrefixKeys; ++i) {
        s[i] = i < kvalid ? __uint_as_float(r[i]) * c : -INFINITY;
        mx = fmaxf(mx, s[i]);
      }
      const float m_new = fmaxf(m_run, mx);
      const bool need = m_new > m_run + 8.0f;
      const float alpha = need ? exp2f(m_run - m_new) : 1.f;
      if (j > 0) {
        // PV_{j-1} has completed: O is current and the P buffer is free
        if (!mbar_wait(&ofull, (j - 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc::tmem_ld32(tO + lane_base + c0, o);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc::tmem_st32(tO + lane_base + c0, o);
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
        const int hf = ch >> 3, cc = ch & 7;
        uint4* dst =
            reinterpret_cast<uint4*>(ps + hf * kHalfBytes + t * 128 + ((cc ^ (t & 7)) << 4));
        *dst = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run += lsum;
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull);
    }
    // ---- epilogue: O / l and the LSE of this row
    const bool done = ok && mbar_wait(&ofull, (J - 1) & 1);
    tc::fence_after_sync();
    if (!done && lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    const int r = mt * RPB + t / G;
    const int g = t % G;
    const bool row_ok = done && r < a.num_seqs;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const int64_t slot =
        ((int64_t)r * a.num_q_heads + (int64_t)kvh * G + g) * a.parts_stride + split;
    if (__all_sync(0xffffffffu, done)) {
      // O row -> registers (one wait), scaled; then through the free K stages
      // (128 rows x D floats, 16-byte chunk i of row t at chunk i ^ (t % 32))
      // so each warp stores whole 4*D-byte rows, one per instruction.
      uint32_t v[D];
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32)
        tc::tmem_ld32(tO + lane_base + c0, *reinterpret_cast<uint32_t(*)[32]>(v + c0));
      tc::wait_ld();
      float4* stage = reinterpret_cast<float4*>(ks);  // K stages are idle: every QK^T completed
      constexpr int kChunks = D / 4;
#pragma unroll
      for (int i = 0; i < kChunks; ++i)
        stage[t * kChunks + (i ^ (t & (kChunks - 1)))] =
            make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                        __uint_as_float(v[4 * i + 2]) * inv, __uint_as_float(v[4 * i + 3]) * inv);
      __syncwarp();
      for (int rr = 0; rr < 32; ++rr) {
        const int row = warp * 32 + rr;
        const int r2 = mt * RPB + row / G;
        if (r2 < a.num_seqs) {
          const int64_t slot2 =
              ((int64_t)r2 * a.num_q_heads + (int64_t)kvh * G + row % G) * a.parts_stride + split;
          for (int i = lane; i < kChunks; i += 32)
            reinterpret_cast<float4*>(a.part_o + slot2 * D)[i] =
                stage[row * kChunks + (i ^ (row & (kChunks - 1)))];
        }
      }
    }
    if (row_ok) a.part_lse[slot] = l_run > 0.f ? (m_run + log2f(l_run)) * a.lse_scale : -INFINITY;
  }
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
  static SmemAttrCache attr_cache;
  cudaError_t e = ensure_smem_limit(kern, (int)smem, attr_cache);
  if (e != cudaSuccess) return e;
  const int m_tiles = (a.num_seqs * G + kPrefixRows - 1) / kPrefixRows;
  dim3 grid((unsigned)num_splits, (unsigned)m_tiles, (unsigned)a.num_kv_heads);
  kern<<<grid, 224, smem, stream>>>(tmq, tmk, tmv, a);
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
