// decode.cu -- split-K paged attention decode on CUDA cores (GQA groups <= 8).
//
// What it computes ("M5.3 - KV Memory Layout and Exact Reuse", 0x0A and
// 0x0BA): for sequence r and query head h, attention of q[r, h] over the
// request-visible rows t < T_r of kv head h / G, where row t lives in physical
// block block_tables[r, t / P] at offset t % P.  A sequence's blocks are cut
// into partitions of `blocks_per_part` blocks; each partition keeps an online
// softmax state (m, l, u) and emits (O_p = u / l, LSE_p = m + log l); a second
// kernel merges the partitions of a row by log-sum-exp, never by averaging
// normalised outputs, with empty partitions as the identity.
//
// Design (GB300):
//   * one CTA per (kv head, partition, sequence); the G query heads of a kv
//     head share every K/V byte the CTA reads;
//   * warp 4 is the producer: it walks the block table and issues one 4-D TMA
//     box (a tile of up to 64 token rows x head_dim of one kv head) for K and
//     one for V into an mbarrier-tracked ring of shared-memory stages;
//   * warps 0-3 consume 16-token chunks: each half-warp owns two token rows,
//     each lane 1/16 of head_dim; q . k partial sums of the 2G (row, head)
//     pairs are folded across the 16 lanes by a transpose-reduction (each
//     shuffle level halves the values a lane carries), the softmax update runs
//     once per (row, head), and P.V accumulates per lane in fp32;
//   * the exponent base is only moved when the running max grows by more than
//     2^8 (exact: output and denominator keep the same base), so the
//     accumulator rescale is rare;
//   * scores are in base 2 (q is pre-multiplied by scale * log2 e);
//   * rows past the request's tail are never multiplied in, so stale or NaN
//     bytes in a recycled block cannot leak (M5.3 0x03G).
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kChunk = 16;             // token rows per softmax update
constexpr int kMaxTileRows = 64;       // token rows per TMA box
constexpr float kRescaleLog2 = 8.0f;   // move the exponent base past 2^8 growth
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int tile_rows_for(int block_size) {
  return block_size < kMaxTileRows ? block_size : kMaxTileRows;
}

// Fold N per-lane values across the 16 lanes of a half-warp (xor offsets
// O, O/2, ..., 1).  While a lane carries more than one value, each level
// sends half of them to its partner and keeps the other half; afterwards the
// lane holds the full 16-lane sum of one of the N values (see held_index).
template <int N, int O>
struct TransposeReduce {
  __device__ __forceinline__ static void run(float* v, int l16) {
    if constexpr (N > 1) {
      constexpr int H = N / 2;
      const bool upper = (l16 & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = upper ? v[i] : v[i + H];
        const float keep = upper ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      if constexpr (O > 1) TransposeReduce<H, O / 2>::run(v, l16);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      if constexpr (O > 1) TransposeReduce<1, O / 2>::run(v, l16);
    }
  }
};

template <int N>
__device__ __forceinline__ int held_index(int l16) {
  int idx = 0, n = N;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    if (n > 1) {
      n >>= 1;
      if (l16 & o) idx += n;
    }
  }
  return idx;
}

template <int N>
__host__ __device__ constexpr int log2_int() {
  return N <= 1 ? 0 : 1 + log2_int<N / 2>();
}

struct DecodeSmem {
  int tile_elems;   // rows * head_dim
  int stages;
  size_t tiles_bytes, bar_off, ok_off, scratch_off, total;
};

__host__ __device__ inline DecodeSmem decode_smem_layout(int block_size, int head_dim,
                                                         int elem_bytes, int group, int stages) {
  DecodeSmem s;
  s.tile_elems = tile_rows_for(block_size) * head_dim;
  s.stages = stages;
  size_t tiles = (size_t)2 * stages * s.tile_elems * elem_bytes;
  const size_t merge = (size_t)(kConsumerWarps * group * head_dim + 2 * kConsumerWarps * group) * 4;
  if (merge > tiles) tiles = merge;
  s.tiles_bytes = (tiles + 127) & ~(size_t)127;
  s.bar_off = s.tiles_bytes;
  s.ok_off = s.bar_off + (size_t)2 * stages * 8;
  s.scratch_off = (s.ok_off + (size_t)stages * 4 + 15) & ~(size_t)15;
  s.total = s.scratch_off + (size_t)kConsumerWarps * 5 * group * 4 + 128;  // +128: base alignment
  return s;
}

int decode_num_stages(int block_size, int head_dim, int elem_bytes) {
  const int stage_bytes = 2 * tile_rows_for(block_size) * head_dim * elem_bytes;
  int ns = (64 * 1024) / stage_bytes;
  if (ns < 2) ns = 2;
  if (ns > 8) ns = 8;
  return ns;
}

size_t decode_smem_bytes(int block_size, int head_dim, int elem_bytes, int group, int stages) {
  return decode_smem_layout(block_size, head_dim, elem_bytes, group, stages).total;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads, (G >= 8 ? 2 : 3))
    decode_partial_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  constexpr int EPL = D / 16;  // head_dim elements per lane
  constexpr int NV = 2 * G;    // (row, head) partial sums per lane per chunk
  constexpr int LEVELS = log2_int<NV>();
  static_assert(NV <= 16 && (NV & (NV - 1)) == 0, "group must be 1, 2, 4 or 8");

  const int kvh = blockIdx.x, part = blockIdx.y, r = blockIdx.z;
  const int P = a.block_size;
  const int TR = tile_rows_for(P);
  const bool reporter = kvh == 0 && part == 0 && threadIdx.x == 0;
  const int T_r = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, reporter);
  const int nblk = (T_r + P - 1) / P;
  const int b0 = part * a.blocks_per_part;
  if (b0 >= nblk) {  // empty partition: the whole CTA leaves before any barrier
    if (a.direct && part == 0) {  // an empty sequence still gets out = 0, lse = -inf
      const int64_t rh0 = (int64_t)r * a.num_q_heads + (int64_t)kvh * G;
      for (int j = threadIdx.x; j < G * D; j += blockDim.x) {
        store_out(static_cast<T*>(a.out) + rh0 * D + j, 0.f);
        if (j % D == 0 && a.lse_out) a.lse_out[rh0 + j / D] = -INFINITY;
      }
    }
    return;
  }
  const int tok0 = b0 * P;
  const int tok_end = min(T_r, (b0 + a.blocks_per_part) * P);
  const int ntiles = (tok_end - tok0 + TR - 1) / TR;
  const int tiles_per_block = P / TR;

  const DecodeSmem L = decode_smem_layout(P, D, (int)sizeof(T), G, a.num_stages);
  const int NS = a.num_stages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  T* ktile = reinterpret_cast<T*>(smem);
  T* vtile = ktile + (size_t)NS * L.tile_elems;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + NS;
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + L.ok_off);
  float* scratch = reinterpret_cast<float*>(smem + L.scratch_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      const int32_t* tbl = a.block_tables + (int64_t)r * a.max_blocks + b0;
      const uint32_t tx = 2u * (uint32_t)(L.tile_elems * sizeof(T));
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % NS;
        if (i >= NS && !mbar_wait(&empty[s], ((i / NS) - 1) & 1)) {
          atomicOr(a.err, PKV_DEVERR_TIMEOUT);
          break;
        }
        const int jb = i / tiles_per_block;             // block within the partition
        const int row = (i % tiles_per_block) * TR;     // first row of the tile in the block
        const int blk = __ldg(tbl + jb);
        if (blk < 0 || (int64_t)blk >= a.num_blocks) {
          atomicOr(a.err, PKV_DEVERR_BLOCK);
          stage_ok[s] = 0;
          mbar_arrive(&full[s]);
        } else {
          stage_ok[s] = 1;
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_4d(ktile + (size_t)s * L.tile_elems, &tmk, 0, kvh, row, blk, &full[s]);
          tma_load_4d(vtile + (size_t)s * L.tile_elems, &tmv, 0, kvh, row, blk, &full[s]);
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int hw = lane >> 4, l16 = lane & 15;
  float qr[G][EPL];
  {
    const T* qp = static_cast<const T*>(a.q) +
                  ((int64_t)r * a.num_q_heads + (int64_t)kvh * G) * D + l16 * EPL;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      VecLoad<T, EPL>::run(qp + g * D, qr[g]);
#pragma unroll
      for (int e = 0; e < EPL; ++e) qr[g][e] *= a.qscale;
    }
  }
  float acc[G][EPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;

  // softmax bookkeeping: lane handles (row stok, head sg) of the warp's 4 x G
  // scores; the state (m_used, l_run) is that of head sg.
  float* sw = scratch + warp * 5 * G;  // [4][G] scores / probabilities, then [G] alpha
  const int sidx = lane & (4 * G - 1);
  const int stok = sidx / G, sg = sidx % G;
  const int ridx = held_index<NV>(l16);
  const int rtk = ridx / G, rg = ridx % G;
  const bool rep = (l16 & ((1 << (4 - LEVELS)) - 1)) == 0;
  float m_used = -INFINITY, l_run = 0.f;

  for (int i = 0; i < ntiles; ++i) {
    const int s = i % NS;
    if (!mbar_wait(&full[s], (i / NS) & 1)) {
      if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
      break;
    }
    const int nvalid = min(TR, tok_end - (tok0 + i * TR));
    if (stage_ok[s]) {
      const T* kt = ktile + (size_t)s * L.tile_elems;
      const T* vt = vtile + (size_t)s * L.tile_elems;
      for (int c = 0; c * kChunk < nvalid; ++c) {
        const int row0 = c * kChunk + warp * 4 + hw * 2;
        // ---- q . k for rows row0, row0 + 1 and the G heads
        float v[NV];
#pragma unroll
        for (int tk = 0; tk < 2; ++tk) {
          float kf[EPL];
          VecLoad<T, EPL>::run(kt + (row0 + tk) * D + l16 * EPL, kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float d0 = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) d0 = fmaf(qr[g][e], kf[e], d0);
            v[tk * G + g] = d0;
          }
        }
        TransposeReduce<NV, 8>::run(v, l16);
        if (rep) sw[(hw * 2 + rtk) * G + rg] = (row0 + rtk < nvalid) ? v[0] : -INFINITY;
        __syncwarp();
        // ---- online softmax over the warp's 4 rows, one lane per (row, head)
        const float sc = sw[stok * G + sg];
        float cmax = sc;
#pragma unroll
        for (int o = G; o < 4 * G; o <<= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
        const float m_new = fmaxf(m_used, cmax);
        const bool need = m_new > m_used + kRescaleLog2;
        const bool any = __any_sync(0xffffffffu, need);
        float alpha = 1.f;
        if (need) {
          alpha = exp2f(m_used - m_new);
          m_used = m_new;
          l_run *= alpha;
        }
        const float p = (sc == -INFINITY) ? 0.f : exp2f(sc - m_used);
        float psum = p;
#pragma unroll
        for (int o = G; o < 4 * G; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
        l_run += psum;
        __syncwarp();
        if (lane < 4 * G) sw[stok * G + sg] = p;
        if (any && lane < G) sw[4 * G + lane] = alpha;
        __syncwarp();
        if (any) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float al = sw[4 * G + g];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[g][e] *= al;
          }
        }
        // ---- P . V for this half-warp's two rows
#pragma unroll
        for (int tk = 0; tk < 2; ++tk) {
          const int row = row0 + tk;
          if (row < nvalid) {
            float pg[G];
#pragma unroll
            for (int g = 0; g < G; ++g) pg[g] = sw[(hw * 2 + tk) * G + g];
            float vf[EPL];
            VecLoad<T, EPL>::run(vt + row * D + l16 * EPL, vf);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(pg[g], vf[e], acc[g][e]);
          }
        }
        __syncwarp();
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ------------------------------------------------------------------ merge the 4 warps
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], 16);

  named_barrier_sync(1, kConsumerWarps * 32);  // every stage consumed: reuse the tiles
  float* macc = reinterpret_cast<float*>(smem);            // [4][G][D]
  float* mm = macc + kConsumerWarps * G * D;               // [4][G]
  float* ml = mm + kConsumerWarps * G;                     // [4][G]
  if (hw == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < EPL; ++e) macc[(warp * G + g) * D + l16 * EPL + e] = acc[g][e];
  }
  if (lane < G) {
    mm[warp * G + lane] = m_used;
    ml[warp * G + lane] = l_run;
  }
  named_barrier_sync(1, kConsumerWarps * 32);

  for (int j = threadIdx.x; j < G * D; j += kConsumerWarps * 32) {
    const int g = j / D, e = j % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * G + g]);
    float Lsum = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float wt = exp2f(mm[w * G + g] - M);
        Lsum = fmaf(wt, ml[w * G + g], Lsum);
        o = fmaf(wt, macc[(w * G + g) * D + e], o);
      }
    }
    const bool nonempty = Lsum > 0.f;
    o = nonempty ? o / Lsum : 0.f;
    const float lse2 = nonempty ? M + log2f(Lsum) : -INFINITY;
    const int64_t rh = (int64_t)r * a.num_q_heads + (int64_t)kvh * G + g;
    if (a.direct) {
      store_out(static_cast<T*>(a.out) + rh * D + e, o);
      if (e == 0 && a.lse_out) a.lse_out[rh] = lse2 * kLn2;
    } else {
      const int64_t slot = rh * a.parts_stride + a.part_offset + part;
      a.part_o[slot * D + e] = o;
      if (e == 0) a.part_lse[slot] = lse2;
    }
  }
}

// One warp per (sequence, query head): merge its partitions by log-sum-exp.
template <typename T, int D>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeArgs a) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rh = (int64_t)blockIdx.x * 4 + warp;
  if (rh >= (int64_t)a.num_seqs * a.num_q_heads) return;
  const int r = (int)(rh / a.num_q_heads);
  const int P = a.block_size;
  const int T_r = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
  const int nblk = (T_r + P - 1) / P;
  const int nparts = a.part_offset + (nblk + a.blocks_per_part - 1) / a.blocks_per_part;
  const float* plse = a.part_lse + rh * a.parts_stride;
  const float* po = a.part_o + rh * a.parts_stride * D;
  float M = -INFINITY;
  for (int p = lane; p < nparts; p += 32) M = fmaxf(M, plse[p]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float Lsum = 0.f;
  if (M != -INFINITY) {
    for (int p = 0; p < nparts; ++p) {
      const float w = exp2f(plse[p] - M);
      Lsum += w;
      float x[EPL];
      VecLoad<float, EPL>::run(po + (int64_t)p * D + lane * EPL, x);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, x[e], acc[e]);
    }
  }
  const bool nonempty = Lsum > 0.f;
  T* out = static_cast<T*>(a.out) + rh * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) store_out(out + e, nonempty ? acc[e] / Lsum : 0.f);
  if (lane == 0 && a.lse_out) a.lse_out[rh] = nonempty ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
}

template <typename T, int D, int G>
static cudaError_t launch_partial(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                  const DecodeArgs& a, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes(a.block_size, D, (int)sizeof(T), G, a.num_stages);
  auto kern = decode_partial_kernel<T, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.num_kv_heads, (unsigned)a.max_parts, (unsigned)a.num_seqs);
  kern<<<grid, kDecodeThreads, smem, stream>>>(tmk, tmv, a);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_reduce_t(const DecodeArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.num_seqs * a.num_q_heads;
  decode_reduce_kernel<T, D><<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_reduce(int dtype, int head_dim, const DecodeArgs& a,
                                 cudaStream_t stream) {
  if (dtype == PKV_BF16)
    return head_dim == 128 ? launch_reduce_t<__nv_bfloat16, 128>(a, stream)
                           : launch_reduce_t<__nv_bfloat16, 64>(a, stream);
  return head_dim == 128 ? launch_reduce_t<float, 128>(a, stream)
                         : launch_reduce_t<float, 64>(a, stream);
}

template <typename T, int D>
static cudaError_t dispatch_group(int group, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                  const DecodeArgs& a, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_partial<T, D, 1>(tmk, tmv, a, stream);
    case 2: return launch_partial<T, D, 2>(tmk, tmv, a, stream);
    case 4: return launch_partial<T, D, 4>(tmk, tmv, a, stream);
    case 8: return launch_partial<T, D, 8>(tmk, tmv, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_paged_decode(int dtype, int head_dim, int group, const CUtensorMap& tmk,
                                const CUtensorMap& tmv, const DecodeArgs& a,
                                cudaStream_t stream) {
  cudaError_t e;
  if (dtype == PKV_BF16)
    e = head_dim == 128 ? dispatch_group<__nv_bfloat16, 128>(group, tmk, tmv, a, stream)
                        : dispatch_group<__nv_bfloat16, 64>(group, tmk, tmv, a, stream);
  else
    e = head_dim == 128 ? dispatch_group<float, 128>(group, tmk, tmv, a, stream)
                        : dispatch_group<float, 64>(group, tmk, tmv, a, stream);
  if (e != cudaSuccess || a.direct) return e;
  return launch_decode_reduce(dtype, head_dim, a, stream);
}

}  // namespace pkv
