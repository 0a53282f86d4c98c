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
//   * one CTA of four warps per (kv head, partition, sequence); the G query
//     heads of a kv head share every K/V byte the CTA reads; four CTAs fit on
//     an SM (registers and a 3 x 16 KiB shared-memory ring each);
//   * warp 0 also issues the loads: it holds the partition's block ids 32 at a
//     time (one coalesced load per 32 blocks, the next group in flight) and
//     fills each 32-row stage with 4-D TMA boxes (one block, or a 32-row slice
//     of a larger block, of one kv head) for K and V, tracked by mbarriers;
//     a stage is refilled as soon as all four warps have released it, so no
//     table lookup sits between two copies;
//   * warps consume 16-row chunks: each half-warp owns two token rows, each
//     lane 1/16 of head_dim; the 2G (row, head) partial dot products are
//     summed across the 16 lanes through a small per-warp shared scratch;
//     the row lands in lane bit 3, so the softmax max and sum over the warp's
//     four rows are two shuffles each; q . k and P . V use packed fp32x2 FMAs;
//   * full stages take a straight-line path with no row masking; only a
//     partition's last stage masks rows;
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
constexpr int kDecodeThreads = kConsumerWarps * 32;
constexpr int kChunk = 16;             // token rows per softmax update
constexpr float kRescaleLog2 = 8.0f;   // move the exponent base past 2^8 growth
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeSmem {
  int tile_elems;   // rows * head_dim
  int stages;
  size_t tiles_bytes, bar_off, ok_off, scratch_off, total;
};

__host__ __device__ inline DecodeSmem decode_smem_layout(int block_size, int head_dim,
                                                         int elem_bytes, int group, int stages) {
  DecodeSmem s;
  s.tile_elems = kStageRows * head_dim;
  s.stages = stages;
  size_t tiles = (size_t)2 * stages * s.tile_elems * elem_bytes;
  const size_t merge = (size_t)(kConsumerWarps * group * head_dim + 2 * kConsumerWarps * group) * 4;
  if (merge > tiles) tiles = merge;
  s.tiles_bytes = (tiles + 127) & ~(size_t)127;
  s.bar_off = s.tiles_bytes;
  s.ok_off = s.bar_off + (size_t)2 * stages * 8;
  s.scratch_off = (s.ok_off + (size_t)stages * 4 + 15) & ~(size_t)15;
  s.total = s.scratch_off + (size_t)kConsumerWarps * 2 * (2 * group * 16) * 4 + 128;  // +128: base alignment
  return s;
}

int decode_num_stages(int block_size, int head_dim, int elem_bytes) {
  (void)block_size;
  const int stage_bytes = 2 * kStageRows * head_dim * elem_bytes;
  int ns = (49 * 1024) / stage_bytes;  // 3 stages of 16 KiB: 4 CTAs per SM
  if (ns < 2) ns = 2;
  if (ns > 8) ns = 8;
  return ns;
}

size_t decode_smem_bytes(int block_size, int head_dim, int elem_bytes, int group, int stages) {
  return decode_smem_layout(block_size, head_dim, elem_bytes, group, stages).total;
}

// One 16-row chunk of a stage for one consumer warp: rows row0 and row0 + 1
// of this half-warp.  kTail = false is the full-stage fast path (every row
// valid, no masking); kTail = true masks rows >= nvalid.
//
// Cross-lane sums go through `red`, this half-warp's [2G][16] scratch: lane
// l16 stores its partial dot product of value i = (row tk, head g) = tk*G + g
// at red[i][l16]; then each value is summed by 8/G lanes that read 2G
// consecutive partials each and combine with 8/G - 1 shuffles.  Lane l16 ends
// up holding value j = l16 / (8/G): row tk = l16 >> 3, head g = j % G.
template <typename T, int D, int G, bool kTail>
__device__ __forceinline__ void decode_chunk(const T* __restrict__ kt, const T* __restrict__ vt,
                                             int row0, int nvalid,
                                             const float2 (&q2)[G][D / 32],
                                             float2 (&acc)[G][D / 32], float& m_used,
                                             float& l_run, float* __restrict__ red, int l16) {
  constexpr int EPL = D / 16;
  constexpr int EP2 = EPL / 2;
  constexpr int NV = 2 * G;    // values per half-warp and chunk
  constexpr int LPV = 16 / NV; // lanes summing one value
  // ---- q . k partial sums for rows row0, row0 + 1 and the G heads
  float v[NV];
#pragma unroll
  for (int tk = 0; tk < 2; ++tk) {
    float kf[EPL];
    VecLoad<T, EPL>::run(kt + (row0 + tk) * D + l16 * EPL, kf);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float2 d2 = __fmul2_rn(q2[g][0], make_float2(kf[0], kf[1]));
#pragma unroll
      for (int j = 1; j < EP2; ++j) d2 = __ffma2_rn(q2[g][j], make_float2(kf[2 * j], kf[2 * j + 1]), d2);
      v[tk * G + g] = d2.x + d2.y;
    }
  }
  // ---- sum each value over the 16 lanes of the half-warp
#pragma unroll
  for (int i = 0; i < NV; ++i) red[i * 16 + l16] = v[i];
  __syncwarp();
  const int j = l16 / LPV, sub = l16 % LPV;
  float part[NV];
  VecLoad<float, NV>::run(red + j * 16 + sub * NV, part);
  __syncwarp();  // the next chunk rewrites red
  float s2 = part[0];
#pragma unroll
  for (int k = 1; k < NV; ++k) s2 += part[k];
#pragma unroll
  for (int o = LPV / 2; o >= 1; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  // ---- online softmax over the warp's 4 rows (rows differ in lane bits 3, 4)
  const float sc = (!kTail || row0 + (l16 >> 3) < nvalid) ? s2 : -INFINITY;
  float cmax = fmaxf(sc, __shfl_xor_sync(0xffffffffu, sc, 8));
  cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 16));
  const float m_new = fmaxf(m_used, cmax);
  const bool need = m_new > m_used + kRescaleLog2;
  const bool any = __any_sync(0xffffffffu, need);
  const float alpha = need ? exp2f(m_used - m_new) : 1.f;
  m_used = need ? m_new : m_used;
  l_run *= alpha;
  const float p = (kTail && sc == -INFINITY) ? 0.f : exp2f(sc - m_used);
  float psum = p + __shfl_xor_sync(0xffffffffu, p, 8);
  psum += __shfl_xor_sync(0xffffffffu, psum, 16);
  l_run += psum;
  if (any) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float al = __shfl_sync(0xffffffffu, alpha, g * LPV, 16);
      const float2 al2 = make_float2(al, al);
#pragma unroll
      for (int e = 0; e < EP2; ++e) acc[g][e] = __fmul2_rn(acc[g][e], al2);
    }
  }
  // ---- P . V for this half-warp's two rows
  float pg[2][G];
#pragma unroll
  for (int tk = 0; tk < 2; ++tk)
#pragma unroll
    for (int g = 0; g < G; ++g) pg[tk][g] = __shfl_sync(0xffffffffu, p, (tk * G + g) * LPV, 16);
#pragma unroll
  for (int tk = 0; tk < 2; ++tk) {
    if (!kTail || row0 + tk < nvalid) {
      float vf[EPL];
      VecLoad<T, EPL>::run(vt + (row0 + tk) * D + l16 * EPL, vf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 p2 = make_float2(pg[tk][g], pg[tk][g]);
#pragma unroll
        for (int e = 0; e < EP2; ++e)
          acc[g][e] = __ffma2_rn(p2, make_float2(vf[2 * e], vf[2 * e + 1]), acc[g][e]);
      }
    }
  }
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads, (G >= 8 ? 2 : 4))
    decode_partial_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  constexpr int EPL = D / 16;  // head_dim elements per lane
  constexpr int EP2 = EPL / 2;
  constexpr int NV = 2 * G;    // (row, head) partial sums per lane per chunk
  static_assert(NV <= 16 && (NV & (NV - 1)) == 0, "group must be 1, 2, 4 or 8");

  const int kvh = blockIdx.x, part = blockIdx.y, r = blockIdx.z;
  const int P = a.block_size;
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
  const int ntiles = (tok_end - tok0 + kStageRows - 1) / kStageRows;  // 64-row stages
  const int nbp = (tok_end - tok0 + P - 1) / P;  // blocks of this partition
  const int TB = box_rows_for(P);                // rows per TMA box
  const int nsub = kStageRows / TB;              // boxes per stage

  const DecodeSmem L = decode_smem_layout(P, D, (int)sizeof(T), G, a.num_stages);
  const int NS = a.num_stages;
  extern __shared__ unsigned char smem_raw[];
  // Align by offsetting the array itself (not through an integer), so the
  // compiler keeps every tile and scratch access in the shared state space.
  unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
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

  // ---------------------------------------------------------------- loads
  // Warp 0 issues the TMA boxes.  It holds the partition's block ids 32 at a
  // time (one coalesced load per 32 blocks, the next group in flight) so no
  // table lookup sits between two copies.  A stage is kStageRows token rows:
  // kStageRows / P boxes of one block each when P < kStageRows, else one
  // box of kStageRows rows of a larger block.  Positions advance
  // incrementally (no division).
  const int32_t* tbl = a.block_tables + (int64_t)r * a.max_blocks + b0;
  int cur = 0, nxt = 0, base = 0;
  int jb = 0, brow = 0, rel = 0;  // next box: block in the partition, row in it, row in partition
  const int avail = tok_end - tok0;
  const uint32_t box_bytes = (uint32_t)(TB * D * sizeof(T));
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    cur = lane < nbp ? __ldg(tbl + lane) : -1;
    nxt = 32 + lane < nbp ? __ldg(tbl + 32 + lane) : -1;
  }
  // Fill stage `st` with the next kStageRows rows (warp 0, all lanes).
  auto issue_stage = [&](int st) {
    int blk[kStageRows / 16], brw[kStageRows / 16];
    int nbox = 0;
#pragma unroll
    for (int j = 0; j < kStageRows / 16; ++j) {
      blk[j] = -1;
      brw[j] = 0;
      if (j < nsub && rel < avail) {
        if (jb >= base + 32) {
          cur = nxt;
          base += 32;
          nxt = base + 32 + lane < nbp ? __ldg(tbl + base + 32 + lane) : -1;
        }
        blk[j] = __shfl_sync(0xffffffffu, cur, jb - base);
        brw[j] = brow;
        nbox = j + 1;
        rel += TB;
        brow += TB;
        if (brow == P) {
          brow = 0;
          ++jb;
        }
      }
    }
    bool valid = true;
#pragma unroll
    for (int j = 0; j < kStageRows / 16; ++j)
      if (j < nbox && (blk[j] < 0 || (int64_t)blk[j] >= a.num_blocks)) valid = false;
    if (!valid) {
      if (lane == 0) {
        atomicOr(a.err, PKV_DEVERR_BLOCK);
        stage_ok[st] = 0;
        mbar_arrive(&full[st]);
      }
    } else {
      if (lane == 0) {
        stage_ok[st] = 1;
        mbar_arrive_expect_tx(&full[st], 2u * box_bytes * (uint32_t)nbox);
      }
      __syncwarp();
      // one box per lane: lanes 0..nbox-1 load K, lanes 16..16+nbox-1 load V
      const int j = lane & 15;
      if (j < nbox) {
        int bj = blk[0], rj = brw[0];
#pragma unroll
        for (int jj = 1; jj < kStageRows / 16; ++jj)
          if (j == jj) {
            bj = blk[jj];
            rj = brw[jj];
          }
        if (lane < 16)
          tma_load_4d(ktile + (size_t)st * L.tile_elems + j * TB * D, &tmk, 0, kvh, rj, bj, &full[st]);
        else
          tma_load_4d(vtile + (size_t)st * L.tile_elems + j * TB * D, &tmv, 0, kvh, rj, bj, &full[st]);
      }
    }
  };
  if (warp == 0) {
    for (int st = 0; st < NS && st < ntiles; ++st) issue_stage(st);
  }

  // ------------------------------------------------------------------ consumers
  const int hw = lane >> 4, l16 = lane & 15;
  float2 q2[G][EP2];
  {
    const T* qp = static_cast<const T*>(a.q) +
                  ((int64_t)r * a.num_q_heads + (int64_t)kvh * G) * D + l16 * EPL;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float f[EPL];
      VecLoad<T, EPL>::run(qp + g * D, f);
#pragma unroll
      for (int j = 0; j < EP2; ++j) q2[g][j] = make_float2(f[2 * j] * a.qscale, f[2 * j + 1] * a.qscale);
    }
  }
  float2 acc[G][EP2];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int j = 0; j < EP2; ++j) acc[g][j] = make_float2(0.f, 0.f);

  // (m_used, l_run): softmax state of head (l16 / (8 / G)) % G of this lane.
  float m_used = -INFINITY, l_run = 0.f;
  float* red = scratch + (warp * 2 + hw) * (2 * G * 16);
  const int rbase = warp * 4 + hw * 2;
  int s = 0, round = 0;
  int remain = tok_end - tok0;  // rows of this partition not yet consumed
  for (int i = 0; i < ntiles; ++i) {
    const int nvalid = min(kStageRows, remain);
    remain -= kStageRows;
    if (!mbar_wait(&full[s], round & 1)) {
      if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
      break;
    }
    if (stage_ok[s]) {
      const T* kt = ktile + (size_t)s * L.tile_elems;
      const T* vt = vtile + (size_t)s * L.tile_elems;
      if (nvalid == kStageRows) {
#pragma unroll 1
        for (int c = 0; c < kStageRows / kChunk; ++c)
          decode_chunk<T, D, G, false>(kt, vt, c * kChunk + rbase, kStageRows, q2, acc, m_used,
                                       l_run, red, l16);
      } else {
        for (int c = 0; c * kChunk < nvalid; ++c)
          decode_chunk<T, D, G, true>(kt, vt, c * kChunk + rbase, nvalid, q2, acc, m_used, l_run,
                                      red, l16);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (warp == 0 && i + NS < ntiles) {
      // every warp has released stage s: refill it with stage i + NS
      int ok = 1;
      if (lane == 0 && !mbar_wait(&empty[s], round & 1)) {
        atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        ok = 0;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issue_stage(s);
    }
    if (++s == NS) {
      s = 0;
      ++round;
    }
  }

  // ------------------------------------------------------------------ merge the 4 warps
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int j = 0; j < EP2; ++j) {
      acc[g][j].x += __shfl_xor_sync(0xffffffffu, acc[g][j].x, 16);
      acc[g][j].y += __shfl_xor_sync(0xffffffffu, acc[g][j].y, 16);
    }

  __syncthreads();  // every stage consumed: reuse the tiles
  float* macc = reinterpret_cast<float*>(smem);            // [4][G][D]
  float* mm = macc + kConsumerWarps * G * D;               // [4][G]
  float* ml = mm + kConsumerWarps * G;                     // [4][G]
  if (hw == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < EP2; ++j) {
        macc[(warp * G + g) * D + l16 * EPL + 2 * j] = acc[g][j].x;
        macc[(warp * G + g) * D + l16 * EPL + 2 * j + 1] = acc[g][j].y;
      }
    constexpr int LPV = 8 / G;  // lanes per (row, head) value
    if (l16 < 8 && l16 % LPV == 0) {  // row 0 of the half-warp, first lane of each head
      mm[warp * G + l16 / LPV] = m_used;
      ml[warp * G + l16 / LPV] = l_run;
    }
  }
  __syncthreads();

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
  static SmemAttrCache attr_cache;
  cudaError_t e = ensure_smem_limit(kern, (int)smem, attr_cache);
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
