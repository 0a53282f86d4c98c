// decode.cu -- split-K paged attention decode on CUDA cores (GQA groups <= 8).
//
// What it computes ("M5.3 - KV Memory Layout and Exact Reuse", 0x0A and
// 0x0BA): for sequence r and query head h, attention of q[r, h] over the
// request-visible rows t < T_r of kv head h / G, where row t lives in physical
// block block_tables[r, t / P] at offset t % P.  The rows of one (sequence,
// kv head) are cut into pieces; each piece keeps an online softmax state
// (m, l, u) and emits (O_p = u / l, LSE_p = m + log l); pieces are merged by
// log-sum-exp, never by averaging normalised outputs, with empty pieces as
// the identity.
//
// Design (GB300):
//   * persistent, balanced CTAs: the work is the list of 32-row stages of
//     every (sequence, kv head) segment, sequence-major; every CTA scans the
//     lengths itself (a block-wide prefix sum, no planning launch), and CTA c
//     of C (one wave: four per SM) takes the c-th equal share of the work
//     units (plan.cuh: a stage costs two, a piece's fixed cost three).  Every
//     CTA does the same work whatever the length mix, there is no tail wave,
//     and a CTA crosses segment boundaries without draining its pipeline;
//   * a segment a CTA covers whole is finished there (output written
//     directly); a segment cut by CTA boundaries leaves one (O, LSE) record
//     per piece -- at most two per CTA, for its first and last segments --
//     and a reduction kernel merges them;
//   * the G query heads of a kv head share every K/V byte the CTA reads;
//   * warp 0 also issues the loads: it walks the CTA's stages, holds the
//     current sequence's block ids 32 at a time (one coalesced load per 32
//     blocks, the next group in flight), and fills each 32-row stage with 4-D
//     TMA boxes (one block, or a 32-row slice of a larger block, of one kv
//     head) for K and V, tracked by mbarriers, plus a small descriptor of the
//     stage (sequence, head, valid rows, piece start / end) for the
//     consumers; a stage is refilled as soon as all four warps released it;
//   * warps consume 16-row chunks: each half-warp owns two token rows, each
//     lane 1/16 of head_dim; the 2G (row, head) partial dot products are
//     summed across the 16 lanes through a small per-warp shared scratch;
//     the row lands in lane bit 3; a vote on each lane's own score decides
//     whether the chunk needs the max over the warp's four rows (two
//     shuffles) and a rescale, and each lane sums its own rows' weights until
//     the piece end adds them; q . k and P . V use packed fp32x2 FMAs;
//   * full stages take a straight-line path with no row masking;
//   * at a piece's end the four warps merge through the stage's own tile
//     (released only afterwards), so the ring keeps streaming the next piece;
//   * the exponent base is only moved when the running max grows by more than
//     2^8 (exact: output and denominator keep the same base), so the
//     accumulator rescale is rare;
//   * scores are in base 2 (q is pre-multiplied by scale * log2 e);
//   * rows past the request's tail are never multiplied in, so stale or NaN
//     bytes in a recycled block cannot leak (M5.3 0x03G).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "plan.cuh"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = kConsumerWarps * 32;
constexpr int kChunk = 16;             // token rows per softmax update
constexpr float kRescaleLog2 = 8.0f;   // move the exponent base past 2^8 growth
constexpr float kLn2 = 0.6931471805599453f;
// Sources a merging warp loads at once (their latencies overlap).
constexpr int kMergeBatch = 8;

// The element storage of the pool -> the type of q and out (bf16 beside an
// MXFP8 pool, whose stages also carry their rows' E8M0 scales).
template <typename T>
struct IoOf {
  using type = T;
};
template <>
struct IoOf<__nv_fp8_e4m3> {
  using type = __nv_bfloat16;
};
template <typename T>
constexpr bool kIsMx = false;
template <>
constexpr bool kIsMx<__nv_fp8_e4m3> = true;

// Stage descriptor flags.
constexpr int kPieceStart = 1;   // first stage of a piece: reset the state, load q
constexpr int kPieceEnd = 2;     // last stage of a piece: merge the warps and write
constexpr int kWhole = 4;        // the piece is its whole segment: write the result
constexpr int kSlot1 = 8;        // a cut piece that is not the CTA's first: record slot 1

struct DecodeSmem {
  int tile_elems;   // rows * head_dim of one K (or V) tile
  int stages;
  size_t tiles_bytes, scale_off, bar_off, ok_off, desc_off, ring_off, scratch_off, total;
};

// Cross-lane sum scratch of one consumer warp, in floats: row i of half-warp
// hw (the 16 lanes' partial sums of value i) starts at red_row<G, kMx>(hw, i).
// Rows are placed so that neither the 32-lane store of a value nor an 8-lane
// phase of the 16-byte reads meets a bank conflict: for G = 4 each phase
// reads four rows whose bank offsets are {0, 4, 16, 20} (half-warp 1 at +16),
// packed into 260 floats; G = 8 takes rows 20 floats apart; G = 1, 2 only
// offset half-warp 1 by 16 banks.  MXFP8 with G = 4 keeps the plain
// 256-float layout (two-way conflicts): the four extra floats per warp would
// cost its six-stage ring a CTA per SM.
__host__ __device__ constexpr int red_warp_floats(int g, int elem_bytes) {
  return g == 4 ? (elem_bytes == 1 ? 256 : 260) : g == 8 ? 672 : 2 * (32 * g + 16);
}
template <int G, bool kMx>
__device__ __forceinline__ int red_row(int hw, int i) {
  if constexpr (G == 4 && kMx)
    return hw * 128 + i * 16;
  else if constexpr (G == 4)
    return ((i & 1) ? 132 : 0) + 16 * (2 * (i >> 2) + (hw ? 5 - ((i >> 1) & 1) : ((i >> 1) & 1)));
  else if constexpr (G == 8)
    return hw * 336 + i * 20;
  else
    return hw * (32 * G + 16) + i * 16;
}

// Stage s holds its K tile then its V tile; both together also hold the
// [4][G][D] fp32 merge of a piece's end (16 G D bytes <= 2 * 32 * D * b for
// G <= 8 with 2- and 4-byte elements, G <= 4 with 1-byte ones).
__host__ __device__ inline DecodeSmem decode_smem_layout(int head_dim, int elem_bytes, int group,
                                                         int stages) {
  DecodeSmem s;
  s.tile_elems = kStageRows * head_dim;
  s.stages = stages;
  s.tiles_bytes = ((size_t)2 * stages * s.tile_elems * elem_bytes + 127) & ~(size_t)127;
  // MXFP8 (1-byte elements): each stage's K then V scale rows [rows][D / 32]
  s.scale_off = s.tiles_bytes;
  const size_t scale_bytes = elem_bytes == 1 ? (size_t)2 * stages * kStageRows * (head_dim / 32) : 0;
  s.bar_off = s.scale_off + ((scale_bytes + 127) & ~(size_t)127);  // full[stages], empty[stages], merge
  s.ok_off = s.bar_off + (size_t)(2 * stages + 1) * 8;
  s.desc_off = (s.ok_off + (size_t)stages * 4 + 15) & ~(size_t)15;
  s.ring_off = s.desc_off + (size_t)stages * 16;
  s.scratch_off = s.ring_off + (size_t)2 * 64 * 16;  // two 64-entry stage descriptor rings
  // scratch: the warps' cross-lane sums (red_warp_floats each), then the
  // merge's per-warp maxima and sums [2][4][G]
  s.total = s.scratch_off + (size_t)kConsumerWarps * red_warp_floats(group, elem_bytes) * 4 +
            (size_t)2 * kConsumerWarps * group * 4 + 128;  // +128: base alignment
  return s;
}

int decode_num_stages(int head_dim, int elem_bytes) {
  const int stage_bytes = 2 * kStageRows * head_dim * elem_bytes;
  int ns = (49 * 1024) / stage_bytes;  // 3 stages of 16 KiB: 4 CTAs per SM
  if (ns < 2) ns = 2;
  if (ns > 8) ns = 8;
  return ns;
}

// One 16-row chunk of a stage for one consumer warp: rows row0 and row0 + 1
// of this half-warp.  kTail = false is the full-stage fast path (every row
// valid, no masking); kTail = true masks rows >= nvalid.
//
// Cross-lane sums go through `red`, this warp's scratch: lane l16 of
// half-warp hw stores its partial dot product of value i = (row tk, head g) =
// tk*G + g at red[red_row(hw, i) + l16]; then each value is summed by 8/G
// lanes that read 2G
// consecutive partials each and combine with 8/G - 1 shuffles.  Lane l16 ends
// up holding value j = l16 / (8/G): row tk = l16 >> 3, head g = j % G.
//
// l_run is this lane's share of its head's softmax sum: the weights of its
// own rows (one per chunk); the piece end adds the four row lanes' shares.
// Store N consecutive outputs (fp32, or bf16 rounded to nearest even) with
// the widest aligned vector stores: the destination is aligned to N elements.
template <int N>
__device__ __forceinline__ void store_vec(float* p, const float (&o)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i)
      reinterpret_cast<float4*>(p)[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  } else if constexpr (N == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(o[0], o[1]);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) p[i] = o[i];
  }
}
template <int N>
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&o)[N]) {
  if constexpr (N % 2 == 0) {
    uint32_t w[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    if constexpr (N == 8)
      *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else if constexpr (N == 4)
      *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
    else
      *reinterpret_cast<uint32_t*>(p) = w[0];
  } else {
    *p = __float2bfloat16_rn(o[0]);
  }
}

template <typename T, int D, int G, bool kTail>
__device__ __forceinline__ void decode_chunk(const T* __restrict__ kt, const T* __restrict__ vt,
                                             const uint8_t* __restrict__ ksc,
                                             const uint8_t* __restrict__ vsc, int row0,
                                             int nvalid, const float2 (&q2)[G][D / 32],
                                             float2 (&acc)[G][D / 32], float& m_used,
                                             float& l_run, float* __restrict__ red, int hw, int l16) {
  constexpr int EPL = D / 16;
  constexpr int EP2 = EPL / 2;
  constexpr int NV = 2 * G;    // values per half-warp and chunk
  constexpr int LPV = 16 / NV; // lanes summing one value
  // MXFP8: this lane's EPL elements lie in one 32-element scale group; its
  // V scale multiplies the weights (a power of two).  The K scales are
  // applied in the cross-lane sum, once per group of partials.
  float vscale[2] = {1.f, 1.f};
  if constexpr (kIsMx<T>) {
    const int grp = l16 * EPL / 32;
#pragma unroll
    for (int tk = 0; tk < 2; ++tk) vscale[tk] = e8m0_value(vsc[(row0 + tk) * (D / 32) + grp]);
  }
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
  for (int i = 0; i < NV; ++i) red[red_row<G, kIsMx<T>>(hw, i) + l16] = v[i];
  __syncwarp();
  const int j = l16 / LPV, sub = l16 % LPV;
  float part[NV];
  VecLoad<float, NV>::run(red + red_row<G, kIsMx<T>>(hw, j) + sub * NV, part);
  __syncwarp();  // the next chunk rewrites red
  float s2;
  if constexpr (kIsMx<T>) {
    // the NV partials span NG scale groups of the row of value j: sum each
    // group's partials, then scale it by that group's K scale
    constexpr int NG = NV * EPL >= 64 ? NV * EPL / 32 : 1;
    constexpr int PPG = NV / NG;  // partials per group
    const int rowj = row0 + j / G;
    s2 = 0.f;
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      float gs = part[q * PPG];
#pragma unroll
      for (int k = 1; k < PPG; ++k) gs += part[q * PPG + k];
      const int grp = (sub * NV + q * PPG) * EPL / 32;
      s2 = fmaf(gs, e8m0_value(ksc[rowj * (D / 32) + grp]), s2);
    }
  } else {
    s2 = part[0];
#pragma unroll
    for (int k = 1; k < NV; ++k) s2 += part[k];
  }
#pragma unroll
  for (int o = LPV / 2; o >= 1; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  // ---- online softmax over the warp's 4 rows (rows differ in lane bits 3, 4)
  const float sc = (!kTail || row0 + (l16 >> 3) < nvalid) ? s2 : -INFINITY;
  // The exponent base of a head moves only when one of its scores passes it
  // by more than 2^8 (m_used = -inf before a piece's first row), so most
  // chunks need neither the cross-row max nor a rescale.
  if (__any_sync(0xffffffffu, sc > m_used + kRescaleLog2)) {
    float cmax = fmaxf(sc, __shfl_xor_sync(0xffffffffu, sc, 8));
    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 16));
    const float m_new = fmaxf(m_used, cmax);
    const bool need = m_new > m_used + kRescaleLog2;
    const float alpha = need ? exp2f(m_used - m_new) : 1.f;
    m_used = need ? m_new : m_used;
    l_run *= alpha;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float al = __shfl_sync(0xffffffffu, alpha, g * LPV, 16);
      const float2 al2 = make_float2(al, al);
#pragma unroll
      for (int e = 0; e < EP2; ++e) acc[g][e] = __fmul2_rn(acc[g][e], al2);
    }
  }
  const float p = (kTail && sc == -INFINITY) ? 0.f : exp2f(sc - m_used);
  l_run += p;
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
        const float pv = kIsMx<T> ? pg[tk][g] * vscale[tk] : pg[tk][g];
        const float2 p2 = make_float2(pv, pv);
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
  using TQ = typename IoOf<T>::type;  // q and out
  constexpr int EPL = D / 16;  // head_dim elements per lane
  constexpr int EP2 = EPL / 2;
  constexpr int NV = 2 * G;    // (row, head) partial sums per lane per chunk
  static_assert(NV <= 16 && (NV & (NV - 1)) == 0, "group must be 1, 2, 4 or 8");
  static_assert(!kIsMx<T> || G <= 4, "an MXFP8 stage tile holds the merge of up to 4 heads");
  constexpr int kScaleRow = D / 32;  // MXFP8 scale bytes per row

  const int c = blockIdx.x;
  const int Hkv = a.num_kv_heads, P = a.block_size;
  const int TB = box_rows_for(P);  // rows per TMA box
  const DecodeSmem L = decode_smem_layout(D, (int)sizeof(T), G, a.num_stages);
  const int NS = a.num_stages;
  extern __shared__ unsigned char smem_raw[];
  // Align by offsetting the array itself (not through an integer), so the
  // compiler keeps every tile and scratch access in the shared state space.
  unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  T* tiles = reinterpret_cast<T*>(smem);  // [NS][K tile, V tile]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + NS;
  uint64_t* mrg = empty + NS;  // all 128 threads arrive: the merge's CTA barrier
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + L.ok_off);
  int4* sdesc = reinterpret_cast<int4*>(smem + L.desc_off);  // per ring slot: (seq, head, rows, flags)
  int4* dA = reinterpret_cast<int4*>(smem + L.ring_off);      // per stage: (id0, id1, row, boxes)
  int4* dB = dA + 64;                                          // per stage: (seq, head, rows, flags)
  float* scratch = reinterpret_cast<float*>(smem + L.scratch_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- plan
  if (!a.plan_before_wait) pdl_wait();  // inputs written by earlier kernels are visible
  pdl_launch_dependents();   // the reduction may be scheduled as CTAs retire
  int4 d0;
  const int n = plan_cta_stages<kDecodeThreads, kStageRows>(
      a, reinterpret_cast<long long*>(scratch), &d0);
  if (n <= 0) return;  // no stages: the whole CTA leaves before any barrier
  const int hw = lane >> 4, l16 = lane & 15;
  float2 q2[G][EP2];
  float2 acc[G][EP2];
  // q of a piece, scaled, into registers.  Every piece after the CTA's
  // first starts right after a piece end, whose merge the load overlaps.
  // The first: where units are stages the plan names its stage, so its q
  // loads now, under the set-up; otherwise it is the first batch's first
  // descriptor.
  auto load_q = [&](int r, int h) {
    const int64_t qr = a.q_rows ? __ldg(a.q_rows + r) : r;
    const TQ* qp = static_cast<const TQ*>(a.q) + (qr * a.num_q_heads + (int64_t)h * G) * D + l16 * EPL;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float f[EPL];
      VecLoad<TQ, EPL>::run(qp + g * D, f);
#pragma unroll
      for (int j = 0; j < EP2; ++j) q2[g][j] = make_float2(f[2 * j] * a.qscale, f[2 * j + 1] * a.qscale);
    }
  };
  // The same in two halves, for a piece end: the raw loads are issued before
  // the merge (from q row qr, the descriptor's) and widened after it, so the
  // merge covers their latency.  The raw words wait in q2's own registers
  // (bf16: in the upper half of each head's q2; fp32: the values themselves),
  // so the hot loop loses no registers to them.
  auto load_q_raw = [&](int64_t qr, int h) {
    const TQ* qp = static_cast<const TQ*>(a.q) + (qr * a.num_q_heads + (int64_t)h * G) * D + l16 * EPL;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if constexpr (sizeof(TQ) == 4) {
#pragma unroll
        for (int j = 0; j < EP2; ++j) q2[g][j] = __ldg(reinterpret_cast<const float2*>(qp + g * D) + j);
      } else {
#pragma unroll
        for (int i = 0; i < EPL / 4; ++i) {
          const uint2 x = __ldg(reinterpret_cast<const uint2*>(qp + g * D) + i);
          q2[g][EP2 / 2 + i] = make_float2(__uint_as_float(x.x), __uint_as_float(x.y));
        }
      }
    }
  };
  auto finish_q = [&]() {
    const float2 s2 = make_float2(a.qscale, a.qscale);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if constexpr (sizeof(TQ) == 4) {
#pragma unroll
        for (int j = 0; j < EP2; ++j) q2[g][j] = __fmul2_rn(q2[g][j], s2);
      } else {
        uint32_t wv[EP2];  // the EPL bf16 as EP2 words
#pragma unroll
        for (int i = 0; i < EPL / 4; ++i) {
          wv[2 * i] = __float_as_uint(q2[g][EP2 / 2 + i].x);
          wv[2 * i + 1] = __float_as_uint(q2[g][EP2 / 2 + i].y);
        }
#pragma unroll
        for (int j = 0; j < EP2; ++j)
          q2[g][j] = make_float2(bf16lo(wv[j]) * a.qscale, bf16hi(wv[j]) * a.qscale);
      }
    }
  };
  const bool d0_exact = a.stage_units == 1 && a.piece_units == 0;
  if (d0_exact && !a.plan_before_wait) load_q(d0.x, d0.y);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(mrg, kDecodeThreads);
    fence_barrier_init();
  }
  __syncthreads();

  // ---------------------------------------------------------------- loads
  // Warp 0 issues the loads.  Once per 32 stages it works out the next 32
  // stages of the CTA's range lane-parallel (lane l: stage kb + l) into a
  // two-batch descriptor ring in shared memory: block ids of the stage's
  // boxes, first row in the block, box count, and (sequence, kv head, valid
  // rows, flags).  The cursor (cr, ch, ci) is the position of the next
  // batch's first stage, cpnt / cT the stages and length of sequence cr.
  int cr = d0.x, ch = d0.y, ci = d0.z, cpnt = 0, cT = 0;
  const uint32_t box_bytes = (uint32_t)(TB * D * sizeof(T));
  const uint32_t scale_box = (uint32_t)(TB * kScaleRow);  // MXFP8 scale bytes of one box
  auto compute_batch = [&](int kb) {
    int r = cr, h = ch, i = ci + lane, pnt = cpnt, len = cT;
    const bool act = kb + lane < n;
    if (act) {
      while (i >= pnt) {  // crossed into a later segment (rare)
        i -= pnt;
        if (++h == Hkv) {
          h = 0;
          do {
            ++r;
            len = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
            pnt = (len + kStageRows - 1) / kStageRows;
          } while (pnt == 0);
        }
      }
      const int k = kb + lane, row0 = i * kStageRows;
      const int nvalid = min(kStageRows, len - row0);
      const int b0 = row0 / P;
      const int nbox = (nvalid + TB - 1) / TB;  // 1 or 2 (two only when P < 32)
      const int32_t* tbl = a.block_tables + (int64_t)r * a.max_blocks + b0;
      const int id0 = __ldg(tbl), id1 = nbox > 1 ? __ldg(tbl + 1) : -1;
      const int dseg = k - i;  // CTA stage index of the segment's first stage
      const bool end = k == n - 1 || i == pnt - 1;
      const int flags = (k == 0 || i == 0 ? kPieceStart : 0) | (end ? kPieceEnd : 0) |
                        (end && i == pnt - 1 && dseg >= 0 ? kWhole : 0) | (dseg > 0 ? kSlot1 : 0);
      if (flags & kPieceStart) {  // the piece's q rows, into L2 long before they are read
        const int64_t qr = a.q_rows ? __ldg(a.q_rows + r) : r;
        prefetch_l2_bulk(static_cast<const TQ*>(a.q) + (qr * a.num_q_heads + (int64_t)h * G) * D,
                         (uint32_t)(G * D * sizeof(TQ)));
      }
      // the piece's q row rides in the box-count word (nbox is 1 or 2)
      const int qrow = a.q_rows ? __ldg(a.q_rows + r) : r;
      dA[k & 63] = make_int4(id0, id1, row0 - b0 * P, nbox | (qrow << 2));
      dB[k & 63] = make_int4(r, h, nvalid, flags);
    }
    // the cursor moves to the stage after lane 31's
    cr = __shfl_sync(0xffffffffu, r, 31);
    ch = __shfl_sync(0xffffffffu, h, 31);
    ci = __shfl_sync(0xffffffffu, i, 31) + 1;
    cpnt = __shfl_sync(0xffffffffu, pnt, 31);
    cT = __shfl_sync(0xffffffffu, len, 31);
    __syncwarp();
  };
  // Fill ring slot `st` with the CTA's k-th stage (warp 0, all lanes).
  auto issue_stage = [&](int st, int k) {
    const int4 da = dA[k & 63];
    const int4 db = dB[k & 63];
    const int nbox = da.w & 3;
    const bool valid = da.x >= 0 && (int64_t)da.x < a.num_blocks &&
                       (nbox < 2 || (da.y >= 0 && (int64_t)da.y < a.num_blocks));
    if (lane == 0) sdesc[st] = db;
    if ((db.w & kPieceStart) && lane == 31)  // refresh the piece's q in L2 shortly before use
      prefetch_l2_bulk(static_cast<const TQ*>(a.q) +
                           ((int64_t)(da.w >> 2) * a.num_q_heads + (int64_t)db.y * G) * D,
                       (uint32_t)(G * D * sizeof(TQ)));
    if (!valid) {
      if (lane == 0) {
        atomicOr(a.err, PKV_DEVERR_BLOCK);
        stage_ok[st] = 0;
        mbar_arrive(&full[st]);
      }
    } else {
      if (lane == 0) {
        stage_ok[st] = 1;
        mbar_arrive_expect_tx(&full[st], 2u * (box_bytes + (kIsMx<T> ? scale_box : 0u)) * (uint32_t)nbox);
      }
      __syncwarp();
      // one box per lane: lanes 0..nbox-1 load K, lanes 16..16+nbox-1 load V;
      // MXFP8: lanes 8.. and 24.. copy the same boxes' scale rows, which lie
      // contiguously in the head-major scale plane
      const int j = lane & 15;
      if (j < nbox) {
        T* dst = tiles + (size_t)st * 2 * L.tile_elems + (lane < 16 ? 0 : L.tile_elems) + j * TB * D;
        tma_load_4d(dst, lane < 16 ? &tmk : &tmv, 0, db.y, j == 0 ? da.z : 0, j == 0 ? da.x : da.y,
                    &full[st]);
      }
      if constexpr (kIsMx<T>) {
        const int js = j - 8;
        if (js >= 0 && js < nbox) {
          const int64_t blk = js == 0 ? da.x : da.y;
          const int row = js == 0 ? da.z : 0;
          const uint8_t* src = (lane < 16 ? a.k_scales : a.v_scales) +
                               ((blk * Hkv + db.y) * P + row) * kScaleRow;
          uint8_t* sdst = smem + L.scale_off + (size_t)st * 2 * kStageRows * kScaleRow +
                          (lane < 16 ? 0 : kStageRows * kScaleRow) + js * TB * kScaleRow;
          bulk_load(sdst, src, scale_box, &full[st]);
        }
      }
    }
    // The next batch (stages kb + 32 ..) overwrites the ring entries of
    // stages kb - 32 .. kb - 1, which a consumer still reads at a piece end
    // (the next stage's q) until it has released stage kb - 1.  So it is
    // worked out with the refill of stage kb + NS - 1, which warp 0 issues
    // only after every warp released stage kb - 1, and still before stage
    // kb + 32 (NS <= 8) is issued.
    const int kb = k - (NS - 1);
    if (kb >= 0 && (kb & 31) == 0 && kb + 32 < n) compute_batch(kb + 32);
  };
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    cT = effective_len(__ldg(a.seq_lens + cr), a.max_blocks, P, a.err, false);
    cpnt = (cT + kStageRows - 1) / kStageRows;
    compute_batch(0);  // lengths, block tables and q rows only
  }
  // With plan_before_wait, what the preceding kernel may still write (K/V
  // rows, q) is read only from here on.
  if (a.plan_before_wait) {
    pdl_wait();
    if (d0_exact) load_q(d0.x, d0.y);
  }
  if (d0_exact && warp == 0)
    for (int st = 0; st < NS && st < n; ++st) issue_stage(st, st);
  if (!d0_exact) {
    __syncthreads();  // the first batch's descriptors: every warp reads its first piece there
    if (warp == 0)
      for (int st = 0; st < NS && st < n; ++st) issue_stage(st, st);
  }

  // ------------------------------------------------------------------ consumers
  if (!d0_exact) load_q(dB[0].x, dB[0].y);
  // (m_used, l_run): softmax state of head (l16 / (8 / G)) % G of this lane
  // (l_run: the weights of this lane's own rows).
  float m_used = -INFINITY, l_run = 0.f;
  float* red = scratch + warp * red_warp_floats(G, (int)sizeof(T));
  const int rbase = warp * 4 + hw * 2;
  int s = 0, round = 0;
  uint32_t mrg_phase = 0;
  // CTA barrier of the merge, bounded like every wait here; warp-uniform.
  auto merge_sync = [&]() -> bool {
    mbar_arrive(mrg);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(mrg, mrg_phase));
    mrg_phase ^= 1u;
    if (!ok && lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    return ok;
  };
  int k = 0;
  for (; k < n; ++k) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], round & 1))) {
      if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
      break;
    }
    const int4 dsc = sdesc[s];  // (sequence, kv head, valid rows, flags)
    const int nvalid = dsc.z, flags = dsc.w;
    const T* kt = tiles + (size_t)s * 2 * L.tile_elems;
    const T* vt = kt + L.tile_elems;
    const uint8_t* ksc = smem + L.scale_off + (size_t)s * 2 * kStageRows * kScaleRow;
    const uint8_t* vsc = ksc + kStageRows * kScaleRow;
    if (flags & kPieceStart) {  // q2 already holds this piece's q
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < EP2; ++j) acc[g][j] = make_float2(0.f, 0.f);
      m_used = -INFINITY;
      l_run = 0.f;
    }
    if (stage_ok[s]) {
      if (nvalid == kStageRows) {
#pragma unroll 1
        for (int cc = 0; cc < kStageRows / kChunk; ++cc)
          decode_chunk<T, D, G, false>(kt, vt, ksc, vsc, cc * kChunk + rbase, kStageRows, q2, acc, m_used,
                                       l_run, red, hw, l16);
      } else {
        for (int cc = 0; cc * kChunk < nvalid; ++cc)
          decode_chunk<T, D, G, true>(kt, vt, ksc, vsc, cc * kChunk + rbase, nvalid, q2, acc, m_used, l_run,
                                      red, hw, l16);
      }
    }
    if (flags & kPieceEnd) {
      // The next stage starts the next piece: issue its q loads now (this
      // piece's is no longer needed) and widen them after the merge, which
      // covers their latency.  Its descriptor was written before this
      // stage's was published (the same batch, or an earlier one).
      const bool next_q = k + 1 < n;
      if (next_q) load_q_raw(dA[(k + 1) & 63].w >> 2, dB[(k + 1) & 63].y);
      // ---- merge the four warps through this stage's tile, then write
      if (!merge_sync()) break;  // every warp is done with the tile
      float* macc = reinterpret_cast<float*>(const_cast<T*>(kt));  // [4][G][D]
      float* mm = scratch + kConsumerWarps * red_warp_floats(G, (int)sizeof(T));  // [4][G]
      float* ml = mm + kConsumerWarps * G;                          // [4][G]
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < EP2; ++j) {
          float2 v = acc[g][j];
          v.x += __shfl_xor_sync(0xffffffffu, v.x, 16);
          v.y += __shfl_xor_sync(0xffffffffu, v.y, 16);
          if (hw == 0) {
            macc[(warp * G + g) * D + l16 * EPL + 2 * j] = v.x;
            macc[(warp * G + g) * D + l16 * EPL + 2 * j + 1] = v.y;
          }
        }
      constexpr int LPV = 8 / G;  // lanes per (row, head) value
      float lsum = l_run + __shfl_xor_sync(0xffffffffu, l_run, 8);  // the warp's four rows
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
      if (lane < 8 && lane % LPV == 0) {  // row 0 of half-warp 0, first lane of each head
        mm[warp * G + lane / LPV] = m_used;
        ml[warp * G + lane / LPV] = lsum;
      }
      if (!merge_sync()) break;
      const int64_t rh0 = (int64_t)dsc.x * a.num_q_heads + (int64_t)dsc.y * G;
      const int64_t rec = (int64_t)2 * c + ((flags & kSlot1) ? 1 : 0);
      // Each thread takes EPT consecutive outputs of one head: the head's
      // weights once, then vector loads, one reciprocal and vector stores.
      constexpr int kOut = G * D;
      constexpr int EPT = kOut >= kDecodeThreads ? kOut / kDecodeThreads : 1;
      const int j0 = threadIdx.x * EPT;
      if (j0 < kOut) {
        const int g = j0 / D, e0 = j0 % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * G + g]);
        float Lsum = 0.f, o[EPT];
#pragma unroll
        for (int i = 0; i < EPT; ++i) o[i] = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = exp2f(mm[w * G + g] - M);
            Lsum = fmaf(wt, ml[w * G + g], Lsum);
            float x[EPT];
            if constexpr (EPT == 1)
              x[0] = macc[(w * G + g) * D + e0];
            else
              VecLoad<float, EPT>::run(macc + (w * G + g) * D + e0, x);
#pragma unroll
            for (int i = 0; i < EPT; ++i) o[i] = fmaf(wt, x[i], o[i]);
          }
        }
        const bool nonempty = Lsum > 0.f;
        const float inv = nonempty ? 1.f / Lsum : 0.f;
#pragma unroll
        for (int i = 0; i < EPT; ++i) o[i] *= inv;
        const int64_t rh = rh0 + g;
        float* dst32 = nullptr;
        if (!(flags & kWhole)) {
          dst32 = a.rec_o + (rec * G + g) * D + e0;
          if (e0 == 0) a.rec_lse[rec * G + g] = nonempty ? M + log2f(Lsum) : -INFINITY;
        } else if (a.st_o) {
          const int64_t slot = rh * a.st_stride + a.st_slot;
          dst32 = a.st_o + slot * D + e0;
          if (e0 == 0) a.st_lse[slot] = nonempty ? M + log2f(Lsum) : -INFINITY;
        } else {
          store_vec(static_cast<TQ*>(a.out) + rh * D + e0, o);
          if (e0 == 0 && a.lse_out) a.lse_out[rh] = nonempty ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
        }
        if (dst32) store_vec(dst32, o);
      }
      if (next_q) finish_q();
      // No barrier here: each warp releases the tile below once its own merge
      // reads are done, and the producer refills it only after all four have;
      // mm / ml are rewritten only after the next piece's first barrier.
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (warp == 0 && k + NS < n) {
      // every warp has released ring slot s: refill it with stage k + NS
      int ok = 1;
      if (lane == 0 && !mbar_wait(&empty[s], round & 1)) {
        atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        ok = 0;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issue_stage(s, k + NS);
    }
    if (++s == NS) {
      s = 0;
      ++round;
    }
  }
  if (k < n && warp == 0 && lane == 0) {
    // left early after a timeout: wait (bounded) for copies still in flight
    // into the ring before the CTA's shared memory is released
    for (int kk = k; kk < min(n, k + NS); ++kk) mbar_wait(&full[kk % NS], (kk / NS) & 1);
  }
}

// One warp per (sequence, query head): merge the pieces of its segment (and,
// in states mode, the extra states before them) by log-sum-exp.  A segment
// one CTA covered whole was written by that CTA (plain mode: nothing to do).
template <typename T, int D>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeArgs a) {
  constexpr int EPL = D / 32;
  pdl_wait();  // the partial kernel's records and plan are complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rh = (int64_t)blockIdx.x * 4 + warp;
  if (rh >= (int64_t)a.num_seqs * a.num_q_heads) return;
  const int r = (int)(rh / a.num_q_heads), qh = (int)(rh % a.num_q_heads);
  const int G = a.num_q_heads / a.num_kv_heads, h = qh / G, g = qh % G;
  const int Hkv = a.num_kv_heads, C = a.num_ctas;
  // the work split of plan.cuh, in units: segment (r, h) starts at unit
  // seg0, its stage i at seg0 + pu + su i, owned by CTA (start) / w
  const long long su = a.stage_units, pu = a.piece_units;
  const long long S = a.plan_pre[a.num_seqs] * Hkv;
  const long long pre = a.plan_pre[r], u = a.plan_pre[r + 1] - pre;
  const long long nt = u > 0 ? (u - pu) / su : 0;
  const int n_ext = a.st_o ? a.st_slot : 0;
  // Sources: extra states [0, n_ext), then either the whole-segment state
  // (states mode) or pieces c_first..c_last.
  const long long w = units_per_cta(S, C, su);
  int c_first = 0, n_pc = 0;  // pieces: CTAs c_first .. c_first + n_pc - 1
  bool whole_state = false;
  bool first_is_slot1 = false;
  if (nt > 0) {
    const long long seg0 = pre * Hkv + (long long)h * u;
    c_first = (int)((seg0 + pu) / w);
    const int c_last = (int)((seg0 + pu + su * (nt - 1)) / w);
    if (c_first == c_last) {
      // written whole by its CTA: to out, or to its state slot, which is
      // already the result when only states are wanted and none merge in
      if (!a.st_o || (!a.out && n_ext == 0)) return;
      whole_state = true;
    } else {
      n_pc = c_last - c_first + 1;
      // a cut segment's first piece is in slot 1 of its CTA when that CTA
      // owns an earlier stage: the stage just before, which starts at
      // seg0 - su, the last of the previous non-empty segment
      first_is_slot1 = seg0 > 0 && seg0 - su >= (long long)c_first * w;
    }
  }
  const float* ext_lse = a.st_o ? a.st_lse + rh * a.st_stride : nullptr;
  const float* ext_o = a.st_o ? a.st_o + rh * a.st_stride * D : nullptr;
  const int n_st = n_ext + (whole_state ? 1 : 0);
  auto piece_rec = [&](int i) -> int64_t {  // record of piece i (CTA c_first + i)
    const int64_t cc = c_first + i;
    return (2 * cc + (i == 0 && first_is_slot1 ? 1 : 0)) * G + g;
  };
  // Sources 0 .. n-1: lane i holds source i's LSE (sources past 32, rare,
  // are read again in pass 2); pass 2 loads the outputs kMergeBatch at a
  // time so their latencies overlap.
  const int n = n_st + n_pc;
  auto src_lse = [&](int i) -> float {
    return i < n_st ? ext_lse[i] : a.rec_lse[piece_rec(i - n_st)];
  };
  auto src_o = [&](int i) -> const float* {
    return i < n_st ? ext_o + (int64_t)i * D : a.rec_o + piece_rec(i - n_st) * D;
  };
  const float my0 = lane < n ? src_lse(lane) : -INFINITY;
  float M = my0;
  for (int i = lane + 32; i < n; i += 32) M = fmaxf(M, src_lse(i));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float Lsum = 0.f;
  if (M != -INFINITY) {
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int m = min(32, n - i0);
      const float my = i0 == 0 ? my0 : (lane < m ? src_lse(i0 + lane) : -INFINITY);
      for (int u0 = 0; u0 < m; u0 += kMergeBatch) {
        float l[kMergeBatch], x[kMergeBatch][EPL];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          l[u] = __shfl_sync(0xffffffffu, my, (u0 + u) & 31);
          if (u0 + u >= m) l[u] = -INFINITY;  // an empty state: the merge's identity
#pragma unroll
          for (int e = 0; e < EPL; ++e) x[u][e] = 0.f;
          if (l[u] != -INFINITY) VecLoad<float, EPL>::run(src_o(i0 + u0 + u) + lane * EPL, x[u]);
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          if (l[u] == -INFINITY) continue;
          const float w = exp2f(l[u] - M);
          Lsum += w;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, x[u][e], acc[e]);
        }
      }
    }
  }
  const bool nonempty = Lsum > 0.f;
  if (!a.out) {  // states only: the merged pieces become the segment's state
    const int64_t slot = rh * a.st_stride + a.st_slot;
    float* so = a.st_o + slot * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) so[e] = nonempty ? acc[e] / Lsum : 0.f;
    if (lane == 0) a.st_lse[slot] = nonempty ? M + log2f(Lsum) : -INFINITY;
    return;
  }
  T* out = static_cast<T*>(a.out) + rh * D + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) store_out(out + e, nonempty ? acc[e] / Lsum : 0.f);
  if (lane == 0 && a.lse_out) a.lse_out[rh] = nonempty ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
}

template <typename T, int D, int G>
static size_t partial_smem_bytes() {
  return decode_smem_layout(D, (int)sizeof(T), G, decode_num_stages(D, (int)sizeof(T))).total;
}

template <typename T, int D, int G>
static cudaError_t launch_partial(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                  const DecodeArgs& a, cudaStream_t stream) {
  const size_t smem = decode_smem_layout(D, (int)sizeof(T), G, a.num_stages).total;
  auto kern = decode_partial_kernel<T, D, G>;
  static SmemAttrCache attr_cache;
  cudaError_t e = ensure_smem_limit(kern, (int)smem, attr_cache);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)a.num_ctas), dim3(kDecodeThreads), smem, stream, tmk, tmv,
                    a);
}

// Resident CTAs per SM of one partial-kernel instance, looked up once per
// device.
template <typename T, int D, int G>
static int resident_ctas() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    const size_t smem = partial_smem_bytes<T, D, G>();
    auto kern = decode_partial_kernel<T, D, G>;
    int per_sm = 0, sms = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, smem) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    cached[dev] = per_sm * sms;
  }
  return cached[dev];
}

template <typename T, int D>
static int resident_for_group(int group) {
  switch (group) {
    case 1: return resident_ctas<T, D, 1>();
    case 2: return resident_ctas<T, D, 2>();
    case 4: return resident_ctas<T, D, 4>();
    case 8:
      if constexpr (!kIsMx<T>) return resident_ctas<T, D, 8>();
      return 0;
    default: return 0;
  }
}

int decode_resident_ctas(int dtype, int head_dim, int group) {
  if (dtype == PKV_MXFP8) {
    if (group > 4) return 0;
    return head_dim == 128 ? resident_for_group<__nv_fp8_e4m3, 128>(group)
                           : resident_for_group<__nv_fp8_e4m3, 64>(group);
  }
  if (dtype == PKV_BF16)
    return head_dim == 128 ? resident_for_group<__nv_bfloat16, 128>(group)
                           : resident_for_group<__nv_bfloat16, 64>(group);
  return head_dim == 128 ? resident_for_group<float, 128>(group)
                         : resident_for_group<float, 64>(group);
}

template <typename T, int D>
static cudaError_t dispatch_group(int group, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                  const DecodeArgs& a, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_partial<T, D, 1>(tmk, tmv, a, stream);
    case 2: return launch_partial<T, D, 2>(tmk, tmv, a, stream);
    case 4: return launch_partial<T, D, 4>(tmk, tmv, a, stream);
    case 8:
      if constexpr (!kIsMx<T>) return launch_partial<T, D, 8>(tmk, tmv, a, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D>
static cudaError_t launch_reduce_t(const DecodeArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.num_seqs * a.num_q_heads;
  return launch_pdl(decode_reduce_kernel<T, D>, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0,
                    stream, a);
}

cudaError_t launch_decode_reduce(int dtype, int head_dim, const DecodeArgs& a,
                                 cudaStream_t stream) {
  if (dtype == PKV_BF16 || dtype == PKV_MXFP8)  // out is bf16 beside an MXFP8 pool
    return head_dim == 128 ? launch_reduce_t<__nv_bfloat16, 128>(a, stream)
                           : launch_reduce_t<__nv_bfloat16, 64>(a, stream);
  return head_dim == 128 ? launch_reduce_t<float, 128>(a, stream)
                         : launch_reduce_t<float, 64>(a, stream);
}

cudaError_t launch_paged_decode(int dtype, int head_dim, int group, const CUtensorMap& tmk,
                                const CUtensorMap& tmv, const DecodeArgs& a,
                                cudaStream_t stream) {
  cudaError_t e;
  if (dtype == PKV_MXFP8)
    e = head_dim == 128 ? dispatch_group<__nv_fp8_e4m3, 128>(group, tmk, tmv, a, stream)
                        : dispatch_group<__nv_fp8_e4m3, 64>(group, tmk, tmv, a, stream);
  else if (dtype == PKV_BF16)
    e = head_dim == 128 ? dispatch_group<__nv_bfloat16, 128>(group, tmk, tmv, a, stream)
                        : dispatch_group<__nv_bfloat16, 64>(group, tmk, tmv, a, stream);
  else
    e = head_dim == 128 ? dispatch_group<float, 128>(group, tmk, tmv, a, stream)
                        : dispatch_group<float, 64>(group, tmk, tmv, a, stream);
  if (e != cudaSuccess) return e;
  return launch_decode_reduce(dtype, head_dim, a, stream);
}

}  // namespace pkv
