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
//   * CTA = (key split, two 128-row query tiles A and B, kv head).  Both
//     tiles use every K/V tile the CTA stages: the prefix blocks arrive as
//     one TMA box each (a 16-row block of head_dim 128 is 4 KiB, both column
//     halves, in the row-group tiles of launch.h), and the TMA engine, not
//     the tensor pipe, bounds a one-tile CTA, so each staged byte feeds two
//     128 x 128 x D MMAs;
//   * thread t of a softmax warpgroup owns query row t of its tile, i.e. TMEM
//     lane t, so the softmax needs no cross-thread reduction;
//   * Q (128 rows x D per tile), K and V tiles (128 keys x D) arrive by TMA
//     with 128-byte swizzle, directly in layouts the UMMA descriptors read
//     (Q in 64-column halves, K and V in row groups); each producer lane
//     issues one box; keys past the prefix read a zero-filled out-of-range
//     box;
//   * warp roles: warps 0-3 softmax of tile A, warps 4-7 softmax of tile B,
//     warp 8 issues the MMAs, warp 9 streams K and V in the order the MMAs
//     need them (K0, V0, K1, V1, ...: the TMA engine serves boxes in issue
//     order), with the prefix block ids loaded at kernel entry; hand-over is
//     by mbarriers and tcgen05.commit, never by a CTA-wide barrier;
//   * TMEM (512 columns): S_A, S_B, O_A, O_B.  The MMA order QK_A, QK_B,
//     then per key tile PV_A, QK_A(next), PV_B, QK_B(next) ping-pongs the
//     tiles, so one tile's softmax runs while the tensor pipe works on the
//     other's;
//   * P is rounded to bf16 into one shared swizzled K-major buffer, written
//     by A and B in turn once the previous PV has read it; V is consumed
//     MN-major (no transpose);
//   * the exponent base moves only when a row's max grows past 2^8 (exact);
//     the rare rescale of O is a TMEM load/multiply/store of that row;
//   * the softmax takes the row max on raw scores and feeds each
//     exponential with one FMA (scale and shift), masks only a split's last
//     tile, and sums on packed fp32 pairs;
//   * each warpgroup stages its normalised O tile in shared memory with the
//     128-byte swizzle, 32 columns at a time, and writes each 32-column plane
//     with a TMA store as soon as it is staged.
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kHalfBytes = kPrefixRows * 128;  // one 64-column half of a 128-row tile
constexpr int kPrefixThreads = 10 * 32;
constexpr int kPBytes = 2 * kHalfBytes;        // P: 128 rows x 128 keys bf16
constexpr int kPlaneBytes = kPrefixRows * 128;  // 32 fp32 columns of a 128-row O tile

__host__ __device__ constexpr int prefix_tile_bytes(int head_dim) {
  return (head_dim / 64) * kHalfBytes;
}

}  // namespace

size_t prefix_smem_bytes(int head_dim, int split_len, int block_size) {
  (void)split_len;
  (void)block_size;
  return (size_t)6 * prefix_tile_bytes(head_dim) + kPBytes + 1024;  // Q[2], K[2], V[2], P; +1024: alignment
}

template <int D, int G>
__global__ void __launch_bounds__(kPrefixThreads, 1)
    prefix_attention_kernel(const __grid_constant__ CUtensorMap tmq,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv,
                            const __grid_constant__ CUtensorMap tmo, const PrefixArgs a) {
  constexpr int H = D / 64;                  // 64-column halves of a row
  constexpr int RPB = kPrefixRows / G;       // requests per query tile
  constexpr uint32_t kTile = prefix_tile_bytes(D);
  constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kPrefixRows, kPrefixKeys, 0, 0);
  constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kPrefixRows, D, 0, 1);

  pdl_launch_dependents();  // the suffix decode may be scheduled as SMs free up
  const int kvh = blockIdx.z;
  const int P = a.block_size;
  // This CTA's keys and query rows: key split blockIdx.x of the one prefix
  // over the query-tile pair blockIdx.y, or item blockIdx.x of a chunk list.
  int split, ids_off, key0, nkeys, req0, nreq, st_req0;
  if (a.items) {
    const int4 w0 = __ldg(reinterpret_cast<const int4*>(a.items + blockIdx.x));
    const int4 w1 = __ldg(reinterpret_cast<const int4*>(a.items + blockIdx.x) + 1);
    ids_off = w0.x;
    key0 = w0.y;
    nkeys = w0.z;
    req0 = w0.w;
    nreq = w1.x;
    st_req0 = w1.y;
    split = w1.z;
  } else {
    split = blockIdx.x;
    ids_off = 0;
    key0 = split * a.split_len;
    nkeys = min(a.split_len, a.prefix_len - key0);
    req0 = 2 * (int)blockIdx.y * RPB;
    nreq = min(a.num_seqs - req0, 2 * RPB);
    st_req0 = req0;
  }
  if (nkeys <= 0 || nreq <= 0) return;
  const int J = (nkeys + kPrefixKeys - 1) / kPrefixKeys;
  const bool hasB = nreq > RPB;  // the pair's second query tile holds rows

  extern __shared__ unsigned char smem_raw[];
  // Align by offsetting the array itself (not through an integer), so the
  // compiler keeps every access in the shared state space.
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* qs = sm;                  // Q_A, Q_B
  unsigned char* ks = qs + 2 * kTile;      // two stages
  unsigned char* vs = ks + 2 * kTile;      // two stages
  unsigned char* ps = vs + 2 * kTile;      // 128 rows x 128 keys bf16 (two halves)
  // qbar[x]: Q of tile x by TMA; kfull/vfull: a producer filled a stage;
  // kfree/vfree: the MMAs that read a stage completed; sfull[x]: QK^T of tile
  // x done; pfull[x]: tile x's softmax wrote P; ofull[x]: PV of tile x done;
  // pfree: a PV read P.
  __shared__ uint64_t qbar[2], kfull[2], vfull[2], kfree[2], vfree[2], sfull[2], pfull[2],
      ofull[2], pfree;
  __shared__ uint32_t tmem_base;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // The producer's block ids: lane l issues box l of every tile (block l,
  // both column halves), K and V alike; the ids of tiles 0 and 1 are
  // requested before the set-up so their latency overlaps it.
  const int PB = P < kPrefixKeys ? P : kPrefixKeys;
  const int nbox = kPrefixKeys / PB;
  const int bsub = lane;
  constexpr int kGroupBytes = kRowGroup * H * 128;  // one 8-row group of a K/V tile
  constexpr int kZeroFill = INT_MIN;  // no key here: read a zero-filled out-of-range box
  auto box_block = [&](int jt) -> int2 {  // (block, first row) of this lane's box of tile jt
    const int key = key0 + jt * kPrefixKeys + bsub * PB;
    if (lane >= nbox || jt >= J || key >= key0 + nkeys) return make_int2(kZeroFill, 0);
    return make_int2(__ldg(a.prefix_block_ids + ids_off + key / P), key % P);
  };
  int2 box0 = make_int2(0, 0), box1 = make_int2(0, 0);
  if (warp == 9) {
    box0 = box_block(0);
    box1 = box_block(1);
  }
  if (t == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qbar[i], 1);
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&kfree[i], 1);
      mbar_init(&vfree[i], 1);
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], 4);
      mbar_init(&ofull[i], 1);
    }
    mbar_init(&pfree, 1);
    fence_barrier_init();
    // tile A's Q needs no block ids: start it before anything else (tile B's
    // follows the first K tile, from the producer)
    prefetch_tensormap(&tmq);
    mbar_arrive_expect_tx(&qbar[0], kTile);
#pragma unroll
    for (int h = 0; h < H; ++h)
      tma_load_3d(qs + h * kHalfBytes, &tmq, h * 64, kvh * G, req0, &qbar[0]);
  }
  __syncthreads();  // barriers initialised: the producer starts streaming now
  // Every warp but the producer waits for the TMEM allocation.
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  if (warp != 9) {
    tc::fence_before_sync();
    named_barrier_sync(3, kPrefixThreads - 32);
    tc::fence_after_sync();
  }
  const uint32_t tmem = tmem_base;  // S_A, S_B at columns 0, 128; O_A, O_B at 256, 384

  if (warp == 9) {
    // ============================================================ producer
    // K and V tiles in the order the MMAs consume them.  A tile is
    // kPrefixKeys / PB TMA boxes (PB rows of both column halves each), lane
    // l issuing box l.  A stage is refilled as soon as the MMAs
    // that read it have completed; keys past the split, and bad block ids
    // (reported), read a zero-filled out-of-range box.
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    __syncwarp();
    int2 bn = box1;  // tile jt + 1
    int blk = box0.x, row = box0.y;  // tile jt
    for (int jt = 0; jt < J; ++jt) {
      const int st = jt & 1;
      if (blk < 0 || (int64_t)blk >= a.num_blocks) {
        if (blk != kZeroFill) atomicOr(a.err, PKV_DEVERR_BLOCK);
        blk = (int)a.num_blocks;
        row = 0;
      }
      int ok = 1;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        uint64_t* fullb = kv ? vfull : kfull;
        if (lane == 0 && jt >= 2 && !mbar_wait(kv ? &vfree[st] : &kfree[st], ((jt - 2) >> 1) & 1)) {
          atomicOr(a.err, PKV_DEVERR_TIMEOUT);
          ok = 0;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        if (lane == 0) mbar_arrive_expect_tx(&fullb[st], kTile);
        __syncwarp();
        if (lane < nbox)
          tma_load_5d((kv ? vs : ks) + st * kTile + bsub * PB * H * 128, kv ? &tmv : &tmk, 0, 0,
                      0, kvh, (int)((int64_t)blk * (P / kRowGroup) + row / kRowGroup),
                      &fullb[st]);
        if (jt == 0 && kv == 0 && hasB && lane == 0) {  // tile B's Q, after the first K tile
          mbar_arrive_expect_tx(&qbar[1], kTile);
#pragma unroll
          for (int h = 0; h < H; ++h)
            tma_load_3d(qs + kTile + h * kHalfBytes, &tmq, h * 64, kvh * G, req0 + RPB,
                        &qbar[1]);
        }
      }
      if (!ok) break;
      blk = bn.x;
      row = bn.y;
      bn = box_block(jt + 2);
    }
  } else if (warp == 8) {
    // ============================================================ MMA issue
    if (lane == 0) {
      auto issue_qk = [&](int x, int jt) -> bool {
        if (jt == 0 && !mbar_wait(&qbar[x], 0)) return false;
        if (!mbar_wait(&kfull[jt & 1], (jt >> 1) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t kb = smem_u32(ks + (jt & 1) * kTile), qb = smem_u32(qs + x * kTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          // Q in 64-column halves (8-row groups 1 KiB apart), K in row groups
          tc::mma_bf16(tmem + x * 128,
                       tc::smem_desc_sw128(qb + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024),
                       tc::smem_desc_sw128(kb + (k >> 2) * 1024 + (k & 3) * 32, 16, kGroupBytes),
                       kIdQK, k > 0 ? 1u : 0u);
        }
        tc::commit(&sfull[x]);
        if (x == 1 || !hasB) tc::commit(&kfree[jt & 1]);
        return true;
      };
      auto issue_pv = [&](int x, int jt) -> bool {
        if (!mbar_wait(&pfull[x], jt & 1)) return false;
        if (x == 0 && !mbar_wait(&vfull[jt & 1], (jt >> 1) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t vb = smem_u32(vs + (jt & 1) * kTile), pb = smem_u32(ps);
#pragma unroll
        for (int k = 0; k < kPrefixKeys / 16; ++k) {
          const uint64_t ad =
              tc::smem_desc_sw128(pb + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
          // V is MN-major: 64-column d chunks 1 KiB apart, 8-key groups kGroupBytes apart
          const uint64_t bd = tc::smem_desc_sw128(vb + k * 2 * kGroupBytes, 1024, kGroupBytes);
          tc::mma_bf16(tmem + 256 + x * 128, ad, bd, kIdPV, (jt > 0 || k > 0) ? 1u : 0u);
        }
        tc::commit(&ofull[x]);
        tc::commit(&pfree);
        if (x == 1 || !hasB) tc::commit(&vfree[jt & 1]);
        return true;
      };
      bool ok = issue_qk(0, 0) && (!hasB || issue_qk(1, 0));
      for (int j = 0; j < J && ok; ++j) {
        ok = issue_pv(0, j) && (j + 1 >= J || issue_qk(0, j + 1));
        if (ok && hasB) ok = issue_pv(1, j) && (j + 1 >= J || issue_qk(1, j + 1));
      }
      if (!ok) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp < 4 || hasB) {
    // ============================================================ softmax rows
    const int x = warp >> 2;                 // query tile A (0) or B (1)
    const int row = (warp & 3) * 32 + lane;  // query row in the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + x * 128, tO = tmem + 256 + x * 128;
    const float c = a.qscale;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < J && ok; ++j) {
      if (!mbar_wait(&sfull[x], j & 1)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t r[kPrefixKeys];
#pragma unroll
      for (int c0 = 0; c0 < kPrefixKeys; c0 += 32)
        tc::tmem_ld32(tS + lane_base + c0, *reinterpret_cast<uint32_t(*)[32]>(r + c0));
      tc::wait_ld();
      const int kvalid = nkeys - j * kPrefixKeys;
      // Row max on the raw scores (the scale c > 0 commutes with max), with 8
      // independent accumulators; keys past the prefix (only in a split's
      // last tile) are masked to -inf.
      if (kvalid < kPrefixKeys) {
#pragma unroll
        for (int i = 0; i < kPrefixKeys; ++i)
          if (i >= kvalid) r[i] = __float_as_uint(-INFINITY);
      }
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = __uint_as_float(r[u]);
#pragma unroll
      for (int i = 8; i < kPrefixKeys; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(r[i]));
      const float mx = c * fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_run, mx);
      const bool need = m_new > m_run + 8.0f;
      const float alpha = need ? exp2f(m_run - m_new) : 1.f;
      if (need) m_run = m_new;
      // ---- P = exp2(c s - m) in bf16 pairs (registers until the buffer is
      // free); one FMA feeds each exponential, the sum runs on packed pairs
      uint32_t pw[kPrefixKeys / 2];
      float2 ls4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ls4[u] = make_float2(0.f, 0.f);
      const float nm = -m_run;
#pragma unroll
      for (int i = 0; i < kPrefixKeys / 2; ++i) {
        const float p0 = exp2f(fmaf(__uint_as_float(r[2 * i]), c, nm));
        const float p1 = exp2f(fmaf(__uint_as_float(r[2 * i + 1]), c, nm));
        ls4[i & 3] = __fadd2_rn(ls4[i & 3], make_float2(p0, p1));
        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
        pw[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      const float2 ls2 = __fadd2_rn(__fadd2_rn(ls4[0], ls4[1]), __fadd2_rn(ls4[2], ls4[3]));
      const float lsum = ls2.x + ls2.y;
      if (j > 0) {
        // PV of this tile's previous keys has completed: O is current
        if (!mbar_wait(&ofull[x], (j - 1) & 1)) { ok = false; break; }
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
      l_run = l_run * alpha + lsum;
      // ---- the P buffer is written A0, B0, A1, B1, ...: wait for the PV
      // that read the previous write
      const int w = 2 * j + x;
      if (w > 0 && (x == 1 || hasB || j > 0)) {
        const int prev = hasB ? w - 1 : j - 1;  // completions of pfree so far
        if (!mbar_wait(&pfree, prev & 1)) { ok = false; break; }
      }
      if (x == 0 && kvalid < kPrefixKeys) {
        // The split's last tile ends inside it.  Rows past the last key hold
        // a zero-filled box, or the stale rest of a chunk's last block: P is
        // 0 there, but 0 * NaN is not, so clear those V rows before the PVs
        // read the tile (tile A's PV is issued after this group's P).
        if (!mbar_wait(&vfull[j & 1], (j >> 1) & 1)) { ok = false; break; }
        if (row >= kvalid) {
#pragma unroll
          for (int h = 0; h < H; ++h) {
            uint4* vr = reinterpret_cast<uint4*>(vs + (j & 1) * kTile + (row / kRowGroup) * kGroupBytes +
                                                 h * 1024 + (row % kRowGroup) * 128);
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) vr[c16] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
#pragma unroll
      for (int ch = 0; ch < kPrefixKeys / 8; ++ch) {
        const int hf = ch >> 3, cc = ch & 7;
        uint4* dst =
            reinterpret_cast<uint4*>(ps + hf * kHalfBytes + row * 128 + ((cc ^ (row & 7)) << 4));
        *dst = make_uint4(pw[4 * ch], pw[4 * ch + 1], pw[4 * ch + 2], pw[4 * ch + 3]);
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[x]);
    }
    // ---- epilogue: O / l and the LSE of this row
    const bool done = ok && mbar_wait(&ofull[x], (J - 1) & 1);
    tc::fence_after_sync();
    if (!done && lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    const int rr = x * RPB + row / G;  // request of the pair
    const int g = row % G;
    const bool row_ok = done && rr < nreq;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const int64_t slot =
        ((int64_t)(st_req0 + rr) * a.num_q_heads + (int64_t)kvh * G + g) * a.parts_stride + split;
    // O row -> registers 32 columns at a time, scaled, into an idle stage
    // pair (tile A: the K stages, every QK^T has completed; tile B: the V
    // stages, its last PV has completed) as D / 32 planes of [128 rows][32
    // floats] with the 128-byte swizzle (16-byte chunk c of row t at
    // c ^ (t % 8)).  One thread stores each plane with TMA as soon as the
    // group has staged it, while the group stages the next (rows of requests
    // past the batch are clipped).  Every warp of the group takes this path,
    // so each group barrier always completes.
    unsigned char* stage = x == 0 ? ks : vs;
    const float sc = done ? inv : 0.f;
#pragma unroll
    for (int plane = 0; plane < D / 32; ++plane) {
      uint32_t v[32];
      tc::tmem_ld32(tO + lane_base + plane * 32, v);
      tc::wait_ld();
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<float4*>(stage + plane * kPlaneBytes + row * 128 +
                                   ((ch ^ (row & 7)) << 4)) =
            make_float4(__uint_as_float(v[4 * ch]) * sc, __uint_as_float(v[4 * ch + 1]) * sc,
                        __uint_as_float(v[4 * ch + 2]) * sc, __uint_as_float(v[4 * ch + 3]) * sc);
      tc::fence_proxy_async_smem();
      named_barrier_sync(1 + x, 128);
      if (row == 0) {
        tma_store_5d(&tmo, plane * 32, split, 0, kvh, st_req0 + x * RPB,
                     stage + plane * kPlaneBytes);
        bulk_commit_group();
      }
    }
    if (row == 0) bulk_wait_group_read0();
    if (row_ok) a.part_lse[slot] = l_run > 0.f ? (m_run + log2f(l_run)) * a.lse_scale : -INFINITY;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <int D, int G>
static cudaError_t launch_prefix_t(int num_splits, const CUtensorMap& tmq, const CUtensorMap& tmk,
                                   const CUtensorMap& tmv, const CUtensorMap& tmo,
                                   const PrefixArgs& a, cudaStream_t stream) {
  const size_t smem = prefix_smem_bytes(D, a.split_len, a.block_size);
  auto kern = prefix_attention_kernel<D, G>;
  static SmemAttrCache attr_cache;
  cudaError_t e = ensure_smem_limit(kern, (int)smem, attr_cache);
  if (e != cudaSuccess) return e;
  const int m_tiles = (a.num_seqs * G + kPrefixRows - 1) / kPrefixRows;
  const dim3 grid = a.items
                        ? dim3((unsigned)a.num_items, 1u, (unsigned)a.num_kv_heads)
                        : dim3((unsigned)num_splits, (unsigned)((m_tiles + 1) / 2),
                               (unsigned)a.num_kv_heads);
  kern<<<grid, kPrefixThreads, smem, stream>>>(tmq, tmk, tmv, tmo, a);
  return cudaGetLastError();
}

template <int D>
static cudaError_t dispatch_prefix_group(int group, int num_splits, const CUtensorMap& tmq,
                                         const CUtensorMap& tmk, const CUtensorMap& tmv,
                                         const CUtensorMap& tmo, const PrefixArgs& a,
                                         cudaStream_t stream) {
  switch (group) {
    case 1: return launch_prefix_t<D, 1>(num_splits, tmq, tmk, tmv, tmo, a, stream);
    case 2: return launch_prefix_t<D, 2>(num_splits, tmq, tmk, tmv, tmo, a, stream);
    case 4: return launch_prefix_t<D, 4>(num_splits, tmq, tmk, tmv, tmo, a, stream);
    case 8: return launch_prefix_t<D, 8>(num_splits, tmq, tmk, tmv, tmo, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefix_attention(int head_dim, int group, int num_splits,
                                    const CUtensorMap& tmq, const CUtensorMap& tmk,
                                    const CUtensorMap& tmv, const CUtensorMap& tmo,
                                    const PrefixArgs& a, cudaStream_t stream) {
  return head_dim == 128
             ? dispatch_prefix_group<128>(group, num_splits, tmq, tmk, tmv, tmo, a, stream)
             : dispatch_prefix_group<64>(group, num_splits, tmq, tmk, tmv, tmo, a, stream);
}

}  // namespace pkv
