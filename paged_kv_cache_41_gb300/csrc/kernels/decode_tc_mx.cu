// decode_tc_mx.cu -- paged attention decode on the tcgen05 tensor cores over
// MXFP8 pools (E4M3 elements, an E8M0 scale per 32 head_dim elements).
//
// What it computes: what decode.cu computes over an MXFP8 pool -- for
// sequence r and query head h, attention of q[r, h] (bf16) over the rows
// t < T_r of kv head h / G, element (t, c) = E4M3 code * 2^(s - 127) with s
// the scale byte of its 32-element group, cut into pieces whose (O, LSE)
// states the reduction merges by log-sum-exp ("M5.3 - KV Memory Layout and
// Exact Reuse", 0x0A, 0x0BA; quantized K/V as a cache-ABI field, 0x0BB).
//
// Design (GB300): the tensor cores take no E4M3 operand beside a bf16 one,
// and q and the weights must stay wider than E4M3, so each stage's E4M3
// tiles are widened to bf16 in shared memory -- exactly: an E4M3 value times
// a power of two is a bf16 value -- and then run through the MMAs of the
// bf16 tensor-core decode (decode_tc.cu):
//     S^T [128 keys x 16] = K_tile . Q^T,  O^T [128 d x 16] += V_tile^T . P^T
// with the G query heads zero-padded to N = 16 and P^T as two bf16 terms.
//   * warp 0 streams each stage's E4M3 K and V rows (one 128-byte-row TMA box
//     per block: half the boxes per row of the bf16 decode), their scale rows
//     (one bulk copy per box from the head-major scale plane) and a piece's Q
//     into one of two raw slots;
//   * warps 6-13 widen a raw slot into one of two bf16 K/V buffers (16 key
//     rows of K and of V per warp, written in the 128-byte swizzled layouts
//     the MMA descriptors expect, with lanes mapped so that neither the raw
//     loads nor the swizzled stores meet bank conflicts; rows past the tail
//     zeroed) with integer operations and one packed multiply per element
//     pair, and release the raw slot at once, so the copies run up to two
//     stages ahead of the widening; a K tile is widened as soon as the
//     softmax two stages back has read its scores, a V tile once that
//     stage's PV MMA has read its buffer, so K need not wait for the PV;
//   * warp 1 issues the MMAs; warps 2-5 run the online softmax, as in
//     decode_tc.cu.
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "plan.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kMxRows = 128;                       // key rows per stage = the QK MMA's M
constexpr int kMxN = 16;                           // query heads, zero-padded to the MMA's N
constexpr int kMxD = 128;                          // head_dim = the PV MMA's M
constexpr int kMxRaw = 2;                          // raw slots
constexpr int kWidenWarps = 8;                     // warps 6 .. 13
constexpr int kMxThreads = (6 + kWidenWarps) * 32;  // producer, MMA, 4 softmax, widening warps
constexpr int kRawTile = kMxRows * kMxD;           // 16 KiB: E4M3 rows of 128 bytes
constexpr int kRawScale = kMxRows * (kMxD / 32);   // 512 B: their scale rows
constexpr int kRawSlot = 2 * kRawTile + 2 * kRawScale;  // K, V, K scales, V scales
constexpr int kBfTile = kMxRows * kMxD * 2;        // 32 KiB: a bf16 tile, two 64-column halves
constexpr int kBfHalf = kMxRows * 128;             // 16 KiB
constexpr int kQB = kMxN * kMxD * 2;               // 4 KiB: Q (or P^T), 16 rows x 128
constexpr int kQH = kMxN * 128;                    // 2 KiB: 64 columns of it
constexpr int kQBufsMx = 3;                        // Q buffers (see decode_tc.cu)
constexpr int kMxSmem = 2 * 2 * kBfTile + kMxRaw * kRawSlot + (kQBufsMx + 2) * kQB + 1024;
constexpr float kLn2m = 0.6931471805599453f;

// Stage descriptor flags (as in decode_tc.cu); bits 4-5 hold the Q buffer.
constexpr int kStart = 1, kEnd = 2, kWholeSeg = 4, kSlotOne = 8;

// Eight E4M3 codes (two words) times 2^(s - 127), as eight bf16 values in a
// uint4, with integer operations and packed bf16 multiplies only.  A code
// s.eeee.mmm placed as bf16 bits s at 15 and eeeemmm at 10..4 reads as the
// E4M3 value times 2^-120 -- normal codes with exponent field e, subnormal
// codes as the bf16 subnormal m/8 2^-126, zero as zero -- so multiplying by
// 2^(s - 7) gives the scaled value: exact, as the product keeps at most four
// significant bits (values below bf16's smallest subnormal aside).  2^(s-7)
// can pass bf16's range (s > 134), so it is applied as 2^a (a <= 127), then,
// in the warps that need it, 2^(s - 7 - a).
__device__ __forceinline__ uint32_t place2(uint32_t pair) {  // bytes in halves -> bf16x2 bits
  // s.eeee.mmm -> s at 15, eeeemmm at 10..4: pair * 16 + sign * 240 (no carries)
  return (pair & 0x00800080u) * 240u + (pair << 4);
}

__device__ __forceinline__ uint4 widen8(uint2 w, __nv_bfloat162 s1, __nv_bfloat162 s2, bool big) {
  uint32_t out[4];
  const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t lo = place2(__byte_perm(ws[i], 0u, 0x4140u));  // bytes 0, 1
    const uint32_t hi = place2(__byte_perm(ws[i], 0u, 0x4342u));  // bytes 2, 3
    __nv_bfloat162 vlo = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&lo), s1);
    __nv_bfloat162 vhi = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&hi), s1);
    if (big) {
      vlo = __hmul2(vlo, s2);
      vhi = __hmul2(vhi, s2);
    }
    out[2 * i] = *reinterpret_cast<const uint32_t*>(&vlo);
    out[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&vhi);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// The two bf16x2 factors for scale byte g of the word sc: 2^a with a =
// min(s - 7, 127), and 2^(s - 7 - a) = 2^max(s - 134, 0).  (Byte g picked by
// a permute, as g varies with the thread.)
__device__ __forceinline__ void scale_factors(uint32_t sc, int g, __nv_bfloat162& s1,
                                              __nv_bfloat162& s2) {
  const uint32_t s = __byte_perm(sc, 0u, 0x4440u | (uint32_t)g);
  const uint32_t m = s < 134u ? s : 134u;
  const uint32_t w1 = m * 0x00800080u + 0x3C003C00u;               // exponent field m + 120
  const uint32_t w2 = (s - m) * 0x00800080u + 0x3F803F80u;         // exponent field s - m + 127
  s1 = *reinterpret_cast<const __nv_bfloat162*>(&w1);
  s2 = *reinterpret_cast<const __nv_bfloat162*>(&w2);
}

}  // namespace

template <int G>
__global__ void __launch_bounds__(kMxThreads, 1)
    decode_tc_mx_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ CUtensorMap tmq, const DecodeArgs a) {
  static_assert(G <= kMxN, "at most 16 query heads per kv head");
  constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kMxRows, kMxN, 0, 0);
  constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kMxD, kMxN, 1, 0);
  // full[r]: raw slot r's copies (and Q) landed; rfree[r]: slot r widened;
  // kready[b] / vready[b]: the K / V tile of bf16 buffer b widened;
  // vfree[b]: the PV MMA that read V completed (K is free once the softmax
  // has read the scores, sfree[b]: the QK MMA completed before, and the
  // softmax waited for kready[b] before, so kready never runs two phases
  // ahead of a waiter)
  // completed; sfull/sfree, pfull, ofull, ofree, rsync as in decode_tc.cu.
  __shared__ uint64_t full[kMxRaw], rfree[kMxRaw], kready[2], vready[2], vfree[2],
      sfull[2], sfree[2], pfull,
      ofull, ofree, rsync;
  // a stage's descriptor, by stage mod 4: stage k + 4 is widened only after
  // QK(k + 2), which waits for the softmax of stage k to have read its own
  __shared__ int4 sdesc_raw[kMxRaw], sdesc_bf[4];
  __shared__ float redm[2][4][kMxN], redl[4][kMxN];
  __shared__ int4 redf[2];  // per stage parity: each softmax warp's "a score passed m + 8"
  __shared__ long long wsum[2 * (kMxThreads / 32) + 4];
  __shared__ uint32_t tmem_base;

  const int c = blockIdx.x;
  if (!a.plan_before_wait) pdl_wait();  // inputs written by earlier kernels are visible
  pdl_launch_dependents();  // the reduction may be scheduled as CTAs retire
  int4 d0;
  const int n = plan_cta_stages<kMxThreads, kMxRows>(a, wsum, &d0);
  if (a.plan_before_wait) pdl_wait();
  if (n <= 0) return;  // no stages: the whole CTA leaves before any barrier
  const int Hkv = a.num_kv_heads, P = a.block_size;
  const int TB = P < kMxRows ? P : kMxRows;  // rows per TMA box

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* bf = sm;                           // [2][bf16 K tile, bf16 V tile]
  unsigned char* raw = bf + 2 * 2 * kBfTile;        // [kMxRaw][K, V, K scales, V scales]
  unsigned char* qs = raw + kMxRaw * kRawSlot;      // Q[kQBufsMx]
  unsigned char* pt = qs + kQBufsMx * kQB;          // P^T: hi term, then lo term

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // rows G..15 of Q and P^T stay zero: the padding of the MMA's N
  for (int i = t; i < (kQBufsMx + 2) * kQB / 16; i += kMxThreads)
    reinterpret_cast<uint4*>(qs)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (t == 0) {
    for (int s = 0; s < kMxRaw; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&rfree[s], kWidenWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kready[b], kWidenWarps);
      mbar_init(&vready[b], kWidenWarps);
      mbar_init(&vfree[b], 1);
      mbar_init(&sfull[b], 1);
      mbar_init(&sfree[b], 4);
    }
    mbar_init(&pfull, 4);
    mbar_init(&ofull, 1);
    mbar_init(&ofree, 4);
    mbar_init(&rsync, 128);
    fence_barrier_init();
  }
  tc::fence_proxy_async_smem();  // the zero padding is visible to the tensor cores
  if (warp == 0) tc::tmem_alloc(&tmem_base, 64);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;  // S^T buffers at columns 0 and 16, O^T at 32
  int issued = 0;                   // stages whose copies warp 0 started

  if (warp == 0) {
    // ============================================================ producer
    // Stage k of the CTA fills raw slot k % 2: boxes of TB 128-byte E4M3
    // rows (lanes 0..7 K, 16..23 V) and their scale rows (lanes 8..15 K,
    // 24..31 V), one per block (or 128-row slice), and a piece's Q.
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      prefetch_tensormap(&tmq);
    }
    int r = d0.x, h = d0.y, i = d0.z;
    int len = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
    int nt = (len + kMxRows - 1) / kMxRows;
    while (i >= nt) {  // the plan may name a segment's end: its next non-empty one
      i -= nt;
      if (++h == Hkv) {
        h = 0;
        do {
          ++r;
          len = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
          nt = (len + kMxRows - 1) / kMxRows;
        } while (nt == 0);
      }
    }
    int pieces = 0;
    const int j = lane & 7, kind = lane >> 3;  // kind: 0 K rows, 1 K scales, 2 V rows, 3 V scales
    for (int k = 0; k < n; ++k) {
      const int s = k % kMxRaw;
      if (k >= kMxRaw) {
        int ok = 1;
        if (lane == 0 && !mbar_wait(&rfree[s], ((k / kMxRaw) - 1) & 1)) {
          atomicOr(a.err, PKV_DEVERR_TIMEOUT);
          ok = 0;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      const int t0 = i * kMxRows;
      const int nvalid = min(kMxRows, len - t0);
      const int dseg = k - i;  // CTA stage index of the segment's first stage
      const bool start = k == 0 || i == 0;
      const bool end = k == n - 1 || i == nt - 1;
      if (start) ++pieces;
      const int qb = (pieces - 1) % kQBufsMx;
      const int flags = (start ? kStart : 0) | (end ? kEnd : 0) |
                        (end && i == nt - 1 && dseg >= 0 ? kWholeSeg : 0) |
                        (dseg > 0 ? kSlotOne : 0) | (qb << 4);
      const int nbox = (nvalid + TB - 1) / TB;  // per tensor, <= 8
      int blk = 0, brow = 0;
      if (j < nbox) {
        const int row = t0 + j * TB;
        const int bi = row / P;
        brow = row - bi * P;
        blk = __ldg(a.block_tables + (int64_t)r * a.max_blocks + bi);
      }
      const bool bad = j < nbox && (blk < 0 || (int64_t)blk >= a.num_blocks);
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.err, PKV_DEVERR_BLOCK);
      if (lane == 0) {
        sdesc_raw[s] = make_int4(r, h, nvalid, flags);
        mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * nbox * TB * (kMxD + kMxD / 32) +
                                                    (start ? 2 * G * 128 : 0)));
      }
      __syncwarp();
      if (j < nbox) {
        unsigned char* slot = raw + (size_t)s * kRawSlot;
        if (kind == 0 || kind == 2) {
          // a bad block id reads a zero-filled out-of-range box
          tma_load_4d(slot + (kind ? kRawTile : 0) + j * TB * kMxD, kind ? &tmv : &tmk, 0, h,
                      bad ? 0 : brow, bad ? (int)a.num_blocks : blk, &full[s]);
        } else {
          // scale rows of the same box; a bad block copies block 0's (its
          // rows are zero-filled and the error bit is set)
          const int64_t sb = bad ? 0 : blk;
          const uint8_t* src = (kind == 3 ? a.v_scales : a.k_scales) +
                               ((sb * Hkv + h) * P + (bad ? 0 : brow)) * (kMxD / 32);
          bulk_load(slot + 2 * kRawTile + (kind == 3 ? kRawScale : 0) + j * TB * (kMxD / 32), src,
                    (uint32_t)(TB * (kMxD / 32)), &full[s]);
        }
      }
      if (start && lane == 0) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(qs + qb * kQB + hf * kQH, &tmq, hf * 64, h * G,
                      a.q_rows ? __ldg(a.q_rows + r) : r, &full[s]);
      }
      issued = k + 1;
      if (k + 1 < n && ++i == nt) {  // on to the next non-empty segment
        i = 0;
        if (++h == Hkv) {
          h = 0;
          do {
            ++r;
            len = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
            nt = (len + kMxRows - 1) / kMxRows;
          } while (nt == 0);
        }
      }
    }
  } else if (warp >= 6) {
    // ============================================================ widening
    // Raw slot k % 2 into bf16 buffer k % 2.  A bf16 row is two 64-column
    // halves of 128 bytes, each 16-byte column j of half h holding chunk
    // c = j ^ row % 8 of that half (the 128-byte swizzle the MMA descriptors
    // expect: K-major for K, MN-major for V); chunk c is 8 elements, 8 raw
    // bytes.  Each step a warp widens 4 rows x 8 columns: lane l takes row
    // (l / 8) and the column j = l % 8, so the 8 lanes of a row store to 8
    // bank groups, and odd rows take the other half first, so the 16 lanes of
    // two rows load from 16 distinct bank pairs.  Rows past the tail are
    // zeroed (their weight is 0, and 0 * NaN is not).
    constexpr int kRowsW = kMxRows / kWidenWarps;  // rows per warp
    const int wrow0 = (warp - 6) * kRowsW, rsub = lane >> 3, col = lane & 7;
    for (int k = 0; k < n; ++k) {
      const int s = k % kMxRaw, b = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / kMxRaw) & 1))) {
        if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        break;
      }
      const int4 dsc = sdesc_raw[s];
      const unsigned char* slot = raw + (size_t)s * kRawSlot;
      bool ok = true;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        // K of stage k waits for the softmax of stage k - 2 to have read its
        // scores (so QK(k - 2) is done), V for PV(k - 2)
        if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(kv ? &vfree[b] : &sfree[b], ((k - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        const unsigned char* src = slot + (kv ? kRawTile : 0);
        const unsigned char* scl = slot + 2 * kRawTile + (kv ? kRawScale : 0);
        unsigned char* dst = bf + (size_t)b * 2 * kBfTile + (kv ? kBfTile : 0);
        // lane i holds the scale word of row wrow0 + i (i < kRowsW); a scale
        // past 2^7 on any valid row of the warp takes the second multiply
        const int mrow = wrow0 + (lane < kRowsW ? lane : 0);
        const uint32_t scw = *reinterpret_cast<const uint32_t*>(scl + mrow * 4);
        const bool big = __any_sync(0xffffffffu, lane < kRowsW && mrow < dsc.z &&
                                                     ((scw & 0xffu) > 134u || ((scw >> 8) & 0xffu) > 134u ||
                                                      ((scw >> 16) & 0xffu) > 134u || (scw >> 24) > 134u));
#pragma unroll
        for (int it = 0; it < kRowsW / 2; ++it) {
          const int rr = (it >> 1) * 4 + rsub;  // row within the warp's
          const int row = wrow0 + rr;
          const uint32_t sc = __shfl_sync(0xffffffffu, scw, rr);
          const int h = (it & 1) ^ (rsub & 1);
          unsigned char* d = dst + h * kBfHalf + row * 128 + col * 16;
          if (row < dsc.z) {
            const int ch = h * 8 + (col ^ (row & 7));  // chunk of the row
            const uint2 w = *reinterpret_cast<const uint2*>(src + row * kMxD + ch * 8);
            __nv_bfloat162 f1, f2;
            scale_factors(sc, ch >> 2, f1, f2);
            *reinterpret_cast<uint4*>(d) = widen8(w, f1, f2, big);
          } else {
            *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        if (kv == 0 && warp == 6 && lane == 0) sdesc_bf[k & 3] = dsc;
        tc::fence_proxy_async_smem();  // the widened tile is visible to the tensor cores
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(kv ? &vready[b] : &kready[b]);
          if (kv) mbar_arrive(&rfree[s]);
        }
      }
      if (!ok) {
        if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        break;
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issue
    if (lane == 0) {
      bool ok = true;
      int pflags = 0, pieces_done = 0;
      auto issue_pv = [&](int jj, int fl) -> bool {
        if (!mbar_wait(&pfull, jj & 1) || !mbar_wait(&vready[jj & 1], (jj >> 1) & 1)) return false;
        if ((fl & kStart) && pieces_done > 0 && !mbar_wait(&ofree, (pieces_done - 1) & 1))
          return false;
        tc::fence_after_sync();
        const uint32_t vb = smem_u32(bf + (size_t)(jj & 1) * 2 * kBfTile + kBfTile);
#pragma unroll
        for (int term = 0; term < 2; ++term) {
          const uint32_t pb = smem_u32(pt + term * kQB);
#pragma unroll
          for (int kk = 0; kk < kMxRows / 16; ++kk) {
            const uint64_t ad = tc::smem_desc_sw128(vb + kk * 2048, kBfHalf, 1024);
            const uint64_t bd = tc::smem_desc_sw128(pb + (kk >> 2) * kQH + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16(tmem + 32, ad, bd, kIdPV,
                         (term > 0 || kk > 0 || !(fl & kStart)) ? 1u : 0u);
          }
        }
        tc::commit(&ofull);
        tc::commit(&vfree[jj & 1]);
        if (fl & kEnd) ++pieces_done;
        return true;
      };
      for (int k = 0; k < n; ++k) {
        const int b = k & 1;
        if (!mbar_wait(&kready[b], (k >> 1) & 1) ||
            (k >= 2 && !mbar_wait(&sfree[b], ((k - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const int fl = sdesc_bf[k & 3].w;
        const uint32_t kb = smem_u32(bf + (size_t)b * 2 * kBfTile);
        const uint32_t qb = smem_u32(qs + ((fl >> 4) & 3) * kQB);
#pragma unroll
        for (int kk = 0; kk < kMxD / 16; ++kk) {
          const uint64_t ad = tc::smem_desc_sw128(kb + (kk >> 2) * kBfHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(qb + (kk >> 2) * kQH + (kk & 3) * 32, 16, 1024);
          tc::mma_bf16(tmem + 16 * b, ad, bd, kIdQK, kk > 0 ? 1u : 0u);
        }
        tc::commit(&sfull[b]);
        if (k >= 1 && !issue_pv(k - 1, pflags)) {
          ok = false;
          break;
        }
        pflags = fl;
      }
      if (ok) ok = issue_pv(n - 1, pflags);
      if (!ok) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
    }
  } else {
    // ============================================================ softmax
    const int q4 = warp & 3;              // TMEM lane quarter of this warp
    const int row = q4 * 32 + lane;       // key row of S^T, head_dim row of O^T
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const float cs = a.qscale;
    float m[G], lp[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      lp[g] = 0.f;
    }
    uint32_t rs = 0;
    auto group_sync = [&]() -> bool {
      mbar_arrive(&rsync);
      const bool okw = __all_sync(0xffffffffu, mbar_wait(&rsync, rs & 1u));
      ++rs;
      if (!okw && lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
      return okw;
    };
    for (int k = 0; k < n; ++k) {
      const int b = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&kready[b], (k >> 1) & 1)) ||
          !__all_sync(0xffffffffu, mbar_wait(&sfull[b], (k >> 1) & 1))) {
        if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        break;
      }
      tc::fence_after_sync();
      const int4 dsc = sdesc_bf[k & 3];
      const int nvalid = dsc.z, flags = dsc.w;
      if (flags & kStart) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          m[g] = -INFINITY;
          lp[g] = 0.f;
        }
      }
      uint32_t v[16];
      tc::tmem_ld16(tmem + 16 * b + lane_base, v);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[b]);
      // the four warps agree on whether any score passes its head's base
      // by 2^8 before taking the per-head max (as in decode_tc.cu)
      float sg[G];
      bool pass = false;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        sg[g] = row < nvalid ? __uint_as_float(v[g]) * cs : -INFINITY;
        pass |= sg[g] > m[g] + 8.0f;
      }
      const bool wpass = __any_sync(0xffffffffu, pass);
      if (lane == 0) reinterpret_cast<int*>(&redf[b])[q4] = wpass ? 1 : 0;
      if (!group_sync()) break;
      const int4 fl = redf[b];
      bool any = false;
      float alpha[G], p[G];
#pragma unroll
      for (int g = 0; g < G; ++g) alpha[g] = 1.f;
      if (fl.x | fl.y | fl.z | fl.w) {  // the same for all four warps
        float mx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = sg[g];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], o));
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (lane == g) redm[b][q4][g] = mx[g];
        if (!group_sync()) break;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float mt = fmaxf(fmaxf(redm[b][0][g], redm[b][1][g]), fmaxf(redm[b][2][g], redm[b][3][g]));
          const float mn = fmaxf(m[g], mt);
          const bool need = mn > m[g] + 8.0f;
          alpha[g] = need ? exp2f(m[g] - mn) : 1.f;
          if (need) {
            m[g] = mn;
            any = true;
          }
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        p[g] = exp2f(sg[g] - m[g]);
        lp[g] = lp[g] * alpha[g] + p[g];
      }
      if (k >= 1) {
        if (!__all_sync(0xffffffffu, mbar_wait(&ofull, (k - 1) & 1))) {
          if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
        if (any && !(flags & kStart)) {
          uint32_t o[16];
          tc::tmem_ld16(tmem + 32 + lane_base, o);
          tc::wait_ld();
#pragma unroll
          for (int g = 0; g < G; ++g) o[g] = __float_as_uint(__uint_as_float(o[g]) * alpha[g]);
          tc::tmem_st16(tmem + 32 + lane_base, o);
          tc::wait_st();
        }
      }
      {  // P^T[g][row] as two bf16 terms (see decode_tc.cu)
        const int hf = row >> 6, cch = (row & 63) >> 3, e = row & 7;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const __nv_bfloat16 hi = __float2bfloat16_rn(p[g]);
          const __nv_bfloat16 lo = __float2bfloat16_rn(p[g] - __bfloat162float(hi));
          unsigned char* at = pt + hf * kQH + g * 128 + ((cch ^ (g & 7)) << 4) + e * 2;
          *reinterpret_cast<__nv_bfloat16*>(at) = hi;
          *reinterpret_cast<__nv_bfloat16*>(at + kQB) = lo;
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull);
      if (flags & kEnd) {
        if (!__all_sync(0xffffffffu, mbar_wait(&ofull, k & 1))) {
          if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
        uint32_t o[16];
        tc::tmem_ld16(tmem + 32 + lane_base, o);
        tc::wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ofree);
        float ls[G];
#pragma unroll
        for (int g = 0; g < G; ++g) ls[g] = lp[g];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) ls[g] += __shfl_xor_sync(0xffffffffu, ls[g], off);
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (lane == g) redl[q4][g] = ls[g];
        if (!group_sync()) break;
        const int64_t rh0 = (int64_t)dsc.x * a.num_q_heads + (int64_t)dsc.y * G;
        const int64_t rec = 2 * (int64_t)c + ((flags & kSlotOne) ? 1 : 0);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float L = (redl[0][g] + redl[1][g]) + (redl[2][g] + redl[3][g]);
          const bool nonempty = L > 0.f;
          const float ov = nonempty ? __uint_as_float(o[g]) / L : 0.f;
          const float lse2 = nonempty ? m[g] + log2f(L) : -INFINITY;
          if (!(flags & kWholeSeg)) {
            a.rec_o[(rec * G + g) * kMxD + row] = ov;
            if (row == 0) a.rec_lse[rec * G + g] = lse2;
          } else if (a.st_o) {
            const int64_t slot = (rh0 + g) * a.st_stride + a.st_slot;
            a.st_o[slot * kMxD + row] = ov;
            if (row == 0) a.st_lse[slot] = lse2;
          } else {
            store_out(static_cast<__nv_bfloat16*>(a.out) + (rh0 + g) * kMxD + row, ov);
            if (row == 0 && a.lse_out) a.lse_out[rh0 + g] = lse2 * kLn2m;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (t == 0) {
    // if anything left early, copies may still be in flight into the raw
    // slots: wait for them (bounded) before the CTA's shared memory is released
    for (int kk = issued > kMxRaw ? issued - kMxRaw : 0; kk < issued; ++kk)
      mbar_wait(&full[kk % kMxRaw], (kk / kMxRaw) & 1);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

// Eight query heads per kv head only: with four or fewer the CUDA-core
// decode reads MXFP8 pools faster than this kernel widens them.
bool decode_tc_mx_supported(int dtype, int head_dim, int group, int block_size) {
  return dtype == PKV_MXFP8 && head_dim == kMxD && group == 8 &&
         (kMxRows % block_size == 0 || block_size % kMxRows == 0);
}

template <int G>
static cudaError_t launch_mx_t(const CUtensorMap& tmk, const CUtensorMap& tmv,
                               const CUtensorMap& tmq, const DecodeArgs& a, cudaStream_t stream) {
  auto kern = decode_tc_mx_kernel<G>;
  static SmemAttrCache attr_cache;
  cudaError_t e = ensure_smem_limit(kern, kMxSmem, attr_cache);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)a.num_ctas), dim3(kMxThreads), kMxSmem, stream, tmk, tmv,
                    tmq, a);
}

int decode_tc_mx_resident_ctas() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    auto kern = decode_tc_mx_kernel<8>;
    int per_sm = 0, sms = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMxThreads, kMxSmem) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    cached[dev] = per_sm * sms;
  }
  return cached[dev];
}

cudaError_t launch_paged_decode_tc_mx(int group, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                      const CUtensorMap& tmq, const DecodeArgs& a,
                                      cudaStream_t stream) {
  cudaError_t e;
  switch (group) {
    case 8: e = launch_mx_t<8>(tmk, tmv, tmq, a, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_decode_reduce(PKV_MXFP8, kMxD, a, stream);
}

}  // namespace pkv
