// decode_tc.cu -- paged attention decode on the tcgen05 tensor cores for GQA
// groups of eight query heads per kv head (bf16, head_dim 128).
//
// What it computes ("M5.3 - KV Memory Layout and Exact Reuse", 0x0A and
// 0x0BA): exactly what decode.cu computes -- for sequence r and query head h,
// attention of q[r, h] over the rows t < T_r of kv head h / G found through
// the block table, cut into pieces whose (O, LSE) states are merged by
// log-sum-exp.
//
// Design (GB300):
//   * with eight query heads per kv head, the CUDA-core decode spends eight
//     FMA pairs per K/V element and is bound by its instruction stream; here
//     both products are MMAs in transposed form, so the key rows fill the
//     MMA's M = 128 and the eight heads (zero-padded to N = 16) its N:
//         S^T [128 keys x 16]  = K_tile [128 x 128] . Q^T
//         O^T [128 d    x 16] += V_tile^T . P^T    (V consumed MN-major)
//     with bf16 operands, fp32 accumulators in TMEM (S^T double-buffered);
//     P^T goes in as two bf16 terms, hi + lo, so the weights keep about 16
//     bits (two PV MMAs per stage: the tensor pipe has room to spare);
//   * the work split, the pieces and their records are those of decode.cu
//     with 128-row stages: one persistent CTA per SM takes an equal share of
//     the stages of every (sequence, kv head) segment, writes whole segments
//     directly and leaves one (O, LSE) record per cut piece, and the same
//     reduction kernel merges them;
//   * warp 0 streams each stage's K and V boxes by TMA (128-byte swizzle,
//     row-group tiles of launch.h: one box brings a whole block, or a
//     128-row slice of a larger one, both column halves; one box per lane)
//     and a piece's Q rows at its first stage, K one stage ahead of V (a K
//     slot is refilled once its QK has run, a V slot once its PV has, on
//     separate K and V barriers); warp 1 issues the MMAs; warps
//     2-5 own one key row (S^T lane) and one head_dim row (O^T lane) each and
//     run the online softmax: a four-warp vote on whether any score passes
//     its head's base by 2^8 (then per-head maxima across the 128 keys by
//     warp shuffles and a four-warp exchange), exp2 on each thread's 8 scores,
//     P^T written in bf16 into the swizzled K-major layout;
//   * the exponent base of a head moves only when its running max grows by
//     more than 2^8 (exact); the rare rescale of O^T is a TMEM
//     load/multiply/store of each thread's row;
//   * rows past a request's tail are masked out of the softmax and their V
//     rows zeroed in shared memory before the PV MMA, so stale or NaN bytes
//     of a recycled block never reach the output (M5.3 0x03G).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "plan.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kTcRows = 128;                  // key rows per stage = the QK MMA's M
constexpr int kTcN = 16;                      // query heads, zero-padded to the MMA's N
constexpr int kTcD = 128;                     // head_dim = the PV MMA's M
constexpr int kTcStages = 3;
constexpr int kTcThreads = 6 * 32;            // producer, MMA, four softmax warps
constexpr int kTcTile = kTcRows * kTcD * 2;   // 32 KiB: one K (or V) tile
constexpr int kTcGroup = kRowGroup * kTcD * 2;  // 2 KiB: one 8-row group, both halves
constexpr int kQBytes = kTcN * kTcD * 2;      // 4 KiB: Q (or P^T) as 16 rows x 128
constexpr int kQHalf = kTcN * 128;            // 2 KiB: 64 columns of it
// Q buffers, one per piece in turn.  A piece's Q is loaded with its first
// stage; with kTcStages ring stages the producer runs at most that many
// stages ahead, and a third piece after p starts at least three stages after
// p's last one, once the ring wait has seen p's last QK complete.  Two
// buffers would let a CTA's third stage overwrite its first piece's Q before
// that piece's QK has run.
constexpr int kQBufs = 3;
// Q[kQBufs], then P^T as two bf16 terms (hi, lo)
constexpr int kTcSmem = kTcStages * 2 * kTcTile + (kQBufs + 2) * kQBytes + 1024;  // +1024: alignment
constexpr float kLn2f = 0.6931471805599453f;

// Stage descriptor flags (as in decode.cu); bits 4-5 hold the Q buffer.
constexpr int kStart = 1, kEnd = 2, kWholeSeg = 4, kSlotOne = 8;

}  // namespace

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmq, const DecodeArgs a) {
  static_assert(G <= kTcN, "at most 16 query heads per kv head");
  constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kTcRows, kTcN, 0, 0);
  constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kTcD, kTcN, 1, 0);
  // kfull/kfree: a stage's K (and Q) landed / its QK completed; dfree: the
  // softmax warps read its descriptor (so the slot's next K may go out
  // without a softmax warp yet to wait for this phase); vfull/vfree: its V
  // landed / its PV completed; sfull/sfree: S^T buffer written / read;
  // pfull: P^T written; ofull: a PV completed; ofree: a piece's epilogue read
  // O^T; rsync: exchange among the softmax warps.
  __shared__ uint64_t kfull[kTcStages], kfree[kTcStages], dfree[kTcStages], vfull[kTcStages],
      vfree[kTcStages], sfull[2], sfree[2], pfull, ofull, ofree, rsync;
  __shared__ int4 sdesc[kTcStages];
  __shared__ float redm[2][4][kTcN], redl[4][kTcN];
  __shared__ int4 redf[2];  // per stage parity: each softmax warp's "a score passed m + 8"
  __shared__ long long wsum[2 * (kTcThreads / 32) + 4];
  __shared__ uint32_t tmem_base;

  const int c = blockIdx.x;
  if (!a.plan_before_wait) pdl_wait();  // inputs written by earlier kernels are visible
  pdl_launch_dependents();  // the reduction may be scheduled as CTAs retire
  int4 d0;
  const int n = plan_cta_stages<kTcThreads, kTcRows>(a, wsum, &d0);
  if (n <= 0) return;  // no stages: the whole CTA leaves before any barrier
  const int Hkv = a.num_kv_heads, P = a.block_size;
  const int TB = P < kTcRows ? P : kTcRows;  // rows per TMA box

  extern __shared__ unsigned char smem_raw[];
  // Align by offsetting the array itself, so accesses stay in shared space.
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* ring = sm;                            // [stage][K tile, V tile]
  unsigned char* qs = ring + kTcStages * 2 * kTcTile;  // Q[kQBufs], one per piece in turn
  unsigned char* pt = qs + kQBufs * kQBytes;           // P^T: hi term, then lo term

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // rows G..15 of Q and P^T stay zero: the padding of the MMA's N
  for (int i = t; i < (kQBufs + 2) * kQBytes / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(qs)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (t == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kfree[s], 1);
      mbar_init(&dfree[s], 4);
      mbar_init(&vfull[s], 1);
      mbar_init(&vfree[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
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
  // With plan_before_wait, what the preceding kernel may still write is read
  // only after the wait: the producer's first block ids come before it.
  if (a.plan_before_wait && warp != 0) pdl_wait();
  int issued_k = 0, issued_v = 0;   // stages whose K / V copies warp 0 started

  if (warp == 0) {
    // ============================================================ producer
    // Walks the CTA's stages (r, h, i) = (sequence, kv head, stage in the
    // segment).  A stage is nbk blocks (or a 128-row slice of a larger one)
    // of TMA boxes per tensor, both column halves in each: lanes 0..7 issue
    // K boxes, lanes 16..23 V boxes, each fetching its own block id.  K runs
    // one stage ahead of V: a K slot is free once its QK has run, a V slot
    // only once its PV has, so stage k's K boxes go out before stage k - 1's
    // V boxes (and the QK and softmax of a stage overlap its V's landing).
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
      prefetch_tensormap(&tmq);
    }
    int r = d0.x, h = d0.y, i = d0.z;
    int len = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
    int nt = (len + kTcRows - 1) / kTcRows;
    while (i >= nt) {  // the plan may name a segment's end: its next non-empty one
      i -= nt;
      if (++h == Hkv) {
        h = 0;
        do {
          ++r;
          len = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
          nt = (len + kTcRows - 1) / kTcRows;
        } while (nt == 0);
      }
    }
    // block id of this lane's box in the stage at row i * kTcRows of
    // sequence r (0 where the lane has no box), loaded one stage ahead: the
    // table read then overlaps the wait for a free slot
    const int j = lane & 15;
    auto box_block = [&](int r_, int i_, int len_) -> int {
      const int row = i_ * kTcRows + j * TB;
      return row < len_ && j * TB < kTcRows
                 ? __ldg(a.block_tables + (int64_t)r_ * a.max_blocks + row / P)
                 : 0;
    };
    int blk_next = box_block(r, i, len);
    if (a.plan_before_wait) pdl_wait();  // the K/V rows and q are read from here on
    int pieces = 0;
    // the previous stage's V boxes: this lane's block and first row, the box
    // count and the kv head
    int v_blk = 0, v_brow = 0, v_nbox = 0, v_h = 0;
    auto issue_v = [&](int kv) -> bool {
      const int sv = kv % kTcStages;
      if (kv >= kTcStages) {
        int ok = 1;
        if (lane == 0 && !mbar_wait(&vfree[sv], ((kv / kTcStages) - 1) & 1)) {
          atomicOr(a.err, PKV_DEVERR_TIMEOUT);
          ok = 0;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      }
      if (lane == 0) mbar_arrive_expect_tx(&vfull[sv], (uint32_t)(v_nbox * TB * kTcD * 2));
      __syncwarp();
      if (lane >= 16 && j < v_nbox)
        tma_load_5d(ring + (size_t)sv * 2 * kTcTile + kTcTile + j * TB * kTcD * 2, &tmv, 0, 0, 0, v_h,
                    (int)((int64_t)v_blk * (P / kRowGroup) + v_brow / kRowGroup), &vfull[sv]);
      issued_v = kv + 1;
      return true;
    };
    bool v_ok = true;
    for (int k = 0; k < n; ++k) {
      const int s = k % kTcStages;
      int blk = blk_next;
      if (k >= kTcStages) {
        int ok = 1;
        if (lane == 0 && (!mbar_wait(&kfree[s], ((k / kTcStages) - 1) & 1) ||
                          !mbar_wait(&dfree[s], ((k / kTcStages) - 1) & 1))) {
          atomicOr(a.err, PKV_DEVERR_TIMEOUT);
          ok = 0;
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          v_ok = false;
          break;
        }
      }
      const int t0 = i * kTcRows;
      const int nvalid = min(kTcRows, len - t0);
      const int dseg = k - i;  // CTA stage index of the segment's first stage
      const bool start = k == 0 || i == 0;
      const bool end = k == n - 1 || i == nt - 1;
      if (start) ++pieces;
      const int qb = (pieces - 1) % kQBufs;
      const int flags = (start ? kStart : 0) | (end ? kEnd : 0) |
                        (end && i == nt - 1 && dseg >= 0 ? kWholeSeg : 0) |
                        (dseg > 0 ? kSlotOne : 0) | (qb << 4);
      const int nbox = (nvalid + TB - 1) / TB;  // per tensor
      int brow = (t0 + j * TB) % P;
      const bool bad = j < nbox && (blk < 0 || (int64_t)blk >= a.num_blocks);
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.err, PKV_DEVERR_BLOCK);
      if (bad) {
        blk = (int)a.num_blocks;  // zero-filled out-of-range box
        brow = 0;
      }
      if (lane == 0) {
        sdesc[s] = make_int4(r, h, nvalid, flags);
        mbar_arrive_expect_tx(&kfull[s], (uint32_t)(nbox * TB * kTcD * 2 + (start ? 2 * G * 128 : 0)));
      }
      __syncwarp();
      if (lane < 16 && j < nbox)
        tma_load_5d(ring + (size_t)s * 2 * kTcTile + j * TB * kTcD * 2, &tmk, 0, 0, 0, h,
                    (int)((int64_t)blk * (P / kRowGroup) + brow / kRowGroup), &kfull[s]);
      if (start && lane == 0) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(qs + qb * kQBytes + hf * kQHalf, &tmq, hf * 64, h * G,
                      a.q_rows ? __ldg(a.q_rows + r) : r, &kfull[s]);
      }
      issued_k = k + 1;
      if (k >= 1 && !issue_v(k - 1)) {
        v_ok = false;
        break;
      }
      v_blk = blk;
      v_brow = brow;
      v_nbox = nbox;
      v_h = h;
      if (k + 1 < n && ++i == nt) {  // on to the next non-empty segment
        i = 0;
        if (++h == Hkv) {
          h = 0;
          do {
            ++r;
            len = effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, false);
            nt = (len + kTcRows - 1) / kTcRows;
          } while (nt == 0);
        }
      }
      if (k + 1 < n) blk_next = box_block(r, i, len);
    }
    if (v_ok) issue_v(n - 1);
  } else if (warp == 1) {
    // ============================================================ MMA issue
    // QK of stage k, then PV of stage k - 1 (whose P^T the softmax wrote
    // while QK ran).  The first PV of a piece starts a fresh O^T, once the
    // previous piece's epilogue has read it.
    if (lane == 0) {
      bool ok = true;
      int pflags = 0, pieces_done = 0;
      auto issue_pv = [&](int j, int fl) -> bool {
        if (!mbar_wait(&pfull, j & 1) || !mbar_wait(&vfull[j % kTcStages], (j / kTcStages) & 1))
          return false;
        if ((fl & kStart) && pieces_done > 0 && !mbar_wait(&ofree, (pieces_done - 1) & 1))
          return false;
        tc::fence_after_sync();
        const uint32_t vb = smem_u32(ring + (size_t)(j % kTcStages) * 2 * kTcTile + kTcTile);
        // P^T = hi + lo: both terms through the same V tile
#pragma unroll
        for (int term = 0; term < 2; ++term) {
          const uint32_t pb = smem_u32(pt + term * kQBytes);
#pragma unroll
          for (int kk = 0; kk < kTcRows / 16; ++kk) {
            // V MN-major: 64-column d chunks 1 KiB apart, 8-key groups 2 KiB apart
            const uint64_t ad = tc::smem_desc_sw128(vb + kk * 2 * kTcGroup, 1024, kTcGroup);
            const uint64_t bd =
                tc::smem_desc_sw128(pb + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16(tmem + 32, ad, bd, kIdPV,
                         (term > 0 || kk > 0 || !(fl & kStart)) ? 1u : 0u);
          }
        }
        tc::commit(&ofull);
        tc::commit(&vfree[j % kTcStages]);
        if (fl & kEnd) ++pieces_done;
        return true;
      };
      for (int k = 0; k < n; ++k) {
        const int s = k % kTcStages, b = k & 1;
        if (!mbar_wait(&kfull[s], (k / kTcStages) & 1) ||
            (k >= 2 && !mbar_wait(&sfree[b], ((k - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const int fl = sdesc[s].w;
        const uint32_t kb = smem_u32(ring + (size_t)s * 2 * kTcTile);
        const uint32_t qb = smem_u32(qs + ((fl >> 4) & 3) * kQBytes);
#pragma unroll
        for (int kk = 0; kk < kTcD / 16; ++kk) {
          const uint64_t ad =
              tc::smem_desc_sw128(kb + (kk >> 2) * 1024 + (kk & 3) * 32, 16, kTcGroup);
          const uint64_t bd = tc::smem_desc_sw128(qb + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024);
          tc::mma_bf16(tmem + 16 * b, ad, bd, kIdQK, kk > 0 ? 1u : 0u);
        }
        tc::commit(&sfull[b]);
        tc::commit(&kfree[s]);
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
    float m[G], lp[G];  // running max (base 2) and this thread's share of the sum
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      lp[g] = 0.f;
    }
    uint32_t rs = 0;  // phases of rsync used so far
    auto group_sync = [&]() -> bool {
      mbar_arrive(&rsync);
      const bool okw = __all_sync(0xffffffffu, mbar_wait(&rsync, rs & 1u));
      ++rs;
      if (!okw && lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
      return okw;
    };
    for (int k = 0; k < n; ++k) {
      const int s = k % kTcStages, b = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&kfull[s], (k / kTcStages) & 1)) ||
          !__all_sync(0xffffffffu, mbar_wait(&sfull[b], (k >> 1) & 1))) {
        if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        break;
      }
      tc::fence_after_sync();
      const int4 dsc = sdesc[s];
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
      if (lane == 0) {
        mbar_arrive(&sfree[b]);
        mbar_arrive(&dfree[s]);  // this warp is done with the slot's descriptor
      }
      // ---- the exponent base of a head moves only when one of its scores
      // passes it by more than 2^8 (m = -inf before a piece's first row): the
      // four warps first agree on whether any score does, and only then
      // take the per-head max over the 128 key rows
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
      // ---- PV of the previous stage has completed: O^T is current and the
      // P^T buffer is free
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
      // ---- P^T[g][row] as two bf16 terms, p = hi + lo to about 2^-17
      // relative (one bf16 term alone errs by up to 2^-9 per weight, which a
      // few keys of opposite-signed values can lift to the attention
      // tolerance): K-major, 128-byte swizzle, 64-key halves
      {
        const int hf = row >> 6, cch = (row & 63) >> 3, e = row & 7;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const __nv_bfloat16 hi = __float2bfloat16_rn(p[g]);
          const __nv_bfloat16 lo = __float2bfloat16_rn(p[g] - __bfloat162float(hi));
          unsigned char* at = pt + hf * kQHalf + g * 128 + ((cch ^ (g & 7)) << 4) + e * 2;
          *reinterpret_cast<__nv_bfloat16*>(at) = hi;
          *reinterpret_cast<__nv_bfloat16*>(at + kQBytes) = lo;
        }
      }
      // zero the rows of V past the tail (weight 0, bytes maybe NaN), once
      // the stage's V has landed
      if (nvalid < kTcRows &&
          !__all_sync(0xffffffffu, mbar_wait(&vfull[s], (k / kTcStages) & 1))) {
        if (lane == 0) atomicOr(a.err, PKV_DEVERR_TIMEOUT);
        break;
      }
      if (row >= nvalid) {
        unsigned char* vrow = ring + (size_t)s * 2 * kTcTile + kTcTile +
                              (row / kRowGroup) * kTcGroup + (row % kRowGroup) * 128;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(vrow + hf * 1024 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull);
      if (flags & kEnd) {
        // ---- epilogue of a piece: O = O^T / l, LSE = m + log2 l
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
            a.rec_o[(rec * G + g) * kTcD + row] = ov;
            if (row == 0) a.rec_lse[rec * G + g] = lse2;
          } else if (a.st_o) {
            const int64_t slot = (rh0 + g) * a.st_stride + a.st_slot;
            a.st_o[slot * kTcD + row] = ov;
            if (row == 0) a.st_lse[slot] = lse2;
          } else {
            store_out(static_cast<__nv_bfloat16*>(a.out) + (rh0 + g) * kTcD + row, ov);
            if (row == 0 && a.lse_out) a.lse_out[rh0 + g] = lse2 * kLn2f;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (t == 0) {
    // if anything left early, copies may still be in flight into the ring:
    // wait for them (bounded) before the CTA's shared memory is released
    for (int kk = issued_k > kTcStages ? issued_k - kTcStages : 0; kk < issued_k; ++kk)
      mbar_wait(&kfull[kk % kTcStages], (kk / kTcStages) & 1);
    for (int kk = issued_v > kTcStages ? issued_v - kTcStages : 0; kk < issued_v; ++kk)
      mbar_wait(&vfull[kk % kTcStages], (kk / kTcStages) & 1);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

bool decode_tc_supported(int dtype, int head_dim, int group, int block_size) {
  return dtype == PKV_BF16 && head_dim == kTcD && group == 8 &&
         (kTcRows % block_size == 0 || block_size % kTcRows == 0);
}

int decode_tc_rows() { return kTcRows; }

int decode_tc_resident_ctas() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    auto kern = decode_tc_kernel<8>;
    int per_sm = 0, sms = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcThreads, kTcSmem) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    cached[dev] = per_sm * sms;
  }
  return cached[dev];
}

cudaError_t launch_paged_decode_tc(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                   const CUtensorMap& tmq, const DecodeArgs& a,
                                   cudaStream_t stream) {
  auto kern = decode_tc_kernel<8>;
  static SmemAttrCache attr_cache;
  cudaError_t e = ensure_smem_limit(kern, kTcSmem, attr_cache);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3((unsigned)a.num_ctas), dim3(kTcThreads), kTcSmem, stream, tmk, tmv,
                 tmq, a);
  if (e != cudaSuccess) return e;
  return launch_decode_reduce(PKV_BF16, kTcD, a, stream);
}

}  // namespace pkv
