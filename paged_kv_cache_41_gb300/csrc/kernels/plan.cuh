// plan.cuh -- the work split of the persistent decode kernels.
//
// The work list is every (sequence, kv head) segment of nt = ceil(T / kRows)
// stages, sequence-major then kv head.  Work is measured in units: a stage
// costs a.stage_units and each non-empty segment a.piece_units more (the
// fixed cost of a piece: its q, its merge, its record), placed before its
// first stage.  So segment (r, h) spans u_r = stage_units * nt_r +
// piece_units units (0 when nt_r = 0) starting at
//   s0 = pre[r] * Hkv + h * u_r,   pre[r] = u_0 + ... + u_{r-1},
// and its stage i starts at unit s0 + piece_units + stage_units * i.  With
// S units in all and w = max(ceil(S / C), stage_units), CTA c owns the stages that start in
// [c w, (c + 1) w): a contiguous run of the global stage order, so only the
// CTAs with a range of nothing but piece units are empty, and the stage
// starting at unit x belongs to CTA x / w.  With stage_units = 1 and
// piece_units = 0 every CTA streams the same number of stages.
#pragma once

#include <limits.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

// Units per CTA: an equal share, and at least one stage's worth, so that a
// CTA whose range lies inside a segment owns at least one of its stages.
__host__ __device__ __forceinline__ long long units_per_cta(long long S, int C, long long stage_units) {
  const long long w = (S + C - 1) / C;
  return w > stage_units ? w : stage_units;
}

// Every CTA scans the lengths (all kThreads threads must call this): units
// per sequence, their total S (times Hkv), this CTA's range, and the
// (sequence, kv head, stage in segment) of its first stage in *d0 -- whose
// stage index may equal that segment's stage count, meaning the first stage
// of the next non-empty segment (never when stage_units = 1 and piece_units
// = 0).  CTA 0 also stores the exclusive prefix of
// units per sequence in a.plan_pre (and the total in a.plan_pre[B]) for the
// reduction, and reports bad lengths (PKV_DEVERR_LENGTH).  The scan runs in
// passes of kThreads * kPer sequences, kPer consecutive ones per thread; up
// to one pass, the lengths are read once and kept in registers.  `wsum` is
// shared scratch of at least 2 * (kThreads / 32) + 4 long longs.  Returns the
// number of stages of this CTA (<= 0: none; the caller leaves).
template <int kThreads, int kRows, int kPer = 8>
__device__ __forceinline__ int plan_cta_stages(const DecodeArgs& a, long long* wsum, int4* d0) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kChunk = kThreads * kPer;
  const int c = blockIdx.x, C = a.num_ctas;
  const int B = a.num_seqs, P = a.block_size, Hkv = a.num_kv_heads;
  const long long su = a.stage_units, pu = a.piece_units;
  const bool weighted = su != 1 || pu != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long* usum = wsum;            // [kWarps] per-warp unit sums
  long long* ssum = wsum + kWarps;   // [kWarps] per-warp stage sums
  long long* found = wsum + 2 * kWarps;  // the stage counts at lo and hi, then the start
  // One pass over sequences [base, base + kChunk): stages nt[] of this
  // thread's sequences, the exclusive prefixes of units and stages before its
  // first one within the pass, and the pass totals.
  auto scan_chunk = [&](int base, int (&nt)[kPer], long long& uex, long long& sex,
                        long long& utot, long long& stot, bool report) {
    long long mu = 0, ms = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int r = base + threadIdx.x * kPer + j;
      nt[j] = r < B ? (effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, report) +
                       kRows - 1) / kRows
                    : 0;
      mu += nt[j] > 0 ? su * nt[j] + pu : 0;
      ms += nt[j];
    }
    long long xu = mu, xs = ms;
    if (weighted) {
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long yu = __shfl_up_sync(0xffffffffu, xu, o);
        const long long ys = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) {
          xu += yu;
          xs += ys;
        }
      }
    } else {  // units are stages: one sum
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long yu = __shfl_up_sync(0xffffffffu, xu, o);
        if (lane >= o) xu += yu;
      }
      xs = xu;
    }
    if (lane == 31) {
      usum[warp] = xu;
      ssum[warp] = xs;
    }
    __syncthreads();
    long long bu = 0, bs = 0;
    utot = 0;
    stot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const long long tu = usum[w], ts = ssum[w];
      if (w < warp) {
        bu += tu;
        bs += ts;
      }
      utot += tu;
      stot += ts;
    }
    uex = bu + xu - mu;
    sex = bs + xs - ms;
    __syncthreads();  // the sums are rewritten by the next pass
  };
  // Stages that start before units lo and hi (hi only when want_hi), for
  // those inside this thread's sequences [base + t kPer, +kPer) (whose first
  // unit and stage are ucar and scar): writes found[0] and found[1], and for
  // lo the CTA's first stage as (sequence, head, stage).  The loop finds the
  // sequences by comparisons alone; the divisions run once, in the thread
  // that holds each.
  auto search = [&](int base, const int (&nt)[kPer], long long ucar, long long scar,
                    long long lo, long long hi, bool want_hi) {
    long long uu = ucar, ss = scar;
    long long u_m[2] = {0, 0}, uu_m[2] = {0, 0}, ss_m[2] = {0, 0};
    int j_m[2] = {-1, -1}, nt_m[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const long long u = nt[j] > 0 ? su * nt[j] + pu : 0;
      const long long a0 = uu * Hkv, a1 = (uu + u) * Hkv;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const long long x = q == 0 ? lo : hi;
        if (u > 0 && (q == 0 || want_hi) && a0 <= x && x < a1) {
          j_m[q] = j;
          nt_m[q] = nt[j];
          u_m[q] = u;
          uu_m[q] = uu;
          ss_m[q] = ss;
        }
      }
      uu += u;
      ss += nt[j];
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (j_m[q] < 0) continue;
      const long long x = q == 0 ? lo : hi;
      const long long off = x - uu_m[q] * Hkv;  // < Hkv * u_m[q]
      const int h = off < INT_MAX && u_m[q] < INT_MAX ? (int)((unsigned)off / (unsigned)u_m[q])
                                                      : (int)(off / u_m[q]);
      const long long in = off - (long long)h * u_m[q] - pu;  // units past the piece units
      long long i = 0;
      if (in > 0) i = min(su == 1 ? in : su == 2 ? (in + 1) >> 1 : (in + su - 1) / su, (long long)nt_m[q]);
      found[q] = ss_m[q] * Hkv + (long long)h * nt_m[q] + i;
      if (q == 0) {
        int* st = reinterpret_cast<int*>(found + 2);
        st[0] = base + threadIdx.x * kPer + j_m[q];
        st[1] = h;
        st[2] = (int)i;
      }
    }
  };
  if (threadIdx.x == 0) {
    found[0] = -1;
    found[1] = -1;
  }
  long long U = 0, ST = 0;  // units and stages of all sequences (per kv head)
  // ---- pass 1: totals, and the prefix for the reduction
  int nt1[kPer];
  long long uex1 = 0, sex1 = 0;
  for (int base = 0; base < B; base += kChunk) {
    int nt[kPer];
    long long uex, sex, utot, stot;
    scan_chunk(base, nt, uex, sex, utot, stot, c == 0);
    if (c == 0) {
      long long p = U + uex;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int r = base + threadIdx.x * kPer + j;
        if (r < B) a.plan_pre[r] = p;
        p += nt[j] > 0 ? su * nt[j] + pu : 0;
      }
    }
    if (base == 0) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) nt1[j] = nt[j];
      uex1 = uex;
      sex1 = sex;
    }
    U += utot;
    ST += stot;
  }
  if (c == 0 && threadIdx.x == 0) a.plan_pre[B] = U;
  const long long S = U * Hkv;
  const long long w = units_per_cta(S, C, su);
  const long long lo = min((long long)c * w, S), hi = min(lo + w, S);
  if (lo >= hi) return 0;  // uniform over the CTA
  // ---- find the stage counts at lo and hi (hi == S: every stage); with
  // units that are stages, the count is hi - lo and only lo is searched
  const bool want_hi = weighted && hi < S;
  if (B <= kChunk) {
    search(0, nt1, uex1, sex1, lo, hi, want_hi);
  } else {
    long long ucar = 0, scar = 0;
    for (int base = 0; base < B; base += kChunk) {
      int nt[kPer];
      long long uex, sex, utot, stot;
      scan_chunk(base, nt, uex, sex, utot, stot, false);
      // lo and hi each lie in one pass; search also matches only inside its
      // own sequences, so passing both is safe
      if (ucar * Hkv <= hi && lo < (ucar + utot) * Hkv)
        search(base, nt, ucar + uex, scar + sex, lo, hi, want_hi);
      ucar += utot;
      scar += stot;
    }
  }
  __syncthreads();
  int n;
  if (weighted) {
    const long long g_lo = found[0];
    const long long g_hi = hi < S ? found[1] : ST * Hkv;
    n = (int)(g_hi - g_lo);
  } else {
    n = (int)(hi - lo);
  }
  const int* st = reinterpret_cast<const int*>(found + 2);
  *d0 = make_int4(st[0], st[1], st[2], 0);
  __syncthreads();  // the scratch is the caller's from here on
  return n;
}

}  // namespace pkv
