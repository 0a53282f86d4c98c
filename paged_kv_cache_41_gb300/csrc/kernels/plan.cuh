// plan.cuh -- the work split of the persistent decode kernels.
//
// The work list is every (sequence, kv head) segment of ceil(T / kRows)
// stages, sequence-major then kv head; S stages in all.  CTA c of C takes
// stages [c w, min((c + 1) w, S)), w = ceil(S / C), so only trailing CTAs
// can be empty and stage p belongs to CTA p / w.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace pkv {

__host__ __device__ __forceinline__ long long stages_per_cta(long long S, int C) {
  return (S + C - 1) / C;
}

// Every CTA scans the lengths (all kThreads threads must call this): stages
// per sequence, their total S (times Hkv), this CTA's range, and the
// (sequence, kv head, stage in segment) of its first stage in *d0.  CTA 0
// also stores the exclusive prefix of stages per sequence in a.plan_pre for
// the reduction, and reports bad lengths (PKV_DEVERR_LENGTH).  The scan runs
// in passes of kThreads * kPer sequences, kPer consecutive ones per thread.
// `wsum` is shared scratch of at least kThreads / 32 + 2 long longs.  Returns
// the number of stages of this CTA (<= 0: none; the caller leaves).  Up to
// kThreads * kPer sequences the lengths are read once and kept in registers.
template <int kThreads, int kRows, int kPer = 8>
__device__ __forceinline__ int plan_cta_stages(const DecodeArgs& a, long long* wsum, int4* d0) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kChunk = kThreads * kPer;
  const int c = blockIdx.x, C = a.num_ctas;
  const int B = a.num_seqs, P = a.block_size, Hkv = a.num_kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto scan_chunk = [&](int base, int (&nt)[kPer], long long& excl, long long& total, bool report) {
    long long mine = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int r = base + threadIdx.x * kPer + j;
      nt[j] = r < B ? (effective_len(__ldg(a.seq_lens + r), a.max_blocks, P, a.err, report) +
                       kRows - 1) / kRows
                    : 0;
      mine += nt[j];
    }
    long long x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    long long before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const long long t = wsum[w];
      if (w < warp) before += t;
      total += t;
    }
    excl = before + x - mine;
    __syncthreads();  // wsum is rewritten by the next pass
  };
  int* start = reinterpret_cast<int*>(wsum + kWarps);
  if (B <= kChunk) {
    // one pass: the lengths stay in registers for the search
    int nt[kPer];
    long long excl, total;
    scan_chunk(0, nt, excl, total, c == 0);
    if (c == 0) {
      long long p = excl;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int r = threadIdx.x * kPer + j;
        if (r < B) a.plan_pre[r] = p;
        p += nt[j];
      }
      if (threadIdx.x == 0) a.plan_pre[B] = total;
    }
    const long long S = total * Hkv;
    const long long wct = stages_per_cta(S, C);
    const long long p0 = min((long long)c * wct, S);
    const int n = (int)(min(p0 + wct, S) - p0);
    if (n <= 0) return n;  // uniform over the CTA
    long long p = excl;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (nt[j] > 0 && p * Hkv <= p0 && p0 < (p + nt[j]) * Hkv) {
        const long long off = p0 - p * Hkv;
        start[0] = threadIdx.x * kPer + j;
        start[1] = (int)(off / nt[j]);
        start[2] = (int)(off % nt[j]);
      }
      p += nt[j];
    }
    __syncthreads();
    *d0 = make_int4(start[0], start[1], start[2], 0);
    __syncthreads();  // the scratch is the caller's from here on
    return n;
  }
  long long carry = 0;
  for (int base = 0; base < B; base += kChunk) {
    int nt[kPer];
    long long excl, total;
    scan_chunk(base, nt, excl, total, c == 0);
    if (c == 0) {
      long long p = carry + excl;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int r = base + threadIdx.x * kPer + j;
        if (r < B) a.plan_pre[r] = p;
        p += nt[j];
      }
    }
    carry += total;
  }
  if (c == 0 && threadIdx.x == 0) a.plan_pre[B] = carry;
  const long long S = carry * Hkv;
  const long long wct = stages_per_cta(S, C);
  const long long p0 = min((long long)c * wct, S);
  const int n = (int)(min(p0 + wct, S) - p0);
  if (n <= 0) return n;  // uniform over the CTA
  // the sequence holding stage p0, found in a second pass
  carry = 0;
  for (int base = 0; base < B; base += kChunk) {
    int nt[kPer];
    long long excl, total;
    scan_chunk(base, nt, excl, total, false);
    if (p0 < (carry + total) * Hkv) {
      long long p = carry + excl;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (nt[j] > 0 && p * Hkv <= p0 && p0 < (p + nt[j]) * Hkv) {
          const long long off = p0 - p * Hkv;
          start[0] = base + threadIdx.x * kPer + j;
          start[1] = (int)(off / nt[j]);
          start[2] = (int)(off % nt[j]);
        }
        p += nt[j];
      }
      __syncthreads();
      break;
    }
    carry += total;
  }
  *d0 = make_int4(start[0], start[1], start[2], 0);
  __syncthreads();  // the scratch is the caller's from here on
  return n;
}

}  // namespace pkv
