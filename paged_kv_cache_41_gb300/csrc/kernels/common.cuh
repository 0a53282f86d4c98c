// common.cuh -- device helpers shared by the libpkv kernels (sm_103a only).
//
// Inline PTX for mbarriers and the tensor memory accelerator (TMA), bounded
// waits that report a timeout instead of spinning forever, and bf16 <-> fp32
// packing.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// A wait on an mbarrier gives up after this many nanoseconds of %globaltimer
// and reports PKV_DEVERR_TIMEOUT.  Every wait in this library normally ends
// within microseconds.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// the caller must record PKV_DEVERR_TIMEOUT) if limit_ns nanoseconds pass
// first.  The library's kernels keep the default limit everywhere; the
// drains after a timeout (waits for their own copies in flight) must too.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// 4-D tiled TMA load global -> shared, completing on `bar` (complete_tx).
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// 5-D tiled TMA load global -> shared, completing on `bar` (complete_tx).
__device__ __forceinline__ void tma_load_5d(void* smem_dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, int c4, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled TMA load global -> shared, completing on `bar` (complete_tx).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 5-D tiled TMA store shared -> global (bulk async-group completion).
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                             int c4, const void* smem_src) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group"
      " [%0, {%1, %2, %3, %4, %5}], [%6];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(smem_src))
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Bulk copy global -> shared of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), completing on `bar` (complete_tx).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch `bytes` (a multiple of 16) of global memory from a 16-byte
// aligned address into L2, asynchronously.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of
// the stream (launched with the programmatic-serialisation attribute) be
// scheduled now; that kernel's pdl_wait still blocks until this grid has
// completed and its memory is visible.  Without such a launch both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier over `nthreads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- conversions
// bf16 is the upper half of a binary32, so widening is a shift or a mask.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Load N consecutive elements (N * sizeof(T) a multiple of 8 bytes) and widen
// them to fp32.  `p` must be aligned to min(16, N * sizeof(T)) bytes.
template <typename T, int N>
struct VecLoad;

template <int N>
struct VecLoad<float, N> {
  static_assert(N % 2 == 0, "fp32 vectors are loaded two at a time at least");
  __device__ __forceinline__ static void run(const float* p, float (&f)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        float4 x = reinterpret_cast<const float4*>(p)[i];
        f[4 * i] = x.x;
        f[4 * i + 1] = x.y;
        f[4 * i + 2] = x.z;
        f[4 * i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        float2 x = reinterpret_cast<const float2*>(p)[i];
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
      }
    }
  }
};

template <int N>
struct VecLoad<__nv_bfloat16, N> {
  static_assert(N % 4 == 0, "bf16 vectors are loaded four at a time at least");
  __device__ __forceinline__ static void run(const __nv_bfloat16* p, float (&f)[N]) {
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N / 8; ++i) {
        uint4 x = reinterpret_cast<const uint4*>(p)[i];
        f[8 * i + 0] = bf16lo(x.x);
        f[8 * i + 1] = bf16hi(x.x);
        f[8 * i + 2] = bf16lo(x.y);
        f[8 * i + 3] = bf16hi(x.y);
        f[8 * i + 4] = bf16lo(x.z);
        f[8 * i + 5] = bf16hi(x.z);
        f[8 * i + 6] = bf16lo(x.w);
        f[8 * i + 7] = bf16hi(x.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        uint2 x = reinterpret_cast<const uint2*>(p)[i];
        f[4 * i + 0] = bf16lo(x.x);
        f[4 * i + 1] = bf16hi(x.x);
        f[4 * i + 2] = bf16lo(x.y);
        f[4 * i + 3] = bf16hi(x.y);
      }
    }
  }
};

// E4M3 codes (the elements of an MXFP8 pool), widened exactly through fp16.
// The caller applies the group's power-of-two scale.
template <int N>
struct VecLoad<__nv_fp8_e4m3, N> {
  static_assert(N % 4 == 0, "fp8 vectors are loaded four at a time at least");
  __device__ __forceinline__ static void run(const __nv_fp8_e4m3* p, float (&f)[N]) {
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N / 8; ++i) {
        const uint2 x = reinterpret_cast<const uint2*>(p)[i];
        widen4(x.x, f + 8 * i);
        widen4(x.y, f + 8 * i + 4);
      }
    } else {
#pragma unroll
      for (int i = 0; i < N / 4; ++i) widen4(reinterpret_cast<const uint32_t*>(p)[i], f + 4 * i);
    }
  }
  __device__ __forceinline__ static void widen4(uint32_t w, float* f) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
  }
};

// 2^(s - 127) for an E8M0 scale byte s in [0, 254] (s = 0 is the fp32
// subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t s) {
  return __uint_as_float(s ? s << 23 : 0x00400000u);
}

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Effective context length of a request: negative lengths count as empty and
// lengths beyond the block table row are clamped; both set PKV_DEVERR_LENGTH.
__device__ __forceinline__ int effective_len(int len, int max_blocks, int block_size,
                                             unsigned int* err, bool report) {
  const long long cap = (long long)max_blocks * block_size;
  if (len < 0) {
    if (report) atomicOr(err, PKV_DEVERR_LENGTH);
    return 0;
  }
  if ((long long)len > cap) {
    if (report) atomicOr(err, PKV_DEVERR_LENGTH);
    return (int)cap;
  }
  return len;
}

}  // namespace pkv
