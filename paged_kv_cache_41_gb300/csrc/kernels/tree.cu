// tree.cu -- the last step of attention over a prefix tree: merge each
// sequence's states.
//
// What it computes ("M5.3 - KV Memory Layout and Exact Reuse", 0x0BA and
// 0x0BD, the sequence-first phase): a sequence's keys are the rows of the
// chunks on its root-to-leaf path.  Every chunk on the path has left one or
// more (O, LSE) states for the sequence over disjoint key sets -- one per key
// split of a chunk attended chunk-first, one per chunk attended by the paged
// decode -- and attention over the whole path is their log-sum-exp merge:
//   M = max LSE_i,  w_i = 2^(LSE_i - M),  O = sum w_i O_i / sum w_i,
//   LSE = M + log2 sum w_i,
// with an empty state (LSE = -inf) the merge's identity.
//
// Design: one warp per (sequence, query head), D / 32 columns per lane.  The
// states a sequence merges are listed on the host (a CSR of (base, head
// stride) references), so the kernel walks no tree: pass 1 takes the max LSE
// with one state per lane, pass 2 accumulates, loading several states'
// outputs at once so their latencies overlap.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr float kLn2 = 0.6931471805599453f;

// Sources a warp loads at once (their latencies overlap).
constexpr int kBatch = 8;

template <typename T, int D>
__global__ void __launch_bounds__(128) tree_merge_kernel(const TreeMergeArgs a) {
  constexpr int EPL = D / 32;
  pdl_wait();  // every state of this call has been written
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rh = (int64_t)blockIdx.x * 4 + warp;
  if (rh >= (int64_t)a.num_seqs * a.num_q_heads) return;
  const int r = (int)(rh / a.num_q_heads), qh = (int)(rh % a.num_q_heads);
  const int s0 = __ldg(a.seq_ptr + r), n = __ldg(a.seq_ptr + r + 1) - s0;
  // state i of this sequence: base + qh * head_stride
  auto state = [&](int i) -> int64_t {
    const longlong2 ref = __ldg(reinterpret_cast<const longlong2*>(a.states) + s0 + i);
    return ref.x + (int64_t)qh * ref.y;
  };
  // lane i holds state i's index and LSE (states past 32, rare, are read
  // again in pass 2)
  int64_t my_si0 = 0;
  float my0 = -INFINITY;
  if (lane < n) {
    my_si0 = state(lane);
    my0 = a.st_lse[my_si0];
  }
  float M = my0;
  for (int i = lane + 32; i < n; i += 32) M = fmaxf(M, a.st_lse[state(i)]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int m = min(32, n - i0);
      int64_t my_si = my_si0;
      float my = my0;
      if (i0 > 0) {
        my = -INFINITY;
        if (lane < m) {
          my_si = state(i0 + lane);
          my = a.st_lse[my_si];
        }
      }
      for (int u0 = 0; u0 < m; u0 += kBatch) {
        float l[kBatch], x[kBatch][EPL];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          l[u] = __shfl_sync(0xffffffffu, my, (u0 + u) & 31);
          const int64_t si = __shfl_sync(0xffffffffu, my_si, (u0 + u) & 31);
          if (u0 + u >= m) l[u] = -INFINITY;  // an empty part: the identity
#pragma unroll
          for (int e = 0; e < EPL; ++e) x[u][e] = 0.f;
          if (l[u] != -INFINITY) VecLoad<float, EPL>::run(a.st_o + si * D + lane * EPL, x[u]);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (l[u] == -INFINITY) continue;
          const float w = exp2f(l[u] - M);
          L += w;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, x[u][e], acc[e]);
        }
      }
    }
  }
  const bool nonempty = L > 0.f;
  const float inv = nonempty ? 1.f / L : 0.f;
  T* out = static_cast<T*>(a.out) + rh * D + lane * EPL;
#pragma unroll
  for (int i = 0; i < EPL; ++i) store_out(out + i, acc[i] * inv);
  if (lane == 0 && a.lse_out) a.lse_out[rh] = nonempty ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <typename T, int D>
static cudaError_t launch_merge_t(const TreeMergeArgs& a, cudaStream_t stream) {
  const int64_t warps = (int64_t)a.num_seqs * a.num_q_heads;
  return launch_pdl(tree_merge_kernel<T, D>, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0,
                    stream, a);
}

cudaError_t launch_tree_merge(int dtype, int head_dim, const TreeMergeArgs& a,
                              cudaStream_t stream) {
  if (dtype == PKV_BF16 || dtype == PKV_MXFP8)  // out is bf16 beside an MXFP8 pool
    return head_dim == 128 ? launch_merge_t<__nv_bfloat16, 128>(a, stream)
                           : launch_merge_t<__nv_bfloat16, 64>(a, stream);
  return head_dim == 128 ? launch_merge_t<float, 128>(a, stream)
                         : launch_merge_t<float, 64>(a, stream);
}

}  // namespace pkv
