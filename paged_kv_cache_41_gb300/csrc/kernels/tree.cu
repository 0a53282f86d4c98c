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
// states a sequence merges are listed on the host (a CSR of (row, count)
// entries), so the kernel walks no tree: pass 1 takes the max LSE, pass 2
// accumulates.  The states are a few per sequence and are read once.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr float kLn2 = 0.6931471805599453f;

template <typename T, int D>
__global__ void __launch_bounds__(128) tree_merge_kernel(const TreeMergeArgs a) {
  constexpr int EPL = D / 32;
  pdl_wait();  // every state of this call has been written
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rh = (int64_t)blockIdx.x * 4 + warp;
  if (rh >= (int64_t)a.num_seqs * a.num_q_heads) return;
  const int r = (int)(rh / a.num_q_heads), qh = (int)(rh % a.num_q_heads);
  const int e0 = __ldg(a.seq_ptr + r), e1 = __ldg(a.seq_ptr + r + 1);
  const int Hq = a.num_q_heads, S = a.s_max;
  // state i of entry (row, n): chunk-first rows [0, cf_rows) keep n split
  // slots each; later rows are the paged decode's, one state each
  auto state_index = [&](int row, int s) -> int64_t {
    return row < a.cf_rows ? ((int64_t)row * Hq + qh) * S + s
                           : (int64_t)a.cf_rows * Hq * S + (int64_t)(row - a.cf_rows) * Hq + qh;
  };
  float M = -INFINITY;
  for (int e = e0; e < e1; ++e) {
    const int2 en = __ldg(a.entries + e);
    for (int s = lane; s < en.y; s += 32) M = fmaxf(M, a.st_lse[state_index(en.x, s)]);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int e = e0; e < e1; ++e) {
      const int2 en = __ldg(a.entries + e);
      for (int s = 0; s < en.y; ++s) {
        const int64_t si = state_index(en.x, s);
        const float l = a.st_lse[si];
        if (l == -INFINITY) continue;  // an empty part: the identity
        const float w = exp2f(l - M);
        L += w;
        float x[EPL];
        VecLoad<float, EPL>::run(a.st_o + si * D + lane * EPL, x);
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[i] = fmaf(w, x[i], acc[i]);
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
  if (dtype == PKV_BF16)
    return head_dim == 128 ? launch_merge_t<__nv_bfloat16, 128>(a, stream)
                           : launch_merge_t<__nv_bfloat16, 64>(a, stream);
  return head_dim == 128 ? launch_merge_t<float, 128>(a, stream)
                         : launch_merge_t<float, 64>(a, stream);
}

}  // namespace pkv
