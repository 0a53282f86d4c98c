// wait_probe.cu -- test-only kernel for the bounded mbarrier wait of
// common.cuh.  Built into its own library beside the tests; libpkv does not
// contain or export it.
//
// One CTA of one thread initialises an mbarrier expecting one arrival.  With
// `arrive` set the thread arrives first and the wait must succeed at once;
// otherwise nothing ever arrives and no copy is in flight, so the wait must
// give up after `limit_ns` and the kernel records PKV_DEVERR_TIMEOUT in its
// own error word, which the host reads back.  The kernel always returns.
#include "kernels/common.cuh"

namespace {

__device__ unsigned int g_probe_err;

__global__ void wait_probe_kernel(uint64_t limit_ns, int arrive, unsigned long long* elapsed_ns) {
  __shared__ uint64_t bar;
  pkv::mbar_init(&bar, 1);
  pkv::fence_barrier_init();
  if (arrive) pkv::mbar_arrive(&bar);
  const uint64_t t0 = pkv::global_timer_ns();
  const bool ok = pkv::mbar_wait(&bar, 0, limit_ns);
  *elapsed_ns = pkv::global_timer_ns() - t0;
  if (!ok) atomicOr(&g_probe_err, PKV_DEVERR_TIMEOUT);
}

}  // namespace

// Runs the probe on the current device and waits for it.  Returns 0 and
// fills *err_out (the error word, then cleared) and *elapsed_ns_out (the
// wait's duration on %globaltimer), or a nonzero cudaError_t.
extern "C" int pkv_test_wait_probe(uint64_t limit_ns, int arrive, unsigned int* err_out,
                                   unsigned long long* elapsed_ns_out) {
  unsigned long long* d_elapsed = nullptr;
  cudaError_t e = cudaMalloc(&d_elapsed, sizeof(*d_elapsed));
  if (e != cudaSuccess) return (int)e;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_probe_err, &zero, sizeof(zero));
  if (e == cudaSuccess) {
    wait_probe_kernel<<<1, 1>>>(limit_ns, arrive, d_elapsed);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(err_out, g_probe_err, sizeof(*err_out));
  if (e == cudaSuccess) e = cudaMemcpy(elapsed_ns_out, d_elapsed, sizeof(*d_elapsed),
                                       cudaMemcpyDeviceToHost);
  cudaFree(d_elapsed);
  return (int)e;
}
