// Test-only probe of the bounded mbarrier wait every pipeline wait of the library's kernels
// goes through (device_utils.cuh); compiled by tests/test_gpu_wait_timeout.py, never linked
// into libpfkv.so. Thread 0 of each CTA waits on an mbarrier of its own shared memory: with
// arrive = 0 nothing ever arrives, so the wait must give up after limit_ns, report it with
// the library's timeout bit and return; with arrive = 1 the phase completes first and the
// wait succeeds at once. Nothing here can hang: the only wait is the bounded one under test.
#include "../../paged_fp8_kv_cache_gb300/csrc/device_utils.cuh"
#include "../../paged_fp8_kv_cache_gb300/csrc/pfkv_internal.h"

namespace {

__global__ void wait_probe_kernel(unsigned* err, unsigned long long* elapsed_ns, int* waited_ok,
                                  unsigned long long limit_ns, int arrive) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pfkv::mbar_init(&bar, 1);
    pfkv::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive) pfkv::mbar_arrive(&bar);
    const uint64_t t0 = pfkv::global_ns();
    const bool ok = pfkv::mbar_wait_limit(&bar, 0, limit_ns);
    elapsed_ns[blockIdx.x] = pfkv::global_ns() - t0;
    waited_ok[blockIdx.x] = ok ? 1 : 0;
    if (!ok) atomicOr(err, pfkv::kDevErrTimeout);
  }
}

}  // namespace

extern "C" int pfkv_test_wait_probe(unsigned* err, unsigned long long* elapsed_ns, int* waited_ok,
                                    unsigned long long limit_ns, int arrive, int num_ctas, cudaStream_t stream) {
  if (num_ctas < 1 || num_ctas > 1024 || limit_ns > 100000000ull) return -1;  // at most 100 ms per wait
  wait_probe_kernel<<<num_ctas, 32, 0, stream>>>(err, elapsed_ns, waited_ok, limit_ns, arrive);
  return static_cast<int>(cudaGetLastError());
}
