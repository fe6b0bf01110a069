// Diagnostic entry point: exercises the bounded mbarrier wait that every
// tensor-core wait of the scans uses, on a barrier that nothing completes, so
// that the timeout path (status word in the workspace, normal kernel exit, a
// usable context afterwards) can be tested without a fault or a hang.
#include "m3_internal.cuh"
#include "tc_ptx.cuh"

namespace m3 {
namespace {

__global__ void k_wait_timeout(uint32_t* status, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::bar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  __syncthreads();
  // no thread arrives: phase 0 never completes, the wait gives up after `budget`
  const bool ok = tc::bar_wait(&bar, 0, budget);
  __syncthreads();
  if (!ok && threadIdx.x == 0) atomicExch(status, kStatusTimeout);
}

}  // namespace
}  // namespace m3

extern "C" int m3_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                        int64_t budget_cycles, m3_stream_t stream) {
  if (!workspace || workspace_bytes < 16 || budget_cycles <= 0 || budget_cycles > 4000000000LL)
    return M3_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return M3_ERR_UNALIGNED;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* status = static_cast<uint32_t*>(workspace);
  if (cudaMemsetAsync(status, 0, 16, s) != cudaSuccess) return M3_ERR_CUDA;
  m3::k_wait_timeout<<<1, 32, 0, s>>>(status, (long long)budget_cycles);
  m3::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}
