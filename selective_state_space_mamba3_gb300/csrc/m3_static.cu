// m3_siso_forward_static: the SISO scan for callers that cannot allocate
// device memory.
//
// m3_siso_forward asks its caller for a workspace (scratch device memory that
// its kernels use during the call: the chunked tensor-core path keeps a
// device status word there). Some callers cannot provide one: code embedded
// in a host that owns every device allocation (a framework plugin or an
// inference runtime with its own memory pool and no allocator hook), or a
// latency-critical loop in which a cudaMalloc would synchronize the device.
// This entry point takes no workspace: it uses a fixed scratch array that
// lives in this library's device image (a file-scope __device__ array of
// kStaticScratchBytes), so the library itself allocates nothing either.
//
// Every GPU that loads the library holds the array until the process exits.
// All calls on a device share it and it keeps the last call's contents; the
// scan clears what must start at zero on every call. Calls that overlap on
// the GPU (different streams without ordering between them) race on the
// array and must not be issued.
#include <mutex>

#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;  // 1 MiB per device
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address per device, set once

// Device address of the scratch array on the current device. The first call
// on a device looks it up with cudaGetSymbolAddress (with that device
// current) and caches it; later calls reuse the cached address.
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M3_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return M3_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return M3_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return M3_OK;
}

}  // namespace
}  // namespace m3

extern "C" int m3_siso_forward_static(const m3_ssm_config* cfg, const float* c, const float* b,
                                      const float* x, const float* z, const float* adt,
                                      const float* dt, const float* trap, const float* angle,
                                      const float* c_bias, const float* b_bias, const float* d,
                                      float* out, m3_stream_t stream) {
  size_t need = 0;
  int st = m3_siso_forward_workspace(cfg, &need);
  if (st != M3_OK) return st;
  if (need > m3::kStaticScratchBytes) return M3_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = m3::static_scratch(&scratch);
  if (st != M3_OK) return st;
  return m3_siso_forward(cfg, c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d, out, scratch,
                         m3::kStaticScratchBytes, stream);
}
