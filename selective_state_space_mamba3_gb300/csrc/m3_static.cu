// m3_siso_forward_static: the SISO scan for callers that cannot allocate
// device memory.
//
// m3_siso_forward asks its caller for a workspace (scratch device memory that
// its kernels use during the call: the chunked tensor-core path keeps a
// device status word there, and per-segment summary states when it splits
// long sequences). Some callers cannot provide one: code embedded in a host
// that owns every device allocation (a framework plugin or an inference
// runtime with its own memory pool and no allocator hook), or a
// latency-critical loop in which a cudaMalloc would synchronize the device.
// This entry point takes no workspace: it uses a fixed scratch array that
// lives in this library's device image (a file-scope __device__ array of
// kStaticScratchBytes), so the library itself allocates nothing either.
//
// Every GPU that loads the library holds the array until the process exits.
// All calls on a device share it and it keeps the last call's contents; the
// scan clears what must start at zero on every call (the status word; the
// summary and entry states are written before they are read). Calls that
// overlap on the GPU (different streams without ordering between them) race
// on the array and must not be issued.
//
// The array's device address belongs to the CUDA context that loaded the
// module, so it is looked up (cudaGetSymbolAddress, a host-side query) in the
// current context on every call rather than cached: a host that runs its own
// context, or calls after cudaDeviceReset, gets the address that is valid
// there.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;  // 1 MiB per device
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the scratch array in the current context.
int static_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
    cudaGetLastError();  // clear the error the failed query left
    return M3_ERR_CUDA;
  }
  *out = p;
  return M3_OK;
}

}  // namespace
}  // namespace m3

extern "C" int m3_siso_forward_static(const m3_ssm_config* cfg, const float* c, const float* b,
                                      const float* x, const float* z, const float* adt,
                                      const float* dt, const float* trap, const float* angle,
                                      const float* c_bias, const float* b_bias, const float* d,
                                      float* out, m3_stream_t stream) {
  m3::NvtxRange nvtx_range("m3_siso_forward_static");
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

// Status word of the last m3_siso_forward_static call on `stream`'s device:
// the first bytes of the scratch array, where the scan's bounded waits record
// a timeout (as in a caller workspace read by m3_workspace_status).
extern "C" int m3_siso_forward_static_status(m3_stream_t stream) {
  void* scratch = nullptr;
  const int st = m3::static_scratch(&scratch);
  if (st != M3_OK) return st;
  return m3_workspace_status(scratch, m3::kStaticScratchBytes, stream);
}
