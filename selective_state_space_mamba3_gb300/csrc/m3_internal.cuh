// Internal declarations shared by the CUDA translation units of libm3.
// Host validation lives in m3_api.cu; each k_*.cu file holds one kernel family
// and its launcher.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/m3.h"

namespace m3 {

// Resolved scan geometry (num_groups == 0 already replaced by H).
struct ScanGeom {
  int B, L, H, G, P, N, A, R;
  int has_z, has_d, has_norm;
  int math_mode;
};

struct ScanArgs {
  const float *c, *b, *x, *z, *adt, *dt, *trap, *angle, *c_bias, *b_bias, *d;
  const float *mimo_x, *mimo_z, *mimo_o, *norm_weight;  // null for SISO
  float* out;
};

struct StepState {
  float *ssm, *angle, *k, *v;
};

struct PreGeom {
  int64_t rows;
  int I, N, H, A, G, R, W;
  float eps, dt_min, dt_max, a_floor;
};

struct PreOut {
  float *x, *z, *bh, *ch, *dt, *adt, *trap, *angle;
};

// Device status word written by bounded waits (lives in the caller's workspace).
constexpr uint32_t kStatusTimeout = 0x54494d45u;  // "TIME"

// Launchers: return cudaSuccess or the launch error. Each increments the
// library's launch counter by the number of kernels it enqueued.
cudaError_t launch_preprocess(const PreGeom& g, const float* projected, const float* dt_bias,
                              const PreOut& o, cudaStream_t s);
cudaError_t launch_step(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                        cudaStream_t s);
cudaError_t launch_scan_seq(const ScanGeom& g, const ScanArgs& a, cudaStream_t s);
bool chunk_supported(const ScanGeom& g);
cudaError_t launch_scan_chunk(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                              cudaStream_t s);

// Scan entry chosen by the host: workspace bytes for geometry g, then launch.
size_t scan_workspace_bytes(const ScanGeom& g);
cudaError_t launch_scan(const ScanGeom& g, const ScanArgs& a, void* ws, size_t ws_bytes,
                        cudaStream_t s);

void count_launches(uint64_t n);

// ---------------------------------------------------------------------------
// Scalar maps of the method, in float32 (overflow-safe softplus as in the
// `softplus` op of the oa::ml::matrix API reference).
__device__ __forceinline__ float softplus_f(float v) {
  return v > 20.0f ? v : log1pf(expf(v));
}
__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + expf(-v)); }
__device__ __forceinline__ float silu_f(float v) { return v * sigmoid_f(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace m3
