// Internal declarations shared by the CUDA translation units of libm3.
// Host validation lives in m3_api.cu; each k_*.cu file holds one kernel family
// and its launcher.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/m3.h"

namespace m3 {

// Resolved scan geometry (num_groups == 0 already replaced by H).
struct ScanGeom {
  int B, L, H, G, P, N, A, R;
  int has_z, has_d, has_norm;
  int math_mode;
  int mimo;  // the MIMO operation (mimo_x / mimo_z / mimo_o operands)
  // packed-projection scan only: width W of a packed row and the preprocess
  // settings (`Mamba3PreprocessConfig`)
  int W;
  float eps, dt_min, dt_max, a_floor;
};

// Scan operands. For the packed-projection scan, x and z point at their
// columns of the packed rows, trap / angle at the trap / angle columns (row
// stride W), dt / adt at the row pass's [rows][H] arrays, c and b are unused
// (the C and B rows are read through tensor maps of the packed rows) and
// row_inv holds the inverse RMS of every B and C row ([rows][2 G R]: the G R
// B rows, then the G R C rows, as launch_row_pre writes them).
struct ScanArgs {
  const float *c, *b, *x, *z, *adt, *dt, *trap, *angle, *c_bias, *b_bias, *d;
  const float *mimo_x, *mimo_z, *mimo_o, *norm_weight;  // null for SISO
  float* out;
  const float* dt_bias;  // packed-projection scan only
  const float* row_inv;  // packed-projection scan only
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

// Gradients of the eight preprocess outputs (`mamba3_preprocess_backward`), in
// the layouts of PreOut.
struct PreGrads {
  const float *x, *z, *bh, *ch, *dt, *adt, *trap, *angle;
};

// Recurrent-state inputs / outputs of the chunked scan. A CTA handles segment
// `seg` of sequence `bh`: tokens [seg * seg_len, min(L, (seg + 1) * seg_len)).
// States are "pre-loaded" (h plus the next token's trapezoid term), fp32,
// [cta][P][N] with cta = bh * nseg + seg; angles [cta][A].
struct ChunkIO {
  int seg_len, nseg;
  // launched as a programmatic dependent of the kernel just before it in the
  // stream (the packed scan after its row-norm pass): wait for that kernel's
  // results before the first token preload
  int pdl;
  // summary pass: its last sum_skip segments (the pieces of the main pass's
  // last segment) have no use and return at once
  int sum_skip;
  const float* g0;   // initial state per CTA (null: zero)
  const float* th0;  // initial cumulative angle per CTA (null: zero)
  float* g1;         // final state per CTA (null: not written)
  float* th1;        // final cumulative angle per CTA
  float* e1;         // exp(sum of adt over the segment) per CTA
  // written by the CTA whose segment ends the sequence, indexed by bh:
  float* g_last;     // [BH][P][N] final state (= h after token L-1)
  float* th_last;    // [BH][A] final cumulative angle
  float* k_last;     // [BH][R][N] rotated, biased key of token L-1 (fp32)
  float* v_last;     // [BH][R][P] rank-scaled value of token L-1
};

// Device status word written by bounded waits (lives in the caller's workspace).
constexpr uint32_t kStatusTimeout = 0x54494d45u;  // "TIME"
// A wait gave up and the kernel's bounded wait for its own copies still in
// flight gave up too: it exited with those copies unfinished.
constexpr uint32_t kStatusUndrained = 0x44524e58u;  // "DRNX"

// Launchers: return cudaSuccess or the launch error. Each increments the
// library's launch counter by the number of kernels it enqueued.
// Per-row scalars of the packed scan, computed exactly as the preprocess
// computes them (W, I, N multiples of 4 and N <= 128): the inverse RMS of
// every B and C row, inv[row][j] for the j-th of the 2 G R rows, and the
// clamped dt and floored adt, dt[row][h] and adt[row][h].
cudaError_t launch_row_pre(const PreGeom& g, const float* projected, const float* dt_bias,
                           float* inv, float* dt, float* adt, cudaStream_t s);
cudaError_t launch_preprocess(const PreGeom& g, const float* projected, const float* dt_bias,
                              const PreOut& o, cudaStream_t s);
// The preprocess adjoint: gproj [rows, W] and gdt_bias [H]; `partial` holds
// preprocess_backward_workspace_bytes(g) of per-(chunk of rows, head) sums.
size_t preprocess_backward_workspace_bytes(const PreGeom& g);
cudaError_t launch_preprocess_backward(const PreGeom& g, const float* projected,
                                       const float* dt_bias, const PreGrads& gr, float* gproj,
                                       float* gdt_bias, float* partial, cudaStream_t s);
cudaError_t launch_step(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                        cudaStream_t s);
// st: optional step state (null ssm: zero state, nothing written back).
cudaError_t launch_scan_seq(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                            cudaStream_t s);
cudaError_t launch_state_init(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                              float* g0, float* th0, cudaStream_t s);
cudaError_t launch_state_prefix(const ScanGeom& g, int nseg, int pieces, const float* g_init,
                                const float* th_init, const float* gsum, const float* thsum,
                                const float* esum, float* g_entry, float* th_entry,
                                cudaStream_t s);
bool chunk_supported(const ScanGeom& g);
// the split-operand (3xTF32) flavour fits the device's shared memory for g
bool chunk_split_supported(const ScanGeom& g);
// summary: state-only pass (no outputs), used to split long sequences.
// split: the split-operand flavour (one CTA per SM) instead of single-pass TF32.
cudaError_t launch_scan_chunk(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                              const ChunkIO& io, bool summary, bool split, cudaStream_t s);
int chunk_rows_per_token(const ScanGeom& g);  // 64 / R: tokens per chunk
// the SISO scan of a packed projection (ScanArgs as described above)
bool chunk_packed_supported(const ScanGeom& g);
cudaError_t launch_scan_chunk_packed(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                                     const ChunkIO& io, bool summary, bool split,
                                     cudaStream_t s);
// `PreprocessGeometry::resolve` rules for `rows` packed rows; fills g
int resolve_pre(const m3_preprocess_config* cfg, int64_t rows, PreGeom* g);

// SISO adjoints (`mamba3_siso_backward`): the gradient of the scan output and
// the eleven gradient outputs, each in its forward operand's layout.
struct BwdArgs {
  const float* dout;
  float *gc, *gb, *gx, *gz, *gadt, *gdt, *gtrap, *gangle, *gc_bias, *gb_bias, *gd;
};
size_t backward_workspace_bytes(const ScanGeom& g);
// MIMO adjoints (`mamba3_mimo_backward`): the eleven of the SISO set plus the
// gradients of mimo_x, mimo_z, mimo_o [H,R,P] and norm_weight [H,P].
struct MBwdArgs {
  BwdArgs g;
  float *gmx, *gmz, *gmo, *gnw;
};
size_t mimo_backward_workspace_bytes(const ScanGeom& g);
cudaError_t launch_mimo_backward(const ScanGeom& g, const ScanArgs& a, const MBwdArgs& o,
                                 void* ws, cudaStream_t s);
cudaError_t launch_siso_backward(const ScanGeom& g, const ScanArgs& a, const BwdArgs& o,
                                 void* ws, cudaStream_t s);

// Scan entry chosen by the host: workspace bytes for geometry g (with or
// without a recurrent state), then launch (st null: zero state).
size_t scan_workspace_bytes(const ScanGeom& g, bool with_state);
cudaError_t launch_scan(const ScanGeom& g, const ScanArgs& a, const StepState* st, void* ws,
                        size_t ws_bytes, cudaStream_t s);

void count_launches(uint64_t n);

// NVTX range around one C-ABI call (header-only NVTX 3: a no-op unless a
// profiler injects its tool library), so that timelines show each m3_* call.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---------------------------------------------------------------------------
// Scalar maps of the method, in float32 (overflow-safe softplus as in the
// `softplus` op of the oa::ml::matrix API reference).
__device__ __forceinline__ float softplus_f(float v) {
  return v > 20.0f ? v : log1pf(expf(v));
}
__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + expf(-v)); }
__device__ __forceinline__ float silu_f(float v) { return v * sigmoid_f(v); }

// Preprocess maps (`mamba3_preprocess`), shared by the preprocess kernel and
// the fused packed-projection scan so that both produce the same bits: the
// clamped dt, the floored negative log decay adt, the sum of squares of four
// B/C values (a fixed FMA chain), and the inverse RMS of a row from its sum of
// squares (IEEE division and square root).
__device__ __forceinline__ float pre_dt(float raw, float bias, float lo, float hi) {
  return fminf(fmaxf(softplus_f(__fadd_rn(raw, bias)), lo), hi);
}
__device__ __forceinline__ float pre_adt(float a_raw, float a_floor, float dt) {
  return __fmul_rn(-fmaxf(softplus_f(a_raw), a_floor), dt);
}
__device__ __forceinline__ float sumsq4(float4 v) {
  return __fmaf_rn(v.w, v.w, __fmaf_rn(v.z, v.z, __fmaf_rn(v.y, v.y, __fmul_rn(v.x, v.x))));
}
__device__ __forceinline__ float rms_inv(float ss, int n, float eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)n), eps)));
}

// sin and cos of v: Cody-Waite reduction by 2 pi (2 pi split into its float
// value and the float remainder), then the SFU sine / cosine on [-pi, pi]
// (absolute error about 2^-21). Arguments beyond 2^15 take sincosf.
__device__ __forceinline__ void sincos_fast(float v, float* s, float* c) {
  if (fabsf(v) > 32768.0f) {
    sincosf(v, s, c);
    return;
  }
  const float k = rintf(v * 0.159154943f);
  float r = fmaf(-k, 6.28318548f, v);
  r = fmaf(-k, -1.74845553e-7f, r);
  *s = __sinf(r);
  *c = __cosf(r);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace m3
