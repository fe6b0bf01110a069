// Fused Mamba-3 projection preprocess (oarust mamba3.rs, `mamba3_preprocess`:
// one packed projection row -> z, x, RMS-normalised B/C rows, clamped dt,
// adt = -max(softplus(a_raw), a_floor) * dt, raw trap and angle).
//
// HBM-bound streaming: every byte of `projected` is read once and every output
// byte written once. One 256-thread block handles one row at a time
// (grid-stride over rows): the z|x slices move as 128-bit streaming loads and
// stores (four loads in flight per thread before their stores), each B/C row
// is owned by one warp whose lanes hold one float4 each
// (N <= 128) and reduce the mean square with shuffles, and the 3H + A scalar
// columns are mapped by the first threads. Rows whose width or slice offsets
// are not multiples of 4 floats take the scalar path of the same kernel.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;

template <bool VEC>
__global__ void __launch_bounds__(kThreads) k_preprocess(PreGeom g, const float* __restrict__ proj,
                                                         const float* __restrict__ dt_bias,
                                                         PreOut o) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = kThreads / 32;
  const int I = g.I, N = g.N, H = g.H, A = g.A, W = g.W;
  const int RG = g.G * g.R;
  const int BC = RG * N;
  for (int64_t r = blockIdx.x; r < g.rows; r += gridDim.x) {
    const float* p = proj + r * (int64_t)W;
    // z | x slices (columns [0, 2I)): four float4 loads per thread in flight
    // before their stores (memory-level parallelism of the stream).
    if (VEC) {
      const float4* p4 = reinterpret_cast<const float4*>(p);
      const int I4 = I >> 2, Z4 = 2 * I4;
      float4* z4 = reinterpret_cast<float4*>(o.z + r * (int64_t)I);
      float4* x4 = reinterpret_cast<float4*>(o.x + r * (int64_t)I);
      for (int base = tid; base < Z4; base += 4 * kThreads) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = base + u * kThreads;
          if (i < Z4) v[u] = __ldcs(p4 + i);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = base + u * kThreads;
          if (i < Z4) {
            if (i < I4)
              __stcs(z4 + i, v[u]);
            else
              __stcs(x4 + (i - I4), v[u]);
          }
        }
      }
    } else {
      for (int i = tid; i < 2 * I; i += kThreads) {
        float v = __ldcs(p + i);
        if (i < I)
          __stcs(o.z + r * (int64_t)I + i, v);
        else
          __stcs(o.x + r * (int64_t)I + (i - I), v);
      }
    }
    // B rows then C rows (columns [2I, 2I + 2BC)), one warp per N-row.
    for (int j = warp; j < 2 * RG; j += nwarps) {
      const float* src = p + 2 * I + (int64_t)j * N;
      float* dst = (j < RG ? o.bh + r * (int64_t)BC + (int64_t)j * N
                           : o.ch + r * (int64_t)BC + (int64_t)(j - RG) * N);
      if (VEC && N <= 128) {
        const int N4 = N >> 2;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane < N4) v = __ldcs(reinterpret_cast<const float4*>(src) + lane);
        // (the fused packed-projection scan reduces in this same order: lane
        // = float4 group, then the 16-8-4-2-1 butterfly)
        const float ss = warp_sum(sumsq4(v));
        const float inv = rms_inv(ss, N, g.eps);
        if (lane < N4)
          __stcs(reinterpret_cast<float4*>(dst) + lane,
                 make_float4(__fmul_rn(v.x, inv), __fmul_rn(v.y, inv), __fmul_rn(v.z, inv),
                             __fmul_rn(v.w, inv)));
      } else {
        float ss = 0.f;
        for (int n = lane; n < N; n += 32) {
          float v = src[n];
          ss += v * v;
        }
        ss = warp_sum(ss);
        const float inv = rms_inv(ss, N, g.eps);
        for (int n = lane; n < N; n += 32) __stcs(dst + n, src[n] * inv);
      }
    }
    // dt_raw | a_raw | trap (H each) | angle (A).
    const float* s = p + 2 * I + 2 * BC;
    for (int h = tid; h < H; h += kThreads) {
      const float d = pre_dt(__ldcs(s + h), __ldg(dt_bias + h), g.dt_min, g.dt_max);
      __stcs(o.dt + r * (int64_t)H + h, d);
      __stcs(o.adt + r * (int64_t)H + h, pre_adt(__ldcs(s + H + h), g.a_floor, d));
      __stcs(o.trap + r * (int64_t)H + h, __ldcs(s + 2 * H + h));
    }
    for (int a = tid; a < A; a += kThreads) __stcs(o.angle + r * (int64_t)A + a, __ldcs(s + 3 * H + a));
  }
}

// Per-row scalars of the packed scan, computed exactly as k_preprocess<true>
// computes them: blocks [0, nb_rms) give one warp kRmsUnits (row, B/C row)
// units with their loads issued together (each unit's float4 groups in lanes
// 0 .. N/4 - 1, the same sum of squares, butterfly and inverse); the other
// blocks give one thread per (row, head) its dt and adt.
constexpr int kRmsUnits = 4;
__global__ void __launch_bounds__(kThreads) k_row_pre(PreGeom g, const float* __restrict__ proj,
                                                      const float* __restrict__ dt_bias,
                                                      float* __restrict__ inv,
                                                      float* __restrict__ dt,
                                                      float* __restrict__ adt, int nb_rms) {
  // the packed scan that follows may start its prologue now (it waits for
  // this grid's results before reading them)
  asm volatile("griddepcontrol.launch_dependents;");
  if ((int)blockIdx.x >= nb_rms) {
    const int64_t u = (int64_t)(blockIdx.x - nb_rms) * kThreads + threadIdx.x;
    if (u >= g.rows * g.H) return;
    const int64_t r = u / g.H;
    const int h = (int)(u - r * g.H);
    const float* s = proj + r * (int64_t)g.W + 2 * (int64_t)g.I + 2 * (int64_t)g.G * g.R * g.N;
    const float d = pre_dt(__ldcs(s + h), __ldg(dt_bias + h), g.dt_min, g.dt_max);
    dt[u] = d;
    adt[u] = pre_adt(__ldcs(s + g.H + h), g.a_floor, d);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int RG2 = 2 * g.G * g.R;
  const int64_t units = g.rows * RG2;
  const int64_t u0 = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kRmsUnits;
  float4 v[kRmsUnits];
#pragma unroll
  for (int k = 0; k < kRmsUnits; ++k) {
    const int64_t unit = u0 + k;
    v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (unit < units && lane < (g.N >> 2)) {
      const int64_t r = unit / RG2;
      const int j = (int)(unit - r * RG2);
      const float* src = proj + r * (int64_t)g.W + 2 * (int64_t)g.I + (int64_t)j * g.N;
      v[k] = __ldcs(reinterpret_cast<const float4*>(src) + lane);
    }
  }
#pragma unroll
  for (int k = 0; k < kRmsUnits; ++k) {
    const float ss = warp_sum(sumsq4(v[k]));
    if (lane == 0 && u0 + k < units) inv[u0 + k] = rms_inv(ss, g.N, g.eps);
  }
}

}  // namespace

cudaError_t launch_row_pre(const PreGeom& g, const float* projected, const float* dt_bias,
                           float* inv, float* dt, float* adt, cudaStream_t s) {
  const int64_t units = g.rows * 2 * g.G * g.R;
  const int64_t per_block = (int64_t)(kThreads / 32) * kRmsUnits;
  const int64_t nb_rms = (units + per_block - 1) / per_block;
  const int64_t nb_dt = (g.rows * g.H + kThreads - 1) / kThreads;
  if (nb_rms + nb_dt > 0x7fffffff) return cudaErrorInvalidValue;
  k_row_pre<<<(unsigned)(nb_rms + nb_dt), kThreads, 0, s>>>(g, projected, dt_bias, inv, dt, adt,
                                                            (int)nb_rms);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const PreGeom& g, const float* projected, const float* dt_bias,
                              const PreOut& o, cudaStream_t s) {
  const bool vec = (g.W % 4 == 0) && (g.I % 4 == 0) && (g.N % 4 == 0);
  const int64_t blocks = g.rows < (int64_t)(1 << 20) ? g.rows : (int64_t)(1 << 20);
  if (vec)
    k_preprocess<true><<<(unsigned)blocks, kThreads, 0, s>>>(g, projected, dt_bias, o);
  else
    k_preprocess<false><<<(unsigned)blocks, kThreads, 0, s>>>(g, projected, dt_bias, o);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace m3
