// Fused Mamba-3 projection preprocess (oarust mamba3.rs, `mamba3_preprocess`:
// one packed projection row -> z, x, RMS-normalised B/C rows, clamped dt,
// adt = -max(softplus(a_raw), a_floor) * dt, raw trap and angle).
//
// HBM-bound streaming: every byte of `projected` is read once and every output
// byte written once. One 256-thread block handles one row at a time
// (grid-stride over rows), no block barriers. Every thread first issues its
// share of the z|x slices (128-bit streaming loads, four in flight), then does
// its own column task while they land, then stores them. The column tasks are
// spread so that no warp chains more than one: each B/C row is owned by one
// warp, from the last warp down, whose lanes hold one float4 each (N <= 128)
// and reduce the mean square with shuffles; the 3H scalar columns go to the
// threads from 0, the A angle columns to the warp after those. Rows whose
// width or slice offsets are not multiples of 4 floats take the scalar path of
// the same kernel.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 4) k_preprocess(PreGeom g, const float* __restrict__ proj,
                                                         const float* __restrict__ dt_bias,
                                                         PreOut o) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int nwarps = kThreads / 32;
  const int I = g.I, N = g.N, H = g.H, A = g.A, W = g.W;
  const int RG = g.G * g.R;
  const int BC = RG * N;
  const int aoff = ((H + 31) / 32 * 32) % kThreads;
  const int ta = tid >= aoff ? tid - aoff : tid - aoff + kThreads;
  for (int64_t r = blockIdx.x; r < g.rows; r += gridDim.x) {
    const float* p = proj + r * (int64_t)W;
    const float4* p4 = reinterpret_cast<const float4*>(p);
    const int I4 = I >> 2, Z4 = 2 * I4;
    float4* z4 = reinterpret_cast<float4*>(o.z + r * (int64_t)I);
    float4* x4 = reinterpret_cast<float4*>(o.x + r * (int64_t)I);
    float4 v[4];
    if (VEC) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = tid + u * kThreads;
        if (i < Z4) v[u] = __ldcs(p4 + i);
      }
    }
    // B rows then C rows (columns [2I, 2I + 2BC)), one warp per N-row.
    for (int j = nwarps - 1 - warp; j < 2 * RG; j += nwarps) {
      const float* src = p + 2 * I + (int64_t)j * N;
      float* dst = (j < RG ? o.bh + r * (int64_t)BC + (int64_t)j * N
                           : o.ch + r * (int64_t)BC + (int64_t)(j - RG) * N);
      if (VEC && N <= 128) {
        const int N4 = N >> 2;
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane < N4) u = __ldcs(reinterpret_cast<const float4*>(src) + lane);
        // (the fused packed-projection scan reduces in this same order: lane
        // = float4 group, then the 16-8-4-2-1 butterfly)
        const float ss = warp_sum(sumsq4(u));
        const float inv = rms_inv(ss, N, g.eps);
        if (lane < N4)
          __stcs(reinterpret_cast<float4*>(dst) + lane,
                 make_float4(__fmul_rn(u.x, inv), __fmul_rn(u.y, inv), __fmul_rn(u.z, inv),
                             __fmul_rn(u.w, inv)));
      } else {
        float ss = 0.f;
        for (int n = lane; n < N; n += 32) {
          float x = src[n];
          ss += x * x;
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
    for (int a = ta; a < A; a += kThreads)
      __stcs(o.angle + r * (int64_t)A + a, __ldcs(s + 3 * H + a));
    // z | x slices (columns [0, 2I)): the loads issued above, then the rest
    // four at a time
    if (VEC) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = tid + u * kThreads;
        if (i < Z4) {
          if (i < I4)
            __stcs(z4 + i, v[u]);
          else
            __stcs(x4 + (i - I4), v[u]);
        }
      }
      for (int base = tid + 4 * kThreads; base < Z4; base += 4 * kThreads) {
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
        float x = __ldcs(p + i);
        if (i < I)
          __stcs(o.z + r * (int64_t)I + i, x);
        else
          __stcs(o.x + r * (int64_t)I + (i - I), x);
      }
    }
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

// Adjoint of the preprocess (oarust mamba3.rs, `mamba3_preprocess_backward`),
// HBM-bound streaming like k_preprocess: one 256-thread block per row
// (grid-stride), no block barriers. Every thread first issues its share of the
// z | x copy (the z / x output gradients, 128-bit streaming loads, four in
// flight), then does its own column task while those loads land, then stores
// them. The column tasks are spread over the warps so that no warp chains
// more than one of them: B / C rows from the last warp down (one warp per
// row: the projection row u and gradient row g, one float4 each per lane,
// sum u^2 and sum g u by shuffles, du = s g - s^3 u (sum g u) / N with s the
// forward's inverse RMS), the scalar columns from thread 0, the angle columns
// from the next warp on. Scalar columns, with dt and a_mag recomputed as the
// forward computes them (bounds inclusive):
//   d dt_raw = (g_dt - a_mag g_adt) sigmoid(dt_raw + dt_bias)  (clamp passing),
//   d a_raw  = -dt g_adt sigmoid(a_raw)                       (floor passing),
// trap copied.
__device__ __forceinline__ void pre_bwd_scalar(const PreGeom& g, const float* s, float bias,
                                                const PreGrads& gr, int64_t r, int h,
                                                float* qs) {
  const int H = g.H;
  const float raw = __fadd_rn(__ldcs(s + h), bias);
  const float ar = __ldcs(s + H + h);
  const float gd = __ldcs(gr.dt + r * (int64_t)H + h), ga = __ldcs(gr.adt + r * (int64_t)H + h);
  const float gt = __ldcs(gr.trap + r * (int64_t)H + h);
  const float sp = softplus_f(raw);
  const float dt = fminf(fmaxf(sp, g.dt_min), g.dt_max);
  const float sa = softplus_f(ar);
  const float a_mag = fmaxf(sa, g.a_floor);
  const bool dt_pass = sp >= g.dt_min && sp <= g.dt_max;
  const float draw = dt_pass ? fmaf(-a_mag, ga, gd) * sigmoid_f(raw) : 0.f;
  // the dt_raw column is read back by the dt_bias sum: a normal store
  qs[h] = draw;
  __stcs(qs + H + h, sa >= g.a_floor ? -dt * ga * sigmoid_f(ar) : 0.f);
  __stcs(qs + 2 * H + h, gt);
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 4) k_preprocess_bwd(PreGeom g,
                                                                const float* __restrict__ proj,
                                                                const float* __restrict__ dt_bias,
                                                                PreGrads gr,
                                                                float* __restrict__ gp) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int nwarps = kThreads / 32;
  const int I = g.I, N = g.N, H = g.H, A = g.A, W = g.W;
  const int RG = g.G * g.R;
  const int BC = RG * N;
  // the angle columns start on the warp after the scalar columns' warps
  const int aoff = ((H + 31) / 32 * 32) % kThreads;
  const int ta = tid >= aoff ? tid - aoff : tid - aoff + kThreads;
  for (int64_t r = blockIdx.x; r < g.rows; r += gridDim.x) {
    float* q = gp + r * (int64_t)W;
    const int I4 = I >> 2, Z4 = 2 * I4;
    const float4* z4 = reinterpret_cast<const float4*>(gr.z + r * (int64_t)I);
    const float4* x4 = reinterpret_cast<const float4*>(gr.x + r * (int64_t)I);
    float4* q4 = reinterpret_cast<float4*>(q);
    float4 v[4];
    if (VEC) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = tid + u * kThreads;
        if (i < Z4) v[u] = i < I4 ? __ldcs(z4 + i) : __ldcs(x4 + (i - I4));
      }
    }
    for (int j = nwarps - 1 - warp; j < 2 * RG; j += nwarps) {
      const float* src = proj + r * (int64_t)W + 2 * I + (int64_t)j * N;
      const float* gs = j < RG ? gr.bh + r * (int64_t)BC + (int64_t)j * N
                               : gr.ch + r * (int64_t)BC + (int64_t)(j - RG) * N;
      float* dst = q + 2 * I + (int64_t)j * N;
      if (VEC && N <= 128) {
        const int N4 = N >> 2;
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f), gv = u;
        if (lane < N4) {
          u = __ldcs(reinterpret_cast<const float4*>(src) + lane);
          gv = __ldcs(reinterpret_cast<const float4*>(gs) + lane);
        }
        const float ss = warp_sum(sumsq4(u));
        const float gu = warp_sum(fmaf(gv.w, u.w, fmaf(gv.z, u.z, fmaf(gv.y, u.y, gv.x * u.x))));
        const float inv = rms_inv(ss, N, g.eps);
        const float c = inv * inv * inv * gu / (float)N;
        if (lane < N4)
          __stcs(reinterpret_cast<float4*>(dst) + lane,
                 make_float4(fmaf(-c, u.x, inv * gv.x), fmaf(-c, u.y, inv * gv.y),
                             fmaf(-c, u.z, inv * gv.z), fmaf(-c, u.w, inv * gv.w)));
      } else {
        float ss = 0.f, gu = 0.f;
        for (int n = lane; n < N; n += 32) {
          const float x = src[n];
          ss = fmaf(x, x, ss);
          gu = fmaf(gs[n], x, gu);
        }
        ss = warp_sum(ss);
        gu = warp_sum(gu);
        const float inv = rms_inv(ss, N, g.eps);
        const float c = inv * inv * inv * gu / (float)N;
        for (int n = lane; n < N; n += 32) __stcs(dst + n, fmaf(-c, src[n], inv * gs[n]));
      }
    }
    const float* s = proj + r * (int64_t)W + 2 * I + 2 * BC;
    float* qs = q + 2 * I + 2 * BC;
    for (int h = tid; h < H; h += kThreads) pre_bwd_scalar(g, s, __ldg(dt_bias + h), gr, r, h, qs);
    for (int a = ta; a < A; a += kThreads)
      __stcs(qs + 3 * H + a, __ldcs(gr.angle + r * (int64_t)A + a));
    if (VEC) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = tid + u * kThreads;
        if (i < Z4) __stcs(q4 + i, v[u]);
      }
      for (int base = tid + 4 * kThreads; base < Z4; base += 4 * kThreads) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = base + u * kThreads;
          if (i < Z4) v[u] = i < I4 ? __ldcs(z4 + i) : __ldcs(x4 + (i - I4));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = base + u * kThreads;
          if (i < Z4) __stcs(q4 + i, v[u]);
        }
      }
    } else {
      for (int i = tid; i < 2 * I; i += kThreads)
        __stcs(q + i, i < I ? __ldcs(gr.z + r * (int64_t)I + i)
                            : __ldcs(gr.x + r * (int64_t)I + (i - I)));
    }
  }
  // the dt_bias partial pass may be scheduled now (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;");
}

// d dt_bias[h] = sum over rows of d dt_raw[row, h], in a fixed order that
// depends on the row count alone, in two passes of one round of loads each.
// k_pre_bias_part: one block per (chunk of rows, 32 heads), lane = head; warp
// w adds rows [w c, (w + 1) c) of the chunk (c = chunk / 8, sixteen loads in
// flight at a time) in row order, then thread (0, lane) adds the eight warp
// sums in order. k_pre_bias_sum: one 1024-thread block per 32 heads; warp w
// adds partials [w per, (w + 1) per) in order, then thread (0, lane) adds the
// 32 warp sums in order. Both are launched as programmatic dependents of the
// kernel before them and wait for it before reading.
constexpr int kBiasUnroll = 16;
constexpr int kBiasChunk = 128;  // rows per partial, at least
__global__ void __launch_bounds__(kThreads) k_pre_bias_part(PreGeom g, const float* __restrict__ gp,
                                                            int64_t chunk, int hblocks,
                                                            float* __restrict__ part) {
  __shared__ float sw[kThreads / 32][33];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = blockIdx.x / hblocks;
  const int h = (int)(blockIdx.x - c * hblocks) * 32 + lane;
  const int64_t per = chunk / (kThreads / 32);
  const int64_t r0 = c * chunk + warp * per;
  int64_t r1 = r0 + per;
  if (r1 > g.rows) r1 = g.rows;
  const float* col = gp + 2 * (int64_t)g.I + 2 * (int64_t)g.G * g.R * g.N + h;
  float acc = 0.f;
  if (h < g.H)
    for (int64_t rb = r0; rb < r1; rb += kBiasUnroll) {
      float v[kBiasUnroll];
#pragma unroll
      for (int u = 0; u < kBiasUnroll; ++u) v[u] = rb + u < r1 ? col[(rb + u) * g.W] : 0.f;
#pragma unroll
      for (int u = 0; u < kBiasUnroll; ++u) acc += v[u];
    }
  sw[warp][lane] = acc;
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;");
  if (warp == 0 && h < g.H) {
    float t = sw[0][lane];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) t += sw[w][lane];
    part[c * g.H + h] = t;
  }
}

constexpr int kSumThreads = 1024;
__global__ void __launch_bounds__(kSumThreads) k_pre_bias_sum(int H, int64_t nparts,
                                                              const float* __restrict__ part,
                                                              float* __restrict__ out) {
  __shared__ float sw[kSumThreads / 32][33];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.x * 32 + lane;
  const int64_t per = (nparts + kSumThreads / 32 - 1) / (kSumThreads / 32);
  const int64_t c0 = warp * per, c1 = c0 + per < nparts ? c0 + per : nparts;
  float acc = 0.f;
  if (h < H)
    for (int64_t cb = c0; cb < c1; cb += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = cb + u < c1 ? part[(cb + u) * H + h] : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) acc += v[u];
    }
  sw[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && h < H) {
    float t = sw[0][lane];
    for (int w = 1; w < kSumThreads / 32; ++w) t += sw[w][lane];
    out[h] = t;
  }
}

// rows per dt_bias partial: 128, or a larger multiple of 128 so that there are
// at most 1024 partials (the sum kernel's 32 warps then take at most 32 each)
int64_t bias_chunk_rows(int64_t rows) {
  int64_t c = (rows + 1023) / 1024;
  c = (c + kBiasChunk - 1) / kBiasChunk * kBiasChunk;
  return c < kBiasChunk ? kBiasChunk : c;
}

// Launch configuration of a programmatic dependent of the previous kernel on
// the stream (the kernel waits for it with griddepcontrol.wait before reading
// its results). Used in place: cfg points at the object's own attribute.
struct PdlLaunch {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg;
  PdlLaunch(unsigned grid, unsigned block, cudaStream_t s) : cfg{} {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  PdlLaunch(const PdlLaunch&) = delete;
};

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

size_t preprocess_backward_workspace_bytes(const PreGeom& g) {
  const int64_t chunk = bias_chunk_rows(g.rows);
  return (size_t)((g.rows + chunk - 1) / chunk) * g.H * sizeof(float);
}

cudaError_t launch_preprocess_backward(const PreGeom& g, const float* projected,
                                       const float* dt_bias, const PreGrads& gr, float* gproj,
                                       float* gdt_bias, float* partial, cudaStream_t s) {
  const bool vec = (g.W % 4 == 0) && (g.I % 4 == 0) && (g.N % 4 == 0);
  const int64_t blocks = g.rows < (int64_t)(1 << 20) ? g.rows : (int64_t)(1 << 20);
  if (vec)
    k_preprocess_bwd<true><<<(unsigned)blocks, kThreads, 0, s>>>(g, projected, dt_bias, gr, gproj);
  else
    k_preprocess_bwd<false><<<(unsigned)blocks, kThreads, 0, s>>>(g, projected, dt_bias, gr, gproj);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t chunk = bias_chunk_rows(g.rows);
  const int64_t nchunk = (g.rows + chunk - 1) / chunk;
  const int hblocks = (g.H + 31) / 32;
  if (nchunk * hblocks > 0x7fffffff) return cudaErrorInvalidValue;
  PdlLaunch part(static_cast<unsigned>(nchunk * hblocks), kThreads, s);
  e = cudaLaunchKernelEx(&part.cfg, k_pre_bias_part, g, static_cast<const float*>(gproj), chunk,
                         hblocks, partial);
  if (e != cudaSuccess) return e;
  PdlLaunch sum(static_cast<unsigned>(hblocks), kSumThreads, s);
  e = cudaLaunchKernelEx(&sum.cfg, k_pre_bias_sum, static_cast<int>(g.H), nchunk,
                         static_cast<const float*>(partial), gdt_bias);
  count_launches(3);
  return e;
}

}  // namespace m3
