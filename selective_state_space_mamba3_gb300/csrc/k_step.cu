// Single-token Mamba-3 step with explicit recurrent state (oarust mamba3.rs,
// `mamba3_siso_step` / `mamba3_mimo_step`: ssm [B,H,P,N], cumulative angle
// [B,H,A], previous key [B,H,R,N], previous value [B,H,R,P]).
//
// One 256-thread block per (b, h). The [P, N] state is the only large operand
// (96% of the bytes at decode shapes), so the kernel is an HBM stream over it:
// warp w owns rows p = w, w + 8, ...; lane l owns the float4 at n = 4l (N <= 128
// gives one float4 per lane per row), reads it once with a 128-bit load,
// applies the exponential-trapezoidal update
//   h = decay * h + scale * decay * sum_r v_prev[r][p] k_prev[r][n]
//                 + gamma * sum_r v[r][p] k[r][n]
// and writes it back once, while the readout h . q_r is reduced across the
// warp with shuffles. The rotated q/k rows, the previous key/value and the
// new angle are staged in shared memory first; k/v/angle states are written
// after the block has read their previous values.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct StepSmem {
  float q[8 * 128], k[8 * 128], kp[8 * 128];  // [R][N]
  float v[8 * 128], vp[8 * 128];              // [R][P]
  float y[8 * 128];                           // [R][P] readouts
  float zz[128];
  float theta[64];
  float red[kWarps];
};

template <int RMAX, bool VEC>
__global__ void __launch_bounds__(kThreads) k_step(ScanGeom g, ScanArgs a, StepState st) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  StepSmem& sm = *reinterpret_cast<StepSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / g.H, h = bh % g.H;
  const int grp = h / (g.H / g.G);
  const int P = g.P, N = g.N, A = g.A, R = g.R;
  const int64_t sc = (int64_t)b * g.H + h;  // [B,1,H] index

  // 0. issue the loads of this warp's first group of state rows (one float4 per
  // lane per row, rows p = warp + 8i) so that their latency overlaps staging.
  float* hs = st.ssm + sc * (int64_t)P * N;
  constexpr int kGroup = 4;
  float4 hreg[kGroup];
  if (VEC) {
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int p = warp + kWarps * u;
      if (p < P && lane < (N >> 2)) hreg[u] = __ldcs(reinterpret_cast<const float4*>(hs + (int64_t)p * N) + lane);
    }
  }
  const float dtv = a.dt[sc];
  // 1. cumulative angle theta = angle_state + dt * angle (per head).
  for (int i = tid; i < A; i += kThreads) {
    const float th = st.angle[sc * A + i] + dtv * a.angle[(int64_t)b * A + i];
    sm.theta[i] = th;
    st.angle[sc * A + i] = th;
  }
  __syncthreads();
  // 2. rotated, biased q/k per rank; previous key/value; x, z.
  for (int idx = tid; idx < R * N; idx += kThreads) {
    const int r = idx / N, n = idx - r * N;
    const int64_t row = ((int64_t)b * g.G * R + (int64_t)grp * R + r) * N;
    const float* cb = a.c_bias + ((int64_t)h * R + r) * N;
    const float* bb = a.b_bias + ((int64_t)h * R + r) * N;
    sm.kp[idx] = st.k[(sc * R + r) * N + n];
    if (n < A) {
      float sn, cs;
      sincosf(sm.theta[n], &sn, &cs);
      const float qu = a.c[row + n] + cb[n], qv = a.c[row + n + A] + cb[n + A];
      const float ku = a.b[row + n] + bb[n], kv = a.b[row + n + A] + bb[n + A];
      sm.q[r * N + n] = qu * cs - qv * sn;
      sm.q[r * N + n + A] = qu * sn + qv * cs;
      sm.k[r * N + n] = ku * cs - kv * sn;
      sm.k[r * N + n + A] = ku * sn + kv * cs;
    } else if (n >= 2 * A) {
      sm.q[idx] = a.c[row + n] + cb[n];
      sm.k[idx] = a.b[row + n] + bb[n];
    }
  }
  for (int idx = tid; idx < R * P; idx += kThreads) {
    const int r = idx / P, p = idx - r * P;
    const float xv = a.x[sc * P + p];
    sm.v[idx] = a.mimo_x ? xv * a.mimo_x[((int64_t)h * R + r) * P + p] : xv;
    sm.vp[idx] = st.v[(sc * R + r) * P + p];
  }
  for (int p = tid; p < P; p += kThreads) sm.zz[p] = a.z[sc * P + p];
  __syncthreads();
  // 3. new previous-key / previous-value states (old values already staged).
  for (int idx = tid; idx < R * N; idx += kThreads) st.k[sc * R * N + idx] = sm.k[idx];
  for (int idx = tid; idx < R * P; idx += kThreads) st.v[sc * R * P + idx] = sm.v[idx];

  // 4. state update + readout. Coefficients of the exponential-trapezoidal rule.
  const float lam = sigmoid_f(a.trap[sc]);
  const float decay = expf(a.adt[sc]);
  const float gam = lam * dtv;
  const float sdec = (1.0f - lam) * dtv * decay;
  const float dskip = g.has_d ? a.d[h] : 0.0f;
  // Readout of row p: y_r[p] = sum_n h[p][n] q_r[n] (+ D v_r[p]).
  auto finish_row = [&](int p, const float* acc) {
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const float yv = warp_sum(acc[r]);
        if (lane == 0) sm.y[r * P + p] = yv + dskip * sm.v[r * P + p];
      }
    }
  };
  if (VEC) {
    const int N4 = N >> 2;
    for (int i0 = 0; warp + kWarps * i0 < P; i0 += kGroup) {
      if (i0 > 0) {
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          const int p = warp + kWarps * (i0 + u);
          if (p < P && lane < N4) hreg[u] = __ldcs(reinterpret_cast<const float4*>(hs + (int64_t)p * N) + lane);
        }
      }
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int p = warp + kWarps * (i0 + u);
        if (p >= P) break;
        float acc[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) acc[r] = 0.f;
        if (lane < N4) {
          float4 hv = hreg[u];
          float4 upd = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int r = 0; r < RMAX; ++r) {
            if (r < R) {
              const float cp = sdec * sm.vp[r * P + p], cc = gam * sm.v[r * P + p];
              const float4 kp4 = reinterpret_cast<const float4*>(sm.kp + r * N)[lane];
              const float4 k4 = reinterpret_cast<const float4*>(sm.k + r * N)[lane];
              upd.x += cp * kp4.x + cc * k4.x;
              upd.y += cp * kp4.y + cc * k4.y;
              upd.z += cp * kp4.z + cc * k4.z;
              upd.w += cp * kp4.w + cc * k4.w;
            }
          }
          hv.x = decay * hv.x + upd.x;
          hv.y = decay * hv.y + upd.y;
          hv.z = decay * hv.z + upd.z;
          hv.w = decay * hv.w + upd.w;
          __stcs(reinterpret_cast<float4*>(hs + (int64_t)p * N) + lane, hv);
#pragma unroll
          for (int r = 0; r < RMAX; ++r) {
            if (r < R) {
              const float4 q4 = reinterpret_cast<const float4*>(sm.q + r * N)[lane];
              acc[r] = hv.x * q4.x + hv.y * q4.y + hv.z * q4.z + hv.w * q4.w;
            }
          }
        }
        finish_row(p, acc);
      }
    }
  } else {
    for (int p = warp; p < P; p += kWarps) {
      float acc[RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) acc[r] = 0.f;
      for (int n = lane; n < N; n += 32) {
        float upd = 0.f;
        for (int r = 0; r < R; ++r)
          upd += sdec * sm.vp[r * P + p] * sm.kp[r * N + n] + gam * sm.v[r * P + p] * sm.k[r * N + n];
        const float hv = decay * hs[(int64_t)p * N + n] + upd;
        hs[(int64_t)p * N + n] = hv;
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
          if (r < R) acc[r] += hv * sm.q[r * N + n];
      }
      finish_row(p, acc);
    }
  }
  __syncthreads();
  // 5. gate (SISO) or per-rank gate + mimo_o contraction + output norm (MIMO).
  float* outp = a.out + sc * P;
  if (!a.mimo_o) {
    for (int p = tid; p < P; p += kThreads) {
      const float yv = sm.y[p];
      outp[p] = g.has_z ? yv * silu_f(sm.zz[p]) : yv;
    }
    return;
  }
  float ov = 0.f;
  const int p = tid;
  if (p < P) {
    for (int r = 0; r < R; ++r) {
      float yv = sm.y[r * P + p];
      if (g.has_z) yv *= silu_f(sm.zz[p] * a.mimo_z[((int64_t)h * R + r) * P + p]);
      ov += a.mimo_o[((int64_t)h * R + r) * P + p] * yv;
    }
  }
  if (g.has_norm) {
    float ss = warp_sum(p < P ? ov * ov : 0.f);
    if (lane == 0) sm.red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < kWarps; ++w) tot += sm.red[w];
    const float inv = 1.0f / sqrtf(tot / (float)P + 1.0e-5f);
    if (p < P) ov = ov * inv * a.norm_weight[(int64_t)h * P + p];
  }
  if (p < P) outp[p] = ov;
}

}  // namespace

cudaError_t launch_step(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                        cudaStream_t s) {
  const bool vec = (g.N % 4 == 0);
  const size_t smem = sizeof(StepSmem);
  const unsigned grid = (unsigned)(g.B * g.H);
  cudaError_t e;
#define M3_STEP_LAUNCH(RM, V)                                                              \
  do {                                                                                     \
    e = cudaFuncSetAttribute(k_step<RM, V>, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                             (int)smem);                                                   \
    if (e != cudaSuccess) return e;                                                        \
    k_step<RM, V><<<grid, kThreads, smem, s>>>(g, a, st);                                  \
  } while (0)
  if (g.R == 1) {
    if (vec) M3_STEP_LAUNCH(1, true); else M3_STEP_LAUNCH(1, false);
  } else {
    if (vec) M3_STEP_LAUNCH(8, true); else M3_STEP_LAUNCH(8, false);
  }
#undef M3_STEP_LAUNCH
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace m3
