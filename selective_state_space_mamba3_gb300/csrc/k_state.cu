// Recurrent-state helpers of the chunked scan (oarust mamba3.rs: the step
// state layouts of `mamba3_siso_step` / `mamba3_mimo_step`, and the chunk
// summary -> prefix -> entry-state pattern of the chunked SISO backward).
//
// k_state_init: converts a step state (h [P,N], cumulative angle, previous key
// per rank, previous value per rank) into the chunked scan's "pre-loaded"
// state g = h + scale_0 * sum_r v_prev[r] k_prev[r]^T, where scale_0 is the
// trapezoid weight the first new token puts on the previous one.
//
// k_state_prefix: with a sequence split into segments, segment s's summary
// (its state contribution computed from a zero state with its angles counted
// from zero) is carried into the true entry states:
//   G_entry[s+1] = e_s G_entry[s] + rot(G_sum[s], theta_entry[s]),
//   theta_entry[s+1] = theta_entry[s] + theta_sum[s],
// rot() rotating the rotary pairs (a, a + A) of each state row by the entry
// angle: rotations of a pair compose additively, so a key rotated by
// theta_entry + phi is the summary's key rotated once more by theta_entry.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;

// Grid (b * H + h, block of 16 state rows): one thread per float4 of the rows
// when N % 4 == 0 (every state base is 16-byte aligned by the host checks),
// else per element; the rank sum in rank order.
constexpr int kInitRows = 16;
__global__ void __launch_bounds__(kThreads) k_state_init(ScanGeom g, ScanArgs a, StepState st,
                                                          float* g0, float* th0) {
  const int bh = blockIdx.x;
  const int b = bh / g.H, h = bh % g.H;
  const int P = g.P, N = g.N, A = g.A, R = g.R;
  const int p0 = blockIdx.y * kInitRows, p1 = min(P, p0 + kInitRows);
  const int64_t sc = (int64_t)b * g.L * g.H + h;  // token 0 of batch row b
  const float lam = sigmoid_f(a.trap[sc]);
  const float s0 = (1.0f - lam) * a.dt[sc];
  const float* hs = st.ssm + (int64_t)bh * P * N;
  const float* kp = st.k + (int64_t)bh * R * N;
  const float* vp = st.v + (int64_t)bh * R * P;
  float* gd = g0 + (int64_t)bh * P * N;
  if (N % 4 == 0) {
    const int N4 = N >> 2;
    for (int i = p0 * N4 + threadIdx.x; i < p1 * N4; i += kThreads) {
      const int p = i / N4, n4 = i - p * N4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < R; ++r) {
        const float v = vp[r * P + p];
        const float4 k = reinterpret_cast<const float4*>(kp + r * N)[n4];
        acc.x += v * k.x;
        acc.y += v * k.y;
        acc.z += v * k.z;
        acc.w += v * k.w;
      }
      const float4 hv = reinterpret_cast<const float4*>(hs)[i];
      reinterpret_cast<float4*>(gd)[i] =
          make_float4(hv.x + s0 * acc.x, hv.y + s0 * acc.y, hv.z + s0 * acc.z, hv.w + s0 * acc.w);
    }
  } else {
    for (int i = p0 * N + threadIdx.x; i < p1 * N; i += kThreads) {
      const int p = i / N, n = i - p * N;
      float acc = 0.f;
      for (int r = 0; r < R; ++r) acc += vp[r * P + p] * kp[r * N + n];
      gd[i] = hs[i] + s0 * acc;
    }
  }
  if (blockIdx.y == 0)
    for (int i = threadIdx.x; i < A; i += kThreads)
      th0[(int64_t)bh * A + i] = st.angle ? st.angle[(int64_t)bh * A + i] : 0.f;
}

// Grid (b * H + h, unit block): one thread per unit, a unit being a rotary
// pair (p, a) for a < A or a single column (p, n >= 2A); each thread walks
// the segments in order (the units are independent, so the walks of all units
// of all sequences overlap), writing each segment's entry state and folding in
// the summaries of its `pieces` pieces (summary index (bh * nseg + s) * pieces
// + k for piece k of segment s).
__global__ void __launch_bounds__(kThreads) k_state_prefix(ScanGeom g, int nseg, int pieces,
                                                            const float* g_init,
                                                            const float* th_init,
                                                            const float* gsum,
                                                            const float* thsum,
                                                            const float* esum, float* g_entry,
                                                            float* th_entry) {
  const int bh = blockIdx.x;
  const int P = g.P, N = g.N, A = g.A;
  const int U = N - A;
  const int64_t PN = (int64_t)P * N;
  const int i = blockIdx.y * kThreads + threadIdx.x;
  if (i < P * U) {
    const int p = i / U, u = i - p * U;
    const int n0 = u < A ? u : u + A;  // first column of the unit
    const bool pair = u < A;
    const int64_t row = (int64_t)p * N;
    float x0 = 0.f, x1 = 0.f;
    float th = 0.f;
    if (g_init) {
      x0 = g_init[(int64_t)bh * PN + row + n0];
      if (pair) x1 = g_init[(int64_t)bh * PN + row + n0 + A];
    }
    if (pair && th_init) th = th_init[(int64_t)bh * A + u];
    for (int s = 0; s < nseg; ++s) {
      const int64_t cs = (int64_t)bh * nseg + s;
      float* ge = g_entry + cs * PN + row;
      ge[n0] = x0;
      if (pair) ge[n0 + A] = x1;
      if (p == 0 && pair) th_entry[cs * A + u] = th;
      if (s + 1 == nseg) break;
      for (int k = 0; k < pieces; ++k) {
        const int64_t cp = cs * pieces + k;
        const float e = esum[cp];
        const float* gs = gsum + cp * PN + row;
        if (pair) {
          float sn, c;
          sincosf(th, &sn, &c);
          const float y0 = gs[n0], y1 = gs[n0 + A];
          x0 = e * x0 + (y0 * c - y1 * sn);
          x1 = e * x1 + (y0 * sn + y1 * c);
          th += thsum[cp * A + u];
        } else {
          x0 = e * x0 + gs[n0];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_state_init(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                              float* g0, float* th0, cudaStream_t s) {
  const dim3 grid((unsigned)(g.B * g.H), (unsigned)((g.P + kInitRows - 1) / kInitRows));
  k_state_init<<<grid, kThreads, 0, s>>>(g, a, st, g0, th0);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_state_prefix(const ScanGeom& g, int nseg, int pieces, const float* g_init,
                                const float* th_init, const float* gsum, const float* thsum,
                                const float* esum, float* g_entry, float* th_entry,
                                cudaStream_t s) {
  const dim3 grid((unsigned)(g.B * g.H),
                  (unsigned)max(1, (g.P * (g.N - g.A) + kThreads - 1) / kThreads));
  k_state_prefix<<<grid, kThreads, 0, s>>>(g, nseg, pieces, g_init, th_init, gsum, thsum, esum, g_entry,
                                           th_entry);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace m3
