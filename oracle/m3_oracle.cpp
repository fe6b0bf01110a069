// Plain, slow, FP64 CPU oracle for the Mamba-3 selective-state scan.
//
// TEST INFRASTRUCTURE ONLY. This file is the reference that the CUDA library is
// checked against. Only the test suite, the smoke check and the benchmark's CPU
// baseline leg load it; the product path never does. It shares no code, header
// or constant with the CUDA sources.
//
// Source: oarust 0.8.6, `src/rs/ml/matrix/mamba3.rs` (docs.rs source view) and
// the `oa::ml::matrix` API reference. Those pages give the operands, shapes,
// limits, dataflow and docstrings of the Mamba-3 ops but print no formula. Each
// function below names the passage it follows; every step the pages leave open
// is marked READING and is listed, with the alternatives, in the design notes.
//
// Everything is computed in double from the float32 inputs the GPU also gets.
// Parallelism: one std::thread per slice of (batch, head) pairs. No blocking,
// fusion or reordering beyond the token-by-token recurrence itself.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>
#include <functional>

namespace {

using i64 = int64_t;

// Overflow-safe softplus: `softplus` in the `oa::ml::matrix` API reference is
// "the overflow-safe Softplus formulation". log(1 + e^v) is returned as v once
// e^-v is below double rounding.
double softplus(double v) { return v > 36.0 ? v : std::log1p(std::exp(v)); }

double sigmoid(double v) { return 1.0 / (1.0 + std::exp(-v)); }

// SiLU gate, `has_z` in SsmConfig ("Apply the SiLU z gate").
double silu(double v) { return v * sigmoid(v); }

// Runs fn(i) for i in [0, n) on up to `threads` std::threads.
void parallel_for(i64 n, int threads, const std::function<void(i64)>& fn) {
  if (threads <= 1 || n <= 1) {
    for (i64 i = 0; i < n; ++i) fn(i);
    return;
  }
  int t = (int)std::min<i64>(threads, n);
  std::vector<std::thread> pool;
  for (int w = 0; w < t; ++w) {
    pool.emplace_back([=, &fn]() {
      for (i64 i = w; i < n; i += t) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

// READING (rotation pairing): the rotary pairs of the state axis are split-half
// over the first 2A state dims, pair a = (a, a + A), the same convention as the
// `rope` op of the API reference ("split-half rotary"). Dims >= 2A are kept.
// Rotation by theta: (u, v) -> (u cos - v sin, u sin + v cos).
void rotate(std::vector<double>& vec, const std::vector<double>& theta, i64 A) {
  for (i64 a = 0; a < A; ++a) {
    double u = vec[a], v = vec[a + A];
    double c = std::cos(theta[a]), s = std::sin(theta[a]);
    vec[a] = u * c - v * s;
    vec[a + A] = u * s + v * c;
  }
}

struct Ssm {
  i64 B, L, H, G, P, N, A, R;
  int has_z, has_d, has_norm;
};

// Per-token scalars of one (b, t, h): the decay, gamma and scale values the
// backward kernels of mamba3.rs recompute from (adt) and (dt, trap) alone.
// READING (trapezoid gate): lambda = sigmoid(trap) ("raw trapezoidal gates");
// gamma = lambda * dt weights the current token, scale = (1 - lambda) * dt the
// previous one, decay = exp(adt).
struct TokenCoef {
  double decay, gamma, scale;
};

TokenCoef coef(double adt, double dt, double trap) {
  double lam = sigmoid(trap);
  return {std::exp(adt), lam * dt, (1.0 - lam) * dt};
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Fused projection preprocess. Follows `Mamba3PreprocessConfig`,
// `Mamba3PreprocessResult` and `PreprocessGeometry::resolve` of mamba3.rs and the
// `mamba3_preprocess` docstring (packed width 2I + 2GRN + 3H + A).
//
// READING (column order): z, x, B rows, C rows, dt, A, trap, angle - the order
// of the kernel's output bindings (z before x, B before C).
// READING (B/C rows): row j of the G*R rows sits at columns [j*N, (j+1)*N) of the
// B (resp. C) slice; each row is divided by sqrt(mean square + epsilon); no
// weight (the preprocess adjoint returns only d(projected) and d(dt_bias)).
// READING (dt): dt = clamp(softplus(dt_raw + dt_bias[h]), dt_min, dt_max), the
// bounds inclusive ("Inclusive lower/upper bound for transformed dt").
// READING (adt): adt = -max(softplus(a_raw), a_floor) * dt ("positive floor for
// the magnitude of the negative A token"; "negative A-times-dt log decays").
// trap and angle pass through raw ("Raw trapezoidal gates", "Raw rotary angular
// velocities").
// Returns 0, or 1 for an invalid geometry.
int m3o_preprocess(i64 rows, i64 inner, i64 N, i64 H, i64 A, i64 G, i64 R, double eps,
                   double dt_min, double dt_max, double a_floor, const float* projected,
                   const float* dt_bias, double* x, double* z, double* bh, double* ch,
                   double* dt, double* adt, double* trap, double* angle, int threads) {
  if (rows <= 0 || inner <= 0 || N <= 0 || H <= 0 || G <= 0 || R <= 0 || 2 * A > N) return 1;
  const i64 bc = G * R * N;
  const i64 W = 2 * inner + 2 * bc + 3 * H + A;
  const i64 o_b = 2 * inner, o_c = o_b + bc, o_s = o_c + bc;
  parallel_for(rows, threads, [&](i64 r) {
    const float* p = projected + r * W;
    for (i64 i = 0; i < inner; ++i) {
      z[r * inner + i] = p[i];
      x[r * inner + i] = p[inner + i];
    }
    for (int which = 0; which < 2; ++which) {
      const float* src = p + (which == 0 ? o_b : o_c);
      double* dst = (which == 0 ? bh : ch) + r * bc;
      for (i64 j = 0; j < G * R; ++j) {
        double ms = 0.0;
        for (i64 n = 0; n < N; ++n) ms += (double)src[j * N + n] * (double)src[j * N + n];
        ms /= (double)N;
        double inv = 1.0 / std::sqrt(ms + eps);
        for (i64 n = 0; n < N; ++n) dst[j * N + n] = (double)src[j * N + n] * inv;
      }
    }
    for (i64 h = 0; h < H; ++h) {
      double d = softplus((double)p[o_s + h] + (double)dt_bias[h]);
      d = std::min(std::max(d, dt_min), dt_max);
      double a_mag = std::max(softplus((double)p[o_s + H + h]), a_floor);
      dt[r * H + h] = d;
      adt[r * H + h] = -a_mag * d;
      trap[r * H + h] = p[o_s + 2 * H + h];
    }
    for (i64 a = 0; a < A; ++a) angle[r * A + a] = p[o_s + 3 * H + a];
  });
  return 0;
}

// ---------------------------------------------------------------------------
// Adjoint of the fused projection preprocess. Follows
// `Mamba3PreprocessBackward` / `mamba3_preprocess_backward` of mamba3.rs: from
// the projection, dt_bias and the gradients of the eight preprocess outputs
// (x, z, bh, ch, dt, adt, trap, angle, the order of
// `Mamba3PreprocessResult::matrices`), the gradient of the packed projection
// [rows, W] and of dt_bias [H]. The pages give only the kernel's bindings
// (projection, dt_bias and the eight output gradients in; the projection
// gradient and per-(row, head) dt_bias partials out, the partials summed over
// rows by a second kernel), so each step below is the chain rule applied to
// m3o_preprocess above:
//   z, x, trap, angle columns: the output gradient itself (identity slices);
//   B / C row u (N values) -> y = u s, s = 1 / sqrt(mean(u^2) + eps):
//     du_n = s g_n - s^3 u_n (sum_m g_m u_m) / N;
//   dt = clamp(softplus(dt_raw + dt_bias), dt_min, dt_max),
//   adt = -a_mag dt with a_mag = max(softplus(a_raw), a_floor):
//     ddt_total = g_dt - a_mag g_adt;
//     d dt_raw = ddt_total * sigmoid(dt_raw + dt_bias)   while the clamp passes;
//     d a_raw  = -dt g_adt * sigmoid(a_raw)               while the floor passes;
//   d dt_bias[h] = sum over rows of d dt_raw[row, h].
// READING (bounds): the clamp passes the gradient for dt_min <= softplus <=
// dt_max, the floor for softplus(a_raw) >= a_floor (bounds inclusive, as the
// forward's "inclusive" dt bounds; at an exact tie the forward value is the
// same on both sides, so either derivative is a valid one-sided choice).
// Returns 0, or 1 for an invalid geometry.
int m3o_preprocess_backward(i64 rows, i64 inner, i64 N, i64 H, i64 A, i64 G, i64 R, double eps,
                            double dt_min, double dt_max, double a_floor, const float* projected,
                            const float* dt_bias, const float* gx, const float* gz,
                            const float* gbh, const float* gch, const float* gdt,
                            const float* gadt, const float* gtrap, const float* gangle,
                            double* gproj, double* gdt_bias, int threads) {
  if (rows <= 0 || inner <= 0 || N <= 0 || H <= 0 || G <= 0 || R <= 0 || 2 * A > N) return 1;
  const i64 bc = G * R * N;
  const i64 W = 2 * inner + 2 * bc + 3 * H + A;
  const i64 o_b = 2 * inner, o_c = o_b + bc, o_s = o_c + bc;
  parallel_for(rows, threads, [&](i64 r) {
    const float* p = projected + r * W;
    double* gp = gproj + r * W;
    for (i64 i = 0; i < inner; ++i) {
      gp[i] = gz[r * inner + i];
      gp[inner + i] = gx[r * inner + i];
    }
    for (int which = 0; which < 2; ++which) {
      const float* src = p + (which == 0 ? o_b : o_c);
      const float* g = (which == 0 ? gbh : gch) + r * bc;
      double* dst = gp + (which == 0 ? o_b : o_c);
      for (i64 j = 0; j < G * R; ++j) {
        double ms = 0.0, gu = 0.0;
        for (i64 n = 0; n < N; ++n) {
          const double u = src[j * N + n];
          ms += u * u;
          gu += (double)g[j * N + n] * u;
        }
        ms /= (double)N;
        const double s = 1.0 / std::sqrt(ms + eps);
        for (i64 n = 0; n < N; ++n)
          dst[j * N + n] = s * (double)g[j * N + n] - s * s * s * (double)src[j * N + n] * gu / (double)N;
      }
    }
    for (i64 h = 0; h < H; ++h) {
      const double raw = (double)p[o_s + h] + (double)dt_bias[h];
      const double sp = softplus(raw);
      const double dt = std::min(std::max(sp, dt_min), dt_max);
      const double sa = softplus((double)p[o_s + H + h]);
      const double a_mag = std::max(sa, a_floor);
      const double g_dt = (double)gdt[r * H + h], g_adt = (double)gadt[r * H + h];
      const bool dt_pass = sp >= dt_min && sp <= dt_max;
      const bool a_pass = sa >= a_floor;
      gp[o_s + h] = dt_pass ? (g_dt - a_mag * g_adt) * sigmoid(raw) : 0.0;
      gp[o_s + H + h] = a_pass ? -dt * g_adt * sigmoid((double)p[o_s + H + h]) : 0.0;
      gp[o_s + 2 * H + h] = gtrap[r * H + h];
    }
    for (i64 a = 0; a < A; ++a) gp[o_s + 3 * H + a] = gangle[r * A + a];
  });
  for (i64 h = 0; h < H; ++h) {
    double s = 0.0;
    for (i64 r = 0; r < rows; ++r) s += gproj[r * W + o_s + h];
    gdt_bias[h] = s;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// SISO / MIMO selective-state recurrence, token by token.
//
// Follows `mamba3_siso` / `mamba3_mimo` (operand layouts C/B [B,L,R*G,N],
// x/z/out [B,L,H,P], adt/dt/trap [B,L,H], angle [B,L,A], biases [H,R,N],
// D [H], mimo_x/z/o [H,R,P], norm_weight [H,P]; R = 1 for SISO), the
// `SsmConfig` field docs, and the dataflow of the backward "prepare" and
// "state" kernels, which recompute c_rot/b_rot (per head), theta [BH,L,A], qk,
// decay, gamma and scale, and read the previous state, decay and gamma to form
// the output.
//
// Per (b, h), with h_0 = 0, previous key/value 0, theta_{-1} = 0:
//   theta_t[a] = theta_{t-1}[a] + dt_t * angle_t[a]      (READING: linear cumsum;
//               "cumulative angle" is the step state)
//   q_{t,r} = Rot(theta_t)(C_t[row(g,r)] + c_bias[h,r]),
//   k_{t,r} = Rot(theta_t)(B_t[row(g,r)] + b_bias[h,r])    (bias before rotation)
//   x_{t,r} = x_t * mimo_x[h,r]   (SISO: x_t)
//   h_t = decay_t * h_{t-1} + scale_t * decay_t * sum_r x_{t-1,r} k_{t-1,r}^T
//                            + gamma_t * sum_r x_{t,r} k_{t,r}^T
//        READING: exponential-trapezoidal update; the previous-token term
//        carries the current decay.
//   y_{t,r} = h_t q_{t,r} + D[h] x_{t,r}                   (READING: D before gate)
//   SISO: out_t = y_t * silu(z_t)
//   MIMO: o_t = sum_r mimo_o[h,r] * y_{t,r} * silu(z_t * mimo_z[h,r])
//         then, if has_output_norm, o_t / sqrt(mean_p o_t^2 + 1e-5) * norm_weight[h]
//         (READING: per-rank gate, then the mimo_o contraction, then the norm;
//         epsilon 1.0e-5 is the push constant of the MIMO dispatch).
// Head h reads group g = h / (H / G) (READING: contiguous heads per group);
// num_groups == 0 means G = H ("A zero num_groups means one Q/K group per head").
// B/C row of (g, r) is g * R + r (READING: "Number of B/C rows per group").
//
// Optional recurrent state (all may be null, then zero in / not written):
//   ssm [B,H,P,N], angle_state [B,H,A], k_state [B,H,R,N], v_state [B,H,R,P],
// the `mamba3_siso_step` / `mamba3_mimo_step` state layouts. k_state holds the
// rotated, biased key of the last token, v_state its (rank-scaled) value.
// When state_in_out is nonzero the states are read first and written back.
// Returns 0, or 1 for an invalid geometry.
int m3o_scan(i64 B, i64 L, i64 H, i64 num_groups, i64 P, i64 N, i64 A, i64 R, int has_z,
             int has_d, int has_norm, const float* c, const float* b, const float* x,
             const float* z, const float* adt, const float* dt, const float* trap,
             const float* angle, const float* c_bias, const float* b_bias, const float* d,
             const float* mimo_x, const float* mimo_z, const float* mimo_o,
             const float* norm_weight, double* out, double* ssm, double* angle_state,
             double* k_state, double* v_state, int threads) {
  const i64 G = num_groups == 0 ? H : num_groups;
  if (B <= 0 || L <= 0 || H <= 0 || G <= 0 || H % G != 0 || P <= 0 || N <= 0 || A < 0 ||
      2 * A > N || R <= 0)
    return 1;
  const i64 heads_per_group = H / G;
  const i64 RG = R * G;
  parallel_for(B * H, threads, [&](i64 bh_idx) {
    const i64 bb = bh_idx / H, h = bh_idx % H, g = h / heads_per_group;
    std::vector<double> state(P * N, 0.0), theta(A, 0.0);
    std::vector<double> k_prev(R * N, 0.0), v_prev(R * P, 0.0);
    if (ssm) {
      for (i64 i = 0; i < P * N; ++i) state[i] = ssm[bh_idx * P * N + i];
      for (i64 a = 0; a < A; ++a) theta[a] = angle_state[bh_idx * A + a];
      for (i64 i = 0; i < R * N; ++i) k_prev[i] = k_state[bh_idx * R * N + i];
      for (i64 i = 0; i < R * P; ++i) v_prev[i] = v_state[bh_idx * R * P + i];
    }
    std::vector<double> q(R * N), k(R * N), v(R * P), tmp(N), y(R * P), o(P);
    for (i64 t = 0; t < L; ++t) {
      const i64 tok = bb * L + t;           // [B, L] index
      const i64 sc = tok * H + h;           // [B, L, H] index
      const TokenCoef cf = coef(adt[sc], dt[sc], trap[sc]);
      for (i64 a = 0; a < A; ++a) theta[a] += (double)dt[sc] * (double)angle[tok * A + a];
      for (i64 r = 0; r < R; ++r) {
        const i64 row = tok * RG + g * R + r;
        for (i64 n = 0; n < N; ++n) tmp[n] = (double)c[row * N + n] + (double)c_bias[(h * R + r) * N + n];
        rotate(tmp, theta, A);
        for (i64 n = 0; n < N; ++n) q[r * N + n] = tmp[n];
        for (i64 n = 0; n < N; ++n) tmp[n] = (double)b[row * N + n] + (double)b_bias[(h * R + r) * N + n];
        rotate(tmp, theta, A);
        for (i64 n = 0; n < N; ++n) k[r * N + n] = tmp[n];
        for (i64 p = 0; p < P; ++p) {
          double xv = (double)x[sc * P + p];
          v[r * P + p] = mimo_x ? xv * (double)mimo_x[(h * R + r) * P + p] : xv;
        }
      }
      for (i64 p = 0; p < P; ++p) {
        for (i64 n = 0; n < N; ++n) {
          double prev_term = 0.0, cur_term = 0.0;
          for (i64 r = 0; r < R; ++r) {
            prev_term += v_prev[r * P + p] * k_prev[r * N + n];
            cur_term += v[r * P + p] * k[r * N + n];
          }
          double& hs = state[p * N + n];
          hs = cf.decay * hs + cf.scale * cf.decay * prev_term + cf.gamma * cur_term;
        }
      }
      for (i64 r = 0; r < R; ++r) {
        for (i64 p = 0; p < P; ++p) {
          double acc = 0.0;
          for (i64 n = 0; n < N; ++n) acc += state[p * N + n] * q[r * N + n];
          if (has_d) acc += (double)d[h] * v[r * P + p];
          y[r * P + p] = acc;
        }
      }
      if (!mimo_o) {
        // SISO readout and gate.
        for (i64 p = 0; p < P; ++p) {
          double val = y[p];
          if (has_z) val *= silu((double)z[sc * P + p]);
          out[sc * P + p] = val;
        }
      } else {
        for (i64 p = 0; p < P; ++p) {
          double acc = 0.0;
          for (i64 r = 0; r < R; ++r) {
            double val = y[r * P + p];
            if (has_z) val *= silu((double)z[sc * P + p] * (double)mimo_z[(h * R + r) * P + p]);
            acc += (double)mimo_o[(h * R + r) * P + p] * val;
          }
          o[p] = acc;
        }
        if (has_norm) {
          double ms = 0.0;
          for (i64 p = 0; p < P; ++p) ms += o[p] * o[p];
          ms /= (double)P;
          double inv = 1.0 / std::sqrt(ms + 1.0e-5);
          for (i64 p = 0; p < P; ++p) o[p] = o[p] * inv * (double)norm_weight[h * P + p];
        }
        for (i64 p = 0; p < P; ++p) out[sc * P + p] = o[p];
      }
      k_prev = k;
      v_prev = v;
    }
    if (ssm) {
      for (i64 i = 0; i < P * N; ++i) ssm[bh_idx * P * N + i] = state[i];
      for (i64 a = 0; a < A; ++a) angle_state[bh_idx * A + a] = theta[a];
      for (i64 i = 0; i < R * N; ++i) k_state[bh_idx * R * N + i] = k_prev[i];
      for (i64 i = 0; i < R * P; ++i) v_state[bh_idx * R * P + i] = v_prev[i];
    }
  });
  return 0;
}

// ---------------------------------------------------------------------------
// SISO adjoints: reverse-mode differentiation of the token loop of m3o_scan
// (R = 1, zero initial state), returning the eleven gradients of `SsmBackward`
// in mamba3.rs (`mamba3_siso_backward`: c, b, x, z, adt, dt, trap, angle,
// c_bias, b_bias, d) in the layouts of the forward operands: c/b [B,L,G,N],
// x/z [B,L,H,P], adt/dt/trap [B,L,H], angle [B,L,A], c_bias/b_bias [H,N],
// d [H]. dout [B,L,H,P] is the gradient of the scan's output.
//
// The forward pass of each (b, h) is re-run and every state h_t kept; the
// reverse pass then walks t = L-1 .. 0 and takes the adjoint of each forward
// statement in reverse order (the chain rule written out, nothing fused):
//   out_t = y_t * silu(z_t):  dy_t = dout_t silu(z_t),  dz_t = dout_t y_t silu'(z_t)
//   y_t = h_t q_t + D v_t:    Lam_t += dy_t q_t^T,  dq_t = h_t^T dy_t,
//                             dD += dy_t . v_t,  dv_t += D dy_t
//   h_t = a_t h_{t-1} + s_t a_t v_{t-1} k_{t-1}^T + g_t v_t k_t^T:
//       da_t = <Lam_t, h_{t-1} + s_t v_{t-1} k_{t-1}^T>,
//       ds_t = a_t <Lam_t, v_{t-1} k_{t-1}^T>,  dg_t = <Lam_t, v_t k_t^T>,
//       dv_t += g_t Lam_t k_t,  dk_t += g_t Lam_t^T v_t,
//       dv_{t-1} += s_t a_t Lam_t k_{t-1},  dk_{t-1} += s_t a_t Lam_t^T v_{t-1},
//       Lam_{t-1} = a_t Lam_t
//   a_t = exp(adt_t), g_t = sigmoid(trap_t) dt_t, s_t = (1 - sigmoid(trap_t)) dt_t
//   q_t = Rot(theta_t)(C_t + c_bias), k_t = Rot(theta_t)(B_t + b_bias):
//       d(C_t + c_bias) = Rot(theta_t)^T dq_t, and d theta_t[a] from both pairs
//   theta_t = theta_{t-1} + dt_t angle_t: the running adjoint of theta carries
//       back, adding to d dt_t and d angle_t.
// Sums over heads (c, b within a group; angle over all heads) and over batch
// and tokens (c_bias, b_bias, d) are taken after the parallel part, in a fixed
// order. Returns 0, or 1 for an invalid geometry.
int m3o_siso_backward(i64 B, i64 L, i64 H, i64 num_groups, i64 P, i64 N, i64 A, int has_z,
                      int has_d, const float* dout, const float* c, const float* b,
                      const float* x, const float* z, const float* adt, const float* dt,
                      const float* trap, const float* angle, const float* c_bias,
                      const float* b_bias, const float* d, double* gc, double* gb, double* gx,
                      double* gz, double* gadt, double* gdt, double* gtrap, double* gangle,
                      double* gc_bias, double* gb_bias, double* gd, int threads) {
  const i64 G = num_groups == 0 ? H : num_groups;
  if (B <= 0 || L <= 0 || H <= 0 || G <= 0 || H % G != 0 || P <= 0 || N <= 0 || A < 0 ||
      2 * A > N)
    return 1;
  const i64 hpg = H / G;
  // per-head parts, summed below
  std::vector<double> pc(B * L * H * N), pb(B * L * H * N), pang(B * L * H * A);
  std::vector<double> pcb(B * H * N), pbb(B * H * N), pd(B * H);
  parallel_for(B * H, threads, [&](i64 bh) {
    const i64 bb = bh / H, h = bh % H, g = h / hpg;
    const double dd = has_d ? (double)d[h] : 0.0;
    // forward, keeping every state and per-token quantity
    std::vector<double> hs((L + 1) * P * N, 0.0);  // hs[t + 1] = h_t, hs[0] = 0
    std::vector<double> q(L * N), k(L * N), ch(L * N), bhat(L * N), th(L * A), v(L * P);
    std::vector<double> al(L), ga(L), sc(L), lam(L), y(L * P);
    std::vector<double> theta(A, 0.0), tmp(N);
    for (i64 t = 0; t < L; ++t) {
      const i64 tok = bb * L + t, s = tok * H + h;
      const double l = sigmoid((double)trap[s]);
      lam[t] = l;
      al[t] = std::exp((double)adt[s]);
      ga[t] = l * (double)dt[s];
      sc[t] = (1.0 - l) * (double)dt[s];
      for (i64 a = 0; a < A; ++a) theta[a] += (double)dt[s] * (double)angle[tok * A + a];
      for (i64 a = 0; a < A; ++a) th[t * A + a] = theta[a];
      for (i64 n = 0; n < N; ++n) tmp[n] = (double)c[(tok * G + g) * N + n] + (double)c_bias[h * N + n];
      for (i64 n = 0; n < N; ++n) ch[t * N + n] = tmp[n];
      rotate(tmp, theta, A);
      for (i64 n = 0; n < N; ++n) q[t * N + n] = tmp[n];
      for (i64 n = 0; n < N; ++n) tmp[n] = (double)b[(tok * G + g) * N + n] + (double)b_bias[h * N + n];
      for (i64 n = 0; n < N; ++n) bhat[t * N + n] = tmp[n];
      rotate(tmp, theta, A);
      for (i64 n = 0; n < N; ++n) k[t * N + n] = tmp[n];
      for (i64 p = 0; p < P; ++p) v[t * P + p] = (double)x[s * P + p];
      const double* hp = &hs[t * P * N];
      double* hc = &hs[(t + 1) * P * N];
      for (i64 p = 0; p < P; ++p)
        for (i64 n = 0; n < N; ++n) {
          const double prev = t > 0 ? v[(t - 1) * P + p] * k[(t - 1) * N + n] : 0.0;
          hc[p * N + n] = al[t] * hp[p * N + n] + sc[t] * al[t] * prev +
                          ga[t] * v[t * P + p] * k[t * N + n];
        }
      for (i64 p = 0; p < P; ++p) {
        double acc = 0.0;
        for (i64 n = 0; n < N; ++n) acc += hc[p * N + n] * q[t * N + n];
        y[t * P + p] = acc + dd * v[t * P + p];
      }
    }
    // reverse
    std::vector<double> Lam(P * N, 0.0), dv(L * P, 0.0), dk(L * N, 0.0), dq(N), dy(P);
    std::vector<double> gth(A, 0.0);  // running adjoint of theta
    double dsum = 0.0;
    for (i64 t = L - 1; t >= 0; --t) {
      const i64 tok = bb * L + t, s = tok * H + h;
      // out_t = y_t * silu(z_t)
      for (i64 p = 0; p < P; ++p) {
        const double go = (double)dout[s * P + p];
        if (has_z) {
          const double zv = (double)z[s * P + p], sg = sigmoid(zv);
          dy[p] = go * zv * sg;
          gz[s * P + p] = go * y[t * P + p] * (sg + zv * sg * (1.0 - sg));
        } else {
          dy[p] = go;
          gz[s * P + p] = 0.0;
        }
      }
      // y_t = h_t q_t + D v_t
      const double* hc = &hs[(t + 1) * P * N];
      for (i64 n = 0; n < N; ++n) dq[n] = 0.0;
      for (i64 p = 0; p < P; ++p) {
        for (i64 n = 0; n < N; ++n) {
          Lam[p * N + n] += dy[p] * q[t * N + n];
          dq[n] += hc[p * N + n] * dy[p];
        }
        dsum += dy[p] * v[t * P + p];
        dv[t * P + p] += dd * dy[p];
      }
      // h_t = a h_{t-1} + s a v_{t-1} k_{t-1}^T + g v_t k_t^T
      const double* hp = &hs[t * P * N];
      double da = 0.0, ds = 0.0, dg = 0.0;
      for (i64 p = 0; p < P; ++p)
        for (i64 n = 0; n < N; ++n) {
          const double lm = Lam[p * N + n];
          const double prev = t > 0 ? v[(t - 1) * P + p] * k[(t - 1) * N + n] : 0.0;
          da += lm * (hp[p * N + n] + sc[t] * prev);
          ds += al[t] * lm * prev;
          dg += lm * v[t * P + p] * k[t * N + n];
          dv[t * P + p] += ga[t] * lm * k[t * N + n];
          dk[t * N + n] += ga[t] * lm * v[t * P + p];
          if (t > 0) {
            dv[(t - 1) * P + p] += sc[t] * al[t] * lm * k[(t - 1) * N + n];
            dk[(t - 1) * N + n] += sc[t] * al[t] * lm * v[(t - 1) * P + p];
          }
        }
      for (i64 i = 0; i < P * N; ++i) Lam[i] *= al[t];
      // a = exp(adt), g = sigmoid(trap) dt, s = (1 - sigmoid(trap)) dt
      gadt[s] = da * al[t];
      double gdt_t = dg * lam[t] + ds * (1.0 - lam[t]);
      gtrap[s] = (dg - ds) * (double)dt[s] * lam[t] * (1.0 - lam[t]);
      for (i64 p = 0; p < P; ++p) gx[s * P + p] = dv[t * P + p];
      // rotations: q = Rot(theta)(chat), k = Rot(theta)(bhat)
      std::vector<double> dth(A, 0.0);
      for (int which = 0; which < 2; ++which) {
        const double* gr = which == 0 ? dq.data() : &dk[t * N];
        const double* rv = which == 0 ? &q[t * N] : &k[t * N];
        double* dst = which == 0 ? &pc[(tok * H + h) * N] : &pb[(tok * H + h) * N];
        double* bias = which == 0 ? &pcb[bh * N] : &pbb[bh * N];
        for (i64 n = 0; n < N; ++n) dst[n] = gr[n];  // the dims >= 2A pass through
        for (i64 a = 0; a < A; ++a) {
          const double cs = std::cos(th[t * A + a]), sn = std::sin(th[t * A + a]);
          const double g0 = gr[a], g1 = gr[a + A];
          // (u, w) -> (u cs - w sn, u sn + w cs); its transpose on the adjoint
          dst[a] = g0 * cs + g1 * sn;
          dst[a + A] = -g0 * sn + g1 * cs;
          // d/dtheta of the rotated pair (r0, r1) is (-r1, r0)
          dth[a] += -g0 * rv[a + A] + g1 * rv[a];
        }
        for (i64 n = 0; n < N; ++n) bias[n] += dst[n];
      }
      // theta_t = theta_{t-1} + dt_t angle_t
      for (i64 a = 0; a < A; ++a) {
        gth[a] += dth[a];
        gdt_t += gth[a] * (double)angle[tok * A + a];
        pang[(tok * H + h) * A + a] = gth[a] * (double)dt[s];
      }
      gdt[s] = gdt_t;
    }
    pd[bh] = dsum;
  });
  // sums over heads, batch and tokens, in index order
  for (i64 tok = 0; tok < B * L; ++tok) {
    for (i64 g = 0; g < G; ++g)
      for (i64 n = 0; n < N; ++n) {
        double sc_ = 0.0, sb_ = 0.0;
        for (i64 j = 0; j < hpg; ++j) {
          sc_ += pc[(tok * H + g * hpg + j) * N + n];
          sb_ += pb[(tok * H + g * hpg + j) * N + n];
        }
        gc[(tok * G + g) * N + n] = sc_;
        gb[(tok * G + g) * N + n] = sb_;
      }
    for (i64 a = 0; a < A; ++a) {
      double sa = 0.0;
      for (i64 h = 0; h < H; ++h) sa += pang[(tok * H + h) * A + a];
      gangle[tok * A + a] = sa;
    }
  }
  for (i64 h = 0; h < H; ++h) {
    for (i64 n = 0; n < N; ++n) {
      double sc_ = 0.0, sb_ = 0.0;
      for (i64 bb = 0; bb < B; ++bb) {
        sc_ += pcb[(bb * H + h) * N + n];
        sb_ += pbb[(bb * H + h) * N + n];
      }
      gc_bias[h * N + n] = sc_;
      gb_bias[h * N + n] = sb_;
    }
    double sd = 0.0;
    for (i64 bb = 0; bb < B; ++bb) sd += pd[bb * H + h];
    gd[h] = has_d ? sd : 0.0;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// MIMO adjoints: reverse-mode differentiation of the MIMO token loop of
// m3o_scan (rank R, zero initial state), returning the fifteen gradients of
// `Mamba3MimoBackward` in mamba3.rs (`mamba3_mimo_backward`): c, b
// [B,L,R*G,N], x, z [B,L,H,P], adt, dt, trap [B,L,H], angle [B,L,A], c_bias,
// b_bias [H,R,N], d [H], mimo_x, mimo_z, mimo_o [H,R,P], norm_weight [H,P].
// As for the SISO adjoints, every state is kept and each forward statement's
// adjoint is taken in reverse order; the MIMO statements add:
//   out_t = o_t rho_t w (has_norm), rho_t = (mean_p o_t^2 + 1e-5)^(-1/2):
//       d w += dout o rho,  d o = rho w dout - rho^3 o (1/P) sum_j dout_j w_j o_j
//   o_t = sum_r mimo_o[r] y_{t,r} silu(z_t mimo_z[r])   (no gate without has_z):
//       d y_{t,r} = d o mimo_o[r] silu(.),  d mimo_o[r] += d o y_{t,r} silu(.),
//       d z_t += d o mimo_o[r] y_{t,r} silu'(.) mimo_z[r],  d mimo_z[r] += ... z_t
//   v_{t,r} = x_t mimo_x[r]:  d x_t += d v_{t,r} mimo_x[r],  d mimo_x[r] += d v_{t,r} x_t
// and the state terms sum their rank products. Returns 0, or 1 for an invalid
// geometry.
int m3o_mimo_backward(i64 B, i64 L, i64 H, i64 num_groups, i64 P, i64 N, i64 A, i64 R,
                      int has_z, int has_d, int has_norm, const float* dout, const float* c,
                      const float* b, const float* x, const float* z, const float* adt,
                      const float* dt, const float* trap, const float* angle,
                      const float* c_bias, const float* b_bias, const float* d,
                      const float* mimo_x, const float* mimo_z, const float* mimo_o,
                      const float* norm_weight, double* gc, double* gb, double* gx, double* gz,
                      double* gadt, double* gdt, double* gtrap, double* gangle, double* gc_bias,
                      double* gb_bias, double* gd, double* gmx, double* gmz, double* gmo,
                      double* gnw, int threads) {
  const i64 G = num_groups == 0 ? H : num_groups;
  if (B <= 0 || L <= 0 || H <= 0 || G <= 0 || H % G != 0 || P <= 0 || N <= 0 || A < 0 ||
      2 * A > N || R <= 0)
    return 1;
  const i64 hpg = H / G, RG = R * G;
  // per-(b, h) parts, summed below
  std::vector<double> pc(B * L * H * R * N), pb(B * L * H * R * N), pang(B * L * H * A);
  std::vector<double> pcb(B * H * R * N), pbb(B * H * R * N), pd(B * H);
  std::vector<double> pmx(B * H * R * P), pmz(B * H * R * P), pmo(B * H * R * P), pnw(B * H * P);
  parallel_for(B * H, threads, [&](i64 bh) {
    const i64 bb = bh / H, h = bh % H, g = h / hpg;
    const double dd = has_d ? (double)d[h] : 0.0;
    const float* mx = mimo_x + h * R * P;
    const float* mz = mimo_z + h * R * P;
    const float* mo = mimo_o + h * R * P;
    // forward, keeping every state and per-token quantity
    std::vector<double> hs((L + 1) * P * N, 0.0);
    std::vector<double> q(L * R * N), k(L * R * N), th(L * A), v(L * R * P), y(L * R * P);
    std::vector<double> o(L * P), rho(L, 1.0), al(L), ga(L), sc(L), lam(L);
    std::vector<double> theta(A, 0.0), tmp(N);
    for (i64 t = 0; t < L; ++t) {
      const i64 tok = bb * L + t, s = tok * H + h;
      const double l = sigmoid((double)trap[s]);
      lam[t] = l;
      al[t] = std::exp((double)adt[s]);
      ga[t] = l * (double)dt[s];
      sc[t] = (1.0 - l) * (double)dt[s];
      for (i64 a = 0; a < A; ++a) theta[a] += (double)dt[s] * (double)angle[tok * A + a];
      for (i64 a = 0; a < A; ++a) th[t * A + a] = theta[a];
      for (i64 r = 0; r < R; ++r) {
        const i64 row = tok * RG + g * R + r;
        for (i64 n = 0; n < N; ++n) tmp[n] = (double)c[row * N + n] + (double)c_bias[(h * R + r) * N + n];
        rotate(tmp, theta, A);
        for (i64 n = 0; n < N; ++n) q[(t * R + r) * N + n] = tmp[n];
        for (i64 n = 0; n < N; ++n) tmp[n] = (double)b[row * N + n] + (double)b_bias[(h * R + r) * N + n];
        rotate(tmp, theta, A);
        for (i64 n = 0; n < N; ++n) k[(t * R + r) * N + n] = tmp[n];
        for (i64 p = 0; p < P; ++p) v[(t * R + r) * P + p] = (double)x[s * P + p] * (double)mx[r * P + p];
      }
      const double* hp = &hs[t * P * N];
      double* hc = &hs[(t + 1) * P * N];
      for (i64 p = 0; p < P; ++p)
        for (i64 n = 0; n < N; ++n) {
          double prev = 0.0, cur = 0.0;
          for (i64 r = 0; r < R; ++r) {
            if (t > 0) prev += v[((t - 1) * R + r) * P + p] * k[((t - 1) * R + r) * N + n];
            cur += v[(t * R + r) * P + p] * k[(t * R + r) * N + n];
          }
          hc[p * N + n] = al[t] * hp[p * N + n] + sc[t] * al[t] * prev + ga[t] * cur;
        }
      for (i64 r = 0; r < R; ++r)
        for (i64 p = 0; p < P; ++p) {
          double acc = 0.0;
          for (i64 n = 0; n < N; ++n) acc += hc[p * N + n] * q[(t * R + r) * N + n];
          y[(t * R + r) * P + p] = acc + dd * v[(t * R + r) * P + p];
        }
      double ms = 0.0;
      for (i64 p = 0; p < P; ++p) {
        double acc = 0.0;
        for (i64 r = 0; r < R; ++r) {
          double val = y[(t * R + r) * P + p];
          if (has_z) val *= silu((double)z[s * P + p] * (double)mz[r * P + p]);
          acc += (double)mo[r * P + p] * val;
        }
        o[t * P + p] = acc;
        ms += acc * acc;
      }
      if (has_norm) rho[t] = 1.0 / std::sqrt(ms / (double)P + 1.0e-5);
    }
    // reverse
    std::vector<double> Lam(P * N, 0.0), dv(L * R * P, 0.0), dk(L * R * N, 0.0);
    std::vector<double> dq(R * N), dy(R * P), dob(P), gth(A, 0.0);
    double dsum = 0.0;
    for (i64 t = L - 1; t >= 0; --t) {
      const i64 tok = bb * L + t, s = tok * H + h;
      // out_t = o_t rho_t w (or o_t)
      const float* go = dout + s * P;
      if (has_norm) {
        const float* w = norm_weight + h * P;
        double cdot = 0.0;
        for (i64 p = 0; p < P; ++p) cdot += (double)go[p] * (double)w[p] * o[t * P + p];
        cdot /= (double)P;
        const double r3 = rho[t] * rho[t] * rho[t];
        for (i64 p = 0; p < P; ++p) {
          pnw[bh * P + p] += (double)go[p] * o[t * P + p] * rho[t];
          dob[p] = rho[t] * (double)w[p] * (double)go[p] - r3 * o[t * P + p] * cdot;
        }
      } else {
        for (i64 p = 0; p < P; ++p) dob[p] = (double)go[p];
      }
      // o_t = sum_r mimo_o[r] y_{t,r} silu(z_t mimo_z[r])
      for (i64 p = 0; p < P; ++p) {
        double gzp = 0.0;
        for (i64 r = 0; r < R; ++r) {
          const double yv = y[(t * R + r) * P + p], mov = (double)mo[r * P + p];
          double gate = 1.0, dgate = 0.0, arg = 0.0;
          if (has_z) {
            arg = (double)z[s * P + p] * (double)mz[r * P + p];
            const double sg = sigmoid(arg);
            gate = arg * sg;
            dgate = sg + arg * sg * (1.0 - sg);
          }
          dy[r * P + p] = dob[p] * mov * gate;
          pmo[(bh * R + r) * P + p] += dob[p] * yv * gate;
          if (has_z) {
            const double da = dob[p] * mov * yv * dgate;
            gzp += da * (double)mz[r * P + p];
            pmz[(bh * R + r) * P + p] += da * (double)z[s * P + p];
          }
        }
        gz[s * P + p] = gzp;
      }
      // y_{t,r} = h_t q_{t,r} + D v_{t,r}
      const double* hc = &hs[(t + 1) * P * N];
      for (i64 i = 0; i < R * N; ++i) dq[i] = 0.0;
      for (i64 r = 0; r < R; ++r)
        for (i64 p = 0; p < P; ++p) {
          const double dyv = dy[r * P + p];
          for (i64 n = 0; n < N; ++n) {
            Lam[p * N + n] += dyv * q[(t * R + r) * N + n];
            dq[r * N + n] += hc[p * N + n] * dyv;
          }
          dsum += dyv * v[(t * R + r) * P + p];
          dv[(t * R + r) * P + p] += dd * dyv;
        }
      // h_t = a h_{t-1} + s a sum_r v_{t-1,r} k_{t-1,r}^T + g sum_r v_{t,r} k_{t,r}^T
      const double* hp = &hs[t * P * N];
      double da = 0.0, ds = 0.0, dg = 0.0;
      for (i64 p = 0; p < P; ++p)
        for (i64 n = 0; n < N; ++n) {
          const double lm = Lam[p * N + n];
          double prev = 0.0, cur = 0.0;
          for (i64 r = 0; r < R; ++r) {
            if (t > 0) prev += v[((t - 1) * R + r) * P + p] * k[((t - 1) * R + r) * N + n];
            cur += v[(t * R + r) * P + p] * k[(t * R + r) * N + n];
          }
          da += lm * (hp[p * N + n] + sc[t] * prev);
          ds += al[t] * lm * prev;
          dg += lm * cur;
          for (i64 r = 0; r < R; ++r) {
            dv[(t * R + r) * P + p] += ga[t] * lm * k[(t * R + r) * N + n];
            dk[(t * R + r) * N + n] += ga[t] * lm * v[(t * R + r) * P + p];
            if (t > 0) {
              dv[((t - 1) * R + r) * P + p] += sc[t] * al[t] * lm * k[((t - 1) * R + r) * N + n];
              dk[((t - 1) * R + r) * N + n] += sc[t] * al[t] * lm * v[((t - 1) * R + r) * P + p];
            }
          }
        }
      for (i64 i = 0; i < P * N; ++i) Lam[i] *= al[t];
      gadt[s] = da * al[t];
      double gdt_t = dg * lam[t] + ds * (1.0 - lam[t]);
      gtrap[s] = (dg - ds) * (double)dt[s] * lam[t] * (1.0 - lam[t]);
      // v_{t,r} = x_t mimo_x[r]
      for (i64 p = 0; p < P; ++p) {
        double acc = 0.0;
        for (i64 r = 0; r < R; ++r) {
          acc += dv[(t * R + r) * P + p] * (double)mx[r * P + p];
          pmx[(bh * R + r) * P + p] += dv[(t * R + r) * P + p] * (double)x[s * P + p];
        }
        gx[s * P + p] = acc;
      }
      // rotations of every rank's q and k
      std::vector<double> dth(A, 0.0);
      for (i64 r = 0; r < R; ++r)
        for (int which = 0; which < 2; ++which) {
          const double* gr = which == 0 ? &dq[r * N] : &dk[(t * R + r) * N];
          const double* rv = which == 0 ? &q[(t * R + r) * N] : &k[(t * R + r) * N];
          double* dst = (which == 0 ? &pc[0] : &pb[0]) + ((tok * H + h) * R + r) * N;
          double* bias = (which == 0 ? &pcb[0] : &pbb[0]) + (bh * R + r) * N;
          for (i64 n = 0; n < N; ++n) dst[n] = gr[n];
          for (i64 a = 0; a < A; ++a) {
            const double cs = std::cos(th[t * A + a]), sn = std::sin(th[t * A + a]);
            const double g0 = gr[a], g1 = gr[a + A];
            dst[a] = g0 * cs + g1 * sn;
            dst[a + A] = -g0 * sn + g1 * cs;
            dth[a] += -g0 * rv[a + A] + g1 * rv[a];
          }
          for (i64 n = 0; n < N; ++n) bias[n] += dst[n];
        }
      for (i64 a = 0; a < A; ++a) {
        gth[a] += dth[a];
        gdt_t += gth[a] * (double)angle[tok * A + a];
        pang[(tok * H + h) * A + a] = gth[a] * (double)dt[s];
      }
      gdt[s] = gdt_t;
    }
    pd[bh] = dsum;
  });
  // sums over heads, batch and tokens, in index order
  for (i64 tok = 0; tok < B * L; ++tok) {
    for (i64 g = 0; g < G; ++g)
      for (i64 r = 0; r < R; ++r)
        for (i64 n = 0; n < N; ++n) {
          double sc_ = 0.0, sb_ = 0.0;
          for (i64 j = 0; j < hpg; ++j) {
            sc_ += pc[((tok * H + g * hpg + j) * R + r) * N + n];
            sb_ += pb[((tok * H + g * hpg + j) * R + r) * N + n];
          }
          gc[(tok * RG + g * R + r) * N + n] = sc_;
          gb[(tok * RG + g * R + r) * N + n] = sb_;
        }
    for (i64 a = 0; a < A; ++a) {
      double sa = 0.0;
      for (i64 h = 0; h < H; ++h) sa += pang[(tok * H + h) * A + a];
      gangle[tok * A + a] = sa;
    }
  }
  for (i64 h = 0; h < H; ++h) {
    for (i64 i = 0; i < R * N; ++i) {
      double sc_ = 0.0, sb_ = 0.0;
      for (i64 bb = 0; bb < B; ++bb) {
        sc_ += pcb[(bb * H + h) * R * N + i];
        sb_ += pbb[(bb * H + h) * R * N + i];
      }
      gc_bias[h * R * N + i] = sc_;
      gb_bias[h * R * N + i] = sb_;
    }
    for (i64 i = 0; i < R * P; ++i) {
      double sx = 0.0, sz = 0.0, so = 0.0;
      for (i64 bb = 0; bb < B; ++bb) {
        sx += pmx[(bb * H + h) * R * P + i];
        sz += pmz[(bb * H + h) * R * P + i];
        so += pmo[(bb * H + h) * R * P + i];
      }
      gmx[h * R * P + i] = sx;
      gmz[h * R * P + i] = has_z ? sz : 0.0;
      gmo[h * R * P + i] = so;
    }
    for (i64 p = 0; p < P; ++p) {
      double sw = 0.0;
      for (i64 bb = 0; bb < B; ++bb) sw += pnw[(bb * H + h) * P + p];
      gnw[h * P + p] = has_norm ? sw : 0.0;
    }
    double sd = 0.0;
    for (i64 bb = 0; bb < B; ++bb) sd += pd[bb * H + h];
    gd[h] = has_d ? sd : 0.0;
  }
  return 0;
}

}  // extern "C"
