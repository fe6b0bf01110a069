// MIMO adjoints of the Mamba-3 scan (oarust mamba3.rs, `mamba3_mimo_backward`:
// the fifteen gradients of `Mamba3MimoBackward`), FP32 on the CUDA cores.
//
// The MIMO forward adds ranks r < R to the SISO recurrence: q_{t,r}, k_{t,r}
// from the rank's C / B rows, v_{t,r} = x_t mimo_x[r], the state update summing
// the ranks' products, y_{t,r} = h_t q_{t,r} + D v_{t,r}, the per-rank gate and
// the mimo_o contraction o_t = sum_r mimo_o[r] y_{t,r} silu(z_t mimo_z[r]), and
// the output norm out_t = o_t rho_t w. The gradient of y_{t,r} depends on the
// whole row o_t through the norm, so the forward sweep runs twice:
//  * k_mbwd_fwd<..., false>: the state, y_{t,r} for every (t, r) into the
//    workspace (and the running angle, and the state at every tile start);
//  * k_mbwd_out: per token the norm, gate and contraction adjoints: dy_{t,r}
//    (over y_{t,r} in place), dz, and the per-(b, h) sums for mimo_o, mimo_z,
//    norm_weight and D;
//  * k_mbwd_fwd<..., true>: one tile per block, all tiles at once, the state
//    again from the tile's recorded start and dq_{t,r} = h_t^T dy_{t,r}: the
//    C gradient parts, Q_t = sum_r q_{t,r} . dq_{t,r}, the query part of the
//    angle adjoint;
//  * k_mbwd_rev: the adjoint state Lam_t = a_{t+1} Lam_{t+1} + sum_r dy_{t,r}
//    q_{t,r}^T from the last token; with M = a_{t+1} Lam_{t+1}, w_t = g_t +
//    s_{t+1}, and the rank cross products dyv[r'][r] = dy_{t,r'} . v_{t,r},
//    qk[r'][r] = q_{t,r'} . k_{t,r}:
//      dk_{t,r} = w_t M^T v_{t,r} + g_t sum_r' dyv[r'][r] q_{t,r'}
//      dv_{t,r} = w_t M k_{t,r} + g_t sum_r' qk[r'][r] dy_{t,r'} + D dy_{t,r}
//      dg_t = sum_r v_{t,r} . M k_{t,r} + sum_{r,r'} dyv[r'][r] qk[r'][r]
//      ds_{t+1} = sum_r v_{t,r} . M k_{t,r}
//    then dx_t = sum_r dv_{t,r} mimo_x[r], the mimo_x sums, and the running
//    sums for d adt and the angle as in the SISO adjoints;
//  * k_mbwd_finish: d dt, d trap and the ordered sums over heads and batch.
// A tile holds tokens_per_tile(RM, NB) tokens (RM = 1, 2, 4 or 8, the
// instance's rank bound): for N <= 64, 16 when RM = 1, else 32 / RM; for
// N > 64 half of that for RM > 1. The two sweeps run 512 threads (16 warps)
// per (b, h), one block per SM, with the thread layout of the SISO adjoint
// kernels; the query-gradient pass runs 256 threads per (b, h, tile).
#include <algorithm>

#include "k_backward.cuh"

namespace m3 {

struct MBwdWs {
  float *theta, *dthq, *Q, *dgam, *ds, *yd, *dc_h, *db_h, *dang_h;
  float *pcb, *pbb, *pd, *pmx, *pmz, *pmo, *pnw;
  float* ckpt;  // [B H][tiles][Ppad][Npad] the state before each tile's first token
  int out_tb;   // token blocks per sequence of k_mbwd_out (pd, pmz, pmo, pnw per block)
  int tiles;    // tiles per sequence (pcb holds one c_bias sum per (b, h, tile))
};

namespace {

// (the sweeps' column partials, tokens x 16 warps x RM x 64 NB floats, stay
// within 128 KB)
__host__ __device__ constexpr int tokens_per_tile(int RM, int NB) {
  return NB == 1 ? (RM == 1 ? 16 : 32 / RM) : 16 / RM;
}

struct MBwdLayout {
  int Npad, Ppad, AS;
  int q, k, v, dy, y, part, coef, th, cs, sn, dth, red, floats;
};

// tokens_per_tile(RM, NB) tokens per tile, arrays sized for RM >= R ranks. The
// query-gradient kernel (dq) uses neither the readout rows nor the reverse
// sweep's arrays and leaves them out (two of its blocks then fit an SM).
inline MBwdLayout mbwd_layout(int A, int RM, int RPT, int NB, bool dq = false, int warps = 16) {
  MBwdLayout l;
  const int kTM = tokens_per_tile(RM, NB), R = RM;
  l.Npad = 64 * NB;
  l.Ppad = 2 * warps * RPT;
  l.AS = A > 0 ? A : 1;
  int off = 0;
  auto take = [&](int n) {
    const int o = off;
    off += (n + 3) / 4 * 4;
    return o;
  };
  l.q = take(kTM * R * l.Npad);
  l.k = take((kTM + 1) * R * l.Npad);
  l.v = take((kTM + 1) * R * l.Ppad);
  l.dy = take(kTM * R * l.Ppad);
  l.y = take(dq ? 0 : kTM * R * l.Ppad);
  l.part = take(kTM * warps * R * l.Npad);
  l.coef = take(kTM * 8);
  l.th = take(kTM * l.AS);
  l.cs = take(kTM * l.AS);
  l.sn = take(kTM * l.AS);
  l.dth = take(dq ? 0 : kTM * l.AS);
  l.red = take(dq ? 0 : kTM * (2 * R * R + R + 8));
  l.floats = off;
  return l;
}

// Rotated, biased q_{t,r} (into sq[tt R + r]) and k_{t,r} (into
// sk[(tt + koff) R + r]) of the tile's tokens; cos / sin into scs / ssn.
template <int BT>
__device__ __forceinline__ void stage_qk_ranks(const ScanGeom& g, const ScanArgs& a, int b,
                                               int h, int grp, int t0, int tv,
                                               const MBwdLayout& lay, float* sq, float* sk,
                                               int koff, const float* sth, float* scs,
                                               float* ssn) {
  const int N = g.N, A = g.A, U = N - A, R = g.R;
  for (int i = threadIdx.x; i < tv * R * U; i += BT) {
    const int row = i / U, u = i - row * U;  // row = tt R + r
    const int tt = row / R, r = row - tt * R;
    const int64_t src = (((int64_t)b * g.L + t0 + tt) * g.G * R + (int64_t)grp * R + r) * N;
    const float* cb = a.c_bias + ((int64_t)h * R + r) * N;
    const float* bb = a.b_bias + ((int64_t)h * R + r) * N;
    float* qd = sq + row * lay.Npad;
    float* kd = sk + ((tt + koff) * R + r) * lay.Npad;
    if (u < A) {
      float sn, cs;
      sincosf(sth[tt * lay.AS + u], &sn, &cs);
      if (r == 0) {
        scs[tt * lay.AS + u] = cs;
        ssn[tt * lay.AS + u] = sn;
      }
      const float cu = a.c[src + u] + cb[u], cw = a.c[src + u + A] + cb[u + A];
      const float bu = a.b[src + u] + bb[u], bw = a.b[src + u + A] + bb[u + A];
      qd[u] = cu * cs - cw * sn;
      qd[u + A] = cu * sn + cw * cs;
      kd[u] = bu * cs - bw * sn;
      kd[u + A] = bu * sn + bw * cs;
    } else {
      const int n = u + A;
      qd[n] = a.c[src + n] + cb[n];
      kd[n] = a.b[src + n] + bb[n];
    }
  }
}

// Per-token scalars a_t, s_t a_t, g_t (forward sweeps) into scoef, the values
// v_{t,r} = x_t mimo_x[r] into sv[(tt + voff) R + r], and, with dy, the
// workspace's dy_{t,r} into sdy[tt R + r].
template <int BT>
__device__ __forceinline__ void stage_values(const ScanGeom& g, const ScanArgs& a,
                                             const MBwdWs& w, int bh, int b, int h, int t0,
                                             int tv, const MBwdLayout& lay, float* sv, int voff,
                                             float* sdy) {
  const int P = g.P, L = g.L, H = g.H, R = g.R;
  for (int i = threadIdx.x; i < tv * R * P; i += BT) {
    const int row = i / P, p = i - row * P;
    const int tt = row / R, r = row - tt * R;
    const float xv = a.x[(((int64_t)b * L + t0 + tt) * H + h) * P + p];
    sv[((tt + voff) * R + r) * lay.Ppad + p] = xv * a.mimo_x[((int64_t)h * R + r) * P + p];
    if (sdy) sdy[row * lay.Ppad + p] = w.yd[(((int64_t)bh * L + t0 + tt) * R + r) * P + p];
  }
}

}  // namespace

namespace {

// DQ = false: the forward sweep of one (b, h), the state in registers (rows
// of the thread as in the SISO sweeps): each token's y_{t,r}, and the state
// before each tile's first token into the workspace.
// DQ = true: one tile of one (b, h) per block, parallel over tiles: the state
// from that record, the previous token's key and value staged, and each
// token's dq_{t,r} = h_t^T dy_{t,r} with the C gradient parts, Q_t and the
// query part of the angle adjoint.
template <int RPT, int NB, int RM, bool DQ, int BT>
__global__ void __launch_bounds__(BT, DQ ? 2 : 1)
    k_mbwd_fwd(ScanGeom g, ScanArgs a, MBwdWs w, MBwdLayout lay) {
  constexpr int kTM = tokens_per_tile(RM, NB), kW = BT / 32;
  const int R = g.R;
  extern __shared__ __align__(16) float sm[];
  float* sq = sm + lay.q;
  float* sk = sm + lay.k;
  float* sv = sm + lay.v;
  float* sdy = sm + lay.dy;
  float* sy = sm + lay.y;
  float* spart = sm + lay.part;
  float* scoef = sm + lay.coef;
  float* sth = sm + lay.th;
  float* scs = sm + lay.cs;
  float* ssn = sm + lay.sn;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rq = lane >> 4, cq = lane & 15;
  const int P = g.P, N = g.N, A = g.A, L = g.L, H = g.H;
  const int Npad = lay.Npad, Ppad = lay.Ppad, AS = lay.AS;
  const int ntiles = (L + kTM - 1) / kTM;
  const int bh = DQ ? (int)(blockIdx.x / ntiles) : (int)blockIdx.x;
  const int tile_first = DQ ? (int)(blockIdx.x % ntiles) : 0;
  const int tile_end = DQ ? tile_first + 1 : ntiles;
  const int b = bh / H, h = bh % H, grp = h / (H / g.G);
  const int prow0 = warp * 2 * RPT + rq * RPT;
  const float dskip = g.has_d ? a.d[h] : 0.f;

  for (int i = tid; i < lay.part; i += BT) sm[i] = 0.f;
  float hs[RPT][4 * NB];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int e = 0; e < 4 * NB; ++e) hs[i][e] = 0.f;
  if (DQ && tile_first > 0) {
    const float* ck = w.ckpt + ((int64_t)bh * ntiles + tile_first) * Ppad * Npad;
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const float4 v =
            *reinterpret_cast<const float4*>(ck + (prow0 + i) * Npad + 64 * j + 4 * cq);
        hs[i][4 * j] = v.x;
        hs[i][4 * j + 1] = v.y;
        hs[i][4 * j + 2] = v.z;
        hs[i][4 * j + 3] = v.w;
      }
  }
  float th_run = 0.f;
  constexpr int kCb = (RM * 128 + BT - 1) / BT;  // c_bias sums per thread (R Npad <= 128 RM)
  float cbacc[kCb];
#pragma unroll
  for (int j = 0; j < kCb; ++j) cbacc[j] = 0.f;
  __syncthreads();

  for (int tile = tile_first; tile < tile_end; ++tile) {
    const int t0 = tile * kTM, tv = min(kTM, L - t0);
    if (DQ && t0 > 0) {
      // the previous token's value and key into slot 0 (its q row is
      // overwritten by the tile's own staging below)
      for (int u = tid; u < A; u += BT) sth[u] = w.theta[((int64_t)bh * L + t0 - 1) * A + u];
      stage_values<BT>(g, a, w, bh, b, h, t0 - 1, 1, lay, sv, 0, nullptr);
      __syncthreads();
      stage_qk_ranks<BT>(g, a, b, h, grp, t0 - 1, 1, lay, sq, sk, 0, sth, scs, ssn);
      __syncthreads();
    }
    if (tid < tv) {
      const int64_t s = ((int64_t)b * L + t0 + tid) * H + h;
      const float al = expf(a.adt[s]), dtv = a.dt[s], lam = sigmoid_f(a.trap[s]);
      scoef[tid * 8 + 0] = al;
      scoef[tid * 8 + 1] = (1.f - lam) * dtv * al;
      scoef[tid * 8 + 2] = lam * dtv;
    }
    stage_values<BT>(g, a, w, bh, b, h, t0, tv, lay, sv, 1, DQ ? sdy : nullptr);
    if (!DQ && tid < A) {
      for (int tt = 0; tt < tv; ++tt) {
        const int64_t tok = (int64_t)b * L + t0 + tt;
        th_run = fmaf(a.dt[tok * H + h], a.angle[tok * A + tid], th_run);
        sth[tt * AS + tid] = th_run;
        w.theta[((int64_t)bh * L + t0 + tt) * A + tid] = th_run;
      }
    }
    if (DQ)
      for (int i = tid; i < tv * A; i += BT) {
        const int tt = i / A, u = i - tt * A;
        sth[tt * AS + u] = w.theta[((int64_t)bh * L + t0 + tt) * A + u];
      }
    __syncthreads();
    stage_qk_ranks<BT>(g, a, b, h, grp, t0, tv, lay, sq, sk, 1, sth, scs, ssn);
    __syncthreads();
    if constexpr (!DQ) {
      // the state before this tile's first token, for the query-gradient kernel
      if (tile > 0) {
        float* ck = w.ckpt + ((int64_t)bh * ntiles + tile) * Ppad * Npad;
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
          for (int j = 0; j < NB; ++j)
            *reinterpret_cast<float4*>(ck + (prow0 + i) * Npad + 64 * j + 4 * cq) =
                make_float4(hs[i][4 * j], hs[i][4 * j + 1], hs[i][4 * j + 2], hs[i][4 * j + 3]);
      }
      // the next tile's operands into L2 while the recurrence runs
      if (t0 + kTM < L)
        prefetch_tile<BT>(g, a, nullptr, nullptr, bh, b, h, grp, t0 + kTM, min(kTM, L - t0 - kTM));
    }
    for (int tt = 0; tt < tv; ++tt) {
      const float al = scoef[tt * 8], sal = scoef[tt * 8 + 1], gm = scoef[tt * 8 + 2];
#pragma unroll
      for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) hs[i][e] *= al;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float kp[4 * NB], kc[4 * NB], vp[RPT], vc[RPT];
        load_cols<NB>(sk + (tt * R + r) * Npad, cq, kp);
        load_cols<NB>(sk + ((tt + 1) * R + r) * Npad, cq, kc);
        load_rows<RPT>(sv + (tt * R + r) * Ppad + prow0, vp);
        load_rows<RPT>(sv + ((tt + 1) * R + r) * Ppad + prow0, vc);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const float cp = sal * vp[i], cc = gm * vc[i];
#pragma unroll
          for (int e = 0; e < 4 * NB; ++e) hs[i][e] = fmaf(cp, kp[e], fmaf(cc, kc[e], hs[i][e]));
        }
      }
      if constexpr (!DQ) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float qv[4 * NB], yv[RPT];
          load_cols<NB>(sq + (tt * R + r) * Npad, cq, qv);
#pragma unroll
          for (int i = 0; i < RPT; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e) acc = fmaf(hs[i][e], qv[e], acc);
            yv[i] = acc;
          }
          int row;
          const float ysum = rows_sum16<RPT>(yv, cq, row);
          if ((cq & (16 / RPT - 1)) == 0) sy[(tt * R + r) * Ppad + prow0 + row] = ysum;
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float dyr[RPT], dq[4 * NB];
          load_rows<RPT>(sdy + (tt * R + r) * Ppad + prow0, dyr);
#pragma unroll
          for (int e = 0; e < 4 * NB; ++e) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < RPT; ++i) acc = fmaf(hs[i][e], dyr[i], acc);
            dq[e] = acc;
          }
          cols_sum_store<NB>(dq, rq, cq, spart + ((tt * kW + warp) * R + r) * Npad);
        }
      }
    }
    __syncthreads();
    if constexpr (!DQ) {
      // y_{t,r} = h_t q_{t,r} + D v_{t,r} into the workspace
      for (int i = tid; i < tv * R * P; i += BT) {
        const int row = i / P, p = i - row * P;
        const int tt = row / R, r = row - tt * R;
        w.yd[(((int64_t)bh * L + t0 + tt) * R + r) * P + p] =
            fmaf(dskip, sv[((tt + 1) * R + r) * Ppad + p], sy[row * Ppad + p]);
      }
    } else {
      // dq_{t,r}: the warps' column sums, into slot 0
      for (int i = tid; i < tv * R * Npad; i += BT) {
        const int row = i / Npad, n = i - row * Npad;
        const int tt = row / R, r = row - tt * R;
        float* pp = spart + (tt * kW * R + r) * Npad + n;
        float s = pp[0];
#pragma unroll
        for (int x = 1; x < kW; ++x) s += pp[x * R * Npad];
        pp[0] = s;
      }
      __syncthreads();
      // the head's C gradient parts Rot(theta)^T dq_{t,r} and the c_bias sums
      // (thread tid + BT j keeps the sum of (r, n) = that index over R Npad)
#pragma unroll
      for (int j = 0; j < kCb; ++j) {
        const int idx = tid + BT * j;
        if (idx < R * Npad) {
          const int r = idx / Npad, n = idx - r * Npad;
          if (n < N)
            for (int tt = 0; tt < tv; ++tt) {
              const float v = unrotate(spart + (tt * kW * R + r) * Npad, scs + tt * AS,
                                       ssn + tt * AS, n, A);
              w.dc_h[((((int64_t)b * L + t0 + tt) * H + h) * R + r) * N + n] = v;
              cbacc[j] += v;
            }
        }
      }
      // Q_t = sum_r q_{t,r} . dq_{t,r} and the query part of theta_t's adjoint
      for (int tt = warp; tt < tv; tt += kW) {
        float s = 0.f;
        for (int r = 0; r < R; ++r) {
          const float* dq = spart + (tt * kW * R + r) * Npad;
          const float* q = sq + (tt * R + r) * Npad;
          for (int n = lane; n < N; n += 32) s = fmaf(q[n], dq[n], s);
        }
        s = warp_sum(s);
        const int64_t tix = (int64_t)bh * L + t0 + tt;
        if (lane == 0) w.Q[tix] = s;
        for (int u = lane; u < A; u += 32) {
          float d = 0.f;
          for (int r = 0; r < R; ++r) {
            const float* dq = spart + (tt * kW * R + r) * Npad;
            const float* q = sq + (tt * R + r) * Npad;
            d += dq[u + A] * q[u] - dq[u] * q[u + A];
          }
          w.dthq[tix * A + u] = d;
        }
      }
    }
    // this tile's last token becomes the next tile's previous token
    if (tv == kTM) {
      for (int i = tid; i < R * Npad; i += BT) sk[i] = sk[kTM * R * Npad + i];
      for (int i = tid; i < R * Ppad; i += BT) sv[i] = sv[kTM * R * Ppad + i];
    }
    __syncthreads();
  }
  if constexpr (DQ) {
#pragma unroll
    for (int j = 0; j < kCb; ++j) {
      const int idx = tid + BT * j;
      if (idx < R * Npad) {
        const int r = idx / Npad, n = idx - r * Npad;
        if (n < N) w.pcb[(((int64_t)bh * ntiles + tile_first) * R + r) * N + n] = cbacc[j];
      }
    }
  }
}

}  // namespace

namespace {

// Per token of one (b, h) (a warp per token, lane p = lane + 32 j; block
// bh * out_tb + tb takes the tb-th of out_tb equal token ranges): from
// y_{t,r} in the workspace, o_t = sum_r mimo_o[r] y_{t,r} silu(z_t mimo_z[r]),
// the norm's adjoint d o = rho w dout - rho^3 o (1/P) sum_j dout_j w_j o_j (or
// d o = dout), then dy_{t,r} = d o mimo_o[r] silu(.) over y_{t,r}, dz_t, and
// the block's sums for mimo_o, mimo_z, norm_weight and D. P <= 128.
template <int RM, int kJ>  // kJ: P <= 32 kJ
__global__ void __launch_bounds__(kBT) k_mbwd_out(ScanGeom g, ScanArgs a, BwdArgs o,
                                                  MBwdWs w) {
  __shared__ float red[kWarps][RM * 128 + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = g.P, L = g.L, H = g.H, R = g.R;
  const int blk = blockIdx.x, bh = blk / w.out_tb, tb = blk - bh * w.out_tb;
  const int b = bh / H, h = bh % H;
  const int per = (L + w.out_tb - 1) / w.out_tb;
  const int t_end = min(L, (tb + 1) * per);
  float mo[kJ][RM], mz[kJ][RM], mx[kJ][RM], nw[kJ];
  float smo[kJ][RM], smz[kJ][RM], snw[kJ], sd = 0.f;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int p = lane + 32 * j;
    nw[j] = p < P ? a.norm_weight[(int64_t)h * P + p] : 0.f;
    snw[j] = 0.f;
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      const int64_t i = ((int64_t)h * R + r) * P + p;
      if (r >= R) {
        mo[j][r] = mz[j][r] = mx[j][r] = smo[j][r] = smz[j][r] = 0.f;
        continue;
      }
      mo[j][r] = p < P ? a.mimo_o[i] : 0.f;
      mz[j][r] = p < P ? a.mimo_z[i] : 0.f;
      mx[j][r] = p < P ? a.mimo_x[i] : 0.f;
      smo[j][r] = smz[j][r] = 0.f;
    }
  }
  for (int t = tb * per + warp; t < t_end; t += kWarps) {
    const int64_t e0 = (((int64_t)b * L + t) * H + h) * P;
    float* yd = w.yd + ((int64_t)bh * L + t) * R * P;
    // this warp's next token into L2 while this one is formed
    if (t + kWarps < t_end && lane < 4) {
      const int64_t e1 = e0 + (int64_t)kWarps * H * P;
      if (lane == 0) prefetch_range(yd + (int64_t)kWarps * R * P, R * P * 4);
      else if (lane == 1) prefetch_range(a.x + e1, P * 4);
      else if (lane == 2) prefetch_range(o.dout + e1, P * 4);
      else if (g.has_z) prefetch_range(a.z + e1, P * 4);
    }
    float y[kJ][RM], gate[kJ][RM], dgate[kJ][RM], zv[kJ], go[kJ], ov[kJ];
    float ms = 0.f, cdot = 0.f;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int p = lane + 32 * j;
      const bool in = p < P;
      zv[j] = in && g.has_z ? a.z[e0 + p] : 0.f;
      go[j] = in ? o.dout[e0 + p] : 0.f;
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < RM; ++r) {
        y[j][r] = in && r < R ? yd[r * P + p] : 0.f;
        gate[j][r] = 1.f;
        dgate[j][r] = 0.f;
        if (g.has_z) {
          const float arg = zv[j] * mz[j][r], sg = sigmoid_f(arg);
          gate[j][r] = arg * sg;
          dgate[j][r] = sg + arg * sg * (1.f - sg);
        }
        acc = fmaf(mo[j][r], y[j][r] * gate[j][r], acc);
      }
      ov[j] = acc;
      ms = fmaf(acc, acc, ms);
      cdot = fmaf(go[j] * nw[j], acc, cdot);
    }
    float rho = 1.f, r3c = 0.f;
    if (g.has_norm) {
      ms = warp_sum(ms);
      cdot = warp_sum(cdot);
      rho = 1.f / sqrtf(ms / (float)P + 1.0e-5f);
      r3c = rho * rho * rho * (cdot / (float)P);
    }
    float dd = 0.f;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int p = lane + 32 * j;
      if (p >= P) continue;
      float dob = go[j];
      if (g.has_norm) {
        snw[j] = fmaf(go[j] * ov[j], rho, snw[j]);
        dob = rho * nw[j] * go[j] - r3c * ov[j];
      }
      const float xv = a.x[e0 + p];
      float gz = 0.f;
#pragma unroll
      for (int r = 0; r < RM; ++r) {
        if (r >= R) break;
        const float dy = dob * mo[j][r] * gate[j][r];
        yd[r * P + p] = dy;
        smo[j][r] = fmaf(dob * y[j][r], gate[j][r], smo[j][r]);
        if (g.has_z) {
          const float da = dob * mo[j][r] * y[j][r] * dgate[j][r];
          gz = fmaf(da, mz[j][r], gz);
          smz[j][r] = fmaf(da, zv[j], smz[j][r]);
        }
        dd = fmaf(dy, xv * mx[j][r], dd);
      }
      o.gz[e0 + p] = gz;
    }
    sd += dd;
  }
  // the warps' sums, combined in warp order: mimo_o, then mimo_z, then
  // norm_weight and D, through one shared array
  for (int round = 0; round < 3; ++round) {
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int p = lane + 32 * j;
#pragma unroll
      for (int r = 0; r < RM; ++r)
        red[warp][r * 128 + p] = round == 0 ? smo[j][r] : round == 1 ? smz[j][r] : 0.f;
      if (round == 2) red[warp][p] = snw[j];
    }
    if (round == 2) {
      sd = warp_sum(sd);
      if (lane == 0) red[warp][128] = sd;
    }
    __syncthreads();
    if (round < 2) {
      float* dst = round == 0 ? w.pmo : w.pmz;
      for (int i = tid; i < R * P; i += kBT) {
        const int r = i / P, p = i - r * P;
        float s = 0.f;
        for (int x = 0; x < kWarps; ++x) s += red[x][r * 128 + p];
        dst[((int64_t)blk * R + r) * P + p] = s;
      }
    } else {
      for (int p = tid; p < P; p += kBT) {
        float s = 0.f;
        for (int x = 0; x < kWarps; ++x) s += red[x][p];
        w.pnw[(int64_t)blk * P + p] = s;
      }
      if (tid == 0) {
        float s = 0.f;
        for (int x = 0; x < kWarps; ++x) s += red[x][128];
        w.pd[blk] = s;
      }
    }
    __syncthreads();
  }
}

}  // namespace
namespace {

// The reverse sweep of one (b, h) with R ranks (see the file comment).
template <int RPT, int NB, int RM, int BT>
__global__ void __launch_bounds__(BT, 1)
    k_mbwd_rev(ScanGeom g, ScanArgs a, BwdArgs o, MBwdWs w, MBwdLayout lay) {
  constexpr int kTM = tokens_per_tile(RM, NB), kW = BT / 32;
  const int R = g.R;
  extern __shared__ __align__(16) float sm[];
  float* sq = sm + lay.q;
  float* sk = sm + lay.k;
  float* sv = sm + lay.v;
  float* sdy = sm + lay.dy;
  float* smk = sm + lay.y;
  float* spart = sm + lay.part;
  float* scoef = sm + lay.coef;
  float* sth = sm + lay.th;
  float* scs = sm + lay.cs;
  float* ssn = sm + lay.sn;
  float* sdth = sm + lay.dth;
  float* sred = sm + lay.red;  // per token: dyv [R][R], qk [R][R], vmk [R], then 8 scalars
  constexpr int kRed = 2 * RM * RM + RM + 8;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rq = lane >> 4, cq = lane & 15;
  const int P = g.P, N = g.N, A = g.A, L = g.L, H = g.H;
  const int Npad = lay.Npad, Ppad = lay.Ppad, AS = lay.AS;
  const int bh = blockIdx.x, b = bh / H, h = bh % H, grp = h / (H / g.G);
  const int prow0 = warp * 2 * RPT + rq * RPT;
  const float dskip = g.has_d ? a.d[h] : 0.f;

  for (int i = tid; i < lay.part; i += BT) sm[i] = 0.f;
  float lam[RPT][4 * NB];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int e = 0; e < 4 * NB; ++e) lam[i][e] = 0.f;
  float gth = 0.f, cadt = 0.f;
  constexpr int kCb = (RM * 128 + BT - 1) / BT;
  float bbacc[kCb];
#pragma unroll
  for (int j = 0; j < kCb; ++j) bbacc[j] = 0.f;
  // mimo_x sums: thread keeps column p = tid % Ppad for every rank (Ppad divides BT)
  float mxacc[RM];
#pragma unroll
  for (int r = 0; r < RM; ++r) mxacc[r] = 0.f;
  __syncthreads();

  const int ntiles = (L + kTM - 1) / kTM;
  for (int tile = ntiles - 1; tile >= 0; --tile) {
    const int t0 = tile * kTM, tv = min(kTM, L - t0);
    if (tid < tv) {
      const int t = t0 + tid;
      const int64_t s = ((int64_t)b * L + t) * H + h;
      const float dtv = a.dt[s], gm = sigmoid_f(a.trap[s]) * dtv;
      float al1 = 0.f, s1 = 0.f;
      if (t + 1 < L) {
        const int64_t s2 = s + H;
        al1 = expf(a.adt[s2]);
        s1 = (1.f - sigmoid_f(a.trap[s2])) * a.dt[s2];
      }
      scoef[tid * 8 + 0] = al1;
      scoef[tid * 8 + 1] = gm + s1;
      scoef[tid * 8 + 2] = gm;
      scoef[tid * 8 + 3] = s1;
      scoef[tid * 8 + 4] = dtv;
    }
    stage_values<BT>(g, a, w, bh, b, h, t0, tv, lay, sv, 0, sdy);
    for (int i = tid; i < tv * A; i += BT) {
      const int tt = i / A, u = i - tt * A;
      sth[tt * AS + u] = w.theta[((int64_t)bh * L + t0 + tt) * A + u];
    }
    __syncthreads();
    stage_qk_ranks<BT>(g, a, b, h, grp, t0, tv, lay, sq, sk, 0, sth, scs, ssn);
    __syncthreads();
    // the previous tile's operands into L2 while the recurrence runs
    if (t0 > 0) prefetch_tile<BT>(g, a, nullptr, w.theta, bh, b, h, grp, t0 - kTM, kTM, w.yd);
    for (int tt = tv - 1; tt >= 0; --tt) {
      const float al1 = scoef[tt * 8];
#pragma unroll
      for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) lam[i][e] *= al1;  // M
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float kv[4 * NB], vr[RPT], mk[RPT], mv[4 * NB];
        load_cols<NB>(sk + (tt * R + r) * Npad, cq, kv);
        load_rows<RPT>(sv + (tt * R + r) * Ppad + prow0, vr);
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) mv[e] = 0.f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < 4 * NB; ++e) {
            acc = fmaf(lam[i][e], kv[e], acc);
            mv[e] = fmaf(lam[i][e], vr[i], mv[e]);
          }
          mk[i] = acc;
        }
        int row;
        const float msum = rows_sum16<RPT>(mk, cq, row);
        if ((cq & (16 / RPT - 1)) == 0) smk[(tt * R + r) * Ppad + prow0 + row] = msum;
        cols_sum_store<NB>(mv, rq, cq, spart + ((tt * kW + warp) * R + r) * Npad);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float qv[4 * NB], dyr[RPT];
        load_cols<NB>(sq + (tt * R + r) * Npad, cq, qv);
        load_rows<RPT>(sdy + (tt * R + r) * Ppad + prow0, dyr);
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
          for (int e = 0; e < 4 * NB; ++e) lam[i][e] = fmaf(dyr[i], qv[e], lam[i][e]);
      }
    }
    __syncthreads();
    // M^T v_{t,r}: the warps' column sums, into slot 0
    for (int i = tid; i < tv * R * Npad; i += BT) {
      const int row = i / Npad, n = i - row * Npad;
      const int tt = row / R, r = row - tt * R;
      float* pp = spart + (tt * kW * R + r) * Npad + n;
      float s = pp[0];
#pragma unroll
      for (int x = 1; x < kW; ++x) s += pp[x * R * Npad];
      pp[0] = s;
    }
    // the rank cross products of each token: dyv[r'][r] = dy_{r'} . v_r,
    // qk[r'][r] = q_{r'} . k_r
    if constexpr (RM <= 4) {
      // a warp per token: each lane sums its columns of all 2 RM^2 products,
      // then one halving exchange leaves lane l with product l / (32 / V)
      constexpr int V = 2 * RM * RM;
      for (int tt = warp; tt < tv; tt += kW) {
        float v[V];
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] = 0.f;
        for (int p = lane; p < P; p += 32) {
          float dyp[RM], vp[RM];
#pragma unroll
          for (int r = 0; r < RM; ++r) {
            dyp[r] = r < R ? sdy[(tt * R + r) * Ppad + p] : 0.f;
            vp[r] = r < R ? sv[(tt * R + r) * Ppad + p] : 0.f;
          }
#pragma unroll
          for (int r1 = 0; r1 < RM; ++r1)
#pragma unroll
            for (int r = 0; r < RM; ++r) v[r1 * RM + r] = fmaf(dyp[r1], vp[r], v[r1 * RM + r]);
        }
        for (int n = lane; n < N; n += 32) {
          float qn[RM], kn[RM];
#pragma unroll
          for (int r = 0; r < RM; ++r) {
            qn[r] = r < R ? sq[(tt * R + r) * Npad + n] : 0.f;
            kn[r] = r < R ? sk[(tt * R + r) * Npad + n] : 0.f;
          }
#pragma unroll
          for (int r1 = 0; r1 < RM; ++r1)
#pragma unroll
            for (int r = 0; r < RM; ++r)
              v[RM * RM + r1 * RM + r] = fmaf(qn[r1], kn[r], v[RM * RM + r1 * RM + r]);
        }
        int idx = 0, o = 16;
#pragma unroll
        for (int c = V; c > 1; c >>= 1) {
          const bool up = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < c / 2; ++i) {
            const float send = up ? v[i] : v[i + c / 2];
            const float keep = up ? v[i + c / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
          if (up) idx += c / 2;
          o >>= 1;
        }
        float tot = v[0];
#pragma unroll
        for (int x = 32 / V / 2; x > 0; x >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, x);
        if ((lane & (32 / V - 1)) == 0) {
          const int half = idx >= RM * RM, j = idx - half * RM * RM;
          const int r1 = j / RM, r = j - r1 * RM;
          if (r1 < R && r < R) sred[tt * kRed + half * R * R + r1 * R + r] = tot;
        }
      }
    } else {
      // one warp per (token, r', r) pair
      for (int i = warp; i < tv * R * R; i += kW) {
        const int tt = i / (R * R), rr = i - tt * R * R, r1 = rr / R, r = rr - r1 * R;
        float dv = 0.f, qk = 0.f;
        for (int p = lane; p < P; p += 32)
          dv = fmaf(sdy[(tt * R + r1) * Ppad + p], sv[(tt * R + r) * Ppad + p], dv);
        for (int n = lane; n < N; n += 32)
          qk = fmaf(sq[(tt * R + r1) * Npad + n], sk[(tt * R + r) * Npad + n], qk);
        dv = warp_sum(dv);
        qk = warp_sum(qk);
        if (lane == 0) {
          sred[tt * kRed + rr] = dv;
          sred[tt * kRed + R * R + rr] = qk;
        }
      }
    }
    __syncthreads();
    // v_r . M k_r; dg_t, ds_{t+1} and the d adt term
    for (int tt = warp; tt < tv; tt += kW) {
      float vmk_all = 0.f;
      for (int r = 0; r < R; ++r) {
        float s = 0.f;
        for (int p = lane; p < P; p += 32)
          s = fmaf(smk[(tt * R + r) * Ppad + p], sv[(tt * R + r) * Ppad + p], s);
        vmk_all += warp_sum(s);
      }
      if (lane == 0) {
        const int t = t0 + tt;
        const int64_t tix = (int64_t)bh * L + t;
        const float gm = scoef[tt * 8 + 2], s1 = scoef[tt * 8 + 3];
        float cross = 0.f;
        for (int rr = 0; rr < R * R; ++rr)
          cross = fmaf(sred[tt * kRed + rr], sred[tt * kRed + R * R + rr], cross);
        const float dg = vmk_all + cross;
        w.dgam[tix] = dg;
        if (t + 1 < L) w.ds[tix + 1] = vmk_all;
        if (t == 0) w.ds[tix] = 0.f;
        sred[tt * kRed + 2 * R * R + R] = w.Q[tix] - gm * dg - s1 * vmk_all;
      }
    }
    __syncthreads();
    // dk_{t,r} into slot 1; dv_{t,r}, dx_t and the mimo_x sums
    for (int i = tid; i < tv * R * Npad; i += BT) {
      const int row = i / Npad, n = i - row * Npad;
      const int tt = row / R, r = row - tt * R;
      const float* red = sred + tt * kRed;
      float acc = 0.f;
      for (int r1 = 0; r1 < R; ++r1) acc = fmaf(red[r1 * R + r], sq[(tt * R + r1) * Npad + n], acc);
      spart[((tt * kW + 1) * R + r) * Npad + n] =
          fmaf(scoef[tt * 8 + 1], spart[(tt * kW * R + r) * Npad + n], scoef[tt * 8 + 2] * acc);
    }
    {
      const int p = tid % Ppad;
      for (int tt = tid / Ppad; tt < tv; tt += BT / Ppad) {
        if (p >= P) continue;
        const float* red = sred + tt * kRed;
        const int64_t e = (((int64_t)b * L + t0 + tt) * H + h) * P + p;
        const float xv = a.x[e];
        float dx = 0.f;
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          if (r >= R) break;
          float acc = dskip * sdy[(tt * R + r) * Ppad + p];
          for (int r1 = 0; r1 < R; ++r1)
            acc = fmaf(scoef[tt * 8 + 2] * red[R * R + r1 * R + r], sdy[(tt * R + r1) * Ppad + p], acc);
          const float dv = fmaf(scoef[tt * 8 + 1], smk[(tt * R + r) * Ppad + p], acc);
          dx = fmaf(dv, a.mimo_x[((int64_t)h * R + r) * P + p], dx);
          mxacc[r] = fmaf(dv, xv, mxacc[r]);
        }
        o.gx[e] = dx;
      }
    }
    // d adt_t: suffix sums of the tile's terms plus the later tiles' total
    if (warp == 0) {
      float v = lane < tv ? sred[lane * kRed + 2 * R * R + R] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float t = __shfl_down_sync(0xffffffffu, v, off);
        if (lane + off < 32) v += t;
      }
      if (lane < tv) o.gadt[((int64_t)b * L + t0 + lane) * H + h] = cadt + v;
      cadt += __shfl_sync(0xffffffffu, v, 0);
    }
    __syncthreads();
    // the head's B gradient parts Rot(theta)^T dk_{t,r}, the b_bias sums, and
    // theta's adjoint: the query part plus every rank's key part
#pragma unroll
    for (int j = 0; j < kCb; ++j) {
      const int idx = tid + BT * j;
      if (idx < R * Npad) {
        const int r = idx / Npad, n = idx - r * Npad;
        if (n < N)
          for (int tt = 0; tt < tv; ++tt) {
            const float v = unrotate(spart + ((tt * kW + 1) * R + r) * Npad, scs + tt * AS,
                                     ssn + tt * AS, n, A);
            w.db_h[((((int64_t)b * L + t0 + tt) * H + h) * R + r) * N + n] = v;
            bbacc[j] += v;
          }
      }
    }
    for (int i = tid; i < tv * A; i += BT) {
      const int tt = i / A, u = i - tt * A;
      float d = w.dthq[((int64_t)bh * L + t0 + tt) * A + u];
      for (int r = 0; r < R; ++r) {
        const float* dk = spart + ((tt * kW + 1) * R + r) * Npad;
        const float* k = sk + (tt * R + r) * Npad;
        d += dk[u + A] * k[u] - dk[u] * k[u + A];
      }
      sdth[tt * AS + u] = d;
    }
    __syncthreads();
    if (tid < A) {
      for (int tt = tv - 1; tt >= 0; --tt) {
        gth += sdth[tt * AS + tid];
        sdth[tt * AS + tid] = gth;
      }
    }
    __syncthreads();
    for (int i = tid; i < tv * A; i += BT) {
      const int tt = i / A, u = i - tt * A;
      w.dang_h[(((int64_t)b * L + t0 + tt) * H + h) * A + u] = sdth[tt * AS + u] * scoef[tt * 8 + 4];
    }
    for (int tt = warp; tt < tv; tt += kW) {
      const int64_t tok = (int64_t)b * L + t0 + tt;
      float s = 0.f;
      for (int u = lane; u < A; u += 32) s = fmaf(sdth[tt * AS + u], a.angle[tok * A + u], s);
      s = warp_sum(s);
      if (lane == 0) o.gdt[tok * H + h] = s;
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < kCb; ++j) {
    const int idx = tid + BT * j;
    if (idx < R * Npad) {
      const int r = idx / Npad, n = idx - r * Npad;
      if (n < N) w.pbb[((int64_t)bh * R + r) * N + n] = bbacc[j];
    }
  }
  // mimo_x sums: threads sharing a column, in order
#pragma unroll
  for (int r = 0; r < RM; ++r) spart[r * BT + tid] = mxacc[r];
  __syncthreads();
  for (int i = tid; i < R * P; i += BT) {
    const int r = i / P, p = i - r * P;
    float s = 0.f;
    for (int x = p; x < BT; x += Ppad) s += spart[r * BT + x];
    w.pmx[((int64_t)bh * R + r) * P + p] = s;
  }
}

}  // namespace
namespace {

// d dt, d trap, and the ordered sums over heads and batch. Job blockIdx.y: 0
// d dt / d trap, 1 C / B rows of each rank over a group's heads, 2 angle over
// heads, 3 biases over batch, 4 D over batch, 5 mimo_x / mimo_z / mimo_o and
// norm_weight over batch.
__global__ void __launch_bounds__(kBT) k_mbwd_finish(ScanGeom g, ScanArgs a, MBwdArgs o,
                                                     MBwdWs w) {
  const int B = g.B, L = g.L, H = g.H, G = g.G, N = g.N, A = g.A, P = g.P, R = g.R;
  const int hpg = H / G;
  const int64_t stride = (int64_t)gridDim.x * kBT;
  const int64_t i0 = (int64_t)blockIdx.x * kBT + threadIdx.x;
  switch (blockIdx.y) {
    case 0:
      for (int64_t i = i0; i < (int64_t)B * L * H; i += stride) {
        const int h = (int)(i % H);
        const int64_t tok = i / H;
        const int b = (int)(tok / L), t = (int)(tok % L);
        const int64_t tix = ((int64_t)b * H + h) * L + t;
        const float dg = w.dgam[tix], ds = w.ds[tix];
        const float lam = sigmoid_f(a.trap[i]), dtv = a.dt[i];
        o.g.gdt[i] += fmaf(lam, dg, (1.f - lam) * ds);
        o.g.gtrap[i] = (dg - ds) * dtv * (lam * (1.f - lam));
      }
      break;
    case 1:
      if (hpg > 1)
        for (int64_t i = i0; i < (int64_t)B * L * G * R * N; i += stride) {
          const int n = (int)(i % N);
          const int64_t q = i / N;
          const int r = (int)(q % R);
          const int64_t q2 = q / R;
          const int grp = (int)(q2 % G);
          const int64_t tok = q2 / G;
          float sc = 0.f, sb = 0.f;
          for (int j = 0; j < hpg; ++j) {
            const int64_t src = ((tok * H + (int64_t)grp * hpg + j) * R + r) * N + n;
            sc += w.dc_h[src];
            sb += w.db_h[src];
          }
          o.g.gc[i] = sc;
          o.g.gb[i] = sb;
        }
      break;
    case 2:
      if (H > 1 && A > 0)
        for (int64_t i = i0; i < (int64_t)B * L * A; i += stride) {
          const int u = (int)(i % A);
          const int64_t tok = i / A;
          float s = 0.f;
          for (int h = 0; h < H; ++h) s += w.dang_h[(tok * H + h) * A + u];
          o.g.gangle[i] = s;
        }
      break;
    case 3:
      for (int64_t i = i0; i < (int64_t)H * R * N; i += stride) {
        const int64_t hh = i / (R * N), rn = i - hh * R * N;
        float sc = 0.f, sb = 0.f;
        for (int b = 0; b < B; ++b) {
          for (int tl = 0; tl < w.tiles; ++tl)
            sc += w.pcb[(((int64_t)b * H + hh) * w.tiles + tl) * R * N + rn];
          sb += w.pbb[(int64_t)b * H * R * N + i];
        }
        o.g.gc_bias[i] = sc;
        o.g.gb_bias[i] = sb;
      }
      break;
    case 4:
      for (int64_t i = i0; i < H; i += stride) {
        float s = 0.f;
        for (int b = 0; b < B; ++b)
          for (int tb = 0; tb < w.out_tb; ++tb) s += w.pd[((int64_t)b * H + i) * w.out_tb + tb];
        o.g.gd[i] = g.has_d ? s : 0.f;
      }
      break;
    default:
      for (int64_t i = i0; i < (int64_t)H * R * P; i += stride) {
        const int64_t hh = i / (R * P), rp = i - hh * R * P;
        float sx = 0.f, sz = 0.f, so = 0.f;
        for (int b = 0; b < B; ++b) {
          sx += w.pmx[(int64_t)b * H * R * P + i];
          for (int tb = 0; tb < w.out_tb; ++tb) {
            const int64_t j = (((int64_t)b * H + hh) * w.out_tb + tb) * R * P + rp;
            sz += w.pmz[j];
            so += w.pmo[j];
          }
        }
        o.gmx[i] = sx;
        o.gmz[i] = g.has_z ? sz : 0.f;
        o.gmo[i] = so;
      }
      for (int64_t i = i0; i < (int64_t)H * P; i += stride) {
        const int64_t hh = i / P, p = i - hh * P;
        float s = 0.f;
        for (int b = 0; b < B; ++b)
          for (int tb = 0; tb < w.out_tb; ++tb)
            s += w.pnw[(((int64_t)b * H + hh) * w.out_tb + tb) * P + p];
        o.gnw[i] = g.has_norm ? s : 0.f;
      }
      break;
  }
}

struct MBwdPlan {
  size_t theta, dthq, Q, dgam, ds, yd, dc_h, db_h, dang_h, pcb, pbb, pd, pmx, pmz, pmo, pnw,
      ckpt, bytes;
  bool own_c, own_ang;
  int out_tb, tiles;
};

MBwdPlan mbwd_plan(const ScanGeom& g) {
  MBwdPlan p{};
  const size_t bh = (size_t)g.B * g.H, BL = (size_t)g.B * g.L, R = (size_t)g.R;
  p.own_c = g.H / g.G > 1;
  p.own_ang = g.H > 1 && g.A > 0;
  size_t off = 0;
  auto take = [&](size_t floats) {
    const size_t o = off;
    off += (floats * 4 + 255) / 256 * 256;
    return o;
  };
  p.theta = take(bh * g.L * g.A);
  p.dthq = take(bh * g.L * g.A);
  p.Q = take(bh * g.L);
  p.dgam = take(bh * g.L);
  p.ds = take(bh * g.L);
  p.yd = take(bh * g.L * R * g.P);
  p.dc_h = take(p.own_c ? BL * g.H * R * g.N : 0);
  p.db_h = take(p.own_c ? BL * g.H * R * g.N : 0);
  p.dang_h = take(p.own_ang ? BL * g.H * g.A : 0);
  // the instance's rank bound and tile length (as launch_mimo_backward picks it)
  const int rm = g.R == 1 ? 1 : g.R == 2 ? 2 : g.R <= 4 ? 4 : 8;
  const int ktm = tokens_per_tile(rm, g.N <= 64 ? 1 : 2);
  p.tiles = (g.L + ktm - 1) / ktm;
  const size_t ppad = g.P <= 32 ? 32 : g.P <= 64 ? 64 : 128, npad = g.N <= 64 ? 64 : 128;
  p.ckpt = take(bh * (size_t)p.tiles * ppad * npad);
  p.pcb = take(bh * (size_t)p.tiles * R * g.N);
  p.pbb = take(bh * R * g.N);
  // k_mbwd_out: about four blocks per SM, ranges of at least 64 tokens
  p.out_tb = (int)std::max<int64_t>(
      1, std::min<int64_t>((g.L + 63) / 64, (4 * 152 + (int64_t)bh - 1) / (int64_t)bh));
  const size_t nb = bh * (size_t)p.out_tb;
  p.pd = take(nb);
  p.pmx = take(bh * R * g.P);
  p.pmz = take(nb * R * g.P);
  p.pmo = take(nb * R * g.P);
  p.pnw = take(nb * g.P);
  p.bytes = off;
  return p;
}

// RPT: rows per thread of the two sweeps (512 threads, 16 warps: P <= 32 RPT);
// the query-gradient pass runs 256-thread blocks, two per SM, with 2 RPT rows
// per thread (the same padded row count, so that the state records match).
constexpr int kSweepBT = 512;

template <int RPT, int NB, int RM>
cudaError_t launch_mbwd(const ScanGeom& g, const ScanArgs& a, const MBwdArgs& o,
                        const MBwdWs& w, cudaStream_t s) {
  constexpr int kSW = kSweepBT / 32;
  const MBwdLayout lay = mbwd_layout(g.A, RM, RPT, NB, false, kSW);
  const MBwdLayout lay_dq = mbwd_layout(g.A, RM, 2 * RPT, NB, true, kWarps);
  const size_t smem = (size_t)lay.floats * sizeof(float);
  const size_t smem_dq = (size_t)lay_dq.floats * sizeof(float);
  {  // the opt-in above 48 KB, for A up to 64 (set on every call: it is per device)
    const int most = mbwd_layout(64, RM, RPT, NB, false, kSW).floats * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_mbwd_fwd<RPT, NB, RM, false, kSweepBT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(
          k_mbwd_fwd<2 * RPT, NB, RM, true, kBT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
          mbwd_layout(64, RM, 2 * RPT, NB, true, kWarps).floats * (int)sizeof(float));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_mbwd_rev<RPT, NB, RM, kSweepBT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = (unsigned)(g.B * g.H);
  k_mbwd_fwd<RPT, NB, RM, false, kSweepBT><<<grid, kSweepBT, smem, s>>>(g, a, w, lay);
  const unsigned out_grid = grid * (unsigned)w.out_tb;
  if (g.P <= 32) k_mbwd_out<RM, 1><<<out_grid, kBT, 0, s>>>(g, a, o.g, w);
  else if (g.P <= 64) k_mbwd_out<RM, 2><<<out_grid, kBT, 0, s>>>(g, a, o.g, w);
  else k_mbwd_out<RM, 4><<<out_grid, kBT, 0, s>>>(g, a, o.g, w);
  k_mbwd_fwd<2 * RPT, NB, RM, true, kBT><<<grid * (unsigned)w.tiles, kBT, smem_dq, s>>>(g, a, w,
                                                                                      lay_dq);
  k_mbwd_rev<RPT, NB, RM, kSweepBT><<<grid, kSweepBT, smem, s>>>(g, a, o.g, w, lay);
  count_launches(4);
  return cudaGetLastError();
}

template <int RM>
cudaError_t launch_mbwd_rank(const ScanGeom& g, const ScanArgs& a, const MBwdArgs& o,
                             const MBwdWs& w, cudaStream_t s) {
  // (P N <= 4096 for MIMO, so N > 64 leaves P < 64)
  const int rpt = g.P <= 32 ? 1 : g.P <= 64 ? 2 : 4;
  const int nb = g.N <= 64 ? 1 : 2;
  switch (rpt * 10 + nb) {
    case 11: return launch_mbwd<1, 1, RM>(g, a, o, w, s);
    case 12: return launch_mbwd<1, 2, RM>(g, a, o, w, s);
    case 21: return launch_mbwd<2, 1, RM>(g, a, o, w, s);
    case 22: return launch_mbwd<2, 2, RM>(g, a, o, w, s);
    case 41: return launch_mbwd<4, 1, RM>(g, a, o, w, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t mimo_backward_workspace_bytes(const ScanGeom& g) { return mbwd_plan(g).bytes; }

cudaError_t launch_mimo_backward(const ScanGeom& g, const ScanArgs& a, const MBwdArgs& o,
                                 void* ws, cudaStream_t s) {
  const MBwdPlan p = mbwd_plan(g);
  char* base = static_cast<char*>(ws);
  auto f = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
  MBwdWs w;
  w.theta = f(p.theta);
  w.dthq = f(p.dthq);
  w.Q = f(p.Q);
  w.dgam = f(p.dgam);
  w.ds = f(p.ds);
  w.yd = f(p.yd);
  w.dc_h = p.own_c ? f(p.dc_h) : o.g.gc;
  w.db_h = p.own_c ? f(p.db_h) : o.g.gb;
  w.dang_h = p.own_ang ? f(p.dang_h) : o.g.gangle;
  w.pcb = f(p.pcb);
  w.pbb = f(p.pbb);
  w.pd = f(p.pd);
  w.pmx = f(p.pmx);
  w.pmz = f(p.pmz);
  w.pmo = f(p.pmo);
  w.pnw = f(p.pnw);
  w.out_tb = p.out_tb;
  w.ckpt = f(p.ckpt);
  w.tiles = p.tiles;
  cudaError_t e;
  // instances for up to 1, 2, 4 or 8 ranks (16 / that many tokens per tile)
  if (g.R == 1) e = launch_mbwd_rank<1>(g, a, o, w, s);
  else if (g.R == 2) e = launch_mbwd_rank<2>(g, a, o, w, s);
  else if (g.R <= 4) e = launch_mbwd_rank<4>(g, a, o, w, s);
  else e = launch_mbwd_rank<8>(g, a, o, w, s);
  if (e != cudaSuccess) return e;
  const int64_t most = std::max<int64_t>(
      {(int64_t)g.B * g.L * g.H, (int64_t)g.B * g.L * g.G * g.R * g.N, (int64_t)g.B * g.L * g.A,
       (int64_t)g.H * g.R * g.N, (int64_t)g.H * g.R * g.P});
  const unsigned blocks = (unsigned)std::min<int64_t>((most + kBT - 1) / kBT, 152 * 8);
  k_mbwd_finish<<<dim3(blocks, 6), kBT, 0, s>>>(g, a, o, w);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace m3
