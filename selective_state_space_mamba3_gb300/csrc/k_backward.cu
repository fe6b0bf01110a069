// SISO adjoints of the Mamba-3 scan (oarust mamba3.rs, `mamba3_siso_backward`:
// the eleven gradients of `SsmBackward`), FP32 on the CUDA cores.
//
// With a_t = exp(adt_t), g_t = sigmoid(trap_t) dt_t, s_t = (1 - sigmoid(trap_t))
// dt_t, q_t / k_t the rotated, biased C / B rows, v_t = x_t and the forward
// recurrence h_t = a_t h_{t-1} + s_t a_t v_{t-1} k_{t-1}^T + g_t v_t k_t^T,
// y_t = h_t q_t + D v_t, out_t = y_t silu(z_t), the adjoints come from two
// token-sequential sweeps per (b, h) and a reduce:
//
//  * forward sweep (k_bwd_fwd): re-runs h_t and reads out y_t (for dz) and
//    dq_t = h_t^T dy_t, dy_t = dout_t silu(z_t); from dq_t the C gradient of
//    the head (dq_t rotated back), Q_t = q_t . dq_t and the query part of the
//    angle adjoint. It saves the running angle theta_t for the reverse sweep.
//  * reverse sweep (k_bwd_rev): the adjoint state Lam_t = a_{t+1} Lam_{t+1} +
//    dy_t q_t^T from the last token down; with M = a_{t+1} Lam_{t+1} and
//    w_t = g_t + s_{t+1}:
//      dk_t = w_t M^T v_t + g_t (dy_t . v_t) q_t
//      dv_t = w_t M k_t + (g_t (q_t . k_t) + D) dy_t
//      dg_t = v_t . M k_t + (dy_t . v_t)(q_t . k_t),  ds_{t+1} = v_t . M k_t
//    and two running sums from the last token: theta's adjoint (which feeds
//    d angle and d dt), and
//      d adt_t = sum_{tau >= t} (Q_tau - g_tau dg_tau - s_{tau+1} ds_{tau+1}),
//    which equals a_t <Lam_t, h_{t-1} + s_t v_{t-1} k_{t-1}^T> (the sum
//    telescopes through Lam_t = a_{t+1} Lam_{t+1} + dy_t q_t^T), so the
//    reverse sweep never needs h_t.
//  * finish (k_bwd_finish): d dt and d trap from dg and ds, and the sums over
//    heads (C / B rows shared by a group's heads, the angle by all heads) and
//    over the batch (c_bias, b_bias, D), each in a fixed order.
//
// Block layout of both sweeps: 256 threads own the [P, N] state; warp w holds
// rows 2 RPT w .. 2 RPT w + 2 RPT - 1, half warp rq the RPT rows from
// 2 RPT w + RPT rq, lane cq of the half the columns 64 j + 4 cq .. + 3
// (j < NB). Row readouts (sums over n) reduce within the half warp; column
// readouts (sums over p) reduce across the half warps by a shuffle and across
// warps through shared memory, once per tile of kT tokens.
#include <algorithm>

#include "k_backward.cuh"

namespace m3 {
namespace {

constexpr int kT = 16;  // tokens per staging tile

// Shared-memory layout (float offsets, 16-byte aligned) for padded sizes
// Npad = 64 NB, Ppad = 16 RPT (P64 N128: 108 KB at A = 32, 112 KB at A = 64,
// two blocks per SM).
struct BwdLayout {
  int Npad, Ppad, AS;
  int q, k, v, dy, y, part, coef, th, cs, sn, dz, dth, red, floats;
};

inline BwdLayout bwd_layout(int A, int RPT, int NB, int warps = kWarps) {
  BwdLayout l;
  l.Npad = 64 * NB;
  l.Ppad = 2 * warps * RPT;
  l.AS = A > 0 ? A : 1;
  int off = 0;
  auto take = [&](int n) {
    const int o = off;
    off += (n + 3) / 4 * 4;
    return o;
  };
  l.q = take(kT * l.Npad);
  l.k = take((kT + 1) * l.Npad);
  l.v = take((kT + 1) * l.Ppad);
  l.dy = take(kT * l.Ppad);
  l.y = take(kT * l.Ppad);
  l.part = take(kT * warps * l.Npad);
  l.coef = take(kT * 8);
  l.th = take(kT * l.AS);
  l.cs = take(kT * l.AS);
  l.sn = take(kT * l.AS);
  // dz (forward sweep) and dth (reverse sweep) share one region
  l.dz = take(kT * (l.Ppad > l.AS ? l.Ppad : l.AS));
  l.dth = l.dz;
  l.red = take(kT * 8);
  l.floats = off;
  return l;
}

// Stages the rotated, biased q_t (into sq[tt]) and k_t (into sk[tt + koff])
// of the tile's tv tokens from the running angles in sth, writing the cosines
// and sines to scs / ssn: q = Rot(theta)(C + c_bias), k = Rot(theta)(B + b_bias),
// split-half pairs (u, u + A) rotated by (u cos - w sin, u sin + w cos).
template <int NB, int BT>
__device__ __forceinline__ void stage_qk(const ScanGeom& g, const ScanArgs& a, int b, int h,
                                         int grp, int t0, int tv, const BwdLayout& lay,
                                         float* sq, float* sk, int koff, const float* sth,
                                         float* scs, float* ssn) {
  constexpr int Npad = 64 * NB;
  const int N = g.N, A = g.A;
  // item (tt, u): u < A the pair (u, u + A), 2A <= u < N the plain dim u
  for (int i = threadIdx.x; i < tv * Npad; i += BT) {
    const int tt = i / Npad, u = i - tt * Npad;
    if ((u >= A && u < 2 * A) || u >= N) continue;
    const int64_t row = (((int64_t)b * g.L + t0 + tt) * g.G + grp) * N;
    const float* cb = a.c_bias + (int64_t)h * N;
    const float* bb = a.b_bias + (int64_t)h * N;
    float* qd = sq + tt * Npad;
    float* kd = sk + (tt + koff) * Npad;
    if (u < A) {
      float sn, cs;
      sincosf(sth[tt * lay.AS + u], &sn, &cs);
      scs[tt * lay.AS + u] = cs;
      ssn[tt * lay.AS + u] = sn;
      const float cu = a.c[row + u] + cb[u], cw = a.c[row + u + A] + cb[u + A];
      const float bu = a.b[row + u] + bb[u], bw = a.b[row + u + A] + bb[u + A];
      qd[u] = cu * cs - cw * sn;
      qd[u + A] = cu * sn + cw * cs;
      kd[u] = bu * cs - bw * sn;
      kd[u + A] = bu * sn + bw * cs;
    } else {
      qd[u] = a.c[row + u] + cb[u];
      kd[u] = a.b[row + u] + bb[u];
    }
  }
}

}  // namespace

// Workspace of the backward (device pointers; see backward_workspace_bytes).
struct BwdWs {
  float *theta, *dthq, *Q, *dgam, *ds, *dc_h, *db_h, *dang_h, *pcb, *pbb, *pd;
};

namespace {

template <int RPT, int NB, int BT>
__global__ void __launch_bounds__(BT, BT > 256 || RPT >= 8 ? 1 : 2)
    k_bwd_fwd(ScanGeom g, ScanArgs a, BwdArgs o, BwdWs w, BwdLayout lay) {
  constexpr int kW = BT / 32;
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
  float* sdz = sm + lay.dz;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rq = lane >> 4, cq = lane & 15;
  const int P = g.P, N = g.N, A = g.A, L = g.L, H = g.H;
  constexpr int Npad = 64 * NB, Ppad = 2 * kW * RPT;
  const int AS = lay.AS;
  const int bh = blockIdx.x, b = bh / H, h = bh % H, hpg = H / g.G, grp = h / hpg;
  const int prow0 = warp * 2 * RPT + rq * RPT;
  const float dskip = g.has_d ? a.d[h] : 0.f;

  // zero tiles: the padding (n >= N, p >= P) and the previous-token slots
  // (zero state) are never written otherwise
  for (int i = tid; i < lay.part; i += BT) sm[i] = 0.f;
  float hs[RPT][4 * NB];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int e = 0; e < 4 * NB; ++e) hs[i][e] = 0.f;
  float th_run = 0.f;  // thread a < A: running angle
  float dsum = 0.f;    // this thread's share of sum_t dy_t . x_t
  float cbacc = 0.f;   // this thread's share of the c_bias sum, column tid % Npad
  __syncthreads();

  const int ntiles = (L + kT - 1) / kT;
  for (int tile = 0; tile < ntiles; ++tile) {
    const int t0 = tile * kT, tv = min(kT, L - t0);
    // (1) per-token scalars, values, gate factors; the running angle
    if (tid < tv) {
      const int64_t s = ((int64_t)b * L + t0 + tid) * H + h;
      const float al = expf(a.adt[s]), dtv = a.dt[s], lam = sigmoid_f(a.trap[s]);
      scoef[tid * 8 + 0] = al;
      scoef[tid * 8 + 1] = (1.f - lam) * dtv * al;
      scoef[tid * 8 + 2] = lam * dtv;
    }
    for (int i = tid; i < tv * Ppad; i += BT) {
      const int tt = i / Ppad, p = i - tt * Ppad;
      if (p >= P) continue;
      const int64_t e = (((int64_t)b * L + t0 + tt) * H + h) * P + p;
      const float go = o.dout[e];
      sv[(tt + 1) * Ppad + p] = a.x[e];
      float dyv = go, dzf = 0.f;
      if (g.has_z) {
        const float zv = a.z[e], sg = sigmoid_f(zv);
        dyv = go * (zv * sg);
        dzf = go * (sg + zv * sg * (1.f - sg));
      }
      sdy[tt * Ppad + p] = dyv;
      sdz[tt * Ppad + p] = dzf;
    }
    if (tid < A) {
      float dts[kT], ang[kT];
#pragma unroll
      for (int tt = 0; tt < kT; ++tt) {
        const int64_t tok = (int64_t)b * L + t0 + tt;
        dts[tt] = tt < tv ? a.dt[tok * H + h] : 0.f;
        ang[tt] = tt < tv ? a.angle[tok * A + tid] : 0.f;
      }
#pragma unroll
      for (int tt = 0; tt < kT; ++tt) {
        if (tt < tv) {
          th_run = fmaf(dts[tt], ang[tt], th_run);
          sth[tt * AS + tid] = th_run;
          w.theta[((int64_t)bh * L + t0 + tt) * A + tid] = th_run;
        }
      }
    }
    __syncthreads();
    // (2) rotated q_t into sq[tt], k_t into sk[tt + 1] (sk[0]: previous token)
    stage_qk<NB, BT>(g, a, b, h, grp, t0, tv, lay, sq, sk, 1, sth, scs, ssn);
    __syncthreads();
    // (3) the recurrence over the tile's tokens, the next tile's operands
    // prefetched into L2 meanwhile
    if (t0 + kT < L)
      prefetch_tile<BT>(g, a, o.dout, nullptr, bh, b, h, grp, t0 + kT, min(kT, L - t0 - kT));
    for (int tt = 0; tt < tv; ++tt) {
      const float al = scoef[tt * 8], sal = scoef[tt * 8 + 1], gm = scoef[tt * 8 + 2];
      float kp[4 * NB], kc[4 * NB], qv[4 * NB];
      load_cols<NB>(sk + tt * Npad, cq, kp);
      load_cols<NB>(sk + (tt + 1) * Npad, cq, kc);
      load_cols<NB>(sq + tt * Npad, cq, qv);
      float vp[RPT], vc[RPT], dyr[RPT];
      load_rows<RPT>(sv + tt * Ppad + prow0, vp);
      load_rows<RPT>(sv + (tt + 1) * Ppad + prow0, vc);
      load_rows<RPT>(sdy + tt * Ppad + prow0, dyr);
      float yv[RPT], dq[4 * NB];
#pragma unroll
      for (int e = 0; e < 4 * NB; ++e) dq[e] = 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float cp = sal * vp[i], cc = gm * vc[i];
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) {
          hs[i][e] = fmaf(al, hs[i][e], fmaf(cp, kp[e], cc * kc[e]));
          acc = fmaf(hs[i][e], qv[e], acc);
          dq[e] = fmaf(hs[i][e], dyr[i], dq[e]);
        }
        yv[i] = acc;
      }
      int row;
      const float ysum = rows_sum16<RPT>(yv, cq, row);
      if ((cq & (16 / RPT - 1)) == 0) sy[tt * Ppad + prow0 + row] = ysum;
      cols_sum_store<NB>(dq, rq, cq, spart + (tt * kW + warp) * Npad);
    }
    __syncthreads();
    // (4) dq_t: the warps' column sums, into slot 0
    for (int i = tid; i < tv * Npad; i += BT) {
      const int tt = i / Npad, n = i - tt * Npad;
      float* pp = spart + tt * kW * Npad + n;
      float s = pp[0];
#pragma unroll
      for (int x = 1; x < kW; ++x) s += pp[x * Npad];
      pp[0] = s;
    }
    __syncthreads();
    // (5a) the head's C gradient Rot(theta)^T dq_t and the c_bias sum
    {
      const int n = tid % Npad;
      for (int tt = tid / Npad; tt < tv; tt += BT / Npad) {
        if (n < N) {
          const float v = unrotate(spart + tt * kW * Npad, scs + tt * AS, ssn + tt * AS, n, A);
          w.dc_h[(((int64_t)b * L + t0 + tt) * H + h) * N + n] = v;
          cbacc += v;
        }
      }
    }
    // (5b) Q_t = q_t . dq_t and the query part of theta_t's adjoint
    for (int tt = warp; tt < tv; tt += kW) {
      const float* dq = spart + tt * kW * Npad;
      const float* q = sq + tt * Npad;
      float s = 0.f;
      for (int n = lane; n < N; n += 32) s = fmaf(q[n], dq[n], s);
      s = warp_sum(s);
      const int64_t tix = (int64_t)bh * L + t0 + tt;
      if (lane == 0) w.Q[tix] = s;
      for (int u = lane; u < A; u += 32) w.dthq[tix * A + u] = dq[u + A] * q[u] - dq[u] * q[u + A];
    }
    // (5c) dz_t = dout_t (y_t + D x_t) silu'(z_t); the D sum
    for (int i = tid; i < tv * Ppad; i += BT) {
      const int tt = i / Ppad, p = i - tt * Ppad;
      if (p >= P) continue;
      const float xv = sv[(tt + 1) * Ppad + p];
      o.gz[(((int64_t)b * L + t0 + tt) * H + h) * P + p] =
          g.has_z ? sdz[tt * Ppad + p] * fmaf(dskip, xv, sy[tt * Ppad + p]) : 0.f;
      dsum = fmaf(sdy[tt * Ppad + p], xv, dsum);
    }
    // (5d) this tile's last key and value become the next tile's previous token
    if (tv == kT) {
      for (int n = tid; n < Npad; n += BT) sk[n] = sk[kT * Npad + n];
      for (int p = tid; p < Ppad; p += BT) sv[p] = sv[kT * Ppad + p];
    }
    __syncthreads();
  }
  // per-(b, h) shares of the c_bias and D sums
  spart[tid] = cbacc;
  spart[BT + tid] = dsum;
  __syncthreads();
  if (tid < N) {
    float s = 0.f;
    for (int x = tid; x < BT; x += Npad) s += spart[x];
    w.pcb[(int64_t)bh * N + tid] = s;
  }
  if (warp == 0) {
    float s = 0.f;
    for (int x = lane; x < BT; x += 32) s += spart[BT + x];
    s = warp_sum(s);
    if (lane == 0) w.pd[bh] = s;
  }
}

template <int RPT, int NB, int BT>
__global__ void __launch_bounds__(BT, BT > 256 || RPT >= 8 ? 1 : 2)
    k_bwd_rev(ScanGeom g, ScanArgs a, BwdArgs o, BwdWs w, BwdLayout lay) {
  constexpr int kW = BT / 32;
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
  float* sred = sm + lay.red;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rq = lane >> 4, cq = lane & 15;
  const int P = g.P, N = g.N, A = g.A, L = g.L, H = g.H;
  constexpr int Npad = 64 * NB, Ppad = 2 * kW * RPT;
  const int AS = lay.AS;
  const int bh = blockIdx.x, b = bh / H, h = bh % H, hpg = H / g.G, grp = h / hpg;
  const int prow0 = warp * 2 * RPT + rq * RPT;
  const float dskip = g.has_d ? a.d[h] : 0.f;

  for (int i = tid; i < lay.part; i += BT) sm[i] = 0.f;
  float lam[RPT][4 * NB];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int e = 0; e < 4 * NB; ++e) lam[i][e] = 0.f;
  float gth = 0.f;   // thread a < A: adjoint of theta summed from the last token
  float cadt = 0.f;  // warp 0: d adt summed from the last token
  float bbacc = 0.f;
  __syncthreads();

  const int ntiles = (L + kT - 1) / kT;
  for (int tile = ntiles - 1; tile >= 0; --tile) {
    const int t0 = tile * kT, tv = min(kT, L - t0);
    // (1) scalars of token t and of token t + 1 (zero past the end)
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
      scoef[tid * 8 + 1] = gm + s1;  // w_t
      scoef[tid * 8 + 2] = gm;
      scoef[tid * 8 + 3] = s1;
      scoef[tid * 8 + 4] = dtv;
    }
    for (int i = tid; i < tv * Ppad; i += BT) {
      const int tt = i / Ppad, p = i - tt * Ppad;
      if (p >= P) continue;
      const int64_t e = (((int64_t)b * L + t0 + tt) * H + h) * P + p;
      const float go = o.dout[e];
      sv[tt * Ppad + p] = a.x[e];
      float dyv = go;
      if (g.has_z) {
        const float zv = a.z[e];
        dyv = go * (zv * sigmoid_f(zv));
      }
      sdy[tt * Ppad + p] = dyv;
    }
    for (int i = tid; i < tv * 64; i += BT) {
      const int tt = i >> 6, u = i & 63;
      if (u >= A) continue;
      sth[tt * AS + u] = w.theta[((int64_t)bh * L + t0 + tt) * A + u];
    }
    __syncthreads();
    // (2) rotated q_t into sq[tt], k_t into sk[tt]
    stage_qk<NB, BT>(g, a, b, h, grp, t0, tv, lay, sq, sk, 0, sth, scs, ssn);
    __syncthreads();
    // (3) the adjoint recurrence, last token first, the previous tile's
    // operands prefetched into L2 meanwhile
    if (t0 > 0) prefetch_tile<BT>(g, a, o.dout, w.theta, bh, b, h, grp, t0 - kT, kT);
    for (int tt = tv - 1; tt >= 0; --tt) {
      const float al1 = scoef[tt * 8];
      float kv[4 * NB], qv[4 * NB];
      load_cols<NB>(sk + tt * Npad, cq, kv);
      load_cols<NB>(sq + tt * Npad, cq, qv);
      float vr[RPT], dyr[RPT];
      load_rows<RPT>(sv + tt * Ppad + prow0, vr);
      load_rows<RPT>(sdy + tt * Ppad + prow0, dyr);
      float mk[RPT], mv[4 * NB];
#pragma unroll
      for (int e = 0; e < 4 * NB; ++e) mv[e] = 0.f;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) {
          const float m = al1 * lam[i][e];
          acc = fmaf(m, kv[e], acc);
          mv[e] = fmaf(m, vr[i], mv[e]);
          lam[i][e] = fmaf(dyr[i], qv[e], m);
        }
        mk[i] = acc;
      }
      int row;
      const float msum = rows_sum16<RPT>(mk, cq, row);
      if ((cq & (16 / RPT - 1)) == 0) smk[tt * Ppad + prow0 + row] = msum;
      cols_sum_store<NB>(mv, rq, cq, spart + (tt * kW + warp) * Npad);
    }
    __syncthreads();
    // (4) M^T v_t: the warps' column sums, into slot 0
    for (int i = tid; i < tv * Npad; i += BT) {
      const int tt = i / Npad, n = i - tt * Npad;
      float* pp = spart + tt * kW * Npad + n;
      float s = pp[0];
#pragma unroll
      for (int x = 1; x < kW; ++x) s += pp[x * Npad];
      pp[0] = s;
    }
    __syncthreads();
    // (5) per token: dy . v, q . k, v . M k; dg_t, ds_{t+1} and the d adt term
    for (int tt = warp; tt < tv; tt += kW) {
      float dyv = 0.f, vmk = 0.f, qk = 0.f;
      for (int p = lane; p < P; p += 32) {
        const float v = sv[tt * Ppad + p];
        dyv = fmaf(sdy[tt * Ppad + p], v, dyv);
        vmk = fmaf(smk[tt * Ppad + p], v, vmk);
      }
      for (int n = lane; n < N; n += 32) qk = fmaf(sq[tt * Npad + n], sk[tt * Npad + n], qk);
      dyv = warp_sum(dyv);
      vmk = warp_sum(vmk);
      qk = warp_sum(qk);
      if (lane == 0) {
        const int t = t0 + tt;
        const int64_t tix = (int64_t)bh * L + t;
        const float gm = scoef[tt * 8 + 2], s1 = scoef[tt * 8 + 3];
        const float dg = fmaf(dyv, qk, vmk);
        w.dgam[tix] = dg;
        if (t + 1 < L) w.ds[tix + 1] = vmk;
        if (t == 0) w.ds[tix] = 0.f;
        sred[tt * 8 + 0] = dyv;
        sred[tt * 8 + 1] = qk;
        sred[tt * 8 + 2] = w.Q[tix] - gm * dg - s1 * vmk;
      }
    }
    __syncthreads();
    // (6) dk_t into slot 1; dv_t = dx_t
    for (int i = tid; i < tv * Npad; i += BT) {
      const int tt = i / Npad, n = i - tt * Npad;
      spart[(tt * kW + 1) * Npad + n] =
          fmaf(scoef[tt * 8 + 1], spart[tt * kW * Npad + n],
               scoef[tt * 8 + 2] * sred[tt * 8] * sq[tt * Npad + n]);
    }
    for (int i = tid; i < tv * Ppad; i += BT) {
      const int tt = i / Ppad, p = i - tt * Ppad;
      if (p >= P) continue;
      const float coef = fmaf(scoef[tt * 8 + 2], sred[tt * 8 + 1], dskip);
      o.gx[(((int64_t)b * L + t0 + tt) * H + h) * P + p] =
          fmaf(scoef[tt * 8 + 1], smk[tt * Ppad + p], coef * sdy[tt * Ppad + p]);
    }
    // (7) d adt_t: suffix sums of the tile's terms plus the later tiles' total
    if (warp == 0) {
      float v = lane < tv ? sred[lane * 8 + 2] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float t = __shfl_down_sync(0xffffffffu, v, off);
        if (lane + off < 32) v += t;
      }
      if (lane < tv) o.gadt[((int64_t)b * L + t0 + lane) * H + h] = cadt + v;
      cadt += __shfl_sync(0xffffffffu, v, 0);
    }
    __syncthreads();
    // (8) the head's B gradient Rot(theta)^T dk_t, the b_bias sum, and theta's
    // adjoint at each token: the query part plus the key part
    {
      const int n = tid % Npad;
      for (int tt = tid / Npad; tt < tv; tt += BT / Npad) {
        if (n < N) {
          const float v =
              unrotate(spart + (tt * kW + 1) * Npad, scs + tt * AS, ssn + tt * AS, n, A);
          w.db_h[(((int64_t)b * L + t0 + tt) * H + h) * N + n] = v;
          bbacc += v;
        }
      }
    }
    for (int i = tid; i < tv * 64; i += BT) {
      const int tt = i >> 6, u = i & 63;
      if (u >= A) continue;
      const float* dk = spart + (tt * kW + 1) * Npad;
      const float* k = sk + tt * Npad;
      sdth[tt * AS + u] = w.dthq[((int64_t)bh * L + t0 + tt) * A + u] +
                          (dk[u + A] * k[u] - dk[u] * k[u + A]);
    }
    __syncthreads();
    // (9) theta's adjoint summed from the last token
    if (tid < A) {
      for (int tt = tv - 1; tt >= 0; --tt) {
        gth += sdth[tt * AS + tid];
        sdth[tt * AS + tid] = gth;
      }
    }
    __syncthreads();
    // (10) theta_t = theta_{t-1} + dt_t angle_t: d angle (this head) and the
    // angle part of d dt
    for (int i = tid; i < tv * 64; i += BT) {
      const int tt = i >> 6, u = i & 63;
      if (u >= A) continue;
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
  spart[tid] = bbacc;
  __syncthreads();
  if (tid < N) {
    float s = 0.f;
    for (int x = tid; x < BT; x += Npad) s += spart[x];
    w.pbb[(int64_t)bh * N + tid] = s;
  }
}

// d dt and d trap per (b, t, h); the sums over heads and batch. Job
// blockIdx.y: 0 d dt / d trap, 1 C / B rows over a group's heads, 2 angle
// over heads, 3 biases over batch, 4 D over batch.
__global__ void __launch_bounds__(kBT) k_bwd_finish(ScanGeom g, ScanArgs a, BwdArgs o, BwdWs w) {
  const int B = g.B, L = g.L, H = g.H, G = g.G, N = g.N, A = g.A, hpg = H / G;
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
        o.gdt[i] += fmaf(lam, dg, (1.f - lam) * ds);
        o.gtrap[i] = (dg - ds) * dtv * (lam * (1.f - lam));
      }
      break;
    case 1:
      if (hpg > 1)
        for (int64_t i = i0; i < (int64_t)B * L * G * N; i += stride) {
          const int n = (int)(i % N);
          const int64_t r = i / N;
          const int grp = (int)(r % G);
          const int64_t tok = r / G;
          const int64_t base = (tok * H + (int64_t)grp * hpg) * N + n;
          float sc = 0.f, sb = 0.f;
          for (int j = 0; j < hpg; ++j) {
            sc += w.dc_h[base + (int64_t)j * N];
            sb += w.db_h[base + (int64_t)j * N];
          }
          o.gc[i] = sc;
          o.gb[i] = sb;
        }
      break;
    case 2:
      if (H > 1 && A > 0)
        for (int64_t i = i0; i < (int64_t)B * L * A; i += stride) {
          const int u = (int)(i % A);
          const int64_t tok = i / A;
          float s = 0.f;
          for (int h = 0; h < H; ++h) s += w.dang_h[(tok * H + h) * A + u];
          o.gangle[i] = s;
        }
      break;
    case 3:
      for (int64_t i = i0; i < (int64_t)H * N; i += stride) {
        float sc = 0.f, sb = 0.f;
        for (int b = 0; b < B; ++b) {
          sc += w.pcb[(int64_t)b * H * N + i];
          sb += w.pbb[(int64_t)b * H * N + i];
        }
        o.gc_bias[i] = sc;
        o.gb_bias[i] = sb;
      }
      break;
    default:
      for (int64_t i = i0; i < H; i += stride) {
        float s = 0.f;
        for (int b = 0; b < B; ++b) s += w.pd[(int64_t)b * H + i];
        o.gd[i] = g.has_d ? s : 0.f;
      }
      break;
  }
}

}  // namespace

namespace {
// Workspace layout (byte offsets, 256-byte aligned), from the geometry alone.
struct BwdPlan {
  size_t theta, dthq, Q, dgam, ds, dc_h, db_h, dang_h, pcb, pbb, pd, bytes;
  bool own_c, own_ang;  // per-head C / B, angle parts need their own arrays
};

BwdPlan bwd_plan(const ScanGeom& g) {
  BwdPlan p{};
  const size_t bh = (size_t)g.B * g.H, BL = (size_t)g.B * g.L;
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
  p.dc_h = take(p.own_c ? BL * g.H * g.N : 0);
  p.db_h = take(p.own_c ? BL * g.H * g.N : 0);
  p.dang_h = take(p.own_ang ? BL * g.H * g.A : 0);
  p.pcb = take(bh * g.N);
  p.pbb = take(bh * g.N);
  p.pd = take(bh);
  p.bytes = off;
  return p;
}

template <int RPT, int NB, int BT>
cudaError_t launch_bwd_sweeps(const ScanGeom& g, const ScanArgs& a, const BwdArgs& o,
                              const BwdWs& w, cudaStream_t s) {
  const BwdLayout lay = bwd_layout(g.A, RPT, NB, BT / 32);
  const size_t smem = (size_t)lay.floats * sizeof(float);
  {  // the opt-in above 48 KB, for A up to 64 (set on every call: it is per device)
    const int most = bwd_layout(64, RPT, NB, BT / 32).floats * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_bwd_fwd<RPT, NB, BT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_bwd_rev<RPT, NB, BT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = (unsigned)(g.B * g.H);
  k_bwd_fwd<RPT, NB, BT><<<grid, BT, smem, s>>>(g, a, o, w, lay);
  k_bwd_rev<RPT, NB, BT><<<grid, BT, smem, s>>>(g, a, o, w, lay);
  count_launches(2);
  return cudaGetLastError();
}

// SMs of the current device (also the answer when none can be queried).
int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  return n;
}
}  // namespace

size_t backward_workspace_bytes(const ScanGeom& g) { return bwd_plan(g).bytes; }

cudaError_t launch_siso_backward(const ScanGeom& g, const ScanArgs& a, const BwdArgs& o,
                                 void* ws, cudaStream_t s) {
  const BwdPlan p = bwd_plan(g);
  char* base = static_cast<char*>(ws);
  auto f = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
  BwdWs w;
  w.theta = f(p.theta);
  w.dthq = f(p.dthq);
  w.Q = f(p.Q);
  w.dgam = f(p.dgam);
  w.ds = f(p.ds);
  // one head per group: the head's C / B gradient is the output itself; one
  // head: so is its angle gradient
  w.dc_h = p.own_c ? f(p.dc_h) : o.gc;
  w.db_h = p.own_c ? f(p.db_h) : o.gb;
  w.dang_h = p.own_ang ? f(p.dang_h) : o.gangle;
  w.pcb = f(p.pcb);
  w.pbb = f(p.pbb);
  w.pd = f(p.pd);
  const int nb = g.N <= 64 ? 1 : 2;
  cudaError_t e;
  if ((int64_t)g.B * g.H < device_sms()) {
    // fewer sequences than SMs: one 512-thread block (16 warps) per sequence
    const int rpt = g.P <= 32 ? 1 : g.P <= 64 ? 2 : 4;
    switch (rpt * 10 + nb) {
      case 11: e = launch_bwd_sweeps<1, 1, 512>(g, a, o, w, s); break;
      case 12: e = launch_bwd_sweeps<1, 2, 512>(g, a, o, w, s); break;
      case 21: e = launch_bwd_sweeps<2, 1, 512>(g, a, o, w, s); break;
      case 22: e = launch_bwd_sweeps<2, 2, 512>(g, a, o, w, s); break;
      case 41: e = launch_bwd_sweeps<4, 1, 512>(g, a, o, w, s); break;
      default: e = launch_bwd_sweeps<4, 2, 512>(g, a, o, w, s); break;
    }
  } else {
    // two 256-thread blocks per SM
    const int rpt = g.P <= 32 ? 2 : g.P <= 64 ? 4 : 8;
    switch (rpt * 10 + nb) {
      case 21: e = launch_bwd_sweeps<2, 1, kBT>(g, a, o, w, s); break;
      case 22: e = launch_bwd_sweeps<2, 2, kBT>(g, a, o, w, s); break;
      case 41: e = launch_bwd_sweeps<4, 1, kBT>(g, a, o, w, s); break;
      case 42: e = launch_bwd_sweeps<4, 2, kBT>(g, a, o, w, s); break;
      case 81: e = launch_bwd_sweeps<8, 1, kBT>(g, a, o, w, s); break;
      default: e = launch_bwd_sweeps<8, 2, kBT>(g, a, o, w, s); break;
    }
  }
  if (e != cudaSuccess) return e;
  const int64_t most = std::max<int64_t>({(int64_t)g.B * g.L * g.H, (int64_t)g.B * g.L * g.G * g.N,
                                          (int64_t)g.B * g.L * g.A, (int64_t)g.H * g.N});
  const unsigned blocks = (unsigned)std::min<int64_t>((most + kBT - 1) / kBT, 152 * 8);
  k_bwd_finish<<<dim3(blocks, 5), kBT, 0, s>>>(g, a, o, w);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace m3
