// Token-sequential Mamba-3 scan on the CUDA cores, FP32 throughout (oarust
// mamba3.rs, `mamba3_siso` / `mamba3_mimo`: the recurrence run token by token).
//
// The rows p of the [P, N] state evolve independently given the per-token
// q, k, decay and trapezoid weights, so a block owns one (b, h) and a tile of
// PT state rows; LPR lanes share a row, each holding 4 * NPT4 state values in
// registers (float4-interleaved so that shared-memory reads are broadcasts),
// and the row's readouts are reduced across those lanes by shuffles, once per
// batch of LPR / RMAX tokens (recursive halving) where the ranks allow it.
// Per tile of kT tokens (16, 32 or 64: the longest that fits) the
// block stages the coefficients, the cumulative rotary angle, the rotated q/k
// rows and x/z in shared memory, runs the recurrence over the tile, then
// writes the gated outputs coalesced. MIMO blocks own all P rows so that the
// output RMS norm is block-local.
//
// This is the FP32 reference path of the library and the fallback for shapes
// outside the tensor-core chunked kernels.
#include "m3_internal.cuh"

namespace m3 {
namespace {


struct SeqLayout {
  int Npad, RS, PT, R, A, kT;  // kT: tokens per staging tile; RS: q / k row stride
  size_t q, k, coef, theta, cs, xs, zs, ys, os, bias, bytes;
};

// RS is the q / k row stride in floats: 4 * NPT4 * LPR of the kernel instance
// (>= Npad), so that every lane's state groups lie inside a row; the columns
// Npad .. RS stay zero.
__host__ __device__ inline SeqLayout seq_layout(int N, int PT, int R, int A, int kT, int RS) {
  SeqLayout l;
  l.Npad = (N + 15) / 16 * 16;
  l.RS = RS;
  l.PT = PT;
  l.R = R;
  l.A = A;
  l.kT = kT;
  size_t off = 0;
  auto take = [&](size_t floats) {
    size_t o = off;
    off += (floats + 3) / 4 * 4;  // keep 16-byte alignment
    return o;
  };
  l.q = take((size_t)kT * R * RS);
  l.k = take((size_t)(kT + 1) * R * RS);
  l.coef = take((size_t)kT * 4);
  l.theta = take((size_t)kT * (A > 0 ? A : 1));
  l.cs = take((size_t)2 * kT * (A > 0 ? A : 1));
  l.xs = take((size_t)kT * PT);
  l.zs = take((size_t)kT * PT);
  l.ys = take((size_t)kT * R * PT);
  l.os = take((size_t)kT * PT);
  l.bias = take((size_t)2 * R * l.Npad);  // c_bias, b_bias of this head, zero-padded
  l.bytes = off * sizeof(float);
  return l;
}

template <int NPT4, int RMAX, int LPR>
__global__ void __launch_bounds__(512, RMAX == 1 ? 2 : 1) k_scan_seq(ScanGeom g, ScanArgs a, SeqLayout lay,
                                                  StepState st) {
  extern __shared__ __align__(16) float sm[];
  float* sq = sm + lay.q;
  float* sk = sm + lay.k;
  float* scoef = sm + lay.coef;
  float* sth = sm + lay.theta;
  float* scs = sm + lay.cs;
  float* sx = sm + lay.xs;
  float* sz = sm + lay.zs;
  float* sy = sm + lay.ys;
  float* so = sm + lay.os;
  float* sbc = sm + lay.bias;          // [R][Npad] c_bias
  float* sbb = sbc + lay.R * lay.Npad;  // [R][Npad] b_bias

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int P = g.P, N = g.N, A = g.A, R = g.R, L = g.L, H = g.H;
  const int Npad = lay.Npad, PT = lay.PT, kT = lay.kT;
  constexpr int RS = 4 * NPT4 * LPR;  // q / k row stride (the launcher sets lay.RS to it)
  const int ptiles = (P + PT - 1) / PT;
  const int bh = blockIdx.x / ptiles;
  const int p0 = (blockIdx.x % ptiles) * PT;
  const int b = bh / H, h = bh % H;
  const int grp = h / (H / g.G);
  const int pi = tid / LPR, j = tid % LPR;
  const int p = p0 + pi;
  const bool row_ok = (pi < PT) && (p < P);

  // Recurrent state: zero, or (with st.ssm set; one block per (b, h) then) the
  // step state h [P,N], previous key [R,N], previous value [R,P] and cumulative
  // angle, which are read here and overwritten with the final state at the end.
  const bool has_state = st.ssm != nullptr;
  float* hrow = has_state && row_ok ? st.ssm + ((int64_t)bh * P + p) * N : nullptr;
  float hst[NPT4 * 4];
#pragma unroll
  for (int i = 0; i < NPT4; ++i) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = 4 * (j + LPR * i) + e;
      hst[4 * i + e] = (hrow && n < N) ? hrow[n] : 0.f;
    }
  }
  float mx[RMAX], xprev[RMAX];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    mx[r] = (r < R && row_ok) ? (a.mimo_x ? a.mimo_x[((int64_t)h * R + r) * P + p] : 1.f) : 0.f;
    xprev[r] = (has_state && r < R && row_ok) ? st.v[((int64_t)bh * R + r) * P + p] : 0.f;
  }
  const float dskip = g.has_d ? a.d[h] : 0.f;
  // q / k tiles start zeroed (columns Npad .. RS are never written again);
  // previous-token key slot (zero or the state's key); the running angle lives
  // in sth[(kT-1)*A + a]
  for (int i = tid; i < (2 * kT + 1) * R * RS; i += nthr) sq[i] = 0.f;  // sq, then sk
  __syncthreads();
  for (int i = tid; i < R * Npad; i += nthr) {
    const int r = i / Npad, n = i - r * Npad;
    sk[r * RS + n] = (has_state && n < N) ? st.k[((int64_t)bh * R + r) * N + n] : 0.f;
  }
  for (int i = tid; i < A; i += nthr)
    sth[(kT - 1) * A + i] = (has_state && st.angle) ? st.angle[(int64_t)bh * A + i] : 0.f;
  for (int i = tid; i < R * Npad; i += nthr) {
    const int r = i / Npad, n = i - r * Npad;
    sbc[i] = n < N ? a.c_bias[((int64_t)h * R + r) * N + n] : 0.f;
    sbb[i] = n < N ? a.b_bias[((int64_t)h * R + r) * N + n] : 0.f;
  }
  // float4 staging of q/k items and x/z rows when the shapes allow it
  const bool vec_qk = (A % 4 == 0) && (N % 4 == 0);
  const bool vec_xz = (P % 4 == 0) && (PT % 4 == 0);
  __syncthreads();

  for (int t0 = 0; t0 < L; t0 += kT) {
    const int tv = min(kT, L - t0);
    // 1. per-token coefficients, cumulative angle, x/z tiles
    for (int t = tid; t < tv; t += nthr) {
      const int64_t sc = ((int64_t)b * L + t0 + t) * H + h;
      const float dtv = a.dt[sc];
      const float lam = sigmoid_f(a.trap[sc]);
      const float dec = expf(a.adt[sc]);
      scoef[t * 4 + 0] = dec;
      scoef[t * 4 + 1] = lam * dtv;
      scoef[t * 4 + 2] = (1.0f - lam) * dtv * dec;
    }
    // dt * angle increments of the tile, loaded coalesced into the sin/cos
    // table's slot (it is overwritten below once the running sums exist)
    for (int i = tid; i < tv * A; i += nthr) {
      const int t = i / A, aa = i - t * A;
      const int64_t tok = (int64_t)b * L + t0 + t;
      scs[i] = a.dt[tok * H + h] * a.angle[tok * A + aa];
    }
    __syncthreads();
    for (int i = tid; i < A; i += nthr) {
      float th = sth[(kT - 1) * A + i];  // running angle from the previous tile
      for (int t = 0; t < tv; ++t) {
        th += scs[t * A + i];
        sth[t * A + i] = th;
      }
      for (int t = tv; t < kT; ++t) sth[t * A + i] = th;
    }
    __syncthreads();
    for (int i = tid; i < tv * A; i += nthr) sincosf(sth[i], &scs[2 * i + 1], &scs[2 * i]);
    if (vec_xz) {
      const int PT4 = PT / 4;
      for (int i = tid; i < kT * PT4; i += nthr) {
        const int t = i / PT4, q4 = i - t * PT4;
        float4 xv = make_float4(0.f, 0.f, 0.f, 0.f), zv = xv;
        if (t < tv && p0 + 4 * q4 < P) {
          const int64_t off = (((int64_t)b * L + t0 + t) * H + h) * P + p0 + 4 * q4;
          xv = *reinterpret_cast<const float4*>(a.x + off);
          zv = *reinterpret_cast<const float4*>(a.z + off);
        }
        reinterpret_cast<float4*>(sx)[i] = xv;
        reinterpret_cast<float4*>(sz)[i] = zv;
      }
    } else {
      for (int i = tid; i < kT * PT; i += nthr) {
        const int t = i / PT, pp = i % PT;
        float xv = 0.f, zv = 0.f;
        if (t < tv && p0 + pp < P) {
          const int64_t off = (((int64_t)b * L + t0 + t) * H + h) * P + p0 + pp;
          xv = a.x[off];
          zv = a.z[off];
        }
        sx[i] = xv;
        sz[i] = zv;
      }
    }
    __syncthreads();
    // 2. rotated q/k rows (zero-padded to Npad), k into slots 1..kT
    if (vec_qk) {
      // item = 4 dims n0..n0+3 of one (token, rank) row; for n0 < A also their
      // rotary partners n0+A..n0+A+3; padding dims N..Npad are zero
      const int PQ = A / 4, QW = PQ + (Npad - 2 * A) / 4;
      for (int i = tid; i < kT * R * QW; i += nthr) {
        const int row = i / QW, jq = i - row * QW;
        const int t = row / R, r = row - t * R;
        const int n0 = jq < PQ ? 4 * jq : 2 * A + 4 * (jq - PQ);
        const bool live = t < tv && n0 < N;
        const int64_t tok = (int64_t)b * L + t0 + t;
        const int64_t roff = (tok * g.G * R + (int64_t)grp * R + r) * N;
        const float* csn = scs + 2 * (t * A + n0);  // (cos, sin) pairs of angles n0..n0+3
        // one operand (C into q, then B into k) at a time: fewer live registers
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const float* src = (which ? a.b : a.c) + roff;
          const float* bias = (which ? sbb : sbc) + r * Npad;
          float* dst = which ? sk + (size_t)(R + t * R + r) * RS : sq + (size_t)(t * R + r) * RS;
          float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
          if (live) {
            const float4 u = *reinterpret_cast<const float4*>(src + n0);
            const float4 ub = *reinterpret_cast<const float4*>(bias + n0);
            if (jq < PQ) {
              const float4 w = *reinterpret_cast<const float4*>(src + n0 + A);
              const float4 wb = *reinterpret_cast<const float4*>(bias + n0 + A);
#define M3_SEQ_ROT(E, K)                                                      \
  {                                                                           \
    const float cs = csn[2 * K], sn = csn[2 * K + 1];                         \
    const float uu = u.E + ub.E, ww = w.E + wb.E;                             \
    v0.E = uu * cs - ww * sn;                                                 \
    v1.E = uu * sn + ww * cs;                                                 \
  }
              M3_SEQ_ROT(x, 0) M3_SEQ_ROT(y, 1) M3_SEQ_ROT(z, 2) M3_SEQ_ROT(w, 3)
#undef M3_SEQ_ROT
            } else {
              v0 = make_float4(u.x + ub.x, u.y + ub.y, u.z + ub.z, u.w + ub.w);
            }
          }
          *reinterpret_cast<float4*>(dst + n0) = v0;
          if (jq < PQ) *reinterpret_cast<float4*>(dst + n0 + A) = v1;
        }
      }
    } else
    for (int i = tid; i < kT * R * Npad; i += nthr) {
      const int t = i / (R * Npad);
      const int rem = i - t * R * Npad;
      const int r = rem / Npad, n = rem - r * Npad;
      float qv = 0.f, kv = 0.f;
      if (t < tv && n < N) {
        const int64_t tok = (int64_t)b * L + t0 + t;
        const int64_t row = (tok * g.G * R + (int64_t)grp * R + r) * N;
        const float* cb = a.c_bias + ((int64_t)h * R + r) * N;
        const float* bb = a.b_bias + ((int64_t)h * R + r) * N;
        if (n < 2 * A) {
          const int pa = n < A ? n : n - A;
          const float cs = scs[2 * (t * A + pa)], sn = scs[2 * (t * A + pa) + 1];
          const float qu = a.c[row + pa] + cb[pa], qw = a.c[row + pa + A] + cb[pa + A];
          const float ku = a.b[row + pa] + bb[pa], kw = a.b[row + pa + A] + bb[pa + A];
          if (n < A) {
            qv = qu * cs - qw * sn;
            kv = ku * cs - kw * sn;
          } else {
            qv = qu * sn + qw * cs;
            kv = ku * sn + kw * cs;
          }
        } else {
          qv = a.c[row + n] + cb[n];
          kv = a.b[row + n] + bb[n];
        }
      }
      sq[(t * R + r) * RS + n] = qv;
      sk[(R + t * R + r) * RS + n] = kv;
    }
    __syncthreads();
    // 3. recurrence over the tile. token_step advances the lane's state groups
    // by token t and returns the lane's partial readouts per rank.
    auto token_step = [&](int t, float* acc) {
      const float dec = scoef[t * 4 + 0], gam = scoef[t * 4 + 1], sdec = scoef[t * 4 + 2];
      const float xv = row_ok ? sx[t * PT + pi] : 0.f;
      float cp[RMAX], cc[RMAX], xr[RMAX], acc2[RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        xr[r] = xv * mx[r];
        cp[r] = sdec * xprev[r];
        cc[r] = gam * xr[r];
        acc[r] = 0.f;
        acc2[r] = 0.f;  // second readout chain (odd groups)
      }
      const float4* kp4 = reinterpret_cast<const float4*>(sk + (size_t)t * R * RS);
      const float4* kc4 = reinterpret_cast<const float4*>(sk + (size_t)(t + 1) * R * RS);
      const float4* q4 = reinterpret_cast<const float4*>(sq + (size_t)t * R * RS);
#pragma unroll
      for (int i = 0; i < NPT4; ++i) {
        const int n4 = j + LPR * i;  // always inside the row (RS = 4 NPT4 LPR)
        float ux = 0.f, uy = 0.f, uz = 0.f, uw = 0.f;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < R) {
            const float4 kp = kp4[r * (RS / 4) + n4];
            const float4 kc = kc4[r * (RS / 4) + n4];
            ux += cp[r] * kp.x + cc[r] * kc.x;
            uy += cp[r] * kp.y + cc[r] * kc.y;
            uz += cp[r] * kp.z + cc[r] * kc.z;
            uw += cp[r] * kp.w + cc[r] * kc.w;
          }
        }
        float* hh = hst + 4 * i;
        hh[0] = dec * hh[0] + ux;
        hh[1] = dec * hh[1] + uy;
        hh[2] = dec * hh[2] + uz;
        hh[3] = dec * hh[3] + uw;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < R) {
            const float4 qq = q4[r * (RS / 4) + n4];
            const float part = (hh[0] * qq.x + hh[1] * qq.y) + (hh[2] * qq.z + hh[3] * qq.w);
            if (i & 1)
              acc2[r] += part;
            else
              acc[r] += part;
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        acc[r] += acc2[r];
        xprev[r] = xr[r];
      }
    };
    if constexpr (RMAX <= LPR) {
      // Batches of TB = LPR / RMAX tokens: each lane keeps its partial readouts
      // of the batch (value u * RMAX + r for token tb + u, rank r); the LPR
      // lanes of the row then reduce them together by recursive halving
      // (LPR - 1 shuffles per batch instead of log2(LPR) per token and rank),
      // leaving lane j with value j.
      constexpr int TB = LPR / RMAX;
      for (int tb = 0; tb < tv; tb += TB) {
        float part[LPR];
#pragma unroll
        for (int u = 0; u < TB; ++u) {
          float acc[RMAX];
#pragma unroll
          for (int r = 0; r < RMAX; ++r) acc[r] = 0.f;
          if (tb + u < tv) token_step(tb + u, acc);
#pragma unroll
          for (int r = 0; r < RMAX; ++r) part[u * RMAX + r] = acc[r];
        }
#pragma unroll
        for (int o = LPR / 2; o >= 1; o >>= 1) {
          const bool upper = (j & o) != 0;  // this lane keeps the upper half
#pragma unroll
          for (int k = 0; k < o; ++k) {
            const float send = upper ? part[k] : part[k + o];
            const float keep = upper ? part[k + o] : part[k];
            part[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        const int r = j % RMAX, t = tb + j / RMAX;
        float mxr = 0.f;
#pragma unroll
        for (int k = 0; k < RMAX; ++k)
          if (k == r) mxr = mx[k];
        if (row_ok && t < tv && r < R)
          sy[(t * R + r) * PT + pi] = part[0] + dskip * (sx[t * PT + pi] * mxr);
      }
    } else {
      for (int t = 0; t < tv; ++t) {
        float acc[RMAX];
        token_step(t, acc);
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
#pragma unroll
          for (int o = 1; o < LPR; o <<= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
          if (r < R && j == 0 && row_ok) sy[(t * R + r) * PT + pi] = acc[r] + dskip * xprev[r];
        }
      }
    }
    __syncthreads();
    // 4. outputs
    if (!a.mimo_o) {
      for (int i = tid; i < tv * PT; i += nthr) {
        const int t = i / PT, pp = i % PT;
        if (p0 + pp < P) {
          float yv = sy[t * PT + pp];
          if (g.has_z) yv *= silu_f(sz[i]);
          a.out[(((int64_t)b * L + t0 + t) * H + h) * P + p0 + pp] = yv;
        }
      }
    } else {
      // MIMO: PT == P
      for (int i = tid; i < tv * P; i += nthr) {
        const int t = i / P, pp = i % P;
        float ov = 0.f;
        for (int r = 0; r < R; ++r) {
          float yv = sy[(t * R + r) * P + pp];
          if (g.has_z) yv *= silu_f(sz[i] * a.mimo_z[((int64_t)h * R + r) * P + pp]);
          ov += a.mimo_o[((int64_t)h * R + r) * P + pp] * yv;
        }
        so[i] = ov;
      }
      __syncthreads();
      const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
      for (int t = warp; t < tv; t += nw) {
        float inv = 1.f;
        if (g.has_norm) {
          float ss = 0.f;
          for (int pp = lane; pp < P; pp += 32) ss += so[t * P + pp] * so[t * P + pp];
          ss = warp_sum(ss);
          inv = 1.0f / sqrtf(ss / (float)P + 1.0e-5f);
        }
        for (int pp = lane; pp < P; pp += 32) {
          float ov = so[t * P + pp];
          if (g.has_norm) ov = ov * inv * a.norm_weight[(int64_t)h * P + pp];
          a.out[(((int64_t)b * L + t0 + t) * H + h) * P + pp] = ov;
        }
      }
    }
    // carry the last token's key into slot 0
    for (int i = tid; i < R * RS; i += nthr) sk[i] = sk[(size_t)tv * R * RS + i];
    __syncthreads();
  }
  if (has_state) {
#pragma unroll
    for (int i = 0; i < NPT4; ++i) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = 4 * (j + LPR * i) + e;
        if (hrow && n < N) hrow[n] = hst[4 * i + e];
      }
    }
    for (int i = tid; i < R * Npad; i += nthr) {
      const int r = i / Npad, n = i - r * Npad;
      if (n < N) st.k[((int64_t)bh * R + r) * N + n] = sk[r * RS + n];
    }
    if (row_ok && j == 0) {
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
        if (r < R) st.v[((int64_t)bh * R + r) * P + p] = xprev[r];
    }
    if (st.angle)
      for (int i = tid; i < A; i += nthr) st.angle[(int64_t)bh * A + i] = sth[(kT - 1) * A + i];
  }
}

int device_sm_count() {
  static const int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 152;
    return v;
  }();
  return n;
}

// State rows per block: all P rows (one block per (b, h): the MIMO output norm
// and the step state need it, and it stages each (b, h)'s q / k once) while
// 8 lanes per row keep the block within 512 threads; otherwise 32-row tiles.
// (Splitting the rows of a few long sequences over more blocks does not help:
// a block's time is its token loop's latency, not its share of the SM.)
int seq_rows_per_block(const ScanGeom& g, const ScanArgs& a, const StepState& st, int rmax) {
  if (rmax > 1 || a.mimo_o || st.ssm || g.P * 8 <= 512) return g.P;
  return g.P < 32 ? g.P : 32;
}

template <int NPT4, int RMAX, int LPR>
cudaError_t launch_seq_t(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                         cudaStream_t s) {
  // one block per (b, h) for MIMO (block-local output norm) and with state
  // (the per-(b, h) key / angle state is read first and written last)
  const int PT = seq_rows_per_block(g, a, st, RMAX);
  constexpr int RS = 4 * NPT4 * LPR;
  // Staging tiles as long as they fit (the per-tile staging is a chain of
  // dependent loads and block barriers, so longer tiles amortise it): 64
  // tokens in 200 KB when the grid has no more blocks than SMs; 32 tokens in
  // 200 KB for the one-block-per-SM instances (RMAX > 1, MIMO, step state) or
  // in 100 KB (two blocks per SM) otherwise; else 16 tokens.
  SeqLayout lay = seq_layout(g.N, PT, g.R, g.A, 16, RS);
  {
    const bool one_per_sm = RMAX > 1 || a.mimo_o || st.ssm;
    const int64_t blocks = (int64_t)g.B * g.H * ((g.P + PT - 1) / PT);
    const SeqLayout mid = seq_layout(g.N, PT, g.R, g.A, 32, RS);
    const SeqLayout big = seq_layout(g.N, PT, g.R, g.A, 64, RS);
    if (blocks <= device_sm_count() && big.bytes <= 200u * 1024u)
      lay = big;
    else if (mid.bytes <= (one_per_sm ? 200u : 100u) * 1024u)
      lay = mid;
  }
  const int threads = ((PT * LPR + 31) / 32) * 32;
  const int ptiles = (g.P + PT - 1) / PT;
  cudaError_t e = cudaFuncSetAttribute(k_scan_seq<NPT4, RMAX, LPR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)lay.bytes);
  if (e != cudaSuccess) return e;
  k_scan_seq<NPT4, RMAX, LPR><<<(unsigned)(g.B * g.H * ptiles), threads, lay.bytes, s>>>(g, a, lay,
                                                                                         st);
  count_launches(1);
  return cudaGetLastError();
}

// Lanes per state row: 8 while the block stays within 512 threads, else 4.
template <int RMAX>
cudaError_t launch_seq_r(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                         cudaStream_t s) {
  const int PT = seq_rows_per_block(g, a, st, RMAX);
  const int groups = (g.N + 15) / 16 * 4;  // float4 groups of a padded row
  if (PT * 8 <= 512) {
    if (groups <= 8) return launch_seq_t<1, RMAX, 8>(g, a, st, s);
    if (groups <= 16) return launch_seq_t<2, RMAX, 8>(g, a, st, s);
    return launch_seq_t<4, RMAX, 8>(g, a, st, s);
  }
  if (groups <= 4) return launch_seq_t<1, RMAX, 4>(g, a, st, s);
  if (groups <= 8) return launch_seq_t<2, RMAX, 4>(g, a, st, s);
  if (groups <= 16) return launch_seq_t<4, RMAX, 4>(g, a, st, s);
  return launch_seq_t<8, RMAX, 4>(g, a, st, s);
}

}  // namespace

cudaError_t launch_scan_seq(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                            cudaStream_t s) {
  if (g.R == 1 && !a.mimo_o) return launch_seq_r<1>(g, a, st, s);
  if (g.R <= 4) return launch_seq_r<4>(g, a, st, s);
  return launch_seq_r<8>(g, a, st, s);
}

}  // namespace m3
