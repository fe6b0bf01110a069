// Chunked Mamba-3 scan on the tcgen05 tensor cores (TF32 operands, FP32
// accumulation in tensor memory). Covers `mamba3_siso` and `mamba3_mimo`
// (oarust mamba3.rs) for mimo_rank R in {1, 2, 4, 8}, P <= 128, N <= 128.
//
// Algebra. Unrolling the exponential-trapezoidal recurrence gives, for a chunk
// starting at token t0 with cum_t = sum_{t0 <= i <= t} adt_i,
//   h_t = e^{cum_t} g_{t0-1} + sum_{t0 <= s <= t} e^{cum_t - cum_s} c_{t,s} x_s k_s^T,
//   c_{t,s} = gamma_s + scale_{s+1} [s < t],
// where g is the "pre-loaded" state (h plus the next token's trapezoid term),
// carried from chunk to chunk as
//   g_end = e^{cum_end} g_{t0-1} + sum_s w_s x_s k_s^T,
//   w_s = e^{cum_end - cum_s} (gamma_s + scale_{s+1}).
// MIMO expands every token into R rows (t, r) that share the token's decay
// and rotation; SISO is R = 1. A chunk holds 64 such rows.
//
// Per chunk and (b, h), every contraction is a tcgen05.mma (kind::tf32):
//   S    = Q K^T               [64 x 64],  K = N     (A, B in shared memory)
//   Yo^T = G Q^T               [P  x 64],  K = N     (A = state G in TMEM)
//   Yi^T = X^T (M o S)^T       [P  x 64],  K = 64    (decay/trapezoid mask M)
//   G   += X^T (w K)           [P  x N],   K = 64    (after G *= e^{cum_end})
// The state G [P x N] stays in TMEM for the whole sequence; outputs come out
// transposed (TMEM lane = p): each output column p is finished by the two
// lanes that share its TMEM row (D skip, SiLU gate, the MIMO mimo_o
// contraction over its R rows) and, through shared memory, the MIMO output
// RMS norm. Rotary cos/sin, the local log-decay cumsum and the trapezoid
// weights are formed by the CUDA cores while staging operands; every operand
// is rounded to TF32 (round to nearest).
//
// One CTA of 256 threads runs one (b, h) sequence chunk after chunk; thread 0
// issues the MMAs and the CTA waits on mbarriers signalled by tcgen05.commit.
// Waits are bounded: on timeout the kernel records a status word and exits.
// Shared memory (about 100 KB for P <= 64, N = 128: the tiles share three
// regions whose contents change phase by phase) and TMEM (256 columns) admit
// two CTAs per SM, and the next chunk's inputs are prefetched into L2 while
// the current chunk runs.
#include "m3_internal.cuh"
#include "tc_ptx.cuh"

namespace m3 {
namespace {

constexpr int kRows = 64;       // (token, rank) rows per chunk
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTok = 72;        // per-token scalar array stride (>= 65)
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (~2 s)

struct ChunkLayout {
  int Npad, MP, CS;
  int q, k, kt, bias, tok, thbase;  // float offsets of the regions
  size_t bytes;
};

int imax(int a, int b) { return a > b ? a : b; }

ChunkLayout chunk_layout(int N, int P, int A, int R) {
  ChunkLayout l;
  l.Npad = (N + 15) / 16 * 16;
  l.MP = P <= 64 ? 64 : 128;
  l.CS = (A + 4) & ~3;  // cos / sin table row stride (16-byte rows, A + 1 <= CS)
  int off = 0;
  auto take = [&](int floats) {
    int o = off;
    off += (floats + 31) / 32 * 32;  // 128-byte aligned regions
    return o;
  };
  // Q region: q tile [64][Npad] until the first MMA batch completes, then the
  // masked scores [64][64] followed by the values X^T [MP][64].
  l.q = take(imax(kRows * l.Npad, kRows * kRows + l.MP * kRows));
  // K region: k tile [64][Npad]; MIMO norm staging [64][MP] in the epilogue.
  l.k = take(kRows * imax(l.Npad, l.MP));
  // Kt region: rotary angle increments, then cos / sin tables [64][CS] each
  // while the q/k tiles are formed, then the w-scaled transposed keys [Npad][64].
  l.kt = take(imax(l.Npad * kRows, 2 * kRows * l.CS));
  l.bias = take(2 * R * l.Npad);  // c_bias, b_bias of this head, zero-padded
  l.tok = take(8 * kTok);
  l.thbase = take(64);
  l.bytes = (size_t)off * sizeof(float);
  return l;
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

// Per-token scalars and angle increments of one chunk, loaded into registers
// one chunk ahead (thread t <= Qt holds token t's dt / adt / trap; the angle
// increments follow the (token = warp + 8 i, angle = lane + 32 j) tiling of
// the staging loop).
struct TokenPreload {
  float dt, adt, trap;
  float ang[16];
};

__device__ __forceinline__ void preload_tokens(TokenPreload& pl, const ScanArgs& a, int64_t tok,
                                               int cn, int L, int Qt, int A, int H, int h,
                                               int tid, int warp, int lane) {
  pl.dt = pl.adt = pl.trap = 0.f;
  if (tid <= Qt && cn + tid < L) {
    const int64_t sc = (tok + tid) * H + h;
    pl.dt = a.dt[sc];
    pl.adt = a.adt[sc];
    pl.trap = a.trap[sc];
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int t = warp + 8 * i, aa = lane + 32 * j;
      pl.ang[2 * i + j] = (t < Qt && aa < A && cn + t < L) ? a.angle[(tok + t) * A + aa] : 0.f;
    }
  }
}

// SiLU with the hardware exp / divide approximations (relative error a few
// float32 ulps, far inside the scan tolerances).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

template <int MP, bool MIMO, bool SUMMARY>
__global__ void __launch_bounds__(kThreads, 2)
    k_scan_chunk(ScanGeom g, ScanArgs a, ChunkLayout lay, ChunkIO io, uint32_t* status) {
  extern __shared__ __align__(1024) float sm[];
  // MMA completion barriers: S, Yo, Yi, state update (each completes once per chunk)
  __shared__ __align__(8) uint64_t bars[4];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = g.H, L = g.L, P = g.P, N = g.N, A = g.A, R = g.R;
  const int lgR = __ffs(R) - 1;  // R is a power of two here
  const int Npad = lay.Npad;
  const int Qt = kRows >> lgR;  // tokens per chunk
  const int cta = blockIdx.x;
  const int bh = cta / io.nseg, seg = cta - bh * io.nseg;
  const int b = bh / H, h = bh % H;
  const int l0 = seg * io.seg_len, l1 = min(L, l0 + io.seg_len);
  // the summary of the last segment is never used
  if (SUMMARY && seg == io.nseg - 1) return;
  const int grp = h / (H / g.G);
  const int RG = g.G * R;

  float* sQ = sm + lay.q;              // [64 rows][Npad] K-major, K = n
  float* sP = sQ;                      // [64][64]        masked scores (after batch 1)
  float* sXt = sQ + kRows * kRows;     // [MP][64 rows]   values (after batch 1)
  float* sK = sm + lay.k;              // [64 rows][Npad] K-major, K = n
  float* sO = sK;                      // [Qt][MP]        MIMO epilogue staging
  const int CS = lay.CS;
  float* sCos = sm + lay.kt;           // [Qt][CS]        angle increments, then cos
  float* sSin = sCos + kRows * CS;     // [Qt][CS]        sin
  float* sBiasC = sm + lay.bias;       // [R][Npad]
  float* sBiasB = sBiasC + R * Npad;   // [R][Npad]
  float* sKt = sm + lay.kt;            // [Npad][64 rows] K-major, K = row (w-scaled keys)
  float* tAdt = sm + lay.tok;
  float* tCum = tAdt + kTok;
  float* tEc = tCum + kTok;   // e^{cum_t}
  float* tGam = tEc + kTok;   // gamma_t
  float* tScl = tGam + kTok;  // scale_t, t in [0, Qt]
  float* tW = tScl + kTok;    // gamma_t + scale_{t+1}
  float* tOm = tW + kTok;     // e^{cum_end - cum_t} * tW[t]
  float* tDt = tOm + kTok;
  float* sThBase = sm + lay.thbase;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) tc::bar_init(&bars[i], 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 256);
  for (int i = tid; i < A; i += kThreads) sThBase[i] = io.th0 ? io.th0[(int64_t)cta * A + i] : 0.f;
  for (int i = tid; i < R * Npad; i += kThreads) {
    const int r = i / Npad, n = i - r * Npad;
    sBiasC[i] = n < N ? a.c_bias[((int64_t)h * R + r) * N + n] : 0.f;
    sBiasB[i] = n < N ? a.b_bias[((int64_t)h * R + r) * N + n] : 0.f;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = tmem_slot;
  // TMEM lane quadrant of this warp (warps w and w + 4 share quadrant w % 4 and
  // split the columns of the row-wise TMEM work between them)
  const int quad = warp & 3, wg = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const uint32_t tG = tbase, tS = tbase + 128, tYo = tbase + 192;
  // Row p of the transposed tiles handled by this thread (TMEM data path:
  // M = 128 -> lane p; M = 64 -> lanes 0..15 of each 32-lane quadrant, and
  // lane l + 16 shares the row of lane l, taking the upper half of the columns).
  const int half = (MP == 64) ? (lane >> 4) : 0;
  const int prow = (MP == 64) ? 16 * quad + (lane & 15) : 32 * quad + lane;
  const bool pvalid = prow < P;
  const bool g_lane = pvalid && (MP == 128 || half == 0);  // TMEM lane holding row prow
  {
    // initial state G (zero, or this segment's entry state)
    const float* g0 = io.g0 ? io.g0 + ((int64_t)cta * P + prow) * N : nullptr;
    for (int c = 16 * wg; c < Npad; c += 32) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = (g0 && g_lane && c + j < N) ? g0[c + j] : 0.f;
      tc::tmem_st16(tG + lane_base + c, v);
    }
  }
  constexpr bool mimo = MIMO;
  constexpr int kRmax = MIMO ? 8 : 1;
  float mxr[kRmax], mzr[kRmax], mor[kRmax];
#pragma unroll
  for (int r = 0; r < kRmax; ++r) {
    const bool ok = mimo && pvalid && r < R;
    mxr[r] = ok ? a.mimo_x[((int64_t)h * R + r) * P + prow] : 1.f;
    mzr[r] = ok ? a.mimo_z[((int64_t)h * R + r) * P + prow] : 1.f;
    mor[r] = ok ? a.mimo_o[((int64_t)h * R + r) * P + prow] : 0.f;
  }
  const float dsk = g.has_d ? a.d[h] : 0.f;
  const uint32_t id_S = tc::idesc_tf32(64, 64);
  const uint32_t id_Y = tc::idesc_tf32(MP, 64);
  const uint32_t id_D = tc::idesc_tf32(MP, Npad);
  const int64_t HP = (int64_t)H * P;
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  TokenPreload pl;
  preload_tokens(pl, a, (int64_t)b * L + l0, l0, L, Qt, A, H, h, tid, warp, lane);
  float esum = 0.f;  // sum of adt over the segment

  int it = 0;
  for (int c0 = l0; c0 < l1; c0 += Qt, ++it) {
    const int tv = min(Qt, l1 - c0);
    const int64_t tok0 = (int64_t)b * L + c0;   // first token of the chunk in [B, L]
    // (0) L2 prefetch of the next chunk's operands. The next chunk's blocks of
    // x, z, C, B, dt, adt, trap and angle are contiguous across the heads of a
    // batch row, so the H CTAs of that row (resident together) each prefetch
    // one 16-byte-aligned slice of every block.
    if (c0 + Qt < l1 && tid < 8) {
      const int nv = min(Qt, l1 - c0 - Qt);
      const int64_t ntok = tok0 + Qt;
      const float* base = nullptr;
      int64_t floats = 0;
      switch (tid) {
        case 0: base = a.x + ntok * HP; floats = (int64_t)nv * HP; break;
        case 1: base = a.z + ntok * HP; floats = (int64_t)nv * HP; break;
        case 2: base = a.c + ntok * RG * N; floats = (int64_t)nv * RG * N; break;
        case 3: base = a.b + ntok * RG * N; floats = (int64_t)nv * RG * N; break;
        case 4: base = a.dt + ntok * H; floats = (int64_t)nv * H; break;
        case 5: base = a.adt + ntok * H; floats = (int64_t)nv * H; break;
        case 6: base = a.trap + ntok * H; floats = (int64_t)nv * H; break;
        default: base = a.angle + ntok * A; floats = (int64_t)nv * A; break;
      }
      const uintptr_t lo = reinterpret_cast<uintptr_t>(base);
      const uintptr_t hi = reinterpret_cast<uintptr_t>(base + floats);
      if (floats > 0 && (lo & 15) == 0 && (hi & 15) == 0) {
        const uintptr_t span = hi - lo;
        const uintptr_t s0 = lo + (span * h / H & ~uintptr_t(15));
        const uintptr_t s1 = (h + 1 == H) ? hi : lo + (span * (h + 1) / H & ~uintptr_t(15));
        if (s1 > s0) tc::prefetch_l2(reinterpret_cast<const void*>(s0), (uint32_t)(s1 - s0));
      }
    }
    // (1) per-token scalars of tokens c0 .. c0 + Qt (the last one is the next
    // chunk's first token: only its trapezoid scale is used); angle increments
    if (tid <= Qt) {
      const int t = tid;
      float dtv = 0.f, adtv = 0.f, gam = 0.f, scl = 0.f;
      if (c0 + t < L) {
        dtv = pl.dt;
        adtv = pl.adt;
        const float lam = sigmoid_f(pl.trap);
        gam = lam * dtv;
        scl = (1.0f - lam) * dtv;
      }
      tScl[t] = scl;
      if (t < Qt) {
        const bool in = t < tv;
        tAdt[t] = in ? adtv : 0.f;
        tGam[t] = in ? gam : 0.f;
        tDt[t] = in ? dtv : 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int t = warp + 8 * i, aa = lane + 32 * j;
        if (t < Qt && aa < A) sCos[t * CS + aa] = pl.ang[2 * i + j];
      }
    }
    __syncthreads();
    // (2) local cumulative log decay (warp 0, two tokens per lane); rotary
    // angle: per-angle scan of dt * angle over the chunk, then cos / sin of
    // each (token, angle) once
    if (warp == 0) {
      const int t0 = 2 * lane, t1 = 2 * lane + 1;
      const float a0 = t0 < Qt ? tAdt[t0] : 0.f, a1 = t1 < Qt ? tAdt[t1] : 0.f;
      float s = a0 + a1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += v;
      }
      const float ex = s - (a0 + a1);
      if (t0 < Qt) tCum[t0] = ex + a0;
      if (t1 < Qt) tCum[t1] = ex + a0 + a1;
    }
    for (int aa = warp; aa < A; aa += kWarps) {
      float v0 = lane < Qt ? tDt[lane] * sCos[lane * CS + aa] : 0.f;
      float v1 = lane + 32 < Qt ? tDt[lane + 32] * sCos[(lane + 32) * CS + aa] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, v0, o);
        const float u1 = __shfl_up_sync(0xffffffffu, v1, o);
        if (lane >= o) {
          v0 += u0;
          v1 += u1;
        }
      }
      v1 += __shfl_sync(0xffffffffu, v0, 31);
      const float base = sThBase[aa];
      const float th0 = base + v0, th1 = base + v1;
      const float last = __shfl_sync(0xffffffffu, Qt > 32 ? th1 : th0, Qt > 32 ? Qt - 33 : Qt - 1);
      if (lane < Qt) sincos_fast(th0, &sSin[lane * CS + aa], &sCos[lane * CS + aa]);
      if (lane + 32 < Qt) sincos_fast(th1, &sSin[(lane + 32) * CS + aa], &sCos[(lane + 32) * CS + aa]);
      __syncwarp();
      if (lane == 0) sThBase[aa] = last;
    }
    __syncthreads();
    // (3) decay / trapezoid coefficients
    esum += tCum[Qt - 1];
    if (tid < Qt) {
      const int t = tid;
      const float cum = tCum[t], cend = tCum[Qt - 1];
      const float w = tGam[t] + tScl[t + 1];
      tEc[t] = expf(cum);
      tW[t] = w;
      tOm[t] = expf(cend - cum) * w;
    }
    // (4a) rotated, biased q / k rows into the K-major q / k tiles.
    if ((A & 3) == 0 && (N & 3) == 0) {
      // Vector path: an item is 4 consecutive dims n0..n0+3 of one row; for
      // n0 < A it also produces their rotary partners n0+A..n0+A+3. Lane l
      // takes row 8 * rb + l % 8 and item 4 * jb + l / 8, so that each 16-byte
      // store of the warp lands in a distinct 16-byte slot (512 contiguous
      // bytes per warp).
      const int PQ = A >> 2, QW = PQ + ((N - 2 * A) >> 2), QW4 = (QW + 3) >> 2;
      const int rl = lane & 7, jl = lane >> 3;
#pragma unroll 2
      for (int item = warp; item < (kRows / 8) * QW4; item += kWarps) {
        const int rb = item / QW4, jb = item - rb * QW4;
        const int rho = 8 * rb + rl;
        const int t = rho >> lgR, r = rho & (R - 1);
        const bool in = t < tv;
        const int64_t roff = ((tok0 + t) * RG + (int64_t)grp * R + r) * N;
        const float* crow = a.c + roff;
        const float* brow = a.b + roff;
        const float* cb = sBiasC + r * Npad;
        const float* bb = sBiasB + r * Npad;
        {
          const int j = 4 * jb + jl;
          if (j >= QW) continue;
          if (j < PQ) {
            const int n0 = 4 * j;
            float4 q0 = make_float4(0.f, 0.f, 0.f, 0.f), q1 = q0, k0 = q0, k1 = q0;
            if (in) {
              const float4 cu = *reinterpret_cast<const float4*>(crow + n0);
              const float4 cw = *reinterpret_cast<const float4*>(crow + n0 + A);
              const float4 bu = *reinterpret_cast<const float4*>(brow + n0);
              const float4 bw = *reinterpret_cast<const float4*>(brow + n0 + A);
              const float4 cbu = *reinterpret_cast<const float4*>(cb + n0);
              const float4 cbw = *reinterpret_cast<const float4*>(cb + n0 + A);
              const float4 bbu = *reinterpret_cast<const float4*>(bb + n0);
              const float4 bbw = *reinterpret_cast<const float4*>(bb + n0 + A);
              const float4 cs = *reinterpret_cast<const float4*>(sCos + t * CS + n0);
              const float4 sn = *reinterpret_cast<const float4*>(sSin + t * CS + n0);
#define M3_ROT(E)                                                            \
  {                                                                          \
    const float qu = cu.E + cbu.E, qw = cw.E + cbw.E;                        \
    const float ku = bu.E + bbu.E, kw = bw.E + bbw.E;                        \
    q0.E = qu * cs.E - qw * sn.E;                                            \
    q1.E = qu * sn.E + qw * cs.E;                                            \
    k0.E = ku * cs.E - kw * sn.E;                                            \
    k1.E = ku * sn.E + kw * cs.E;                                            \
  }
              M3_ROT(x) M3_ROT(y) M3_ROT(z) M3_ROT(w)
#undef M3_ROT
            }
            if (!SUMMARY) {
              *reinterpret_cast<float4*>(sQ + tc::kmaj(rho, n0, Npad)) = tc::to_tf32(q0);
              *reinterpret_cast<float4*>(sQ + tc::kmaj(rho, n0 + A, Npad)) = tc::to_tf32(q1);
            }
            *reinterpret_cast<float4*>(sK + tc::kmaj(rho, n0, Npad)) = tc::to_tf32(k0);
            *reinterpret_cast<float4*>(sK + tc::kmaj(rho, n0 + A, Npad)) = tc::to_tf32(k1);
          } else {
            const int n0 = 2 * A + 4 * (j - PQ);
            float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), kv = qv;
            if (in) {
              const float4 cu = *reinterpret_cast<const float4*>(crow + n0);
              const float4 bu = *reinterpret_cast<const float4*>(brow + n0);
              const float4 cbu = *reinterpret_cast<const float4*>(cb + n0);
              const float4 bbu = *reinterpret_cast<const float4*>(bb + n0);
              qv = make_float4(cu.x + cbu.x, cu.y + cbu.y, cu.z + cbu.z, cu.w + cbu.w);
              kv = make_float4(bu.x + bbu.x, bu.y + bbu.y, bu.z + bbu.z, bu.w + bbu.w);
            }
            if (!SUMMARY) *reinterpret_cast<float4*>(sQ + tc::kmaj(rho, n0, Npad)) = tc::to_tf32(qv);
            *reinterpret_cast<float4*>(sK + tc::kmaj(rho, n0, Npad)) = tc::to_tf32(kv);
          }
        }
      }
    } else {
      // Scalar path for A or N not a multiple of 4: unit u of a row is the
      // rotary pair (u, u + A) for u < A, else the single dim u + A.
      const int U = N - A;
      const int U4 = (U + 3) >> 2;
      const int rl = lane & 7, ul = lane >> 3;
      for (int rb = 0; rb < kRows / 8; ++rb) {
        const int rho = 8 * rb + rl;
        const int t = rho >> lgR, r = rho & (R - 1);
        const bool in = t < tv;
        const float* crow = a.c + ((tok0 + t) * RG + (int64_t)grp * R + r) * N;
        const float* brow = a.b + ((tok0 + t) * RG + (int64_t)grp * R + r) * N;
        const float* cb = sBiasC + r * Npad;
        const float* bb = sBiasB + r * Npad;
        for (int ub = warp; ub < U4; ub += kWarps) {
          const int u = 4 * ub + ul;
          if (u >= U) continue;
          if (u < A) {
            float q0 = 0.f, q1 = 0.f, k0 = 0.f, k1 = 0.f;
            if (in) {
              const float cs = sCos[t * CS + u], sn = sSin[t * CS + u];
              const float qu = crow[u] + cb[u], qw = crow[u + A] + cb[u + A];
              const float ku = brow[u] + bb[u], kw = brow[u + A] + bb[u + A];
              q0 = qu * cs - qw * sn;
              q1 = qu * sn + qw * cs;
              k0 = ku * cs - kw * sn;
              k1 = ku * sn + kw * cs;
            }
            if (!SUMMARY) {
              sQ[tc::kmaj(rho, u, Npad)] = tc::to_tf32(q0);
              sQ[tc::kmaj(rho, u + A, Npad)] = tc::to_tf32(q1);
            }
            sK[tc::kmaj(rho, u, Npad)] = tc::to_tf32(k0);
            sK[tc::kmaj(rho, u + A, Npad)] = tc::to_tf32(k1);
          } else {
            const int n = u + A;
            float qv = 0.f, kv = 0.f;
            if (in) {
              qv = crow[n] + cb[n];
              kv = brow[n] + bb[n];
            }
            if (!SUMMARY) sQ[tc::kmaj(rho, n, Npad)] = tc::to_tf32(qv);
            sK[tc::kmaj(rho, n, Npad)] = tc::to_tf32(kv);
          }
        }
      }
    }
    // key of the sequence's last token in fp32 for the step state (last chunk only)
    if (io.k_last && c0 + tv == L) {
      const int t = tv - 1;
      for (int i = tid; i < R * (N - A); i += kThreads) {
        const int r = i / (N - A), u = i - r * (N - A);
        const float* brow = a.b + ((tok0 + t) * RG + (int64_t)grp * R + r) * N;
        const float* bb = sBiasB + r * Npad;
        float* kl = io.k_last + ((int64_t)bh * R + r) * N;
        if (u < A) {
          const float cs = sCos[t * CS + u], sn = sSin[t * CS + u];
          const float ku = brow[u] + bb[u], kw = brow[u + A] + bb[u + A];
          kl[u] = ku * cs - kw * sn;
          kl[u + A] = ku * sn + kw * cs;
        } else {
          kl[u + A] = brow[u + A] + bb[u + A];
        }
      }
    }
    // zero padding columns N .. Npad
    for (int i = tid; i < kRows * (Npad - N); i += kThreads) {
      const int rho = i / (Npad - N), n = N + i % (Npad - N);
      sQ[tc::kmaj(rho, n, Npad)] = 0.f;
      sK[tc::kmaj(rho, n, Npad)] = 0.f;
    }
    __syncthreads();
    // (4b) w-scaled transposed keys Kt[n][row] = w_t * k[row][n] from the
    // TF32 k tile: lane l reads the 16 bytes of row 8 * rb + l % 8, dims
    // 4 * (4 * nb + l / 8) .. +3 (conflict-free), and writes them as four
    // scalars of column `row` of Kt.
    {
      const int rl = lane & 7, nl = lane >> 3;
      const int NQ = Npad >> 2;
      for (int rb = 0; rb < kRows / 8; ++rb) {
        const int rho = 8 * rb + rl;
        const int t = rho >> lgR;
        const float om = t < tv ? tOm[t] : 0.f;
        for (int nb = warp; nb < (NQ >> 2); nb += kWarps) {
          const int n0 = 4 * (4 * nb + nl);
          const float4 kv = *reinterpret_cast<const float4*>(sK + tc::kmaj(rho, n0, Npad));
          sKt[tc::kmaj(n0, rho, kRows)] = tc::to_tf32(om * kv.x);
          sKt[tc::kmaj(n0 + 1, rho, kRows)] = tc::to_tf32(om * kv.y);
          sKt[tc::kmaj(n0 + 2, rho, kRows)] = tc::to_tf32(om * kv.z);
          sKt[tc::kmaj(n0 + 3, rho, kRows)] = tc::to_tf32(om * kv.w);
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // (5) S = Q K^T and Yo^T = G Q^T
    if (!SUMMARY && tid == 0) {
      for (int ks = 0; ks < Npad / 8; ++ks)
        tc::mma_ss(tS, tc::kdesc(sQ, Npad, ks), tc::kdesc(sK, Npad, ks), id_S, ks > 0);
      tc::commit(&bars[0]);
      for (int ks = 0; ks < Npad / 8; ++ks)
        tc::mma_ts(tYo, tG + ks * 8, tc::kdesc(sQ, Npad, ks), id_Y, ks > 0);
      tc::commit(&bars[1]);
    }
    if (!SUMMARY) {
      if (!tc::bar_wait(&bars[0], it & 1, kWaitBudget)) abort_flag = 1;
      tc::fence_after();
      __syncthreads();
      if (abort_flag) break;
    }
    // (6) masked scores P = M o S (S rows: TMEM M = 64 layout, lanes 0..15 of
    // each quadrant; lane l + 16 takes the upper 8 columns of each 16-column
    // block of row l), values X^T, and G *= e^{cum_end}. The value loads are
    // issued first so that their latency overlaps the mask.
    {
      constexpr int kXr = (kRows / 4 + kWarps - 1) / kWarps;  // row blocks per warp
      float xreg[kXr][MP / 8];
      {
        const int pl8 = lane & 7, rl = lane >> 3;
#pragma unroll
        for (int q = 0; q < kXr; ++q) {
          const int rb = warp + kWarps * q;
          const int rho2 = 4 * rb + rl;
          const int t2 = rho2 >> lgR, r2 = rho2 & (R - 1);
          const bool in = rb < kRows / 4 && t2 < tv;
          const float* xrow = a.x + (tok0 + t2) * HP + (int64_t)h * P;
          const float* mx = mimo ? a.mimo_x + ((int64_t)h * R + r2) * P : nullptr;
#pragma unroll
          for (int pb = 0; pb < MP / 8; ++pb) {
            const int p = 8 * pb + pl8;
            float xv = (in && p < P) ? xrow[p] : 0.f;
            if (mimo && in && p < P) xv *= mx[p];
            xreg[q][pb] = xv;
          }
        }
      }
      if (!SUMMARY) {
      const int rho = 16 * quad + (lane & 15);
      const int t = rho >> lgR;
      const float cum_t = tCum[t];
      const float gam_t = tGam[t];
      const int sh = lane >> 4;
      for (int cb = 2 * wg; cb < 2 * wg + 2; ++cb) {
        float v[16];
        tc::tmem_ld16(tS + lane_base + cb * 16, v);
        float w8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float hi = __shfl_sync(0xffffffffu, v[j + 8], lane & 15);
          w8[j] = sh ? hi : v[j];
        }
        const int col0 = cb * 16 + 8 * sh;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int s = (col0 + j) >> lgR;
          float m = 0.f;
          if (s < t)
            m = __expf(cum_t - tCum[s]) * tW[s];
          else if (s == t)
            m = gam_t;
          w8[j] = tc::to_tf32(w8[j] * m);
        }
        *reinterpret_cast<float4*>(sP + tc::kmaj(rho, col0, kRows)) =
            make_float4(w8[0], w8[1], w8[2], w8[3]);
        *reinterpret_cast<float4*>(sP + tc::kmaj(rho, col0 + 4, kRows)) =
            make_float4(w8[4], w8[5], w8[6], w8[7]);
      }
      }
      // values X^T [p][row] (x * mimo_x for MIMO): lane l takes p = 8 * pb +
      // l % 8 and row 4 * rb + l / 8 (conflict-free scalar stores)
      {
        const int pl8 = lane & 7, rl = lane >> 3;
#pragma unroll
        for (int q = 0; q < kXr; ++q) {
          const int rb = warp + kWarps * q;
          if (rb >= kRows / 4) break;
          const int rho2 = 4 * rb + rl;
#pragma unroll
          for (int pb = 0; pb < MP / 8; ++pb)
            sXt[tc::kmaj(8 * pb + pl8, rho2, kRows)] = tc::to_tf32(xreg[q][pb]);
        }
      }
      // value of the sequence's last token for the step state (last chunk only)
      if (io.v_last && c0 + tv == L) {
        const float* xrow = a.x + (tok0 + tv - 1) * HP + (int64_t)h * P;
        for (int i = tid; i < R * P; i += kThreads) {
          const int r = i / P, p = i - r * P;
          io.v_last[((int64_t)bh * R + r) * P + p] =
              mimo ? xrow[p] * a.mimo_x[((int64_t)h * R + r) * P + p] : xrow[p];
        }
      }
      // G may be rescaled only once Yo^T = G Q^T has read it
      if (!SUMMARY) {
        if (!tc::bar_wait(&bars[1], it & 1, kWaitBudget)) abort_flag = 1;
        tc::fence_after();
      }
      const float ec = expf(tCum[Qt - 1]);
      for (int c = 16 * wg; c < Npad; c += 32) {
        float v[16];
        tc::tmem_ld16(tG + lane_base + c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = tc::to_tf32(v[j] * ec);
        tc::tmem_st16(tG + lane_base + c, v);
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // (7) Yi^T = X^T P^T and G += X^T (w K)
    if (abort_flag) break;
    if (tid == 0) {
      if (!SUMMARY) {
        for (int ks = 0; ks < kRows / 8; ++ks)
          tc::mma_ss(tS, tc::kdesc(sXt, kRows, ks), tc::kdesc(sP, kRows, ks), id_Y, ks > 0);
        tc::commit(&bars[2]);
      }
      for (int ks = 0; ks < kRows / 8; ++ks)
        tc::mma_ss(tG, tc::kdesc(sXt, kRows, ks), tc::kdesc(sKt, kRows, ks), id_D, 1);
      tc::commit(&bars[3]);
    }
    // next chunk's per-token scalars and angles: loads in flight during the
    // MMAs and the epilogue
    if (c0 + Qt < l1) preload_tokens(pl, a, tok0 + Qt, c0 + Qt, L, Qt, A, H, h, tid, warp, lane);
    if (!SUMMARY) {
      // SISO epilogue operands x, z of this thread's output column, loaded while
      // the MMAs run
      constexpr int kCols = (MP == 64) ? 8 : 16;
      float xe[2][kCols], ze[2][kCols];
      if (!mimo) {
        const float* xcol = a.x + tok0 * HP + (int64_t)h * P + prow;
        const float* zcol = a.z + tok0 * HP + (int64_t)h * P + prow;
  #pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col0 = (2 * wg + u) * 16 + 8 * half;
  #pragma unroll
          for (int j = 0; j < kCols; ++j) {
            const int t = col0 + j;
            const bool ok = pvalid && t < tv;
            xe[u][j] = ok ? xcol[t * HP] : 0.f;
            ze[u][j] = (ok && g.has_z) ? zcol[t * HP] : 0.f;
          }
        }
      }
      // the epilogue needs Yi only; the state update runs on under it
      if (!tc::bar_wait(&bars[2], it & 1, kWaitBudget)) abort_flag = 1;
      tc::fence_after();
      __syncthreads();
      if (abort_flag) break;
      // (8) epilogue: output column p of this chunk's tokens. With MP = 64 the
      // two lanes of a row split each 16-column block into 8 + 8 columns.
      {
        const float* xcol = a.x + tok0 * HP + (int64_t)h * P + prow;
        const float* zcol = a.z + tok0 * HP + (int64_t)h * P + prow;
        float* ocol = a.out + tok0 * HP + (int64_t)h * P + prow;
        for (int cb = 2 * wg; cb < 2 * wg + 2; ++cb) {
          float yo[16], yi[16];
          tc::tmem_ld16(tYo + lane_base + cb * 16, yo);
          tc::tmem_ld16(tS + lane_base + cb * 16, yi);
          if (MP == 64) {
  #pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float ho = __shfl_sync(0xffffffffu, yo[j + 8], lane & 15);
              const float hi = __shfl_sync(0xffffffffu, yi[j + 8], lane & 15);
              if (half) {
                yo[j] = ho;
                yi[j] = hi;
              }
            }
          }
          if (!pvalid) continue;
          const int col0 = cb * 16 + 8 * half;
          if (!mimo) {
            const int u = cb - 2 * wg;
  #pragma unroll
            for (int j = 0; j < kCols; ++j) {
              const int t = col0 + j;
              if (t < tv) {
                const float xv = u ? xe[1][j] : xe[0][j];
                const float zv = u ? ze[1][j] : ze[0][j];
                float y = tEc[t] * yo[j] + yi[j] + dsk * xv;
                if (g.has_z) y *= silu_fast(zv);
                ocol[t * HP] = y;
              }
            }
          } else {
            const int tpb = kCols >> lgR;  // whole tokens in this lane's columns
            for (int tt = 0; tt < tpb; ++tt) {
              const int t = (col0 >> lgR) + tt;
              if (t >= tv) break;
              const float xv = xcol[t * HP];
              const float zv = g.has_z ? zcol[t * HP] : 0.f;
              const float ec = tEc[t];
              float o = 0.f;
  #pragma unroll
              for (int r = 0; r < kRmax; ++r) {
                if (r < R) {
                  const int j = (tt << lgR) + r;
                  float y = ec * yo[j] + yi[j] + dsk * xv * mxr[r];
                  if (g.has_z) y *= silu_fast(zv * mzr[r]);
                  o += mor[r] * y;
                }
              }
              if (g.has_norm)
                sO[t * MP + prow] = o;
              else
                ocol[t * HP] = o;
            }
          }
        }
      }
      if (mimo && g.has_norm) {
        __syncthreads();
        for (int t = warp; t < tv; t += kWarps) {
          float ss = 0.f;
          for (int p = lane; p < P; p += 32) ss += sO[t * MP + p] * sO[t * MP + p];
          ss = warp_sum(ss);
          const float inv = 1.0f / sqrtf(ss / (float)P + 1.0e-5f);
          float* orow = a.out + (tok0 + t) * HP + (int64_t)h * P;
          for (int p = lane; p < P; p += 32)
            orow[p] = sO[t * MP + p] * inv * a.norm_weight[(int64_t)h * P + p];
        }
      }
    }
    // the state update must finish before the next chunk rewrites the tiles it
    // reads and issues Yo^T = G Q^T
    if (!tc::bar_wait(&bars[3], it & 1, kWaitBudget)) abort_flag = 1;
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (abort_flag) break;
  }
  if (abort_flag && tid == 0) atomicExch(status, kStatusTimeout);
  if (!abort_flag) {
    // final state, cumulative angle and decay of this segment
    if (io.g1) {
      float* g1 = io.g1 + ((int64_t)cta * P + prow) * N;
      for (int c = 16 * wg; c < Npad; c += 32) {
        float v[16];
        tc::tmem_ld16(tG + lane_base + c, v);
        if (g_lane) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < N) g1[c + j] = v[j];
        }
      }
    }
    if (io.g_last && l1 == L) {
      float* gl = io.g_last + ((int64_t)bh * P + prow) * N;
      for (int c = 16 * wg; c < Npad; c += 32) {
        float v[16];
        tc::tmem_ld16(tG + lane_base + c, v);
        if (g_lane) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < N) gl[c + j] = v[j];
        }
      }
    }
    if (io.th1)
      for (int i = tid; i < A; i += kThreads) io.th1[(int64_t)cta * A + i] = sThBase[i];
    if (io.th_last && l1 == L)
      for (int i = tid; i < A; i += kThreads) io.th_last[(int64_t)bh * A + i] = sThBase[i];
    if (io.e1 && tid == 0) io.e1[cta] = expf(esum);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, 256);
}

}  // namespace

bool chunk_supported(const ScanGeom& g) {
  return (g.R == 1 || g.R == 2 || g.R == 4 || g.R == 8) && g.N <= 128 && g.P <= 128;
}

int chunk_rows_per_token(const ScanGeom& g) { return kRows / g.R; }

cudaError_t launch_scan_chunk(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                              const ChunkIO& io, bool summary, cudaStream_t s) {
  const ChunkLayout lay = chunk_layout(g.N, g.P, g.A, g.R);
  const unsigned grid = (unsigned)(g.B * g.H * io.nseg);
  const bool mimo = a.mimo_o != nullptr;
  auto run = [&](auto kernel) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)lay.bytes);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, lay.bytes, s>>>(g, a, lay, io, status);
    return cudaSuccess;
  };
  cudaError_t e;
  if (summary) {
    if (lay.MP == 64)
      e = mimo ? run(k_scan_chunk<64, true, true>) : run(k_scan_chunk<64, false, true>);
    else
      e = mimo ? run(k_scan_chunk<128, true, true>) : run(k_scan_chunk<128, false, true>);
  } else {
    if (lay.MP == 64)
      e = mimo ? run(k_scan_chunk<64, true, false>) : run(k_scan_chunk<64, false, false>);
    else
      e = mimo ? run(k_scan_chunk<128, true, false>) : run(k_scan_chunk<128, false, false>);
  }
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace m3
