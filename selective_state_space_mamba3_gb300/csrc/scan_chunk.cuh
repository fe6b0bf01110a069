// Chunked Mamba-3 scan on the tcgen05 tensor cores (TF32 operands, FP32
// accumulation in tensor memory). Covers `mamba3_siso` and `mamba3_mimo`
// (oarust mamba3.rs) for mimo_rank R in {1, 2, 4, 8}, P <= 128, N <= 128.
// This header holds the kernel template; k_scan_chunk.cu instantiates the
// single-pass TF32 flavour and k_scan_chunk_split.cu the split-operand
// (3xTF32) flavour, in which every operand x is carried as hi(x) + lo(x) and
// every product takes three MMAs (hi hi + hi lo + lo hi), giving FP32-level
// accuracy (FP32-exact mode, and the MIMO output norm in TF32 mode).
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
//   Yi^T = X^T (M o S + D I)^T [P  x 64],  K = 64    (decay/trapezoid mask M;
//                                                   the D skip on the diagonal)
//   G   += X^T (w K)           [P  x N],   K = 64    (after G *= e^{cum_end})
// The state G [P x N] stays in TMEM for the whole sequence; outputs come out
// transposed (TMEM lane = p): each output column p is finished by the two
// lanes that share its TMEM row (e^{cum_t} Yo + Yi, SiLU gate, the MIMO mimo_o
// contraction over its R rows) and, through shared memory, the MIMO output
// RMS norm. Every operand is rounded to TF32 (round to nearest).
//
// One CTA of 256 threads runs one (b, h) sequence chunk after chunk; threads 0
// and 32 issue the MMAs (one independent chain each), and threads wait on
// mbarriers signalled by tcgen05.commit. Staging is warp-local: warp w owns
// rows 8w .. 8w + 7 of the chunk (its tokens' scalars, rotary angles and the
// q / k / w-scaled transposed key tiles), so three block barriers precede the
// epilogue (after the per-warp totals, before the first and before the second
// MMA batch); the staged SISO epilogue adds two (its output rows, and before
// the next chunk's B rows reuse the region). The state update of a chunk runs
// on under its epilogue and the next chunk's scalar work. The C / B rows of a
// chunk arrive by TMA (one issuing thread, 4-D boxes into 128-byte-swizzled
// tiles) a chunk ahead of their use.
// Waits are bounded: on timeout the kernel records a status word and exits.
// Shared memory (at most about 114 KB for P <= 64, N = 128) and TMEM (256
// columns) admit two CTAs per SM, and the next chunk's other inputs are
// prefetched into L2 while the current chunk runs.
//
// The kernel is a template over the shape: the generic instance reads N, A, R
// and P at run time; instances for common shapes have them as constants. The
// compile-time shape selects these variants (constexpr flags in the kernel):
//   kAsync     C / B rows by TMA into swizzled tiles (N % 32 == 0, A <= 64,
//              A % 4 == 0); otherwise 128-bit loads into unswizzled tiles.
//   kSplitK    (kAsync, N <= 64) the scores get a region of their own, so the
//              k tile is dead once S is done.
//   kEarlyB    the next chunk's B rows are copied as soon as the k tile is
//              dead: after the tile phase in the summary pass, after S with
//              kSplitK.
//   kBAtEpi    (kAsync SISO main pass without kEarlyB) the epilogue stages its
//              rows in the transposed-key tile and the B copy starts with the
//              epilogue; otherwise it follows a final block barrier.
//   kThInKt    (kAsync, A > 32) the rotary angles live in each warp's part of
//              the transposed-key tile; with kAsync and A <= 32 in their own
//              region; without kAsync in the warp's q rows.
//   kCosSin    (kAsync MIMO) the angle slots hold cos and sin per (token,
//              angle), computed once instead of per rank row.
//   kFactMask  (SISO) the factored decay mask for chunks with sum |adt| <= 85.
//   kXVec, kStaged, kTpb: float4 value loads, staged float4 epilogue (SISO),
//              z preloaded before the epilogue waits (MIMO).
#pragma once

#include <cuda.h>
#include <string.h>
#include <cudaTypedefs.h>

#include "m3_internal.cuh"
#include "tc_ptx.cuh"

namespace m3 {
namespace {

constexpr int kRows = 64;       // (token, rank) rows per chunk
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTok = 72;        // per-token array stride (>= 65)
constexpr int kAngMax = 64;     // A <= 64
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (~2 s)
// Lazy state scaling: TMEM holds G~ with G = e^{lgE} G~, and G~ is rescaled
// only when the log decay accumulated since the last rescale would pass
// -kLazyRange (so |G~| <= e^{kLazyRange} |G|).
constexpr float kLazyRange = 40.0f;

struct ChunkLayout {
  int Npad, MP;
  int q, k, kt, tot, bias, tok, thbase, th, o, p;  // float offsets of the regions
  int lo;        // split operands: float distance from each operand tile to its low part
  size_t bytes;
};

// Instances with compile-time N and A (N a multiple of 32, A <= 64 and a
// multiple of 4) stage the C / B rows of a chunk by TMA: one 4-D box per
// 32-column block lands in a 128-byte-swizzled K-major q / k tile, which the
// threads then rotate in place. Each warp's rotary angles live in a region of
// their own for A <= 32; for larger A, which would not fit beside the tiles,
// in the warp's private part of the transposed key tile (rows 8w .. 8w + 7 of
// every 8-dim group: 64 contiguous floats per group), which is free from the
// previous state update until the warp writes its own keys. The MIMO norm
// staging has a region of its own.
__host__ __device__ constexpr bool chunk_async(int KN, int KA) {
  return KN > 0 && KA > 0 && KA <= 64 && KN % 32 == 0 && KA % 4 == 0 &&
         8 * (KA + 4) <= 64 * (KN / 8);  // a warp's angles fit its key-tile part
}
constexpr int kTmaThread = 64;  // issues the TMA copies (warp 2, lane 0)

int imax(int a, int b) { return a > b ? a : b; }

ChunkLayout chunk_layout(int N, int P, int A, int R, bool mimo, bool async, bool split) {
  ChunkLayout l;
  l.Npad = (N + 15) / 16 * 16;
  l.MP = P <= 64 ? 64 : 128;
  const int Qt = kRows / R;
  int off = 0;
  auto take = [&](int floats) {
    int o = off;
    off += (floats + 31) / 32 * 32;  // 128-byte aligned regions
    return o;
  };
  // Q region: q tile [64][Npad]; without TMA staging each warp's 8-row
  // block first holds that warp's rotary angles, and the MIMO norm staging
  // [Qt][MP] uses the region in the epilogue.
  l.q = take(async ? kRows * l.Npad : imax(kRows * l.Npad, Qt * l.MP));
  // K region: k tile [64][Npad] until S = Q K^T completes, then the masked
  // scores [64][64] followed by the values X^T [MP][64]. With TMA staging and
  // N <= 64 (split), the values follow the k tile and the scores have a region
  // of their own, so that the next chunk's B rows can land once S is done.
  const bool split_k = async && N <= 64;
  const bool split_ops = split;
  l.k = take(split_k ? kRows * l.Npad + l.MP * kRows
                     : imax(kRows * l.Npad, kRows * kRows + l.MP * kRows));
  // Kt region: w-scaled transposed keys [Npad][64] (K-major, K = row).
  l.kt = take(l.Npad * kRows);
  l.p = split_k ? take(kRows * kRows) : 0;               // masked scores (split K region)
  // Split operands: the low parts of every operand tile (q, K region, Kt,
  // scores) sit `lo` floats after their high parts, in the same layout; `lo`
  // is a multiple of 1024 bytes so that swizzled tiles stay aligned.
  l.lo = split_ops ? (off + 255) / 256 * 256 : 0;
  if (split_ops) off = 2 * l.lo;
  l.tot = take(kWarps * kAngMax + 2 * kWarps);  // per-warp angle, log-decay, |log-decay| totals
  l.bias = take(2 * R * (l.Npad + 4));      // c_bias, b_bias of this head, zero-padded rows
  l.tok = take(6 * kTok);                   // cum, e^{cum + lgE}, gamma, w, e^cum, e^-cum w
  l.thbase = take(2 * kAngMax);             // cumulative angle at the chunk start (x2)
  // per-warp angles [TPW][A + 4] (TMA staging with A <= 32); MIMO keeps their
  // cosines and sines instead (two such blocks per warp)
  l.th = (async && A <= 32) ? take(kWarps * (8 / R) * (A + 4) * (mimo && R > 1 ? 2 : 1)) : 0;
  l.o = (async && mimo) ? take(Qt * l.MP) : 0;          // MIMO norm staging
  l.bytes = (size_t)off * sizeof(float);
  return l;
}

__host__ __device__ constexpr int ilog2c(int v) { return v <= 1 ? 0 : 1 + ilog2c(v >> 1); }

// Per-token scalars and angle increments of one chunk, loaded into registers
// one chunk ahead. Warp w owns tokens TPW * w .. TPW * w + TPW - 1 (TPW = 8 /
// R); lane i <= TPW holds the dt / adt / trap of token TPW * w + i (lane TPW:
// the first token after the warp's, whose trapezoid scale the warp's last
// token needs), and ang[2 i + j] is the increment of angle lane + 32 j of the
// warp's token i.
struct TokenPreload {
  float dt, adt, trap;
  float inv_b, inv_c;  // packed projection: inverse RMS of the token's B / C row
  float ang[16];
};

// Packed projection (PACKED): trap and angle from their columns of the packed
// rows (row stride W), dt / adt and the B / C inverse RMS from the row pass.
template <bool PACKED>
__device__ __forceinline__ void preload_tokens(TokenPreload& pl, const ScanArgs& a,
                                               const ScanGeom& g, int64_t tok, int cn, int L,
                                               int TPW, int A, int H, int h, int warp, int lane) {
  pl.dt = pl.adt = pl.trap = 0.f;
  pl.inv_b = pl.inv_c = 1.f;
  const int tw = TPW * warp + lane;
  const int64_t rs = PACKED ? (int64_t)g.W : (int64_t)H;  // row stride of the trap column
  if (lane <= TPW && cn + tw < L) {
    const int64_t sc = (tok + tw) * H + h;
    pl.dt = a.dt[sc];
    pl.adt = a.adt[sc];
    pl.trap = a.trap[(tok + tw) * rs + h];
    if constexpr (PACKED) {
      // (SISO: one B and one C row per group)
      const int grp = h / (H / g.G);
      const float* ri = a.row_inv + (tok + tw) * 2 * g.G;
      pl.inv_b = ri[grp];
      pl.inv_c = ri[g.G + grp];
    }
  }
  const int64_t ars = PACKED ? (int64_t)g.W : (int64_t)A;  // row stride of the angle columns
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int t = TPW * warp + i, aa = lane + 32 * j;
      pl.ang[2 * i + j] =
          (i < TPW && aa < A && cn + t < L) ? a.angle[(tok + t) * ars + aa] : 0.f;
    }
  }
}

// Writes w * v, rounded for the tensor core, into rows n0..n0+3 (n0 % 4 == 0) of column
// rho of the transposed key tile. Step i stores component (i + rot) & 3: with
// the phase-(4) lane mapping and rot = 2 * (lane / 16) + (lane / 4) % 2, the
// 32 lanes' stores of one step land in 32 distinct banks.
// Paired FP32 arithmetic (FADD2 / FMUL2 / FFMA2: two IEEE single-precision
// operations per instruction) on the (x, y) and (z, w) halves of float4s.
__device__ __forceinline__ float4 cat4(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return cat4(__fadd2_rn(lo2(a), lo2(b)), __fadd2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  return cat4(__fmul2_rn(lo2(a), lo2(b)), __fmul2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {
  return cat4(__ffma2_rn(lo2(a), lo2(b), lo2(c)), __ffma2_rn(hi2(a), hi2(b), hi2(c)));
}
// Paired multiply in inline PTX: the compiler cannot merge it with a
// following add into a fused multiply-add, so each product is rounded on its
// own (as a separately stored product would be).
__device__ __forceinline__ float2 mul2_sep(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ta, tb, td;\n\tmov.b64 ta, {%2, %3};\n\tmov.b64 tb, {%4, %5};\n\t"
      "mul.rn.f32x2 td, ta, tb;\n\tmov.b64 {%0, %1}, td;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Split operands: the low part (the rounded remainder) of each value goes to
// the same position LO floats further on.
template <bool SPLIT>
__device__ __forceinline__ void store_kt4(float* kt, int LO, int n0, int rho, float4 v, float w,
                                          int rot) {
  const float4 pw = mul4(v, make_float4(w, w, w, w));
  const float p0 = pw.x, p1 = pw.y, p2 = pw.z, p3 = pw.w;
  const float a0 = SPLIT ? tc::tf32_clean(p0) : tc::tf32_feed(p0);
  const float a1 = SPLIT ? tc::tf32_clean(p1) : tc::tf32_feed(p1);
  const float a2 = SPLIT ? tc::tf32_clean(p2) : tc::tf32_feed(p2);
  const float a3 = SPLIT ? tc::tf32_clean(p3) : tc::tf32_feed(p3);
  const bool r1 = rot & 1, r2 = rot & 2;
  float* base = kt + tc::kmaj(n0, rho, 64);  // row n0 + c is 4 * c floats further
  {
    const float s0 = r1 ? a1 : a0, s1 = r1 ? a2 : a1, s2 = r1 ? a3 : a2, s3 = r1 ? a0 : a3;
    const float t0 = r2 ? s2 : s0, t1 = r2 ? s3 : s1, t2 = r2 ? s0 : s2, t3 = r2 ? s1 : s3;
    base[((rot + 0) & 3) * 4] = t0;
    base[((rot + 1) & 3) * 4] = t1;
    base[((rot + 2) & 3) * 4] = t2;
    base[((rot + 3) & 3) * 4] = t3;
  }
  if constexpr (SPLIT) {
    const float b0 = tc::tf32_feed(p0 - a0), b1 = tc::tf32_feed(p1 - a1);
    const float b2 = tc::tf32_feed(p2 - a2), b3 = tc::tf32_feed(p3 - a3);
    const float s0 = r1 ? b1 : b0, s1 = r1 ? b2 : b1, s2 = r1 ? b3 : b2, s3 = r1 ? b0 : b3;
    const float t0 = r2 ? s2 : s0, t1 = r2 ? s3 : s1, t2 = r2 ? s0 : s2, t3 = r2 ? s1 : s3;
    base[LO + ((rot + 0) & 3) * 4] = t0;
    base[LO + ((rot + 1) & 3) * 4] = t1;
    base[LO + ((rot + 2) & 3) * 4] = t2;
    base[LO + ((rot + 3) & 3) * 4] = t3;
  }
}

// Operand stores. Single pass: the value with half a TF32 unit added (the MMA
// then sees it rounded to nearest). Split: the value rounded to TF32 (low bits
// cleared) into the tile and the rounded remainder into its low part at LO.
template <bool SPLIT>
__device__ __forceinline__ void put1(float* dst, int LO, float v) {
  if constexpr (SPLIT) {
    const float hi = tc::tf32_clean(v);
    dst[0] = hi;
    dst[LO] = tc::tf32_feed(v - hi);
  } else {
    dst[0] = tc::tf32_feed(v);
  }
}
template <bool SPLIT>
__device__ __forceinline__ void put4(float* dst, int LO, float4 v) {
  if constexpr (SPLIT) {
    const float4 hi = make_float4(tc::tf32_clean(v.x), tc::tf32_clean(v.y), tc::tf32_clean(v.z),
                                  tc::tf32_clean(v.w));
    *reinterpret_cast<float4*>(dst) = hi;
    *reinterpret_cast<float4*>(dst + LO) =
        make_float4(tc::tf32_feed(v.x - hi.x), tc::tf32_feed(v.y - hi.y),
                    tc::tf32_feed(v.z - hi.z), tc::tf32_feed(v.w - hi.w));
  } else {
    *reinterpret_cast<float4*>(dst) = tc::tf32_feed(v);
  }
}

// SiLU with the hardware exp / divide approximations (relative error a few
// float32 ulps, far inside the scan tolerances).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }
// SFU base-2 exponential and reciprocal (PTX ex2.approx / rcp.approx).
__device__ __forceinline__ float ex2_sfu(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float rcp_sfu(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// y * silu(z) = y z / (1 + 2^(-z log2 e)) for four values: the exponential
// and the reciprocal on the SFU, the rest as paired FP32 operations (relative
// error a few float32 units, like the scalar silu_fast).
__device__ __forceinline__ float4 gate4(float4 y, float4 z) {
  const float l2e = -1.4426950408889634f;
  const float4 a = mul4(z, make_float4(l2e, l2e, l2e, l2e));
  const float4 e = make_float4(ex2_sfu(a.x), ex2_sfu(a.y), ex2_sfu(a.z), ex2_sfu(a.w));
  const float4 d = add4(e, make_float4(1.f, 1.f, 1.f, 1.f));
  const float4 r = make_float4(rcp_sfu(d.x), rcp_sfu(d.y), rcp_sfu(d.z), rcp_sfu(d.w));
  return mul4(y, mul4(z, r));
}

template <int MP, bool MIMO, bool SUMMARY, int KN, int KA, int KR, int KP, bool SPLIT,
          bool PACKED>
__global__ void __launch_bounds__(kThreads, SPLIT ? 1 : 2)
    k_scan_chunk(ScanGeom g, ScanArgs a, ChunkLayout lay, ChunkIO io, uint32_t* status,
                 const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ __align__(1024) float sm_raw[];
  constexpr bool kAsync = chunk_async(KN, KA);
  // swizzled tiles start on a 1024-byte boundary (1 KB of slack is allocated)
  float* sm = kAsync ? sm_raw + ((1024u - (tc::smem_u32(sm_raw) & 1023u)) & 1023u) / 4 : sm_raw;
  // Completion barriers, each completing once per chunk: MMAs S, Yo, Yi and
  // state update; TMA copies of the C rows and of the B rows.
  __shared__ __align__(8) uint64_t bars[6];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = g.H, L = g.L;
  const int P = KP ? KP : g.P;
  const int N = KN ? KN : g.N;
  const int A = KA ? KA : g.A;
  const int R = KR ? KR : g.R;
  const int lgR = KR ? ilog2c(KR) : __ffs(R) - 1;  // R is a power of two here
  const int Npad = KN ? (KN + 15) / 16 * 16 : lay.Npad;
  const int Qt = kRows >> lgR;  // tokens per chunk
  const int TPW = Qt >> 3;      // tokens per warp
  const int cta = blockIdx.x;
  const int bh = cta / io.nseg, seg = cta - bh * io.nseg;
  const int b = bh / H, h = bh % H;
  const int l0 = seg * io.seg_len, l1 = min(L, l0 + io.seg_len);
  // the summaries of the main pass's last segment are never used
  if (SUMMARY && seg >= io.nseg - io.sum_skip) return;
  const int grp = h / (H / g.G);
  const int RG = g.G * R;

  // Split operands (3xTF32): every operand tile X has a low part at X + LO
  // holding x - hi(x), and each product takes three MMAs (hi hi, hi lo, lo hi).
  const int LO = SPLIT ? lay.lo : 0;
  float* sQ = sm + lay.q;              // [64 rows][Npad] K-major, K = n
  float* sO = (kAsync && MIMO) ? sm + lay.o : sQ;  // [Qt][MP] MIMO epilogue staging
  float* sK = sm + lay.k;              // [64 rows][Npad] K-major, K = n
  // With TMA staging the next chunk's B rows are copied as soon as the k tile
  // is dead (kEarlyB): in the summary pass (no S; the values then use the
  // unused q tile) right after the tiles are built, and with split regions
  // (N <= 64) once S = Q K^T completes; otherwise after the state update.
  constexpr bool kSplitK = kAsync && KN <= 64;
  constexpr bool kFactMask = KR == 1;  // factored decay mask (compile-time SISO)
  constexpr bool kEarlyB = kAsync && (SUMMARY || kSplitK);
  float* sP = kSplitK ? sm + lay.p : sK;  // [64][64]      masked scores (after S)
  // [MP][64 rows] values (after S)
  float* sXt = (kAsync && SUMMARY) ? sQ : sK + (kSplitK ? kRows * Npad : kRows * kRows);
  float* sKt = sm + lay.kt;            // [Npad][64 rows] K-major, K = row (w-scaled keys)
  // Staged SISO epilogue with TMA staging and no early B copy: the output rows
  // are staged in the transposed key tile, free once the chunk's state update
  // has read it, so the next chunk's B rows can be copied into the K region as
  // soon as Yi and the state update are done (start of the epilogue).
  constexpr bool kStagedEpi = !MIMO && !SUMMARY && KP > 0 && KP % 4 == 0 && KP <= 64;
  constexpr bool kBAtEpi = kAsync && !kEarlyB && kStagedEpi;
  float* sStage = kBAtEpi ? sKt : sP;  // [t][P] pre-gate output rows
  // Row t starts at t * P + 16 (t / 8) (in the transposed key tile, which has
  // room): lanes l and l + 16 stage tokens t and t + 8 of the same column, and
  // the extra 16 floats per group of 8 rows put their stores in different
  // banks while keeping the rows disjoint and 16-byte aligned.
  constexpr int kStageSkew = kBAtEpi ? 16 : 0;
  float* sTot = sm + lay.tot;          // [8 warps][64]   per-warp angle totals
  float* sTotAdt = sTot + kWarps * kAngMax;  // [8 warps] per-warp log-decay totals
  // bias rows of Npad + 4 floats: the ranks of a row block read the same
  // columns at once, and the extra 16 bytes per row put them on different banks
  const int BS = Npad + 4;
  float* sBiasC = sm + lay.bias;       // [R][BS]
  float* sBiasB = sBiasC + R * BS;     // [R][BS]
  float* tCum = sm + lay.tok;          // local cumulative log decay
  float* tEc = tCum + kTok;            // e^{cum_t}
  float* tGam = tEc + kTok;            // gamma_t
  float* tW = tGam + kTok;             // gamma_t + scale_{t+1}
  float* tEa = tW + kTok;              // e^{cum_t}            (factored mask)
  float* tEb = tEa + kTok;             // e^{-cum_t} w_t       (factored mask)
  float* sAbsAdt = sTotAdt + kWarps;   // [8 warps] per-warp totals of |adt|
  float* sThBase = sm + lay.thbase;    // [2][64] cumulative angle before the chunk
  const int AS = A + 4;                // angle row stride of a warp's angle block
  // this warp's angles [TPW][AS]: element k at thp(k) (TMA staging: in their
  // own region for A <= 32, else in the warp's part of the transposed key
  // tile; without TMA staging: in the warp's q rows)
  constexpr bool kThInKt = kAsync && KA > 32;
  // MIMO with TMA staging: phase (2) stores cos and sin per (token, angle) once,
  // instead of every one of a token's R rows computing them in phase (4)
  constexpr bool kCosSin = MIMO && KR > 1 && kAsync && !kThInKt;
  float* sTh = kAsync ? sm + lay.th + warp * TPW * AS * (kCosSin ? 2 : 1) : sQ + warp * 8 * Npad;
  auto thp = [&](int k) -> float* {
    return kThInKt ? sKt + (((k >> 6) * 16 + 2 * warp) << 5) + (k & 63) : sTh + k;
  };

  if (tid == 0) {
    for (int i = 0; i < 6; ++i) tc::bar_init(&bars[i], 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  // TMEM columns: G [0, 128), S / Yi [128, 192), Yo [192, 256); split: the low
  // part of G at [256, 384) (one CTA per SM then, so 512 columns are free)
  constexpr uint32_t kTmemCols = SPLIT ? 512 : 256;
  if (warp == 0) tc::tmem_alloc(&tmem_slot, kTmemCols);
  for (int i = tid; i < A; i += kThreads) sThBase[i] = io.th0 ? io.th0[(int64_t)cta * A + i] : 0.f;
  for (int i = tid; i < R * BS; i += kThreads) {
    const int r = i / BS, n = i - r * BS;
    sBiasC[i] = n < N ? a.c_bias[((int64_t)h * R + r) * N + n] : 0.f;
    sBiasB[i] = n < N ? a.b_bias[((int64_t)h * R + r) * N + n] : 0.f;
  }
  // padding rows N .. Npad of the transposed key tile stay zero
  for (int i = tid; i < (Npad - N) * kRows; i += kThreads) {
    const int n = N + i / kRows, rho = i % kRows;
    sKt[tc::kmaj(n, rho, kRows)] = 0.f;
    if (SPLIT) sKt[tc::kmaj(n, rho, kRows) + LO] = 0.f;
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = tmem_slot;
  // TMEM lane quadrant of this warp (warps w and w + 4 share quadrant w % 4 and
  // split the columns of the row-wise TMEM work between them)
  const int quad = warp & 3, wg = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
  const uint32_t tG = tbase, tS = tbase + 128, tYo = tbase + 192, tGl = tbase + 256;
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
    // (N % 16 == 0: a 16-column block is wholly inside the row or wholly past
    // it, and the row bases are 16-byte aligned, so it moves as four float4s)
    const bool vec16 = N % 16 == 0;
    for (int c = 16 * wg; c < Npad; c += 32) {
      float v[16];
      if (vec16) {
        const bool on = g0 && g_lane && c < N;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 u = on ? reinterpret_cast<const float4*>(g0 + c)[q]
                              : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * q] = u.x;
          v[4 * q + 1] = u.y;
          v[4 * q + 2] = u.z;
          v[4 * q + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = (g0 && g_lane && c + j < N) ? g0[c + j] : 0.f;
      }
      tc::tmem_st16(tG + lane_base + c, v);
    }
  }
  constexpr bool mimo = MIMO;
  constexpr int kRmax = MIMO ? 8 : 1;
  float mzr[kRmax], mor[kRmax];
#pragma unroll
  for (int r = 0; r < kRmax; ++r) {
    const bool ok = mimo && pvalid && r < R;
    mzr[r] = ok ? a.mimo_z[((int64_t)h * R + r) * P + prow] : 1.f;
    mor[r] = ok ? a.mimo_o[((int64_t)h * R + r) * P + prow] : 0.f;
  }
  const float dsk = g.has_d ? a.d[h] : 0.f;
  // MIMO with compile-time R <= 4: the value rows 4 rb + l / 8 of this lane all
  // have rank (l / 8) mod R, so its mimo_x factors (columns 8 pb + l % 8) are
  // loaded once and applied when the values are stored
  constexpr bool kMxPre = MIMO && KR > 0 && KR <= 4;
  float mxr[kMxPre ? MP / 8 : 1];
#pragma unroll
  for (int pb = 0; pb < (kMxPre ? MP / 8 : 1); ++pb) {
    const int p = 8 * pb + (lane & 7), r2 = (lane >> 3) & (R - 1);
    mxr[pb] = (kMxPre && p < P) ? a.mimo_x[((int64_t)h * R + r2) * P + p] : 1.f;
  }
  const uint32_t id_S = tc::idesc_tf32(64, 64);
  const uint32_t id_Y = tc::idesc_tf32(MP, 64);
  const uint32_t id_D = tc::idesc_tf32(MP, Npad);
  const int64_t HP = (int64_t)H * P;
  // row stride of the x and z rows: H * P in their own tensors, W in the
  // packed projection (PACKED: x and z are column slices of the packed rows)
  const int64_t XS = PACKED ? (int64_t)g.W : HP;
  static_assert(!PACKED || kAsync, "the packed projection is read by TMA instances only");
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  // L2 prefetch plan: the blocks of x, z, C, B, dt, adt, trap and angle of a
  // chunk are contiguous across the heads of a batch row, so the H CTAs of the
  // row (resident together) each prefetch one 16-byte-aligned slice of every
  // block; lane 0 of warp i handles block i.
  uintptr_t pf_base = 0, pf_bytes = 0, pf_off0 = 0, pf_off1 = 0;
  if (lane == 0) {
    const float* base = nullptr;
    int64_t per_tok = 0;  // floats per token
    if (PACKED) {
      // the packed rows of a chunk are contiguous: warp 0 takes this head's slice
      if (warp == 0) {
        base = a.z;
        per_tok = g.W;
      }
    } else switch (warp) {
      case 0: base = a.x; per_tok = HP; break;
      case 1: base = a.z; per_tok = HP; break;
      case 2: base = a.c; per_tok = (int64_t)RG * N; break;
      case 3: base = a.b; per_tok = (int64_t)RG * N; break;
      case 4: base = a.dt; per_tok = H; break;
      case 5: base = a.adt; per_tok = H; break;
      case 6: base = a.trap; per_tok = H; break;
      default: base = a.angle; per_tok = A; break;
    }
    if (base && per_tok > 0) {
      pf_base = reinterpret_cast<uintptr_t>(base);
      pf_bytes = (uintptr_t)per_tok * sizeof(float);
      const uintptr_t span = (uintptr_t)Qt * pf_bytes;
      pf_off0 = span * h / H & ~uintptr_t(15);
      pf_off1 = span * (h + 1) / H & ~uintptr_t(15);
    }
  }
  // MMA operand descriptors; K step ks adds 16 * ks (256 bytes) to each
  const uint64_t dQ = kAsync ? tc::swdesc(sQ) : tc::kdesc(sQ, Npad, 0);
  const uint64_t dK = kAsync ? tc::swdesc(sK) : tc::kdesc(sK, Npad, 0);
  const uint64_t dXt = tc::kdesc(sXt, kRows, 0), dP = tc::kdesc(sP, kRows, 0);
  const uint64_t dKt = tc::kdesc(sKt, kRows, 0);
  // low parts (split operands): the same tiles LO floats further on
  const uint64_t dQl = SPLIT ? (kAsync ? tc::swdesc(sQ + LO) : tc::kdesc(sQ + LO, Npad, 0)) : 0;
  const uint64_t dKl = SPLIT ? (kAsync ? tc::swdesc(sK + LO) : tc::kdesc(sK + LO, Npad, 0)) : 0;
  const uint64_t dXtl = SPLIT ? tc::kdesc(sXt + LO, kRows, 0) : 0;
  const uint64_t dPl = SPLIT ? tc::kdesc(sP + LO, kRows, 0) : 0;
  const uint64_t dKtl = SPLIT ? tc::kdesc(sKt + LO, kRows, 0) : 0;

  // Row and items of this lane in phase (4): row 8 * warp + l % 8, items
  // 4 * jb + l / 8.
  const int rl = lane & 7, jl = lane >> 3;
  const int rho = 8 * warp + rl;
  const int t = rho >> lgR, r = rho & (R - 1);
  // Offset of element (row, n) in the q / k tiles, and the descriptor advance
  // of MMA K step ks over them.
  auto toff = [&](int row, int n) { return kAsync ? tc::sw128(row, n, kRows) : tc::kmaj(row, n, Npad); };
  auto qk_step = [&](int ks) -> uint64_t { return kAsync ? tc::swdesc_kstep(ks, kRows) : 16u * ks; };
  // TMA staging (thread kTmaThread): the C (or B) rows of the chunk starting at
  // token t_start of the sequence into a q (or k) tile, one box [Qt tokens][R
  // ranks][32 dims] per column block; rows past the sequence end read zeros.
  int pendC = -1, pendB = -1;  // chunk whose copy is in flight (issuing thread)
  auto issue_rows = [&](const CUtensorMap* tm, float* tile, int t_start, uint64_t* bar) {
    tc::bar_expect_tx(bar, (uint32_t)(kRows * N * 4));
#pragma unroll
    for (int cb = 0; cb < (KN > 0 ? KN : 128) / 32; ++cb)
      tc::tma_load_4d(tile + cb * kRows * 32, tm, 32 * cb, grp * R, t_start, b, bar);
  };
  if (kAsync && tid == kTmaThread && l0 < l1) {
    if (!SUMMARY) {
      issue_rows(&tmC, sQ, l0, &bars[4]);
      pendC = 0;
    }
    issue_rows(&tmB, sK, l0, &bars[5]);
    pendB = 0;
  }

  TokenPreload pl;
  // a programmatic dependent launch runs the prologue above (and the first C /
  // B row copies) under the tail of the kernel before it; its results (the row
  // norms the preload reads) are waited for here
  if constexpr (PACKED) {
    if (io.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  preload_tokens<PACKED>(pl, a, g, (int64_t)b * L + l0, l0, L, TPW, A, H, h, warp, lane);
  float esum = 0.f;  // sum of adt over the segment
  float lgE = 0.f;   // G = e^{lgE} G~ (identical in every thread)

  int it = 0;
  for (int c0 = l0; c0 < l1; c0 += Qt, ++it) {
    const int tv = min(Qt, l1 - c0);
    const int64_t tok0 = (int64_t)b * L + c0;   // first token of the chunk in [B, L]
    const float* thb_cur = sThBase + (it & 1) * kAngMax;
    float* thb_next = sThBase + ((it & 1) ^ 1) * kAngMax;
    // (0) L2 prefetch of the next chunk's operands (slices fixed before the loop)
    if (pf_bytes && c0 + Qt < l1) {
      const int nv = min(Qt, l1 - c0 - Qt);
      const uintptr_t lo = pf_base + (uintptr_t)(tok0 + Qt) * pf_bytes;
      const uintptr_t hi = lo + (uintptr_t)nv * pf_bytes;
      if (((lo | hi) & 15) == 0) {
        const uintptr_t s0 = lo + pf_off0;
        const uintptr_t s1 = (h + 1 == H) ? hi : min(lo + pf_off1, hi);
        if (s1 > s0) tc::prefetch_l2(reinterpret_cast<const void*>(s0), (uint32_t)(s1 - s0));
      }
    }
    // (1) per-warp token scalars; local (within the warp's tokens) inclusive
    // sums of the log decay and of dt * angle, whose warp totals go to shared
    // memory. Lane i <= TPW: token TPW * warp + i.
    const int tw = TPW * warp + lane;
    float dtv = 0.f, adtv = 0.f, gam = 0.f, scl = 0.f;
    if (lane <= TPW) {
      // (single pass: SFU exponential and division; split: the accurate ones)
      const float lam = SPLIT ? sigmoid_f(pl.trap) : __fdividef(1.0f, 1.0f + __expf(-pl.trap));
      if (c0 + tw < L) scl = (1.0f - lam) * pl.dt;
      if (tw < tv && lane < TPW) {
        dtv = pl.dt;
        adtv = pl.adt;
        gam = lam * pl.dt;
      }
    }
    float cl = adtv;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, cl, o);
      if (o < TPW && lane >= o) cl += u;
    }
    const float adt_tot = __shfl_sync(0xffffffffu, cl, TPW - 1);
    if (lane == 0) sTotAdt[warp] = adt_tot;
    if (kFactMask) {
      float aab = fabsf(adtv);  // lanes 0 .. TPW - 1 hold the warp's tokens
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) aab += __shfl_xor_sync(0xffffffffu, aab, o);
      if (lane == 0) sAbsAdt[warp] = aab;
    }
    float thl[2][8], dsh[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) dsh[i] = __shfl_sync(0xffffffffu, dtv, i);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < TPW && 32 * j < A) s = fmaf(dsh[i], pl.ang[2 * i + j], s);
        thl[j][i] = s;
      }
      const int aa = lane + 32 * j;
      if (aa < A) sTot[warp * kAngMax + aa] = s;
    }
    __syncthreads();  // B1: totals visible; previous chunk's epilogue finished
    if (abort_flag) break;
    const bool in = t < tv;  // this lane's phase-(4) row holds a valid token
    const int64_t roff = ((tok0 + t) * RG + (int64_t)grp * R + r) * N;
    const float* crow = a.c + roff;
    const float* brow = a.b + roff;
    // (2) per-token coefficients (lane i < TPW) and this warp's angles
    float cend = 0.f, cbase = 0.f, aabs = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float v = sTotAdt[w];
      if (w < warp) cbase += v;
      cend += v;
      if (kFactMask) aabs += sAbsAdt[w];
    }
    // Factored mask (SISO instances): with sum |adt| <= 85 over the chunk
    // every |cum_t| <= 85, so e^{cum_t - cum_s} w_s = e^{cum_t} (e^{-cum_s} w_s)
    // with both factors normal floats, computed once per token instead of once
    // per (t, s)
    const bool fact = kFactMask && aabs <= 85.0f;
    esum += cend;
    // lazy chunk: G~ keeps its scale, e^{-lgE_new} goes into the w-scaled keys
    // and e^{lgE} into the Yo readout; otherwise G~ *= e^{lgE + cend} below
    const bool lazy = lgE + cend >= -kLazyRange;
    const float lg_new = lazy ? lgE + cend : 0.f;
    const float cum = cbase + cl;
    const float wt = gam + __shfl_down_sync(0xffffffffu, scl, 1);
    auto xpf = [](float v) { return SPLIT ? expf(v) : __expf(v); };
    const float om = (lane < TPW && tw < tv) ? xpf(cend - cum - lg_new) * wt : 0.f;
    if (lane < TPW) {
      tCum[tw] = cum;
      tEc[tw] = xpf(cum + lgE);
      tGam[tw] = gam;
      tW[tw] = wt;
      if (kFactMask) {
        tEa[tw] = xpf(cum);
        tEb[tw] = xpf(-cum) * wt;
      }
    }
    // the previous chunk's state update must finish before its tiles are
    // rewritten and before the next Yo reads G (here already when the angles
    // go into the transposed key tile)
    if (kThInKt && it > 0) {
      if (!tc::bar_wait(&bars[3], (it - 1) & 1, kWaitBudget)) abort_flag = 1;
      tc::fence_after();
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int aa = lane + 32 * j;
      if (aa < A) {
        float base = thb_cur[aa];
        for (int w = 0; w < warp; ++w) base += sTot[w * kAngMax + aa];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < TPW) {
            const float th = base + thl[j][i];
            if constexpr (kCosSin) {
              float sn, cs;
              sincos_fast(th, &sn, &cs);
              sTh[i * AS + aa] = cs;
              sTh[TPW * AS + i * AS + aa] = sn;
            } else {
              *thp(i * AS + aa) = th;
            }
          }
        if (warp == kWarps - 1) thb_next[aa] = base + thl[j][TPW - 1];
      }
    }
    __syncwarp();
    if (!kThInKt && it > 0) {
      if (!tc::bar_wait(&bars[3], (it - 1) & 1, kWaitBudget)) abort_flag = 1;
      tc::fence_after();
    }
    if constexpr (SPLIT && !SUMMARY) {
      // low part of the state for this chunk's Yo: G - trunc(G), rounded (the
      // MMA reads G itself truncated to TF32 as the high part); made visible
      // to the MMAs by the block barrier that precedes them
      if (MP == 64 && 32 * wg < Npad) {
        float v0[16], v1[16];
        const bool two = 32 * wg + 64 < Npad;
        tc::tmem_ld_m64_16(tG + lane_base + 32 * wg, v0);
        if (two) tc::tmem_ld_m64_16(tG + lane_base + 32 * wg + 64, v1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          v0[j] = tc::tf32_feed(v0[j] - tc::tf32_trunc(v0[j]));
          v1[j] = tc::tf32_feed(v1[j] - tc::tf32_trunc(v1[j]));
        }
        tc::tmem_st_m64_16(tGl + lane_base + 32 * wg, v0);
        if (two) tc::tmem_st_m64_16(tGl + lane_base + 32 * wg + 64, v1);
      }
      if (MP == 128) for (int c = 16 * wg; c < Npad; c += 64) {
        float v0[16], v1[16];
        const bool two = c + 32 < Npad;
        tc::tmem_ld16x2(tG + lane_base + c, tG + lane_base + (two ? c + 32 : c), v0, v1);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          v0[j] = tc::tf32_feed(v0[j] - tc::tf32_trunc(v0[j]));
          v1[j] = tc::tf32_feed(v1[j] - tc::tf32_trunc(v1[j]));
        }
        tc::tmem_st16_async(tGl + lane_base + c, v0);
        if (two) tc::tmem_st16_async(tGl + lane_base + c + 32, v1);
      }
      tc::tmem_wait_st();
    }
    // (4) rows 8 * warp .. 8 * warp + 7: rotated, biased q / k into the K-major
    // q / k tiles, w-scaled keys into the transposed key tile. Lane l takes
    // row 8 * warp + l % 8 and items 4 * jb + l / 8, so that each 16-byte
    // store of the warp lands in a distinct 16-byte slot.
    const bool last_chunk = io.k_last && c0 + tv == L;
    {
      const int ti = t - TPW * warp;  // token index within the warp
      const float omr = __shfl_sync(0xffffffffu, om, ti);
      const int krot = 2 * (lane >> 4) + ((lane >> 2) & 1);  // store order of the Kt rows
      const float* cb = sBiasC + r * BS;
      const float* bb = sBiasB + r * BS;
      float* kl = last_chunk && t == tv - 1 ? io.k_last + ((int64_t)bh * R + r) * N : nullptr;
      // Rotary item: dims n0..n0+3 and their partners n0+A..n0+A+3.
      // th: the four angles (or, with kCosSin, their cosines; sv their sines)
      auto pair_item = [&](int n0, float4 cu, float4 cw, float4 bu, float4 bw, float4 th,
                           float4 sv) {
        float4 q0 = make_float4(0.f, 0.f, 0.f, 0.f), q1 = q0, k0 = q0, k1 = q0;
        if (in) {
          const float4 cbu = *reinterpret_cast<const float4*>(cb + n0);
          const float4 cbw = *reinterpret_cast<const float4*>(cb + n0 + A);
          const float4 bbu = *reinterpret_cast<const float4*>(bb + n0);
          const float4 bbw = *reinterpret_cast<const float4*>(bb + n0 + A);
          float4 cs4, sn4;
          if constexpr (kCosSin) {
            cs4 = th;
            sn4 = sv;
          } else {
            sincos_fast(th.x, &sn4.x, &cs4.x);
            sincos_fast(th.y, &sn4.y, &cs4.y);
            sincos_fast(th.z, &sn4.z, &cs4.z);
            sincos_fast(th.w, &sn4.w, &cs4.w);
          }
          const float4 nsn4 = make_float4(-sn4.x, -sn4.y, -sn4.z, -sn4.w);
          // biased pair (u, w) = (C + c_bias, its partner); rotated:
          // (u cos - w sin, u sin + w cos), likewise for the key
          const float4 qu = add4(cu, cbu), qw = add4(cw, cbw);
          const float4 ku = add4(bu, bbu), kw = add4(bw, bbw);
          q0 = fma4(qu, cs4, mul4(qw, nsn4));
          q1 = fma4(qu, sn4, mul4(qw, cs4));
          k0 = fma4(ku, cs4, mul4(kw, nsn4));
          k1 = fma4(ku, sn4, mul4(kw, cs4));
        }
        if (!SUMMARY) {
          put4<SPLIT>(sQ + toff(rho, n0), LO, q0);
          put4<SPLIT>(sQ + toff(rho, n0 + A), LO, q1);
          put4<SPLIT>(sK + toff(rho, n0), LO, k0);
          put4<SPLIT>(sK + toff(rho, n0 + A), LO, k1);
        }
        store_kt4<SPLIT>(sKt, LO, n0, rho, k0, omr, krot);
        store_kt4<SPLIT>(sKt, LO, n0 + A, rho, k1, omr, krot);
        if (kl) {
          *reinterpret_cast<float4*>(kl + n0) = k0;
          *reinterpret_cast<float4*>(kl + n0 + A) = k1;
        }
      };
      // Plain item: dims n0..n0+3 >= 2A.
      auto single_item = [&](int n0, float4 cu, float4 bu) {
        float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), kv = qv;
        if (in) {
          const float4 cbu = *reinterpret_cast<const float4*>(cb + n0);
          const float4 bbu = *reinterpret_cast<const float4*>(bb + n0);
          qv = add4(cu, cbu);
          kv = add4(bu, bbu);
        }
        if (!SUMMARY) {
          put4<SPLIT>(sQ + toff(rho, n0), LO, qv);
          put4<SPLIT>(sK + toff(rho, n0), LO, kv);
        }
        store_kt4<SPLIT>(sKt, LO, n0, rho, kv, omr, krot);
        if (kl) *reinterpret_cast<float4*>(kl + n0) = kv;
      };
      if ((A & 3) == 0 && (N & 3) == 0) {
        // Vector path: an item is 4 consecutive dims n0..n0+3 of one row; for
        // n0 < A it also produces their rotary partners n0+A..n0+A+3.
        const int PQ = A >> 2, QW = PQ + ((N - 2 * A) >> 2), QW4 = (QW + 3) >> 2;
        // angles of this lane's rotary items, read before the q rows (which
        // share this warp's angle block) are written
        // Compile-time shapes with A a multiple of 16 and N of 4: item step jb
        // holds rotary pairs exactly when jb < A / 16 and real dims when
        // jb < QW / 4, whatever the lane, so the item kind is known per step.
        constexpr bool kStaticItems = KA > 0 && KA % 16 == 0 && KN > 0 && KN % 4 == 0;
        constexpr int kPairSteps = kStaticItems ? KA / 16 : 0;
        constexpr int kSteps = kStaticItems ? (KA / 4 + (KN - 2 * KA) / 4) / 4 : 0;
        auto is_pair = [&](int jb, int j) { return kStaticItems ? jb < kPairSteps : j < PQ; };
        auto is_item = [&](int jb, int j) { return kStaticItems ? jb < kSteps : j < QW; };
        float4 th4[4], sn4[kCosSin ? 4 : 1];
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          const int j = 4 * jb + jl;
          th4[jb] = is_pair(jb, j) ? *reinterpret_cast<const float4*>(thp(ti * AS + 4 * j))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (kCosSin)
            sn4[jb] = is_pair(jb, j) ? *reinterpret_cast<const float4*>(sTh + TPW * AS + ti * AS + 4 * j)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncwarp();
        if (kAsync) {
          // operands staged by TMA in the q / k tile positions
          bool ok = SUMMARY || tc::bar_wait(&bars[4], it & 1, kWaitBudget);
          ok = tc::bar_wait(&bars[5], it & 1, kWaitBudget) && ok;
          if (!ok) abort_flag = 1;
          if (pendC == it) pendC = -1;
          if (pendB == it) pendB = -1;
          // Packed projection: the B / C rows arrive raw and are scaled here by
          // their inverse RMS, which a pass over the packed rows has computed
          // exactly as the preprocess does (this row's token is the warp's
          // token ti, whose preloaded scalars sit in lane ti)
          float inv_c = 1.f, inv_b = 1.f;
          if constexpr (PACKED) {
            static_assert(KR == 1, "the packed projection is read by SISO instances only");
            inv_c = __shfl_sync(0xffffffffu, pl.inv_c, ti);
            inv_b = __shfl_sync(0xffffffffu, pl.inv_b, ti);
          }
          // (the raw row times its inverse RMS, as the preprocess writes it)
          // (never merged with the bias add that follows, so the normalised
          // value is rounded on its own, as the preprocess stores it)
          auto nrm = [&](float4 v, float inv) -> float4 {
            if constexpr (PACKED)
              return cat4(mul2_sep(lo2(v), make_float2(inv, inv)),
                          mul2_sep(hi2(v), make_float2(inv, inv)));
            else
              return v;
          };
#pragma unroll
          for (int jb = 0; jb < QW4; ++jb) {
            const int j = 4 * jb + jl;
            if (!is_item(jb, j)) continue;
            if (is_pair(jb, j)) {
              const int n0 = 4 * j;
              float4 th;
              float4 sv = make_float4(0.f, 0.f, 0.f, 0.f);
              switch (jb) {  // registers, not a local array
                case 0: th = th4[0]; if constexpr (kCosSin) sv = sn4[0]; break;
                case 1: th = th4[1]; if constexpr (kCosSin) sv = sn4[kCosSin ? 1 : 0]; break;
                case 2: th = th4[2]; if constexpr (kCosSin) sv = sn4[kCosSin ? 2 : 0]; break;
                default: th = th4[3]; if constexpr (kCosSin) sv = sn4[kCosSin ? 3 : 0]; break;
              }
              pair_item(n0, nrm(*reinterpret_cast<const float4*>(sQ + toff(rho, n0)), inv_c),
                        nrm(*reinterpret_cast<const float4*>(sQ + toff(rho, n0 + A)), inv_c),
                        nrm(*reinterpret_cast<const float4*>(sK + toff(rho, n0)), inv_b),
                        nrm(*reinterpret_cast<const float4*>(sK + toff(rho, n0 + A)), inv_b), th,
                        sv);
            } else {
              const int n0 = 2 * A + 4 * (j - PQ);
              single_item(n0, nrm(*reinterpret_cast<const float4*>(sQ + toff(rho, n0)), inv_c),
                          nrm(*reinterpret_cast<const float4*>(sK + toff(rho, n0)), inv_b));
            }
          }
        } else {
#pragma unroll 2
          for (int jb = 0; jb < QW4; ++jb) {
            const int j = 4 * jb + jl;
            if (j >= QW) continue;
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < PQ) {
              const int n0 = 4 * j;
              float4 th;
              switch (jb) {  // registers, not a local array
                case 0: th = th4[0]; break;
                case 1: th = th4[1]; break;
                case 2: th = th4[2]; break;
                default: th = th4[3]; break;
              }
              pair_item(n0, in ? *reinterpret_cast<const float4*>(crow + n0) : z4,
                        in ? *reinterpret_cast<const float4*>(crow + n0 + A) : z4,
                        in ? *reinterpret_cast<const float4*>(brow + n0) : z4,
                        in ? *reinterpret_cast<const float4*>(brow + n0 + A) : z4, th, z4);
            } else {
              const int n0 = 2 * A + 4 * (j - PQ);
              single_item(n0, in ? *reinterpret_cast<const float4*>(crow + n0) : z4,
                          in ? *reinterpret_cast<const float4*>(brow + n0) : z4);
            }
          }
        }
      } else {
        // Scalar path for A or N not a multiple of 4: unit u of a row is the
        // rotary pair (u, u + A) for u < A, else the single dim u + A.
        const int U = N - A;
        const int U4 = (U + 3) >> 2;
        float thr[16];
#pragma unroll
        for (int ub = 0; ub < 16; ++ub) {
          const int u = 4 * ub + jl;
          thr[ub] = u < A ? *thp(ti * AS + u) : 0.f;
        }
        __syncwarp();
        for (int ub = 0; ub < U4; ++ub) {
          const int u = 4 * ub + jl;
          if (u >= U) continue;
          if (u < A) {
            float q0 = 0.f, q1 = 0.f, k0 = 0.f, k1 = 0.f;
            if (in) {
              float th = 0.f;
#pragma unroll
              for (int x = 0; x < 16; ++x)
                if (x == ub) th = thr[x];
              float sn, cs;
              sincos_fast(th, &sn, &cs);
              const float qu = crow[u] + cb[u], qw = crow[u + A] + cb[u + A];
              const float ku = brow[u] + bb[u], kw = brow[u + A] + bb[u + A];
              q0 = qu * cs - qw * sn;
              q1 = qu * sn + qw * cs;
              k0 = ku * cs - kw * sn;
              k1 = ku * sn + kw * cs;
            }
            if (!SUMMARY) {
              put1<SPLIT>(sQ + tc::kmaj(rho, u, Npad), LO, q0);
              put1<SPLIT>(sQ + tc::kmaj(rho, u + A, Npad), LO, q1);
              put1<SPLIT>(sK + tc::kmaj(rho, u, Npad), LO, k0);
              put1<SPLIT>(sK + tc::kmaj(rho, u + A, Npad), LO, k1);
            }
            put1<SPLIT>(sKt + tc::kmaj(u, rho, kRows), LO, omr * k0);
            put1<SPLIT>(sKt + tc::kmaj(u + A, rho, kRows), LO, omr * k1);
            if (kl) {
              kl[u] = k0;
              kl[u + A] = k1;
            }
          } else {
            const int n = u + A;
            float qv = 0.f, kv = 0.f;
            if (in) {
              qv = crow[n] + cb[n];
              kv = brow[n] + bb[n];
            }
            if (!SUMMARY) {
              put1<SPLIT>(sQ + tc::kmaj(rho, n, Npad), LO, qv);
              put1<SPLIT>(sK + tc::kmaj(rho, n, Npad), LO, kv);
            }
            put1<SPLIT>(sKt + tc::kmaj(n, rho, kRows), LO, omr * kv);
            if (kl) kl[n] = kv;
          }
        }
      }
      // zero padding columns N .. Npad of this warp's q / k rows
      if (!SUMMARY && Npad > N) {
        const int pad = Npad > N ? Npad - N : 1;
        for (int i = lane; i < 8 * (Npad - N); i += 32) {
          const int rr = 8 * warp + i / pad, n = N + i % pad;
          sQ[tc::kmaj(rr, n, Npad)] = 0.f;
          sK[tc::kmaj(rr, n, Npad)] = 0.f;
          if (SPLIT) {
            sQ[tc::kmaj(rr, n, Npad) + LO] = 0.f;
            sK[tc::kmaj(rr, n, Npad) + LO] = 0.f;
          }
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();  // B2: tiles complete
    tc::fence_after();
    if (abort_flag) break;
    if (kEarlyB && SUMMARY && tid == kTmaThread && c0 + Qt < l1) {
      issue_rows(&tmB, sK, c0 + Qt, &bars[5]);
      pendB = it + 1;
    }
    // (5) S = Q K^T and Yo^T = G Q^T
    // (MMAs issued by one thread run one after another; the two independent
    // chains come from threads of different warps so that they overlap)
    // (split: three MMAs per K step, hi * hi + hi * lo + lo * hi; the state's
    // high part is the MMA's own truncation of G, its low part sits at tGl)
    // (an issuing thread's warp waits about a hundred cycles per MMA: in the
    // MIMO instances, whose values come from scalar loads, the issue comes
    // after the warp's value loads are in flight)
    auto issue_s_yo = [&] {
    if (!SUMMARY && tid == 0) {
#pragma unroll
      for (int ks = 0; ks < Npad / 8; ++ks) {
        tc::mma_ss(tS, dQ + qk_step(ks), dK + qk_step(ks), id_S, ks > 0);
        if (SPLIT) {
          tc::mma_ss(tS, dQ + qk_step(ks), dKl + qk_step(ks), id_S, 1);
          tc::mma_ss(tS, dQl + qk_step(ks), dK + qk_step(ks), id_S, 1);
        }
      }
      tc::commit(&bars[0]);
    }
    if (!SUMMARY && tid == 32) {
#pragma unroll
      for (int ks = 0; ks < Npad / 8; ++ks) {
        tc::mma_ts(tYo, tG + ks * 8, dQ + qk_step(ks), id_Y, ks > 0);
        if (SPLIT) {
          tc::mma_ts(tYo, tG + ks * 8, dQl + qk_step(ks), id_Y, 1);
          tc::mma_ts(tYo, tGl + ks * 8, dQ + qk_step(ks), id_Y, 1);
        }
      }
      tc::commit(&bars[1]);
    }
    };
    if constexpr (!kMxPre) issue_s_yo();
    // (6) masked scores P = M o S + D I (S rows: TMEM M = 64 layout, lanes
    // 0..15 of each quadrant; lane l + 16 takes the upper 8 columns of each
    // 16-column block of row l) and values X^T, both into the K region (or
    // their own regions) once S is done; then, in a chunk that is not lazy,
    // G~ *= e^{lgE + cum_end} once Yo has read G~. The value loads are issued
    // first so that their latency overlaps the wait.
    {
      constexpr int kXr = (kRows / 4 + kWarps - 1) / kWarps;  // row blocks per warp
      // SISO with P = 64 (compile time): x rows as float4 (warp w: tokens 8w ..
      // 8w + 7; lane l: token 8w + 4 (k / 2) + l / 8, dims 4 (8 (k % 2) + l % 8) ..)
      constexpr bool kXVec = !MIMO && KP == 64 && MP == 64;
      float4 xq[4];
      float xreg[kXVec ? 1 : kXr][kXVec ? 1 : MP / 8];
      if (kXVec) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = 8 * warp + 4 * (k >> 1) + (lane >> 3), pq = 8 * (k & 1) + (lane & 7);
          xq[k] = t < tv ? *reinterpret_cast<const float4*>(a.x + (tok0 + t) * XS + (int64_t)h * P + 4 * pq)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      } else {
        const int pl8 = lane & 7, rl = lane >> 3;
#pragma unroll
        for (int q = 0; q < kXr; ++q) {
          const int rb = warp + kWarps * q;
          const int rho2 = 4 * rb + rl;
          const int t2 = rho2 >> lgR, r2 = rho2 & (R - 1);
          const bool in = rb < kRows / 4 && t2 < tv;
          const float* xrow = a.x + (tok0 + t2) * XS + (int64_t)h * P;
          const float* mx = mimo ? a.mimo_x + ((int64_t)h * R + r2) * P : nullptr;
#pragma unroll
          for (int pb = 0; pb < MP / 8; ++pb) {
            const int p = 8 * pb + pl8;
            float xv = (in && p < P) ? xrow[p] : 0.f;
            if (!kMxPre && mimo && in && p < P) xv *= mx[p];
            xreg[q][pb] = xv;
          }
        }
      }
      if constexpr (kMxPre) issue_s_yo();
      if (!SUMMARY) {
        const bool s_done = tc::bar_wait(&bars[0], it & 1, kWaitBudget);
        if (!s_done) abort_flag = 1;
        tc::fence_after();
        // the k tile is dead once S has read it (split regions)
        if (kEarlyB && s_done && tid == kTmaThread && c0 + Qt < l1) {
          issue_rows(&tmB, sK, c0 + Qt, &bars[5]);
          pendB = it + 1;
        }
        const int rho = 16 * quad + (lane & 15);
        const int t = rho >> lgR;
        const float cum_t = tCum[t];
        const float gam_t = tGam[t];
        const float ea_t = kFactMask ? tEa[t] : 0.f;
        const int sh = lane >> 4;
        // lane l and l + 16 share row rho: columns cb * 16 + 8 * sh .. + 8
        float sv[2][8];
        tc::tmem_ld_m64_8x2(tS + lane_base + 32 * wg, tS + lane_base + 32 * wg + 16, sv[0], sv[1]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int cb = 2 * wg + u;
          float w8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) w8[j] = sv[u][j];
          const int col0 = cb * 16 + 8 * sh;
          // coefficients of the 8 key tokens of these columns (vector loads
          // when a row is a token)
          // (factored: ws = e^{-cum_s} w_s; otherwise cs = cum_s, ws = w_s)
          float cs[8], ws[8];
          const float* wsrc = fact ? tEb : tW;
          if (KR == 1) {
            const float4 w0 = *reinterpret_cast<const float4*>(wsrc + col0);
            const float4 w1 = *reinterpret_cast<const float4*>(wsrc + col0 + 4);
            ws[0] = w0.x; ws[1] = w0.y; ws[2] = w0.z; ws[3] = w0.w;
            ws[4] = w1.x; ws[5] = w1.y; ws[6] = w1.z; ws[7] = w1.w;
            if (!fact) {
              const float4 c0 = *reinterpret_cast<const float4*>(tCum + col0);
              const float4 c1 = *reinterpret_cast<const float4*>(tCum + col0 + 4);
              cs[0] = c0.x; cs[1] = c0.y; cs[2] = c0.z; cs[3] = c0.w;
              cs[4] = c1.x; cs[5] = c1.y; cs[6] = c1.z; cs[7] = c1.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              ws[j] = wsrc[(col0 + j) >> lgR];
              if (!fact) cs[j] = tCum[(col0 + j) >> lgR];
            }
          }
          if constexpr (KR == 1) {
            // a row is a token: columns before the diagonal position kd take
            // S e^{cum_t - cum_s} w_s, the diagonal gamma_t S + D (the D skip
            // rides on the diagonal: Yi then includes D * x), later ones zero
            const int kd = rho - col0;
            float pr[8];
            if (fact) {
              const float4 e4 = make_float4(ea_t, ea_t, ea_t, ea_t);
              const float4 m0 = mul4(make_float4(ws[0], ws[1], ws[2], ws[3]), e4);
              const float4 m1 = mul4(make_float4(ws[4], ws[5], ws[6], ws[7]), e4);
              const float4 p0 = mul4(make_float4(w8[0], w8[1], w8[2], w8[3]), m0);
              const float4 p1 = mul4(make_float4(w8[4], w8[5], w8[6], w8[7]), m1);
              pr[0] = p0.x; pr[1] = p0.y; pr[2] = p0.z; pr[3] = p0.w;
              pr[4] = p1.x; pr[5] = p1.y; pr[6] = p1.z; pr[7] = p1.w;
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) pr[j] = w8[j] * (__expf(cum_t - cs[j]) * ws[j]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              w8[j] = j < kd ? pr[j] : (j == kd ? fmaf(w8[j], gam_t, dsk) : 0.f);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int s = (col0 + j) >> lgR;
              float m = 0.f;
              if (s < t)
                m = fact ? ea_t * ws[j] : __expf(cum_t - cs[j]) * ws[j];
              else if (s == t)
                m = gam_t;
              // the D skip rides on the diagonal: Yi then includes D * x
              w8[j] = col0 + j == rho ? fmaf(w8[j], m, dsk) : w8[j] * m;
            }
          }
          put4<SPLIT>(sP + tc::kmaj(rho, col0, kRows), LO, make_float4(w8[0], w8[1], w8[2], w8[3]));
          put4<SPLIT>(sP + tc::kmaj(rho, col0 + 4, kRows), LO,
                      make_float4(w8[4], w8[5], w8[6], w8[7]));
        }
      }
      // values X^T [p][row] (x * mimo_x for MIMO): lane l takes p = 8 * pb +
      // l % 8 and row 4 * rb + l / 8 (conflict-free scalar stores); the float4
      // rows go out in a lane-rotated component order (conflict-free as well)
      if (kXVec) {
        const int rot = (lane >> 1) & 3;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = 8 * warp + 4 * (k >> 1) + (lane >> 3), pq = 8 * (k & 1) + (lane & 7);
          store_kt4<SPLIT>(sXt, LO, 4 * pq, t, xq[k], 1.0f, rot);
        }
      } else {
        const int pl8 = lane & 7, rl = lane >> 3;
#pragma unroll
        for (int q = 0; q < kXr; ++q) {
          const int rb = warp + kWarps * q;
          if (rb >= kRows / 4) break;
          const int rho2 = 4 * rb + rl;
#pragma unroll
          for (int pb = 0; pb < MP / 8; ++pb)
            put1<SPLIT>(sXt + tc::kmaj(8 * pb + pl8, rho2, kRows), LO,
                        kMxPre ? xreg[q][pb] * mxr[pb] : xreg[q][pb]);
        }
      }
      // value of the sequence's last token for the step state (last chunk only)
      if (io.v_last && c0 + tv == L) {
        const float* xrow = a.x + (tok0 + tv - 1) * XS + (int64_t)h * P;
        for (int i = tid; i < R * P; i += kThreads) {
          const int r = i / P, p = i - r * P;
          io.v_last[((int64_t)bh * R + r) * P + p] =
              mimo ? xrow[p] * a.mimo_x[((int64_t)h * R + r) * P + p] : xrow[p];
        }
      }
      // G~ may be rescaled only once Yo^T = G~ Q^T has read it
      if (!SUMMARY && !lazy) {
        if (!tc::bar_wait(&bars[1], it & 1, kWaitBudget)) abort_flag = 1;
        tc::fence_after();
        // the q tile is free: stage the next chunk's C rows
        if (kAsync && c0 + Qt < l1 && tid == kTmaThread) {
          issue_rows(&tmC, sQ, c0 + Qt, &bars[4]);
          pendC = it + 1;
        }
      }
      const float ec = expf(lgE + cend);
      // M = 64 state (P <= 64): the half-split loads give each thread 16 useful
      // columns of its row; warp group wg takes the 32-column blocks 32 wg and
      // 32 wg + 64. M = 128: two 16-column blocks per pass. One wait per pair
      // of loads, stores unwaited until the end.
      if (!lazy && MP == 64 && 32 * wg < Npad) {
        float v0[16], v1[16];
        const bool two = 32 * wg + 64 < Npad;
        tc::tmem_ld_m64_16(tG + lane_base + 32 * wg, v0);
        if (two) tc::tmem_ld_m64_16(tG + lane_base + 32 * wg + 64, v1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          v0[j] = SPLIT ? v0[j] * ec : tc::tf32_clean(v0[j] * ec);
          v1[j] = SPLIT ? v1[j] * ec : tc::tf32_clean(v1[j] * ec);
        }
        tc::tmem_st_m64_16(tG + lane_base + 32 * wg, v0);
        if (two) tc::tmem_st_m64_16(tG + lane_base + 32 * wg + 64, v1);
      }
      if (!lazy && MP == 128) for (int c = 16 * wg; c < Npad; c += 64) {
        float v0[16], v1[16];
        const bool two = c + 32 < Npad;
        tc::tmem_ld16x2(tG + lane_base + c, tG + lane_base + (two ? c + 32 : c), v0, v1);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          // single pass: the state is the A operand of Yo, so it is kept
          // rounded to TF32; split: full FP32 (its low part is derived below)
          v0[j] = SPLIT ? v0[j] * ec : tc::tf32_clean(v0[j] * ec);
          v1[j] = SPLIT ? v1[j] * ec : tc::tf32_clean(v1[j] * ec);
        }
        tc::tmem_st16_async(tG + lane_base + c, v0);
        if (two) tc::tmem_st16_async(tG + lane_base + c + 32, v1);
      }
      tc::tmem_wait_st();
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();  // B3: scores, values and the rescaled state complete
    tc::fence_after();
    if (abort_flag) break;
    // (7) Yi^T = X^T P^T and G~ += X^T (w e^{-lgE} K)
    // (Yi and the state update come from threads of different warps)
    if (!SUMMARY && tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kRows / 8; ++ks) {
        tc::mma_ss(tS, dXt + 16ull * ks, dP + 16ull * ks, id_Y, ks > 0);
        if (SPLIT) {
          tc::mma_ss(tS, dXt + 16ull * ks, dPl + 16ull * ks, id_Y, 1);
          tc::mma_ss(tS, dXtl + 16ull * ks, dP + 16ull * ks, id_Y, 1);
        }
      }
      tc::commit(&bars[2]);
    }
    if (tid == 32) {
      // a lazy chunk adds to G~ without the rescale pass: the Yo MMAs
      // (issued by this thread) must have read G~ first
      bool ok = true;
      if (!SUMMARY && lazy) {
        ok = tc::bar_wait(&bars[1], it & 1, kWaitBudget);
        tc::fence_after();
      }
      if (ok) {
#pragma unroll
        for (int ks = 0; ks < kRows / 8; ++ks) {
          tc::mma_ss(tG, dXt + 16ull * ks, dKt + 16ull * ks, id_D, 1);
          if (SPLIT) {
            tc::mma_ss(tG, dXt + 16ull * ks, dKtl + 16ull * ks, id_D, 1);
            tc::mma_ss(tG, dXtl + 16ull * ks, dKt + 16ull * ks, id_D, 1);
          }
        }
        tc::commit(&bars[3]);
      } else {
        abort_flag = 1;
      }
    }
    lgE = lg_new;
    // next chunk's per-token scalars and angles: loads in flight during the
    // MMAs and the epilogue
    if (c0 + Qt < l1)
      preload_tokens<PACKED>(pl, a, g, tok0 + Qt, c0 + Qt, L, TPW, A, H, h, warp, lane);
    if (!SUMMARY) {
      // SISO epilogue gate operand z of this thread's output column, loaded while
      // the MMAs run (its x comes from the value tile, rounded to TF32 like
      // every operand of this kernel)
      constexpr int kCols = (MP == 64) ? 8 : 16;
      // Staged SISO output (P a compile-time multiple of 4, P <= 64): the
      // pre-gate outputs go through the free score area of shared memory as
      // [t][P] rows, and the gate and the stores run on float4 rows.
      constexpr bool kStaged = !MIMO && KP > 0 && KP % 4 == 0 && KP <= 64;
      constexpr int kQuads = kStaged ? kRows * KP / 4 / kThreads : 1;  // float4 units per thread
      constexpr int kRowQ = kStaged ? KP / 4 : 1;                       // float4 units per row
      float4 zq[kQuads > 0 ? kQuads : 1];
      float ze[2][kCols];
      if (kStaged) {
#pragma unroll
        for (int k = 0; k < kQuads; ++k) {
          const int unit = tid + kThreads * k;
          const int t = unit / kRowQ, p0 = 4 * (unit % kRowQ);
          zq[k] = (t < tv && g.has_z)
                      ? *reinterpret_cast<const float4*>(a.z + (tok0 + t) * XS + (int64_t)h * P + p0)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      } else if (!mimo) {
        const float* zcol = a.z + tok0 * XS + (int64_t)h * P + prow;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col0 = (2 * wg + u) * 16 + 8 * half;
#pragma unroll
          for (int j = 0; j < kCols; ++j) {
            const int t = col0 + j;
            const bool ok = pvalid && t < tv;
            ze[u][j] = (ok && g.has_z) ? zcol[t * XS] : 0.f;
          }
        }
      }
      // MIMO instances with compile-time R: the z values of this lane's tokens
      // (kTpb per 16-column block), loaded before the waits as well
      constexpr int kTpb = (MIMO && KR > 0) ? kCols / KR : 0;
      float zm[2][kTpb > 0 ? kTpb : 1];
      if (kTpb > 0) {
        const float* zcol = a.z + tok0 * XS + (int64_t)h * P + prow;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int col0 = (2 * wg + u) * 16 + 8 * half;
#pragma unroll
          for (int tt = 0; tt < (kTpb > 0 ? kTpb : 1); ++tt) {
            const int t = (col0 >> lgR) + tt;
            zm[u][tt] = (pvalid && t < tv && g.has_z) ? zcol[t * XS] : 0.f;
          }
        }
      }
      // a lazy chunk waits for Yo only here; the q tile is then free for the
      // next chunk's C rows
      if (lazy) {
        if (!tc::bar_wait(&bars[1], it & 1, kWaitBudget)) abort_flag = 1;
        tc::fence_after();
        if (kAsync && c0 + Qt < l1 && tid == kTmaThread) {
          issue_rows(&tmC, sQ, c0 + Qt, &bars[4]);
          pendC = it + 1;
        }
      }
      // the epilogue needs Yo and Yi; the state update runs on under it
      if (!tc::bar_wait(&bars[2], it & 1, kWaitBudget)) abort_flag = 1;
      tc::fence_after();
      if (kBAtEpi) {
        // the staging area (the transposed key tile) is free once the state
        // update is done; the K region is then free for the next B rows
        const bool st_done = tc::bar_wait(&bars[3], it & 1, kWaitBudget);
        if (!st_done) abort_flag = 1;
        tc::fence_after();
        if (st_done && c0 + Qt < l1 && tid == kTmaThread) {
          issue_rows(&tmB, sK, c0 + Qt, &bars[5]);
          pendB = it + 1;
        }
      }
      // (8) epilogue: output column p of this chunk's tokens. With MP = 64 the
      // two lanes of a row split each 16-column block into 8 + 8 columns.
      {
        const float* zcol = a.z + tok0 * XS + (int64_t)h * P + prow;
        float* ocol = a.out + tok0 * HP + (int64_t)h * P + prow;
#pragma unroll
        for (int cb = 2 * wg; cb < 2 * wg + 2; ++cb) {
          float yo[16], yi[16];
          if constexpr (MP == 64)  // lane l + 16: the upper 8 columns of row l's block
            tc::tmem_ld_m64_8x2(tYo + lane_base + cb * 16, tS + lane_base + cb * 16, yo, yi);
          else
            tc::tmem_ld16x2(tYo + lane_base + cb * 16, tS + lane_base + cb * 16, yo, yi);
          if (!pvalid) continue;
          const int col0 = cb * 16 + 8 * half;
          if (!mimo) {
            const int u = cb - 2 * wg;
            float ec[kCols];
#pragma unroll
            for (int q = 0; q < kCols / 4; ++q) {
              const float4 e4 = *reinterpret_cast<const float4*>(tEc + col0 + 4 * q);
              ec[4 * q] = e4.x;
              ec[4 * q + 1] = e4.y;
              ec[4 * q + 2] = e4.z;
              ec[4 * q + 3] = e4.w;
            }
            float yv[kCols];
#pragma unroll
            for (int j = 0; j < kCols; j += 2) {
              const float2 r = __ffma2_rn(make_float2(ec[j], ec[j + 1]), make_float2(yo[j], yo[j + 1]),
                                          make_float2(yi[j], yi[j + 1]));
              yv[j] = r.x;
              yv[j + 1] = r.y;
            }
#pragma unroll
            for (int j = 0; j < kCols; ++j) {
              const int t = col0 + j;
              if (kStaged) {
                sStage[t * KP + prow + kStageSkew * (t >> 3)] = yv[j];
              } else if (t < tv) {
                const float zv = u ? ze[1][j] : ze[0][j];
                float y = yv[j];
                if (g.has_z) y *= silu_fast(zv);
                ocol[t * HP] = y;
              }
            }
          } else {
            const int tpb = kCols >> lgR;  // whole tokens in this lane's columns
#pragma unroll
            for (int tt = 0; tt < tpb; ++tt) {
              const int t = (col0 >> lgR) + tt;
              if (t >= tv) break;
              float zv;
              if constexpr (kTpb > 0)
                zv = zm[cb - 2 * wg][tt];
              else
                zv = g.has_z ? zcol[t * XS] : 0.f;
              const float ec = tEc[t];
              float o = 0.f;
#pragma unroll
              for (int r = 0; r < kRmax; ++r) {
                if (r < R) {
                  const int j = (tt << lgR) + r;
                  float y = fmaf(ec, yo[j], yi[j]);
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
      if (kStaged) {
        __syncthreads();  // the staged rows are complete
#pragma unroll
        for (int k = 0; k < kQuads; ++k) {
          const int unit = tid + kThreads * k;
          const int t = unit / kRowQ, p0 = 4 * (unit % kRowQ);
          if (t < tv) {
            float4 y = *reinterpret_cast<const float4*>(sStage + t * KP + kStageSkew * (t >> 3) + p0);
            if (g.has_z) y = gate4(y, zq[k]);
            *reinterpret_cast<float4*>(a.out + (tok0 + t) * HP + (int64_t)h * P + p0) = y;
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
    // once the state update has read the K region and every thread is done with
    // its scores, values and staged outputs: stage the next chunk's B rows
    // (the generic-proxy writes of the region are ordered before the TMA's)
    if (kAsync && !kEarlyB && !kBAtEpi && c0 + Qt < l1) {
      if (!SUMMARY) {
        tc::fence_async_smem();
        __syncthreads();
      }
      if (tid == kTmaThread) {
        if (tc::bar_wait(&bars[3], it & 1, kWaitBudget)) {
          tc::fence_after();
          issue_rows(&tmB, sK, c0 + Qt, &bars[5]);
          pendB = it + 1;
        } else {
          abort_flag = 1;
        }
      }
    }
  }
  // the last state update
  if (!abort_flag && it > 0) {
    if (!tc::bar_wait(&bars[3], (it - 1) & 1, kWaitBudget)) abort_flag = 1;
    tc::fence_after();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (abort_flag && tid == 0) atomicExch(status, kStatusTimeout);
  // after a timeout: wait (bounded) for TMA copies still in flight, since
  // shared memory must outlive them; if that wait gives up too, the copies may
  // still land after the kernel exits, which the status records
  if (kAsync && tid == kTmaThread) {
    bool drained = true;
    if (pendC >= 0) drained = tc::bar_wait(&bars[4], pendC & 1, kWaitBudget) && drained;
    if (pendB >= 0) drained = tc::bar_wait(&bars[5], pendB & 1, kWaitBudget) && drained;
    if (!drained) atomicExch(status, kStatusUndrained);
  }
  if (!abort_flag) {
    // final state (G = e^{lgE} G~), cumulative angle and decay of this segment
    const float* thb = sThBase + (it & 1) * kAngMax;
    const float gsc = expf(lgE);
    // this thread's state row (G = e^{lgE} G~) into dst, 16 columns per load
    // (as four float4s when N % 16 == 0, the row bases then 16-byte aligned)
    auto store_state = [&](float* dst) {
      for (int c = 16 * wg; c < Npad; c += 32) {
        float v[16];
        tc::tmem_ld16(tG + lane_base + c, v);
        if (!g_lane) continue;
        if (N % 16 == 0) {
          if (c < N) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              reinterpret_cast<float4*>(dst + c)[q] =
                  make_float4(v[4 * q] * gsc, v[4 * q + 1] * gsc, v[4 * q + 2] * gsc,
                              v[4 * q + 3] * gsc);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < N) dst[c + j] = v[j] * gsc;
        }
      }
    };
    if (io.g1) store_state(io.g1 + ((int64_t)cta * P + prow) * N);
    if (io.g_last && l1 == L) store_state(io.g_last + ((int64_t)bh * P + prow) * N);
    if (io.th1)
      for (int i = tid; i < A; i += kThreads) io.th1[(int64_t)cta * A + i] = thb[i];
    if (io.th_last && l1 == L)
      for (int i = tid; i < A; i += kThreads) io.th_last[(int64_t)bh * A + i] = thb[i];
    if (io.e1 && tid == 0) io.e1[cta] = expf(esum);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_free(tbase, kTmemCols);
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Tensor map of the C or B rows [B, L, G * R, N] for the chunk kernel's TMA
// staging: dimensions (n, group row, token, batch), box [32 dims][R ranks][Qt
// tokens][1], 128-byte swizzle, zero fill outside the tensor. tok_stride is
// the distance in floats between consecutive tokens' rows: G * R * N in the
// C / B tensors, the packed width W when they are column slices of the packed
// projection.
cudaError_t rows_tensor_map(CUtensorMap* m, const float* base, const ScanGeom& g,
                            uint64_t tok_stride) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const uint64_t RG = (uint64_t)g.G * g.R, N = (uint64_t)g.N;
  const cuuint64_t dims[4] = {N, RG, (cuuint64_t)g.L, (cuuint64_t)g.B};
  const cuuint64_t strides[3] = {N * 4, tok_stride * 4, (uint64_t)g.L * tok_stride * 4};
  const cuuint32_t box[4] = {32, (cuuint32_t)g.R, (cuuint32_t)(kRows / g.R), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Dynamic shared memory of an instance: the layout, 1 KB of alignment slack
// for the swizzled tiles, and for split instances at least 120 KB, so that two
// CTAs never share an SM (their 512 TMEM columns take the whole SM).
size_t chunk_smem_bytes(const ChunkLayout& lay, bool async, bool split) {
  size_t b = lay.bytes + (async ? 1024 : 0);
  if (split && b < (size_t)120 * 1024) b = (size_t)120 * 1024;
  return b;
}

template <int MP, bool MIMO, int KN, int KA, int KR, int KP, bool SPLIT, bool PACKED = false>
cudaError_t run_chunk(const ScanGeom& g, const ScanArgs& a, uint32_t* status, const ChunkIO& io,
                      bool summary, unsigned grid, cudaStream_t s) {
  constexpr bool async = chunk_async(KN, KA);
  const ChunkLayout lay = chunk_layout(g.N, g.P, g.A, g.R, MIMO, async, SPLIT);
  const size_t bytes = chunk_smem_bytes(lay, async, SPLIT);
  CUtensorMap tmC, tmB;
  memset(&tmC, 0, sizeof(tmC));
  memset(&tmB, 0, sizeof(tmB));
  cudaError_t e;
  if (PACKED) {
    // B rows at columns [2I, 2I + GRN), C rows at [2I + GRN, 2I + 2GRN) of the
    // packed rows, which start at a.z (z is the first slice)
    const float* rows_b = a.z + 2 * (int64_t)g.H * g.P;
    const float* rows_c = rows_b + (int64_t)g.G * g.R * g.N;
    if ((e = rows_tensor_map(&tmC, rows_c, g, (uint64_t)g.W)) != cudaSuccess) return e;
    if ((e = rows_tensor_map(&tmB, rows_b, g, (uint64_t)g.W)) != cudaSuccess) return e;
  } else if (async) {
    const uint64_t rgn = (uint64_t)g.G * g.R * g.N;
    if ((e = rows_tensor_map(&tmC, a.c, g, rgn)) != cudaSuccess) return e;
    if ((e = rows_tensor_map(&tmB, a.b, g, rgn)) != cudaSuccess) return e;
  }
  auto kernel = summary ? k_scan_chunk<MP, MIMO, true, KN, KA, KR, KP, SPLIT, PACKED>
                        : k_scan_chunk<MP, MIMO, false, KN, KA, KR, KP, SPLIT, PACKED>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (PACKED && io.pdl) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, g, a, lay, io, status, tmC, tmB);
  }
  kernel<<<grid, kThreads, bytes, s>>>(g, a, lay, io, status, tmC, tmB);
  return cudaSuccess;
}

// Launches the instance for g's shape: compile-time shapes SISO P64 N128 with
// A = 32 or 64 and MIMO R4 P64 N64 A32, else the generic instance for P <= 64
// or P <= 128.
template <bool SPLIT>
cudaError_t dispatch_chunk(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                           const ChunkIO& io, bool summary, cudaStream_t s) {
  const unsigned grid = (unsigned)(g.B * g.H * io.nseg);
  const bool mimo = a.mimo_o != nullptr;
  cudaError_t e;
  if (!mimo && g.R == 1 && g.P == 64 && g.N == 128 && g.A == 32)
    e = run_chunk<64, false, 128, 32, 1, 64, SPLIT>(g, a, status, io, summary, grid, s);
  else if (!mimo && g.R == 1 && g.P == 64 && g.N == 128 && g.A == 64)
    e = run_chunk<64, false, 128, 64, 1, 64, SPLIT>(g, a, status, io, summary, grid, s);
  else if (mimo && g.R == 4 && g.P == 64 && g.N == 64 && g.A == 32)
    e = run_chunk<64, true, 64, 32, 4, 64, SPLIT>(g, a, status, io, summary, grid, s);
  else if (g.P <= 64)
    e = mimo ? run_chunk<64, true, 0, 0, 0, 0, SPLIT>(g, a, status, io, summary, grid, s)
             : run_chunk<64, false, 0, 0, 0, 0, SPLIT>(g, a, status, io, summary, grid, s);
  else
    e = mimo ? run_chunk<128, true, 0, 0, 0, 0, SPLIT>(g, a, status, io, summary, grid, s)
             : run_chunk<128, false, 0, 0, 0, 0, SPLIT>(g, a, status, io, summary, grid, s);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

// The SISO scan reading the packed projection directly (compile-time TMA
// shapes P64 N128 with A = 32 or 64 only; the host routes every other shape
// through the preprocess kernel and a workspace instead).
bool packed_instance(const ScanGeom& g) {
  return !g.mimo && g.R == 1 && g.P == 64 && g.N == 128 && (g.A == 32 || g.A == 64);
}
template <bool SPLIT>
cudaError_t dispatch_chunk_packed(const ScanGeom& g, const ScanArgs& a, uint32_t* status,
                                  const ChunkIO& io, bool summary, cudaStream_t s) {
  const unsigned grid = (unsigned)(g.B * g.H * io.nseg);
  cudaError_t e;
  if (!packed_instance(g)) return cudaErrorInvalidValue;
  if (g.A == 32)
    e = run_chunk<64, false, 128, 32, 1, 64, SPLIT, true>(g, a, status, io, summary, grid, s);
  else
    e = run_chunk<64, false, 128, 64, 1, 64, SPLIT, true>(g, a, status, io, summary, grid, s);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace
}  // namespace m3
