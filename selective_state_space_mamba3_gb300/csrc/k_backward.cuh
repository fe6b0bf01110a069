// Device helpers shared by the SISO and MIMO adjoint kernels (k_backward.cu,
// k_backward_mimo.cu): half-warp row sums, cross-half column sums, shared
// memory row / column loads, and the transpose of the split-half rotation.
#pragma once

#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kBT = 256;  // threads per block of the sweeps
constexpr int kWarps = kBT / 32;

// Sums v[i] (i < R, R a power of two <= 16) over the 16 lanes of a half warp.
// Each halving round keeps one half of the values per lane and adds the
// partner's other half; afterwards the lane holds the total of value `row`
// (chosen by its high lane bits) and every lane sharing those bits holds the same.
template <int R>
__device__ __forceinline__ float rows_sum16(float (&v)[R], int cq, int& row) {
  row = 0;
  int o = 8;
#pragma unroll
  for (int c = R; c > 1; c >>= 1) {
    const bool up = (cq & o) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = up ? v[i] : v[i + c / 2];
      const float keep = up ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    if (up) row += c / 2;
    o >>= 1;
  }
  float s = v[0];
#pragma unroll
  for (int r = 16 / R / 2; r > 0; r >>= 1) s += __shfl_xor_sync(0xffffffffu, s, r);
  return s;
}

// Adds the two half warps' column values v[4 NB] (columns 64 j + 4 cq + e)
// and stores this warp's column sums at dst[n]: half warp rq keeps half of
// the values and adds its partner's.
template <int NB>
__device__ __forceinline__ void cols_sum_store(const float (&v)[4 * NB], int rq, int cq,
                                               float* dst) {
  constexpr int kHalf = 2 * NB;
  float r[kHalf];
#pragma unroll
  for (int i = 0; i < kHalf; ++i) {
    const float send = rq ? v[i] : v[i + kHalf];
    const float keep = rq ? v[i + kHalf] : v[i];
    r[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
  if constexpr (NB == 2) {
    *reinterpret_cast<float4*>(dst + 64 * rq + 4 * cq) = make_float4(r[0], r[1], r[2], r[3]);
  } else {
    *reinterpret_cast<float2*>(dst + 4 * cq + 2 * rq) = make_float2(r[0], r[1]);
  }
}

// Loads RPT consecutive floats (16-byte aligned for RPT % 4 == 0, 8-byte for
// RPT = 2).
template <int RPT>
__device__ __forceinline__ void load_rows(const float* src, float (&d)[RPT]) {
  if constexpr (RPT == 1) {
    d[0] = src[0];
  } else if constexpr (RPT % 4 == 0) {
#pragma unroll
    for (int i = 0; i < RPT; i += 4) {
      const float4 t = *reinterpret_cast<const float4*>(src + i);
      d[i] = t.x; d[i + 1] = t.y; d[i + 2] = t.z; d[i + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < RPT; i += 2) {
      const float2 t = *reinterpret_cast<const float2*>(src + i);
      d[i] = t.x; d[i + 1] = t.y;
    }
  }
}

template <int NB>
__device__ __forceinline__ void load_cols(const float* row, int cq, float (&d)[4 * NB]) {
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const float4 t = *reinterpret_cast<const float4*>(row + 64 * j + 4 * cq);
    d[4 * j] = t.x; d[4 * j + 1] = t.y; d[4 * j + 2] = t.z; d[4 * j + 3] = t.w;
  }
}

// Gradient d(row) of the unrotated, biased row from the gradient gr of its
// rotated form (the transpose of the rotation), element n.
__device__ __forceinline__ float unrotate(const float* gr, const float* cs, const float* sn,
                                          int n, int A) {
  if (n < A) return gr[n] * cs[n] + gr[n + A] * sn[n];
  if (n < 2 * A) return -gr[n - A] * sn[n - A] + gr[n] * cs[n - A];
  return gr[n];
}

// L2 prefetch of the 128-byte lines of [p, p + bytes).
__device__ __forceinline__ void prefetch_range(const float* p, int bytes) {
  const uintptr_t first = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(127);
  const uintptr_t last = reinterpret_cast<uintptr_t>(p) + bytes;
  for (uintptr_t q = first; q < last; q += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
}

// L2 prefetch of the operands a sweep stages for tokens [t0, t0 + tv) of
// (b, h): the x, dout and z rows, the group's C and B rows (rank rows
// grp R .. grp R + R - 1), the scalars, the angle row and, when given, the
// saved running angles of the sequence. Thread i takes item i of 8 per token.
// (dout may be null: not prefetched; yd, when given, is the MIMO readout /
// adjoint array [B H][L][R P], prefetched in place of z.)
template <int BT = kBT>
__device__ __forceinline__ void prefetch_tile(const ScanGeom& g, const ScanArgs& a,
                                              const float* dout, const float* theta, int bh,
                                              int b, int h, int grp, int t0, int tv,
                                              const float* yd = nullptr) {
  const int P = g.P, N = g.N, H = g.H, L = g.L, A = g.A, R = g.R;
  for (int i = threadIdx.x; i < tv * 8; i += BT) {
    const int tt = i >> 3, k = i & 7;
    const int64_t tok = (int64_t)b * L + t0 + tt, s = tok * H + h;
    switch (k) {
      case 0: prefetch_range(a.x + s * P, P * 4); break;
      case 1: if (dout) prefetch_range(dout + s * P, P * 4); break;
      case 2:
        if (yd) prefetch_range(yd + ((int64_t)bh * L + t0 + tt) * R * P, R * P * 4);
        else if (g.has_z) prefetch_range(a.z + s * P, P * 4);
        break;
      case 3: prefetch_range(a.c + (tok * g.G * R + (int64_t)grp * R) * N, R * N * 4); break;
      case 4: prefetch_range(a.b + (tok * g.G * R + (int64_t)grp * R) * N, R * N * 4); break;
      case 5:
        prefetch_range(a.adt + s, 4);
        prefetch_range(a.dt + s, 4);
        prefetch_range(a.trap + s, 4);
        break;
      case 6: if (A > 0) prefetch_range(a.angle + tok * A, A * 4); break;
      default: if (theta && A > 0) prefetch_range(theta + ((int64_t)bh * L + t0 + tt) * A, A * 4); break;
    }
  }
}

}  // namespace
}  // namespace m3
