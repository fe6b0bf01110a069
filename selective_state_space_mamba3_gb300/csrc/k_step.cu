// Single-token Mamba-3 step with explicit recurrent state (oarust mamba3.rs,
// `mamba3_siso_step` / `mamba3_mimo_step`: ssm [B,H,P,N], cumulative angle
// [B,H,A], previous key [B,H,R,N], previous value [B,H,R,P]).
//
// One 256-thread block per (b, h). The [P, N] state is the only large operand
// (96% of the bytes at decode shapes), so the kernel is an HBM stream over it.
// When N is a multiple of 4 the block moves the whole state with two bulk
// copies (cp.async.bulk): the load is issued first and lands in shared memory
// while the block stages the rotated q / k rows and the previous key / value;
// the state is then updated in place by the exponential-trapezoidal rule
//   h = decay * h + scale * decay * sum_r v_prev[r][p] k_prev[r][n]
//                 + gamma * sum_r v[r][p] k[r][n]
// (warp w owns rows w, w + 8, ..., lane l the float4 at n = 4l; the readout
// h . q_r is reduced with shuffles) and goes back with one bulk store that
// overlaps the output stage. Other N take a register path with the same
// arithmetic. The k / v / angle states are written after the block has read
// their previous values.
#include "m3_internal.cuh"
#include "tc_ptx.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr long long kWaitBudget = 2000000000LL;  // clock cycles (about a second)

template <int RMAX>
struct StepSmem {
  float q[RMAX * 128], k[RMAX * 128], kp[RMAX * 128];  // [R][N]
  float v[RMAX * 128], vp[RMAX * 128];                 // [R][P]
  float y[RMAX * 128];                                 // [R][P] readouts
  float zz[128];
  float theta[64];
  float red[kWarps];
};

template <int RMAX>
__host__ __device__ constexpr size_t step_smem_head() {
  return (sizeof(StepSmem<RMAX>) + 127) / 128 * 128;
}

// Stages the per-(b, h) operands: the new cumulative angle, the rotated biased
// q / k per rank, the previous key / value, the rank-scaled value and z. The
// units (one rotary pair or lone column of q / k per rank, one value element
// per rank, one z element) are spread over the block so that each thread's
// loads are independent and issue together; all state writes (angle, key,
// value) follow a single block barrier, after every previous value is read.
template <int RMAX>
__device__ __forceinline__ void stage_step(StepSmem<RMAX>& sm, const ScanGeom& g,
                                           const ScanArgs& a, const StepState& st, int b, int h,
                                           int64_t sc, float dtv) {
  const int tid = threadIdx.x;
  const int grp = h / (g.H / g.G);
  const int P = g.P, N = g.N, A = g.A, R = g.R;
  const int UQ = R * N, UV = R * P, U = UQ + UV + P;
  for (int u = tid; u < U; u += kThreads) {
    if (u < UQ) {
      const int r = u / N, n = u - r * N;
      const int64_t row = ((int64_t)b * g.G * R + (int64_t)grp * R + r) * N;
      const float* cb = a.c_bias + ((int64_t)h * R + r) * N;
      const float* bb = a.b_bias + ((int64_t)h * R + r) * N;
      sm.kp[u] = st.k[sc * R * N + u];
      if (n < A) {
        const float th = st.angle[sc * A + n] + dtv * a.angle[(int64_t)b * A + n];
        const float qu = a.c[row + n] + cb[n], qv = a.c[row + n + A] + cb[n + A];
        const float ku = a.b[row + n] + bb[n], kv = a.b[row + n + A] + bb[n + A];
        if (r == 0) sm.theta[n] = th;
        float sn, cs;
        sincos_fast(th, &sn, &cs);
        sm.q[r * N + n] = qu * cs - qv * sn;
        sm.q[r * N + n + A] = qu * sn + qv * cs;
        sm.k[r * N + n] = ku * cs - kv * sn;
        sm.k[r * N + n + A] = ku * sn + kv * cs;
      } else if (n >= 2 * A) {
        sm.q[u] = a.c[row + n] + cb[n];
        sm.k[u] = a.b[row + n] + bb[n];
      }
    } else if (u < UQ + UV) {
      const int i = u - UQ;
      const int r = i / P, p = i - r * P;
      const float xv = a.x[sc * P + p];
      sm.vp[i] = st.v[sc * R * P + i];
      sm.v[i] = a.mimo_x ? xv * a.mimo_x[((int64_t)h * R + r) * P + p] : xv;
    } else {
      const int p = u - UQ - UV;
      sm.zz[p] = a.z[sc * P + p];
    }
  }
  __syncthreads();
  for (int i = tid; i < A; i += kThreads) st.angle[sc * A + i] = sm.theta[i];
  for (int i = tid; i < R * N; i += kThreads) st.k[sc * R * N + i] = sm.k[i];
  for (int i = tid; i < R * P; i += kThreads) st.v[sc * R * P + i] = sm.v[i];
}

// Readout of row p: y_r[p] = sum_n h[p][n] q_r[n] (+ D v_r[p]); acc holds the
// lane's partial sums.
template <int RMAX>
__device__ __forceinline__ void finish_row(StepSmem<RMAX>& sm, int R, int P, int p, float dskip,
                                           const float* acc) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r < R) {
      const float yv = warp_sum(acc[r]);
      if (lane == 0) sm.y[r * P + p] = yv + dskip * sm.v[r * P + p];
    }
  }
}

// Gate (SISO), or per-rank gate + mimo_o contraction + output RMS norm (MIMO).
template <int RMAX>
__device__ __forceinline__ void step_output(StepSmem<RMAX>& sm, const ScanGeom& g,
                                            const ScanArgs& a, int h, int64_t sc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = g.P, R = g.R;
  float* outp = a.out + sc * P;
  if (!a.mimo_o) {
    for (int p = tid; p < P; p += kThreads) {
      const float yv = sm.y[p];
      outp[p] = g.has_z ? yv * silu_f(sm.zz[p]) : yv;
    }
    return;
  }
  // (row p, rank r) of thread 4 p + r when R <= 4 and P <= 64: the gated rank
  // values of a row in four neighbouring lanes, summed in rank order by the
  // rank-0 lane; otherwise thread p loops over the ranks
  const bool quad = RMAX == 4 && P <= kThreads / 4;
  const int p = quad ? tid >> 2 : tid;
  const int r0 = quad ? tid & 3 : 0;
  float ov = 0.f;
  if (quad) {
    float term = 0.f;
    if (p < P && r0 < R) {
      float yv = sm.y[r0 * P + p];
      if (g.has_z) yv *= silu_f(sm.zz[p] * a.mimo_z[((int64_t)h * R + r0) * P + p]);
      term = a.mimo_o[((int64_t)h * R + r0) * P + p] * yv;
    }
    // ov = ((t0 + t1) + t2) + t3 in the rank-0 lane, as the loop below adds
    const float t1 = __shfl_down_sync(0xffffffffu, term, 1);
    const float t2 = __shfl_down_sync(0xffffffffu, term, 2);
    const float t3 = __shfl_down_sync(0xffffffffu, term, 3);
    ov = term;
    if (R > 1) ov += t1;
    if (R > 2) ov += t2;
    if (R > 3) ov += t3;
    if (r0 != 0) ov = 0.f;
  } else if (p < P) {
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
  if (p < P && r0 == 0) outp[p] = ov;
}

// Bulk-copy path (N % 4 == 0): the state travels HBM -> shared -> HBM as two
// cp.async.bulk transfers of P * N * 4 bytes (a multiple of 16; the state base
// is 16-byte aligned by the host checks).
template <int RMAX>
__global__ void __launch_bounds__(kThreads, RMAX == 1 ? 5 : (RMAX == 4 ? 5 : 4)) k_step_bulk(ScanGeom g, ScanArgs a, StepState st) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StepSmem<RMAX>& sm = *reinterpret_cast<StepSmem<RMAX>*>(smem_raw);
  float* hsm = reinterpret_cast<float*>(smem_raw + step_smem_head<RMAX>());
  __shared__ __align__(8) uint64_t bar;
  __shared__ int arrived;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / g.H, h = bh % g.H;
  const int P = g.P, N = g.N, R = g.R;
  const int64_t sc = (int64_t)b * g.H + h;  // [B,1,H] index
  float* hs = st.ssm + sc * (int64_t)P * N;
  const uint32_t bytes = (uint32_t)(P * N) * 4u;
  if (tid == 0) {
    tc::bar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(&bar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_u32(hsm)),
        "l"(hs), "r"(bytes), "r"(tc::smem_u32(&bar))
        : "memory");
    arrived = 1;
  }
  const float dtv = a.dt[sc];
  stage_step<RMAX>(sm, g, a, st, b, h, sc, dtv);
  const float lam = sigmoid_f(a.trap[sc]);
  const float decay = expf(a.adt[sc]);
  const float gam = lam * dtv;
  const float sdec = (1.0f - lam) * dtv * decay;
  const float dskip = g.has_d ? a.d[h] : 0.0f;
  if (!tc::bar_wait(&bar, 0, kWaitBudget)) arrived = 0;
  __syncthreads();
  if (!arrived) {
    // The copy did not complete in time: the ssm state row stays as it was and
    // the output row is NaN. Wait (bounded) once more so that no copy into
    // shared memory outlives the block.
    tc::bar_wait(&bar, 0, kWaitBudget);
    for (int p = tid; p < P; p += kThreads) a.out[sc * P + p] = __int_as_float(0x7fc00000);
    return;
  }
  const int N4 = N >> 2;
  // Row p of the state: h = decay * h + sum_r (sdec v_prev[r][p] k_prev[r] +
  // gamma v[r][p] k[r]) over the lane's float4 of columns, then the readouts
  // h . q_r as lane partial sums.
  auto row_update = [&](int p, int l, float* acc) {
    float4* hp = reinterpret_cast<float4*>(hsm + p * N) + l;
    float4 hv = *hp;
    float4 upd = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const float cp = sdec * sm.vp[r * P + p], cc = gam * sm.v[r * P + p];
        const float4 kp4 = reinterpret_cast<const float4*>(sm.kp + r * N)[l];
        const float4 k4 = reinterpret_cast<const float4*>(sm.k + r * N)[l];
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
    *hp = hv;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const float4 q4 = reinterpret_cast<const float4*>(sm.q + r * N)[l];
        acc[r] = hv.x * q4.x + hv.y * q4.y + hv.z * q4.z + hv.w * q4.w;
      }
    }
  };
  // rows pa and pb together (each with row_update's arithmetic), the key and
  // query float4s loaded once for both
  auto row_update2 = [&](int pa, int pb, int l, float* acc_a, float* acc_b) {
    float4* hpa = reinterpret_cast<float4*>(hsm + pa * N) + l;
    float4* hpb = reinterpret_cast<float4*>(hsm + pb * N) + l;
    float4 ha = *hpa, hb = *hpb;
    float4 ua = make_float4(0.f, 0.f, 0.f, 0.f), ub = ua;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const float cpa = sdec * sm.vp[r * P + pa], cca = gam * sm.v[r * P + pa];
        const float cpb = sdec * sm.vp[r * P + pb], ccb = gam * sm.v[r * P + pb];
        const float4 kp4 = reinterpret_cast<const float4*>(sm.kp + r * N)[l];
        const float4 k4 = reinterpret_cast<const float4*>(sm.k + r * N)[l];
        ua.x += cpa * kp4.x + cca * k4.x;
        ua.y += cpa * kp4.y + cca * k4.y;
        ua.z += cpa * kp4.z + cca * k4.z;
        ua.w += cpa * kp4.w + cca * k4.w;
        ub.x += cpb * kp4.x + ccb * k4.x;
        ub.y += cpb * kp4.y + ccb * k4.y;
        ub.z += cpb * kp4.z + ccb * k4.z;
        ub.w += cpb * kp4.w + ccb * k4.w;
      }
    }
    ha.x = decay * ha.x + ua.x;
    ha.y = decay * ha.y + ua.y;
    ha.z = decay * ha.z + ua.z;
    ha.w = decay * ha.w + ua.w;
    hb.x = decay * hb.x + ub.x;
    hb.y = decay * hb.y + ub.y;
    hb.z = decay * hb.z + ub.z;
    hb.w = decay * hb.w + ub.w;
    *hpa = ha;
    *hpb = hb;
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const float4 q4 = reinterpret_cast<const float4*>(sm.q + r * N)[l];
        acc_a[r] = ha.x * q4.x + ha.y * q4.y + ha.z * q4.z + ha.w * q4.w;
        acc_b[r] = hb.x * q4.x + hb.y * q4.y + hb.z * q4.z + hb.w * q4.w;
      }
    }
  };
  if (N4 <= 16) {
    // rows of at most 16 float4: each half warp takes two rows per step (rows
    // p and p + 16 of the step's 32; p + 8 in the other half), so that the
    // key and query loads serve both
    const int hw = lane >> 4, hl = lane & 15;
    for (int p0 = warp; p0 < P; p0 += 4 * kWarps) {
      const int pa = p0 + hw * kWarps, pb = pa + 2 * kWarps;
      float acc[2][RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) acc[0][r] = acc[1][r] = 0.f;
      if (hl < N4) {
        if (pb < P)
          row_update2(pa, pb, hl, acc[0], acc[1]);
        else if (pa < P)
          row_update(pa, hl, acc[0]);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int p = i ? pb : pa;
        if constexpr (RMAX == 4) {
          // the four rank sums over the half warp by recursive halving: lanes
          // with bit 3 keep ranks 2, 3 and send 0, 1 (and the other way
          // round), then bit 2 picks one rank; each rank's sum is the tree
          // of the 8-4-2-1 butterfly
          const bool b3 = (hl >> 3) & 1, b2 = (hl >> 2) & 1;
          float k0 = b3 ? acc[i][2] : acc[i][0], k1 = b3 ? acc[i][3] : acc[i][1];
          const float s0 = b3 ? acc[i][0] : acc[i][2], s1 = b3 ? acc[i][1] : acc[i][3];
          k0 += __shfl_xor_sync(0xffffffffu, s0, 8);
          k1 += __shfl_xor_sync(0xffffffffu, s1, 8);
          float v = b2 ? k1 : k0;
          v += __shfl_xor_sync(0xffffffffu, b2 ? k0 : k1, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          const int r = hl >> 2;
          if ((hl & 3) == 0 && r < R && p < P) sm.y[r * P + p] = v + dskip * sm.v[r * P + p];
        } else {
#pragma unroll
          for (int r = 0; r < RMAX; ++r) {
            if (r < R) {
              float v = acc[i][r];
#pragma unroll
              for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
              if (hl == 0 && p < P) sm.y[r * P + p] = v + dskip * sm.v[r * P + p];
            }
          }
        }
      }
    }
  } else {
    // a warp per row, two rows (p and p + 8) per step sharing the key and
    // query loads
    for (int p = warp; p < P; p += 2 * kWarps) {
      const int pb = p + kWarps;
      float acc[2][RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) acc[0][r] = acc[1][r] = 0.f;
      if (lane < N4) {
        if (pb < P)
          row_update2(p, pb, lane, acc[0], acc[1]);
        else
          row_update(p, lane, acc[0]);
      }
      finish_row<RMAX>(sm, R, P, p, dskip, acc[0]);
      if (pb < P) finish_row<RMAX>(sm, R, P, pb, dskip, acc[1]);
    }
  }
  // generic-proxy writes of the updated rows -> visible to the bulk store
  tc::fence_async_smem();
  __syncthreads();
  if (tid == 0) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(hs),
                 "r"(tc::smem_u32(hsm)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
  step_output<RMAX>(sm, g, a, h, sc);
  // shared memory must stay valid until the store has read it
  if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Register path for N not a multiple of 4.
template <int RMAX>
__global__ void __launch_bounds__(kThreads) k_step(ScanGeom g, ScanArgs a, StepState st) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StepSmem<RMAX>& sm = *reinterpret_cast<StepSmem<RMAX>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / g.H, h = bh % g.H;
  const int P = g.P, N = g.N, R = g.R;
  const int64_t sc = (int64_t)b * g.H + h;
  float* hs = st.ssm + sc * (int64_t)P * N;
  const float dtv = a.dt[sc];
  stage_step<RMAX>(sm, g, a, st, b, h, sc, dtv);
  const float lam = sigmoid_f(a.trap[sc]);
  const float decay = expf(a.adt[sc]);
  const float gam = lam * dtv;
  const float sdec = (1.0f - lam) * dtv * decay;
  const float dskip = g.has_d ? a.d[h] : 0.0f;
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
    finish_row<RMAX>(sm, R, P, p, dskip, acc);
  }
  __syncthreads();
  step_output<RMAX>(sm, g, a, h, sc);
}

template <int RMAX>
cudaError_t launch_step_r(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                          cudaStream_t s) {
  const unsigned grid = (unsigned)(g.B * g.H);
  cudaError_t e;
  if (g.N % 4 == 0) {
    const size_t smem = step_smem_head<RMAX>() + (size_t)g.P * g.N * 4;
    e = cudaFuncSetAttribute(k_step_bulk<RMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    k_step_bulk<RMAX><<<grid, kThreads, smem, s>>>(g, a, st);
  } else {
    const size_t smem = sizeof(StepSmem<RMAX>);
    e = cudaFuncSetAttribute(k_step<RMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    k_step<RMAX><<<grid, kThreads, smem, s>>>(g, a, st);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_step(const ScanGeom& g, const ScanArgs& a, const StepState& st,
                        cudaStream_t s) {
  if (g.R == 1) return launch_step_r<1>(g, a, st, s);
  if (g.R <= 4) return launch_step_r<4>(g, a, st, s);
  return launch_step_r<8>(g, a, st, s);
}

}  // namespace m3
