// C ABI of libm3: host-side validation and kernel dispatch.
//
// The geometry rules mirror oarust 0.8.6 `src/rs/ml/matrix/mamba3.rs`:
// `Geometry::resolve` (SISO), `MimoGeometry::resolve` (MIMO),
// `PreprocessGeometry::resolve` (preprocess), the step functions' L == 1 and
// state-shape checks, and `shader_u32` (every element count below 2^32).
// Every check runs before anything is enqueued, so a rejected call changes no
// buffer (the step docstring: states are mutated only after validation).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <initializer_list>

#include "m3_internal.cuh"

namespace m3 {

static std::atomic<uint64_t> g_launches{0};
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {

constexpr uint64_t kU32 = 1ull << 32;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Product of non-negative extents, false on overflow or when >= 2^32.
bool count_below_u32(std::initializer_list<int64_t> dims) {
  uint64_t c = 1;
  for (int64_t d : dims) {
    if (d < 0) return false;
    if (d != 0 && c > (kU32 - 1) / (uint64_t)d) return false;
    c *= (uint64_t)d;
  }
  return c < kU32;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? M3_OK : M3_ERR_CUDA; }

// Shared SISO/MIMO geometry check. Fills g; returns M3_OK or an error code.
int resolve_ssm(const m3_ssm_config* cfg, bool mimo, ScanGeom* g) {
  if (!cfg) return M3_ERR_INVALID_ARGUMENT;
  const int64_t B = cfg->batch_size, L = cfg->sequence_length, H = cfg->num_heads;
  const int64_t G = cfg->num_groups == 0 ? H : cfg->num_groups;
  const int64_t P = cfg->head_dim, N = cfg->state_size, A = cfg->num_rope_angles;
  const int64_t R = cfg->mimo_rank;
  if (B <= 0 || L <= 0 || H <= 0 || G <= 0 || cfg->num_groups < 0 || H % G != 0) return M3_ERR_INVALID_ARGUMENT;
  if (P <= 0 || P > 128 || N <= 0 || N > 128 || A < 0 || A > 64 || 2 * A > N) return M3_ERR_INVALID_ARGUMENT;
  if (mimo) {
    if (R < 1 || R > 8 || P * N > 4096) return M3_ERR_INVALID_ARGUMENT;
  } else {
    if (R != 1 || cfg->has_output_norm) return M3_ERR_INVALID_ARGUMENT;
  }
  if (cfg->math_mode != M3_MATH_FP32 && cfg->math_mode != M3_MATH_TF32) return M3_ERR_INVALID_ARGUMENT;
  // every operand element count below 2^32 (`shader_u32`)
  if (!count_below_u32({B, L, R * G, N}) || !count_below_u32({B, L, H, P}) ||
      !count_below_u32({B, L, H}) || !count_below_u32({B, L, A}) ||
      !count_below_u32({H, R, N}) || !count_below_u32({H, R, P}) || !count_below_u32({B, H}))
    return M3_ERR_INVALID_ARGUMENT;
  g->B = (int)B; g->L = (int)L; g->H = (int)H; g->G = (int)G; g->P = (int)P; g->N = (int)N;
  g->A = (int)A; g->R = (int)R;
  g->has_z = cfg->has_z != 0; g->has_d = cfg->has_d != 0;
  g->has_norm = mimo && cfg->has_output_norm != 0;
  g->math_mode = cfg->math_mode;
  g->mimo = mimo ? 1 : 0;
  return M3_OK;
}

int check_ptrs(std::initializer_list<const void*> required) {
  for (const void* p : required)
    if (!p) return M3_ERR_INVALID_ARGUMENT;
  for (const void* p : required)
    if (!aligned16(p)) return M3_ERR_UNALIGNED;
  return M3_OK;
}

int check_angle_ptr(const void* p, int A) {
  if (A == 0) return (p && !aligned16(p)) ? M3_ERR_UNALIGNED : M3_OK;
  if (!p) return M3_ERR_INVALID_ARGUMENT;
  return aligned16(p) ? M3_OK : M3_ERR_UNALIGNED;
}

}  // namespace

// Scan dispatch. The tcgen05 chunked kernel takes R in {1,2,4,8}, P, N <= 128:
//  - TF32 mode: single-pass TF32 operands, except the MIMO output norm, which
//    takes the split-operand (3xTF32) flavour. The norm rescales every token to
//    unit size, so a token's own relative error becomes the normwise error, and
//    single-pass TF32 rounding reaches a few 1e-3 on some tokens.
//  - FP32-exact mode: the split-operand flavour where its doubled tiles fit in
//    shared memory.
// Every other shape, and FP32-exact shapes the split tiles do not fit, run the
// token-sequential FP32 kernel on the CUDA cores.
static bool chunk_split_mode(const ScanGeom& g) {
  return g.math_mode == M3_MATH_FP32 || g.has_norm;
}
static bool use_chunk(const ScanGeom& g) {
  if (!chunk_supported(g)) return false;
  if (chunk_split_mode(g)) return chunk_split_supported(g);
  return g.math_mode == M3_MATH_TF32;
}

// SMs of the current device (152 on GB300; also the answer when no device can
// be queried, so that workspace sizes stay defined without a GPU).
static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // reset the last-error state the failed query left
    return 152;
  }
  return n;
}

// Sequences per launch below the CTAs the SMs hold at once (two per SM for
// single-pass TF32, one for the split flavour) are split into segments of
// whole chunks, at least four chunks long: a summary pass, a prefix over
// segments and the main pass then replace one long serial chain.
static int choose_nseg(const ScanGeom& g) {
  const int64_t bh = (int64_t)g.B * g.H;
  const int64_t target = (chunk_split_mode(g) ? 1 : 2) * (int64_t)sm_count();
  if (bh >= target) return 1;
  const int64_t qt = chunk_rows_per_token(g);
  const int64_t max_seg = g.L / (4 * qt);
  int64_t n = target / bh;
  if (n > max_seg) n = max_seg;
  if (n > 4096) n = 4096;
  return n < 1 ? 1 : (int)n;
}

// Relative time of a pass of C CTAs that each walk c chunks, for SMs holding
// `slots` CTAs at once: each SM takes ceil(C / SMs) CTAs in turns of `slots`;
// a chunk of a CTA that shares its SM takes kShared times as long as one that
// runs alone (the chunk chain is latency-bound, so two CTAs on an SM run each
// at about 0.7 of the lone speed).
static double pass_cost(int64_t C, int64_t c, int slots, int sms) {
  constexpr double kShared = 1.4;
  const int64_t k = (C + sms - 1) / sms;
  const int64_t turns = k / slots, rem = k % slots;
  const double t_full = slots == 1 ? 1.0 : kShared;
  return (double)c * ((double)turns * t_full + (rem == 0 ? 0.0 : rem == 1 ? 1.0 : kShared));
}

namespace {
// Workspace layout of the chunked path (byte offsets, 256-byte aligned).
// Split sequences: nseg segments of seg_len tokens; the summary pass runs
// over `pieces` equal pieces of each segment (pieces * nseg CTAs per
// sequence, the last segment's pieces skipped), so that its short chains
// fill the SMs that the main pass's nseg CTAs per sequence leave idle; the
// prefix folds the pieces of a segment into the next segment's entry state.
struct ChunkWs {
  size_t status, gsum, thsum, esum, gentry, thentry, g0, th0, bytes;
  int nseg, seg_len, pieces;
};

ChunkWs chunk_ws(const ScanGeom& g, bool with_state) {
  ChunkWs w;
  const size_t bh = (size_t)g.B * g.H, pn = (size_t)g.P * g.N, A = (size_t)g.A;
  w.nseg = choose_nseg(g);
  const int qt = chunk_rows_per_token(g);
  const int per = (g.L + w.nseg - 1) / w.nseg;
  w.seg_len = (per + qt - 1) / qt * qt;
  w.pieces = 1;
  if (w.nseg > 1) {
    // pieces per segment: the least modelled time of summary + main pass over
    // 1..4 pieces of at least two chunks (a segment then holds a whole number
    // of pieces, so it may grow by up to pieces - 1 chunks)
    const int sms = sm_count(), slots = chunk_split_mode(g) ? 1 : 2;
    const int64_t seg_chunks = w.seg_len / qt, L_chunks = ((int64_t)g.L + qt - 1) / qt;
    double best = 0.0;
    for (int m = 1; m <= 4; ++m) {
      const int64_t pc = (seg_chunks + m - 1) / m;
      if (m > 1 && pc < 2) break;
      const int64_t sc = pc * m, ns = (L_chunks + sc - 1) / sc;
      if (ns < 2) continue;
      const double t = pass_cost((int64_t)bh * (ns - 1) * m, pc, slots, sms) +
                       pass_cost((int64_t)bh * ns, sc, slots, sms);
      if (m == 1 || t < best) {
        best = t;
        w.pieces = m;
        w.seg_len = (int)(sc * qt);
        w.nseg = (int)ns;
      }
    }
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  w.status = take(256);
  const size_t ns = w.nseg > 1 ? bh * (size_t)w.nseg : 0, np = ns * (size_t)w.pieces;
  w.gsum = take(np * pn * 4);
  w.thsum = take(np * A * 4);
  w.esum = take(np * 4);
  w.gentry = take(ns * pn * 4);
  w.thentry = take(ns * A * 4);
  w.g0 = take(with_state ? bh * pn * 4 : 0);
  w.th0 = take(with_state ? bh * A * 4 : 0);
  w.bytes = off;
  return w;
}
}  // namespace

size_t scan_workspace_bytes(const ScanGeom& g, bool with_state) {
  return use_chunk(g) ? chunk_ws(g, with_state).bytes : 0;
}

namespace {
using ChunkLauncher = cudaError_t (*)(const ScanGeom&, const ScanArgs&, uint32_t*,
                                      const ChunkIO&, bool, bool, cudaStream_t);

// The chunked scan: status word cleared, the step state converted into the
// kernel's entry state (prefill), then one main pass, or for split sequences a
// summary pass, the prefix over segments and the main pass.
// after_kernel: the caller has cleared the status word and launched, just
// before, a kernel whose outputs the scan reads (the packed scan's row norms):
// the first scan launch then follows it as a programmatic dependent launch.
cudaError_t run_chunked(const ScanGeom& g, const ScanArgs& a, const StepState* st, void* ws,
                        cudaStream_t s, ChunkLauncher launch_scan_chunk,
                        bool after_kernel = false) {
  const bool split = chunk_split_mode(g);
  const ChunkWs w = chunk_ws(g, st != nullptr);
  char* base = static_cast<char*>(ws);
  auto f = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
  uint32_t* status = reinterpret_cast<uint32_t*>(base + w.status);
  cudaError_t e = after_kernel ? cudaSuccess : cudaMemsetAsync(status, 0, 16, s);
  if (e != cudaSuccess) return e;
  if (st) {
    e = launch_state_init(g, a, *st, f(w.g0), f(w.th0), s);
    if (e != cudaSuccess) return e;
  }
  ChunkIO io{};
  io.seg_len = w.seg_len;
  io.nseg = w.nseg;
  io.pdl = after_kernel && w.nseg == 1;
  if (st) {
    io.g_last = st->ssm;
    io.th_last = st->angle;
    io.k_last = st->k;
    io.v_last = st->v;
  }
  if (w.nseg == 1) {
    if (st) {
      io.g0 = f(w.g0);
      io.th0 = f(w.th0);
    }
    return launch_scan_chunk(g, a, status, io, false, split, s);
  }
  ChunkIO sum{};
  sum.seg_len = w.seg_len / w.pieces;
  sum.nseg = w.nseg * w.pieces;
  sum.sum_skip = w.pieces;
  sum.pdl = after_kernel;
  sum.g1 = f(w.gsum);
  sum.th1 = f(w.thsum);
  sum.e1 = f(w.esum);
  e = launch_scan_chunk(g, a, status, sum, true, split, s);
  if (e != cudaSuccess) return e;
  e = launch_state_prefix(g, w.nseg, w.pieces, st ? f(w.g0) : nullptr, st ? f(w.th0) : nullptr, f(w.gsum),
                          f(w.thsum), f(w.esum), f(w.gentry), f(w.thentry), s);
  if (e != cudaSuccess) return e;
  io.g0 = f(w.gentry);
  io.th0 = f(w.thentry);
  return launch_scan_chunk(g, a, status, io, false, split, s);
}
}  // namespace

cudaError_t launch_scan(const ScanGeom& g, const ScanArgs& a, const StepState* st, void* ws,
                        size_t, cudaStream_t s) {
  if (!use_chunk(g)) return launch_scan_seq(g, a, st ? *st : StepState{}, s);
  return run_chunked(g, a, st, ws, s, launch_scan_chunk);
}

// ---------------------------------------------------------------------------
// Scans of a packed projection. SISO: fused where the chunked kernel has a TMA
// instance for the shape and the packed rows are 16-byte aligned column by
// column, otherwise m3_preprocess into the workspace followed by the scan.
// MIMO: always the preprocess and then the scan (measured faster than reading
// the packed rows in the latency-bound MIMO kernel).
namespace {
// Workspace: the scan's own workspace first (its status word at offset 0, where
// m3_workspace_status reads it), then, fused, the row pass's outputs (B / C
// inverse RMS, dt, adt) at off[0..2], or, otherwise, the preprocess outputs at
// off[0..7].
struct PackedPlan {
  bool fused;
  size_t scan_bytes;
  size_t off[8];  // fallback: x, z, bh, ch, dt, adt, trap, angle
  size_t bytes;
};

PackedPlan packed_plan(const ScanGeom& g, const PreGeom& p) {
  PackedPlan pl{};
  pl.fused = !g.mimo && use_chunk(g) && chunk_packed_supported(g) && p.W % 4 == 0;
  // (at least the 256 bytes of the status word, which the token-sequential
  // scan does not use but which is cleared for m3_workspace_status)
  pl.scan_bytes = std::max<size_t>(256, (scan_workspace_bytes(g, false) + 255) / 256 * 256);
  if (pl.fused) {
    // the row pass's outputs: B / C inverse RMS, then dt and adt
    pl.off[0] = pl.scan_bytes;
    pl.off[1] = pl.off[0] + ((size_t)p.rows * 2 * p.G * p.R * 4 + 255) / 256 * 256;
    pl.off[2] = pl.off[1] + ((size_t)p.rows * p.H * 4 + 255) / 256 * 256;
    pl.bytes = pl.off[2] + ((size_t)p.rows * p.H * 4 + 255) / 256 * 256;
    return pl;
  }
  const size_t rows = (size_t)p.rows;
  const size_t bc = (size_t)p.G * p.R * p.N;  // B / C rows per packed row
  const size_t cols[8] = {(size_t)p.I, (size_t)p.I, bc, bc, (size_t)p.H, (size_t)p.H,
                          (size_t)p.H, (size_t)p.A};
  size_t o = pl.scan_bytes;
  for (int i = 0; i < 8; ++i) {
    pl.off[i] = o;
    o += (rows * cols[i] * 4 + 255) / 256 * 256;
  }
  pl.bytes = o;
  return pl;
}

// Geometry of the packed scan: the SsmConfig rules (SISO or MIMO), and a
// preprocess config that describes the same layer (inner = H * P, the same N,
// H, A, groups and rank).
int resolve_packed(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg, bool mimo,
                   ScanGeom* g, PreGeom* p) {
  int st = resolve_ssm(cfg, mimo, g);
  if (st != M3_OK) return st;
  if (!pcfg) return M3_ERR_INVALID_ARGUMENT;
  st = resolve_pre(pcfg, (int64_t)g->B * g->L, p);
  if (st != M3_OK) return st;
  if (p->I != g->H * g->P || p->N != g->N || p->H != g->H || p->A != g->A || p->G != g->G ||
      p->R != g->R)
    return M3_ERR_INVALID_ARGUMENT;
  g->W = p->W;
  g->eps = p->eps;
  g->dt_min = p->dt_min;
  g->dt_max = p->dt_max;
  g->a_floor = p->a_floor;
  return M3_OK;
}
}  // namespace

}  // namespace m3

using namespace m3;

extern "C" {

const char* m3_status_string(int status) {
  switch (status) {
    case M3_OK: return "ok";
    case M3_ERR_INVALID_ARGUMENT: return "invalid argument: geometry, limit, null pointer or overflow";
    case M3_ERR_UNALIGNED: return "a base pointer is not 16-byte aligned";
    case M3_ERR_WORKSPACE: return "workspace missing or smaller than required";
    case M3_ERR_CUDA: return "a CUDA launch or runtime call failed";
    case M3_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case M3_ERR_DEVICE_STATE:
      return "a bounded device-side wait gave up and in-flight copies did not drain: context unusable";
    default: return "unknown status";
  }
}

uint64_t m3_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int m3_preprocess(const m3_preprocess_config* cfg, int64_t rows, const float* projected,
                  const float* dt_bias, float* x, float* z, float* bh, float* ch, float* dt,
                  float* adt, float* trap, float* angle, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_preprocess");
  PreGeom g;
  int st = resolve_pre(cfg, rows, &g);
  if (st != M3_OK) return st;
  st = check_ptrs({projected, dt_bias, x, z, bh, ch, dt, adt, trap});
  if (st != M3_OK) return st;
  if ((st = check_angle_ptr(angle, g.A)) != M3_OK) return st;
  PreOut o{x, z, bh, ch, dt, adt, trap, angle};
  return cuda_status(launch_preprocess(g, projected, dt_bias, o, (cudaStream_t)stream));
}

int m3_preprocess_backward_workspace(const m3_preprocess_config* cfg, int64_t rows,
                                     size_t* bytes) {
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  PreGeom g;
  const int st = resolve_pre(cfg, rows, &g);
  if (st != M3_OK) return st;
  *bytes = preprocess_backward_workspace_bytes(g);
  return M3_OK;
}

int m3_preprocess_backward(const m3_preprocess_config* cfg, int64_t rows, const float* projected,
                           const float* dt_bias, const float* grad_x, const float* grad_z,
                           const float* grad_bh, const float* grad_ch, const float* grad_dt,
                           const float* grad_adt, const float* grad_trap,
                           const float* grad_angle, float* grad_projected, float* grad_dt_bias,
                           void* workspace, size_t workspace_bytes, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_preprocess_backward");
  PreGeom g;
  int st = resolve_pre(cfg, rows, &g);
  if (st != M3_OK) return st;
  st = check_ptrs({projected, dt_bias, grad_x, grad_z, grad_bh, grad_ch, grad_dt, grad_adt,
                   grad_trap, grad_projected, grad_dt_bias});
  if (st != M3_OK) return st;
  if ((st = check_angle_ptr(grad_angle, g.A)) != M3_OK) return st;
  const size_t need = preprocess_backward_workspace_bytes(g);
  if (!workspace || workspace_bytes < need) return M3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return M3_ERR_UNALIGNED;
  PreGrads gr{grad_x, grad_z, grad_bh, grad_ch, grad_dt, grad_adt, grad_trap, grad_angle};
  return cuda_status(launch_preprocess_backward(g, projected, dt_bias, gr, grad_projected,
                                                grad_dt_bias, (float*)workspace,
                                                (cudaStream_t)stream));
}

}  // extern "C"

namespace m3 {
// `PreprocessGeometry::resolve` rules; fills g.
int resolve_pre(const m3_preprocess_config* cfg, int64_t rows, PreGeom* out) {
  if (!cfg) return M3_ERR_INVALID_ARGUMENT;
  const int64_t I = cfg->inner_size, N = cfg->state_size, H = cfg->num_heads;
  const int64_t A = cfg->num_rope_angles, G = cfg->num_groups, R = cfg->mimo_rank;
  if (rows <= 0 || I <= 0 || N <= 0 || H <= 0 || G <= 0 || R <= 0 || A < 0 || A > N / 2)
    return M3_ERR_INVALID_ARGUMENT;
  const float eps = cfg->epsilon, lo = cfg->dt_min, hi = cfg->dt_max, fl = cfg->a_floor;
  if (!std::isfinite(eps) || eps <= 0.f || !std::isfinite(lo) || !std::isfinite(hi) ||
      lo <= 0.f || lo > hi || !std::isfinite(fl) || fl <= 0.f)
    return M3_ERR_INVALID_ARGUMENT;
  if (!count_below_u32({G, R, N}) || !count_below_u32({I, 2}) || !count_below_u32({H, 3}))
    return M3_ERR_INVALID_ARGUMENT;
  const int64_t bc = G * R * N;
  const int64_t W = 2 * I + 2 * bc + 3 * H + A;
  if (!count_below_u32({W}) || !count_below_u32({rows, W}) || !count_below_u32({rows, I}) ||
      !count_below_u32({rows, bc}) || !count_below_u32({rows, H}) || !count_below_u32({rows, A}))
    return M3_ERR_INVALID_ARGUMENT;
  PreGeom& g = *out;
  g.rows = rows; g.I = (int)I; g.N = (int)N; g.H = (int)H; g.A = (int)A; g.G = (int)G;
  g.R = (int)R; g.W = (int)W;
  g.eps = eps; g.dt_min = lo; g.dt_max = hi; g.a_floor = fl;
  return M3_OK;
}
}  // namespace m3

extern "C" {

int m3_siso_forward_workspace(const m3_ssm_config* cfg, size_t* bytes) {
  ScanGeom g;
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  int st = resolve_ssm(cfg, false, &g);
  if (st != M3_OK) return st;
  *bytes = scan_workspace_bytes(g, false);
  return M3_OK;
}

int m3_mimo_forward_workspace(const m3_ssm_config* cfg, size_t* bytes) {
  ScanGeom g;
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  int st = resolve_ssm(cfg, true, &g);
  if (st != M3_OK) return st;
  *bytes = scan_workspace_bytes(g, false);
  return M3_OK;
}

static int scan_common(const m3_ssm_config* cfg, bool mimo, const ScanArgs& a,
                       const StepState* st, void* ws, size_t ws_bytes, m3_stream_t stream) {
  ScanGeom g;
  int status = resolve_ssm(cfg, mimo, &g);
  if (status != M3_OK) return status;
  status = check_ptrs({a.c, a.b, a.x, a.z, a.adt, a.dt, a.trap, a.c_bias, a.b_bias, a.d, a.out});
  if (status != M3_OK) return status;
  if ((status = check_angle_ptr(a.angle, g.A)) != M3_OK) return status;
  if (mimo && (status = check_ptrs({a.mimo_x, a.mimo_z, a.mimo_o, a.norm_weight})) != M3_OK)
    return status;
  if (st) {
    if (!count_below_u32({g.B, g.H, g.P, g.N}) || !count_below_u32({g.B, g.H, g.R, g.N}) ||
        !count_below_u32({g.B, g.H, g.R, g.P}) || !count_below_u32({g.B, g.H, g.A}))
      return M3_ERR_INVALID_ARGUMENT;
    if ((status = check_ptrs({st->ssm, st->k, st->v})) != M3_OK) return status;
    if ((status = check_angle_ptr(st->angle, g.A)) != M3_OK) return status;
  }
  const size_t need = scan_workspace_bytes(g, st != nullptr);
  if (need > 0 && (!ws || ws_bytes < need)) return M3_ERR_WORKSPACE;
  if (ws && !aligned16(ws)) return M3_ERR_UNALIGNED;
  return cuda_status(launch_scan(g, a, st, ws, ws_bytes, (cudaStream_t)stream));
}

int m3_siso_forward(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, float* out, void* workspace, size_t workspace_bytes,
                    m3_stream_t stream) {
  NvtxRange nvtx_range("m3_siso_forward");
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             nullptr, nullptr, nullptr, nullptr, out};
  return scan_common(cfg, false, a, nullptr, workspace, workspace_bytes, stream);
}

// `mamba3_siso_backward`: the SISO geometry rules, plus the backward's
// workspace arrays ([B,L,H,N] per-head C / B parts, [B,H,L,A] angles) below
// 2^32 elements.
static int resolve_backward(const m3_ssm_config* cfg, ScanGeom* g) {
  const int st = resolve_ssm(cfg, false, g);
  if (st != M3_OK) return st;
  if (!count_below_u32({g->B, g->L, g->H, g->N}) || !count_below_u32({g->B, g->L, g->H, g->A}))
    return M3_ERR_INVALID_ARGUMENT;
  return M3_OK;
}

int m3_siso_backward_workspace(const m3_ssm_config* cfg, size_t* bytes) {
  ScanGeom g;
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  const int st = resolve_backward(cfg, &g);
  if (st != M3_OK) return st;
  *bytes = backward_workspace_bytes(g);
  return M3_OK;
}

int m3_siso_backward(const m3_ssm_config* cfg, const float* dout, const float* c, const float* b,
                     const float* x, const float* z, const float* adt, const float* dt,
                     const float* trap, const float* angle, const float* c_bias,
                     const float* b_bias, const float* d, float* grad_c, float* grad_b,
                     float* grad_x, float* grad_z, float* grad_adt, float* grad_dt,
                     float* grad_trap, float* grad_angle, float* grad_c_bias, float* grad_b_bias,
                     float* grad_d, void* workspace, size_t workspace_bytes, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_siso_backward");
  ScanGeom g;
  int st = resolve_backward(cfg, &g);
  if (st != M3_OK) return st;
  st = check_ptrs({dout, c, b, x, z, adt, dt, trap, c_bias, b_bias, d, grad_c, grad_b, grad_x,
                   grad_z, grad_adt, grad_dt, grad_trap, grad_c_bias, grad_b_bias, grad_d});
  if (st != M3_OK) return st;
  if ((st = check_angle_ptr(angle, g.A)) != M3_OK) return st;
  if ((st = check_angle_ptr(grad_angle, g.A)) != M3_OK) return st;
  const size_t need = backward_workspace_bytes(g);
  if (!workspace || workspace_bytes < need) return M3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return M3_ERR_UNALIGNED;
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             nullptr, nullptr, nullptr, nullptr, nullptr};
  BwdArgs o{dout, grad_c, grad_b, grad_x, grad_z, grad_adt, grad_dt, grad_trap, grad_angle,
            grad_c_bias, grad_b_bias, grad_d};
  return cuda_status(launch_siso_backward(g, a, o, workspace, (cudaStream_t)stream));
}

// `mamba3_mimo_backward`: the MIMO geometry rules, plus the workspace arrays
// ([B,L,H,R,N] per-head C / B parts, [B,H,L,R,P] readouts) below 2^32 elements.
static int resolve_mimo_backward(const m3_ssm_config* cfg, ScanGeom* g) {
  const int st = resolve_ssm(cfg, true, g);
  if (st != M3_OK) return st;
  if (!count_below_u32({g->B, g->L, g->H, g->R, g->N}) ||
      !count_below_u32({g->B, g->L, g->H, g->R, g->P}) || !count_below_u32({g->B, g->L, g->H, g->A}))
    return M3_ERR_INVALID_ARGUMENT;
  return M3_OK;
}

int m3_mimo_backward_workspace(const m3_ssm_config* cfg, size_t* bytes) {
  ScanGeom g;
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  const int st = resolve_mimo_backward(cfg, &g);
  if (st != M3_OK) return st;
  *bytes = mimo_backward_workspace_bytes(g);
  return M3_OK;
}

int m3_mimo_backward(const m3_ssm_config* cfg, const float* dout, const float* c, const float* b,
                     const float* x, const float* z, const float* adt, const float* dt,
                     const float* trap, const float* angle, const float* c_bias,
                     const float* b_bias, const float* d, const float* mimo_x,
                     const float* mimo_z, const float* mimo_o, const float* norm_weight,
                     float* grad_c, float* grad_b, float* grad_x, float* grad_z, float* grad_adt,
                     float* grad_dt, float* grad_trap, float* grad_angle, float* grad_c_bias,
                     float* grad_b_bias, float* grad_d, float* grad_mimo_x, float* grad_mimo_z,
                     float* grad_mimo_o, float* grad_norm_weight, void* workspace,
                     size_t workspace_bytes, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_mimo_backward");
  ScanGeom g;
  int st = resolve_mimo_backward(cfg, &g);
  if (st != M3_OK) return st;
  st = check_ptrs({dout, c, b, x, z, adt, dt, trap, c_bias, b_bias, d, mimo_x, mimo_z, mimo_o,
                   norm_weight, grad_c, grad_b, grad_x, grad_z, grad_adt, grad_dt, grad_trap,
                   grad_c_bias, grad_b_bias, grad_d, grad_mimo_x, grad_mimo_z, grad_mimo_o,
                   grad_norm_weight});
  if (st != M3_OK) return st;
  if ((st = check_angle_ptr(angle, g.A)) != M3_OK) return st;
  if ((st = check_angle_ptr(grad_angle, g.A)) != M3_OK) return st;
  const size_t need = mimo_backward_workspace_bytes(g);
  if (!workspace || workspace_bytes < need) return M3_ERR_WORKSPACE;
  if (!aligned16(workspace)) return M3_ERR_UNALIGNED;
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             mimo_x, mimo_z, mimo_o, norm_weight, nullptr};
  MBwdArgs o{{dout, grad_c, grad_b, grad_x, grad_z, grad_adt, grad_dt, grad_trap, grad_angle,
              grad_c_bias, grad_b_bias, grad_d},
             grad_mimo_x, grad_mimo_z, grad_mimo_o, grad_norm_weight};
  return cuda_status(launch_mimo_backward(g, a, o, workspace, (cudaStream_t)stream));
}

static int packed_workspace(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                            bool mimo, size_t* bytes) {
  ScanGeom g;
  PreGeom p;
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  const int st = resolve_packed(cfg, pcfg, mimo, &g, &p);
  if (st != M3_OK) return st;
  *bytes = packed_plan(g, p).bytes;
  return M3_OK;
}

// The packed-projection scan, SISO (mimo operands null) or MIMO.
static int packed_common(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg, bool mimo,
                         const float* projected, const float* dt_bias, const float* c_bias,
                         const float* b_bias, const float* d, const float* mimo_x,
                         const float* mimo_z, const float* mimo_o, const float* norm_weight,
                         float* out, void* workspace, size_t workspace_bytes,
                         m3_stream_t stream) {
  ScanGeom g;
  PreGeom p;
  int st = resolve_packed(cfg, pcfg, mimo, &g, &p);
  if (st != M3_OK) return st;
  if ((st = check_ptrs({projected, dt_bias, c_bias, b_bias, d, out})) != M3_OK) return st;
  if (mimo && (st = check_ptrs({mimo_x, mimo_z, mimo_o, norm_weight})) != M3_OK) return st;
  const PackedPlan pl = packed_plan(g, p);
  if (pl.bytes > 0 && (!workspace || workspace_bytes < pl.bytes)) return M3_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return M3_ERR_UNALIGNED;
  const cudaStream_t s = (cudaStream_t)stream;
  if (pl.fused) {
    // the rows' B / C inverse RMS, then the scan: x, z and the scalar columns
    // of the packed rows, C / B through tensor maps
    char* wb = static_cast<char*>(workspace);
    float* inv = reinterpret_cast<float*>(wb + pl.off[0]);
    float* dt = reinterpret_cast<float*>(wb + pl.off[1]);
    float* adt = reinterpret_cast<float*>(wb + pl.off[2]);
    // (the status word is cleared first, so that the scan directly follows the
    // row pass in the stream)
    if (cudaMemsetAsync(workspace, 0, 16, s) != cudaSuccess) return M3_ERR_CUDA;
    if (launch_row_pre(p, projected, dt_bias, inv, dt, adt, s) != cudaSuccess) return M3_ERR_CUDA;
    const int64_t I = p.I, o_s = 2 * I + 2 * (int64_t)p.G * p.R * p.N;
    ScanArgs a{projected, projected, projected + I, projected, adt, dt,
               projected + o_s + 2 * p.H, projected + o_s + 3 * p.H, c_bias, b_bias, d,
               mimo_x, mimo_z, mimo_o, norm_weight, out, dt_bias, inv};
    return cuda_status(
        run_chunked(g, a, nullptr, workspace, s, launch_scan_chunk_packed, /*after_kernel=*/true));
  }
  char* w = static_cast<char*>(workspace);
  if (!use_chunk(g) && cudaMemsetAsync(w, 0, 16, s) != cudaSuccess) return M3_ERR_CUDA;
  float* f[8];
  for (int i = 0; i < 8; ++i) f[i] = reinterpret_cast<float*>(w + pl.off[i]);
  PreOut o{f[0], f[1], f[2], f[3], f[4], f[5], f[6], g.A ? f[7] : nullptr};
  cudaError_t e = launch_preprocess(p, projected, dt_bias, o, s);
  if (e != cudaSuccess) return M3_ERR_CUDA;
  ScanArgs a{o.ch, o.bh, o.x, o.z, o.adt, o.dt, o.trap, o.angle, c_bias, b_bias, d,
             mimo_x, mimo_z, mimo_o, norm_weight, out};
  return cuda_status(launch_scan(g, a, nullptr, w, pl.scan_bytes, s));
}

int m3_siso_forward_packed_workspace(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                                     size_t* bytes) {
  return packed_workspace(cfg, pcfg, false, bytes);
}

int m3_siso_forward_packed(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                           const float* projected, const float* dt_bias, const float* c_bias,
                           const float* b_bias, const float* d, float* out, void* workspace,
                           size_t workspace_bytes, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_siso_forward_packed");
  return packed_common(cfg, pcfg, false, projected, dt_bias, c_bias, b_bias, d, nullptr, nullptr,
                       nullptr, nullptr, out, workspace, workspace_bytes, stream);
}

int m3_mimo_forward_packed_workspace(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                                     size_t* bytes) {
  return packed_workspace(cfg, pcfg, true, bytes);
}

int m3_mimo_forward_packed(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                           const float* projected, const float* dt_bias, const float* c_bias,
                           const float* b_bias, const float* d, const float* mimo_x,
                           const float* mimo_z, const float* mimo_o, const float* norm_weight,
                           float* out, void* workspace, size_t workspace_bytes,
                           m3_stream_t stream) {
  NvtxRange nvtx_range("m3_mimo_forward_packed");
  return packed_common(cfg, pcfg, true, projected, dt_bias, c_bias, b_bias, d, mimo_x, mimo_z,
                       mimo_o, norm_weight, out, workspace, workspace_bytes, stream);
}

int m3_mimo_forward(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, const float* mimo_x, const float* mimo_z,
                    const float* mimo_o, const float* norm_weight, float* out,
                    void* workspace, size_t workspace_bytes, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_mimo_forward");
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             mimo_x, mimo_z, mimo_o, norm_weight, out};
  return scan_common(cfg, true, a, nullptr, workspace, workspace_bytes, stream);
}

int m3_siso_prefill_workspace(const m3_ssm_config* cfg, size_t* bytes) {
  ScanGeom g;
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  int st = resolve_ssm(cfg, false, &g);
  if (st != M3_OK) return st;
  *bytes = scan_workspace_bytes(g, true);
  return M3_OK;
}

int m3_mimo_prefill_workspace(const m3_ssm_config* cfg, size_t* bytes) {
  ScanGeom g;
  if (!bytes) return M3_ERR_INVALID_ARGUMENT;
  int st = resolve_ssm(cfg, true, &g);
  if (st != M3_OK) return st;
  *bytes = scan_workspace_bytes(g, true);
  return M3_OK;
}

int m3_siso_prefill(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, float* ssm_state, float* angle_state, float* k_state,
                    float* v_state, float* out, void* workspace, size_t workspace_bytes,
                    m3_stream_t stream) {
  NvtxRange nvtx_range("m3_siso_prefill");
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             nullptr, nullptr, nullptr, nullptr, out};
  StepState s{ssm_state, angle_state, k_state, v_state};
  return scan_common(cfg, false, a, &s, workspace, workspace_bytes, stream);
}

int m3_mimo_prefill(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, const float* mimo_x, const float* mimo_z,
                    const float* mimo_o, const float* norm_weight, float* ssm_state,
                    float* angle_state, float* k_state, float* v_state, float* out,
                    void* workspace, size_t workspace_bytes, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_mimo_prefill");
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             mimo_x, mimo_z, mimo_o, norm_weight, out};
  StepState s{ssm_state, angle_state, k_state, v_state};
  return scan_common(cfg, true, a, &s, workspace, workspace_bytes, stream);
}

static int step_common(const m3_ssm_config* cfg, bool mimo, const ScanArgs& a,
                       const StepState& s, m3_stream_t stream) {
  ScanGeom g;
  int st = resolve_ssm(cfg, mimo, &g);
  if (st != M3_OK) return st;
  if (g.L != 1) return M3_ERR_INVALID_ARGUMENT;
  // state element counts (`shader_u32` on the four state shapes)
  if (!count_below_u32({g.B, g.H, g.P, g.N}) || !count_below_u32({g.B, g.H, g.A}) ||
      !count_below_u32({g.B, g.H, g.R, g.N}) || !count_below_u32({g.B, g.H, g.R, g.P}))
    return M3_ERR_INVALID_ARGUMENT;
  st = check_ptrs({a.c, a.b, a.x, a.z, a.adt, a.dt, a.trap, a.c_bias, a.b_bias, a.d, a.out,
                   s.ssm, s.k, s.v});
  if (st != M3_OK) return st;
  if ((st = check_angle_ptr(a.angle, g.A)) != M3_OK) return st;
  if ((st = check_angle_ptr(s.angle, g.A)) != M3_OK) return st;
  if (mimo && (st = check_ptrs({a.mimo_x, a.mimo_z, a.mimo_o, a.norm_weight})) != M3_OK) return st;
  return cuda_status(launch_step(g, a, s, (cudaStream_t)stream));
}

int m3_siso_step(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                 const float* z, const float* adt, const float* dt, const float* trap,
                 const float* angle, const float* c_bias, const float* b_bias, const float* d,
                 float* ssm_state, float* angle_state, float* k_state, float* v_state,
                 float* out, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_siso_step");
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             nullptr, nullptr, nullptr, nullptr, out};
  StepState s{ssm_state, angle_state, k_state, v_state};
  return step_common(cfg, false, a, s, stream);
}

int m3_mimo_step(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                 const float* z, const float* adt, const float* dt, const float* trap,
                 const float* angle, const float* c_bias, const float* b_bias, const float* d,
                 const float* mimo_x, const float* mimo_z, const float* mimo_o,
                 const float* norm_weight, float* ssm_state, float* angle_state,
                 float* k_state, float* v_state, float* out, m3_stream_t stream) {
  NvtxRange nvtx_range("m3_mimo_step");
  ScanArgs a{c, b, x, z, adt, dt, trap, angle, c_bias, b_bias, d,
             mimo_x, mimo_z, mimo_o, norm_weight, out};
  StepState s{ssm_state, angle_state, k_state, v_state};
  return step_common(cfg, true, a, s, stream);
}

int m3_workspace_status(const void* workspace, size_t workspace_bytes, m3_stream_t stream) {
  if (!workspace || workspace_bytes < 16) return M3_ERR_INVALID_ARGUMENT;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return M3_ERR_CUDA;
  uint32_t word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return M3_ERR_CUDA;
  if (word == kStatusUndrained) return M3_ERR_DEVICE_STATE;
  return word == kStatusTimeout ? M3_ERR_TIMEOUT : M3_OK;
}

}  // extern "C"
