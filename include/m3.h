/*
 * m3.h - C ABI of the GB300 (sm_103a) Mamba-3 selective-state scan library.
 *
 * Operations follow oarust 0.8.6 `src/rs/ml/matrix/mamba3.rs` (docs.rs source
 * view) and the `oa::ml::matrix` API reference:
 *   m3_preprocess     - `mamba3_preprocess`   (fused split + B/C RMS + dt/adt)
 *   m3_preprocess_backward - `mamba3_preprocess_backward` (its adjoint)
 *   m3_siso_forward   - `mamba3_siso`         (SISO selective-state recurrence)
 *   m3_mimo_forward   - `mamba3_mimo`         (shared-state MIMO recurrence)
 *   m3_siso_step      - `mamba3_siso_step`    (one token, explicit state)
 *   m3_mimo_step      - `mamba3_mimo_step`    (one MIMO token, explicit state)
 *   m3_siso_prefill / m3_mimo_prefill - the forward scans from / to an
 *                       explicit step state (prefill -> decode hand-off)
 *   m3_siso_forward_packed / m3_mimo_forward_packed - `mamba3_preprocess` and
 *                       `mamba3_siso` / `mamba3_mimo` in one call
 *   m3_siso_backward  - `mamba3_siso_backward` (the eleven SISO adjoints)
 *   m3_mimo_backward  - `mamba3_mimo_backward` (the fifteen MIMO adjoints)
 *
 * Conventions for every entry point:
 *  - Every tensor is float32, dense row-major, in device memory owned by the
 *    caller; the library allocates nothing and keeps no pointer after return.
 *  - Every base pointer must be 16-byte aligned (M3_ERR_UNALIGNED otherwise).
 *  - All checks run on the host before anything is enqueued. A rejected call
 *    enqueues no work and leaves every output and state buffer untouched.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream). Calls return once the kernels are enqueued; they do not wait.
 *  - Return value: an m3_status code; m3_status_string() describes it.
 */
#ifndef M3_H_
#define M3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. M3_ERR_INVALID_ARGUMENT mirrors the pages'
 * `Error::invalid_argument` results of the geometry checks. */
enum m3_status {
  M3_OK = 0,
  M3_ERR_INVALID_ARGUMENT = 1, /* geometry, limits, null pointer, overflow */
  M3_ERR_UNALIGNED = 2,        /* a base pointer is not 16-byte aligned */
  M3_ERR_WORKSPACE = 3,        /* workspace missing or smaller than required */
  M3_ERR_CUDA = 4,             /* a CUDA launch or runtime call failed */
  M3_ERR_TIMEOUT = 5,          /* a bounded device-side wait gave up */
  M3_ERR_DEVICE_STATE = 6      /* a bounded wait gave up and copies still in
                                  flight did not drain either: the CUDA
                                  context must be treated as unusable */
};

/* Arithmetic of the scans' dense contractions (an extension of SsmConfig). */
enum m3_math_mode {
  M3_MATH_FP32 = 0, /* FP32-exact: the token-by-token recurrence in FP32 FFMA */
  M3_MATH_TF32 = 1  /* chunked form, single-pass TF32 tensor MMA, FP32 accumulate
                       (shapes the chunked kernel does not take run as FP32) */
};

typedef struct CUstream_st* m3_stream_t; /* same type as cudaStream_t */

/* `Mamba3PreprocessConfig` (mamba3.rs): inner_size I, state_size N,
 * num_heads H, num_rope_angles A, num_groups G (> 0 here: no zero rule),
 * mimo_rank R (B/C rows per group), epsilon of the B/C RMS normalisation,
 * inclusive dt bounds [dt_min, dt_max], a_floor = positive floor of |A|. */
typedef struct {
  int64_t inner_size;
  int64_t state_size;
  int64_t num_heads;
  int64_t num_rope_angles;
  int64_t num_groups;
  int64_t mimo_rank;
  float epsilon;
  float dt_min;
  float dt_max;
  float a_floor;
} m3_preprocess_config;

/* `SsmConfig` (mamba3.rs): B, L, H, num_groups (0 means H), P = head_dim,
 * N = state_size, A = num_rope_angles, R = mimo_rank, and the three optional
 * paths. math_mode is an m3_math_mode (extension; 0 is FP32-exact). */
typedef struct {
  int64_t batch_size;
  int64_t sequence_length;
  int64_t num_heads;
  int64_t num_groups;
  int64_t head_dim;
  int64_t state_size;
  int64_t num_rope_angles;
  int64_t mimo_rank;
  int32_t has_z;
  int32_t has_d;
  int32_t has_output_norm;
  int32_t math_mode;
} m3_ssm_config;

/*
 * m3_preprocess - split and transform one packed Mamba-3 input projection
 * (`mamba3_preprocess`, `PreprocessGeometry::resolve`).
 *
 * projected [rows, W], W = 2I + 2GRN + 3H + A, columns in the order
 *   z | x | B rows (G*R rows of N) | C rows | dt_raw [H] | a_raw [H] | trap [H] | angle [A];
 * dt_bias [H]. Outputs: x, z [rows, I]; bh, ch [rows, G*R*N] (each N-row divided
 * by sqrt(mean square + epsilon)); dt, adt, trap [rows, H]; angle [rows, A]:
 *   dt  = clamp(softplus(dt_raw + dt_bias[h]), dt_min, dt_max)
 *   adt = -max(softplus(a_raw), a_floor) * dt;   trap, angle copied.
 * Checks: rows, I, N, H, G, R > 0; 2A <= N; epsilon, dt_min, dt_max, a_floor
 * finite; epsilon, dt_min, a_floor > 0; dt_min <= dt_max; W and every output
 * element count below 2^32. `angle` may be NULL when A == 0.
 */
int m3_preprocess(const m3_preprocess_config* cfg, int64_t rows, const float* projected,
                  const float* dt_bias, float* x, float* z, float* bh, float* ch, float* dt,
                  float* adt, float* trap, float* angle, m3_stream_t stream);

/*
 * m3_preprocess_backward - the adjoint of m3_preprocess
 * (`mamba3_preprocess_backward`, `Mamba3PreprocessBackward`): the gradients of
 * the packed projection and of dt_bias from those of the eight outputs.
 *
 * projected [rows, W] and dt_bias [H] as given to m3_preprocess; grad_x,
 * grad_z [rows, I]; grad_bh, grad_ch [rows, G*R*N]; grad_dt, grad_adt,
 * grad_trap [rows, H]; grad_angle [rows, A] (may be NULL when A == 0).
 * Outputs: grad_projected [rows, W], every column written:
 *   z, x, trap, angle columns = their output gradients;
 *   each B / C N-row u with output gradient g: s g - s^3 u (sum g u) / N,
 *     s = 1 / sqrt(mean u^2 + epsilon);
 *   dt_raw column = (grad_dt - a_mag grad_adt) sigmoid(dt_raw + dt_bias) while
 *     dt_min <= softplus(dt_raw + dt_bias) <= dt_max, else 0;
 *   a_raw column = -dt grad_adt sigmoid(a_raw) while softplus(a_raw) >= a_floor,
 *     else 0 (a_mag, dt as m3_preprocess computes them);
 * grad_dt_bias [H] = the dt_raw column summed over rows, in a fixed order that
 * depends on rows alone (the result is bit-identical from call to call).
 * Checks: as m3_preprocess, plus a workspace of at least
 * m3_preprocess_backward_workspace() bytes (16-byte aligned, device scratch
 * used only during the call's kernels; M3_ERR_WORKSPACE when missing or small).
 */
int m3_preprocess_backward_workspace(const m3_preprocess_config* cfg, int64_t rows,
                                     size_t* bytes);
int m3_preprocess_backward(const m3_preprocess_config* cfg, int64_t rows, const float* projected,
                           const float* dt_bias, const float* grad_x, const float* grad_z,
                           const float* grad_bh, const float* grad_ch, const float* grad_dt,
                           const float* grad_adt, const float* grad_trap,
                           const float* grad_angle, float* grad_projected, float* grad_dt_bias,
                           void* workspace, size_t workspace_bytes, m3_stream_t stream);

/*
 * m3_siso_forward - the Mamba-3 SISO selective-state recurrence over a whole
 * sequence from a zero state (`mamba3_siso`, `Geometry::resolve`).
 *
 * Operands: c, b [B,L,G,N]; x, z [B,L,H,P]; adt, dt, trap [B,L,H]; angle
 * [B,L,A] (may be NULL when A == 0); c_bias, b_bias [H,N]; d [H]. Output
 * out [B,L,H,P]. Checks: B,L,H,G,P,N > 0, H % G == 0, P <= 128, N <= 128,
 * A <= 64, 2A <= N, mimo_rank == 1, has_output_norm == 0, every element count
 * below 2^32. z and d are read only when has_z / has_d are set but must be
 * valid pointers regardless, as in the pages' shape checks.
 * workspace: device scratch of at least m3_siso_forward_workspace() bytes,
 * 16-byte aligned, used only during the call's kernels (may be NULL when that
 * size is 0). Calls that share a workspace must not overlap on the GPU.
 */
int m3_siso_forward_workspace(const m3_ssm_config* cfg, size_t* bytes);
int m3_siso_forward(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, float* out, void* workspace, size_t workspace_bytes,
                    m3_stream_t stream);

/*
 * m3_siso_forward_packed - m3_preprocess and m3_siso_forward in one call: the
 * SISO scan of a packed input projection (`mamba3_preprocess` feeding
 * `mamba3_siso`; the pages run them as two ops, this entry point fuses them).
 *
 * projected [B*L, W] in the m3_preprocess column order, dt_bias [H]; c_bias,
 * b_bias [H,N]; d [H]; out [B,L,H,P]. pcfg must describe the same layer as
 * cfg: inner_size = H*P, state_size = N, num_heads = H, num_rope_angles = A,
 * num_groups = the resolved G, mimo_rank = 1; its epsilon / dt bounds /
 * a_floor are checked as in m3_preprocess, cfg as in m3_siso_forward.
 * Where the chunked kernel has a TMA instance for the shape (P = 64, N = 128,
 * A = 32 or 64) and W is a multiple of 4, a short pass writes the inverse
 * RMS of every B / C row into the workspace (computed exactly as m3_preprocess
 * computes it) and the scan reads the packed rows directly, scaling the B / C
 * rows in shared memory and forming dt / adt by the same maps, so the output
 * has the bits of m3_preprocess followed by m3_siso_forward in the same math
 * mode. Otherwise the preprocess writes its outputs into the workspace and the
 * scan reads them from there (the same result).
 * workspace: at least m3_siso_forward_packed_workspace() bytes (never 0),
 * 16-byte aligned; its first word is the scan's status word, read by
 * m3_workspace_status.
 */
int m3_siso_forward_packed_workspace(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                                     size_t* bytes);
int m3_siso_forward_packed(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                           const float* projected, const float* dt_bias, const float* c_bias,
                           const float* b_bias, const float* d, float* out, void* workspace,
                           size_t workspace_bytes, m3_stream_t stream);

/*
 * m3_mimo_forward_packed - m3_preprocess and m3_mimo_forward in one call
 * (`mamba3_preprocess` feeding `mamba3_mimo`). As m3_siso_forward_packed, with
 * the MIMO operands and checks of m3_mimo_forward: pcfg->mimo_rank = R (the
 * packed rows hold G*R B / C rows), c_bias / b_bias [H,R,N], mimo_x / mimo_z /
 * mimo_o [H,R,P], norm_weight [H,P]. Every shape runs the preprocess into the
 * workspace and then the MIMO scan (the MIMO scan kernel is bound by its
 * per-chunk latency, and the per-head RMS of R rank rows that reading the
 * packed rows directly adds to it costs more than the preprocess pass), so
 * the output is that of m3_preprocess followed by m3_mimo_forward in the same
 * math mode.
 */
int m3_mimo_forward_packed_workspace(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                                     size_t* bytes);
int m3_mimo_forward_packed(const m3_ssm_config* cfg, const m3_preprocess_config* pcfg,
                           const float* projected, const float* dt_bias, const float* c_bias,
                           const float* b_bias, const float* d, const float* mimo_x,
                           const float* mimo_z, const float* mimo_o, const float* norm_weight,
                           float* out, void* workspace, size_t workspace_bytes,
                           m3_stream_t stream);

/*
 * m3_mimo_forward - the shared-state Mamba-3 MIMO recurrence (`mamba3_mimo`,
 * `MimoGeometry::resolve`).
 *
 * Operands as m3_siso_forward except c, b [B,L,R*G,N] (row g*R + r is rank r
 * of group g) and c_bias, b_bias [H,R,N]; plus mimo_x, mimo_z, mimo_o [H,R,P]
 * and norm_weight [H,P] (read only when has_output_norm; always required).
 * Output RMS norm epsilon is 1.0e-5. Checks: as SISO but 1 <= R <= 8 and
 * P*N <= 4096; has_output_norm allowed.
 */
int m3_mimo_forward_workspace(const m3_ssm_config* cfg, size_t* bytes);
int m3_mimo_forward(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, const float* mimo_x, const float* mimo_z,
                    const float* mimo_o, const float* norm_weight, float* out,
                    void* workspace, size_t workspace_bytes, m3_stream_t stream);

/*
 * m3_siso_backward - the eleven adjoints of m3_siso_forward
 * (`mamba3_siso_backward`, the fields of `SsmBackward`): given grad_out
 * [B,L,H,P], the gradient of a loss with respect to the scan's output, and the
 * forward operands, writes the gradient with respect to each operand in that
 * operand's layout: grad_c, grad_b [B,L,G,N] (summed over the heads that share
 * a group's rows); grad_x, grad_z [B,L,H,P]; grad_adt, grad_dt, grad_trap
 * [B,L,H]; grad_angle [B,L,A] (summed over the heads; may be NULL when
 * A == 0); grad_c_bias, grad_b_bias [H,N] (summed over batch and tokens);
 * grad_d [H]. grad_z is zero without has_z, grad_d zero without has_d. The
 * scan starts from a zero state, as in m3_siso_forward.
 * Arithmetic: FP32 on the CUDA cores whatever cfg->math_mode says (two
 * token-sequential sweeps per (b, h) and a reduction in a fixed order, so
 * that repeated calls give the same bits). Checks: those of m3_siso_forward,
 * plus B*L*H*N and B*L*H*A below 2^32; every pointer but angle / grad_angle
 * (when A == 0) non-NULL and 16-byte aligned.
 * workspace: at least m3_siso_backward_workspace() bytes (never 0), 16-byte
 * aligned, used only during the call's kernels. Outputs must not overlap the
 * inputs or the workspace.
 */
int m3_siso_backward_workspace(const m3_ssm_config* cfg, size_t* bytes);
int m3_siso_backward(const m3_ssm_config* cfg, const float* grad_out, const float* c,
                     const float* b, const float* x, const float* z, const float* adt,
                     const float* dt, const float* trap, const float* angle,
                     const float* c_bias, const float* b_bias, const float* d, float* grad_c,
                     float* grad_b, float* grad_x, float* grad_z, float* grad_adt,
                     float* grad_dt, float* grad_trap, float* grad_angle, float* grad_c_bias,
                     float* grad_b_bias, float* grad_d, void* workspace, size_t workspace_bytes,
                     m3_stream_t stream);

/*
 * m3_mimo_backward - the fifteen adjoints of m3_mimo_forward
 * (`mamba3_mimo_backward`, the fields of `Mamba3MimoBackward`): given grad_out
 * [B,L,H,P] and the forward operands, writes grad_c, grad_b [B,L,R*G,N] (summed
 * over the heads sharing a group's rows); grad_x, grad_z [B,L,H,P]; grad_adt,
 * grad_dt, grad_trap [B,L,H]; grad_angle [B,L,A] (summed over heads; may be
 * NULL when A == 0); grad_c_bias, grad_b_bias [H,R,N]; grad_d [H];
 * grad_mimo_x, grad_mimo_z, grad_mimo_o [H,R,P]; grad_norm_weight [H,P] (the
 * batch and token sums). grad_z and grad_mimo_z are zero without has_z,
 * grad_d without has_d, grad_norm_weight without has_output_norm. The scan
 * starts from a zero state.
 * Arithmetic: FP32 on the CUDA cores whatever cfg->math_mode says: a forward
 * sweep for the readouts y_{t,r} (recording the state at every tile start), a
 * per-token pass for the norm, gate and mimo_o adjoints, a pass over all
 * tiles at once for the query gradients, a reverse sweep and a reduction in a
 * fixed order (repeated calls give the same bits).
 * Checks: those of m3_mimo_forward, plus B*L*H*R*N, B*L*H*R*P and B*L*H*A
 * below 2^32; every pointer but angle / grad_angle (when A == 0) non-NULL and
 * 16-byte aligned. workspace: at least m3_mimo_backward_workspace() bytes,
 * 16-byte aligned. Outputs must not overlap the inputs or the workspace.
 */
int m3_mimo_backward_workspace(const m3_ssm_config* cfg, size_t* bytes);
int m3_mimo_backward(const m3_ssm_config* cfg, const float* grad_out, const float* c,
                     const float* b, const float* x, const float* z, const float* adt,
                     const float* dt, const float* trap, const float* angle,
                     const float* c_bias, const float* b_bias, const float* d,
                     const float* mimo_x, const float* mimo_z, const float* mimo_o,
                     const float* norm_weight, float* grad_c, float* grad_b, float* grad_x,
                     float* grad_z, float* grad_adt, float* grad_dt, float* grad_trap,
                     float* grad_angle, float* grad_c_bias, float* grad_b_bias, float* grad_d,
                     float* grad_mimo_x, float* grad_mimo_z, float* grad_mimo_o,
                     float* grad_norm_weight, void* workspace, size_t workspace_bytes,
                     m3_stream_t stream);

/*
 * m3_siso_prefill / m3_mimo_prefill - the scan of m3_siso_forward /
 * m3_mimo_forward continued from, and handing over, an explicit recurrent
 * state: the prefill -> decode hand-off between the full-sequence ops and the
 * step ops (`mamba3_siso` / `mamba3_siso_step`, `mamba3_mimo` /
 * `mamba3_mimo_step`).
 *
 * The four states use the step layouts: ssm_state [B,H,P,N], angle_state
 * [B,H,A] (may be NULL when A == 0), k_state [B,H,R,N] (rotated, biased key
 * of the last token), v_state [B,H,R,P] (its rank-scaled value). They are read
 * as the state before token 0 (all zero = the start of a sequence) and
 * overwritten with the state after token L-1, so that m3_siso_step can take
 * over at token L. Operands and checks are those of the forward calls;
 * workspace: at least m3_*_prefill_workspace() bytes.
 */
int m3_siso_prefill_workspace(const m3_ssm_config* cfg, size_t* bytes);
int m3_siso_prefill(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, float* ssm_state, float* angle_state, float* k_state,
                    float* v_state, float* out, void* workspace, size_t workspace_bytes,
                    m3_stream_t stream);
int m3_mimo_prefill_workspace(const m3_ssm_config* cfg, size_t* bytes);
int m3_mimo_prefill(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                    const float* z, const float* adt, const float* dt, const float* trap,
                    const float* angle, const float* c_bias, const float* b_bias,
                    const float* d, const float* mimo_x, const float* mimo_z,
                    const float* mimo_o, const float* norm_weight, float* ssm_state,
                    float* angle_state, float* k_state, float* v_state, float* out,
                    void* workspace, size_t workspace_bytes, m3_stream_t stream);

/*
 * m3_siso_forward_static - m3_siso_forward without a workspace argument, for
 * callers that cannot allocate device memory (code running inside a host that
 * owns every device allocation, such as a framework plugin or an inference
 * runtime with its own pool, or a latency-critical loop where a cudaMalloc
 * would synchronize the device). The source pages have no counterpart: this
 * entry point belongs to this library's C ABI only.
 *
 * Operands, checks and results are those of m3_siso_forward. The scratch the
 * scan needs comes from a fixed 1 MiB array in the library's device image
 * (held by every GPU that loads the library until the process exits); this
 * call allocates nothing. Geometries whose m3_siso_forward_workspace() size
 * exceeds 1 MiB are rejected with M3_ERR_WORKSPACE. Every call looks up the
 * array's device address in the current CUDA context (cudaGetSymbolAddress, a
 * host-side query), so hosts that run their own context get the address valid
 * there; the first call on a device may load the library's device code, so
 * make it before any stream capture. All calls on a device share the array
 * and it keeps the last call's contents: calls that overlap on the GPU race
 * and must not be issued; each call clears what must start at zero.
 *
 * m3_siso_forward_static_status - waits for `stream`, then reads the status
 * word that the bounded device-side waits of the last m3_siso_forward_static
 * call on the current device wrote into the array: M3_OK, M3_ERR_TIMEOUT or
 * M3_ERR_DEVICE_STATE (as m3_workspace_status for a caller workspace).
 */
int m3_siso_forward_static(const m3_ssm_config* cfg, const float* c, const float* b,
                           const float* x, const float* z, const float* adt, const float* dt,
                           const float* trap, const float* angle, const float* c_bias,
                           const float* b_bias, const float* d, float* out, m3_stream_t stream);
int m3_siso_forward_static_status(m3_stream_t stream);

/*
 * m3_siso_step - advance one SISO token and update four recurrent states in
 * place (`mamba3_siso_step`). cfg->sequence_length must be 1; operands are the
 * length-one forms of m3_siso_forward. States (read, then overwritten):
 *   ssm_state [B,H,P,N], angle_state [B,H,A] (cumulative angle; may be NULL
 *   when A == 0), k_state [B,H,N] (rotated, biased key of the last token),
 *   v_state [B,H,P] (value of the last token).
 * A zero state equals the start of a sequence. A rejected call leaves the
 * states untouched ("mutated only after the complete operation has been
 * validated"). Output out [B,1,H,P].
 * Device-side waits are bounded: if the copy of a (b, h) state row into the
 * kernel's shared memory does not complete within about a second (a device
 * fault), that output row is set to NaN and that ssm_state row is left as it
 * was (the step has no workspace, hence no status word).
 */
int m3_siso_step(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                 const float* z, const float* adt, const float* dt, const float* trap,
                 const float* angle, const float* c_bias, const float* b_bias, const float* d,
                 float* ssm_state, float* angle_state, float* k_state, float* v_state,
                 float* out, m3_stream_t stream);

/*
 * m3_mimo_step - advance one MIMO token (`mamba3_mimo_step`). Operands as
 * m3_mimo_forward with sequence_length == 1. States: ssm [B,H,P,N], angle
 * [B,H,A], k_state [B,H,R,N], v_state [B,H,R,P] (rank-scaled values).
 */
int m3_mimo_step(const m3_ssm_config* cfg, const float* c, const float* b, const float* x,
                 const float* z, const float* adt, const float* dt, const float* trap,
                 const float* angle, const float* c_bias, const float* b_bias, const float* d,
                 const float* mimo_x, const float* mimo_z, const float* mimo_o,
                 const float* norm_weight, float* ssm_state, float* angle_state,
                 float* k_state, float* v_state, float* out, m3_stream_t stream);

/*
 * m3_workspace_status - waits for `stream`, then reads the device status word
 * that the scans' bounded waits write into `workspace`: M3_OK, M3_ERR_TIMEOUT
 * if a wait gave up during the last call that used it, or M3_ERR_DEVICE_STATE
 * if, after that, the kernel's bounded wait for its own copies still in flight
 * gave up as well (the kernel then exits with those copies unfinished, and the
 * context is in an undefined state).
 */
int m3_workspace_status(const void* workspace, size_t workspace_bytes, m3_stream_t stream);

/*
 * m3_selftest_wait_timeout - diagnostic: enqueues one kernel that waits on an
 * mbarrier nothing completes, with the same bounded wait the scans use, for
 * about `budget_cycles` SM clock cycles (1 .. 4e9), then records
 * M3_ERR_TIMEOUT in the workspace status word (first 16 bytes, zeroed first)
 * and exits normally. m3_workspace_status() then returns M3_ERR_TIMEOUT and
 * the context stays usable. Checks: workspace non-NULL, >= 16 bytes, 16-byte
 * aligned.
 */
int m3_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t budget_cycles,
                             m3_stream_t stream);

/* Human-readable description of a status code (static string). */
const char* m3_status_string(int status);

/* Number of kernels this library has enqueued since it was loaded. */
uint64_t m3_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* M3_H_ */
