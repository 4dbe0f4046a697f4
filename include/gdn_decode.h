/*
 * gdn_decode.h -- C ABI of the GB300 (sm_103a) decode-step front of a Gated
 * DeltaNet (GDN) layer: one persistent launch per layer and step, 1..16 rows.
 *
 * What one step computes, for every row (the step list of sgl-amd-mono #89,
 * Modifications table, gdn.py row; vLLM #60833, Details, "Launches"):
 *   residual add + Gemma RMSNorm, in_proj_qkvz and in_proj_ba, causal
 *   depthwise conv1d update + SiLU, L2-normalised q/k, gates
 *   g = -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b), the gated
 *   delta rule on the row's cached state slot (S <- e^g S;
 *   S += k (x) beta (v - S^T k); o = S^T q; f32 arithmetic, state stored in
 *   place as f32 or bf16), then the gated RMSNorm over each value head times
 *   SiLU(z). A pad row (state index <= 0) writes a zero core row and no state
 *   (sgl-amd-mono #89, Modifications, gdn.py row; Kernel checks, pad rows).
 *
 * Conventions for every entry point:
 *  - Tensor arguments are DEVICE pointers owned by the caller. The library
 *    never allocates device memory; the caller passes a workspace buffer.
 *  - All tensors are dense row-major in the layouts below. Pointers to bf16
 *    or f32 tensors must be 16-byte aligned; state_indices and A_log 4-byte.
 *  - bf16 is IEEE bfloat16 stored as uint16_t.
 *  - A stream argument is a cudaStream_t (passed as void*); NULL means the
 *    legacy default stream.
 *  - Host-side argument errors return before anything is launched. Device
 *    errors (a cross-CTA wait that passed its deadline, a state index >=
 *    num_slots) are recorded in a sticky error word in the workspace; every
 *    later step on that handle returns at once on the device until
 *    gdn_decode_reset(). gdn_decode_check() reads the word.
 *
 * Shapes: H = hidden, Hk/Hv = key/value heads, dk/dv = head dims (dk == dv,
 * 64 or 128), K = conv kernel (4), C = 2*Hk*dk + Hv*dv conv channels,
 * Nqkvz = 2*Hk*dk + 2*Hv*dv, Nba = 2*Hv, W = rows of this step.
 *
 * Layouts (our own; the pages name the tensors but not their layouts):
 *  x, residual, residual_out   [W][H] bf16
 *  core_out                    [W][Hv*dv] bf16 (value head h at columns h*dv..)
 *  state_indices               [W] int32, device; <= 0 marks a pad row
 *  conv_state                  [num_slots][C][K-1] bf16, oldest tap first,
 *                              channels in the order q | k | v
 *  ssm_state                   [num_slots][Hv][dv][dk] f32 or bf16 (S[v][k])
 *  qkvz (bf16)                 [Nqkvz][H] bf16, rows q(Hk*dk) | k(Hk*dk) |
 *                              v(Hv*dv) | z(Hv*dv)
 *  qkvz (MXFP4)                codes [Nqkvz][H/2] uint8 (element 2i in the
 *                              low nibble, OCP E2M1) and qkvz_scales
 *                              [Nqkvz][H/32] uint8 e8m0 (2^(byte-127));
 *                              tensor-core engine only, H a multiple of
 *                              512, dk = 128; the normed input is then
 *                              quantised to MXFP4 per block of 32 as well
 *  ba                          [Nba][H] bf16, rows b(Hv) | a(Hv)
 *  conv_w                      [C][K] bf16, tap K-1 multiplies the new input
 *  input_norm_w                [H] bf16 (Gemma form: x * rstd * (1 + w))
 *  A_log                       [Hv] f32;  dt_bias [Hv] bf16
 *  gated_norm_w                [dv] bf16, shared by all value heads
 *  Value head h reads key head h / (Hv/Hk).
 */
#ifndef GDN_DECODE_H_
#define GDN_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_ARG = 1,          /* bad argument: null, misaligned, aliasing, rows out of range */
  GDN_ERR_UNSUPPORTED = 2,  /* a shape or option this build does not run */
  GDN_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  GDN_ERR_DEADLINE = 4,     /* device: a cross-CTA wait passed its deadline */
  GDN_ERR_INDEX = 5,        /* device: a state index >= num_slots (row treated as a pad row) */
  GDN_ERR_FAILED = 6        /* device: the sticky error word holds an unknown code */
} gdn_status;

typedef enum { GDN_STATE_F32 = 0, GDN_STATE_BF16 = 1 } gdn_state_dtype;
typedef enum { GDN_W_BF16 = 0, GDN_W_MXFP4 = 1 } gdn_weight_format;

/* Which unit runs the in_proj_qkvz / in_proj_ba dot products. */
typedef enum {
  GDN_ENGINE_AUTO = 0,       /* the library's choice per width */
  GDN_ENGINE_CUDA_CORE = 1,  /* f32 FMA dot products on CUDA cores */
  GDN_ENGINE_TCGEN05 = 2     /* tcgen05.mma, TMEM accumulators, TMA-fed operands */
} gdn_engine;

/* Test hooks (debug_flags). Never set in production. */
#define GDN_DEBUG_SKIP_NORM_PUBLISH 0x1 /* CTA 0 never publishes its norm partials,
                                           so every CTA's first wait runs out */
#define GDN_DEBUG_TIMELINE 0x2          /* record %globaltimer stamps of each CTA's
                                           phases (read with gdn_decode_debug_timeline) */

/* Launch options (launch_flags). By default a step is an ordinary launch
 * with programmatic stream serialisation: a step's CTAs start as soon as
 * SMs free up at the end of the previous step in the stream, and stream the
 * step's weights before the previous step's results are needed. The step's
 * CTAs wait on one another, so all of them must be resident at once; create
 * checks that one CTA per SM fits. If other work holds SMs while a step runs,
 * its bounded waits run out and it reports GDN_ERR_DEADLINE (it cannot hang).
 * GDN_LAUNCH_COOPERATIVE makes the runtime guarantee co-residency instead
 * (cooperative launch), at the cost of that overlap. */
#define GDN_LAUNCH_COOPERATIVE 0x1

typedef struct {
  int32_t hidden;
  int32_t num_k_heads;
  int32_t num_v_heads;
  int32_t head_k_dim;
  int32_t head_v_dim;
  int32_t conv_kernel;     /* must be 4 */
  int32_t num_slots;
  int32_t max_rows;        /* 1..16 */
  int32_t ssm_dtype;       /* gdn_state_dtype */
  int32_t qkvz_format;     /* gdn_weight_format */
  int32_t engine;          /* gdn_engine */
  float norm_eps;          /* Gemma input RMSNorm eps */
  float gated_norm_eps;    /* gated RMSNorm eps */
  float l2_eps;            /* q/k L2 norm: x / sqrt(sum(x^2) + l2_eps) */
  float q_scale;           /* multiplies the L2-normalised q */
  uint32_t deadline_us;    /* bound of every cross-CTA wait; 0 = 200000 */
  int32_t num_ctas;        /* persistent grid size; 0 = one CTA per SM */
  int32_t debug_flags;     /* GDN_DEBUG_*; 0 in production */
  int32_t launch_flags;    /* GDN_LAUNCH_*; 0 = overlapped launches */
} gdn_decode_config;

typedef struct {
  const void* input_norm_w;     /* [H] bf16 */
  const void* qkvz;             /* [Nqkvz][H] bf16, or [Nqkvz][H/2] uint8 MXFP4 codes */
  const uint8_t* qkvz_scales;   /* [Nqkvz][H/32] e8m0; MXFP4 only, else NULL */
  const void* ba;               /* [Nba][H] bf16 */
  const void* conv_w;           /* [C][K] bf16 */
  const float* A_log;           /* [Hv] f32 */
  const void* dt_bias;          /* [Hv] bf16 */
  const void* gated_norm_w;     /* [dv] bf16 */
} gdn_decode_weights;

typedef struct gdn_decode gdn_decode_t;

/* Device bytes the caller must provide as the workspace for this config
 * (counters, the sticky error word, the plan tables, norm and projection
 * partials, and for the CUDA-core engine the normed input image). 0 if the
 * config is invalid or unsupported. */
size_t gdn_decode_workspace_bytes(const gdn_decode_config* cfg);

/* Validate the config for the current device, bind the caller's workspace
 * (device memory of at least gdn_decode_workspace_bytes(cfg) bytes, 256-byte
 * aligned; it stays owned by the caller and must outlive the handle) and zero
 * it asynchronously on `stream`. The handle holds host state only.
 * Returns GDN_ERR_ARG / GDN_ERR_UNSUPPORTED / GDN_ERR_CUDA on failure. */
gdn_status gdn_decode_create(const gdn_decode_config* cfg, void* workspace,
                             size_t workspace_bytes, void* stream,
                             gdn_decode_t** out);

/* Run one decode step of `rows` rows (1..max_rows) as one launch on `stream`.
 * Asynchronous and stream-ordered; allocates nothing; may be captured in a
 * CUDA graph. residual == NULL selects the first-layer variant (r = x).
 * Reads x, residual, weights, state_indices; writes residual_out and core_out
 * and updates the rows' conv_state and ssm_state slots in place. Outputs must
 * not overlap any input. state_indices must be distinct among non-pad rows.
 * One step at a time per handle (the workspace is shared by its steps). */
gdn_status gdn_decode_step(gdn_decode_t* h, int32_t rows, const void* x,
                           const void* residual, const gdn_decode_weights* w,
                           const int32_t* state_indices, void* conv_state,
                           void* ssm_state, void* core_out, void* residual_out,
                           void* stream);

/* Synchronise `stream` and read the sticky error word. Returns GDN_OK, or the
 * recorded device status; *detail (optional) receives the raw word:
 * bits 31..24 status, 23..16 the wait that gave up (1 norm, 2 normed input,
 * 3 projection tile, 4 a tensor-core pipeline stage), 15..0 the CTA
 * (deadline) or row (index error). */
gdn_status gdn_decode_check(gdn_decode_t* h, void* stream, uint32_t* detail);

/* Clear the error word, all counters and the partial buffers of the
 * workspace on `stream` (the plan stays). */
gdn_status gdn_decode_reset(gdn_decode_t* h, void* stream);

/* Free the host handle. The workspace stays the caller's. */
void gdn_decode_destroy(gdn_decode_t* h);

const char* gdn_status_string(gdn_status s);

/* Persistent grid size and projection engine a handle launches with
 * (diagnostics for tests and benchmarks). */
gdn_status gdn_decode_launch_info(const gdn_decode_t* h, int32_t rows,
                                  int32_t* num_ctas, int32_t* engine);

/* Diagnostics: synchronise `stream` and copy the phase timeline the last
 * step recorded (handle created with GDN_DEBUG_TIMELINE). cta_stamps receives
 * num_ctas x 48 uint64 nanosecond stamps: 0 start (after the previous step),
 * 1 norm partials out, 2 norm sums in (rstd known), 3 normed input out
 * (CUDA-core engine), 4 projection start, 5 projection end, 6 the first
 * recurrence task's projection partials in, 7 end, 8 that task's inputs
 * done, 9 first MMA, 10 last MMA done, 11 first weight tiles issued,
 * 12 x and residual staged, 13 that task's state written; 32+n the n-th
 * weight tile issued (n < 16, tensor-core engine); other slots unused.
 * tile_stamps receives num_tiles x 2 zeros (kept for the layout of this
 * call). Capacities are in elements; *num_ctas and *num_tiles receive the
 * sizes. */
gdn_status gdn_decode_debug_timeline(gdn_decode_t* h, void* stream, uint64_t* cta_stamps,
                                     int32_t cta_cap, uint64_t* tile_stamps, int32_t tile_cap,
                                     int32_t* num_ctas, int32_t* num_tiles);

/* Host-only diagnostics of the stream-K split of the projection work units
 * (no device call) for a grid of num_ctas CTAs. A unit is one 64-column step
 * (k-step) of one 256-row projection tile (tiles: in_proj_qkvz rows first,
 * then in_proj_ba rows); units are ordered by group g = (k-block g / T,
 * tile g % T) of `kblock` k-steps. Fills *engine (the engine the config runs
 * with), unit_begin[num_ctas+1] (CTA c takes units [unit_begin[c],
 * unit_begin[c+1])), seg_slot[num_ctas][16] (partial slot of the i-th group
 * CTA c touches), ks_first[num_ctas] and nb_slots[num_ctas] (CTA c keeps the
 * normed input of k-steps ks_first[c] + j mod ksteps, j < nb_slots[c]),
 * tile_count[*num_tiles] (partials per tile; capacity tile_cap), *ksteps and
 * *kblock. Errors as for gdn_decode_create. */
gdn_status gdn_decode_plan(const gdn_decode_config* cfg, int32_t num_ctas, int32_t* engine,
                           int32_t* unit_begin, uint8_t* seg_slot, uint16_t* ks_first, uint8_t* nb_slots,
                           uint8_t* tile_count, int32_t tile_cap, int32_t* num_tiles, int32_t* ksteps,
                           int32_t* kblock);

/* Largest scratch gdn_decode_step_static can use, in bytes (8 MiB). */
#define GDN_STATIC_SCRATCH_BYTES (8u << 20)

/* One decode step, computed exactly as gdn_decode_step computes it, for
 * callers that cannot allocate device memory: a C or C++ host program with no
 * PyTorch or other device allocator to provide a workspace, or a runtime
 * whose device memory is all handed out by its own pool, so that a
 * cudaMalloc would fail or fragment it. The pages this library follows have
 * no counterpart of this call.
 *
 * No handle and no workspace: the scratch (counters, sticky error word, plan
 * tables, norm and projection partials) is a fixed device array of
 * GDN_STATIC_SCRATCH_BYTES inside the library, one per device, held by every
 * GPU that loads the library's device code until the process exits. The call
 * allocates nothing on the host or the device, through no API or library.
 *
 * Set-up: the first call on a device (with that device current), and every
 * later call whose *cfg differs from the previous call's on that device,
 * first validates the config, looks up the scratch array's device address,
 * zeroes its counters, error word and partial buffers, and copies the plan
 * tables into it, stream-ordered on `stream`. They must start at zero: a
 * launch takes its number from a counter that grows from zero, and a partial
 * word carries the number of the launch that wrote it, so with the counters
 * back at zero an old word would pass for a new one. That first call must
 * come before any stream capture on `stream`.
 *
 * Arguments, layouts and the launch are those of gdn_decode_step; `cfg` takes
 * the place of the handle. The scratch is shared by every call on a device:
 * two calls whose launches overlap on the GPU (on different streams, or from
 * different host threads) race on it and give wrong results or deadline
 * errors. Calls from several host threads must be serialised by the caller.
 *
 * Errors: GDN_ERR_ARG and GDN_ERR_UNSUPPORTED as for gdn_decode_create and
 * gdn_decode_step, before any launch; GDN_ERR_UNSUPPORTED also when the
 * config's scratch would exceed GDN_STATIC_SCRATCH_BYTES (the layer front of
 * one tensor-parallel shard fits; a full 8192-wide layer with 64 value heads
 * does not: use gdn_decode_create with a workspace). Device errors are sticky
 * in the scratch as for a handle: if `detail` is not NULL the call waits for
 * its launch, stores the error word in *detail (layout of gdn_decode_check),
 * returns its status, and if it is non-zero clears the word, the counters
 * and the partial buffers so the next call runs. With detail == NULL the call does not synchronise. */
gdn_status gdn_decode_step_static(const gdn_decode_config* cfg, int32_t rows, const void* x,
                                  const void* residual, const gdn_decode_weights* w,
                                  const int32_t* state_indices, void* conv_state,
                                  void* ssm_state, void* core_out, void* residual_out,
                                  void* stream, uint32_t* detail);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DECODE_H_ */
