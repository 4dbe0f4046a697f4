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
 *  qkvz (MXFP6)                codes [Nqkvz][3H/4] uint8: each block of 32
 *                              OCP E2M3 codes (sign bit 5, 2 exponent and 3
 *                              mantissa bits) is 24 bytes, code i at bits
 *                              6i..6i+5 little-endian; qkvz_scales as for
 *                              MXFP4; the normed input stays bf16 (W6A16;
 *                              vLLM #60833, review "How to make the MXFP6
 *                              weights"); tensor-core engine only, H a
 *                              multiple of 512, dk = 128
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

/* Rows of one step: up to GDN_ROWS_PER_LAUNCH run as one launch (the row
 * cap of the pages' launch: vLLM #60833, Details, "Steps"; sgl-amd-mono #89,
 * Modifications); wider steps, up to GDN_MAX_ROWS, run as one launch per
 * tile of GDN_ROWS_PER_LAUNCH rows, in row order, each streaming the
 * weights again. */
#define GDN_ROWS_PER_LAUNCH 16
#define GDN_MAX_ROWS 64

typedef enum { GDN_STATE_F32 = 0, GDN_STATE_BF16 = 1 } gdn_state_dtype;
typedef enum { GDN_W_BF16 = 0, GDN_W_MXFP4 = 1, GDN_W_MXFP6 = 2 } gdn_weight_format;

/* Which unit runs the in_proj_qkvz / in_proj_ba dot products. Both engines
 * run the same launch (plan, TMA weight ring, shared-memory normed input,
 * hand-offs, recurrence) and differ only there. */
typedef enum {
  GDN_ENGINE_AUTO = 0,       /* the library's choice: the tensor cores */
  GDN_ENGINE_CUDA_CORE = 1,  /* f32 FMA dot products on CUDA cores (bf16 weights, decode steps) */
  GDN_ENGINE_TCGEN05 = 2     /* tcgen05.mma, TMEM accumulators */
} gdn_engine;

/* Launch options (launch_flags).
 *
 * By default a step is an ordinary launch with programmatic stream
 * serialisation: its CTAs start as soon as SMs free up at the end of the
 * kernel before it in the stream, and they begin streaming the step's
 * weights (in_proj_qkvz, in_proj_ba and the input-norm weight) and reading
 * the handle's plan tables BEFORE that kernel has finished. Only those
 * reads come early; x, residual, state_indices, the states and every other
 * weight are read after the previous kernel's writes are visible. So by
 * default the caller must not have the kernel launched just before the
 * step, in the same stream, write those weights (a weight load, update or
 * quantisation kernel, a copy_ into the weight tensor): the step could read
 * the old values. A copy engine operation, an event wait or any
 * non-kernel operation in between restores the ordering, and so does
 * GDN_LAUNCH_NO_EARLY_WEIGHTS, which makes the step read nothing before the
 * previous kernel is done (it keeps the overlapped launch otherwise; it costs
 * the overlap of the first weight tiles with that kernel's tail).
 *
 * The step's CTAs wait on one another, so all of them must be resident at
 * once; create checks that one CTA per SM fits. If other work holds SMs
 * while a step runs, its bounded waits run out and it reports
 * GDN_ERR_DEADLINE (it cannot hang). GDN_LAUNCH_COOPERATIVE makes the
 * runtime guarantee co-residency instead (cooperative launch), at the cost
 * of the overlap between consecutive steps. */
#define GDN_LAUNCH_COOPERATIVE 0x1
#define GDN_LAUNCH_NO_EARLY_WEIGHTS 0x2

typedef struct {
  int32_t hidden;
  int32_t num_k_heads;
  int32_t num_v_heads;
  int32_t head_k_dim;
  int32_t head_v_dim;
  int32_t conv_kernel;     /* must be 4 */
  int32_t num_slots;
  int32_t max_rows;        /* 1..GDN_MAX_ROWS */
  int32_t ssm_dtype;       /* gdn_state_dtype */
  int32_t qkvz_format;     /* gdn_weight_format */
  int32_t engine;          /* gdn_engine */
  float norm_eps;          /* Gemma input RMSNorm eps */
  float gated_norm_eps;    /* gated RMSNorm eps */
  float l2_eps;            /* q/k L2 norm: x / sqrt(sum(x^2) + l2_eps) */
  float q_scale;           /* multiplies the L2-normalised q */
  uint32_t deadline_us;    /* bound of every cross-CTA wait; 0 = 200000 */
  int32_t num_ctas;        /* persistent grid size; 0 = one CTA per SM */
  int32_t debug_flags;     /* test hooks (gdn_decode_diag.h); 0 in production */
  int32_t launch_flags;    /* GDN_LAUNCH_*; 0 = overlapped launches */
} gdn_decode_config;

typedef struct {
  const void* input_norm_w;     /* [H] bf16 */
  const void* qkvz;             /* [Nqkvz][H] bf16, [Nqkvz][H/2] MXFP4 or [Nqkvz][3H/4] MXFP6 codes */
  const uint8_t* qkvz_scales;   /* [Nqkvz][H/32] e8m0; MXFP4 / MXFP6 only, else NULL */
  const void* ba;               /* [Nba][H] bf16 */
  const void* conv_w;           /* [C][K] bf16 */
  const float* A_log;           /* [Hv] f32 */
  const void* dt_bias;          /* [Hv] bf16 */
  const void* gated_norm_w;     /* [dv] bf16 */
  const void* out_proj;         /* [H][Hv*dv] bf16, read by gdn_decode_step_out only; else NULL */
} gdn_decode_weights;

typedef struct gdn_decode gdn_decode_t;

/* Device bytes the caller must provide as the workspace for this config
 * (counters, the sticky error word, the plan tables, norm and projection
 * partials). 0 if the
 * config is invalid or unsupported. The workspace holds what the pages'
 * runtime helpers keep per launch key: the scratch of the cross-CTA
 * hand-offs and the health word (vLLM #60833, Details, "Shared helpers":
 * launch ABI and health words, a tagged mailbox with bounded waits). */
size_t gdn_decode_workspace_bytes(const gdn_decode_config* cfg);

/* Validate the config for the current device, bind the caller's workspace
 * (device memory of at least gdn_decode_workspace_bytes(cfg) bytes, 256-byte
 * aligned; it stays owned by the caller and must outlive the handle) and zero
 * it asynchronously on `stream`. The handle holds host state only: the
 * shapes, the stream-K plan of the projection units (written once into the
 * workspace) and the weight tile maps. It stands for one build key of the
 * pages' launch (one persistent launch per GDN layer front with its layer
 * shape, state dtype and first-layer variant; sgl-amd-mono #89,
 * Modifications, gdn.py and spec.py rows; vLLM #60833, Details,
 * "Launches"). Returns GDN_ERR_ARG / GDN_ERR_UNSUPPORTED / GDN_ERR_CUDA on
 * failure; a config outside the shapes this build runs is refused up front
 * with GDN_ERR_UNSUPPORTED, as the pages refuse configurations at start-up
 * (sgl-amd-mono #89, "Refusals"). */
gdn_status gdn_decode_create(const gdn_decode_config* cfg, void* workspace,
                             size_t workspace_bytes, void* stream,
                             gdn_decode_t** out);

/* Run one decode step of `rows` rows (1..max_rows) on `stream` (the step
 * list at the top of this header): one launch for up to GDN_ROWS_PER_LAUNCH
 * rows, else one launch per tile of that many rows. Asynchronous and
 * stream-ordered; allocates no memory on the host or the device; may be
 * captured in a CUDA graph. residual == NULL selects the first-layer variant
 * (r = x). See "Launch options" for the weights it reads before the previous
 * kernel in the stream has finished.
 * Reads x, residual, weights, state_indices; writes residual_out and core_out
 * and updates the rows' conv_state and ssm_state slots in place. Outputs must
 * not overlap any input. state_indices must be distinct among non-pad rows.
 * One step at a time per handle (the workspace is shared by its steps). */
gdn_status gdn_decode_step(gdn_decode_t* h, int32_t rows, const void* x,
                           const void* residual, const gdn_decode_weights* w,
                           const int32_t* state_indices, void* conv_state,
                           void* ssm_state, void* core_out, void* residual_out,
                           void* stream);

/* A decode step followed by the layer's out_proj in the same launch:
 * out[w][n] = bf16(sum_j out_proj[n][j] core[w][j]) over the Hv*dv core
 * columns, written to `out` ([rows][H] bf16; core_out is still written).
 * The pages fold out_proj into the GDN launch this way (SGLang #43558,
 * commit text of the SGLANG_QWEN3_8_DENSE_MONO_OPROJ fold, "dense_gdn
 * (K1Build.oproj)": every CTA publishes its core rows with a flag, CTAs poll
 * the flags and each runs its hidden columns of out_proj over the K share);
 * for one tensor-parallel rank's shard `out` is the rank's partial, to be
 * summed across ranks by the caller. Needs w->out_proj, the tensor-core
 * engine, at most 64 output columns per CTA (H <= 64 x grid) and Hv*dv a
 * multiple of 256 (else GDN_ERR_UNSUPPORTED). The out_proj weights are read
 * early like in_proj's (see "Launch options"). Other behaviour as
 * gdn_decode_step. */
gdn_status gdn_decode_step_out(gdn_decode_t* h, int32_t rows, const void* x, const void* residual,
                               const gdn_decode_weights* w, const int32_t* state_indices, void* conv_state,
                               void* ssm_state, void* core_out, void* residual_out, void* out, void* stream);

/* A verify step (multi-token, a state per token): `seqs` sequences of
 * `tokens` tokens each (rows s*tokens + t of x, residual, core_out and
 * residual_out; seqs * tokens <= max_rows, tokens <= GDN_ROWS_PER_LAUNCH).
 * Sequence s starts from the conv and SSM state in slot state_in[s]; after
 * token t, its conv and SSM state are written to slot state_out[s*tokens + t],
 * and token t + 1 continues from that stored state. So the tokens give what
 * as many decode steps would, and accepting a sequence's first a tokens is
 * taking slot state_out[s*tokens + a - 1]: a rejected draft token rolls back
 * by choosing a slot. The pages leave this as a follow-up (sgl-amd-mono #89,
 * Motivation: the launch keeps no state for each draft token, so a rejected
 * draft cannot roll back; vLLM #60833, Details, "Limitations / follow-ups":
 * MTP verify steps).
 * state_in [seqs] and state_out [seqs*tokens] are int32 device arrays; a
 * sequence with state_in <= 0 is padding (zero core rows, no state read or
 * written). Live sequences need distinct state_in slots, and all their
 * state_out slots distinct and apart from every state_in slot; the input
 * slots are only read. A slot >= num_slots (in or out) records GDN_ERR_INDEX
 * and makes the sequence padding. Each launch takes whole sequences
 * (floor(16 / tokens) of them). Tensor-core engine with bf16 in_proj_qkvz
 * only (else GDN_ERR_UNSUPPORTED). Other behaviour as gdn_decode_step. */
gdn_status gdn_decode_verify(gdn_decode_t* h, int32_t seqs, int32_t tokens, const void* x,
                             const void* residual, const gdn_decode_weights* w,
                             const int32_t* state_in, const int32_t* state_out, void* conv_state,
                             void* ssm_state, void* core_out, void* residual_out, void* stream);

/* Synchronise `stream` and read the sticky error word. Returns GDN_OK, or the
 * recorded device status; *detail (optional) receives the raw word:
 * bits 31..24 status, 23..16 the wait that gave up (1 norm, 3 projection
 * tile, 4 a weight-ring stage, 6 the core rows before
 * out_proj, 7 an out_proj weight chunk, 8 a state tile's copy into shared
 * memory, 9 every CTA's projection partials stored), 15..0 the CTA
 * (deadline) or row
 * (index error). This is the host
 * side of the pages' failure design: every wait in the launch is bounded, a
 * CTA that gives up records which wait in a sticky failed word, and the host
 * reads that word after the step without a fallback path (vLLM #60833,
 * Details, "Limitations / follow-ups"; sgl-amd-mono #89, Kernel checks,
 * "fault at the first wait"). */
gdn_status gdn_decode_check(gdn_decode_t* h, void* stream, uint32_t* detail);

/* Clear the error word, all counters and the partial buffers of the
 * workspace on `stream` (the plan stays). Until then every step on the
 * handle returns at once on the device, as a launch does once the pages'
 * sticky failed word is set (vLLM #60833, Details, "Limitations /
 * follow-ups"). */
gdn_status gdn_decode_reset(gdn_decode_t* h, void* stream);

/* Free the host handle. The workspace stays the caller's. */
void gdn_decode_destroy(gdn_decode_t* h);

const char* gdn_status_string(gdn_status s);

/* Persistent grid size and projection engine a handle launches with
 * (diagnostics for tests and benchmarks). */
gdn_status gdn_decode_launch_info(const gdn_decode_t* h, int32_t rows,
                                  int32_t* num_ctas, int32_t* engine);

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
 * Set-up: the first call on a device (with that device current), every
 * later call whose *cfg differs from the previous call's on that device, and
 * the first call in a new CUDA context on the device (after cudaDeviceReset,
 * or with another context current: the library keys its set-up on the
 * context's unique id, so it never reuses an address of a context that is
 * gone) first validates the config, looks up the scratch array's device
 * address, zeroes its counters, error word and partial buffers, and copies
 * the plan tables into it, stream-ordered on `stream`. They must start at
 * zero: a launch takes its number from a counter that grows from zero, and a
 * partial word carries the number of the launch that wrote it, so with the
 * counters back at zero an old word would pass for a new one. A call that
 * does the set-up must come before any stream capture on `stream`.
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
 * and the partial buffers so the next call runs. With detail == NULL the
 * call does not synchronise and nothing reads the word: once a device error
 * is set, that call and every later one return at once on the device
 * without writing their outputs or states, until a call with detail != NULL
 * reads and clears it. A caller that passes NULL for speed should pass
 * detail on some calls (every N-th step, say) to find such an error. */
gdn_status gdn_decode_step_static(const gdn_decode_config* cfg, int32_t rows, const void* x,
                                  const void* residual, const gdn_decode_weights* w,
                                  const int32_t* state_indices, void* conv_state,
                                  void* ssm_state, void* core_out, void* residual_out,
                                  void* stream, uint32_t* detail);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DECODE_H_ */
