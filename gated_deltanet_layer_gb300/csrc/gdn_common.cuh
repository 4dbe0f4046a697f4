// Shared definitions of the GDN decode-step kernels: launch parameters,
// workspace layout, bf16 helpers, release/acquire counters and bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {

constexpr int kThreads = 512;              // one persistent CTA per SM
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 16;               // rows of one launch (wider steps run as several launches)
constexpr int kTileM = 256;                // projection rows per tile (one MMA's N)
constexpr int kTileShift = 8;              // log2(kTileM)
constexpr int kKStep = 64;                 // projection columns per work unit
constexpr int kMaxCtas = 256;
constexpr int kMaxTiles = 512;             // (Nqkvz + Nba) / 128 upper bound
constexpr int kMaxSegs = 16;               // tile segments in one CTA's unit range
constexpr int kKBlock = 16;                // k-steps per k-block in the k-block-major order
constexpr int kKBlockMxfp4 = 8;            // the same with coded (MXFP4, MXFP6) weights
constexpr int kMaxBSlots = 32;             // normed-input k-steps a CTA keeps in shared memory
constexpr int kMaxBSlotsMxfp4 = 24;        // the same with coded weights
constexpr int kMaxKHeads = 64;             // key heads of a layer (conv-group counters)

// Sticky error word: bits 31..24 status, 23..16 wait id, 15..0 CTA or row.
constexpr uint32_t kStatusDeadline = 4;
constexpr uint32_t kStatusIndex = 5;
constexpr uint32_t kWaitNorm = 1, kWaitTile = 3, kWaitProj = 9;  // (2: no longer used)

// in_proj_qkvz weight formats (the values of gdn_weight_format).
constexpr int kFmtBf16 = 0, kFmtMxfp4 = 1, kFmtMxfp6 = 2;
// The step kernel's form for bf16 weights with the projection's dot products
// on the CUDA cores (f32 FMA) instead of the tensor cores: the CUDA-core
// engine. Everything else (weight ring, windows, recurrence) is shared.
constexpr int kFmtBf16Fma = 3;
template <int FMT>
__host__ __device__ constexpr bool bf16_weights() { return FMT == kFmtBf16 || FMT == kFmtBf16Fma; }

constexpr int kDebugSkipNormPublish = 0x1;
constexpr int kDebugTimeline = 0x2;
constexpr int kTlSlots = 48;  // timeline stamps per CTA: 16 phase points, then 16 + 16 per-unit stamps

// Workspace header: counters on separate 128-byte lines. Every counter only
// grows; nothing is reset between launches. The launch number L of a step is
// norm_arrive / num_ctas at its start. The norm and projection partials are
// tagged words (tag = L + 1 beside the value, see tagged()), so a reader
// polls the data itself and no counter or fence guards them.
struct WsCounters {
  unsigned long long norm_arrive;   // +1 per CTA once its norm partials are out
  unsigned long long pad0[15];
  // +1 per CTA (a release) once every projection partial it writes is
  // stored: at (L + 1) x grid, launch L's partials are final
  unsigned long long proj_done;
  unsigned long long pad3[15];
  unsigned int error;               // sticky error word
  unsigned int pad2[63];
  // +1 per recurrence task of (row, key head) once it has read the old q/k
  // conv state; every launch adds the group size G or nothing, so the task
  // that makes the count a multiple of G is the group's last reader
  unsigned int conv_group[kMaxRows][kMaxKHeads];
  // Debug timeline (kDebugTimeline): %globaltimer stamps per CTA at phase
  // boundaries.
  unsigned long long tl_cta[kMaxCtas][kTlSlots];
};

// Timeline stamp points of a CTA.
enum TlPoint { TL_START = 0, TL_NORM_OUT, TL_NORM_IN, TL_XN_OUT, TL_PROJ_START, TL_PROJ_END,
               TL_REC_WAITED, TL_END, TL_REC_INPUTS, TL_MMA_FIRST, TL_MMA_LAST, TL_ISSUED,
               TL_R_STAGED, TL_REC_STATE, TL_TASK = 16, TL_UNIT_ISSUED = 32 };

struct StepParams {
  // shapes
  int H, Hk, Hv, dk, dv, C, Nqkvz, Nba, num_slots, rows;
  int tokens;          // tokens per sequence (rows = sequences x tokens); 1 for a decode step
  int group;           // Hv / Hk
  int tiles_qkvz;      // Nqkvz / kTileM
  int num_tiles;       // tiles_qkvz + ceil(Nba / kTileM)
  int ksteps;          // H / 64
  int kblock;          // k-steps per k-block of the unit order (== ksteps: tile-major)
  int max_contrib;     // most CTAs contributing to one tile
  int num_ctas;
  int fmt;             // in_proj_qkvz format: kFmtBf16, kFmtMxfp4 or kFmtMxfp6 (codes + e8m0 scales)
  int stages;          // bf16 weight tiles in flight per CTA
  int rstages;         // MXFP4 / MXFP6 code tiles in flight per CTA
  int xslots;          // normed-input k-steps a CTA keeps in shared memory
  unsigned int xpad;   // bytes past the window an MMA may read (and norm-sum scratch)
  unsigned int dyn_free;  // dynamic shared memory from the ring's start, free once the projection is done
  float norm_eps, gnorm_eps, l2_eps, q_scale;
  unsigned long long deadline_ns;
  int debug_flags;
  int early_weights;   // stream the weights (and read the plan) before griddepcontrol.wait
  // step tensors
  const __nv_bfloat16* x;
  const __nv_bfloat16* res;   // nullptr: first layer
  __nv_bfloat16* res_out;
  __nv_bfloat16* core_out;
  const int* idx;             // [rows / tokens] state slot each sequence starts from (and, decoding, updates)
  const int* idx_out;         // verify: [rows] slot of each token's state; nullptr when decoding
  __nv_bfloat16* conv_state;
  void* ssm_state;
  // weights
  const __nv_bfloat16* w_in;
  const __nv_bfloat16* w_qkvz;
  const uint8_t* w_qkvz_scales;
  const __nv_bfloat16* w_ba;
  const __nv_bfloat16* conv_w;
  const float* A_log;
  const __nv_bfloat16* dt_bias;
  const __nv_bfloat16* gnorm_w;
  const __nv_bfloat16* w_out;   // out_proj [H][Hv * dv] (with `out`)
  __nv_bfloat16* out;           // out_proj result [rows][H], or nullptr: no out_proj
  // workspace
  WsCounters* ctr;
  unsigned long long* norm_part;  // [kMaxRows][num_ctas] tagged words
  unsigned long long* core_flag;  // [num_ctas] tagged words: a CTA's core rows are written (out_proj)
  unsigned long long* proj_part;  // [num_tiles][max_contrib][kMaxRows][kTileM] tagged words
  // TMA descriptors of the weights: bf16 boxes of 64 columns x 256 rows with
  // 128-byte swizzle, or for MXFP4 / MXFP6 in_proj_qkvz uint8 boxes of one
  // k-step's codes (32 or 48 bytes) x 256 rows.
  CUtensorMap tm_qkvz;
  CUtensorMap tm_ba;
  CUtensorMap tm_out;  // out_proj [H][Hv*dv] bf16: boxes of 64 columns x 64 rows, 128-byte swizzle
  const struct PlanDev* plan;  // stream-K plan, in the workspace (written once at create)
};

// Stream-K plan of the projection work units. Unit u belongs to group
// g = u / kblock (k-block kb = g / num_tiles, tile t = g % num_tiles) and is
// k-step kb * kblock + u % kblock of tile t. CTA c takes units
// [unit_begin[c], unit_begin[c+1]); the i-th group it touches is its segment
// i, whose partial goes to slot seg_slot[c][i] of the tile. Tile t receives
// tile_num_ctas[t] partials. The CTA's normed-input k-steps are
// ks_first[c] + j (mod ksteps) for j < nb_slots[c].
// Each k-step's columns have one owner CTA (the first whose window holds
// it): bit j of own_mask[c] marks window slot j as
// owned; the owner writes residual_out and the norm partial of those columns.
struct PlanDev {
  int unit_begin[kMaxCtas + 1];
  unsigned char seg_slot[kMaxCtas][kMaxSegs];
  unsigned short ks_first[kMaxCtas];
  unsigned char nb_slots[kMaxCtas];
  unsigned char tile_num_ctas[kMaxTiles];
  unsigned int own_mask[kMaxCtas];
};

// ------------------------------------------------------------------ bf16

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ uint16_t f_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)f_to_bf16_bits(lo) | ((uint32_t)f_to_bf16_bits(hi) << 16);
}
__device__ __forceinline__ float round_bf16(float f) { return __bfloat162float(__float2bfloat16_rn(f)); }

// ------------------------------------------------------------------ memory

// Streamed once per launch: read-only, keep out of L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Written by other CTAs during this launch: read at L2.
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ float ld_cg_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ld_cg_f4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Release add: every write of this thread (and, after a bar.sync, of its CTA)
// before the add is visible to a thread that acquires the new value.
__device__ __forceinline__ unsigned long long atom_add_release_u64(unsigned long long* p,
                                                                   unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
// Relaxed add without a result (a count nobody orders data by).
__device__ __forceinline__ void red_add_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Release add without a result: the issuing thread does not wait for it.
__device__ __forceinline__ void red_add_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned int atom_add_relaxed_u32(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.add.relaxed.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned int atom_add_release_u32(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_add_acq_rel_u64(unsigned long long* p,
                                                                   unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

// Tagged words. A partial handed between CTAs is one 64-bit word: the launch
// tag L + 1 in the high half, the f32 value in the low half, written and read
// with relaxed gpu-scope 64-bit accesses (each single-copy atomic). A reader
// that sees its launch's tag sees that launch's value: no counter, no fence
// (vLLM #60833, Details, "Shared helpers": a tagged mailbox with bounded
// waits). The workspace starts zeroed (tag 0); reset zeroes it again.
__device__ __forceinline__ unsigned long long tagged(int L, float v) {
  return ((unsigned long long)(unsigned)(L + 1) << 32) | __float_as_uint(v);
}
__device__ __forceinline__ bool tag_is(unsigned long long w, int L) { return (unsigned)(w >> 32) == (unsigned)(L + 1); }
__device__ __forceinline__ float tagged_value(unsigned long long w) { return __uint_as_float((unsigned)w); }
__device__ __forceinline__ void st_tagged(unsigned long long* p, unsigned long long w) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ void st_tagged2(unsigned long long* p, unsigned long long a, unsigned long long b) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long* p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

// Programmatic dependent launch. wait: block until the launches this one
// depends on in the stream have completed and their writes are visible (a
// no-op when the launch was not made with programmatic serialisation).
// launch_dependents: let the next such launch in the stream be scheduled
// (its CTAs still need an SM that this launch's CTAs free).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Thread 0 of the CTA stamps a phase boundary when the timeline is on.
__device__ __forceinline__ void tl_stamp(const StepParams& p, int point) {
  if ((p.debug_flags & kDebugTimeline) && threadIdx.x == 0)
    p.ctr->tl_cta[blockIdx.x][point] = globaltimer_ns();
}
// The same from whichever single thread calls it.
__device__ __forceinline__ void tl_stamp_here(const StepParams& p, int point) {
  if (p.debug_flags & kDebugTimeline) p.ctr->tl_cta[blockIdx.x][point] = globaltimer_ns();
}

__device__ __forceinline__ void record_error(WsCounters* c, uint32_t status, uint32_t wait_id,
                                             uint32_t who) {
  uint32_t word = (status << 24) | ((wait_id & 0xff) << 16) | (who & 0xffff);
  atomicCAS(&c->error, 0u, word);  // the first error wins
}

// Spin (one thread) until *ctr >= target. Gives up after the deadline, or at
// once when another CTA recorded a deadline error; returns false then. An
// iteration cap backs up the timer.
static __device__ __noinline__ bool wait_counter(const StepParams& p, const unsigned long long* ctr,
                                          unsigned long long target, uint32_t wait_id) {
  if (ld_acquire_u64(ctr) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  const unsigned long long cap = p.deadline_ns / 32 + 4096;
  unsigned ns = 32;
  for (unsigned long long it = 0;; ++it) {
    __nanosleep(ns);
    if (ns < 64) ns <<= 1;
    if (ld_acquire_u64(ctr) >= target) return true;
    if ((ld_relaxed_u32(&p.ctr->error) >> 24) == kStatusDeadline) return false;
    if (globaltimer_ns() - t0 > p.deadline_ns || it > cap) {
      record_error(p.ctr, kStatusDeadline, wait_id, blockIdx.x);
      return false;
    }
  }
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Bounded poll of tagged words this thread has loaded (w[j] from
// base + j * stride, j < n): reloads the ones whose tag is not yet this
// launch's until all are. Gives up at the deadline (recording it) or once
// another CTA recorded a deadline error; returns false then.
template <int N>
__device__ __forceinline__ bool poll_tagged(const StepParams& p, unsigned long long (&w)[N],
                                            const unsigned long long* base, size_t stride, int n, int L,
                                            uint32_t wait_id) {
  static_assert(N <= 32, "one stale bit per word");
  uint32_t stale = 0;
#pragma unroll
  for (int j = 0; j < N; ++j)
    if (j < n && !tag_is(w[j], L)) stale |= 1u << j;
  if (!stale) return true;
  const unsigned long long t0 = globaltimer_ns();
  const unsigned long long cap = p.deadline_ns / 64 + 4096;
  for (unsigned long long it = 0;; ++it) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if ((stale >> j) & 1u) w[j] = ld_tagged(base + (size_t)j * stride);
    stale = 0;
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (j < n && !tag_is(w[j], L)) stale |= 1u << j;
    if (!stale) return true;
    if ((it & 15) == 15) {
      if ((ld_relaxed_u32(&p.ctr->error) >> 24) == kStatusDeadline) return false;
      if (globaltimer_ns() - t0 > p.deadline_ns || it > cap) {
        record_error(p.ctr, kStatusDeadline, wait_id, blockIdx.x);
        return false;
      }
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float t) { return t / (1.0f + expf(-t)); }

}  // namespace gdn
