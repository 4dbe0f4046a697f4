// out_proj folded into the step (SGLang #43558, commit text of the
// SGLANG_QWEN3_8_DENSE_MONO_OPROJ fold, "dense_gdn (K1Build.oproj)": every
// CTA publishes its core rows with a flag, then CTAs poll the flags and each
// runs its hidden columns of out_proj over the K share; the launch writes the
// out_proj result).
//
// After the recurrence, every CTA's core rows are in core_out. Each CTA then
// publishes a tagged word (behind a gpu-scope fence); CTA c owns the output
// columns [c H / G, (c + 1) H / G) of out[w][n] = sum_j W_o[n][j] core[w][j]
// (j over the Hv*dv core columns). It streams its out_proj rows in chunks
// of 256 columns through up to 3 stages (2-D TMA boxes with 128-byte
// swizzle into the weight ring, free after the projection; the first stages'
// copies go out before the hand-off, as no step writes the weights), and, once every CTA's word is
// seen, the core rows of each chunk (cp.async at L2: they were written by
// other CTAs in this launch), as many chunks ahead as there are stages. The contraction runs on the warp
// MMA (m16n8k16, bf16 inputs, f32 accumulation): the 16 rows on M, 8 output
// columns per N tile, each warp one 16-column K slice of every chunk; the 16
// warps' partial tiles are added in warp order and rounded once to bf16.
#pragma once

#include "gdn_common.cuh"
#include "gdn_tc_ptx.cuh"

namespace gdn {

constexpr int kOpKC = 256;                           // K columns per chunk (one k16 slice per warp)
constexpr int kOpMaxCols = 64;                       // output columns one CTA may own
constexpr uint32_t kOpRow = kOpKC * 2 + 16;          // bytes of a staged core row (padded: no bank conflicts)
constexpr uint32_t kOpBox = 64 * 128;                // one TMA box of weights: 64 rows x 64 columns, 128B swizzle
constexpr uint32_t kOpWBytes = 4 * kOpBox;           // a chunk's weights: 4 boxes (256 columns)
// a stage: the weights (swizzled TMA boxes need 1024-byte alignment), then
// core rows 0..15; the size rounded to 1024 so every stage stays aligned
constexpr uint32_t kOpStage = (kOpWBytes + kMaxRows * kOpRow + 1023) / 1024 * 1024;
constexpr int kOpMaxStages = 3;                      // chunks in flight (as the freed ring allows)
constexpr uint32_t kOpRing = 2 * kOpStage;           // shared memory the phase needs at least
constexpr uint32_t kWaitCore = 6, kWaitOutW = 7;     // error-word ids of its waits
static_assert(kOpKC / 16 == kWarps, "one k16 slice of each chunk per warp");
static_assert(kOpStage % 1024 == 0 && kOpBox % 1024 == 0, "swizzled TMA boxes on 1024-byte boundaries");
static_assert((uint32_t)kWarps * kMaxRows * kOpMaxCols * 4 <= kOpRing, "the warp partials fit the stages");

// The out_proj geometry of this CTA: its output columns [n0, n0 + ncols),
// the K chunks, the stages the ring holds.
struct OpShape {
  int n0, ncols, nch, ns;
  __device__ OpShape(const StepParams& p, size_t ring_bytes) {
    const int G = p.num_ctas, cta = blockIdx.x;
    n0 = (int)((long long)cta * p.H / G);
    ncols = (int)((long long)(cta + 1) * p.H / G) - n0;
    nch = p.Hv * p.dv / kOpKC;
    ns = (int)min((size_t)kOpMaxStages, ring_bytes / kOpStage);
  }
};

// The weights of chunk ch into stage ch % ns: rows n0..n0+63 (those past the
// CTA's columns are read and not used; past the last row TMA fills zeros),
// columns ch*256.. as four 64x64 boxes with 128-byte swizzle (one thread,
// lane 0 of warp 0). Weights: no step writes them, so these copies may go out
// before anything of the launch is known.
static __device__ __forceinline__ void op_issue_weights(const StepParams& p, const OpShape& o, uint8_t* ring,
                                                        uint64_t* bar, int ch) {
  const int s = ch % o.ns;
  if ((threadIdx.x & 31) == 0) {
    tc::mbar_arrive_expect_tx(&bar[s], kOpWBytes);
    for (int b = 0; b < 4; ++b)
      tc::tma_load_2d(ring + s * kOpStage + b * kOpBox, &p.tm_out, ch * kOpKC + b * 64, o.n0, &bar[s],
                      tc::policy_evict_first());
  }
  __syncwarp();
}

// The first stages' weight chunks, as soon as the ring is free (warp 0).
static __device__ __forceinline__ void out_proj_prefetch(const StepParams& p, uint8_t* ring, size_t ring_bytes,
                                                         uint64_t* bar) {
  const OpShape o(p, ring_bytes);
  for (int ch = 0; ch < min(o.ns, o.nch); ++ch) op_issue_weights(p, o, ring, bar, ch);
}

__device__ __forceinline__ void mma_m16n8k16_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                  uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Bounded wait on a stage's mbarrier (its weight rows landed).
static __device__ __forceinline__ bool op_wait(const StepParams& p, uint64_t* bar, uint32_t parity) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if ((ld_relaxed_u32(&p.ctr->error) >> 24) == kStatusDeadline) return false;
      if (globaltimer_ns() - t0 > p.deadline_ns) {
        record_error(p.ctr, kStatusDeadline, kWaitOutW, blockIdx.x);
        return false;
      }
    }
  }
}

// The out_proj phase of one CTA. `ring` is kOpRing bytes of shared memory no
// longer in use, `bar` two mbarriers (count 1) in phase 0. Returns false if a
// wait ran out (the error is recorded; the CTA's copies in flight have
// landed before it returns).
static __device__ bool phase_out_proj(const StepParams& p, uint8_t* ring, size_t ring_bytes, uint64_t* bar, int L,
                                      bool prefetch_after_publish) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, cta = blockIdx.x;
  const int W = p.rows, G = p.num_ctas;
  const int K = p.Hv * p.dv;
  const OpShape o(p, ring_bytes);
  const int n0 = o.n0, ncols = o.ncols, nch = o.nch, ns = o.ns, ntiles = (ncols + 7) / 8;
  // 1. this CTA's core rows are written: publish
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    st_tagged(p.core_flag + cta, tagged(L, 0.f));
  }
  if (prefetch_after_publish && warp == 0)
    for (int ch = 0; ch < min(ns, nch); ++ch) op_issue_weights(p, o, ring, bar, ch);
  // the first min(ns, nch) chunks' weights are in flight already (out_proj_prefetch)
  uint32_t inflight = (1u << min(ns, nch)) - 1;  // stages with a copy in flight
  auto drain = [&](uint32_t ph) {  // warp 0: let copies in flight land (bounded)
    for (int s = 0; s < ns; ++s)
      if ((inflight >> s) & 1u) {
        const unsigned long long c0 = globaltimer_ns();
        for (uint32_t it = 0; !tc::mbar_try_wait(&bar[s], (ph >> s) & 1u); ++it)
          if ((it & 63) == 0 && globaltimer_ns() - c0 > 100000000ull) break;
      }
  };
  // 2. every CTA's core rows (bounded poll of the tagged words, then a fence)
  __shared__ int op_ok;
  if (warp == 0) {
    constexpr int M = (kMaxCtas + 31) / 32;
    const unsigned long long* src = p.core_flag + lane;
    const int n = lane < G ? (G - lane + 31) / 32 : 0;
    unsigned long long v[M];
#pragma unroll
    for (int m = 0; m < M; ++m) v[m] = m < n ? ld_tagged(src + 32 * m) : 0ull;
    const bool ok = __all_sync(0xffffffffu, poll_tagged<M>(p, v, src, 32, n, L, kWaitCore));
    __threadfence();
    if (lane == 0) op_ok = ok;
  }
  __syncthreads();
  // the core rows of chunk ch into its stage: thread t < 32 W copies 16 bytes
  // (row t / 32, piece t % 32) with cp.async at L2 (they were written by
  // other CTAs), one commit group per chunk, ns chunks ahead
  const int crow = tid >> 5, c16 = tid & 31;
  const bool loads_core = crow < W;
  auto copy_core = [&](int ch) {
    if (loads_core)
      tc::cp_async16(ring + (ch % ns) * kOpStage + kOpWBytes + crow * kOpRow + c16 * 16,
                     p.core_out + (size_t)crow * K + (size_t)ch * kOpKC + c16 * 8);
    tc::cp_async_commit();
  };
  uint32_t ph = 0;  // parity of each stage's next completion (bit s)
  if (!op_ok) {
    if (warp == 0) drain(ph);
    return false;
  }
  for (int ch = 0; ch < min(ns, nch); ++ch) copy_core(ch);
  float acc[kOpMaxCols / 8][4];
#pragma unroll
  for (int j = 0; j < kOpMaxCols / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const int g = lane >> 2, t = lane & 3;
  const int k0 = warp * 16;  // this warp's k16 slice of every chunk
  bool ok = true;
  for (int ch = 0; ch < nch; ++ch) {
    const int s = ch % ns;
    tc::cp_async_wait_pending(min(ns, nch - ch) - 1);  // this chunk's core rows (this thread's copies)
    ok = __syncthreads_and(op_wait(p, &bar[s], (ph >> s) & 1u));  // and every thread's, and the weights
    if (!ok) break;  // the stage's copy may still be in flight: drained below
    ph ^= 1u << s;
    if (warp == 0) inflight &= ~(1u << s);
    const uint8_t* sw = ring + s * kOpStage;    // weights
    const uint8_t* sc = sw + kOpWBytes;          // core rows
    auto core32 = [&](int row, int col) { return *reinterpret_cast<const uint32_t*>(sc + row * kOpRow + col * 2); };
    // weight (row r, column kk) in the swizzled boxes: box kk / 64, its 16-byte
    // unit (kk % 64) / 8 stored at unit ^ (r % 8)
    auto w32 = [&](int r, int kk) {
      return *reinterpret_cast<const uint32_t*>(sw + (kk >> 6) * kOpBox + r * 128 +
                                                ((((kk & 63) >> 3) ^ (r & 7)) << 4) + (kk & 7) * 2);
    };
    const uint32_t a0 = core32(g, k0 + 2 * t), a1 = core32(g + 8, k0 + 2 * t);
    const uint32_t a2 = core32(g, k0 + 8 + 2 * t), a3 = core32(g + 8, k0 + 8 + 2 * t);
#pragma unroll
    for (int j = 0; j < kOpMaxCols / 8; ++j)
      if (j < ntiles) {
        const int wr = 8 * j + g;  // weight row of output column 8j + g
        mma_m16n8k16_bf16(acc[j], a0, a1, a2, a3, w32(wr, k0 + 2 * t), w32(wr, k0 + 8 + 2 * t));
      }
    __syncthreads();  // stage s read by every warp: it takes chunk ch + ns
    if (ch + ns < nch) {
      copy_core(ch + ns);
      if (warp == 0) {
        op_issue_weights(p, o, ring, bar, ch + ns);
        inflight |= 1u << s;
      }
    }
  }
  if (!ok) {
    tc::cp_async_wait_pending(0);
    if (warp == 0) drain(ph);
    return false;
  }
  // 3. the 16 warps' partial tiles, added in warp order, rounded once
  float* part = reinterpret_cast<float*>(ring);  // [warp][row][col]
#pragma unroll
  for (int j = 0; j < kOpMaxCols / 8; ++j)
    if (j < ntiles) {
      const int c = 8 * j + 2 * t;
      part[(warp * kMaxRows + g) * kOpMaxCols + c] = acc[j][0];
      part[(warp * kMaxRows + g) * kOpMaxCols + c + 1] = acc[j][1];
      part[(warp * kMaxRows + g + 8) * kOpMaxCols + c] = acc[j][2];
      part[(warp * kMaxRows + g + 8) * kOpMaxCols + c + 1] = acc[j][3];
    }
  __syncthreads();
  for (int i = tid; i < W * ncols; i += kThreads) {
    const int w = i / ncols, c = i - w * ncols;
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) sum += part[(k * kMaxRows + w) * kOpMaxCols + c];
    p.out[(size_t)w * p.H + n0 + c] = __float2bfloat16_rn(sum);
  }
  return true;
}

}  // namespace gdn
