// The persistent GDN decode-step kernel. The projections run on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM, weight
// tiles fed by TMA) or, in the CUDA-core engine's instances (kFmtBf16Fma),
// as f32 FMA dot products on the CUDA cores from the same weight ring.
//
// The MMA is D[m][n] += A[m][k] B[n][k] with A = the normed input xn (M = 64:
// the step's up to 16 rows; the MMA also reads 48 rows of whatever lies past
// a slice, whose results land in TMEM lanes nobody reads) and B = a 256-row
// weight tile (N = 256, K-major, 128-byte swizzle). The tensor core's time
// per instruction follows N x K alone (128 cycles at N = 256, the same for
// M = 64 and M = 128; 64 cycles at N = 128), so the weights take the wide N
// side, one instruction consumes 8 KB of weights, and M is the smallest
// shape whose D rows 0..15 sit in TMEM lanes 0..15.
//
// One persistent CTA per SM. Roles during the projection:
//   thread 32           fills the ring's first stages (2..6 tiles of 256 rows
//                       x 64 columns, as shared memory allows) before the norm
//                       hand-off: as soon as the CTA starts when the previous
//                       step is still running (programmatic dependent
//                       launch), else right after issuing its x and residual
//                       loads, so HBM streams weights while the hand-off runs
//   warp 0              TMA producer: refills each stage its consumers
//                       release (lane 0 issues)
//   warp 1              allocates TMEM; issues tcgen05.mma (lane 0) into one
//                       of two 64 x 256 f32 accumulators (512 columns)
// Whole warps run these loops, waiting together, with lane 0 issuing (a
// little faster end to end than a lone thread). In this kernel a 4-MMA unit
// takes ~930 SM cycles of the issuing warp against ~510 for the same MMAs
// issued back to back alone on an SM; the difference is issue overhead
// between units, not tensor-core time.
//   warps 4, 8, 12      drain an accumulator with tcgen05.ld (lane w holds
//                       row w of the step; the warps split the columns) and
//                       write the CTA's partial of the tile as tagged words;
//                       the recurrence tasks reduce the partials they need
//   warps 2, 3, 5-7,    (MXFP4 or MXFP6 in_proj_qkvz) decode each code tile
//   9-11                into a bf16 tile for the MMA
//   warps 8-15          (CUDA-core engine, in place of the MMA, the drain
//                       and TMEM) thread i: row i of each tile, its dot
//                       products with the step's rows, the same partials
// The A operand (xn of the CTA's k-steps, 16 rows, rows past the step's row
// count zero) is built per launch in shared memory: r = x + residual is
// staged while the norm hand-off is in flight and normalised in place once
// rstd is known; there is no global xn image and no second grid-wide
// hand-off. Every mbarrier wait is bounded; a wait that runs out records a
// deadline error, and the CTA waits for its own copies and MMAs in flight,
// frees its TMEM and returns.
#pragma once

#include "gdn_kernels.h"
#include "gdn_outproj.cuh"
#include "gdn_phases.cuh"
#include "gdn_recurrence_staged.cuh"
#include "gdn_tc_ptx.cuh"

namespace gdn {

namespace {
constexpr int kMaxStages = 6;                           // weight tiles in flight per CTA (the plan picks)
constexpr int kFirstTiles = 4;                          // of them issued before the norm hand-off
constexpr uint32_t kWBytes = kTileM * kKStep * 2;       // 32 KB weight tile (B operand)
constexpr uint32_t kXBytes = kMaxRows * kKStep * 2;     // 2 KB normed-input slice (A rows 0..15)
constexpr uint32_t kXPadMin = (64 - kMaxRows) * 128;    // 6 KB an M = 64 MMA reads past the last slice
constexpr uint32_t kWinBytes = kKStep * 2;              // input-norm weights of one k-step
constexpr uint32_t kTmemCols = 2 * kTileM;              // two 256-column f32 accumulators
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(64, kTileM);
static_assert(kMaxBSlots <= 32, "one owner bit per window slot");
// Bytes of one row of a unit's code tile (64 codes: MXFP4 32, MXFP6 48) and
// of the tile (256 rows).
template <int FMT>
__host__ __device__ constexpr uint32_t code_row_bytes() { return FMT == kFmtMxfp6 ? 48u : 32u; }
template <int FMT>
__host__ __device__ constexpr uint32_t code_tile_bytes() { return kTileM * code_row_bytes<FMT>(); }
constexpr int kMaxRStages = 4;                          // code tiles in flight per CTA (MXFP4, MXFP6)
// Warps that decode MXFP4 / MXFP6 code tiles into bf16 tiles: thread i of them owns
// row i of the 256-row tile. Warp 0 holds the TMA producer, warp 1 the MMA
// issuer, warp 4 the drain (with bf16 weights, which have no decode, warps 4,
// 8 and 12). The decode is bound by the integer pipe of its warps' schedulers
// (warp w issues on scheduler w % 4), so its eight warps are two per scheduler:
// 8, 12 | 5, 9 | 2, 6 | 3, 7.
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
__device__ __forceinline__ int conv_index(int warp) {
  switch (warp) {
    case 8: return 0;
    case 12: return 1;
    case 5: return 2;
    case 9: return 3;
    case 2: return 4;
    case 6: return 5;
    case 3: return 6;
    case 7: return 7;
    default: return -1;
  }
}
constexpr uint32_t kWaitPipe = 4;                       // error-word id of a pipeline wait
constexpr unsigned long long kCleanupNs = 100000000ull; // bound of the waits on the abort path
}  // namespace

struct TcShared {
  uint64_t full[kMaxStages];   // bf16 weight tile landed (TMA complete_tx)
  uint64_t dfull[kMaxStages];  // coded weights: the stage's code tile decoded (one arrival per decode warp)
  uint64_t empty[kMaxStages];  // MMAs of the stage done (tcgen05.commit)
  uint64_t rfull[kMaxRStages];   // code tile landed (TMA complete_tx)
  uint64_t rempty[kMaxRStages];  // code tile read by every decode warp
  uint64_t acc_full[2];     // accumulator ready for the drain
  uint64_t acc_empty[2];    // accumulator drained
  uint64_t mma_done;        // every MMA issued by the CTA done
  uint64_t obar[kOpMaxStages];  // out_proj: a stage's weight rows landed
  uint64_t sbar[3];             // recurrence: a state tile landed (one per buffer)
  unsigned char seg_slot[kMaxSegs];  // the CTA's plan entries read late (drain, MMA), copied at kernel start
  unsigned short ks_first;
  uint32_t tmem_base;
  int abort;
  int dec_issued;  // coded formats: units [0, dec_issued) passed by the decode warps (bf16 tiles issued)
};

// Walks a CTA's units in plan order without divisions: unit u is k-step
// kb * kblock + k of tile t, in group g = kb * num_tiles + t.
struct UnitIter {
  int k, t, kb, ks;
  int KB, T;
  __device__ __forceinline__ UnitIter(const StepParams& p, int u) : KB(p.kblock), T(p.num_tiles) {
    const int g = u / KB;
    k = u - g * KB;
    kb = g / T;
    t = g - kb * T;
    ks = kb * KB + k;
  }
  __device__ __forceinline__ bool group_end() const { return k + 1 == KB; }
  __device__ __forceinline__ void next() {
    ++k;
    ++ks;
    if (k == KB) {
      k = 0;
      if (++t == T) {
        t = 0;
        ++kb;
      }
      ks = kb * KB;
    }
  }
};

// Bounded wait for the phase of `bar` with this parity. Gives up when the
// CTA's abort flag is set, or at the deadline (then records the error and
// sets the flag).
static __device__ __forceinline__ bool pipe_wait(const StepParams& p, TcShared& ts, uint64_t* bar,
                                                 uint32_t parity) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ts.abort)) return false;
    if ((it & 63) == 0 && globaltimer_ns() - t0 > p.deadline_ns) {
      record_error(p.ctr, kStatusDeadline, kWaitPipe, blockIdx.x);
      *reinterpret_cast<volatile int*>(&ts.abort) = 1;
      return false;
    }
  }
}

// The same for a whole warp: every lane waits, and the warp goes on only if
// every lane saw the phase (so its lanes never part ways).
static __device__ __forceinline__ bool pipe_wait_warp(const StepParams& p, TcShared& ts, uint64_t* bar,
                                                      uint32_t parity) {
  return __all_sync(0xffffffffu, pipe_wait(p, ts, bar, parity));
}

// Wait (bounded, ignoring the abort flag) on the abort path.
static __device__ void cleanup_wait(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0; !tc::mbar_try_wait(bar, parity); ++it)
    if ((it & 63) == 0 && globaltimer_ns() - t0 > kCleanupNs) return;
}

__device__ __forceinline__ const CUtensorMap* weight_map(const StepParams& p, int t, int& row0) {
  if (t < p.tiles_qkvz) {
    row0 = t * kTileM;
    return &p.tm_qkvz;
  }
  row0 = (t - p.tiles_qkvz) * kTileM;
  return &p.tm_ba;
}

// A unit whose weights are MXFP4 or MXFP6 codes (decoded to bf16 in shared
// memory before the MMA); the others are bf16 tiles the MMA reads as loaded.
template <int FMT>
__device__ __forceinline__ bool unit_coded(const StepParams& p, const UnitIter& it) {
  return !bf16_weights<FMT>() && it.t < p.tiles_qkvz;
}

// Ring positions along a CTA's units: every unit takes the next bf16 stage
// (s, phase ph); a coded unit also the next code stage (r, phase rph).
struct RingPos {
  int s = 0, r = 0;
  uint32_t ph = 0, rph = 0;
  __device__ __forceinline__ void advance(const StepParams& p, bool coded) {
    if (++s == p.stages) { s = 0; ph ^= 1; }
    if (coded && ++r == p.rstages) { r = 0; rph ^= 1; }
  }
};

// Unit n's weights: codes into code stage pos.r, else a bf16 tile into
// stage pos.s (the caller has made sure the stage is free).
template <int FMT>
__device__ __forceinline__ void issue_unit(const StepParams& p, TcShared& ts, uint8_t* sW, uint8_t* sR,
                                           const UnitIter& it, int n, const RingPos& pos, uint64_t pol) {
  int row0;
  const CUtensorMap* m = weight_map(p, it.t, row0);
  if (unit_coded<FMT>(p, it)) {
    tc::mbar_arrive_expect_tx(&ts.rfull[pos.r], code_tile_bytes<FMT>());
    tc::tma_load_2d(sR + (size_t)pos.r * code_tile_bytes<FMT>(), m, it.ks * (int)code_row_bytes<FMT>(), row0,
                    &ts.rfull[pos.r], pol);
  } else {
    tc::mbar_arrive_expect_tx(&ts.full[pos.s], kWBytes);
    tc::tma_load_2d(sW + (size_t)pos.s * kWBytes, m, it.ks * kKStep, row0, &ts.full[pos.s], pol);
  }
  if (n < 16) tl_stamp_here(p, TL_UNIT_ISSUED + n);
}

// Ring positions after the CTA's first n units.
template <int FMT>
__device__ __forceinline__ RingPos ring_pos_at(const StepParams& p, int ub, int n) {
  RingPos pos;
  UnitIter it(p, ub);
  for (int j = 0; j < n; ++j, it.next()) pos.advance(p, unit_coded<FMT>(p, it));
  return pos;
}

// The CTA's leading units that fit the rings before any stage is reused (at
// most `cap`): the ones issued without waiting.
template <int FMT>
__device__ __forceinline__ int prefill_units(const StepParams& p, int ub, int nunits, int cap) {
  UnitIter it(p, ub);
  int coded = 0, n = 0;
  for (; n < min(nunits, cap); ++n, it.next()) {
    if (unit_coded<FMT>(p, it)) {
      if (coded == p.rstages) break;
      ++coded;
    } else if (n >= p.stages) {
      break;
    }
  }
  return n;
}

// Units [from, to) of the CTA's weight stream, all within the prefill (one
// thread, no waits).
template <int FMT>
static __device__ __forceinline__ void start_weight_stream(const StepParams& p, TcShared& ts, uint8_t* sW,
                                                           uint8_t* sR, int ub, int from, int to) {
  if (from >= to) return;
  const uint64_t pol0 = tc::policy_evict_first();
  RingPos pos = ring_pos_at<FMT>(p, ub, from);
  UnitIter it(p, ub + from);
  for (int n = from; n < to; ++n, it.next()) {
    issue_unit<FMT>(p, ts, sW, sR, it, n, pos, pol0);
    pos.advance(p, unit_coded<FMT>(p, it));
  }
  if (from == 0) tl_stamp_here(p, TL_ISSUED);
}

// The A operand of this CTA: the normed input xn of its k-steps as slices in
// shared memory. Slot j holds k-step (ks_first + j) mod ksteps, 16 rows x 64
// columns bf16 in the 128-byte swizzled K-major layout (row r at r * 128
// bytes, its 16-byte chunk c at position c ^ (r % 8)); rows past the step's
// rows are 0. Built in two passes around the norm hand-off:
//   stage_residual_slices: r = bf16(x + residual) of the window; for the
//     k-steps this CTA owns, the sums of r^2 of 8 columns into `sq`
//     ([row][slot * 8 + chunk]); write_residual_out stores them later
//   finish_normed_slices: xn = bf16(r * rstd * (1 + w)) in place.
// One pass over x and the residual serves the residual add, the norm
// partials and the MMA operand (vLLM #60833, Details, "x without an LDS
// tile": each consumer builds the part of x it reads; the sums of squares
// are handed between CTAs).
// `after_issue` runs once every thread has issued the loads of the first
// batch (before any of them is used), so what it starts queues behind them.
template <bool HAS_RES, typename F>
static __device__ __forceinline__ void stage_residual_slices(const StepParams& p, uint8_t* sX, uint8_t* sWin,
                                                            float* sq, F after_issue) {
  const int cta = blockIdx.x, W = p.rows;
  const int nb = p.plan->nb_slots[cta], ks0 = p.plan->ks_first[cta];
  const unsigned own = p.plan->own_mask[cta];
  const int ntask = nb * kMaxRows * 8;  // (slot, row, 16-byte chunk)
  constexpr int B = 4;                  // tasks per thread in flight
  for (int b0 = 0; b0 == 0 || b0 < ntask; b0 += kThreads * B) {  // the first batch runs even if empty
    const int i0 = b0 + threadIdx.x;
    uint4 xv[B], qv[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int i = i0 + k * kThreads;
      const int j = i >> 7, w = (i >> 3) & (kMaxRows - 1), c = i & 7;
      if (i < ntask && w < W) {
        const size_t col = (size_t)((ks0 + j) % p.ksteps) * kKStep + c * 8;
        xv[k] = ld_stream_v4(p.x + (size_t)w * p.H + col);
        qv[k] = HAS_RES ? ld_stream_v4(p.res + (size_t)w * p.H + col) : xv[k];
      }
    }
    if (b0 == 0) {
      __syncthreads();
      after_issue();
    }
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int i = i0 + k * kThreads;
      const int j = i >> 7, w = (i >> 3) & (kMaxRows - 1), c = i & 7;
      if (i < ntask) {
        uint4 r = make_uint4(0, 0, 0, 0);
        if (w < W) {
          r = residual8<HAS_RES>(xv[k], qv[k]);
          if ((own >> j) & 1u) {
            const uint32_t rs[4] = {r.x, r.y, r.z, r.w};
            float s2 = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = bf16_lo(rs[e]), hi = bf16_hi(rs[e]);
              s2 = fmaf(lo, lo, s2);
              s2 = fmaf(hi, hi, s2);
            }
            sq[w * (p.xslots * 8) + j * 8 + c] = s2;
          }
        }
        *reinterpret_cast<uint4*>(sX + (size_t)j * kXBytes + w * 128 + ((c ^ (w & 7)) << 4)) = r;
      }
    }
  }
}

// The input-norm weights of the window, one 16-byte chunk per thread (at
// most 32 k-steps x 8 chunks <= 512 threads). A weight no step writes: the
// load goes out before the previous step is done, the value is stored to
// shared memory once the x and residual loads are out, off the norm path.
static_assert(kMaxBSlots * 8 <= kThreads, "one norm-weight chunk per thread");
static __device__ __forceinline__ uint4 load_norm_weights(const StepParams& p) {
  const int cta = blockIdx.x, i = threadIdx.x;
  const int nb = p.plan->nb_slots[cta], ks0 = p.plan->ks_first[cta];
  if (i >= nb * 8) return make_uint4(0, 0, 0, 0);
  return ld_stream_v4(p.w_in + (size_t)((ks0 + (i >> 3)) % p.ksteps) * kKStep + (i & 7) * 8);
}
static __device__ __forceinline__ void store_norm_weights(const StepParams& p, uint8_t* sWin, uint4 v) {
  const int i = threadIdx.x;
  if (i < p.plan->nb_slots[blockIdx.x] * 8) reinterpret_cast<uint4*>(sWin + (size_t)(i >> 3) * kWinBytes)[i & 7] = v;
}

// residual_out of the owned k-steps, from the staged r (after the norm
// partials are out: these stores need not be visible to other CTAs, so they
// stay out of the release fence).
static __device__ __forceinline__ void write_residual_out(const StepParams& p, const uint8_t* sX) {
  const int cta = blockIdx.x, W = p.rows;
  const int nb = p.plan->nb_slots[cta], ks0 = p.plan->ks_first[cta];
  const unsigned own = p.plan->own_mask[cta];
  for (int i = threadIdx.x; i < nb * W * 8; i += kThreads) {
    const int j = i / (W * 8), rem = i - j * (W * 8), w = rem >> 3, c = rem & 7;
    if ((own >> j) & 1u) {
      const size_t col = (size_t)((ks0 + j) % p.ksteps) * kKStep + c * 8;
      *reinterpret_cast<uint4*>(p.res_out + (size_t)w * p.H + col) =
          *reinterpret_cast<const uint4*>(sX + (size_t)j * kXBytes + w * 128 + ((c ^ (w & 7)) << 4));
    }
  }
}

// Each row's sum of r^2 over the owned k-steps (slot-major, a fixed order),
// published to every CTA as a tagged word: no fence, no release (the launch
// number L was read at kernel entry). The norm counter only counts launches.
static __device__ __forceinline__ void publish_norm_partials(const StepParams& p, const float* sq, int L) {
  const int cta = blockIdx.x, W = p.rows, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int nb = p.plan->nb_slots[cta];
  const unsigned own = p.plan->own_mask[cta];
  const bool publish = !((p.debug_flags & kDebugSkipNormPublish) && cta == 0);  // test hook: never publish
  __syncthreads();
  for (int w = warp; w < W; w += kWarps) {
    float s = 0.f;
    for (int e = lane; e < nb * 8; e += 32)
      if ((own >> (e >> 3)) & 1u) s += sq[w * (p.xslots * 8) + e];
    s = warp_sum(s);
    if (lane == 0 && publish) st_tagged(p.norm_part + w * p.num_ctas + cta, tagged(L, s));
  }
  if (tid == 0 && publish) red_add_relaxed_u64(&p.ctr->norm_arrive, 1ull);
  tl_stamp(p, TL_NORM_OUT);
}

// f32 2^e for e in [-127, 127] (exact; 2^-127 is subnormal).
static __device__ __forceinline__ float exp2_int(int e) {
  return e == -127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(e + 127) << 23);
}

// MXFP4 quantisation of one row's block of 32 normed inputs, 8 of them in
// this thread (the block's 4 chunks are 4 consecutive lanes): the block scale
// 2^E from the block maximum with its mantissa rounded half up to one bit,
// E = its exponent - 2 clamped to [-126, 127] (a normal scale, also for an
// all-zero block); each value |x| / 2^E rounded
// to the e2m1 grid {0, .5, 1, 1.5, 2, 3, 4, 6} (ties to even, saturating at
// 6), returned dequantised (exact in bf16). The dynamic MX quantiser of
// vLLM #60833 (review "How to make the MXFP6 weights", step 2) with E2M1's
// largest exponent, 2.
static __device__ __forceinline__ uint4 quantize8_mxfp4(uint4 xv) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
  float v[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = bf16_lo(xs[e]);
    v[2 * e + 1] = bf16_hi(xs[e]);
  }
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
  const unsigned mask = __activemask();
  m = fmaxf(m, __shfl_xor_sync(mask, m, 1));
  m = fmaxf(m, __shfl_xor_sync(mask, m, 2));
  int E = (int)(((__float_as_uint(m) + (1u << 21)) >> 23) & 0xffu) - 127 - 2;
  E = max(-126, min(127, E));
  const float inv = exp2_int(-E), scale = exp2_int(E);
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float q[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float a = fabsf(v[2 * e + h]) * inv;              // exact
      const float st = a < 2.f ? 0.5f : (a < 4.f ? 1.f : 2.f);  // grid spacing
      const float r = fminf(rintf(a / st) * st, 6.f);           // ties to even
      q[h] = copysignf(r, v[2 * e + h]) * scale;
    }
    o[e] = pack_bf16x2(q[0], q[1]);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// xn = bf16(r * rstd * (1 + w)) in place; with MXFP4 weights also its
// quantised copy in the second window sXq (same layout).
template <int FMT>
static __device__ __forceinline__ void finish_normed_slices(const StepParams& p, const SmemPhases& sm,
                                                            uint8_t* sX, uint8_t* sXq, const uint8_t* sWin) {
  const int cta = blockIdx.x, W = p.rows;
  const int ntask = p.plan->nb_slots[cta] * W * 8;  // (slot, row < W, chunk); a multiple of 8
  for (int i = threadIdx.x; i < ntask; i += kThreads) {
    const int j = i / (W * 8), rem = i - j * (W * 8), w = rem >> 3, c = rem & 7;
    const size_t off = (size_t)j * kXBytes + w * 128 + ((c ^ (w & 7)) << 4);
    uint4* d = reinterpret_cast<uint4*>(sX + off);
    const uint4 xv = normed8(*d, reinterpret_cast<const uint4*>(sWin + (size_t)j * kWinBytes)[c], sm.rstd[w]);
    *d = xv;
    if (FMT == kFmtMxfp4) *reinterpret_cast<uint4*>(sXq + off) = quantize8_mxfp4(xv);
  }
}

// TMA producer (one whole warp; lane 0 issues): units `issued`.. into the
// rings, each into a stage that has been released (a bf16 stage by the MMAs,
// a code stage by the decode). With coded weights it issues the code tiles
// only: the bf16 tiles of the other units (in_proj_ba) go out from the decode
// warps, which wait for every phase of every bf16 stage in unit order. A
// waiter that skipped some phases of a stage could take an older phase's
// parity for the one it waits for. Returns the number of units passed. (An L2 prefetch ahead of the ring was
// measured: the tensor form does not bring tiles in early, and per-row
// prefetches delay the latency-bound norm hand-off more than they shorten
// the projection.)
template <int FMT>
static __device__ __forceinline__ int producer_loop(const StepParams& p, TcShared& ts, uint8_t* sW, uint8_t* sR,
                                                   int ub, int nunits, int issued, uint64_t pol) {
  const bool leader = (threadIdx.x & 31) == 0;
  UnitIter it(p, ub + issued);
  RingPos pos = ring_pos_at<FMT>(p, ub, issued);
  for (int n = issued; n < nunits; ++n) {
    const bool coded = unit_coded<FMT>(p, it);
    if (coded) {
      if (!pipe_wait_warp(p, ts, &ts.rempty[pos.r], pos.rph ^ 1)) return n;
    } else if (bf16_weights<FMT>()) {
      if (!pipe_wait_warp(p, ts, &ts.empty[pos.s], pos.ph ^ 1)) return n;
    }
    if (leader && (coded || bf16_weights<FMT>())) issue_unit<FMT>(p, ts, sW, sR, it, n, pos, pol);
    __syncwarp();
    pos.advance(p, coded);
    it.next();
  }
  return nunits;
}

// Code decode (kConvThreads threads, thread i owns row i of the tile): per
// coded unit, each warp on its own waits for the code tile and for its bf16
// stage to be free, turns its rows' 64 codes (MXFP4 e2m1 or MXFP6 e2m3) and
// their two e8m0 block scales into bf16 (code value x 2^(scale - 127), exact
// in bf16) in the 128-byte swizzled K-major layout the MMA reads, then
// arrives on the code stage's release and on the stage's `dfull` (both count
// one arrival per warp): no barrier among the warps per unit. A row's scales
// for 8 k-steps are one aligned 16-byte load, issued a block ahead.
// 2^(e - 127) of an e8m0 byte as bf16x2 (both halves): bf16 exponent field
// e; e = 0 is 2^-127, the bf16 subnormal 0x0040.
static __device__ __forceinline__ uint32_t e8m0_bf16x2(uint32_t e) {
  const uint32_t h = e == 0 ? 0x0040u : (e << 7);
  return h | (h << 16);
}
static __device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// bf16x2 product, round to nearest even (exact here: a power of two times a
// value with a 2-bit significand).
static __device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Eight e2m1 codes (one 32-bit word, element i in nibble i: sign bit 3,
// exponent bits 2..1 with bias 1, mantissa bit 0) to their bf16 values as
// four bf16x2 words, element 2j in the low half of word j. The magnitudes
// {0, .5, 1, 1.5, 2, 3, 4, 6} have the bf16 patterns 0x0000, 0x3F00, 0x3F80,
// 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0: their high and low bytes are two
// 8-entry byte tables, looked up four codes at a time with PRMT (the code's
// low 3 bits select a byte); the sign bits are shifted into bit 15 / 31.
// The signs: code 2j's sign bit is the top bit of byte j of (w << 4), code
// 2j + 1's the top bit of byte j of w; a PRMT selector nibble with bit 3 set
// replicates the top bit of the byte it selects, which puts them at bits 15
// and 31 (masked in with one logic op).
static __device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, uint32_t (&o)[4]) {
  constexpr uint32_t kHiLo = 0x3F3F3F00u, kHiHi = 0x40404040u;  // high bytes of magnitudes 0..3, 4..7
  constexpr uint32_t kLoLo = 0xC0800000u, kLoHi = 0xC0804000u;  // low bytes
  const uint32_t m = w & 0x77777777u, m2 = m >> 16;
  const uint32_t h0 = prmt(kHiLo, kHiHi, m), l0 = prmt(kLoLo, kLoHi, m);
  const uint32_t h1 = prmt(kHiLo, kHiHi, m2), l1 = prmt(kLoLo, kLoHi, m2);
  const uint32_t ev = w << 4;  // even codes' signs at the bytes' top bits (odd codes': w itself)
  constexpr uint32_t kSignMask = 0x80008000u;
  o[0] = prmt(l0, h0, 0x5140u) | (prmt(ev, w, 0xC080u) & kSignMask);
  o[1] = prmt(l0, h0, 0x7362u) | (prmt(ev, w, 0xD090u) & kSignMask);
  o[2] = prmt(l1, h1, 0x5140u) | (prmt(ev, w, 0xE0A0u) & kSignMask);
  o[3] = prmt(l1, h1, 0x7362u) | (prmt(ev, w, 0xF0B0u) & kSignMask);
}
// Two e2m3 codes (6 bits: sign bit 5, exponent bits 4..3 with bias 1,
// mantissa bits 2..0) to a bf16x2 word, c0 in the low half. With exponent
// field e >= 1 the value (1 + m/8) 2^(e-1) has the bf16 pattern
// 0x3F00 + ((code & 31) << 4); with e = 0 it is m/8, whose eight bf16
// patterns (0, 0x3E00, 0x3E80, 0x3EC0, 0x3F00, 0x3F20, 0x3F40, 0x3F60) are
// looked up bytewise with PRMT; the sign goes to bit 15 / 31.
static __device__ __forceinline__ uint32_t e2m3x2_to_bf16(uint32_t c0, uint32_t c1) {
  uint32_t v = (((c0 & 31u) << 4) | ((c1 & 31u) << 20)) + 0x3F003F00u;
  const uint32_t sel = (c0 & 7u) | ((c1 & 7u) << 4);
  const uint32_t hi = prmt(0x3E3E3E00u, 0x3F3F3F3Fu, sel), lo = prmt(0xC0800000u, 0x60402000u, sel);
  const uint32_t sub = prmt(lo, hi, 0x5140u);
  const uint32_t mask = ((c0 & 24u) ? 0u : 0xFFFFu) | ((c1 & 24u) ? 0u : 0xFFFF0000u);
  v = (v & ~mask) | (sub & mask);
  return v | ((c0 & 32u) << 10) | ((c1 & 32u) << 26);
}

// One row's 64 MXFP6 codes (48 bytes: two 24-byte groups of 32 codes, code i
// of a group at bits 6i..6i+5 little-endian, so code j of the row starts at
// bit 6j) to eight 16-byte chunks of bf16 (chunk c: columns 8c..8c+7),
// scaled by the groups' e8m0 scales, through a table of all 4096 code pairs
// (entry c0 | c1 << 6 holds e2m3x2_to_bf16(c0, c1), built once per launch in
// shared memory): per pair a funnel shift, a mask, a table load and the
// scale. The table's loads are bank-conflicted at random, but they cost the
// integer pipe, which bounds the decode, far less than the conversion.
constexpr uint32_t kE2m3LutEntries = 4096;
static __device__ __forceinline__ void decode_row_mxfp6_lut(const uint8_t* src, const uint32_t (&sc)[2],
                                                            uint8_t* dst, int swz, const uint32_t* lut) {
  const uint4 q0 = reinterpret_cast<const uint4*>(src)[0], q1 = reinterpret_cast<const uint4*>(src)[1],
              q2 = reinterpret_cast<const uint4*>(src)[2];
  const uint32_t w[13] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w, q2.x, q2.y, q2.z, q2.w, 0u};
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // chunk c: code pairs 4c..4c+3, the 12-bit field of pair j at bit 12j
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int b = 48 * c + 12 * e;
      const uint32_t idx = __funnelshift_r(w[b >> 5], w[(b >> 5) + 1], b & 31) & (kE2m3LutEntries - 1);
      o[e] = mul_bf16x2(lut[idx], sc[c >> 2]);
    }
    *reinterpret_cast<uint4*>(dst + ((c ^ swz) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// One row's e8m0 scales of the 8-k-step block of unit `it` (16 bytes).
static __device__ __forceinline__ uint4 scale_block(const StepParams& p, const UnitIter& it, int row) {
  const int grow = (it.t * kTileM) + row;  // coded units are in_proj_qkvz rows
  return ld_stream_v4(p.w_qkvz_scales + (size_t)grow * (p.H / 32) + (it.ks >> 3) * 16);
}
template <int FMT>
static __device__ __forceinline__ void decode_loop(const StepParams& p, TcShared& ts, uint8_t* sW,
                                                   const uint8_t* sR, int ub, int nunits, int prefill, int ci,
                                                   const uint32_t* lut) {
  UnitIter it(p, ub);
  RingPos pos;
  const uint64_t pol = tc::policy_evict_first();
  int blk_t = -1, blk_k = -1;  // the 8-k-step scale block held in `cur`
  uint4 cur = make_uint4(0, 0, 0, 0), nxt = make_uint4(0, 0, 0, 0);
  int nxt_t = -1, nxt_k = -1;
  // the first coded unit's block
  {
    UnitIter f(p, ub);
    for (int n = 0; n < nunits; ++n, f.next())
      if (unit_coded<FMT>(p, f)) {
        nxt = scale_block(p, f, ci);
        nxt_t = f.t;
        nxt_k = f.ks >> 3;
        break;
      }
  }
  // A warp whose wait ran out (the abort flag is then set, and every later
  // wait returns at once) goes on walking the units without work, so that it
  // still meets the other decode warps at every barrier below.
  bool live = true;
  for (int n = 0; n < nunits; ++n) {
    const bool coded = unit_coded<FMT>(p, it);
    if (!coded) {
      // a bf16 tile (the prefill has issued the first ones). A stage's first
      // use has no wait: the MMA may already have taken a prefilled tile.
      // Later, every decode warp waits for the stage's release and the tile
      // goes out only once all of them have: were it to need one warp alone,
      // it could be multiplied and the stage released again before a slower
      // warp had waited for the release before (that warp would then wait
      // for a phase two generations on).
      if (n >= p.stages) {
        live = live && pipe_wait_warp(p, ts, &ts.empty[pos.s], pos.ph ^ 1);
        asm volatile("barrier.sync 2, %0;" ::"n"(kConvThreads) : "memory");
      }
      if (live && ci == 0) {
        if (n >= prefill) issue_unit<FMT>(p, ts, sW, nullptr, it, n, pos, pol);
        *reinterpret_cast<volatile int*>(&ts.dec_issued) = n + 1;
      }
    }
    if (coded && live) {
      if (it.t != blk_t || (it.ks >> 3) != blk_k) {
        // this unit starts a new scale block: take the prefetched one, prefetch the next
        cur = nxt;
        blk_t = nxt_t;
        blk_k = nxt_k;
        UnitIter f = it;
        for (int j = n + 1; j < nunits; ++j) {
          f.next();
          if (unit_coded<FMT>(p, f) && (f.t != blk_t || (f.ks >> 3) != blk_k)) {
            nxt = scale_block(p, f, ci);
            nxt_t = f.t;
            nxt_k = f.ks >> 3;
            break;
          }
        }
      }
      // each warp on its own: it waits for every phase in order, and every
      // barrier it waits on needs all eight decode warps to advance
      live = pipe_wait_warp(p, ts, &ts.rfull[pos.r], pos.rph) && pipe_wait_warp(p, ts, &ts.empty[pos.s], pos.ph ^ 1);
    }
    if (coded && live) {
      const uint8_t* row = sR + (size_t)pos.r * code_tile_bytes<FMT>() + ci * code_row_bytes<FMT>();
      const int kk = it.ks & 7;  // k-step within the block: scale bytes 2kk, 2kk + 1
      const uint32_t sw4 = (kk >> 1) == 0 ? cur.x : (kk >> 1) == 1 ? cur.y : (kk >> 1) == 2 ? cur.z : cur.w;
      const uint32_t sword = sw4 >> ((kk & 1) * 16);
      const uint32_t sc[2] = {e8m0_bf16x2(sword & 0xffu), e8m0_bf16x2((sword >> 8) & 0xffu)};
      uint8_t* dst = sW + (size_t)pos.s * kWBytes + ci * 128;
      if (FMT == kFmtMxfp6) {
        decode_row_mxfp6_lut(row, sc, dst, ci & 7, lut);
      } else {
        const uint4 c0 = reinterpret_cast<const uint4*>(row)[0], c1 = reinterpret_cast<const uint4*>(row)[1];
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 8 columns per 16-byte chunk, from one 32-bit word of codes
          uint32_t o[4];
          e2m1x8_to_bf16(words[c], o);
          const uint32_t scale = sc[c >> 2];
#pragma unroll
          for (int e = 0; e < 4; ++e) o[e] = mul_bf16x2(o[e], scale);  // exact in bf16
          *reinterpret_cast<uint4*>(dst + ((c ^ (ci & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      tc::fence_proxy_async_smem();  // the generic-proxy writes, visible to the MMA
      __syncwarp();
      if ((ci & 31) == 0) {  // this warp's rows: code read, bf16 written
        tc::mbar_arrive(&ts.rempty[pos.r]);
        tc::mbar_arrive(&ts.dfull[pos.s]);
      }
    }
    pos.advance(p, coded);
    it.next();
  }
}

// MMA issuer (one whole warp; lane 0 issues): per unit, 4 MMAs of K = 16 over
// the stage's 64 columns into the segment's accumulator; a segment (the units
// of one group) starts by overwriting. Commits release the stage and, at a
// segment's end, hand the accumulator to the drain.
template <int FMT>
static __device__ __forceinline__ void mma_loop(const StepParams& p, TcShared& ts, uint8_t* sW,
                                                uint8_t* sX, uint8_t* sXq, int ub, int nunits, uint32_t tmem) {
  // Stage and phase advance incrementally: a division per unit by the
  // runtime ring depth costs the loop more than the tensor core's own time.
  const int ks0 = ts.ks_first, KS = p.ksteps, S = p.stages;
  UnitIter it(p, ub);
  int seg = -1;
  bool seg_open = false;
  int s = 0;
  // per stage, the phase parity of its two fill barriers: `full` (a TMA fill)
  // and, with coded weights, `dfull` (a decoded tile); each is waited for at
  // every one of its phases, in order
  uint32_t phu = 0, phc = 0;
  const uint32_t sw0 = tc::smem_u32(sW), sx0 = tc::smem_u32(sX), sxq0 = tc::smem_u32(sXq);
  const bool leader = (threadIdx.x & 31) == 0;
  bool landed = false;  // unit n's tile seen complete while unit n - 1 was issued
  for (int n = 0; n < nunits; ++n) {
    const bool first = !seg_open;
    if (first) {
      ++seg;
      seg_open = true;
      if (!pipe_wait_warp(p, ts, &ts.acc_empty[seg & 1], ((seg >> 1) & 1) ^ 1)) break;
      tc::tc_fence_after();  // these MMAs come after the drain's tcgen05.ld of this accumulator
    }
    // The phase makes the stage's TMA bytes (or the decode's writes, fenced
    // to the async proxy) visible to the MMA: no tcgen05 fence per unit.
    const bool cd = unit_coded<FMT>(p, it);
    uint64_t* fb = cd ? &ts.dfull[s] : &ts.full[s];
    const uint32_t par = ((cd ? phc : phu) >> s) & 1u;
    if (!landed && !__all_sync(0xffffffffu, tc::mbar_try_wait(fb, par) || pipe_wait(p, ts, fb, par))) break;
    // The next unit's stage, tested now: an mbarrier test takes ~200 cycles,
    // which then pass under this unit's MMA issue instead of idling the
    // tensor core between units.
    int s1 = s + 1;
    if (s1 == S) s1 = 0;
    bool landed1 = false;
    if (n + 1 < nunits) {
      UnitIter nx = it;
      nx.next();
      const bool cd1 = unit_coded<FMT>(p, nx);
      landed1 = tc::mbar_test(cd1 ? &ts.dfull[s1] : &ts.full[s1], ((cd1 ? phc : phu) >> s1) & 1u);
    }
    int slot = it.ks - ks0;
    if (slot < 0) slot += KS;
    if (n == 0 && leader) tl_stamp_here(p, TL_MMA_FIRST);
    // MXFP4 in_proj_qkvz: the quantised inputs (W4A4); bf16 or MXFP6 weights: xn itself
    const uint64_t ad = tc::sdesc_k_sw128(((FMT == kFmtMxfp4 && unit_coded<FMT>(p, it)) ? sxq0 : sx0) +
                                          (uint32_t)slot * kXBytes);
    const uint64_t bd = tc::sdesc_k_sw128(sw0 + (uint32_t)s * kWBytes);
    const uint32_t d = tmem + (uint32_t)(seg & 1) * kTileM;
    const bool seg_end = n + 1 == nunits || it.group_end();
    if (leader) {
#pragma unroll
      for (int k = 0; k < kKStep / 16; ++k)
        tc::mma_bf16(d, ad + 2 * k, bd + 2 * k, kIdesc, (first && k == 0) ? 0u : 1u);
      tc::mma_commit(&ts.empty[s]);
      if (seg_end) tc::mma_commit(&ts.acc_full[seg & 1]);
    }
    landed = __all_sync(0xffffffffu, landed1);
    if (seg_end) seg_open = false;
    if (cd)
      phc ^= 1u << s;
    else
      phu ^= 1u << s;
    it.next();
    s = s1;
  }
  if (leader) tc::mma_commit(&ts.mma_done);
  __syncwarp();
  cleanup_wait(&ts.mma_done, 0);
  if (leader) tl_stamp_here(p, TL_MMA_LAST);
}

// Drain (warp 4 with coded weights, warps 4, 8 and 12 with bf16 weights; all
// in TMEM sub-partition 0, so lane w reads row w of the step): per segment,
// the warps split the accumulator's 8 chunks of 32 columns (weight rows) and
// write the CTA's partial of the tile as tagged words; then the accumulator
// is released.
template <int kDrainWarps>
static __device__ __forceinline__ void drain_loop(const StepParams& p, TcShared& ts, int ub, int nunits,
                                                  uint32_t tmem, int gtid, int L) {
  constexpr int kDrainThreads = 32 * kDrainWarps;
  const int W = p.rows, lane = gtid & 31, dw = gtid >> 5;
  UnitIter it(p, ub);
  int seg = 0;
  for (int n = 0; n < nunits; ++seg) {
    const int t = it.t;
    while (n < nunits) {  // to the end of this segment's group
      const bool end = it.group_end();
      it.next();
      ++n;
      if (end) break;
    }
    const int b = seg & 1;
    bool ok = true;
    if (lane == 0) ok = pipe_wait(p, ts, &ts.acc_full[b], (seg >> 1) & 1);
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    tc::tc_fence_after();
    unsigned long long* dst = p.proj_part +
                              ((size_t)t * p.max_contrib + ts.seg_slot[seg]) * kMaxRows * kTileM +
                              (size_t)lane * kTileM;
#pragma unroll 1
    for (int c = dw; c < kTileM / 32; c += kDrainWarps) {
      float v[32];
      tc::tmem_ld32(tmem + (uint32_t)b * kTileM + c * 32, v);
      if (lane < W) {  // the partial as tagged words: readers poll them directly
#pragma unroll
        for (int q = 0; q < 16; ++q)
          st_tagged2(dst + c * 32 + 2 * q, tagged(L, v[2 * q]), tagged(L, v[2 * q + 1]));
      }
    }
    tc::tc_fence_before();
    group_sync<kDrainThreads>();
    if (gtid == 0) tc::mbar_arrive(&ts.acc_empty[b]);
  }
}

// CUDA-core engine: the projection's dot products on the CUDA cores, from the
// same weight ring and normed-input window the MMA reads. kFmaWarps warps;
// thread i owns row i of each 256-row tile: per unit it adds its row's 64
// bf16 weights times each of the step's rows of xn (f32 FMA) to that row's
// two sums (even and odd 8-column chunks, in column order: two chains in
// flight), the rows one by one below 4 rows, else four at a time; at the end
// of a group (or of its units) it stores the two sums' total as the CTA's
// partial of the tile, in the slot and tagged layout the drain writes. A warp
// releases a stage once its rows are read (the stage's `empty` counts one
// arrival per warp).
// One 8-column chunk c of a thread's weight row, as f32, and its dot product
// with a chunk of xn added to a running sum (in column order).
struct FmaChunk {
  float w[8];
  __device__ __forceinline__ FmaChunk(const uint8_t* wr, int c, int rsw) {
    const uint4 v = *reinterpret_cast<const uint4*>(wr + ((c ^ rsw) << 4));
    w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z); w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
  }
  __device__ __forceinline__ float dot8(float a, const uint4& x) const {
    a = fmaf(w[0], bf16_lo(x.x), a);
    a = fmaf(w[1], bf16_hi(x.x), a);
    a = fmaf(w[2], bf16_lo(x.y), a);
    a = fmaf(w[3], bf16_hi(x.y), a);
    a = fmaf(w[4], bf16_lo(x.z), a);
    a = fmaf(w[5], bf16_hi(x.z), a);
    a = fmaf(w[6], bf16_lo(x.w), a);
    return fmaf(w[7], bf16_hi(x.w), a);
  }
};
// Row w's chunk c of the window's k-step slice (a broadcast: every thread
// reads the same bytes).
__device__ __forceinline__ uint4 fma_xrow(const uint8_t* xk, int c, int w) {
  return *reinterpret_cast<const uint4*>(xk + w * 128 + ((c ^ (w & 7)) << 4));
}
constexpr int kFmaWarps = 8;
static_assert(kFmaWarps * 32 == kTileM, "one weight row per thread");
static __device__ __forceinline__ void fma_loop(const StepParams& p, TcShared& ts, const uint8_t* sW,
                                                const uint8_t* sX, int ub, int nunits, int row, int L) {
  const int W = p.rows, KS = p.ksteps, S = p.stages, ks0 = ts.ks_first;
  const int rsw = row & 7;  // the row's 16-byte chunk c sits at position c ^ (row % 8)
  UnitIter it(p, ub);
  int s = 0, seg = 0;
  uint32_t ph = 0;  // per stage, the parity of its next `full` phase
  float acc[kMaxRows][2];
#pragma unroll
  for (int w = 0; w < kMaxRows; ++w) acc[w][0] = acc[w][1] = 0.f;
  for (int n = 0; n < nunits; ++n) {
    if (!pipe_wait_warp(p, ts, &ts.full[s], (ph >> s) & 1u)) return;
    int slot = it.ks - ks0;
    if (slot < 0) slot += KS;
    const uint8_t* wr = sW + (size_t)s * kWBytes + (size_t)row * 128;
    const uint8_t* xk = sX + (size_t)slot * kXBytes;
    // (the two loops differ only in how rows are grouped; a row's sums take
    // the same products in the same order in both)
    if (W < 4) {
#pragma unroll
      for (int c = 0; c < kKStep / 8; ++c) {
        const FmaChunk k(wr, c, rsw);
        uint4 xv[3];  // the rows' loads in flight together
#pragma unroll
        for (int w = 0; w < 3; ++w) xv[w] = w < W ? fma_xrow(xk, c, w) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int w = 0; w < 3; ++w) {
          if (w >= W) break;
          acc[w][c & 1] = k.dot8(acc[w][c & 1], xv[w]);
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < kKStep / 8; ++c) {
        const FmaChunk k(wr, c, rsw);
#pragma unroll
        for (int wb = 0; wb < kMaxRows; wb += 4) {  // rows past W are zero in the window
          if (wb >= W) break;
          uint4 xv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) xv[j] = fma_xrow(xk, c, wb + j);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[wb + j][c & 1] = k.dot8(acc[wb + j][c & 1], xv[j]);
        }
      }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&ts.empty[s]);
    if (n + 1 == nunits || it.group_end()) {
      unsigned long long* dst =
          p.proj_part + ((size_t)it.t * p.max_contrib + ts.seg_slot[seg]) * kMaxRows * kTileM + row;
#pragma unroll
      for (int w = 0; w < kMaxRows; ++w) {
        if (w < W) st_tagged(dst + (size_t)w * kTileM, tagged(L, acc[w][0] + acc[w][1]));
        acc[w][0] = acc[w][1] = 0.f;
      }
      ++seg;
    }
    ph ^= 1u << s;
    if (++s == S) s = 0;
    it.next();
  }
}

// On an exit that skips the projection: wait (bounded) for the TMA loads of
// the CTA's first n units, all within the prefill (first use of each stage).
template <int FMT>
static __device__ void land_prefill(const StepParams& p, TcShared& ts, int ub, int n) {
  RingPos pos;
  UnitIter it(p, ub);
  for (int j = 0; j < n; ++j, it.next()) {
    const bool coded = unit_coded<FMT>(p, it);
    cleanup_wait(coded ? &ts.rfull[pos.r] : &ts.full[pos.s], 0);
    pos.advance(p, coded);
  }
}
// On an aborted projection: wait (bounded) for the last TMA load issued into
// each stage of either ring: the producer's units [0, issued) (with coded
// weights its code tiles and the prefill's bf16 tiles), and with coded
// weights the bf16 tiles of units [0, dec_issued) from the decode warps.
template <int FMT>
static __device__ void land_issued(const StepParams& p, TcShared& ts, int ub, int issued, int prefill,
                                   int dec_issued) {
  const int bf16_end = bf16_weights<FMT>() ? issued : max(prefill, dec_issued);
  const int end = max(issued, bf16_end);
  int last_s[kMaxStages], last_r[kMaxRStages];
  uint32_t ph_s[kMaxStages], ph_r[kMaxRStages];
  for (int i = 0; i < kMaxStages; ++i) last_s[i] = -1;
  for (int i = 0; i < kMaxRStages; ++i) last_r[i] = -1;
  RingPos pos;
  UnitIter it(p, ub);
  for (int j = 0; j < end; ++j, it.next()) {
    const bool coded = unit_coded<FMT>(p, it);
    if (coded) {
      if (j < issued) {
        last_r[pos.r] = j;
        ph_r[pos.r] = pos.rph;
      }
    } else if (j < bf16_end) {
      last_s[pos.s] = j;
      ph_s[pos.s] = pos.ph;
    }
    pos.advance(p, coded);
  }
  for (int i = 0; i < p.stages; ++i)
    if (last_s[i] >= 0) cleanup_wait(&ts.full[i], ph_s[i]);
  for (int i = 0; i < p.rstages; ++i)
    if (last_r[i] >= 0) cleanup_wait(&ts.rfull[i], ph_r[i]);
}

// FMT: the in_proj_qkvz weight format (kFmtBf16, kFmtMxfp4, kFmtMxfp6; the
// coded formats alone carry the decoding warps' code), or kFmtBf16Fma: bf16
// weights with the projection on the CUDA cores (no tcgen05 instruction and
// no TMEM; everything else as with kFmtBf16).
// MULTI: a verify step (sequences of p.tokens rows, a state slot per token).
template <bool HAS_RES, bool STATE_BF16, int DK, int FMT, bool MULTI>
__global__ void __launch_bounds__(kThreads, 1) gdn_step_kernel(const __grid_constant__ StepParams p) {
  constexpr bool kMma = FMT != kFmtBf16Fma;  // the projection on the tensor cores
  extern __shared__ uint8_t dyn_smem[];
  __shared__ SmemPhases sm;
  __shared__ SmemTask st;
  __shared__ TcShared ts;
  uint8_t* sW = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  constexpr int kWindows = FMT == kFmtMxfp4 ? 2 : 1;                         // xn (and its MXFP4 copy)
  uint8_t* sR = sW + (size_t)p.stages * kWBytes;                             // code ring
  uint8_t* sX = sR + (size_t)p.rstages * code_tile_bytes<FMT>();             // normed-input window
  uint8_t* sXq = sX + (size_t)p.xslots * kXBytes;                            // its MXFP4-quantised copy
  uint8_t* sPad = sX + (size_t)kWindows * p.xslots * kXBytes;                // read past the windows; scratch
  uint8_t* sWin = sPad + p.xpad;
  uint32_t* sLut = reinterpret_cast<uint32_t*>(sWin + (size_t)p.xslots * kWinBytes);  // MXFP6 code-pair table
  const int tid = threadIdx.x, warp = tid >> 5, cta = blockIdx.x;
  // Without early weight reads nothing is read before the previous kernel in
  // the stream is done (the caller's kernel just before may write weights).
  if (!p.early_weights) griddep_wait();
  const int ub = p.plan->unit_begin[cta], nunits = p.plan->unit_begin[cta + 1] - ub;
  // The plan entries the drain and the MMA issuer read once the weight stream
  // fills HBM (a cold global load then takes a microsecond): loaded now, with
  // unit_begin, which the first weight tiles wait for anyway.
  if (tid >= 64 && tid < 64 + kMaxSegs) ts.seg_slot[tid - 64] = p.plan->seg_slot[cta][tid - 64];
  if (tid == 64 + kMaxSegs) ts.ks_first = p.plan->ks_first[cta];

  if (tid == 0) {
    tc::prefetch_tensormap(&p.tm_qkvz);
    tc::prefetch_tensormap(&p.tm_ba);
    if (p.out) tc::prefetch_tensormap(&p.tm_out);
    ts.abort = 0;
    ts.dec_issued = 0;
    for (int s = 0; s < p.stages; ++s) {
      tc::mbar_init(&ts.full[s], 1);
      tc::mbar_init(&ts.dfull[s], kConvWarps);
      tc::mbar_init(&ts.empty[s], kMma ? 1 : kFmaWarps);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ts.acc_full[b], 1);
      tc::mbar_init(&ts.acc_empty[b], 1);
    }
    for (int r = 0; r < p.rstages; ++r) {
      tc::mbar_init(&ts.rfull[r], 1);
      tc::mbar_init(&ts.rempty[r], kConvWarps);
    }
    tc::mbar_init(&ts.mma_done, 1);
    for (int s = 0; s < kOpMaxStages; ++s) tc::mbar_init(&ts.obar[s], 1);
    for (int s = 0; s < 3; ++s) tc::mbar_init(&ts.sbar[s], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();

  // The weights are the one input no step writes, so their stream starts
  // before the previous step is known to be done: with programmatic
  // dependent launch this CTA runs as soon as the previous step's CTA on its
  // SM has ended, and its first tiles overlap the previous step's tail. Only
  // kFirstTiles go out now: the x and residual loads that start the norm
  // hand-off queue behind them in HBM (measured on the full layer at 16 rows:
  // 0, 1, 2, 3, 4, 6 early tiles gave 103.9, 102.5, 100.4, 99.6, 99.1,
  // 99.6 µs). The rest of the ring follows once the norm partials are out.
  const int issued = prefill_units<FMT>(p, ub, nunits, kMaxStages + kMaxRStages);
  const int first = min(issued, kFirstTiles);
  if (tid == 32) start_weight_stream<FMT>(p, ts, sW, sR, ub, 0, first);
  const uint4 wnorm = load_norm_weights(p);  // also warms this SM's cache lines of the plan
  // the partials per tile, for the recurrence's loads (kept in shared memory:
  // the L1 left beside this kernel's shared memory does not keep the plan)
  static_assert(kMaxTiles <= kThreads, "one tile count per thread");
  const unsigned tile_cnt = tid < p.num_tiles ? p.plan->tile_num_ctas[tid] : 0u;
  griddep_wait();  // from here on the previous kernel's writes are visible (a no-op if already waited)
  griddep_launch_dependents();
  if (tid == 0) {
    sm.flag = (ld_relaxed_u32(&p.ctr->error) == 0);
    // Launch number: every CTA of the previous launches has published, none
    // of this one has, so the count is in [L * G, (L + 1) * G).
    sm.L = (int)(ld_relaxed_u64(&p.ctr->norm_arrive) / (unsigned long long)p.num_ctas);
  }
  __syncthreads();
  if (!sm.flag) {  // sticky error: every later launch returns at once
    if (tid == 32) land_prefill<FMT>(p, ts, ub, first);  // once the weight tiles in flight have landed
    return;
  }
  tl_stamp(p, TL_START);
  if (kMma && warp == 1) tc::tmem_alloc(&ts.tmem_base, kTmemCols);  // read after the barriers below

  // x and the residual (and the weights, unless already streaming), then the
  // norm partials go out. The sums of squares use the A operand's pad as
  // scratch.
  float* sq = reinterpret_cast<float*>(sPad);
  stage_residual_slices<HAS_RES>(p, sX, sWin, sq, [&] { store_norm_weights(p, sWin, wnorm); });
  tl_stamp(p, TL_R_STAGED);
  const int L = sm.L;
  publish_norm_partials(p, sq, L);
  if (tid == 32) start_weight_stream<FMT>(p, ts, sW, sR, ub, first, issued);
  write_residual_out(p, sX);
  if (FMT == kFmtMxfp6)  // the code-pair table, while the norm hand-off is in flight
    for (uint32_t i = tid; i < kE2m3LutEntries; i += kThreads) sLut[i] = e2m3x2_to_bf16(i & 63u, i >> 6);
  if (!phase_wait_rstd(p, sm, L)) {
    if (tid == 32) land_prefill<FMT>(p, ts, ub, issued);  // let the weight tiles in flight land
    if (kMma && warp == 1) {
      tc::tc_fence_after();
      tc::tmem_dealloc(ts.tmem_base, kTmemCols);
    }
    return;
  }
  finish_normed_slices<FMT>(p, sm, sX, sXq, sWin);
  tl_stamp(p, TL_XN_OUT);
  tc::fence_proxy_async_smem();
  if (kMma) tc::tc_fence_before();
  __syncthreads();
  if (kMma) tc::tc_fence_after();
  const uint32_t tmem = kMma ? ts.tmem_base : 0u;
  tl_stamp(p, TL_PROJ_START);
  // The first recurrence task's state goes into registers now: its latency
  // hides under the projection, which leaves most threads idle.
  StateRegs<DK> first_state;
  int rt0, rt1;
  task_range(p, rt0, rt1);
  // two or more decode tasks: the staged recurrence, in the shared memory
  // the projection leaves
  const bool staged = !MULTI && rt1 - rt0 >= 2 && rt1 - rt0 <= kMaxStagedTasks &&
                      p.dyn_free >= staged_recurrence_bytes<DK, STATE_BF16>();
  if (rt0 < rt1 && !staged) load_state<DK, STATE_BF16>(p, rt0, first_state);
  if (staged && tid == 0) prefetch_state_l2<DK, STATE_BF16>(p, rt0);  // its bulk copy reads L2
  int issued_total = issued;
  if (nunits > 0) {
    if (warp == 0) {
      issued_total = producer_loop<FMT>(p, ts, sW, sR, ub, nunits, issued, tc::policy_evict_first());
    } else if constexpr (!kMma) {
      if (warp >= kWarps - kFmaWarps) fma_loop(p, ts, sW, sX, ub, nunits, tid - (kWarps - kFmaWarps) * 32, L);
    } else {
      if (warp == 1)
        mma_loop<FMT>(p, ts, sW, sX, sXq, ub, nunits, tmem);
      else if (warp == 4 || (FMT == kFmtBf16 && (warp == 8 || warp == 12)))
        drain_loop<FMT == kFmtBf16 ? 3 : 1>(p, ts, ub, nunits, tmem, (warp / 4 - 1) * 32 + (tid & 31), L);
      else if (FMT != kFmtBf16 && conv_index(warp) >= 0)
        decode_loop<FMT>(p, ts, sW, sR, ub, nunits, issued, conv_index(warp) * 32 + (tid & 31), sLut);
    }
  }
  if (tid < p.num_tiles) sm.tiles[tid] = (unsigned char)tile_cnt;
  if (kMma) tc::tc_fence_before();
  __syncthreads();
  const bool aborted = ts.abort != 0;
  // every partial of this CTA is stored (the drain's or the FMA warps'
  // stores are ordered before this release by the barrier above)
  if (!aborted && tid == 0) red_add_release_u64(&p.ctr->proj_done, 1ull);
  if (aborted && tid == 0)  // TMA in flight lands before exit
    land_issued<FMT>(p, ts, ub, issued_total, issued, *reinterpret_cast<volatile int*>(&ts.dec_issued));
  if (kMma && warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  tl_stamp(p, TL_PROJ_END);
  // out_proj's first weight chunks stream into the freed ring: now in a CTA
  // without recurrence tasks, after its tasks in one with (so they do not
  // compete with the tasks' loads)
  const size_t ring_bytes = (size_t)p.stages * kWBytes + (size_t)p.rstages * code_tile_bytes<FMT>();
  if (!aborted && p.out && warp == 0 && rt0 >= rt1) out_proj_prefetch(p, sW, ring_bytes, ts.obar);
  if (!aborted) {
    const bool rec_ok = staged ? phase_recurrence_staged<DK, STATE_BF16>(p, sW, ts.sbar, L, rt0, rt1, sm.tiles)
                               : phase_recurrence<DK, STATE_BF16, MULTI>(p, sm, st, L, first_state, rt0 < rt1, sm.tiles);
    // out_proj over the core rows of every CTA, in the freed weight ring
    if (p.out) {
      if (rec_ok) {
        phase_out_proj(p, sW, ring_bytes, ts.obar, L, rt0 < rt1);
      } else if (warp == 0 && rt0 >= rt1) {  // let the prefetched chunks land before the CTA ends (bounded)
        const OpShape o(p, ring_bytes);
        for (int s2 = 0; s2 < min(o.ns, o.nch); ++s2) {
          const unsigned long long c0 = globaltimer_ns();
          for (uint32_t it = 0; !tc::mbar_try_wait(&ts.obar[s2], 0); ++it)
            if ((it & 63) == 0 && globaltimer_ns() - c0 > kCleanupNs) break;
        }
      }
    }
    tl_stamp(p, TL_END);
  }
}

}  // namespace gdn
