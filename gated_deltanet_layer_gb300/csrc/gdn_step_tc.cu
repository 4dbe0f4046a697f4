// GDN decode-step launch with the projections on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM, weight tiles fed by TMA).
//
// The MMA is D[m][n] += A[m][k] B[n][k] with A = the normed input xn (M = 128:
// the step's up to 16 rows; the MMA also reads 112 rows of whatever lies past
// a slice, whose results land in TMEM lanes nobody reads) and B = a 256-row
// weight tile (N = 256, K-major, 128-byte swizzle). A 128x16x16 MMA costs the
// tensor core about as much issue time as a 128x256x16 one, so the weights
// take the wide N side: one instruction consumes 8 KB of weights.
//
// One persistent CTA per SM. Roles during the projection:
//   thread 0 (warp 0)   TMA producer: 256-row x 64-column bf16 weight tiles
//                       into a ring of shared-memory stages; the first stages
//                       and an L2 prefetch of the following units are issued
//                       at kernel entry, so HBM streams weights while the norm
//                       hand-off runs
//   warp 1              allocates TMEM; its thread 0 issues tcgen05.mma into
//                       one of two 128 x 256 f32 accumulators
//   warp 4              drains an accumulator with tcgen05.ld (lane w holds
//                       row w of the step), writes the CTA's partial of the
//                       tile and publishes it; the recurrence tasks reduce the
//                       partials they need
// The A operand (xn of the CTA's k-steps, 16 rows, rows past the step's row
// count zero) is built per launch in shared memory: r = x + residual is
// staged while the norm hand-off is in flight and normalised in place once
// rstd is known; there is no global xn image and no second grid-wide
// hand-off. Every mbarrier wait is bounded; a wait that runs out records a
// deadline error, and the CTA waits for its own copies and MMAs in flight,
// frees its TMEM and returns.
#include "gdn_kernels.h"
#include "gdn_phases.cuh"
#include "gdn_tc_ptx.cuh"

namespace gdn {

namespace {
constexpr int kStages = 3;                              // weight tiles in flight per CTA
constexpr uint32_t kWBytes = kTileM * kKStep * 2;       // 32 KB weight tile (B operand)
constexpr uint32_t kXBytes = kMaxRows * kKStep * 2;     // 2 KB normed-input slice (A rows 0..15)
constexpr uint32_t kXPad = (128 - kMaxRows) * 128;      // 14 KB an M = 128 MMA reads past the last slice
constexpr uint32_t kWinBytes = kKStep * 2;              // input-norm weights of one k-step
constexpr uint32_t kTmemCols = 2 * kTileM;              // two 128 x 256 f32 accumulators
constexpr int kPrefetchUnits = 4;                       // units prefetched to L2 ahead of the ring
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(128, kTileM);
constexpr size_t kDynSmem = (size_t)kStages * kWBytes + (size_t)kMaxBSlots * kXBytes + kXPad +
                            (size_t)kMaxBSlots * kWinBytes + 1024;
constexpr uint32_t kWaitPipe = 4;                       // error-word id of a pipeline wait
constexpr unsigned long long kCleanupNs = 100000000ull; // bound of the waits on the abort path
}  // namespace

struct TcShared {
  uint64_t full[kStages];   // weight tile landed (TMA complete_tx)
  uint64_t empty[kStages];  // MMAs of the stage done (tcgen05.commit)
  uint64_t acc_full[2];     // accumulator ready for the drain
  uint64_t acc_empty[2];    // accumulator drained
  uint64_t mma_done;        // every MMA issued by the CTA done
  uint32_t tmem_base;
  int abort;
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

__device__ __forceinline__ void issue_weight_tile(const StepParams& p, TcShared& ts, uint8_t* sW,
                                                  const UnitIter& it, int n, uint64_t pol) {
  int row0;
  const CUtensorMap* m = weight_map(p, it.t, row0);
  const int s = n % kStages;
  tc::mbar_arrive_expect_tx(&ts.full[s], kWBytes);
  tc::tma_load_2d(sW + (size_t)s * kWBytes, m, it.ks * kKStep, row0, &ts.full[s], pol);
  if (n < 16) tl_stamp_here(p, TL_UNIT_ISSUED + n);
}

__device__ __forceinline__ void prefetch_weight_tile(const StepParams& p, const UnitIter& it) {
  int row0;
  tc::tma_prefetch_2d(weight_map(p, it.t, row0), it.ks * kKStep, row0);
}

// L2 prefetch of the state this CTA's recurrence tasks read, and of the conv
// state rows of the step (read by the recurrence tasks of each row).
template <int DK, bool STATE_BF16>
static __device__ __forceinline__ void prefetch_states(const StepParams& p) {
  const int cta = blockIdx.x;
  const int T = p.rows * p.Hv;
  const int t0 = (int)(((long long)cta * T) / p.num_ctas);
  const int t1 = (int)(((long long)(cta + 1) * T) / p.num_ctas);
  constexpr uint32_t bytes = DK * DK * (STATE_BF16 ? 2 : 4);
  for (int task = t0; task < t1; ++task) {
    const int w = task / p.Hv, h = task - w * p.Hv;
    const int slot = p.idx[w];
    if (row_is_live(p, slot))
      tc::prefetch_l2_bulk(static_cast<const char*>(p.ssm_state) + ((size_t)slot * p.Hv + h) * bytes, bytes);
  }
  if (cta < p.rows) {
    const int slot = p.idx[cta];
    if (row_is_live(p, slot))
      tc::prefetch_l2_bulk(p.conv_state + (size_t)slot * p.C * 3, (uint32_t)p.C * 6);
  }
}

// The A operand of this CTA: the normed input xn of its k-steps as slices in
// shared memory. Slot j holds k-step (ks_first + j) mod ksteps, 16 rows x 64
// columns bf16 in the 128-byte swizzled K-major layout (row r at r * 128
// bytes, its 16-byte chunk c at position c ^ (r % 8)); rows past the step's
// rows are 0. Built in two passes: r = bf16(x + residual) and the norm
// weights are staged before the norm hand-off completes (they do not need
// rstd), then xn = bf16(r * rstd * (1 + w)) is formed in place.
template <bool HAS_RES>
static __device__ __forceinline__ void stage_residual_slices(const StepParams& p, uint8_t* sX, uint8_t* sWin) {
  const int cta = blockIdx.x, W = p.rows;
  const int nb = p.nb_slots[cta], ks0 = p.ks_first[cta];
  const int ntask = nb * kMaxRows * 8;  // (slot, row, 16-byte chunk)
  constexpr int B = 4;                  // tasks per thread in flight
  for (int i0 = threadIdx.x; i0 < ntask; i0 += kThreads * B) {
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
#pragma unroll
    for (int k = 0; k < B; ++k) {
      const int i = i0 + k * kThreads;
      const int j = i >> 7, w = (i >> 3) & (kMaxRows - 1), c = i & 7;
      if (i < ntask)
        *reinterpret_cast<uint4*>(sX + (size_t)j * kXBytes + w * 128 + ((c ^ (w & 7)) << 4)) =
            w < W ? residual8<HAS_RES>(xv[k], qv[k]) : make_uint4(0, 0, 0, 0);
    }
  }
  for (int i = threadIdx.x; i < nb * 8; i += kThreads) {
    const int j = i >> 3, c = i & 7;
    reinterpret_cast<uint4*>(sWin + (size_t)j * kWinBytes)[c] =
        ld_stream_v4(p.w_in + (size_t)((ks0 + j) % p.ksteps) * kKStep + c * 8);
  }
}

static __device__ __forceinline__ void finish_normed_slices(const StepParams& p, const SmemPhases& sm,
                                                            uint8_t* sX, const uint8_t* sWin) {
  const int cta = blockIdx.x, W = p.rows;
  const int ntask = p.nb_slots[cta] * W * 8;  // (slot, row < W, chunk)
  for (int i = threadIdx.x; i < ntask; i += kThreads) {
    const int j = i / (W * 8), rem = i - j * (W * 8), w = rem >> 3, c = rem & 7;
    uint4* d = reinterpret_cast<uint4*>(sX + (size_t)j * kXBytes + w * 128 + ((c ^ (w & 7)) << 4));
    *d = normed8(*d, reinterpret_cast<const uint4*>(sWin + (size_t)j * kWinBytes)[c], sm.rstd[w]);
  }
}

// TMA producer: weight tiles `issued`.. into the ring, each into a stage the
// MMAs have released; keeps an L2 prefetch kPrefetchUnits units ahead.
// Returns the number of units issued.
static __device__ __forceinline__ int producer_loop(const StepParams& p, TcShared& ts, uint8_t* sW, int ub,
                                                   int nunits, int issued, uint64_t pol) {
  UnitIter it(p, ub + issued);
  UnitIter pf(p, min(ub + issued + kPrefetchUnits, ub + nunits - 1));
  for (int n = issued; n < nunits; ++n) {
    const int s = n % kStages;
    if (!pipe_wait(p, ts, &ts.empty[s], ((n / kStages) & 1) ^ 1)) return n;
    issue_weight_tile(p, ts, sW, it, n, pol);
    it.next();
    if (n + kPrefetchUnits < nunits) {
      prefetch_weight_tile(p, pf);
      pf.next();
    }
  }
  return nunits;
}

// MMA issuer: per unit, 4 MMAs of K = 16 over the stage's 64 columns into the
// segment's accumulator; a segment (the units of one group) starts by
// overwriting. Commits release the stage and, at a segment's end, hand the
// accumulator to the drain.
static __device__ __forceinline__ void mma_loop(const StepParams& p, TcShared& ts, uint8_t* sW,
                                                uint8_t* sX, int ub, int nunits, uint32_t tmem) {
  const int ks0 = p.ks_first[blockIdx.x], KS = p.ksteps;
  UnitIter it(p, ub);
  int seg = -1;
  bool seg_open = false;
  for (int n = 0; n < nunits; ++n) {
    const int s = n % kStages;
    const bool first = !seg_open;
    if (first) {
      ++seg;
      seg_open = true;
      if (!pipe_wait(p, ts, &ts.acc_empty[seg & 1], ((seg >> 1) & 1) ^ 1)) break;
    }
    if (!pipe_wait(p, ts, &ts.full[s], (n / kStages) & 1)) break;
    tc::tc_fence_after();
    if (n == 0) tl_stamp_here(p, TL_MMA_FIRST);
    if (n < 16) tl_stamp_here(p, TL_UNIT_READY + n);
    int slot = it.ks - ks0;
    if (slot < 0) slot += KS;
    const uint64_t ad = tc::sdesc_k_sw128(tc::smem_u32(sX + (size_t)slot * kXBytes));
    const uint64_t bd = tc::sdesc_k_sw128(tc::smem_u32(sW + (size_t)s * kWBytes));
    const uint32_t d = tmem + (uint32_t)(seg & 1) * kTileM;
#pragma unroll
    for (int k = 0; k < kKStep / 16; ++k)  // +32 bytes along K inside the swizzle atom
      tc::mma_bf16(d, ad + 2 * k, bd + 2 * k, kIdesc, (first && k == 0) ? 0u : 1u);
    tc::mma_commit(&ts.empty[s]);
    if (n + 1 == nunits || it.group_end()) {
      tc::mma_commit(&ts.acc_full[seg & 1]);
      seg_open = false;
    }
    it.next();
  }
  tc::mma_commit(&ts.mma_done);
  cleanup_wait(&ts.mma_done, 0);
  tl_stamp_here(p, TL_MMA_LAST);
}

// Drain (warp 4): per segment, read the 128 x 256 accumulator (lane w = row
// w of the step, 256 weight rows), release it, write the CTA's partial of the
// tile and publish it.
static __device__ __forceinline__ void drain_loop(const StepParams& p, TcShared& ts, int ub, int nunits,
                                                  uint32_t tmem, int lane) {
  const int W = p.rows;
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
    float* dst = p.proj_part + ((size_t)t * p.max_contrib + p.seg_slot[blockIdx.x][seg]) * kMaxRows * kTileM +
                 (size_t)lane * kTileM;
#pragma unroll 1
    for (int c = 0; c < kTileM / 32; ++c) {
      float v[32];
      tc::tmem_ld32(tmem + (uint32_t)b * kTileM + c * 32, v);
      if (lane < W) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          reinterpret_cast<float4*>(dst + c * 32)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&ts.acc_empty[b]);
    publish_tile_partial<32>(p, t, lane);
  }
}

template <bool HAS_RES, bool STATE_BF16, int DK>
__global__ void __launch_bounds__(kThreads, 1) gdn_step_tc_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ SmemPhases sm;
  __shared__ SmemTask st;
  __shared__ TcShared ts;
  uint8_t* sW = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = sW + (size_t)kStages * kWBytes;
  uint8_t* sWin = sX + (size_t)kMaxBSlots * kXBytes + kXPad;
  const int tid = threadIdx.x, warp = tid >> 5, cta = blockIdx.x;
  const int ub = p.unit_begin[cta], nunits = p.unit_begin[cta + 1] - ub;

  if (tid == 0) {
    tc::prefetch_tensormap(&p.tm_qkvz);
    tc::prefetch_tensormap(&p.tm_ba);
    sm.flag = (ld_relaxed_u32(&p.ctr->error) == 0);
    ts.abort = 0;
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&ts.full[s], 1);
      tc::mbar_init(&ts.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&ts.acc_full[b], 1);
      tc::mbar_init(&ts.acc_empty[b], 1);
    }
    tc::mbar_init(&ts.mma_done, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (!sm.flag) return;  // sticky error: every later launch returns at once
  tl_stamp(p, TL_START);

  // Start the weight stream before any wait.
  uint64_t pol = 0;
  int issued = 0;
  if (tid == 0 && nunits > 0) {
    pol = tc::policy_evict_first();
    issued = min(nunits, kStages);
    UnitIter it(p, ub);
    for (int n = 0; n < issued; ++n, it.next()) issue_weight_tile(p, ts, sW, it, n, pol);
    for (int n = issued; n < min(nunits, issued + kPrefetchUnits); ++n, it.next()) prefetch_weight_tile(p, it);
    tl_stamp_here(p, TL_ISSUED);
  }

  phase_norm_partials<HAS_RES>(p, sm);
  const int L = sm.L;
  if (tid == 64) prefetch_states<DK, STATE_BF16>(p);
  stage_residual_slices<HAS_RES>(p, sX, sWin);
  tl_stamp(p, TL_R_STAGED);
  if (!phase_wait_rstd(p, sm, L)) {
    if (tid == 0)  // let the weight tiles in flight land before the CTA exits
      for (int n = 0; n < issued; ++n) cleanup_wait(&ts.full[n], 0);
    return;
  }
  if (warp == 1) tc::tmem_alloc(&ts.tmem_base, kTmemCols);
  finish_normed_slices(p, sm, sX, sWin);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = ts.tmem_base;
  tl_stamp(p, TL_PROJ_START);
  if (nunits > 0) {
    if (tid == 0)
      issued = producer_loop(p, ts, sW, ub, nunits, issued, pol);
    else if (tid == 32)
      mma_loop(p, ts, sW, sX, ub, nunits, tmem);
    else if (warp == 4)
      drain_loop(p, ts, ub, nunits, tmem, tid & 31);
  }
  tc::tc_fence_before();
  __syncthreads();
  const bool aborted = ts.abort != 0;
  if (aborted && tid == 0) {
    // the last tile issued into each stage must land before the CTA exits
    for (int s = 0; s < kStages; ++s) {
      int last = -1;
      for (int n = s; n < issued; n += kStages) last = n;
      if (last >= 0) cleanup_wait(&ts.full[s], (last / kStages) & 1);
    }
  }
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  tl_stamp(p, TL_PROJ_END);
  if (aborted) return;
  phase_recurrence<DK, STATE_BF16>(p, sm, st, L);
  tl_stamp(p, TL_END);
}

const void* tensor_core_kernel(bool has_res, bool state_bf16, int dk) {
#define GDN_PICK(R, B, D) \
  if (has_res == R && state_bf16 == B && dk == D) return (const void*)&gdn_step_tc_kernel<R, B, D>;
  GDN_PICK(true, false, 128) GDN_PICK(true, true, 128) GDN_PICK(false, false, 128) GDN_PICK(false, true, 128)
  GDN_PICK(true, false, 64) GDN_PICK(true, true, 64) GDN_PICK(false, false, 64) GDN_PICK(false, true, 64)
#undef GDN_PICK
  return nullptr;
}

size_t tensor_core_smem_bytes() { return kDynSmem; }

}  // namespace gdn
