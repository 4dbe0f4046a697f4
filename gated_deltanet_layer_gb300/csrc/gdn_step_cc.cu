// GDN decode-step launch with the projections on CUDA cores (f32 FMA dot
// products of bf16 weights and the bf16 normed input).
//
// One persistent CTA per SM runs, in order: the residual add and its norm
// partials, the normed input image, its share of the in_proj_qkvz/in_proj_ba
// work units (a stream-K split of (256-row tile, 64-column step) units, so
// every CTA streams the same number of weight bytes), publishing a partial
// per tile it touched, and its share of the (row, value head) recurrence
// tasks, which reduce the partials they need. The norm sums and the
// projection partials are handed over as tagged words, the normed input
// image through a release/acquire counter; every wait is bounded and a
// failed wait leaves a sticky failed word (vLLM #60833, Details,
// "Limitations / follow-ups").
#include "gdn_kernels.h"
#include "gdn_phases.cuh"

namespace gdn {

__device__ __forceinline__ const __nv_bfloat16* weight_row(const StepParams& p, int t, int r, bool& valid) {
  if (t < p.tiles_qkvz) {
    valid = true;
    return p.w_qkvz + (size_t)(t * kTileM + r) * p.H;
  }
  const int n = (t - p.tiles_qkvz) * kTileM + r;
  valid = n < p.Nba;
  return p.w_ba + (size_t)(valid ? n : 0) * p.H;
}

// Projection engine on CUDA cores. Thread (row = tid/2, sub = tid%2) owns one
// weight row of the current 256-row tile and 32 of the 64 columns of each
// unit; its f32 sums over the CTA's units of one tile are combined over the 2
// lanes of the row and written as this CTA's partial of the tile.
static __device__ __forceinline__ bool phase_proj_cuda_core(const StepParams& p, SmemPhases& sm,
                                                            float (*xs)[kMaxRows][kKStep], int L) {
  const int cta = blockIdx.x, tid = threadIdx.x, W = p.rows;
  const int ub = p.plan->unit_begin[cta], ue = p.plan->unit_begin[cta + 1];
  if (ub >= ue) return true;
  if (tid == 0)
    sm.flag = wait_counter(p, &p.ctr->xn_arrive, (unsigned long long)(L + 1) * p.num_ctas, kWaitXn);
  tl_stamp(p, TL_PROJ_START);
  __syncthreads();
  if (!sm.flag) return false;

  const int row = tid >> 1, sub = tid & 1;
  auto stage = [&](int u, int buf) {
    if (tid < W * 8) {
      const int ks = u % p.ksteps;
      const int w = tid >> 3, c = (tid & 7) * 8;
      const uint4 v = ld_cg_v4(p.xn + (size_t)w * p.H + ks * kKStep + c);
      float4* d = reinterpret_cast<float4*>(&xs[buf][w][c]);
      d[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
      d[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
    }
  };
  auto wload = [&](int u, uint4 (&a)[4]) {
    const int t = u / p.ksteps, ks = u - t * p.ksteps;
    bool valid;
    const __nv_bfloat16* rp = weight_row(p, t, row, valid);
    if (valid) {
      const __nv_bfloat16* q = rp + ks * kKStep + sub * 32;
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] = ld_stream_v4(q + e * 8);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] = make_uint4(0, 0, 0, 0);
    }
  };

  float acc[kMaxRows];
#pragma unroll
  for (int w = 0; w < kMaxRows; ++w) acc[w] = 0.f;

  int seg = 0;  // segment index within this CTA's range (tile-major order)
  auto flush = [&](int t) {
#pragma unroll
    for (int w = 0; w < kMaxRows; ++w) acc[w] += __shfl_xor_sync(0xffffffffu, acc[w], 1);
    const int j = p.plan->seg_slot[cta][seg];
    unsigned long long* dst = p.proj_part + ((size_t)t * p.max_contrib + j) * kMaxRows * kTileM;
    if (sub == 0) {
#pragma unroll
      for (int w = 0; w < kMaxRows; ++w)
        if (w < W) st_tagged(dst + w * kTileM + row, tagged(L, acc[w]));
    }
#pragma unroll
    for (int w = 0; w < kMaxRows; ++w) acc[w] = 0.f;
  };

  constexpr int D = 2;  // units of weights in flight per thread
  uint4 wr[D][4];
#pragma unroll
  for (int j = 0; j < D; ++j)
    if (ub + j < ue) wload(ub + j, wr[j]);
  stage(ub, 0);
  __syncthreads();

  int cur = ub / p.ksteps;
  for (int u0 = ub; u0 < ue; u0 += D) {
#pragma unroll
    for (int j = 0; j < D; ++j) {
      const int u = u0 + j;
      if (u < ue) {
        const int t = u / p.ksteps;
        if (t != cur) {
          flush(cur);
          cur = t;
          ++seg;
        }
        if (u + 1 < ue) stage(u + 1, (u + 1 - ub) & 1);
        const float(*x)[kKStep] = xs[(u - ub) & 1];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t ws_[4] = {wr[j][e].x, wr[j][e].y, wr[j][e].z, wr[j][e].w};
          float wv[8];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            wv[2 * h] = bf16_lo(ws_[h]);
            wv[2 * h + 1] = bf16_hi(ws_[h]);
          }
#pragma unroll
          for (int w = 0; w < kMaxRows; ++w) {
            if (w < W) {
              const float4* xr = reinterpret_cast<const float4*>(&x[w][sub * 32 + e * 8]);
              const float4 x0 = xr[0], x1 = xr[1];
              float sacc = acc[w];
              sacc = fmaf(wv[0], x0.x, sacc); sacc = fmaf(wv[1], x0.y, sacc);
              sacc = fmaf(wv[2], x0.z, sacc); sacc = fmaf(wv[3], x0.w, sacc);
              sacc = fmaf(wv[4], x1.x, sacc); sacc = fmaf(wv[5], x1.y, sacc);
              sacc = fmaf(wv[6], x1.z, sacc); sacc = fmaf(wv[7], x1.w, sacc);
              acc[w] = sacc;
            }
          }
        }
        if (u + D < ue) wload(u + D, wr[j]);
        __syncthreads();
      }
    }
  }
  flush(cur);
  tl_stamp(p, TL_PROJ_END);
  return true;
}

// Dynamic shared memory of the CUDA-core kernel: the double-buffered
// normed-input slice of the current unit.
struct CcDynSmem {
  alignas(16) float xs[2][kMaxRows][kKStep];
};

template <bool HAS_RES, bool STATE_BF16, int DK>
__global__ void __launch_bounds__(kThreads, 1) gdn_step_cc_kernel(const __grid_constant__ StepParams p) {
  __shared__ SmemPhases sm;
  __shared__ SmemTask st;
  extern __shared__ __align__(16) uint8_t cc_dyn[];
  CcDynSmem& ds = *reinterpret_cast<CcDynSmem*>(cc_dyn);
  griddep_wait();  // the previous step's writes first
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    sm.flag = (ld_relaxed_u32(&p.ctr->error) == 0);
    // launch number: every CTA of the previous launches has counted itself
    sm.L = (int)(ld_relaxed_u64(&p.ctr->norm_arrive) / (unsigned long long)p.num_ctas);
  }
  __syncthreads();
  if (!sm.flag) return;  // sticky error: every later launch returns at once
  tl_stamp(p, TL_START);
  const int L = sm.L;
  phase_norm_partials<HAS_RES>(p, sm, L);
  if (!phase_normed_input(p, sm, L)) return;
  if (!phase_proj_cuda_core(p, sm, ds.xs, L)) return;
  StateRegs<DK> none;
  phase_recurrence<DK, STATE_BF16>(p, sm, st, L, none, false, p.plan->tile_num_ctas);
  tl_stamp(p, TL_END);
}

size_t cuda_core_smem_bytes() { return sizeof(CcDynSmem); }

const void* cuda_core_kernel(bool has_res, bool state_bf16, int dk) {
#define GDN_PICK(R, B, D) \
  if (has_res == R && state_bf16 == B && dk == D) return (const void*)&gdn_step_cc_kernel<R, B, D>;
  GDN_PICK(true, false, 128) GDN_PICK(true, true, 128) GDN_PICK(false, false, 128) GDN_PICK(false, true, 128)
  GDN_PICK(true, false, 64) GDN_PICK(true, true, 64) GDN_PICK(false, false, 64) GDN_PICK(false, true, 64)
#undef GDN_PICK
  return nullptr;
}

}  // namespace gdn
