// Phases of the persistent GDN decode-step launch that do not depend on the
// projection engine: residual add + norm partials, the normed input image,
// the per-tile epilogue (partial reduction, conv update + SiLU, q/k L2 norm)
// and the per-(row, value head) gated delta rule with the gated RMSNorm.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Every array is 16-byte aligned: several are accessed with 16-byte vectors.
struct SmemPhases {
  alignas(16) __nv_bfloat16 rbuf[kMaxRows][kMaxNormChunk];  // r = x + residual of this CTA's columns
  alignas(16) float part8[kMaxRows * (kMaxNormChunk / 8)];  // sums of 8 squares
  alignas(16) float ep[kMaxRows][kTileM];                   // tile epilogue values
  alignas(16) float v[128];                                 // recurrence task vectors (dv <= 128)
  alignas(16) float z[128];
  alignas(16) float o[128];
  alignas(16) float rstd[kMaxRows];
  alignas(16) float inv[kMaxRows * 2];                      // q/k inverse norms of one tile
  alignas(16) float red[kWarps];
  alignas(16) __nv_bfloat16 cst[kMaxRows][kTileM * 3];      // conv state of one tile's channels
  alignas(16) __nv_bfloat16 cw[kTileM * 4];                 // conv weights of one tile's channels
  int slot[kMaxRows];                                       // state index of each row
  int L;                 // launch number on this workspace
  int flag;              // CTA-wide decision broadcast by thread 0
};

// xn = bf16(r * rstd * (1 + w_in)) of 8 consecutive columns (r, w_in as bf16x2 words).
__device__ __forceinline__ uint4 normed8(uint4 rv, uint4 gv, float rstd) {
  const uint32_t rs[4] = {rv.x, rv.y, rv.z, rv.w}, gs[4] = {gv.x, gv.y, gv.z, gv.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    o[j] = pack_bf16x2(bf16_lo(rs[j]) * rstd * (1.0f + bf16_lo(gs[j])),
                       bf16_hi(rs[j]) * rstd * (1.0f + bf16_hi(gs[j])));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// r = bf16(x + residual) of 8 consecutive columns.
template <bool HAS_RES>
__device__ __forceinline__ uint4 residual8(uint4 xv, uint4 qv) {
  if (!HAS_RES) return xv;
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, qs[4] = {qv.x, qv.y, qv.z, qv.w};
  uint32_t rs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    rs[j] = pack_bf16x2(bf16_lo(xs[j]) + bf16_lo(qs[j]), bf16_hi(xs[j]) + bf16_hi(qs[j]));
  return make_uint4(rs[0], rs[1], rs[2], rs[3]);
}

// ---------------------------------------------------------------------------
// Phase 1: r = x + residual (bf16), residual_out, and each row's sum of r^2
// over this CTA's hidden columns. The sums are handed to every CTA through
// global memory and a release counter (vLLM #60833, Details, "x without an
// LDS tile": the norm CTAs publish their columns' sums of squares and each
// consumer builds the x it reads). Returns the launch number.
// ---------------------------------------------------------------------------
template <bool HAS_RES>
__device__ void phase_norm_partials(const StepParams& p, SmemPhases& sm) {
  const int W = p.rows, cta = blockIdx.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int c0 = cta * p.norm_chunk;
  const int ncol = max(0, min(p.H, c0 + p.norm_chunk) - c0);
  const int nvec = ncol >> 3;
  for (int i = tid; i < W * nvec; i += kThreads) {
    const int w = i / nvec, v = i - w * nvec;
    const size_t off = (size_t)w * p.H + c0 + v * 8;
    const uint4 xv = *reinterpret_cast<const uint4*>(p.x + off);
    const uint4 qv = HAS_RES ? *reinterpret_cast<const uint4*>(p.res + off) : xv;
    const uint4 rv = residual8<HAS_RES>(xv, qv);
    const uint32_t rs[4] = {rv.x, rv.y, rv.z, rv.w};
    *reinterpret_cast<uint4*>(p.res_out + off) = rv;
    *reinterpret_cast<uint4*>(&sm.rbuf[w][v * 8]) = rv;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(rs[j]), b = bf16_hi(rs[j]);
      s = fmaf(a, a, s);
      s = fmaf(b, b, s);
    }
    sm.part8[w * (kMaxNormChunk / 8) + v] = s;
  }
  __syncthreads();
  for (int w = warp; w < W; w += kWarps) {
    float s = 0.f;
    for (int v = lane; v < nvec; v += 32) s += sm.part8[w * (kMaxNormChunk / 8) + v];
    s = warp_sum(s);
    if (lane == 0) p.norm_part[w * p.num_ctas + cta] = s;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned long long old;
    if ((p.debug_flags & kDebugSkipNormPublish) && cta == 0)
      old = ld_acquire_u64(&p.ctr->norm_arrive);  // test hook: never publish
    else
      old = atom_add_release_u64(&p.ctr->norm_arrive, 1ull);
    sm.L = (int)(old / (unsigned long long)p.num_ctas);
  }
  tl_stamp(p, TL_NORM_OUT);
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Phase 1b: wait for every CTA's sums, form rstd per row (Gemma RMSNorm:
// rstd = 1/sqrt(mean(r^2) + eps), xn = r * rstd * (1 + w)) and write this
// CTA's columns of the normed input xn (bf16) to the workspace image.
// ---------------------------------------------------------------------------
static __device__ bool phase_wait_rstd(const StepParams& p, SmemPhases& sm, int L) {
  const int W = p.rows, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0)
    sm.flag = wait_counter(p, &p.ctr->norm_arrive,
                           (unsigned long long)(L + 1) * p.num_ctas, kWaitNorm);
  tl_stamp(p, TL_NORM_IN);
  __syncthreads();
  if (!sm.flag) return false;
  for (int w = warp; w < W; w += kWarps) {
    float s = 0.f;
    for (int c = lane; c < p.num_ctas; c += 32) s += ld_cg_f(p.norm_part + w * p.num_ctas + c);
    s = warp_sum(s);
    if (lane == 0) sm.rstd[w] = 1.0f / sqrtf(s / (float)p.H + p.norm_eps);
  }
  __syncthreads();
  return true;
}

static __device__ bool phase_normed_input(const StepParams& p, SmemPhases& sm, int L) {
  const int W = p.rows, cta = blockIdx.x, tid = threadIdx.x;
  if (!phase_wait_rstd(p, sm, L)) return false;
  const int c0 = cta * p.norm_chunk;
  const int ncol = max(0, min(p.H, c0 + p.norm_chunk) - c0);
  const int nvec = ncol >> 3;
  for (int i = tid; i < W * nvec; i += kThreads) {
    const int w = i / nvec, v = i - w * nvec;
    const uint4 rv = *reinterpret_cast<const uint4*>(&sm.rbuf[w][v * 8]);
    const uint4 gv = *reinterpret_cast<const uint4*>(p.w_in + c0 + v * 8);
    *reinterpret_cast<uint4*>(p.xn + (size_t)w * p.H + c0 + v * 8) = normed8(rv, gv, sm.rstd[w]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) atom_add_release_u64(&p.ctr->xn_arrive, 1ull);
  tl_stamp(p, TL_XN_OUT);
  return true;
}

__device__ __forceinline__ bool row_is_live(const StepParams& p, int slot) {
  return slot > 0 && slot < p.num_slots;
}

// Synchronise the threads that run an epilogue: the whole CTA (barrier 0) or
// the 128-thread drain group of the tensor-core engine (named barrier 1).
template <int NT>
__device__ __forceinline__ void group_sync() {
  if (NT == kThreads)
    __syncthreads();
  else
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// ---------------------------------------------------------------------------
// Tile epilogue, run by the last CTA to deliver a partial of projection tile t
// (NT threads, group thread index gtid): sum the partials in slot order, round
// to bf16 (the projection output), then by row kind: q/k/v channels -> conv
// update + SiLU (and the L2 norm for q, k); z -> stored; b/a -> stored for the
// gates. Pad rows write no state. (sgl-amd-mono #89, "Kernels before and
// after": the split, the conv update and the gated delta rule's q/k
// normalisation all move into one launch.)
// ---------------------------------------------------------------------------
template <int NT>
static __device__ void tile_epilogue(const StepParams& p, SmemPhases& sm, int t, int gtid) {
  constexpr int NW = NT / 32;
  constexpr int IT = (kMaxRows * (kTileM / 4) + NT - 1) / NT;  // float4 items per thread
  const int W = p.rows;
  const int warp = gtid >> 5, lane = gtid & 31;
  const bool is_ba = t >= p.tiles_qkvz;
  const int n0 = is_ba ? (t - p.tiles_qkvz) * kTileM : t * kTileM;
  const int rows_t = is_ba ? min(kTileM, p.Nba - n0) : kTileM;
  const int nc = p.tile_num_ctas[t];
  const float* part = p.proj_part + (size_t)t * p.max_contrib * kMaxRows * kTileM;
  const bool conv_tile = !is_ba && n0 < p.C;
  if (gtid < W) sm.slot[gtid] = p.idx[gtid];
  // conv state and weights of this tile's channels, staged while the partials load
  if (conv_tile) {
    for (int i = gtid; i < W * (kTileM * 3 / 8); i += NT) {
      const int w = i / (kTileM * 3 / 8), q = i - w * (kTileM * 3 / 8);
      const int slot = p.idx[w];
      if (row_is_live(p, slot))
        reinterpret_cast<uint4*>(sm.cst[w])[q] =
            *reinterpret_cast<const uint4*>(p.conv_state + ((size_t)slot * p.C + n0) * 3 + q * 8);
    }
    for (int i = gtid; i < kTileM * 4 / 8; i += NT)
      reinterpret_cast<uint4*>(sm.cw)[i] = *reinterpret_cast<const uint4*>(p.conv_w + (size_t)n0 * 4 + i * 8);
  }
  // partial sums: float4 items (row w, rows 4*r4 .. 4*r4+3), slots added in order
  float4 acc[IT];
#pragma unroll
  for (int it = 0; it < IT; ++it) acc[it] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < nc; j0 += 4) {
    float4 v[4][IT];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int q = gtid + it * NT, w = q >> 5, r4 = q & 31;
        if (j0 + jj < nc && w < W && r4 * 4 < rows_t)
          v[jj][it] = ld_cg_f4(part + ((size_t)(j0 + jj) * kMaxRows + w) * kTileM + r4 * 4);
      }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int q = gtid + it * NT, w = q >> 5, r4 = q & 31;
        if (j0 + jj < nc && w < W && r4 * 4 < rows_t) {
          acc[it].x += v[jj][it].x; acc[it].y += v[jj][it].y;
          acc[it].z += v[jj][it].z; acc[it].w += v[jj][it].w;
        }
      }
  }
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int q = gtid + it * NT, w = q >> 5, r4 = q & 31;
    if (w < W && r4 * 4 < rows_t)
      *reinterpret_cast<float4*>(&sm.ep[w][r4 * 4]) =
          make_float4(round_bf16(acc[it].x), round_bf16(acc[it].y), round_bf16(acc[it].z), round_bf16(acc[it].w));
  }
  group_sync<NT>();
  if (is_ba) {
    for (int i = gtid; i < W * kTileM; i += NT) {
      const int w = i >> 7, r = i & (kTileM - 1);
      if (r < rows_t) p.act_ba[(size_t)w * p.Nba + n0 + r] = sm.ep[w][r];
    }
    return;
  }
  if (!conv_tile) {  // z rows
    for (int i = gtid; i < W * kTileM; i += NT) {
      const int w = i >> 7, r = i & (kTileM - 1);
      p.act[(size_t)w * p.Nqkvz + n0 + r] = sm.ep[w][r];
    }
    return;
  }
  // conv channels c = n0 + r over [q | k | v]: y = silu(w0 s0 + w1 s1 + w2 s2 + w3 p),
  // state <- [s1, s2, p]
  for (int i = gtid; i < W * kTileM; i += NT) {
    const int w = i >> 7, r = i & (kTileM - 1);
    if (!row_is_live(p, sm.slot[w])) continue;
    __nv_bfloat16* cs = &sm.cst[w][r * 3];
    const __nv_bfloat16* cw = &sm.cw[r * 4];
    const float pv = sm.ep[w][r];
    const float s1 = bf16_to_f(cs[1]), s2 = bf16_to_f(cs[2]);
    float acc1 = bf16_to_f(cw[0]) * bf16_to_f(cs[0]);
    acc1 = fmaf(bf16_to_f(cw[1]), s1, acc1);
    acc1 = fmaf(bf16_to_f(cw[2]), s2, acc1);
    acc1 = fmaf(bf16_to_f(cw[3]), pv, acc1);
    cs[0] = __float2bfloat16_rn(s1);
    cs[1] = __float2bfloat16_rn(s2);
    cs[2] = __float2bfloat16_rn(pv);
    sm.ep[w][r] = silu_f(acc1);
  }
  group_sync<NT>();
  for (int i = gtid; i < W * (kTileM * 3 / 8); i += NT) {
    const int w = i / (kTileM * 3 / 8), q = i - w * (kTileM * 3 / 8);
    const int slot = sm.slot[w];
    if (row_is_live(p, slot))
      *reinterpret_cast<uint4*>(p.conv_state + ((size_t)slot * p.C + n0) * 3 + q * 8) =
          reinterpret_cast<const uint4*>(sm.cst[w])[q];
  }
  const bool is_qk = n0 < 2 * p.Hk * p.dk;
  if (is_qk) {
    const bool is_q = n0 < p.Hk * p.dk;
    const int hpt = kTileM / p.dk;  // heads in this tile
    for (int pr = warp; pr < W * hpt; pr += NW) {
      const int w = pr / hpt, hd = pr - w * hpt;
      float s = 0.f;
      for (int j = lane; j < p.dk; j += 32) {
        const float y = sm.ep[w][hd * p.dk + j];
        s = fmaf(y, y, s);
      }
      s = warp_sum(s);
      if (lane == 0) sm.inv[pr] = (1.0f / sqrtf(s + p.l2_eps)) * (is_q ? p.q_scale : 1.0f);
    }
    group_sync<NT>();
    for (int i = gtid; i < W * kTileM; i += NT) {
      const int w = i >> 7, r = i & (kTileM - 1);
      p.act[(size_t)w * p.Nqkvz + n0 + r] = sm.ep[w][r] * sm.inv[w * hpt + r / p.dk];
    }
  } else {
    for (int i = gtid; i < W * kTileM; i += NT) {
      const int w = i >> 7, r = i & (kTileM - 1);
      p.act[(size_t)w * p.Nqkvz + n0 + r] = sm.ep[w][r];
    }
  }
}

// Publish a finished partial of tile t and count it. Called by all NT
// threads of a group after the partial is written; returns (to every thread
// of the group) whether this was the tile's last partial.
template <int NT>
static __device__ bool arrive_tile_partial(const StepParams& p, SmemPhases& sm, int t, int L, int gtid) {
  __threadfence();
  group_sync<NT>();
  if (gtid == 0) {
    const unsigned long long old = atom_add_acq_rel_u64(&p.ctr->tile_arrive[t], 1ull);
    const unsigned long long full = (unsigned long long)(L + 1) * p.tile_num_ctas[t];
    sm.flag = (old + 1 == full);
  }
  group_sync<NT>();
  const bool last = sm.flag;
  group_sync<NT>();
  return last;
}

// Run tile t's epilogue (all partials are in) and publish the tile as done.
template <int NT>
static __device__ void finish_tile(const StepParams& p, SmemPhases& sm, int t, int gtid) {
  __threadfence();
  if ((p.debug_flags & kDebugTimeline) && gtid == 0) {
    p.ctr->tl_tile[t][0] = globaltimer_ns();
    p.ctr->tl_cta[blockIdx.x][TL_EPI_COUNT] += 1;
  }
  tile_epilogue<NT>(p, sm, t, gtid);
  __threadfence();
  group_sync<NT>();
  if (gtid == 0) {
    if (p.debug_flags & kDebugTimeline) p.ctr->tl_tile[t][1] = globaltimer_ns();
    atom_add_release_u64(&p.ctr->tile_done[t], 1ull);
  }
  group_sync<NT>();
}

// Deliver a partial and, as the tile's last contributor, finish the tile.
template <int NT>
static __device__ void deliver_tile_partial(const StepParams& p, SmemPhases& sm, int t, int L, int gtid) {
  if (arrive_tile_partial<NT>(p, sm, t, L, gtid)) finish_tile<NT>(p, sm, t, gtid);
}

// ---------------------------------------------------------------------------
// Phase 3: per (row w, value head h) task: gates, the gated delta rule on
// the row's state slot, and the gated RMSNorm x SiLU(z).
//   g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)
//   S <- e^g S;  u = beta (v - S k);  S <- S + u k^T;  o = S q   (S[v][k])
//   core = bf16(o * rsqrt(mean(o^2) + eps) * w_g * silu(z))
// Each warp owns whole state rows S[v][:], so S k and S q are reductions over
// one row's lanes (sgl-amd-mono #89, Modifications, gdn.py row: f32
// recurrence, state stored in f32 or bf16 in place; pad rows write a zero
// core row and no state).
// ---------------------------------------------------------------------------
template <int DK, bool STATE_BF16>
__device__ bool phase_recurrence(const StepParams& p, SmemPhases& sm, int L) {
  constexpr int LPR = DK / 4;            // lanes per state row, 4 elements each
  constexpr int RPW = 32 / LPR;          // rows per warp per step
  constexpr int NR = DK / (kWarps * RPW);  // rows per lane (dv == dk)
  static_assert(NR >= 1, "state rows per lane");
  const int W = p.rows, cta = blockIdx.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int sub = lane % LPR, rw = lane / LPR;
  const int T = W * p.Hv;
  const int t0 = (int)(((long long)cta * T) / p.num_ctas);
  const int t1 = (int)(((long long)(cta + 1) * T) / p.num_ctas);
  for (int task = t0; task < t1; ++task) {
    const int w = task / p.Hv, h = task - w * p.Hv;
    const int slot = p.idx[w];
    __nv_bfloat16* core = p.core_out + (size_t)w * p.Hv * DK + (size_t)h * DK;
    if (!row_is_live(p, slot)) {
      if (slot >= p.num_slots && h == 0 && tid == 0) record_error(p.ctr, kStatusIndex, 0, w);
      for (int i = tid; i < DK; i += kThreads) core[i] = __float2bfloat16_rn(0.f);
      continue;
    }
    const int kh = h / p.group;
    // The state rows go into registers first, so their latency overlaps the
    // wait for this task's projection tiles.
    const size_t sbase = ((size_t)slot * p.Hv + h) * (size_t)DK * DK;
    uint2 rawb[NR];
    float4 rawf[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const int v = (j * kWarps + warp) * RPW + rw;
      const size_t off = sbase + (size_t)v * DK + sub * 4;
      if (STATE_BF16)
        rawb[j] = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.ssm_state) + off);
      else
        rawf[j] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.ssm_state) + off);
    }
    if (tid == 0) {
      const unsigned long long* ctrs[6] = {
          &p.ctr->tile_done[(kh * DK) / kTileM],
          &p.ctr->tile_done[(p.Hk * DK + kh * DK) / kTileM],
          &p.ctr->tile_done[(2 * p.Hk * DK + h * DK) / kTileM],
          &p.ctr->tile_done[(p.C + h * DK) / kTileM],
          &p.ctr->tile_done[p.tiles_qkvz + h / kTileM],
          &p.ctr->tile_done[p.tiles_qkvz + (p.Hv + h) / kTileM]};
      sm.flag = wait_counters(p, ctrs, 6, (unsigned long long)(L + 1), kWaitTile);
      if ((p.debug_flags & kDebugTimeline) && task == t0) p.ctr->tl_cta[cta][TL_REC_WAITED] = globaltimer_ns();
    }
    __syncthreads();
    if (!sm.flag) return false;
    const float* actw = p.act + (size_t)w * p.Nqkvz;
    for (int i = tid; i < DK; i += kThreads) {
      sm.v[i] = ld_cg_f(actw + 2 * p.Hk * DK + h * DK + i);
      sm.z[i] = ld_cg_f(actw + p.C + h * DK + i);
    }
    const float4 k4 = ld_cg_f4(actw + p.Hk * DK + kh * DK + sub * 4);
    const float4 q4 = ld_cg_f4(actw + kh * DK + sub * 4);
    const float bv = ld_cg_f(p.act_ba + (size_t)w * p.Nba + h);
    const float av = ld_cg_f(p.act_ba + (size_t)w * p.Nba + p.Hv + h);
    const float sp_in = av + bf16_to_f(p.dt_bias[h]);
    const float sp = sp_in > 20.f ? sp_in : log1pf(expf(sp_in));
    const float g = -expf(p.A_log[h]) * sp;
    const float eg = expf(g);
    const float beta = 1.0f / (1.0f + expf(-bv));
    __syncthreads();

    float s[NR][4];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      if (STATE_BF16) {
        s[j][0] = bf16_lo(rawb[j].x); s[j][1] = bf16_hi(rawb[j].x);
        s[j][2] = bf16_lo(rawb[j].y); s[j][3] = bf16_hi(rawb[j].y);
      } else {
        s[j][0] = rawf[j].x; s[j][1] = rawf[j].y; s[j][2] = rawf[j].z; s[j][3] = rawf[j].w;
      }
    }
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const int v = (j * kWarps + warp) * RPW + rw;
      float e[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) e[c] = eg * s[j][c];
      float a = e[0] * k4.x;
      a = fmaf(e[1], k4.y, a); a = fmaf(e[2], k4.z, a); a = fmaf(e[3], k4.w, a);
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      const float u = beta * (sm.v[v] - a);
      e[0] = fmaf(k4.x, u, e[0]); e[1] = fmaf(k4.y, u, e[1]);
      e[2] = fmaf(k4.z, u, e[2]); e[3] = fmaf(k4.w, u, e[3]);
      float ov = e[0] * q4.x;
      ov = fmaf(e[1], q4.y, ov); ov = fmaf(e[2], q4.z, ov); ov = fmaf(e[3], q4.w, ov);
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) ov += __shfl_xor_sync(0xffffffffu, ov, o);
      const size_t off = sbase + (size_t)v * DK + sub * 4;
      if (STATE_BF16) {
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.ssm_state) + off) =
            make_uint2(pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]));
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.ssm_state) + off) =
            make_float4(e[0], e[1], e[2], e[3]);
      }
      if (sub == 0) sm.o[v] = ov;
    }
    __syncthreads();
    if (warp == 0) {
      float q = 0.f;
      for (int i = lane; i < DK; i += 32) q = fmaf(sm.o[i], sm.o[i], q);
      q = warp_sum(q);
      if (lane == 0) sm.red[0] = 1.0f / sqrtf(q / (float)DK + p.gnorm_eps);
    }
    __syncthreads();
    const float rn = sm.red[0];
    for (int i = tid; i < DK; i += kThreads)
      core[i] = __float2bfloat16_rn(sm.o[i] * rn * bf16_to_f(p.gnorm_w[i]) * silu_f(sm.z[i]));
    __syncthreads();
  }
  return true;
}

}  // namespace gdn
