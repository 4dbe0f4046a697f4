// Phases of the persistent GDN decode-step launch that do not depend on how
// the projection runs: the residual add and normalisation helpers, the end of
// the norm hand-off, and the per-(row, value head) task: partial reduction,
// conv update + SiLU, q/k L2 norm, the gated delta rule and the gated
// RMSNorm.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Every array is 16-byte aligned: several are accessed with 16-byte vectors.
struct SmemPhases {
  alignas(16) float rstd[kMaxRows];
  alignas(16) float red[kWarps];
  unsigned char tiles[kMaxTiles];  // partials per projection tile (the plan's, staged)
  int L;                 // launch number on this workspace
  int flag;              // CTA-wide decision (set by thread 0, cleared by any thread that gives up)
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
// The norm hand-off's end: every CTA's sums (polled as tagged words of this launch), rstd
// per row (Gemma RMSNorm: rstd = 1/sqrt(mean(r^2) + eps)). The sums are added
// in CTA order, so every CTA forms the same rstd bit for bit.
// ---------------------------------------------------------------------------
static __device__ __forceinline__ bool phase_wait_rstd(const StepParams& p, SmemPhases& sm, int L) {
  const int W = p.rows, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) sm.flag = 1;
  __syncthreads();
  for (int w = warp; w < W; w += kWarps) {
    // lane l holds CTAs l, l + 32, ...: all in flight at once
    constexpr int M = (kMaxCtas + 31) / 32;
    const unsigned long long* src = p.norm_part + w * p.num_ctas + lane;
    const int n = lane < p.num_ctas ? (p.num_ctas - lane + 31) / 32 : 0;
    unsigned long long v[M];
#pragma unroll
    for (int m = 0; m < M; ++m) v[m] = m < n ? ld_tagged(src + 32 * m) : 0ull;
    if (!poll_tagged<M>(p, v, src, 32, n, L, kWaitNorm)) sm.flag = 0;
    float s = 0.f;
#pragma unroll
    for (int m = 0; m < M; ++m)
      if (m < n) s += tagged_value(v[m]);
    s = warp_sum(s);
    if (lane == 0) sm.rstd[w] = 1.0f / sqrtf(s / (float)p.H + p.norm_eps);
  }
  tl_stamp(p, TL_NORM_IN);
  __syncthreads();
  return sm.flag != 0;
}

__device__ __forceinline__ bool row_is_live(const StepParams& p, int slot) {
  return slot > 0 && slot < p.num_slots;
}

// Synchronise the threads of a group: the whole CTA (barrier 0), one warp, or
// another group of whole warps (named barrier 1).
template <int NT>
__device__ __forceinline__ void group_sync() {
  if (NT == kThreads)
    __syncthreads();
  else if (NT == 32)
    __syncwarp();
  else
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");  // callers reach it with converged warps
}

// Shared memory of one recurrence task.
struct SmemTask {
  alignas(16) float q[128];     // q^ (after conv + SiLU, L2 norm, q_scale)
  alignas(16) float k[128];     // k^
  alignas(16) float v[128];     // v after conv + SiLU
  alignas(16) float z[128];     // z (bf16 projection)
  alignas(16) float o[128];     // o = S q
  alignas(16) float cnew[2 * 128][3];  // new q/k conv taps, written by the group's last reader
  float ba[2];                  // b, a (bf16 projections)
  float red[kWarps];
  int last;
};

// ---------------------------------------------------------------------------
// The recurrence: per (row w, value head h) task, all of the layer front after the
// projections for that head:
//   * the task's 4*dk + 2 projection outputs (q, k of key head kh = h / G; v,
//     z of head h; b, a) as the sum of the tiles' partials in slot order,
//     rounded to bf16
//   * causal conv update + SiLU over its q, k, v channels (old taps read,
//     new taps [s1, s2, p]); the v channels are this task's alone; the q/k
//     channels are shared by the G value heads of kh, and the last of those
//     G tasks to read the old taps writes the new ones
//   * q^ = q / sqrt(sum q^2 + eps) * q_scale, k^ likewise without the scale
//   * g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)
//   * S <- e^g S;  u = beta (v - S k^);  S <- S + u k^T;  o = S q^   (S[v][k])
//   * core = bf16(o * rsqrt(mean(o^2) + eps) * w_g * silu(z))
// Each warp owns whole state rows S[v][:], so S k and S q are reductions
// over one row's lanes (sgl-amd-mono #89, Modifications, gdn.py row: f32
// recurrence, state stored in f32 or bf16 in place; pad rows write a zero
// core row and no state).
// ---------------------------------------------------------------------------
// A thread's share of one (row, value head) state tile: NR rows, CH chunks
// of 4 elements of each. Eight lanes share a row; lane sub holds chunks
// sub, sub + 8, sub + 16, ... so that the eight lanes of a row read 128
// contiguous bytes per chunk, and a row's dot products reduce in 3 shuffle
// rounds (a warp holds 4 rows at a time).
template <int DK>
struct StateRegs {
  static constexpr int LPR = 8;                   // lanes per state row
  static constexpr int CH = DK / (4 * LPR);       // chunks of 4 elements per lane and row
  static constexpr int RPW = 32 / LPR;            // rows per warp per step
  static constexpr int NR = DK / (kWarps * RPW);  // rows per lane (dv == dk)
  static_assert(NR >= 1 && CH >= 1, "state layout");
  uint2 b[NR][CH];   // bf16 state
  float4 f[NR][CH];  // f32 state
};

// The CTA's recurrence tasks: (sequence, value head h) = task / Hv, task % Hv
// for task in [t0, t1); a sequence is one row when decoding, `tokens` rows
// in a verify step.
__device__ __forceinline__ void task_range(const StepParams& p, int& t0, int& t1) {
  const int T = p.rows / p.tokens * p.Hv;
  t0 = (int)(((long long)blockIdx.x * T) / p.num_ctas);
  t1 = (int)(((long long)(blockIdx.x + 1) * T) / p.num_ctas);
}

// Issue the loads of this thread's share of a task's state tile (nothing for
// a pad row).
template <int DK, bool STATE_BF16>
__device__ __forceinline__ void load_state(const StepParams& p, int task, StateRegs<DK>& r) {
  constexpr int NR = StateRegs<DK>::NR, CH = StateRegs<DK>::CH, LPR = StateRegs<DK>::LPR;
  constexpr int RPW = StateRegs<DK>::RPW;
  const int sq = task / p.Hv, h = task - sq * p.Hv;  // sequence, value head
  const int slot = p.idx[sq];
  if (!row_is_live(p, slot)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t sbase = ((size_t)slot * p.Hv + h) * (size_t)DK * DK;
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    const int v = (j * kWarps + warp) * RPW + lane / LPR;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const size_t off = sbase + (size_t)v * DK + (lane % LPR + LPR * c) * 4;
      if (STATE_BF16)
        r.b[j][c] = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.ssm_state) + off);
      else
        r.f[j][c] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.ssm_state) + off);
    }
  }
}

// `raw` holds the first task's state when `have_first` (loaded early, so
// that its latency hides under the projection); later tasks load into it.
// tile_cnt[t]: the partials of projection tile t (the plan's table, or its
// copy in shared memory).
// sm.flag is 1 on entry (every earlier phase of the launch succeeded); a
// thread whose wait runs out clears it.
// MULTI (verify steps): a task is (sequence, value head) and runs the
// sequence's tokens in order; token t starts from the state (and conv taps)
// token t - 1 stored, and its state goes to its own slot idx_out[row]. The
// conv taps of a channel stay in its thread's registers from token to token;
// the state between tokens is the stored one (rounded to bf16 for a bf16
// state), held in `raw`. The q/k taps of a key-head group are written by its
// first value head's task (no counter: the input slot is never written).
template <int DK, bool STATE_BF16, bool MULTI = false>
__device__ __forceinline__ bool phase_recurrence(const StepParams& p, SmemPhases& sm, SmemTask& st, int L,
                                                 StateRegs<DK>& raw, bool have_first,
                                                 const unsigned char* tile_cnt) {
  constexpr int LPR = StateRegs<DK>::LPR;
  constexpr int RPW = StateRegs<DK>::RPW;
  constexpr int NR = StateRegs<DK>::NR;
  constexpr int CH = StateRegs<DK>::CH;
  static_assert(4 * DK <= kThreads, "task layout");
  const int cta = blockIdx.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int sub = lane % LPR, rw = lane / LPR;
  int t0, t1;
  task_range(p, t0, t1);
  const int TK = MULTI ? p.tokens : 1;
  for (int task = t0; task < t1; ++task) {
    const int sq = task / p.Hv, h = task - sq * p.Hv;  // sequence (one row when decoding), value head
    const int slot = p.idx[sq];
    bool live = row_is_live(p, slot);
    bool bad = slot >= p.num_slots;
    if (MULTI && live)
      for (int t = 0; t < TK; ++t) {
        const int o = p.idx_out[sq * TK + t];
        if (!(o > 0 && o < p.num_slots)) live = false, bad = true;
      }
    if (!live) {
      if (bad && h == 0 && tid == 0) record_error(p.ctr, kStatusIndex, 0, sq * TK);
      for (int i = tid; i < DK * TK; i += kThreads)
        p.core_out[(size_t)(sq * TK + i / DK) * p.Hv * DK + (size_t)h * DK + i % DK] = __float2bfloat16_rn(0.f);
      continue;
    }
    const int kh = h / p.group;
    // The state rows go into registers first, so their latency overlaps the
    // wait for the projections (the first task's were loaded earlier still).
    if (!(have_first && task == t0)) load_state<DK, STATE_BF16>(p, task, raw);
    // the conv taps of this thread's channel, carried from token to token (MULTI)
    float tap0 = 0.f, tap1 = 0.f, tap2 = 0.f;
#pragma unroll 1
    for (int tk = 0; tk < TK; ++tk) {
    const int w = sq * TK + tk;  // the row of this token
    const int oslot = MULTI ? p.idx_out[w] : slot;  // where its state goes
    __nv_bfloat16* core = p.core_out + (size_t)w * p.Hv * DK + (size_t)h * DK;
    const size_t sbase = ((size_t)oslot * p.Hv + h) * (size_t)DK * DK;
    // Per-head constants, also loaded now.
    const float A_log_h = p.A_log[h];
    const float dt_bias_h = bf16_to_f(p.dt_bias[h]);
    const float gw = tid < DK ? bf16_to_f(p.gnorm_w[tid]) : 0.f;
    // Projection row of each task output, its tile and row in the tile.
    auto proj_row = [&](int i) -> int {
      if (i < DK) return kh * DK + i;
      if (i < 2 * DK) return p.Hk * DK + kh * DK + (i - DK);
      if (i < 3 * DK) return 2 * p.Hk * DK + h * DK + (i - 2 * DK);
      if (i < 4 * DK) return p.C + h * DK + (i - 3 * DK);
      return p.Nqkvz + (i == 4 * DK ? h : p.Hv + h);
    };
    auto tile_of = [&](int n) -> int {
      return n < p.Nqkvz ? (n >> kTileShift) : p.tiles_qkvz + ((n - p.Nqkvz) >> kTileShift);
    };
    // Projection outputs, each the sum of its tile's partials in slot order,
    // polled as tagged words of this launch. Thread i < 4*dk takes output i
    // (q, k, v, z); b and a take one slot per lane of the last two warps.
    constexpr size_t kSlot = (size_t)kMaxRows * kTileM;
    constexpr int kMaxSlots = 24;  // partials per tile (the plan's bound)
    auto part_src = [&](int n, int& nc) {
      const int t = tile_of(n);
      const int r = (n < p.Nqkvz ? n : n - p.Nqkvz) & (kTileM - 1);
      nc = tile_cnt[t];
      return p.proj_part + ((size_t)t * p.max_contrib * kMaxRows + w) * kTileM + r;
    };
    const bool ba_warp = warp >= kWarps - 2;
    int ba_nc = 0;
    const unsigned long long* ba_src = nullptr;
    unsigned long long ba_w[1] = {0ull};
    if (ba_warp) {  // issued first: these lanes also have an output of their own
      ba_src = part_src(proj_row(4 * DK + (warp - (kWarps - 2))), ba_nc) + (size_t)lane * kSlot;
      if (lane < ba_nc) ba_w[0] = ld_tagged(ba_src);
    }
    if (tid < 4 * DK) {
      const int i = tid;
      const int n = proj_row(i);
      int nc;
      const unsigned long long* src = part_src(n, nc);
      uint2 cwv;
      if (i < 3 * DK) {  // old taps and weights of channel n
        if (tk == 0) {
          const __nv_bfloat16* cs = p.conv_state + ((size_t)slot * p.C + n) * 3;
          tap0 = bf16_to_f(cs[0]); tap1 = bf16_to_f(cs[1]); tap2 = bf16_to_f(cs[2]);
        }
        cwv = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)n * 4);
      }
      unsigned long long pw[kMaxSlots];
#pragma unroll
      for (int jj = 0; jj < kMaxSlots; ++jj) pw[jj] = jj < nc ? ld_tagged(src + (size_t)jj * kSlot) : 0ull;
      if (!poll_tagged<kMaxSlots>(p, pw, src, kSlot, nc, L, kWaitTile)) sm.flag = 0;
      if (i == 0 && (p.debug_flags & kDebugTimeline) && task == t0)
        p.ctr->tl_cta[cta][TL_REC_WAITED] = globaltimer_ns();
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < kMaxSlots; ++jj)
        if (jj < nc) acc += tagged_value(pw[jj]);
      const float pv = round_bf16(acc);
      float y2 = 0.f;  // y^2 of a q or k output, for the L2 norms
      if (i < 3 * DK) {
        const float c0 = tap0, c1 = tap1, c2 = tap2;
        tap0 = c1; tap1 = c2; tap2 = pv;  // the taps after this token
        float y = bf16_lo(cwv.x) * c0;
        y = fmaf(bf16_hi(cwv.x), c1, y);
        y = fmaf(bf16_lo(cwv.y), c2, y);
        y = fmaf(bf16_hi(cwv.y), pv, y);
        y = silu_f(y);
        if (i < DK) {
          st.q[i] = y;
        } else if (i < 2 * DK) {
          st.k[i - DK] = y;
        } else {
          st.v[i - 2 * DK] = y;
          __nv_bfloat16* cs = p.conv_state + ((size_t)oslot * p.C + n) * 3;  // this head's own channel
          cs[0] = __float2bfloat16_rn(c1);
          cs[1] = __float2bfloat16_rn(c2);
          cs[2] = __float2bfloat16_rn(pv);
        }
        if (i < 2 * DK) {
          y2 = y * y;
          if (MULTI) {
            if (h % p.group == 0) {  // the group's first value head writes its q/k taps
              __nv_bfloat16* cs = p.conv_state + ((size_t)oslot * p.C + n) * 3;
              cs[0] = __float2bfloat16_rn(c1);
              cs[1] = __float2bfloat16_rn(c2);
              cs[2] = __float2bfloat16_rn(pv);
            }
          } else {
            st.cnew[i][0] = c1;
            st.cnew[i][1] = c2;
            st.cnew[i][2] = pv;
          }
        }
      } else {
        st.z[i - 3 * DK] = pv;
      }
      if (warp < 2 * DK / 32) {  // whole warps of q (then k) outputs: their sums of squares
        y2 = warp_sum(y2);
        if (lane == 0) st.red[warp] = y2;
      }
    }
    if (ba_warp) {
      if (!poll_tagged<1>(p, ba_w, ba_src, 0, lane < ba_nc ? 1 : 0, L, kWaitTile)) sm.flag = 0;
      const float v = tagged_value(ba_w[0]);
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < kMaxSlots; ++jj) {  // slot order, as for the other outputs
        const float x = __shfl_sync(0xffffffffu, v, jj);
        if (jj < ba_nc) acc += x;
      }
      if (lane == 0) st.ba[warp - (kWarps - 2)] = round_bf16(acc);
    }
    __syncthreads();
    if (!sm.flag) return false;
    unsigned int group_old = 0;
    if (!MULTI && tid == 0) {
      // Every thread's reads of the old q/k taps are done: their values were
      // used before the barrier above, so no later store can reach them. The
      // count needs no release (a release here waits for every store the CTA
      // has in flight); its result is needed only at the end.
      group_old = atom_add_relaxed_u32(&p.ctr->conv_group[w][kh], 1u);
      if ((p.debug_flags & kDebugTimeline) && task == t0) p.ctr->tl_cta[cta][TL_REC_INPUTS] = globaltimer_ns();
    }
    // L2 norms of q and k from the per-warp sums of squares, added in warp
    // order (the same arithmetic in every thread, and in the pipelined phase)
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int i = 0; i < DK / 32; ++i) {
      sq += st.red[i];
      sk += st.red[DK / 32 + i];
    }
    const float inv_q = (1.0f / sqrtf(sq + p.l2_eps)) * p.q_scale;
    const float inv_k = 1.0f / sqrtf(sk + p.l2_eps);
    float4 k4[CH], q4[CH];  // this lane's chunks of k^ and q^
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const float4 kq = *reinterpret_cast<const float4*>(&st.k[(sub + LPR * c) * 4]);
      const float4 qq = *reinterpret_cast<const float4*>(&st.q[(sub + LPR * c) * 4]);
      k4[c] = make_float4(kq.x * inv_k, kq.y * inv_k, kq.z * inv_k, kq.w * inv_k);
      q4[c] = make_float4(qq.x * inv_q, qq.y * inv_q, qq.z * inv_q, qq.w * inv_q);
    }
    const float sp_in = st.ba[1] + dt_bias_h;
    const float sp = sp_in > 20.f ? sp_in : log1pf(expf(sp_in));
    const float g = -expf(A_log_h) * sp;
    const float eg = expf(g);
    const float beta = 1.0f / (1.0f + expf(-st.ba[0]));

    float4 s[NR][CH];
#pragma unroll
    for (int j = 0; j < NR; ++j)
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        if (STATE_BF16)
          s[j][c] = make_float4(bf16_lo(raw.b[j][c].x), bf16_hi(raw.b[j][c].x), bf16_lo(raw.b[j][c].y),
                                bf16_hi(raw.b[j][c].y));
        else
          s[j][c] = raw.f[j][c];
      }
    // S k over all rows of this lane at once (independent butterflies)
    float a[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      a[j] = 0.f;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        s[j][c].x *= eg; s[j][c].y *= eg; s[j][c].z *= eg; s[j][c].w *= eg;
        a[j] = fmaf(s[j][c].x, k4[c].x, a[j]);
        a[j] = fmaf(s[j][c].y, k4[c].y, a[j]);
        a[j] = fmaf(s[j][c].z, k4[c].z, a[j]);
        a[j] = fmaf(s[j][c].w, k4[c].w, a[j]);
      }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1)
#pragma unroll
      for (int j = 0; j < NR; ++j) a[j] += __shfl_xor_sync(0xffffffffu, a[j], o);
    float ov[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const int v = (j * kWarps + warp) * RPW + rw;
      const float u = beta * (st.v[v] - a[j]);
      ov[j] = 0.f;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        s[j][c].x = fmaf(k4[c].x, u, s[j][c].x); s[j][c].y = fmaf(k4[c].y, u, s[j][c].y);
        s[j][c].z = fmaf(k4[c].z, u, s[j][c].z); s[j][c].w = fmaf(k4[c].w, u, s[j][c].w);
        ov[j] = fmaf(s[j][c].x, q4[c].x, ov[j]);
        ov[j] = fmaf(s[j][c].y, q4[c].y, ov[j]);
        ov[j] = fmaf(s[j][c].z, q4[c].z, ov[j]);
        ov[j] = fmaf(s[j][c].w, q4[c].w, ov[j]);
        const size_t off = sbase + (size_t)v * DK + (sub + LPR * c) * 4;
        if (STATE_BF16) {
          const uint2 sb = make_uint2(pack_bf16x2(s[j][c].x, s[j][c].y), pack_bf16x2(s[j][c].z, s[j][c].w));
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.ssm_state) + off) = sb;
          if (MULTI) raw.b[j][c] = sb;  // the next token starts from the stored state
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.ssm_state) + off) = s[j][c];
          if (MULTI) raw.f[j][c] = s[j][c];
        }
      }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1)
#pragma unroll
      for (int j = 0; j < NR; ++j) ov[j] += __shfl_xor_sync(0xffffffffu, ov[j], o);
#pragma unroll
    for (int j = 0; j < NR; ++j)
      if (sub == 0) st.o[(j * kWarps + warp) * RPW + rw] = ov[j];
    if (tid == 0) st.last = !MULTI && ((group_old + 1) % (unsigned)p.group) == 0;
    __syncthreads();
    float rn = 0.f;
    if (warp < DK / 32) {  // the warps that write core: each sums o^2 itself (same order)
      float q = 0.f;
#pragma unroll
      for (int i = 0; i < DK / 32; ++i) q = fmaf(st.o[i * 32 + lane], st.o[i * 32 + lane], q);
      q = warp_sum(q);
      rn = 1.0f / sqrtf(q / (float)DK + p.gnorm_eps);
    }
    if (st.last) {  // the last reader of the group writes the new q/k taps
      for (int i = tid; i < 2 * DK; i += kThreads) {
        const int n = proj_row(i);
        __nv_bfloat16* cs = p.conv_state + ((size_t)oslot * p.C + n) * 3;
        cs[0] = __float2bfloat16_rn(st.cnew[i][0]);
        cs[1] = __float2bfloat16_rn(st.cnew[i][1]);
        cs[2] = __float2bfloat16_rn(st.cnew[i][2]);
      }
    }
    if (tid < DK) core[tid] = __float2bfloat16_rn(st.o[tid] * rn * gw * silu_f(st.z[tid]));
    if ((p.debug_flags & kDebugTimeline) && task == t0 && tid == 0)
      p.ctr->tl_cta[cta][TL_REC_STATE] = globaltimer_ns();
    __syncthreads();
    }  // tokens
  }
  return true;
}

}  // namespace gdn
