// The recurrence phase of a CTA with two or more (row, value head) tasks,
// with the state traffic moved off the threads and the input loads issued a
// task ahead:
//   * state tiles (DK x DK contiguous elements per task) live in a ring of
//     three shared-memory buffers, task j in buffer j % 3: bulk copies bring
//     task j + 2's tile in while task j runs; the threads update a tile in
//     place; a bulk copy takes it back out (task 0's tile was prefetched
//     into L2 under the projection);
//   * task 0's projection partials are polled as tagged words of the
//     launch, so it starts as soon as its own tiles are done; task j + 1's
//     (and its old conv taps) are loaded while task j updates its state,
//     once every CTA has counted itself on the projection counter (a release
//     after its last partial): they are then final and are read as plain f32
//     values (the low halves of the tagged words), with half the registers
//     and no tags to check;
//   * the key-head group's counter of task j is read back at task j + 1, and
//     the new q/k taps of task j (held in the registers of their threads)
//     are written then if j was the group's last reader.
// Every value is computed with the single-task phase's arithmetic in the
// same order (the same state layout per row, the same sums), so a row's
// results do not depend on which path ran it. All threads pass the same
// barriers; a wait that runs out stops the phase at the next barrier (the
// error is recorded) after the copies in flight have landed.
#pragma once

#include <type_traits>

#include "gdn_phases.cuh"
#include "gdn_tc_ptx.cuh"

namespace gdn {

constexpr uint32_t kWaitState = 8;  // error-word id: a state tile's copy into shared memory

// One task's inputs (two, alternating between tasks).
struct StagedTask {
  alignas(16) float q[128];  // q, k after conv + SiLU (not yet normalised)
  alignas(16) float k[128];
  alignas(16) float v[128];  // v after conv + SiLU
  alignas(16) float z[128];  // z (bf16 projection)
  alignas(16) float o[128];  // o = S q^
  float red[kWarps];         // per-warp sums of q^2 (warps 0 .. dk/32-1), then k^2
  float eg, beta;            // the head's gates e^g and beta
  int last;                  // the previous task was its key-head group's last reader
};
constexpr int kMaxStagedTasks = 64;  // (row, value head) tasks of one CTA the staged phase takes
constexpr int kBulkTid = 128;        // the thread that issues and waits for the state tiles' bulk copies
// A task's indices, worked out once per phase (no divisions in the loop).
struct StagedTaskIdx {
  short w, h, kh;      // row, value head, key head
  unsigned char same;  // the same (row, key head) as the task before: same q/k
  unsigned char pad;
};
// The state slots of the launch's rows and the CTA's tasks (once per phase).
struct StagedSlots {
  int idx[kMaxRows];
  int go;  // every CTA's projection partials are stored
  StagedTaskIdx task[kMaxStagedTasks];
};

template <int DK, bool STATE_BF16>
struct StagedLayout {
  static constexpr uint32_t kStateBytes = DK * DK * (STATE_BF16 ? 2 : 4);
  static constexpr int kBufs = 3;
  static constexpr size_t kBytes = kBufs * (size_t)kStateBytes + 2 * sizeof(StagedTask) + sizeof(StagedSlots);
  static_assert(kStateBytes % 16 == 0, "bulk copy size");
};

// The shared memory the staged phase needs.
template <int DK, bool STATE_BF16>
__host__ __device__ constexpr size_t staged_recurrence_bytes() {
  return StagedLayout<DK, STATE_BF16>::kBytes;
}

// A thread's loads of one task's inputs: the partials of output `i` = tid
// (q, k, v, z) and its conv taps and weights; b and a one slot per lane of
// the last two warps.
struct StagedLoads {
  static constexpr int kMaxSlots = 24;  // partials per tile (the plan's bound)
  uint32_t pv[kMaxSlots];    // the partials' f32 bits
  int nc;
  uint32_t bav;              // b or a: this lane's slot
  int ba_nc;
  uint2 cwv;                 // conv weights of the channel
  __nv_bfloat16 tap[3];      // its old taps
  float A_log;               // the head's constants
  __nv_bfloat16 dt_bias;
};

// The L2 prefetch of a task's state tile (nothing for a pad row).
template <int DK, bool STATE_BF16>
__device__ __forceinline__ void prefetch_state_l2(const StepParams& p, int task) {
  using SL = StagedLayout<DK, STATE_BF16>;
  const int w = task / p.Hv, h = task - w * p.Hv;
  const int slot = p.idx[w];
  if (!row_is_live(p, slot)) return;
  tc::prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(p.ssm_state) + ((size_t)slot * p.Hv + h) * SL::kStateBytes,
                       SL::kStateBytes);
}

template <int DK, bool STATE_BF16>
__device__ bool phase_recurrence_staged(const StepParams& p, uint8_t* ring, uint64_t* sbar, int L, int t0,
                                        int t1, const unsigned char* tile_cnt) {
  using SL = StagedLayout<DK, STATE_BF16>;
  constexpr int LPR = StateRegs<DK>::LPR;
  constexpr int RPW = StateRegs<DK>::RPW;
  constexpr int NR = StateRegs<DK>::NR;
  constexpr int CH = StateRegs<DK>::CH;
  constexpr int kMaxSlots = StagedLoads::kMaxSlots;
  constexpr size_t kSlot = (size_t)kMaxRows * kTileM;
  static_assert(4 * DK <= kThreads, "task layout");
  const int cta = blockIdx.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int sub = lane % LPR, rw = lane / LPR;
  const int n = t1 - t0;
  auto sbuf = [&](int j) { return ring + (size_t)(j % SL::kBufs) * SL::kStateBytes; };  // task j's tile
  StagedTask* tb = reinterpret_cast<StagedTask*>(ring + SL::kBufs * (size_t)SL::kStateBytes);
  StagedSlots* sst = reinterpret_cast<StagedSlots*>(tb + 2);
  int* sidx = sst->idx;  // the rows' state slots
  if (tid < p.rows) sidx[tid] = p.idx[tid];
  if (tid < n) {  // task tid's indices
    const int task = t0 + tid, w = task / p.Hv, h = task - w * p.Hv, kh = h / p.group;
    const int pt = task - 1, pw = pt / p.Hv, pkh = (pt - pw * p.Hv) / p.group;
    sst->task[tid] = StagedTaskIdx{(short)w, (short)h, (short)kh, (unsigned char)(tid > 0 && pw == w && pkh == kh), 0};
  }
  __syncthreads();
  const bool ba_warp = warp >= kWarps - 2;

  auto proj_row = [&](int i, int h, int kh) -> int {
    if (i < DK) return kh * DK + i;
    if (i < 2 * DK) return p.Hk * DK + kh * DK + (i - DK);
    if (i < 3 * DK) return 2 * p.Hk * DK + h * DK + (i - 2 * DK);
    if (i < 4 * DK) return p.C + h * DK + (i - 3 * DK);
    return p.Nqkvz + (i == 4 * DK ? h : p.Hv + h);
  };
  auto part_src = [&](int n_row, int w, int& nc) {
    const int t = n_row < p.Nqkvz ? (n_row >> kTileShift) : p.tiles_qkvz + ((n_row - p.Nqkvz) >> kTileShift);
    const int r = (n_row < p.Nqkvz ? n_row : n_row - p.Nqkvz) & (kTileM - 1);
    nc = tile_cnt[t];
    return p.proj_part + ((size_t)t * p.max_contrib * kMaxRows + w) * kTileM + r;
  };

  auto state_src = [&](int slot, int h) {
    return reinterpret_cast<uint8_t*>(p.ssm_state) + ((size_t)slot * p.Hv + h) * SL::kStateBytes;
  };
  // The bulk thread: the bulk copy of task j's state tile into its buffer,
  // completing on that buffer's mbarrier. Returns whether one was issued
  // (not for a pad row).
  auto issue_state = [&](int j) -> bool {
    const int w = sst->task[j].w, h = sst->task[j].h;
    const int slot = sidx[w];
    if (!row_is_live(p, slot)) return false;
    uint64_t* bar = &sbar[j % SL::kBufs];
    tc::mbar_arrive_expect_tx(bar, SL::kStateBytes);
    tc::bulk_load(sbuf(j), state_src(slot, h), SL::kStateBytes, bar);
    return true;
  };
  // Task j reads the same q/k channels (row and key head) as task j - 1:
  // their conv + SiLU outputs are the previous task's, copied, not reloaded.
  auto same_qk = [&](int j) { return sst->task[j].same != 0; };
  // Every thread: issue its loads of task j's inputs (nothing for a pad row,
  // or when `real` is false: then the fields are only cleared).
  StagedLoads ld;
  auto issue_inputs = [&](int j, bool real) {
    const int jj0 = real ? j : 0;
    const int w = sst->task[jj0].w, h = sst->task[jj0].h, kh = sst->task[jj0].kh;
    const int slot = real ? sidx[w] : 0;
    // every field is assigned on every path (and the call made after every
    // task), so nothing of a task's loads stays live past its use
    ld.nc = 0;
    ld.ba_nc = 0;
    ld.bav = 0u;
#pragma unroll
    for (int jj = 0; jj < kMaxSlots; ++jj) ld.pv[jj] = 0u;
    ld.cwv = make_uint2(0u, 0u);
    ld.tap[0] = ld.tap[1] = ld.tap[2] = __float2bfloat16_rn(0.f);
    ld.A_log = 0.f;
    ld.dt_bias = __float2bfloat16_rn(0.f);
    if (!row_is_live(p, slot)) return;
    ld.A_log = p.A_log[h];
    ld.dt_bias = p.dt_bias[h];
    // a partial's f32 bits: the low half of its tagged word
    auto ld_part = [](const unsigned long long* q) { return ld_relaxed_u32(reinterpret_cast<const unsigned*>(q)); };
    if (ba_warp) {  // first: these lanes also have an output of their own
      const unsigned long long* bsrc =
          part_src(proj_row(4 * DK + (warp - (kWarps - 2)), h, kh), w, ld.ba_nc) + (size_t)lane * kSlot;
      if (lane < ld.ba_nc) ld.bav = ld_part(bsrc);
    }
    if (tid < 4 * DK && !(tid < 2 * DK && same_qk(j))) {
      const int nr = proj_row(tid, h, kh);
      const unsigned long long* src = part_src(nr, w, ld.nc);
#pragma unroll
      for (int jj = 0; jj < kMaxSlots; ++jj)
        if (jj < ld.nc) ld.pv[jj] = ld_part(src + (size_t)jj * kSlot);
      if (tid < 3 * DK) {
        const __nv_bfloat16* cs = p.conv_state + ((size_t)slot * p.C + nr) * 3;
        ld.tap[0] = cs[0];
        ld.tap[1] = cs[1];
        ld.tap[2] = cs[2];
        ld.cwv = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)nr * 4);
      }
    }
  };

  // bulk copies in flight into each buffer (the bulk thread: its warp has no
  // core row to write, so the copies stay off the path of the next task) and
  // the buffers' mbarrier phases (every thread)
  uint32_t pending = 0, ph = 0;
  if (tid == kBulkTid) {
    tc::fence_proxy_async_smem();  // the ring's earlier generic accesses before the copies
    for (int j = 0; j < min(n, SL::kBufs); ++j)
      if (issue_state(j)) pending |= 1u << j;
  }
  bool ok = true;
  // timeline (test hook): stamps 16 + 4 j + k of the first four tasks
  auto stamp = [&](int j, int k) {
    if ((p.debug_flags & kDebugTimeline) && j < 4 && tid == 0) p.ctr->tl_cta[cta][TL_TASK + 4 * j + k] = globaltimer_ns();
  };
  const float gw = tid < DK ? bf16_to_f(p.gnorm_w[tid]) : 0.f;
  // Task j's inputs (its row live): partial sums, conv update + SiLU, per-warp
  // sums of squares into tb[j & 1], this thread's new q/k taps into c1, c2,
  // pvq. Task 0 (TAGGED): its partials polled as tagged words of this launch,
  // so it starts as soon as its own tiles are done; later tasks: loaded once
  // the projection counter was seen complete, so read as plain f32 values.
  struct TaggedLoads {
    unsigned long long pw[kMaxSlots];
    const unsigned long long* src;
    unsigned long long baw[1];
    const unsigned long long* ba_src;
  } ld0;
  float c1 = 0.f, c2 = 0.f, pvq = 0.f;    // this task's new q/k taps (threads < 2 dk)
  float nt0 = 0.f, nt1 = 0.f, nt2 = 0.f;  // the previous task's
  auto gather = [&](int j, auto tagged) {
    constexpr bool TAGGED = decltype(tagged)::value;
    const int w = sst->task[j].w, h = sst->task[j].h, kh = sst->task[j].kh;
    const int slot = sidx[w];
    StagedTask& T = tb[j & 1];
    if (tid < 2 * DK && same_qk(j)) {
      // q/k as the previous task had them (same values, so the same sums)
      const StagedTask& P = tb[(j - 1) & 1];
      const float y = tid < DK ? P.q[tid] : P.k[tid - DK];
      if (tid < DK)
        T.q[tid] = y;
      else
        T.k[tid - DK] = y;
      c1 = nt0;
      c2 = nt1;
      pvq = nt2;
      const float y2 = warp_sum(y * y);
      if (lane == 0) T.red[warp] = y2;
    } else if (tid < 4 * DK) {
      const int i = tid;
      float acc = 0.f;
      if constexpr (TAGGED) {
        if (!poll_tagged<kMaxSlots>(p, ld0.pw, ld0.src, kSlot, ld.nc, L, kWaitTile)) ok = false;
        if (i == 0 && (p.debug_flags & kDebugTimeline)) p.ctr->tl_cta[cta][TL_REC_WAITED] = globaltimer_ns();
#pragma unroll
        for (int jj = 0; jj < kMaxSlots; ++jj)
          if (jj < ld.nc) acc += tagged_value(ld0.pw[jj]);
      } else {
#pragma unroll
        for (int jj = 0; jj < kMaxSlots; ++jj)
          if (jj < ld.nc) acc += __uint_as_float(ld.pv[jj]);
      }
      const float pv = round_bf16(acc);
      float y2 = 0.f;
      if (i < 3 * DK) {
        const float c0 = bf16_to_f(ld.tap[0]);
        c1 = bf16_to_f(ld.tap[1]);
        c2 = bf16_to_f(ld.tap[2]);
        float y = bf16_lo(ld.cwv.x) * c0;
        y = fmaf(bf16_hi(ld.cwv.x), c1, y);
        y = fmaf(bf16_lo(ld.cwv.y), c2, y);
        y = fmaf(bf16_hi(ld.cwv.y), pv, y);
        y = silu_f(y);
        if (i < DK) {
          T.q[i] = y;
        } else if (i < 2 * DK) {
          T.k[i - DK] = y;
        } else {
          T.v[i - 2 * DK] = y;
          __nv_bfloat16* cs = p.conv_state + ((size_t)slot * p.C + proj_row(i, h, kh)) * 3;  // own channel
          cs[0] = __float2bfloat16_rn(c1);
          cs[1] = __float2bfloat16_rn(c2);
          cs[2] = __float2bfloat16_rn(pv);
        }
        if (i < 2 * DK) {
          y2 = y * y;
          pvq = pv;
        }
      } else {
        T.z[i - 3 * DK] = pv;
      }
      if (warp < 2 * DK / 32) {
        y2 = warp_sum(y2);
        if (lane == 0) T.red[warp] = y2;
      }
    }
    if (ba_warp) {
      float v;
      if constexpr (TAGGED) {
        if (!poll_tagged<1>(p, ld0.baw, ld0.ba_src, 0, lane < ld.ba_nc ? 1 : 0, L, kWaitTile)) ok = false;
        v = tagged_value(ld0.baw[0]);
      } else {
        v = __uint_as_float(ld.bav);
      }
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < kMaxSlots; ++jj) {  // slot order, as for the other outputs
        const float x = __shfl_sync(0xffffffffu, v, jj);
        if (jj < ld.ba_nc) acc += x;
      }
      if (lane == 0) {  // the head's gates, once (the one-task phase's arithmetic)
        const float x = round_bf16(acc);
        if (warp == kWarps - 2) {
          T.beta = 1.0f / (1.0f + expf(-x));  // b
        } else {
          const float sp_in = x + bf16_to_f(ld.dt_bias);  // a
          const float sp = sp_in > 20.f ? sp_in : log1pf(expf(sp_in));
          const float g = -expf(ld.A_log) * sp;
          T.eg = expf(g);
        }
      }
    }
  };
  // task 0: its loads as tagged words (the non-partial ones into `ld`), then
  // its inputs
  issue_inputs(0, false);  // clears `ld`
  {
    const int w0 = sst->task[0].w, h0 = sst->task[0].h, kh0 = sst->task[0].kh;
    const int slot0 = sidx[w0];
    if (row_is_live(p, slot0)) {
      ld.A_log = p.A_log[h0];
      ld.dt_bias = p.dt_bias[h0];
      if (ba_warp) {
        ld0.ba_src = part_src(proj_row(4 * DK + (warp - (kWarps - 2)), h0, kh0), w0, ld.ba_nc) + (size_t)lane * kSlot;
        ld0.baw[0] = lane < ld.ba_nc ? ld_tagged(ld0.ba_src) : 0ull;
      }
      if (tid < 4 * DK) {
        const int nr = proj_row(tid, h0, kh0);
        ld0.src = part_src(nr, w0, ld.nc);
#pragma unroll
        for (int jj = 0; jj < kMaxSlots; ++jj) ld0.pw[jj] = jj < ld.nc ? ld_tagged(ld0.src + (size_t)jj * kSlot) : 0ull;
        if (tid < 3 * DK) {
          const __nv_bfloat16* cs = p.conv_state + ((size_t)slot0 * p.C + nr) * 3;
          ld.tap[0] = cs[0];
          ld.tap[1] = cs[1];
          ld.tap[2] = cs[2];
          ld.cwv = *reinterpret_cast<const uint2*>(p.conv_w + (size_t)nr * 4);
        }
      }
      gather(0, std::true_type());
    }
  }
  unsigned int group_old = 0;  // thread 0: the previous task's group counter
  bool prev_live = false;
  int prev_slot = 0, prev_row = 0;
  for (int j = 0; j < n && ok; ++j) {
    const int w = sst->task[j].w, h = sst->task[j].h, kh = sst->task[j].kh;
    const int slot = sidx[w];
    const bool live = row_is_live(p, slot);
    StagedTask& T = tb[j & 1];
    __nv_bfloat16* core = p.core_out + (size_t)w * p.Hv * DK + (size_t)h * DK;
    const int b = j % SL::kBufs;  // the tile's buffer and its mbarrier
    if (j > 0) {  // (task 0's inputs were gathered before the loop)
      c1 = c2 = pvq = 0.f;
      if (live) gather(j, std::false_type());
    }
    if (live) {
      stamp(j, 0);  // inputs in
      // ---- this task's state tile in shared memory (bounded wait)
      if (ok) {
        const uint32_t par = (ph >> b) & 1u;
        bool landed = tc::mbar_try_wait(&sbar[b], par);
        if (!landed) {
          const unsigned long long c0 = globaltimer_ns();
          for (uint32_t it = 1;; ++it) {
            if (tc::mbar_try_wait(&sbar[b], par)) { landed = true; break; }
            if ((it & 63) == 0) {
              if ((ld_relaxed_u32(&p.ctr->error) >> 24) == kStatusDeadline) break;
              if (globaltimer_ns() - c0 > p.deadline_ns) {
                record_error(p.ctr, kStatusDeadline, kWaitState, cta);
                break;
              }
            }
          }
        }
        if (landed) {
          ph ^= 1u << b;  // this buffer's copy is consumed
          if (tid == kBulkTid) pending &= ~(1u << b);
        } else {
          ok = false;
        }
      }
    }
    if (!__syncthreads_and(ok)) {  // S1: T complete, the state tile landed
      ok = false;
      break;
    }
    stamp(j, 1);
    // thread 0: this task's group counter (read back at the next task); the
    // previous task's flag for its new q/k taps
    if (tid == 0) {
      T.last = prev_live && ((group_old + 1) % (unsigned)p.group) == 0;
      if (live) group_old = atom_add_relaxed_u32(&p.ctr->conv_group[w][kh], 1u);
      if ((p.debug_flags & kDebugTimeline) && j == 0) p.ctr->tl_cta[cta][TL_REC_INPUTS] = globaltimer_ns();
    }
    float inv_q = 0.f, inv_k = 0.f, eg = 0.f, beta = 0.f;
    if (live) {
      // ---- L2 norms of q and k, gates (the single-task phase's arithmetic)
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int i = 0; i < DK / 32; ++i) {
        sq += T.red[i];
        sk += T.red[DK / 32 + i];
      }
      inv_q = (1.0f / sqrtf(sq + p.l2_eps)) * p.q_scale;
      inv_k = 1.0f / sqrtf(sk + p.l2_eps);
      eg = T.eg;
      beta = T.beta;
    }
    // the next task's inputs (this task's head constants are used above),
    // while this one updates its state. From task 1 on they are read as
    // plain values: first, every CTA's partials must be stored (the acquire,
    // and the barrier after it, order the loads after them).
    if (j == 0 && n > 1) {
      if (tid == 0)
        sst->go = wait_counter(p, &p.ctr->proj_done, (unsigned long long)(L + 1) * p.num_ctas, kWaitProj) ? 1 : 0;
      __syncthreads();
      if (!sst->go) ok = false;  // (the error is recorded; the loop ends after this task)
    }
    issue_inputs(j + 1, j + 1 < n && ok);
    if (live) {
      uint8_t* sb = sbuf(j);  // each thread reads and writes only its own elements
      float4 k4[CH], q4[CH];  // this lane's chunks of k^ and q^
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const float4 kq = *reinterpret_cast<const float4*>(&T.k[(sub + LPR * c) * 4]);
        const float4 qq = *reinterpret_cast<const float4*>(&T.q[(sub + LPR * c) * 4]);
        k4[c] = make_float4(kq.x * inv_k, kq.y * inv_k, kq.z * inv_k, kq.w * inv_k);
        q4[c] = make_float4(qq.x * inv_q, qq.y * inv_q, qq.z * inv_q, qq.w * inv_q);
      }
      // one state row of this lane at a time (the tile is in shared memory):
      // the same arithmetic per row as with all rows in registers
#pragma unroll 1
      for (int jr = 0; jr < NR; ++jr) {
        const int v = (jr * kWarps + warp) * RPW + rw;
        float4 s[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int e = v * DK + (sub + LPR * c) * 4;  // element offset in the tile
          if (STATE_BF16) {
            const uint2 u = *reinterpret_cast<const uint2*>(sb + (size_t)e * 2);
            s[c] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
          } else {
            s[c] = *reinterpret_cast<const float4*>(sb + (size_t)e * 4);
          }
        }
        float a = 0.f;  // (S k)[v]
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          s[c].x *= eg; s[c].y *= eg; s[c].z *= eg; s[c].w *= eg;
          a = fmaf(s[c].x, k4[c].x, a);
          a = fmaf(s[c].y, k4[c].y, a);
          a = fmaf(s[c].z, k4[c].z, a);
          a = fmaf(s[c].w, k4[c].w, a);
        }
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        const float u = beta * (T.v[v] - a);
        float ov = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          s[c].x = fmaf(k4[c].x, u, s[c].x); s[c].y = fmaf(k4[c].y, u, s[c].y);
          s[c].z = fmaf(k4[c].z, u, s[c].z); s[c].w = fmaf(k4[c].w, u, s[c].w);
          ov = fmaf(s[c].x, q4[c].x, ov);
          ov = fmaf(s[c].y, q4[c].y, ov);
          ov = fmaf(s[c].z, q4[c].z, ov);
          ov = fmaf(s[c].w, q4[c].w, ov);
          const int e = v * DK + (sub + LPR * c) * 4;
          if (STATE_BF16)
            *reinterpret_cast<uint2*>(sb + (size_t)e * 2) =
                make_uint2(pack_bf16x2(s[c].x, s[c].y), pack_bf16x2(s[c].z, s[c].w));
          else
            *reinterpret_cast<float4*>(sb + (size_t)e * 4) = s[c];
        }
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) ov += __shfl_xor_sync(0xffffffffu, ov, o);
        if (sub == 0) T.o[v] = ov;
      }
    }
    stamp(j, 2);
    tc::fence_proxy_async_smem();  // this thread's tile writes before the bulk copy out
    __syncthreads();  // S2: o, last and the updated tile complete
    stamp(j, 3);
    if (tid == kBulkTid) {
      // the tile back to its slot (an empty group for a pad row), then task
      // j + 2's tile into the buffer task j - 1's copy out has finished reading
      if (live) tc::bulk_store(state_src(slot, h), sbuf(j), SL::kStateBytes);
      tc::bulk_commit();
      if (j >= 1 && j + 2 < n) {
        tc::bulk_wait_read_1();
        if (issue_state(j + 2)) pending |= 1u << ((j + 2) % SL::kBufs);
      }
    }
    // the previous task's new q/k taps, if it was its group's last reader
    if (T.last && tid < 2 * DK) {
      __nv_bfloat16* cs = p.conv_state + ((size_t)prev_slot * p.C + prev_row) * 3;
      cs[0] = __float2bfloat16_rn(nt0);
      cs[1] = __float2bfloat16_rn(nt1);
      cs[2] = __float2bfloat16_rn(nt2);
    }
    if (live) {
      float rn = 0.f;
      if (warp < DK / 32) {  // the warps that write core: each sums o^2 itself (same order)
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < DK / 32; ++i) q = fmaf(T.o[i * 32 + lane], T.o[i * 32 + lane], q);
        q = warp_sum(q);
        rn = 1.0f / sqrtf(q / (float)DK + p.gnorm_eps);
      }
      if (tid < DK) {
        core[tid] = __float2bfloat16_rn(T.o[tid] * rn * gw * silu_f(T.z[tid]));
      }
    } else if (tid < DK) {
      core[tid] = __float2bfloat16_rn(0.f);
      if (slot >= p.num_slots && h == 0 && tid == 0) record_error(p.ctr, kStatusIndex, 0, w);
    }
    if ((p.debug_flags & kDebugTimeline) && j == 0 && tid == 0) p.ctr->tl_cta[cta][TL_REC_STATE] = globaltimer_ns();
    prev_live = live;
    prev_slot = slot;
    prev_row = tid < 2 * DK ? proj_row(tid, h, kh) : 0;
    nt0 = c1;
    nt1 = c2;
    nt2 = pvq;
  }
  if (ok) {
    // the last task's new q/k taps
    StagedTask& T = tb[n & 1];
    if (tid == 0) T.last = prev_live && ((group_old + 1) % (unsigned)p.group) == 0;
    __syncthreads();
    if (T.last && tid < 2 * DK) {
      __nv_bfloat16* cs = p.conv_state + ((size_t)prev_slot * p.C + prev_row) * 3;
      cs[0] = __float2bfloat16_rn(nt0);
      cs[1] = __float2bfloat16_rn(nt1);
      cs[2] = __float2bfloat16_rn(nt2);
    }
  } else if (tid == kBulkTid) {
    // let the copies in flight land before the ring is reused or the CTA ends (bounded)
    for (int bb = 0; bb < SL::kBufs; ++bb) {
      if (!((pending >> bb) & 1u)) continue;
      const unsigned long long c0 = globaltimer_ns();
      for (uint32_t it = 0; !tc::mbar_try_wait(&sbar[bb], (ph >> bb) & 1u); ++it)
        if ((it & 63) == 0 && globaltimer_ns() - c0 > p.deadline_ns) break;
    }
  }
  // the tiles' copies out complete (written to global memory, the ring free)
  if (tid == kBulkTid) tc::bulk_wait_all();
  // the buffers' generic accesses before any later copy into the ring
  tc::fence_proxy_async_smem();
  __syncthreads();
  return ok;
}

}  // namespace gdn
