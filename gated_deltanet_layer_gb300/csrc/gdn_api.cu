// Host side of the C ABI in include/gdn_decode.h: config validation, the
// workspace layout, the stream-K plan of the projection units, argument
// checks and the cooperative launch of the persistent step kernel.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "../../include/gdn_decode.h"
#include "gdn_kernels.h"

using namespace gdn;

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
  size_t ctr, norm_part, xn, proj_part, act, act_ba, total;
};

struct Plan {
  int G, tiles_qkvz, num_tiles, ksteps, norm_chunk, max_contrib;
  int unit_begin[kMaxCtas + 1];
  unsigned char cta_slot0[kMaxCtas];
  unsigned char tile_count[kMaxTiles];
};

}  // namespace

struct gdn_decode {
  gdn_decode_config cfg;
  int device;
  int num_sms;
  void* ws;
  size_t ws_bytes;
  Layout lay;
  Plan plan;
};

namespace {

int n_qkvz(const gdn_decode_config& c) {
  return 2 * c.num_k_heads * c.head_k_dim + 2 * c.num_v_heads * c.head_v_dim;
}
int n_ba(const gdn_decode_config& c) { return 2 * c.num_v_heads; }
int n_conv(const gdn_decode_config& c) {
  return 2 * c.num_k_heads * c.head_k_dim + c.num_v_heads * c.head_v_dim;
}

gdn_status validate(const gdn_decode_config* c) {
  if (!c) return GDN_ERR_ARG;
  if (c->hidden <= 0 || c->num_k_heads <= 0 || c->num_v_heads <= 0 || c->head_k_dim <= 0 ||
      c->head_v_dim <= 0 || c->num_slots <= 0 || c->max_rows < 1 || c->max_rows > kMaxRows)
    return GDN_ERR_ARG;
  if (c->ssm_dtype != GDN_STATE_F32 && c->ssm_dtype != GDN_STATE_BF16) return GDN_ERR_ARG;
  if (c->qkvz_format != GDN_W_BF16 && c->qkvz_format != GDN_W_MXFP4) return GDN_ERR_ARG;
  if (c->engine < GDN_ENGINE_AUTO || c->engine > GDN_ENGINE_TCGEN05) return GDN_ERR_ARG;
  if (!(c->norm_eps >= 0.f) || !(c->gated_norm_eps >= 0.f) || !(c->l2_eps >= 0.f)) return GDN_ERR_ARG;
  if (c->num_ctas < 0 || c->num_ctas > kMaxCtas) return GDN_ERR_ARG;
  // Shapes this build runs.
  if (c->conv_kernel != 4) return GDN_ERR_UNSUPPORTED;
  if (c->head_k_dim != c->head_v_dim) return GDN_ERR_UNSUPPORTED;
  if (c->head_k_dim != 64 && c->head_k_dim != 128) return GDN_ERR_UNSUPPORTED;
  if (c->num_v_heads % c->num_k_heads != 0) return GDN_ERR_UNSUPPORTED;
  if ((c->num_k_heads * c->head_k_dim) % kTileM != 0) return GDN_ERR_UNSUPPORTED;
  if ((c->num_v_heads * c->head_v_dim) % kTileM != 0) return GDN_ERR_UNSUPPORTED;
  if (c->hidden % kKStep != 0 || c->hidden > (1 << 20)) return GDN_ERR_UNSUPPORTED;
  if (c->qkvz_format == GDN_W_MXFP4) return GDN_ERR_UNSUPPORTED;
  if (c->engine == GDN_ENGINE_TCGEN05) return GDN_ERR_UNSUPPORTED;
  const int tiles = n_qkvz(*c) / kTileM + (n_ba(*c) + kTileM - 1) / kTileM;
  if (tiles > kMaxTiles) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// Stream-K split of the projection units over G CTAs. A unit is one 64-column
// step of one 128-row tile; a unit of a partial in_proj_ba tile costs its row
// count, so every CTA streams about the same number of weight bytes. CTA c
// takes units [unit_begin[c], unit_begin[c+1]).
gdn_status make_plan(const gdn_decode_config& c, int G, Plan* pl) {
  pl->G = G;
  pl->tiles_qkvz = n_qkvz(c) / kTileM;
  const int nba = n_ba(c);
  pl->num_tiles = pl->tiles_qkvz + (nba + kTileM - 1) / kTileM;
  pl->ksteps = c.hidden / kKStep;
  int chunk = (c.hidden + G - 1) / G;
  chunk = (chunk + 7) / 8 * 8;
  pl->norm_chunk = chunk;
  if (chunk > kMaxNormChunk) return GDN_ERR_UNSUPPORTED;
  const long long KS = pl->ksteps;
  const long long U = (long long)pl->num_tiles * KS;
  auto cost = [&](long long t) -> long long {
    return t < pl->tiles_qkvz ? kTileM : std::min<long long>(kTileM, nba - (t - pl->tiles_qkvz) * kTileM);
  };
  long long total = 0;
  for (long long t = 0; t < pl->num_tiles; ++t) total += cost(t) * KS;
  // unit_begin[c] = first unit whose cost prefix reaches c * total / G
  long long u = 0, prefix = 0;
  for (int cta = 0; cta <= G; ++cta) {
    while (u < U && prefix * G < (long long)cta * total) {
      prefix += cost(u / KS);
      ++u;
    }
    pl->unit_begin[cta] = (int)(cta == G ? U : u);
  }
  // Contributors of a tile are the CTAs with at least one unit in it, slotted
  // in CTA order. A CTA whose range starts inside tile t0 takes the next slot
  // of t0; every later tile it touches starts inside its range, so it is that
  // tile's first contributor.
  int count[kMaxTiles];
  for (int t = 0; t < pl->num_tiles; ++t) count[t] = 0;
  for (int cta = 0; cta < G; ++cta) {
    pl->cta_slot0[cta] = 0;
    const int b = pl->unit_begin[cta], e = pl->unit_begin[cta + 1];
    if (b >= e) continue;
    const int t0 = (int)(b / KS);
    for (int t = t0; t <= (int)((e - 1) / KS); ++t) {
      if (t == t0) {
        if (count[t] > 255) return GDN_ERR_UNSUPPORTED;
        pl->cta_slot0[cta] = (unsigned char)count[t];
      } else if (count[t] != 0) {
        return GDN_ERR_UNSUPPORTED;  // cannot happen with contiguous ranges
      }
      ++count[t];
    }
  }
  int maxc = 1;
  for (int t = 0; t < pl->num_tiles; ++t) {
    if (count[t] < 1 || count[t] > 255) return GDN_ERR_UNSUPPORTED;
    pl->tile_count[t] = (unsigned char)count[t];
    maxc = std::max(maxc, count[t]);
  }
  pl->max_contrib = maxc;
  return GDN_OK;
}

Layout make_layout(const gdn_decode_config& c, const Plan& pl) {
  Layout l;
  size_t off = 0;
  l.ctr = off;        off += align_up(sizeof(WsCounters), 256);
  l.norm_part = off;  off += align_up((size_t)kMaxRows * pl.G * sizeof(float), 256);
  l.xn = off;         off += align_up((size_t)kMaxRows * c.hidden * 2, 256);
  l.proj_part = off;  off += align_up((size_t)pl.num_tiles * pl.max_contrib * kMaxRows * kTileM * sizeof(float), 256);
  l.act = off;        off += align_up((size_t)kMaxRows * n_qkvz(c) * sizeof(float), 256);
  l.act_ba = off;     off += align_up((size_t)kMaxRows * n_ba(c) * sizeof(float), 256);
  l.total = off;
  return l;
}

gdn_status device_grid(const gdn_decode_config& c, int* device, int* num_sms, int* G) {
  if (cudaGetDevice(device) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess)
    return GDN_ERR_CUDA;
  *G = c.num_ctas > 0 ? c.num_ctas : std::min(*num_sms, kMaxCtas);
  if (*G > *num_sms) return GDN_ERR_UNSUPPORTED;  // one co-resident CTA per SM
  return GDN_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const char* pa = (const char*)a;
  const char* pb = (const char*)b;
  return pa < pb + nb && pb < pa + na;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

const void* pick_kernel(const gdn_decode_config& c, bool has_res) {
  return cuda_core_kernel(has_res, c.ssm_dtype == GDN_STATE_BF16, c.head_k_dim);
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported shape or option";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_DEADLINE: return "a cross-CTA wait passed its deadline";
    case GDN_ERR_INDEX: return "state index out of range";
    case GDN_ERR_FAILED: return "device error word set";
  }
  return "unknown status";
}

size_t gdn_decode_workspace_bytes(const gdn_decode_config* cfg) {
  if (validate(cfg) != GDN_OK) return 0;
  int dev, sms, G;
  if (device_grid(*cfg, &dev, &sms, &G) != GDN_OK) return 0;
  Plan* pl = new (std::nothrow) Plan;
  if (!pl) return 0;
  size_t bytes = 0;
  if (make_plan(*cfg, G, pl) == GDN_OK) bytes = make_layout(*cfg, *pl).total;
  delete pl;
  return bytes;
}

gdn_status gdn_decode_create(const gdn_decode_config* cfg, void* workspace, size_t workspace_bytes,
                             void* stream, gdn_decode_t** out) {
  if (!out) return GDN_ERR_ARG;
  *out = nullptr;
  gdn_status st = validate(cfg);
  if (st != GDN_OK) return st;
  if (!workspace || !aligned(workspace, 256)) return GDN_ERR_ARG;
  gdn_decode* h = new (std::nothrow) gdn_decode;
  if (!h) return GDN_ERR_ARG;
  h->cfg = *cfg;
  if (h->cfg.deadline_us == 0) h->cfg.deadline_us = 200000;
  int G;
  st = device_grid(h->cfg, &h->device, &h->num_sms, &G);
  if (st == GDN_OK) st = make_plan(h->cfg, G, &h->plan);
  if (st != GDN_OK) {
    delete h;
    return st;
  }
  h->lay = make_layout(h->cfg, h->plan);
  if (workspace_bytes < h->lay.total) {
    delete h;
    return GDN_ERR_ARG;
  }
  int coop = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device) != cudaSuccess || !coop) {
    delete h;
    return GDN_ERR_UNSUPPORTED;
  }
  // Every CTA of the persistent grid must be co-resident.
  for (int r = 0; r < 2; ++r) {
    const void* k = pick_kernel(h->cfg, r == 1);
    int per_sm = 0;
    if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, 0) != cudaSuccess ||
        per_sm < 1) {
      delete h;
      return GDN_ERR_UNSUPPORTED;
    }
  }
  h->ws = workspace;
  h->ws_bytes = workspace_bytes;
  if (cudaMemsetAsync(workspace, 0, h->lay.total, (cudaStream_t)stream) != cudaSuccess) {
    delete h;
    return GDN_ERR_CUDA;
  }
  *out = h;
  return GDN_OK;
}

gdn_status gdn_decode_step(gdn_decode_t* h, int32_t rows, const void* x, const void* residual,
                           const gdn_decode_weights* w, const int32_t* state_indices,
                           void* conv_state, void* ssm_state, void* core_out, void* residual_out,
                           void* stream) {
  if (!h || !w) return GDN_ERR_ARG;
  const gdn_decode_config& c = h->cfg;
  if (rows < 1 || rows > c.max_rows) return GDN_ERR_ARG;
  if (!x || !state_indices || !conv_state || !ssm_state || !core_out || !residual_out) return GDN_ERR_ARG;
  if (!w->input_norm_w || !w->qkvz || !w->ba || !w->conv_w || !w->A_log || !w->dt_bias || !w->gated_norm_w)
    return GDN_ERR_ARG;
  const void* a16[] = {x, residual, core_out, residual_out, conv_state, ssm_state, w->input_norm_w,
                       w->qkvz, w->ba, w->conv_w, w->gated_norm_w};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return GDN_ERR_ARG;
  if (!aligned(state_indices, 4) || !aligned(w->A_log, 4) || !aligned(w->dt_bias, 2)) return GDN_ERR_ARG;
  const size_t H = (size_t)c.hidden;
  const size_t xb = (size_t)rows * H * 2;
  const size_t coreb = (size_t)rows * c.num_v_heads * c.head_v_dim * 2;
  const size_t sdt = c.ssm_dtype == GDN_STATE_BF16 ? 2 : 4;
  const size_t ssmb = (size_t)c.num_slots * c.num_v_heads * c.head_v_dim * c.head_k_dim * sdt;
  const size_t convb = (size_t)c.num_slots * n_conv(c) * (c.conv_kernel - 1) * 2;
  struct Rg { const void* p; size_t n; };
  const Rg ins[] = {{x, xb}, {residual, residual ? xb : 0}, {state_indices, (size_t)rows * 4},
                    {conv_state, convb}, {ssm_state, ssmb}, {w->qkvz, (size_t)n_qkvz(c) * H * 2},
                    {w->ba, (size_t)n_ba(c) * H * 2}, {w->input_norm_w, H * 2},
                    {h->ws, h->lay.total}};
  const Rg outs[] = {{core_out, coreb}, {residual_out, xb}};
  for (const Rg& o : outs)
    for (const Rg& i : ins)
      if (overlaps(o.p, o.n, i.p, i.n)) return GDN_ERR_ARG;
  if (overlaps(core_out, coreb, residual_out, xb)) return GDN_ERR_ARG;
  if (overlaps(conv_state, convb, ssm_state, ssmb)) return GDN_ERR_ARG;

  const Plan& pl = h->plan;
  StepParams* p = new (std::nothrow) StepParams;
  if (!p) return GDN_ERR_ARG;
  memset(p, 0, sizeof(*p));
  p->H = c.hidden; p->Hk = c.num_k_heads; p->Hv = c.num_v_heads;
  p->dk = c.head_k_dim; p->dv = c.head_v_dim; p->C = n_conv(c);
  p->Nqkvz = n_qkvz(c); p->Nba = n_ba(c); p->num_slots = c.num_slots; p->rows = rows;
  p->group = c.num_v_heads / c.num_k_heads;
  p->tiles_qkvz = pl.tiles_qkvz; p->num_tiles = pl.num_tiles; p->ksteps = pl.ksteps;
  p->norm_chunk = pl.norm_chunk; p->max_contrib = pl.max_contrib; p->num_ctas = pl.G;
  p->norm_eps = c.norm_eps; p->gnorm_eps = c.gated_norm_eps; p->l2_eps = c.l2_eps; p->q_scale = c.q_scale;
  p->deadline_ns = (unsigned long long)c.deadline_us * 1000ull;
  p->debug_flags = c.debug_flags;
  p->x = (const __nv_bfloat16*)x;
  p->res = (const __nv_bfloat16*)residual;
  p->res_out = (__nv_bfloat16*)residual_out;
  p->core_out = (__nv_bfloat16*)core_out;
  p->idx = state_indices;
  p->conv_state = (__nv_bfloat16*)conv_state;
  p->ssm_state = ssm_state;
  p->w_in = (const __nv_bfloat16*)w->input_norm_w;
  p->w_qkvz = (const __nv_bfloat16*)w->qkvz;
  p->w_qkvz_scales = w->qkvz_scales;
  p->w_ba = (const __nv_bfloat16*)w->ba;
  p->conv_w = (const __nv_bfloat16*)w->conv_w;
  p->A_log = w->A_log;
  p->dt_bias = (const __nv_bfloat16*)w->dt_bias;
  p->gnorm_w = (const __nv_bfloat16*)w->gated_norm_w;
  char* base = (char*)h->ws;
  p->ctr = (WsCounters*)(base + h->lay.ctr);
  p->norm_part = (float*)(base + h->lay.norm_part);
  p->xn = (__nv_bfloat16*)(base + h->lay.xn);
  p->proj_part = (float*)(base + h->lay.proj_part);
  p->act = (float*)(base + h->lay.act);
  p->act_ba = (float*)(base + h->lay.act_ba);
  memcpy(p->unit_begin, pl.unit_begin, sizeof(int) * (pl.G + 1));
  memcpy(p->cta_slot0, pl.cta_slot0, pl.G);
  memcpy(p->tile_num_ctas, pl.tile_count, pl.num_tiles);

  const void* kern = pick_kernel(c, residual != nullptr);
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(pl.G);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = 0;
  lc.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  void* args[] = {p};
  const cudaError_t e = cudaLaunchKernelExC(&lc, kern, args);
  delete p;
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_decode_check(gdn_decode_t* h, void* stream, uint32_t* detail) {
  if (!h) return GDN_ERR_ARG;
  uint32_t word = 0;
  const char* base = (const char*)h->ws;
  const void* err = base + h->lay.ctr + offsetof(WsCounters, error);
  if (cudaMemcpyAsync(&word, err, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
  if (detail) *detail = word;
  if (word == 0) return GDN_OK;
  const uint32_t s = word >> 24;
  if (s == GDN_ERR_DEADLINE) return GDN_ERR_DEADLINE;
  if (s == GDN_ERR_INDEX) return GDN_ERR_INDEX;
  return GDN_ERR_FAILED;
}

gdn_status gdn_decode_reset(gdn_decode_t* h, void* stream) {
  if (!h) return GDN_ERR_ARG;
  return cudaMemsetAsync(h->ws, 0, h->lay.total, (cudaStream_t)stream) == cudaSuccess ? GDN_OK
                                                                                      : GDN_ERR_CUDA;
}

void gdn_decode_destroy(gdn_decode_t* h) { delete h; }

gdn_status gdn_decode_launch_info(const gdn_decode_t* h, int32_t rows, int32_t* num_ctas,
                                  int32_t* engine) {
  if (!h || rows < 1 || rows > h->cfg.max_rows) return GDN_ERR_ARG;
  if (num_ctas) *num_ctas = h->plan.G;
  if (engine) *engine = GDN_ENGINE_CUDA_CORE;
  return GDN_OK;
}

gdn_status gdn_decode_plan(const gdn_decode_config* cfg, int32_t num_ctas, int32_t* unit_begin,
                           uint8_t* cta_slot0, uint8_t* tile_count, int32_t tile_cap,
                           int32_t* num_tiles, int32_t* ksteps) {
  gdn_status st = validate(cfg);
  if (st != GDN_OK) return st;
  if (num_ctas < 1 || num_ctas > kMaxCtas || !unit_begin || !cta_slot0 || !tile_count || !num_tiles ||
      !ksteps)
    return GDN_ERR_ARG;
  Plan* pl = new (std::nothrow) Plan;
  if (!pl) return GDN_ERR_ARG;
  st = make_plan(*cfg, num_ctas, pl);
  if (st == GDN_OK && pl->num_tiles > tile_cap) st = GDN_ERR_ARG;
  if (st == GDN_OK) {
    memcpy(unit_begin, pl->unit_begin, sizeof(int32_t) * (num_ctas + 1));
    memcpy(cta_slot0, pl->cta_slot0, num_ctas);
    memcpy(tile_count, pl->tile_count, pl->num_tiles);
    *num_tiles = pl->num_tiles;
    *ksteps = pl->ksteps;
  }
  delete pl;
  return st;
}

}  // extern "C"
