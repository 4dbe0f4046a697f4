// Host side of the C ABI in include/gdn_decode.h: config validation, the
// workspace layout, the stream-K plan of the projection units, argument
// checks and the cooperative launch of the persistent step kernel.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "gdn_decode.h"
#include "gdn_decode_diag.h"
#include "gdn_kernels.h"

using namespace gdn;

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
  size_t ctr, plan, norm_part, core_flag, proj_part, total;
};

struct Plan {
  int engine;  // GDN_ENGINE_CUDA_CORE or GDN_ENGINE_TCGEN05
  int G, tiles_qkvz, num_tiles, ksteps, kblock, max_contrib;
  int unit_begin[kMaxCtas + 1];
  unsigned char seg_slot[kMaxCtas][kMaxSegs];
  unsigned short ks_first[kMaxCtas];
  unsigned char nb_slots[kMaxCtas];
  unsigned char tile_count[kMaxTiles];
  unsigned int own_mask[kMaxCtas];
  // weight ring depth (bf16 tiles), code ring depth (MXFP4 / MXFP6 code
  // tiles), normed-input window (k-steps), the pad past it, and the launch's
  // dynamic shared memory (the same for both engines)
  int stages, rstages, xslots;
  unsigned int xpad;
  size_t smem;
};

// Weight tile maps, re-encoded only when the weight pointers change.
struct MapCache {
  const void* qkvz_ptr = nullptr;
  const void* ba_ptr = nullptr;
  const void* out_ptr = nullptr;
  CUtensorMap qkvz;
  CUtensorMap ba;
  CUtensorMap out;
};

// Shared memory a CTA may use on sm_100-class GPUs (opt-in limit per block).
constexpr size_t kSmemOptin = 232448;

}  // namespace

struct gdn_decode {
  gdn_decode_config cfg;
  int device;
  int num_sms;
  void* ws;
  size_t ws_bytes;
  Layout lay;
  Plan plan;
  bool pdl;  // launch with programmatic stream serialisation
  MapCache maps;  // TMA maps of the last weights a step used
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
      c->head_v_dim <= 0 || c->num_slots <= 0 || c->max_rows < 1 || c->max_rows > GDN_MAX_ROWS)
    return GDN_ERR_ARG;
  if (c->ssm_dtype != GDN_STATE_F32 && c->ssm_dtype != GDN_STATE_BF16) return GDN_ERR_ARG;
  if (c->qkvz_format != GDN_W_BF16 && c->qkvz_format != GDN_W_MXFP4 && c->qkvz_format != GDN_W_MXFP6)
    return GDN_ERR_ARG;
  if (c->engine < GDN_ENGINE_AUTO || c->engine > GDN_ENGINE_TCGEN05) return GDN_ERR_ARG;
  if (!(c->norm_eps >= 0.f) || !(c->gated_norm_eps >= 0.f) || !(c->l2_eps >= 0.f)) return GDN_ERR_ARG;
  if (c->num_ctas < 0 || c->num_ctas > kMaxCtas) return GDN_ERR_ARG;
  if (c->launch_flags & ~(GDN_LAUNCH_COOPERATIVE | GDN_LAUNCH_NO_EARLY_WEIGHTS)) return GDN_ERR_ARG;
  // Shapes this build runs.
  if (c->conv_kernel != 4) return GDN_ERR_UNSUPPORTED;
  if (c->head_k_dim != c->head_v_dim) return GDN_ERR_UNSUPPORTED;
  if (c->head_k_dim != 64 && c->head_k_dim != 128) return GDN_ERR_UNSUPPORTED;
  if (c->num_v_heads % c->num_k_heads != 0) return GDN_ERR_UNSUPPORTED;
  if (c->num_k_heads > kMaxKHeads) return GDN_ERR_UNSUPPORTED;
  if (c->num_v_heads % 2 != 0) return GDN_ERR_UNSUPPORTED;  // in_proj_ba rows come in fours
  if ((c->num_k_heads * c->head_k_dim) % kTileM != 0) return GDN_ERR_UNSUPPORTED;
  if ((c->num_v_heads * c->head_v_dim) % kTileM != 0) return GDN_ERR_UNSUPPORTED;
  if (c->hidden % kKStep != 0 || c->hidden > (1 << 20)) return GDN_ERR_UNSUPPORTED;
  // MXFP4 / MXFP6: a row's e8m0 scales for 8 k-steps are one aligned 16-byte load
  if (c->qkvz_format != GDN_W_BF16 && (c->hidden % 512 != 0 || c->head_k_dim != 128)) return GDN_ERR_UNSUPPORTED;
  const int tiles = n_qkvz(*c) / kTileM + (n_ba(*c) + kTileM - 1) / kTileM;
  if (tiles > kMaxTiles) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// Stream-K split of the projection units over G CTAs. A unit is one 64-column
// step (k-step) of one 256-row tile. Units are ordered by group: group g =
// (k-block kb = g / T, tile t = g % T) holds the `kblock` k-steps kb*kblock ..
// of tile t. With kblock = ksteps the order is tile-major (a CTA sweeps K of
// one tile, then the next); a large layer uses kblock = 16 (8 with MXFP4 or MXFP6 weights, whose second window or code
// ring takes the room), so a CTA's units touch at most two k-blocks and the
// normed input it needs (<= 32 k-steps; 24 with coded weights) fits in shared
// memory. Longer k-blocks also mean
// fewer partials per tile for the recurrence to add. Every unit counts the
// same, also one of the partial in_proj_ba tile: a unit's time is set by its
// fixed per-unit cost, not by its row count. CTA c takes units
// [unit_begin[c], unit_begin[c+1]) with unit_begin[c] = floor(c * U / G).
gdn_status make_plan(const gdn_decode_config& c, int G, int engine, Plan* pl) {
  pl->engine = engine;
  pl->G = G;
  pl->tiles_qkvz = n_qkvz(c) / kTileM;
  const int nba = n_ba(c);
  const int T = pl->tiles_qkvz + (nba + kTileM - 1) / kTileM;
  pl->num_tiles = T;
  const int KS = c.hidden / kKStep;
  pl->ksteps = KS;
  const long long U = (long long)T * KS;
  const long long per_cta = (U + G - 1) / G;
  // the normed-input window, in k-steps, and the k-block that keeps a CTA's
  // units inside it
  // coded weights (MXFP4: two windows; MXFP6: the code ring) keep the ring
  // deeper with the shorter k-block
  const bool coded = c.qkvz_format != GDN_W_BF16;
  const int max_window = coded ? kMaxBSlotsMxfp4 : kMaxBSlots;
  int KB = KS;
  if (per_cta + 1 > max_window) {
    KB = coded ? kKBlockMxfp4 : kKBlock;
    if (KS % KB != 0) return GDN_ERR_UNSUPPORTED;
  }
  pl->kblock = KB;
  for (int cta = 0; cta <= G; ++cta) pl->unit_begin[cta] = (int)((long long)cta * U / G);
  // Partial slots: the pieces of tile t in unit order (k-block, then CTA)
  // take slots 0, 1, ... of the tile; the epilogue adds them in slot order.
  int count[kMaxTiles];
  for (int t = 0; t < T; ++t) count[t] = 0;
  std::vector<char> need(KS);
  for (int cta = 0; cta < G; ++cta) {
    const long long b = pl->unit_begin[cta], e = pl->unit_begin[cta + 1];
    for (int i = 0; i < kMaxSegs; ++i) pl->seg_slot[cta][i] = 0;
    pl->ks_first[cta] = 0;
    pl->nb_slots[cta] = 0;
    if (b >= e) continue;
    int seg = 0;
    for (long long g = b / KB; g <= (e - 1) / KB; ++g, ++seg) {
      if (seg >= kMaxSegs) return GDN_ERR_UNSUPPORTED;
      const int t = (int)(g % T);
      if (count[t] > 254) return GDN_ERR_UNSUPPORTED;
      pl->seg_slot[cta][seg] = (unsigned char)count[t]++;
    }
    // the k-steps this CTA multiplies, as one cyclic window ks_first + j
    std::fill(need.begin(), need.end(), 0);
    int nneed = 0;
    for (long long u = b; u < e; ++u) {
      const long long g = u / KB;
      const int ks = (int)((g / T) * KB + u % KB);
      if (!need[ks]) { need[ks] = 1; ++nneed; }
    }
    int first = 0, len = KS;
    if (nneed < KS) {
      // the window starts after the longest cyclic run of unneeded k-steps
      int best_gap = -1, best_end = 0;
      for (int i = 0; i < KS; ++i) {
        if (need[i] || !need[(i + KS - 1) % KS]) continue;  // i starts a gap run
        int j = i;
        while (!need[j % KS]) ++j;
        if (j - i > best_gap) { best_gap = j - i; best_end = j % KS; }
      }
      first = best_end;
      len = KS - best_gap;
    }
    pl->ks_first[cta] = (unsigned short)first;
    pl->nb_slots[cta] = (unsigned char)std::min(len, 255);
    if (len > max_window) return GDN_ERR_UNSUPPORTED;
  }
  // k-step owners: the first CTA whose window holds it
  for (int cta = 0; cta < G; ++cta) pl->own_mask[cta] = 0;
  for (int ks = 0; ks < KS; ++ks) {
    int owner = -1;
    for (int cta = 0; cta < G && owner < 0; ++cta) {
      const int j = (ks - pl->ks_first[cta] + KS) % KS;
      if (j < pl->nb_slots[cta]) {
        owner = cta;
        pl->own_mask[cta] |= 1u << j;
      }
    }
    if (owner < 0) return GDN_ERR_UNSUPPORTED;
  }
  int maxc = 1;
  for (int t = 0; t < T; ++t) {
    // a recurrence task reduces one output's partials in one batch of <= 24
    if (count[t] < 1 || count[t] > 24) return GDN_ERR_UNSUPPORTED;
    pl->tile_count[t] = (unsigned char)count[t];
    maxc = std::max(maxc, count[t]);
  }
  pl->max_contrib = maxc;
  // the ring takes what the window (two windows with MXFP4 weights: xn and
  // its quantised copy) and the code ring leave: 2..6 tiles of 32 KB
  const int fmt = c.qkvz_format;
  int xs = 1;
  for (int cta = 0; cta < G; ++cta) xs = std::max(xs, (int)pl->nb_slots[cta]);
  pl->xslots = xs;
  pl->xpad = tensor_core_xpad(xs);
  const size_t avail = kSmemOptin - tensor_core_static_smem() - 1024;
  const size_t wtile = (size_t)kTileM * kKStep * 2;
  pl->rstages = fmt != GDN_W_BF16 ? tensor_core_max_rstages() : 0;
  const size_t fixed = tensor_core_smem_bytes(0, pl->rstages, xs, fmt);
  if (fixed + 2 * wtile > avail) return GDN_ERR_UNSUPPORTED;
  pl->stages = (int)std::min<size_t>((avail - fixed) / wtile, (size_t)tensor_core_max_stages());
  pl->smem = tensor_core_smem_bytes(pl->stages, pl->rstages, xs, fmt);
  return GDN_OK;
}

Layout make_layout(const gdn_decode_config& c, const Plan& pl) {
  Layout l;
  size_t off = 0;
  l.ctr = off;        off += align_up(sizeof(WsCounters), 256);
  l.plan = off;       off += align_up(sizeof(PlanDev), 256);
  l.norm_part = off;  off += align_up((size_t)kMaxRows * pl.G * sizeof(unsigned long long), 256);
  l.core_flag = off;  off += align_up((size_t)pl.G * sizeof(unsigned long long), 256);
  l.proj_part = off;
  off += align_up((size_t)pl.num_tiles * pl.max_contrib * kMaxRows * kTileM * sizeof(unsigned long long), 256);
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

// The step kernel of a config: the engine's, for a decode step or (multi) a
// verify step (tensor-core engine with bf16 weights only); nullptr if none.
const void* pick_kernel(const gdn_decode_config& c, int engine, bool has_res, bool multi = false) {
  const bool b16 = c.ssm_dtype == GDN_STATE_BF16;
  if (engine == GDN_ENGINE_TCGEN05) return tensor_core_kernel(has_res, b16, c.head_k_dim, c.qkvz_format, multi);
  return multi || c.qkvz_format != GDN_W_BF16 ? nullptr : cuda_core_kernel(has_res, b16, c.head_k_dim);
}

size_t kernel_smem(const Plan& pl) { return pl.smem; }

// Zero what a workspace's launches count on: the counters and error word, and
// the tagged partials (a zero tag is no launch's; with the counters back at
// zero, old tags would otherwise match new launches). The plan stays.
bool clear_launch_state(char* base, const Layout& l, cudaStream_t s) {
  return cudaMemsetAsync(base + l.ctr, 0, sizeof(WsCounters), s) == cudaSuccess &&
         cudaMemsetAsync(base + l.norm_part, 0, l.total - l.norm_part, s) == cudaSuccess;
}

// Launch fields of the plan that the kernels read.
void set_plan_params(const Plan& pl, StepParams* p) {
  p->tiles_qkvz = pl.tiles_qkvz; p->num_tiles = pl.num_tiles; p->ksteps = pl.ksteps;
  p->max_contrib = pl.max_contrib; p->num_ctas = pl.G;
  p->kblock = pl.kblock;
  p->stages = pl.stages; p->rstages = pl.rstages; p->xslots = pl.xslots; p->xpad = pl.xpad;
  p->dyn_free = pl.smem > 1024 ? (unsigned int)(pl.smem - 1024) : 0u;  // 1 KB of it aligns the ring
}

// The engine a config runs with and its plan (the engines share the plan:
// the same units, windows and weight ring): the requested engine, or for
// GDN_ENGINE_AUTO the tensor-core engine. MXFP4 and MXFP6 weights run on the
// tensor-core engine only.
gdn_status resolve_plan(const gdn_decode_config& c, int G, Plan* pl) {
  if (c.engine == GDN_ENGINE_CUDA_CORE && c.qkvz_format != GDN_W_BF16) return GDN_ERR_UNSUPPORTED;
  return make_plan(c, G, c.engine == GDN_ENGINE_CUDA_CORE ? GDN_ENGINE_CUDA_CORE : GDN_ENGINE_TCGEN05, pl);
}

// cuTensorMapEncodeTiled from the driver, looked up once.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  }
  return fn;
}

// Tile map of a row-major [rows][H] bf16 weight: box 64 columns x 128 rows,
// 128-byte swizzle (the K-major layout tcgen05.mma reads), zero fill past the
// last row.
bool encode_weight_map(CUtensorMap* m, const void* base, int rows, int H) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kKStep, (cuuint32_t)kTileM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile map of out_proj [H][K] bf16 (K = Hv*dv): box 64 columns x 64 rows,
// 128-byte swizzle, zero fill past the last row.
bool encode_out_map(CUtensorMap* m, const void* base, int rows, int K) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile map of codes [rows][H * bits / 8] uint8 (MXFP4 4 bits, MXFP6 6 bits a
// code): box of one k-step's codes (32 or 48 bytes) x 256 rows, no swizzle
// (the decoding warps read each row's bytes).
bool encode_code_map(CUtensorMap* m, const void* base, int rows, int H, int bits) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)H * bits / 8, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)H * bits / 8};
  const cuuint32_t box[2] = {(cuuint32_t)kKStep * bits / 8, (cuuint32_t)kTileM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes of in_proj_qkvz as the config stores it.
size_t qkvz_bytes(const gdn_decode_config& c) {
  const size_t n = (size_t)n_qkvz(c), H = (size_t)c.hidden;
  return c.qkvz_format == GDN_W_MXFP4 ? n * H / 2 : c.qkvz_format == GDN_W_MXFP6 ? n * H * 3 / 4 : n * H * 2;
}

// The weight tile maps of a step: in_proj_qkvz (bf16, or MXFP4 / MXFP6
// codes) and in_proj_ba (bf16).
bool encode_maps(const gdn_decode_config& c, const gdn_decode_weights* w, CUtensorMap* mq, CUtensorMap* mba) {
  const bool okq = c.qkvz_format == GDN_W_BF16
                       ? encode_weight_map(mq, w->qkvz, n_qkvz(c), c.hidden)
                       : encode_code_map(mq, w->qkvz, n_qkvz(c), c.hidden, c.qkvz_format == GDN_W_MXFP4 ? 4 : 6);
  return okq && encode_weight_map(mba, w->ba, n_ba(c), c.hidden);
}


// The tensors of one step call. A verify step has `tokens` rows per
// sequence, idx holds one slot per sequence and idx_out one per row; a
// decode step has tokens = 1 and no idx_out.
struct StepArgs {
  int32_t rows;
  const void* x;
  const void* residual;
  const gdn_decode_weights* w;
  const int32_t* idx;
  void* conv_state;
  void* ssm_state;
  void* core_out;
  void* residual_out;
  int32_t tokens = 1;
  const int32_t* idx_out = nullptr;
  void* out = nullptr;  // out_proj result [rows][H] (weights out_proj), or nullptr
};

// Host-side checks of a step's arguments (before any launch): rows in range,
// non-null and aligned pointers, no output overlapping an input, the
// scratch or the other output, conv and SSM state apart.
gdn_status check_step_args(const gdn_decode_config& c, const StepArgs& a, const void* scratch,
                           size_t scratch_bytes) {
  const gdn_decode_weights* w = a.w;
  if (!w) return GDN_ERR_ARG;
  if (a.rows < 1 || a.rows > c.max_rows) return GDN_ERR_ARG;
  if (!a.x || !a.idx || !a.conv_state || !a.ssm_state || !a.core_out || !a.residual_out) return GDN_ERR_ARG;
  if (!w->input_norm_w || !w->qkvz || !w->ba || !w->conv_w || !w->A_log || !w->dt_bias || !w->gated_norm_w)
    return GDN_ERR_ARG;
  if (c.qkvz_format != GDN_W_BF16 && !w->qkvz_scales) return GDN_ERR_ARG;
  const void* a16[] = {a.x, a.residual, a.core_out, a.residual_out, a.conv_state, a.ssm_state, w->input_norm_w,
                       w->qkvz, w->ba, w->conv_w, w->gated_norm_w};
  for (const void* q : a16)
    if (q && !aligned(q, 16)) return GDN_ERR_ARG;
  if (!aligned(a.idx, 4) || !aligned(w->A_log, 4) || !aligned(w->dt_bias, 2)) return GDN_ERR_ARG;
  if (a.tokens > 1 && (!a.idx_out || !aligned(a.idx_out, 4))) return GDN_ERR_ARG;
  if (a.out && (!w->out_proj || !aligned(a.out, 16) || !aligned(w->out_proj, 16))) return GDN_ERR_ARG;
  const size_t H = (size_t)c.hidden;
  const size_t xb = (size_t)a.rows * H * 2;
  const size_t coreb = (size_t)a.rows * c.num_v_heads * c.head_v_dim * 2;
  const size_t sdt = c.ssm_dtype == GDN_STATE_BF16 ? 2 : 4;
  const size_t ssmb = (size_t)c.num_slots * c.num_v_heads * c.head_v_dim * c.head_k_dim * sdt;
  const size_t convb = (size_t)c.num_slots * n_conv(c) * (c.conv_kernel - 1) * 2;
  struct Rg { const void* p; size_t n; };
  const Rg ins[] = {{a.x, xb}, {a.residual, a.residual ? xb : 0}, {a.idx, (size_t)(a.rows / a.tokens) * 4},
                    {a.idx_out, a.idx_out ? (size_t)a.rows * 4 : 0},
                    {a.conv_state, convb}, {a.ssm_state, ssmb}, {w->qkvz, qkvz_bytes(c)},
                    {w->ba, (size_t)n_ba(c) * H * 2}, {w->input_norm_w, H * 2},
                    {w->qkvz_scales, c.qkvz_format != GDN_W_BF16 ? (size_t)n_qkvz(c) * H / 32 : 0},
                    {a.out ? w->out_proj : nullptr, a.out ? H * c.num_v_heads * c.head_v_dim * 2 : 0},
                    {scratch, scratch_bytes}};
  const Rg outs[] = {{a.core_out, coreb}, {a.residual_out, xb}, {a.out, a.out ? xb : 0}};
  for (const Rg& o : outs)
    for (const Rg& i : ins)
      if (overlaps(o.p, o.n, i.p, i.n)) return GDN_ERR_ARG;
  if (overlaps(a.core_out, coreb, a.residual_out, xb)) return GDN_ERR_ARG;
  if (overlaps(a.out, a.out ? xb : 0, a.core_out, coreb) || overlaps(a.out, a.out ? xb : 0, a.residual_out, xb))
    return GDN_ERR_ARG;
  if (overlaps(a.conv_state, convb, a.ssm_state, ssmb)) return GDN_ERR_ARG;
  return GDN_OK;
}

// The launch parameters of a step on scratch `base` (a workspace or the
// static scratch) laid out as `lay`.
void fill_params(const gdn_decode_config& c, const Plan& pl, const Layout& lay, char* base, const StepArgs& a,
                 StepParams* p) {
  memset(p, 0, sizeof(*p));
  p->H = c.hidden; p->Hk = c.num_k_heads; p->Hv = c.num_v_heads;
  p->dk = c.head_k_dim; p->dv = c.head_v_dim; p->C = n_conv(c);
  p->Nqkvz = n_qkvz(c); p->Nba = n_ba(c); p->num_slots = c.num_slots; p->rows = a.rows;
  p->tokens = a.tokens;
  p->idx_out = a.idx_out;
  p->group = c.num_v_heads / c.num_k_heads;
  set_plan_params(pl, p);
  p->norm_eps = c.norm_eps; p->gnorm_eps = c.gated_norm_eps; p->l2_eps = c.l2_eps; p->q_scale = c.q_scale;
  p->deadline_ns = (unsigned long long)c.deadline_us * 1000ull;
  p->debug_flags = c.debug_flags;
  p->early_weights = (c.launch_flags & GDN_LAUNCH_NO_EARLY_WEIGHTS) ? 0 : 1;
  p->x = (const __nv_bfloat16*)a.x;
  p->res = (const __nv_bfloat16*)a.residual;
  p->res_out = (__nv_bfloat16*)a.residual_out;
  p->core_out = (__nv_bfloat16*)a.core_out;
  p->idx = a.idx;
  p->conv_state = (__nv_bfloat16*)a.conv_state;
  p->ssm_state = a.ssm_state;
  const gdn_decode_weights* w = a.w;
  p->w_in = (const __nv_bfloat16*)w->input_norm_w;
  p->w_qkvz = (const __nv_bfloat16*)w->qkvz;
  p->w_qkvz_scales = w->qkvz_scales;
  p->fmt = c.qkvz_format;
  p->w_ba = (const __nv_bfloat16*)w->ba;
  p->conv_w = (const __nv_bfloat16*)w->conv_w;
  p->A_log = w->A_log;
  p->dt_bias = (const __nv_bfloat16*)w->dt_bias;
  p->gnorm_w = (const __nv_bfloat16*)w->gated_norm_w;
  p->out = (__nv_bfloat16*)a.out;
  p->w_out = a.out ? (const __nv_bfloat16*)w->out_proj : nullptr;
  p->ctr = (WsCounters*)(base + lay.ctr);
  p->core_flag = (unsigned long long*)(base + lay.core_flag);
  p->norm_part = (unsigned long long*)(base + lay.norm_part);
  p->proj_part = (unsigned long long*)(base + lay.proj_part);
  p->plan = (const PlanDev*)(base + lay.plan);
}

bool weight_maps(const gdn_decode_config& c, const gdn_decode_weights* w, MapCache* m, StepParams* p) {
  if (m->qkvz_ptr != w->qkvz || m->ba_ptr != w->ba) {
    if (!encode_maps(c, w, &m->qkvz, &m->ba)) {
      m->qkvz_ptr = m->ba_ptr = nullptr;
      return false;
    }
    m->qkvz_ptr = w->qkvz;
    m->ba_ptr = w->ba;
  }
  p->tm_qkvz = m->qkvz;
  p->tm_ba = m->ba;
  if (p->out) {
    if (m->out_ptr != w->out_proj) {
      if (!encode_out_map(&m->out, w->out_proj, c.hidden, c.num_v_heads * c.head_v_dim)) {
        m->out_ptr = nullptr;
        return false;
      }
      m->out_ptr = w->out_proj;
    }
    p->tm_out = m->out;
  }
  return true;
}

// One launch of the step kernel. Programmatic stream serialisation (while
// *pdl): the launch may start while the previous kernel in the stream
// finishes; the kernel reads only the weights it streams and the plan
// before its griddepcontrol.wait, or nothing with
// GDN_LAUNCH_NO_EARLY_WEIGHTS. Cooperative (on request): every CTA resident
// at once, guaranteed by the runtime. If the runtime refuses programmatic
// serialisation, *pdl is cleared and the launch goes without it.
gdn_status launch_step(const gdn_decode_config& c, const Plan& pl, bool* pdl, const StepParams& p, bool has_res,
                       cudaStream_t s) {
  const void* kern = pick_kernel(c, pl.engine, has_res, p.tokens > 1 || p.idx_out != nullptr);
  if (!kern) return GDN_ERR_UNSUPPORTED;
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(pl.G);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = kernel_smem(pl);
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (c.launch_flags & GDN_LAUNCH_COOPERATIVE) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na++].val.cooperative = 1;
  }
  if (*pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na++].val.programmaticStreamSerializationAllowed = 1;
  }
  lc.attrs = attr;
  lc.numAttrs = na;
  void* args[] = {const_cast<StepParams*>(&p)};
  cudaError_t e = cudaLaunchKernelExC(&lc, kern, args);
  if (e != cudaSuccess && *pdl) {
    (void)cudaGetLastError();
    *pdl = false;
    lc.numAttrs = na - 1;
    e = cudaLaunchKernelExC(&lc, kern, args);
  }
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// The launches of one step: rows in tiles of at most kMaxRows, one launch
// per tile in row order, each a whole step over its rows (rows are
// independent: distinct state slots; a verify step's tiles hold whole
// sequences). A step of up to kMaxRows rows is one launch; wider steps
// stream the weights once per tile.
gdn_status launch_row_tiles(const gdn_decode_config& c, const Plan& pl, const Layout& lay, char* base,
                            const StepArgs& a, MapCache* maps, bool* pdl, cudaStream_t s) {
  const size_t xrow = (size_t)c.hidden * 2, crow = (size_t)c.num_v_heads * c.head_v_dim * 2;
  const int tile_rows = kMaxRows / a.tokens * a.tokens;
  for (int r0 = 0; r0 < a.rows; r0 += tile_rows) {
    StepArgs t = a;
    t.rows = std::min(tile_rows, a.rows - r0);
    t.x = (const char*)a.x + r0 * xrow;
    t.residual = a.residual ? (const char*)a.residual + r0 * xrow : nullptr;
    t.idx = a.idx + r0 / a.tokens;
    t.idx_out = a.idx_out ? a.idx_out + r0 : nullptr;
    t.out = a.out ? (char*)a.out + r0 * xrow : nullptr;
    t.core_out = (char*)a.core_out + r0 * crow;
    t.residual_out = (char*)a.residual_out + r0 * xrow;
    StepParams p;  // on the stack: the step allocates nothing
    fill_params(c, pl, lay, base, t, &p);
    if (!weight_maps(c, a.w, maps, &p)) return GDN_ERR_CUDA;
    const gdn_status st = launch_step(c, pl, pdl, p, a.residual != nullptr, s);
    if (st != GDN_OK) return st;
  }
  return GDN_OK;
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
  if (resolve_plan(*cfg, G, pl) == GDN_OK) bytes = make_layout(*cfg, *pl).total;
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
  h->pdl = true;
  if (h->cfg.deadline_us == 0) h->cfg.deadline_us = 200000;
  int G;
  st = device_grid(h->cfg, &h->device, &h->num_sms, &G);
  if (st == GDN_OK) st = resolve_plan(h->cfg, G, &h->plan);
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
  const size_t smem = kernel_smem(h->plan);
  for (int r = 0; r < 4; ++r) {
    const void* k = pick_kernel(h->cfg, h->plan.engine, r & 1, r >= 2);
    if (!k && r >= 2) continue;  // no verify kernel for this config
    int per_sm = 0;
    if (!k || (smem && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                           cudaSuccess) ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem) != cudaSuccess || per_sm < 1) {
      delete h;
      return GDN_ERR_UNSUPPORTED;
    }
  }
  h->ws = workspace;
  h->ws_bytes = workspace_bytes;
  PlanDev* pd = new (std::nothrow) PlanDev;
  if (!pd) {
    delete h;
    return GDN_ERR_ARG;
  }
  memset(pd, 0, sizeof(*pd));
  memcpy(pd->unit_begin, h->plan.unit_begin, sizeof(int) * (h->plan.G + 1));
  memcpy(pd->seg_slot, h->plan.seg_slot, sizeof(h->plan.seg_slot[0]) * h->plan.G);
  memcpy(pd->ks_first, h->plan.ks_first, sizeof(unsigned short) * h->plan.G);
  memcpy(pd->nb_slots, h->plan.nb_slots, h->plan.G);
  memcpy(pd->tile_num_ctas, h->plan.tile_count, h->plan.num_tiles);
  memcpy(pd->own_mask, h->plan.own_mask, sizeof(unsigned int) * h->plan.G);
  // pageable source: the copy has staged it when the call returns
  const bool ok = cudaMemsetAsync(workspace, 0, h->lay.total, (cudaStream_t)stream) == cudaSuccess &&
                  cudaMemcpyAsync((char*)workspace + h->lay.plan, pd, sizeof(PlanDev), cudaMemcpyHostToDevice,
                                  (cudaStream_t)stream) == cudaSuccess;
  delete pd;
  if (!ok) {
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
  if (!h) return GDN_ERR_ARG;
  const StepArgs a{rows, x, residual, w, state_indices, conv_state, ssm_state, core_out, residual_out};
  gdn_status st = check_step_args(h->cfg, a, h->ws, h->lay.total);
  if (st != GDN_OK) return st;
  return launch_row_tiles(h->cfg, h->plan, h->lay, (char*)h->ws, a, &h->maps, &h->pdl, (cudaStream_t)stream);
}

gdn_status gdn_decode_step_out(gdn_decode_t* h, int32_t rows, const void* x, const void* residual,
                               const gdn_decode_weights* w, const int32_t* state_indices, void* conv_state,
                               void* ssm_state, void* core_out, void* residual_out, void* out, void* stream) {
  if (!h || !out) return GDN_ERR_ARG;
  StepArgs a{rows, x, residual, w, state_indices, conv_state, ssm_state, core_out, residual_out};
  a.out = out;
  gdn_status st = check_step_args(h->cfg, a, h->ws, h->lay.total);
  if (st != GDN_OK) return st;
  // the tensor-core kernel's out_proj phase: a freed weight ring large enough,
  // at most kOpMaxCols output columns per CTA, K a multiple of its chunk
  const Plan& pl = h->plan;
  const size_t ring = (size_t)pl.stages * kTileM * kKStep * 2 + (size_t)pl.rstages * (size_t)kTileM *
                                                                     (h->cfg.qkvz_format == GDN_W_MXFP6 ? 48 : 32);
  if (pl.engine != GDN_ENGINE_TCGEN05 || ring < tensor_core_out_proj_smem() ||
      (h->cfg.hidden + pl.G - 1) / pl.G > 64 || (h->cfg.num_v_heads * h->cfg.head_v_dim) % 256 != 0)
    return GDN_ERR_UNSUPPORTED;
  return launch_row_tiles(h->cfg, pl, h->lay, (char*)h->ws, a, &h->maps, &h->pdl, (cudaStream_t)stream);
}

gdn_status gdn_decode_verify(gdn_decode_t* h, int32_t seqs, int32_t tokens, const void* x, const void* residual,
                             const gdn_decode_weights* w, const int32_t* state_in, const int32_t* state_out,
                             void* conv_state, void* ssm_state, void* core_out, void* residual_out,
                             void* stream) {
  if (!h) return GDN_ERR_ARG;
  if (seqs < 1 || tokens < 1 || tokens > kMaxRows || (long long)seqs * tokens > h->cfg.max_rows) return GDN_ERR_ARG;
  StepArgs a{seqs * tokens, x, residual, w, state_in, conv_state, ssm_state, core_out, residual_out};
  a.tokens = tokens;
  a.idx_out = state_out;
  if (!state_out) return GDN_ERR_ARG;
  gdn_status st = check_step_args(h->cfg, a, h->ws, h->lay.total);
  if (st != GDN_OK) return st;
  if (!pick_kernel(h->cfg, h->plan.engine, residual != nullptr, true)) return GDN_ERR_UNSUPPORTED;
  return launch_row_tiles(h->cfg, h->plan, h->lay, (char*)h->ws, a, &h->maps, &h->pdl, (cudaStream_t)stream);
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
  return clear_launch_state((char*)h->ws, h->lay, (cudaStream_t)stream) ? GDN_OK : GDN_ERR_CUDA;
}

void gdn_decode_destroy(gdn_decode_t* h) { delete h; }

gdn_status gdn_decode_launch_info(const gdn_decode_t* h, int32_t rows, int32_t* num_ctas,
                                  int32_t* engine) {
  if (!h || rows < 1 || rows > h->cfg.max_rows) return GDN_ERR_ARG;
  if (num_ctas) *num_ctas = h->plan.G;
  if (engine) *engine = h->plan.engine;
  return GDN_OK;
}

gdn_status gdn_decode_debug_timeline(gdn_decode_t* h, void* stream, uint64_t* cta_stamps, int32_t cta_cap,
                                     int32_t* num_ctas) {
  if (!h || !cta_stamps || !num_ctas) return GDN_ERR_ARG;
  const int G = h->plan.G;
  if (cta_cap < G * kTlSlots) return GDN_ERR_ARG;
  const char* base = (const char*)h->ws + h->lay.ctr;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(cta_stamps, base + offsetof(WsCounters, tl_cta), sizeof(uint64_t) * G * kTlSlots,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return GDN_ERR_CUDA;
  *num_ctas = G;
  return GDN_OK;
}

gdn_status gdn_decode_plan(const gdn_decode_config* cfg, int32_t num_ctas, int32_t* engine,
                           int32_t* unit_begin, uint8_t* seg_slot, uint16_t* ks_first, uint8_t* nb_slots,
                           uint32_t* own_mask, uint8_t* tile_count, int32_t tile_cap, int32_t* num_tiles,
                           int32_t* ksteps, int32_t* kblock) {
  gdn_status st = validate(cfg);
  if (st != GDN_OK) return st;
  if (num_ctas < 1 || num_ctas > kMaxCtas || !engine || !unit_begin || !seg_slot || !ks_first ||
      !nb_slots || !own_mask || !tile_count || !num_tiles || !ksteps || !kblock)
    return GDN_ERR_ARG;
  Plan* pl = new (std::nothrow) Plan;
  if (!pl) return GDN_ERR_ARG;
  st = resolve_plan(*cfg, num_ctas, pl);
  if (st == GDN_OK && pl->num_tiles > tile_cap) st = GDN_ERR_ARG;
  if (st == GDN_OK) {
    *engine = pl->engine;
    memcpy(unit_begin, pl->unit_begin, sizeof(int32_t) * (num_ctas + 1));
    memcpy(seg_slot, pl->seg_slot, (size_t)kMaxSegs * num_ctas);
    memcpy(ks_first, pl->ks_first, sizeof(uint16_t) * num_ctas);
    memcpy(nb_slots, pl->nb_slots, num_ctas);
    memcpy(own_mask, pl->own_mask, sizeof(uint32_t) * num_ctas);
    memcpy(tile_count, pl->tile_count, pl->num_tiles);
    *num_tiles = pl->num_tiles;
    *ksteps = pl->ksteps;
    *kblock = pl->kblock;
  }
  delete pl;
  return st;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gdn_decode_step_static: the step with a fixed device scratch in place of a
// caller workspace. It serves callers that cannot allocate device memory: a
// host program with no PyTorch or other device allocator to hand over a
// workspace, or a runtime whose device memory all belongs to its own pool
// (a cudaMalloc would fail there, or fragment the pool). Nothing on this
// path allocates: the scratch is a file-scope device array, reserved when
// this module's device code is loaded, and the host state is file-scope too.
// ---------------------------------------------------------------------------

// One scratch per device: the layout of a caller workspace (counters, error
// word, plan tables, norm and projection partials) for configs that fit. In
// host code this name is only a handle for cudaGetSymbolAddress, never a
// device address.
static __device__ __align__(256) unsigned char g_static_scratch[GDN_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kStaticMaxDevices = 32;

// The unique id of the CUDA context current on this thread (0 if none), from
// the driver, looked up once. Ids are never reused within a process, so a
// set-up keyed on one cannot outlive its context (cudaDeviceReset, or
// another context made current).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = (CtxGetCurrentFn)f;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = (CtxGetIdFn)f;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

struct StaticDevice {
  bool ready;                // set up for `cfg` in context `ctx_id`
  unsigned long long ctx_id; // the context the scratch address belongs to
  gdn_decode_config cfg;     // the caller's config the scratch is set up for
  gdn_decode_config run;     // the same with defaults filled in
  void* scratch;             // this context's device address of g_static_scratch
  Layout lay;
  Plan plan;
  PlanDev staging;           // host image of the plan tables
  bool pdl;                  // launch with programmatic stream serialisation
  MapCache maps;             // weights the cached tile maps describe
};
StaticDevice g_static[kStaticMaxDevices];

// Set the current device's scratch up for `cfg` unless it already is in the
// current context: validate, plan, look up the scratch address, zero the
// counters, the error word and the partials, and copy the plan tables in,
// ordered on `stream`.
gdn_status static_setup(int dev, const gdn_decode_config* cfg, cudaStream_t stream, StaticDevice** out) {
  if (dev < 0 || dev >= kStaticMaxDevices) return GDN_ERR_UNSUPPORTED;
  StaticDevice& d = g_static[dev];
  *out = &d;
  const unsigned long long ctx = current_context_id();
  if (d.ready && ctx != 0 && ctx == d.ctx_id && memcmp(&d.cfg, cfg, sizeof(*cfg)) == 0) return GDN_OK;
  d.ready = false;
  gdn_status st = validate(cfg);
  if (st != GDN_OK) return st;
  d.run = *cfg;
  if (d.run.deadline_us == 0) d.run.deadline_us = 200000;
  int device, sms, G;
  st = device_grid(d.run, &device, &sms, &G);
  if (st == GDN_OK) st = resolve_plan(d.run, G, &d.plan);
  if (st != GDN_OK) return st;
  d.lay = make_layout(d.run, d.plan);
  if (d.lay.total > GDN_STATIC_SCRATCH_BYTES) return GDN_ERR_UNSUPPORTED;  // needs a caller workspace
  int coop = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
    return GDN_ERR_UNSUPPORTED;
  const size_t smem = kernel_smem(d.plan);
  for (int r = 0; r < 2; ++r) {
    const void* k = pick_kernel(d.run, d.plan.engine, r == 1);
    int per_sm = 0;
    if (!k || (smem && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                           cudaSuccess) ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem) != cudaSuccess || per_sm < 1)
      return GDN_ERR_UNSUPPORTED;
  }
  // the address of this context's copy of the array (the runtime has made a
  // context current by now)
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return GDN_ERR_CUDA;
  d.scratch = ptr;
  d.ctx_id = current_context_id();
  PlanDev& pd = d.staging;
  memset(&pd, 0, sizeof(pd));
  memcpy(pd.unit_begin, d.plan.unit_begin, sizeof(int) * (d.plan.G + 1));
  memcpy(pd.seg_slot, d.plan.seg_slot, sizeof(d.plan.seg_slot[0]) * d.plan.G);
  memcpy(pd.ks_first, d.plan.ks_first, sizeof(unsigned short) * d.plan.G);
  memcpy(pd.nb_slots, d.plan.nb_slots, d.plan.G);
  memcpy(pd.tile_num_ctas, d.plan.tile_count, d.plan.num_tiles);
  memcpy(pd.own_mask, d.plan.own_mask, sizeof(unsigned int) * d.plan.G);
  char* base = (char*)d.scratch;
  // pageable source: the copy has staged it when the call returns
  if (!clear_launch_state(base, d.lay, stream) ||
      cudaMemcpyAsync(base + d.lay.plan, &pd, sizeof(PlanDev), cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  d.maps = MapCache();
  d.pdl = true;
  d.cfg = *cfg;
  d.ready = d.ctx_id != 0;
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_decode_step_static(const gdn_decode_config* cfg, int32_t rows, const void* x,
                                             const void* residual, const gdn_decode_weights* w,
                                             const int32_t* state_indices, void* conv_state, void* ssm_state,
                                             void* core_out, void* residual_out, void* stream,
                                             uint32_t* detail) {
  if (!cfg || !w) return GDN_ERR_ARG;
  if (rows < 1 || rows > cfg->max_rows || cfg->max_rows > GDN_MAX_ROWS) return GDN_ERR_ARG;
  // argument errors come back before any CUDA call
  const StepArgs a{rows, x, residual, w, state_indices, conv_state, ssm_state, core_out, residual_out};
  gdn_status st = check_step_args(*cfg, a, nullptr, 0);
  if (st != GDN_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  StaticDevice* dp = nullptr;
  st = static_setup(dev, cfg, s, &dp);
  if (st != GDN_OK) return st;
  StaticDevice& d = *dp;
  st = check_step_args(d.run, a, d.scratch, d.lay.total);  // now also against the scratch
  if (st != GDN_OK) return st;
  char* base = (char*)d.scratch;
  st = launch_row_tiles(d.run, d.plan, d.lay, base, a, &d.maps, &d.pdl, s);
  if (st != GDN_OK || !detail) return st;

  uint32_t word = 0;
  const char* err = base + d.lay.ctr + offsetof(WsCounters, error);
  if (cudaMemcpyAsync(&word, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return GDN_ERR_CUDA;
  *detail = word;
  if (word == 0) return GDN_OK;
  // read and cleared: the next call starts from zero counters
  if (!clear_launch_state(base, d.lay, s)) return GDN_ERR_CUDA;
  const uint32_t code = word >> 24;
  if (code == GDN_ERR_DEADLINE) return GDN_ERR_DEADLINE;
  if (code == GDN_ERR_INDEX) return GDN_ERR_INDEX;
  return GDN_ERR_FAILED;
}
