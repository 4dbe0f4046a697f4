// The step kernel's tensor-core instances (tcgen05.mma projection) and the
// sizes the host plans its launches with.
#include "gdn_step_kernel.cuh"

namespace gdn {

const void* tensor_core_kernel(bool has_res, bool state_bf16, int dk, int fmt, bool multi) {
#define GDN_PICK(R, B, D, F, M)                                                         \
  if (has_res == R && state_bf16 == B && dk == D && fmt == F && multi == M)             \
    return (const void*)&gdn_step_kernel<R, B, D, F, M>;
  // decode steps: bf16 weights (head dim 64 or 128), MXFP4 and MXFP6 (head dim 128)
  GDN_PICK(true, false, 128, kFmtBf16, false) GDN_PICK(true, true, 128, kFmtBf16, false)
  GDN_PICK(false, false, 128, kFmtBf16, false) GDN_PICK(false, true, 128, kFmtBf16, false)
  GDN_PICK(true, false, 64, kFmtBf16, false) GDN_PICK(true, true, 64, kFmtBf16, false)
  GDN_PICK(false, false, 64, kFmtBf16, false) GDN_PICK(false, true, 64, kFmtBf16, false)
  GDN_PICK(true, false, 128, kFmtMxfp4, false) GDN_PICK(true, true, 128, kFmtMxfp4, false)
  GDN_PICK(false, false, 128, kFmtMxfp4, false) GDN_PICK(false, true, 128, kFmtMxfp4, false)
  GDN_PICK(true, false, 128, kFmtMxfp6, false) GDN_PICK(true, true, 128, kFmtMxfp6, false)
  GDN_PICK(false, false, 128, kFmtMxfp6, false) GDN_PICK(false, true, 128, kFmtMxfp6, false)
  // verify steps: bf16 weights
  GDN_PICK(true, false, 128, kFmtBf16, true) GDN_PICK(true, true, 128, kFmtBf16, true)
  GDN_PICK(false, false, 128, kFmtBf16, true) GDN_PICK(false, true, 128, kFmtBf16, true)
  GDN_PICK(true, false, 64, kFmtBf16, true) GDN_PICK(true, true, 64, kFmtBf16, true)
  GDN_PICK(false, false, 64, kFmtBf16, true) GDN_PICK(false, true, 64, kFmtBf16, true)
#undef GDN_PICK
  return nullptr;
}

// Dynamic shared memory of a launch: the bf16 weight ring, the code ring
// (MXFP4 or MXFP6), the normed-input window (and with MXFP4 weights its
// quantised copy) with the pad an M = 64 MMA reads past the last slice (also
// the norm sums' scratch), the window's input-norm weights, with MXFP6 the
// code-pair table, and 1 KB of alignment.
uint32_t tensor_core_xpad(int xslots) {
  const uint32_t sums = (uint32_t)(kMaxRows * xslots * 8 * sizeof(float));
  return sums > kXPadMin ? (sums + 127) / 128 * 128 : kXPadMin;
}
size_t tensor_core_smem_bytes(int stages, int rstages, int xslots, int fmt) {
  const size_t rtile = fmt == kFmtMxfp6 ? code_tile_bytes<kFmtMxfp6>() : code_tile_bytes<kFmtMxfp4>();
  return (size_t)stages * kWBytes + (size_t)rstages * rtile + (size_t)(fmt == kFmtMxfp4 ? 2 : 1) * xslots * kXBytes +
         tensor_core_xpad(xslots) + (size_t)xslots * kWinBytes + (fmt == kFmtMxfp6 ? kE2m3LutEntries * 4 : 0) + 1024;
}
size_t tensor_core_static_smem() { return sizeof(SmemPhases) + sizeof(SmemTask) + sizeof(TcShared); }
int tensor_core_max_stages() { return kMaxStages; }
size_t tensor_core_out_proj_smem() { return kOpRing; }
int tensor_core_max_rstages() { return kMaxRStages; }

}  // namespace gdn
