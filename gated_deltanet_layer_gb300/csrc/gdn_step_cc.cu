// The step kernel's CUDA-core instances: bf16 in_proj_qkvz and in_proj_ba
// with the projection's dot products as f32 FMA on the CUDA cores, reading the
// same TMA-fed weight ring and shared-memory normed input as the tensor-core
// instances, with the same plan, hand-offs and recurrence. It is the engine
// the tensor cores are measured against, width by width.
#include "gdn_step_kernel.cuh"

namespace gdn {

const void* cuda_core_kernel(bool has_res, bool state_bf16, int dk) {
#define GDN_PICK(R, B, D)                           \
  if (has_res == R && state_bf16 == B && dk == D) \
    return (const void*)&gdn_step_kernel<R, B, D, kFmtBf16Fma, false>;
  GDN_PICK(true, false, 128) GDN_PICK(true, true, 128) GDN_PICK(false, false, 128) GDN_PICK(false, true, 128)
  GDN_PICK(true, false, 64) GDN_PICK(true, true, 64) GDN_PICK(false, false, 64) GDN_PICK(false, true, 64)
#undef GDN_PICK
  return nullptr;
}

}  // namespace gdn
