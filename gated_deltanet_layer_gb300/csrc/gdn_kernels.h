// Internal: kernel lookup between the host API and the kernel translation units.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Address of the persistent step kernel with the projection on the CUDA
// cores (bf16 weights, decode steps) for a combination of first-layer
// variant, state dtype and head dim; nullptr if there is none.
const void* cuda_core_kernel(bool has_res, bool state_bf16, int dk);

// The same with the projection on the tensor cores (tcgen05), for a decode
// step or (multi) a verify step. Both engines' dynamic shared memory depends
// on the weight ring's depth (stages), the code ring's (rstages; MXFP4 or
// MXFP6), the normed input window (xslots k-steps, doubled for MXFP4
// weights); the pad past the window; the static shared memory of the
// kernel; the deepest ring it supports.
const void* tensor_core_kernel(bool has_res, bool state_bf16, int dk, int fmt, bool multi);
size_t tensor_core_smem_bytes(int stages, int rstages, int xslots, int fmt);
uint32_t tensor_core_xpad(int xslots);
size_t tensor_core_static_smem();
int tensor_core_max_stages();
// Shared memory the out_proj phase needs in the freed weight ring.
size_t tensor_core_out_proj_smem();
int tensor_core_max_rstages();

}  // namespace gdn
