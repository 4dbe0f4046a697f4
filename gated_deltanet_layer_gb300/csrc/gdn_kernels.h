// Internal: kernel lookup between the host API and the kernel translation units.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Address of the persistent step kernel (CUDA-core projection engine) for a
// combination of first-layer variant, state dtype and head dim; nullptr if
// there is none.
const void* cuda_core_kernel(bool has_res, bool state_bf16, int dk);

}  // namespace gdn
