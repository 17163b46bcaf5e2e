// Library-internal entry points shared between the translation units of the CUDA library.
// Not part of the C ABI.
#pragma once

#include "blasst.h"

namespace blasst {

// The head-group pipeline of blasst_attn_fwd_host, on the device workspace named in `a`.
blasst_status run_host_pipeline(const blasst_host_args& a);

// BLASST_OK when the current device is compute capability 10.3 and the kernels are set up on it.
blasst_status check_device();

}  // namespace blasst
