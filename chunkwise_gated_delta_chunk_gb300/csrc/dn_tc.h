// Tensor-core kernel entry (bf16, dk = 128, dv a multiple of 128).
#pragma once

#include "dn_internal.h"

namespace dn {

bool tc_supported(int dk, int dv, bool bf16);
cudaError_t tc_launch(const Params &p, cudaStream_t stream, const char **name);

}  // namespace dn
