// Tensor-core path (bf16, dk = 128 or 256, dv a multiple of 128): the WY
// kernel (T of every chunk, into the workspace) and the scan kernel that
// reads it (dn_tc.cu for dk = 128, dn_tc_wide.cu for dk = 256).
#pragma once

#include <cuda.h>

#include "dn_internal.h"

namespace dn {

// chunk: tokens per chunk (16, 32 or 64; a chunk occupies the first `chunk`
// rows of the kernels' 64-row tiles).
bool tc_supported(int dk, int dv, bool bf16, int chunk);
// Workspace bytes the tensor-core path needs (0 for no tokens).
size_t tc_workspace_bytes(long long tokens, int N, int Nv, int dk, int chunk);
// The WY kernel and the scan kernel for p.dk (128 or 256).
cudaError_t tc_launch(const Params &p, cudaStream_t stream, const char **name);
cudaError_t tc_wide_launch(const Params &p, cudaStream_t stream, const char **name);
cudaError_t wy_launch(const Params &p, const CUtensorMap &mK, const CUtensorMap &mQ, cudaStream_t stream);

}  // namespace dn
