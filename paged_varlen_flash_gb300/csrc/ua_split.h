// ua_split.h -- launchers of the split-KV CUDA-core path (internal).
#pragma once

#include "ua_common.cuh"

namespace ua {

// Dynamic shared memory of the split kernel for head size d and row tile `rows`
// (-1 for an unsupported pair).
int split_smem_bytes(int d, int rows);

// Launch the split kernel with a row tile of `rows` packed rows (1, 2, 4, 8 or
// 16).  p.splits > 1 writes fp32 partials for launch_combine; p.splits == 1
// writes the final bf16 output directly.
cudaError_t launch_split(int rows, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                         const FwdParams& p, cudaStream_t stream);

// Merge the split partials of every row into the bf16 output.
cudaError_t launch_combine(const FwdParams& p, cudaStream_t stream);

}  // namespace ua
