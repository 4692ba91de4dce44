// ua_topk.h -- launcher of the sparse top-k decode kernel (internal).
#pragma once

#include "ua_common.cuh"

namespace ua {

struct TopkPlan {
    int splits = 1;    // list segments per (query token, kv head)
    int chunk = 0;     // list entries per segment (a multiple of 128)
    int launches = 0;  // kernels enqueued per call
};

// True when the call fits the kernel: d = 128, g <= 16.
bool topk_shape_ok(const FwdParams& p);

// 2-D gather view of a bf16 cache: [num_blocks * b * H_k rows, d columns],
// box = one 64-column panel of one row.  False if the rows overflow int32.
bool encode_gather_map(CUtensorMap* m, const void* cache, int64_t num_blocks, int b, int hk, int d);

void plan_topk(const FwdParams& p, int num_sms, size_t workspace_bytes, TopkPlan* plan);

// Enqueue the kernel (p.splits / p.chunk / partial pointers set from the plan).
cudaError_t launch_topk(const TopkPlan& plan, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const FwdParams& p, cudaStream_t stream);

}  // namespace ua
