// ua_decode_tc.h -- launcher of the transposed tensor-core decode kernel (internal).
#pragma once

#include "ua_common.cuh"

namespace ua {

struct DecodePlan {
    int kv_box_rows = 64;  // slots per TMA box of the paged caches
    int splits = 1;        // KV segments per (sequence, kv head)
    int chunk = 0;         // keys per segment (a multiple of 128)
    int launches = 0;      // kernels enqueued per call
};

// True when the call fits the kernel: d = 128, g <= 16 and every KV head
// has at most 16 packed query rows (g * max_seqlen_q <= 16).
bool decode_tc_shape_ok(const FwdParams& p);

void plan_decode_tc(const FwdParams& p, int num_sms, size_t workspace_bytes, DecodePlan* plan);

// Enqueue the kernel (p.splits / p.chunk / partial pointers set from the plan).
cudaError_t launch_decode_tc(const DecodePlan& plan, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const FwdParams& p, cudaStream_t stream);

}  // namespace ua
