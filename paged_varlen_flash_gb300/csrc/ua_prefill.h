// ua_prefill.h -- launcher of the tensor-core prefill path (internal).
#pragma once

#include "ua_common.cuh"

namespace ua {

struct PrefillPlan {
    int kv_box_rows = 64;  // slots per TMA box of the paged caches
    int grid = 0;          // persistent CTAs
    int num_tiles = 0;     // work items (q tile, kv head, sequence)
    int launches = 0;      // kernels enqueued per call
};

// True when the tensor-core path is built for head size d.
bool prefill_supported(int d);

// True when the call's shape fits the tensor-core tile (128 packed rows hold
// whole GQA groups: g divides 128).
bool prefill_shape_ok(const FwdParams& p);

// Fill *plan for the call described by p.
void plan_prefill(const FwdParams& p, int num_sms, PrefillPlan* plan);

// Enqueue the prefill path (p.out receives the final bf16 rows).
cudaError_t launch_prefill(const PrefillPlan& plan, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, const FwdParams& p, cudaStream_t stream);

}  // namespace ua
