// ua_prefill.h -- launcher of the tensor-core prefill path (internal).
#pragma once

#include "ua_common.cuh"

namespace ua {

struct PrefillPlan {
    int kv_box_rows = 64;  // slots per TMA box of the paged caches
    int num_tiles = 0;     // query tiles per (sequence, kv head) (grid x / splits)
    int splits = 1;        // KV segments per tile (1 = the kernel writes O itself)
    int chunk = 0;         // keys per segment (a multiple of the KV tile)
    int ctas = 0;          // persistent CTAs of the two-tile kernel (one per SM at most)
    bool dense = false;    // two-tile kernel as one CTA per unit over the padded grid
    int launches = 0;      // kernels enqueued per call
};

// True when the tensor-core path is built for head size d.
bool prefill_supported(int d);

// True when the call's shape fits the tensor-core tile (128 packed rows hold
// floor(128 / g) positions of whole GQA groups: g <= 128).
bool prefill_shape_ok(const FwdParams& p);

// Fill *plan for the call described by p; split partials may use up to
// `workspace_bytes` of the problem workspace.
void plan_prefill(const FwdParams& p, int num_sms, size_t workspace_bytes, PrefillPlan* plan);

// Head sizes served by the two-tiles-per-CTA kernel (256 query rows share each
// K/V tile); the others use one 128-row tile per CTA.
bool prefill_pair_supported(int d);

// Upper bound on the work-list entries (sequence, tile pair, KV segment) of
// the two-tile kernel for a call with `splits` segments:
// (total_q / (2 floor(128 / g)) + num_seqs) * splits.
int64_t pair_work_entries_bound(const FwdParams& p, int splits);

// Enqueue the two-tile kernel as one CTA per (tile pair, KV head, sequence[,
// segment]) over the padded grid of `pairs` tile pairs per sequence: the form
// for batches whose padded grid is nearly all real units (ua_prefill_grid.cu).
// `to` maps the output like tq maps Q (full tiles are stored through it).
cudaError_t launch_prefill_grid(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& to, const FwdParams& p, int pairs, cudaStream_t stream);

// Enqueue the planner (the longest-first work list in p.work_list) and the
// persistent two-tile kernel on `ctas` CTAs; tq is the Q tensor map (boxes of
// a tile's packed rows).
cudaError_t launch_prefill_pair(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const FwdParams& p, int ctas, cudaStream_t stream);

// Enqueue the head-size-256 kernel on CTA pairs: one cluster of two CTAs per
// (pair of adjacent query tiles, KV head, sequence[, segment]) over the padded
// grid of `pairs` tile pairs per sequence (ua_prefill_cta2.cu).
// `to` maps the output like tq maps Q (full tiles are stored through it).
cudaError_t launch_prefill_cta2(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& to, const FwdParams& p, int pairs, cudaStream_t stream);

// Enqueue the prefill path (p.out receives the final bf16 rows).
cudaError_t launch_prefill(const PrefillPlan& plan, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, const FwdParams& p, cudaStream_t stream);

}  // namespace ua
