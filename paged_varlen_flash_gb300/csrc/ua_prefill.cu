// ua_prefill.cu -- planner and launcher of the tensor-core prefill path.
// Head sizes 64 and 128 run the two-tile kernel (ua_prefill_pair.cu as the
// persistent work-list form, ua_prefill_grid.cu as the one-CTA-per-unit
// form); head size 256 runs the CTA-pair kernel of ua_prefill_cta2.cu.  The
// plan picks the KV segments (split partials merged by the combine kernel)
// and the launch form.
#include <algorithm>
#include <cstdint>

#include "ua_common.cuh"
#include "ua_prefill.h"
#include "ua_prefill_common.cuh"
#include "ua_tmap.h"

namespace ua {

using pf::kRows;

bool prefill_supported(int d) { return d == 64 || d == 128 || d == 256; }

void plan_prefill(const FwdParams& p, int num_sms, size_t workspace_bytes, PrefillPlan* plan) {
    *plan = PrefillPlan();
    plan->kv_box_rows = p.b;
    const int bn = 128;   // keys per KV tile of every tensor-core prefill kernel
    const int ppt = kRows / p.g;
    plan->num_tiles = (p.max_seqlen_q + ppt - 1) / ppt;
    // Split the keys into segments only when the (tile, kv head, sequence)
    // grid is too small to give every SM about four CTAs; each segment keeps
    // at least eight KV tiles.
    // CTAs per (sequence, kv head): tile pairs where the pair kernel serves d.
    // (the d = 256 kernel runs the tiles of a pair on two CTAs of a cluster)
    const int ctas = prefill_pair_supported(p.d) ? (plan->num_tiles + 1) / 2 : 2 * ((plan->num_tiles + 1) / 2);
    const int64_t base = (int64_t)ctas * p.hk * p.num_seqs;
    int splits = 1;
    if (base < 4LL * num_sms) {
        const int64_t want = (4LL * num_sms + base - 1) / base;
        const int64_t by_len = std::max<int64_t>(1, p.max_seqlen_k / (8 * bn));
        splits = (int)std::min<int64_t>(std::min<int64_t>(want, by_len), 64);
        const size_t per_split = (size_t)p.total_q * p.hq * (p.d + 2) * sizeof(float);
        splits = (int)std::min<size_t>((size_t)splits, per_split ? workspace_bytes / per_split : 1);
        if (splits < 1) splits = 1;
    }
    const bool pair = prefill_pair_supported(p.d);
    // The two-tile kernel's work list must hold every entry.
    while (pair && splits > 1 && pair_work_entries_bound(p, splits) > p.work_cap) --splits;
    if (splits > 1) {
        const int per = (p.max_seqlen_k + splits - 1) / splits;
        plan->chunk = (per + bn - 1) / bn * bn;
        splits = (p.max_seqlen_k + plan->chunk - 1) / plan->chunk;
    }
    plan->splits = splits;
    if (pair) {
        // Dense batches -- the padded grid (num_seqs x max_seqlen_q rows)
        // wastes at most a quarter on padding and fills every SM at least
        // twice -- run one CTA per unit over that grid; ragged ones run
        // persistent CTAs over the longest-first list (measured: the long
        // prefill 1.87 ms dense vs 2.06 persistent, the chunked batch 0.171
        // dense vs 0.137 persistent).
        const int64_t grid = (int64_t)p.num_seqs * ctas * splits * p.hk;
        plan->dense = (int64_t)p.num_seqs * p.max_seqlen_q * 4 <= (int64_t)p.total_q * 5 &&
                      grid >= 2LL * num_sms && grid <= 0x7fffffffLL;
        if (plan->dense) {
            plan->launches = splits > 1 ? 2 : 1;
        } else {
            // Persistent CTAs: one per SM, fewer when the call has fewer
            // units (bounded from the host-side maxima).
            plan->ctas = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms, grid));
            plan->launches = splits > 1 ? 3 : 2;   // planner, kernel[, combine]
        }
    } else {
        plan->launches = splits > 1 ? 2 : 1;
    }
}

bool prefill_shape_ok(const FwdParams& p) {
    // A tile holds floor(128 / g) positions of all g heads of one KV head;
    // when g does not divide 128 the last 128 mod g rows are padding.
    return prefill_supported(p.d) && p.g >= 1 && p.g <= kRows;
}

cudaError_t launch_prefill(const PrefillPlan& plan, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const FwdParams& p, cudaStream_t stream) {
    // Q map: [total_q, H_q, d] innermost first; box = one 64-wide panel x g heads
    // x floor(128/g) positions: the tile's packed rows (all 128 when g divides 128).
    CUtensorMap tq;
    cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.hq, (cuuint64_t)p.total_q};
    cuuint64_t strides[2] = {2ull * p.d, 2ull * p.d * p.hq};
    cuuint32_t box[3] = {64, (cuuint32_t)p.g, (cuuint32_t)(kRows / p.g)};
    if (!encode_bf16_sw128(&tq, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (plan.num_tiles <= 0) return cudaSuccess;
    CUtensorMap to;   // the output, boxed like Q
    if (!encode_bf16_sw128(&to, p.out, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (prefill_pair_supported(p.d))
        return plan.dense ? launch_prefill_grid(tq, tm_k, tm_v, to, p, (plan.num_tiles + 1) / 2, stream)
                          : launch_prefill_pair(tq, tm_k, tm_v, p, plan.ctas, stream);
    if (p.d != 256) return cudaErrorInvalidValue;
    return launch_prefill_cta2(tq, tm_k, tm_v, to, p, (plan.num_tiles + 1) / 2, stream);
}

}  // namespace ua
