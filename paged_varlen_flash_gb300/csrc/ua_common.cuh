// ua_common.cuh -- parameters shared by the forward kernels and the host
// planner, and the per-sequence metadata check every kernel applies the same way.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/ua.h"

namespace ua {

struct FwdParams {
    const __nv_bfloat16* q;        // [total_q, hq, d]
    const void* k_cache;           // [num_blocks, b, hk, d] (paths that read rows directly)
    const void* v_cache;
    const int32_t* block_table;    // [num_seqs, bt_stride]
    const int32_t* cu_seqlens_q;   // [num_seqs + 1]
    const int32_t* seqused_k;      // [num_seqs]
    const float* sinks;            // [hq] or null
    const float* alibi;            // [hq] or null
    const float* qq_bias;          // query-query bias B, element (a, c) at a * qq_stride + c, or null
    __nv_bfloat16* out;            // [total_q, hq, d]
    float* part_o;                 // [total_q * hq, splits, d] split partials
    float* part_ml;                // [total_q * hq, splits, 2] (m in log2 units, l)
    int32_t* err;                  // device error word
    int64_t total_q;
    int64_t num_blocks;
    int32_t num_seqs;
    int32_t bt_stride;
    int32_t max_seqlen_q;
    int32_t max_seqlen_k;
    int32_t hq, hk, g, d, b;
    uint32_t flags;
    float scale;                   // tau
    float softcap;                 // c
    int32_t window;                // W
    int32_t splits;                // split-KV segments per row (1 = direct)
    int32_t chunk;                 // keys per segment (multiple of 64)
    int32_t row_tiles;             // row tiles per (sequence, kv head)
    int32_t kv_fp8;                // caches hold e4m3 codes
    float k_scale, v_scale;        // fp8 caches: K = code * k_scale, V = code * v_scale
    int64_t qq_stride;             // row stride of qq_bias
    int32_t part_bf16;             // part_o holds bf16 (same element indexing) instead of fp32
    const int32_t* topk_idx;       // [total_q, topk_stride] key positions per query token, or null
    const int32_t* topk_len;       // [total_q] list lengths (with topk_idx)
    int32_t topk_stride;
    // Persistent prefill: the work list the planner kernel writes (entries
    // (sequence, tile pair << 7 | KV segment), longest first), its length and
    // claim counter, and the per-sequence exclusive prefix of entry counts.
    int2* work_list;
    int32_t* work_info;            // [0] entries, [1] claim counter
    int32_t* seq_prefix;           // [num_seqs + 1]
    int32_t work_cap;              // capacity of work_list in entries
    // Testing hook (ua_debug_stall_data_waits): when set, each kernel's first
    // consumer-side K/V data wait waits on a barrier that nothing completes,
    // bounded by stall_ns, so the bounded-wait abort path runs.
    int32_t stall;
    int64_t stall_ns;
};

// Per-sequence metadata check.  Returns UA_DEVERR_* bits (0 = well formed) and
// the sequence's S_q, S_k and first packed row.
__device__ __forceinline__ uint32_t seq_status(const FwdParams& p, int s, int& sq, int& sk,
                                               int64_t& q0) {
    const int32_t a = __ldg(p.cu_seqlens_q + s);
    const int32_t e = __ldg(p.cu_seqlens_q + s + 1);
    sk = __ldg(p.seqused_k + s);
    q0 = a;
    sq = e - a;
    uint32_t st = 0;
    if (a < 0 || e < a || (int64_t)e > p.total_q) {
        st |= UA_DEVERR_CU_SEQLENS;
        sq = 0;
        return st;
    }
    if (sk < sq) st |= UA_DEVERR_CONTEXT;
    if (sq > p.max_seqlen_q || sk > p.max_seqlen_k ||
        (int64_t)sk > (int64_t)p.bt_stride * p.b)
        st |= UA_DEVERR_BOUNDS;
    return st;
}

// Top-k calls: the list length of query token `token`, or -1 when it lies
// outside [0, topk_stride] (a malformed list; the token's rows are written as 0).
__device__ __forceinline__ int topk_length(const FwdParams& p, int64_t token) {
    const int n = __ldg(p.topk_len + token);
    return (n < 0 || n > p.topk_stride) ? -1 : n;
}

// Segments the token's list is split into (the top-k kernel and the combine
// kernel must agree): one per `chunk` entries, at least one.
__device__ __forceinline__ int topk_segments(const FwdParams& p, uint32_t st, int64_t token) {
    const int n = topk_length(p, token);
    if (st != 0 || n <= 0) return 1;
    const int k = (n + p.chunk - 1) / p.chunk;
    return k < p.splits ? k : p.splits;
}

// Split partials of o: fp32, or bf16 when p.part_bf16 (half the bytes, same
// element index; m and l stay fp32).
__device__ __forceinline__ void part_store(const FwdParams& p, int64_t idx, float v) {
    if (p.part_bf16)
        reinterpret_cast<__nv_bfloat16*>(p.part_o)[idx] = __float2bfloat16_rn(v);
    else
        p.part_o[idx] = v;
}

__device__ __forceinline__ float part_load(const FwdParams& p, int64_t idx) {
    return p.part_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.part_o)[idx])
                       : p.part_o[idx];
}

// 32 consecutive elements from fp32 bit patterns; idx is a multiple of 32.
__device__ __forceinline__ void part_store32(const FwdParams& p, int64_t idx, const uint32_t* o) {
    if (p.part_bf16) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.part_o) + idx);
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(o[e + 2 * k]),
                                                               __uint_as_float(o[e + 2 * k + 1]));
                w[k] = *reinterpret_cast<const uint32_t*>(&h);
            }
            dst[e / 8] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        float4* dst = reinterpret_cast<float4*>(p.part_o + idx);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
            dst[e / 4] = make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                     __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
    }
}

// Number of split segments sequence s uses (the split kernel and the combine
// kernel must agree on it).
__device__ __forceinline__ int seq_segments(const FwdParams& p, uint32_t st, int sk) {
    if (st != 0 || sk <= 0) return 1;
    int n = (sk + p.chunk - 1) / p.chunk;
    return n < p.splits ? n : p.splits;
}

}  // namespace ua
