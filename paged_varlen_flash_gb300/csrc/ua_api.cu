// ua_api.cu -- the C ABI of include/ua.h: argument validation, the problem-
// owned workspace, tensor-map encoding, and the host planner that picks the
// execution path and launch shape for each call (gfx950 "Unified paged
// attention on gfx950, from the math up", section 6: choose between a path
// whose query-tile grid already fills the device and a split-KV path plus a
// reduction when it does not).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ua_common.cuh"
#include "ua_decode_tc.h"
#include "ua_prefill.h"
#include "ua_split.h"
#include "ua_tmap.h"
#include "ua_topk.h"

namespace {

thread_local char g_cuda_err[256] = "";

void note_cuda(cudaError_t e, const char* where) {
    std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", where, cudaGetErrorString(e));
}

constexpr int kMaxSplits = 64;
constexpr size_t kWorkspaceCap = size_t(128) << 20;  // bytes of split partials

// Cache map of the problem's caches with boxes of `box_rows` slots.
bool encode_cache_map(CUtensorMap* m, const void* base, const ua_problem_desc& d, int box_rows) {
    return ua::encode_cache_map(m, base, d.head_size, d.num_kv_heads, d.block_size, d.num_blocks,
                                d.kv_dtype == UA_DTYPE_FP8_E4M3, box_rows);
}

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

}  // namespace

struct ua_problem {
    ua_problem_desc desc;
    int device = 0;
    int num_sms = 0;
    int32_t* d_err = nullptr;
    float* d_ws = nullptr;
    size_t ws_bytes = 0;
    // work list of the persistent prefill kernel: entries, then the
    // per-sequence prefix, then [entries, claim counter]
    void* d_work = nullptr;
    int32_t work_cap = 0;
    // staging buffers of ua_forward_host (allocated on first use)
    void* st_q = nullptr;
    void* st_out = nullptr;
    int32_t* st_bt = nullptr;
    int32_t* st_cu = nullptr;
    int32_t* st_su = nullptr;
    float* st_sinks = nullptr;
    float* st_alibi = nullptr;
    // query-query bias set by ua_set_qq_bias (caller-owned device memory)
    const float* qq_bias = nullptr;
    int64_t qq_n = 0;
    int64_t qq_stride = 0;
    // tensor maps of the most recent caches (re-encoded when the pointers change)
    const void* map_k_ptr = nullptr;
    const void* map_v_ptr = nullptr;
    CUtensorMap map_k16, map_v16;       // 16-slot boxes (split path)
    CUtensorMap map_kp, map_vp;         // prefill-path boxes
    int map_p_rows = 0;
    const void* map_g_k_ptr = nullptr;  // row-gather views of the caches (top-k calls)
    const void* map_g_v_ptr = nullptr;
    CUtensorMap map_kg, map_vg;
    int last_launches = 0;
    const char* last_path = "none";
    cudaEvent_t prof_begin = nullptr;
    cudaEvent_t prof_end = nullptr;
    // testing hook of ua_debug_stall_data_waits
    int32_t stall = 0;
    int64_t stall_ns = 0;
};

namespace {
void prof_mark(const ua_problem* p, bool begin, cudaStream_t st) {
    if (p->prof_begin && p->prof_end) cudaEventRecord(begin ? p->prof_begin : p->prof_end, st);
}
}  // namespace

extern "C" {

const char* ua_status_string(ua_status s) {
    switch (s) {
        case UA_OK: return "ok";
        case UA_ERR_INVALID_ARG: return "invalid argument";
        case UA_ERR_UNSUPPORTED: return "unsupported configuration";
        case UA_ERR_CUDA: return "CUDA error";
        case UA_ERR_OUT_OF_MEMORY: return "out of device memory";
        case UA_ERR_DEVICE: return "device reported an input error";
    }
    return "unknown status";
}

const char* ua_last_cuda_error(void) { return g_cuda_err; }

ua_status ua_problem_create(const ua_problem_desc* d, ua_problem** out) {
    if (!d || !out) return UA_ERR_INVALID_ARG;
    *out = nullptr;
    const uint32_t known = UA_FLAG_CAUSAL | UA_FLAG_SOFTCAP | UA_FLAG_ALIBI | UA_FLAG_WINDOW |
                           UA_FLAG_SINKS | UA_FLAG_QQ_BIAS;
    if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_q_heads % d->num_kv_heads != 0)
        return UA_ERR_INVALID_ARG;
    if (d->num_blocks <= 0 || d->max_num_seqs <= 0 || d->max_blocks_per_seq <= 0 ||
        d->max_total_q <= 0 || d->head_size <= 0 || d->block_size <= 0)
        return UA_ERR_INVALID_ARG;
    if (d->flags & ~known) return UA_ERR_INVALID_ARG;
    if (!(d->scale > 0.f) || !std::isfinite(d->scale)) return UA_ERR_INVALID_ARG;
    if ((d->flags & UA_FLAG_SOFTCAP) && !(d->softcap > 0.f && std::isfinite(d->softcap)))
        return UA_ERR_INVALID_ARG;
    if ((d->flags & UA_FLAG_WINDOW) && (d->window < 1 || !(d->flags & UA_FLAG_CAUSAL)))
        return UA_ERR_INVALID_ARG;
    if (d->dtype != UA_DTYPE_BF16) return UA_ERR_UNSUPPORTED;
    if (d->kv_dtype != UA_DTYPE_BF16 && d->kv_dtype != UA_DTYPE_FP8_E4M3) return UA_ERR_INVALID_ARG;
    if (d->kv_dtype == UA_DTYPE_FP8_E4M3) {
        if (!(d->k_scale > 0.f) || !std::isfinite(d->k_scale) || !(d->v_scale > 0.f) ||
            !std::isfinite(d->v_scale))
            return UA_ERR_INVALID_ARG;
        // Only the decode tensor-core kernel reads an fp8 cache.
        if (d->head_size != 128) return UA_ERR_UNSUPPORTED;
        if (d->path != UA_PATH_AUTO && d->path != UA_PATH_DECODE_TC) return UA_ERR_UNSUPPORTED;
    }
    if (d->head_size != 64 && d->head_size != 128 && d->head_size != 256) return UA_ERR_UNSUPPORTED;
    if (d->block_size != 16 && d->block_size != 32 && d->block_size != 64) return UA_ERR_UNSUPPORTED;
    if (d->num_blocks > (int64_t(1) << 31) - 1) return UA_ERR_UNSUPPORTED;
    if (d->path > UA_PATH_DECODE_TC) return UA_ERR_INVALID_ARG;
    if (d->split_partials != UA_PARTIALS_F32 && d->split_partials != UA_PARTIALS_BF16)
        return UA_ERR_INVALID_ARG;

    ua_problem* p = new (std::nothrow) ua_problem();
    if (!p) return UA_ERR_OUT_OF_MEMORY;
    p->desc = *d;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) {
        note_cuda(e, "ua_problem_create");
        delete p;
        return UA_ERR_CUDA;
    }
    const size_t row_bytes = size_t(d->head_size + 2) * sizeof(float);
    const size_t want = size_t(d->max_total_q) * d->num_q_heads * row_bytes * 16;
    p->ws_bytes = std::min(want, kWorkspaceCap);
    // Work-list entries: every call's (total_q / (2 ppt) + num_seqs) entries
    // without a KV split, and room for the splits the planner makes when the
    // grid is small (about 4 x 152 units per KV head x up to 64 segments).
    const int64_t cap = std::min<int64_t>(d->max_total_q + d->max_num_seqs + 64 * 4 * 160,
                                          int64_t(1) << 30);
    p->work_cap = (int32_t)cap;
    const size_t work_bytes = (size_t)cap * sizeof(int2) + (size_t)(d->max_num_seqs + 1) * 4 + 16;
    if (cudaMalloc(&p->d_err, sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&p->d_ws, p->ws_bytes) != cudaSuccess ||
        cudaMalloc(&p->d_work, work_bytes) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->d_err);
        cudaFree(p->d_ws);
        delete p;
        return UA_ERR_OUT_OF_MEMORY;
    }
    e = cudaMemset(p->d_err, 0, sizeof(int32_t));
    if (e != cudaSuccess) {
        note_cuda(e, "ua_problem_create");
        cudaFree(p->d_err);
        cudaFree(p->d_ws);
        cudaFree(p->d_work);
        delete p;
        return UA_ERR_CUDA;
    }
    *out = p;
    return UA_OK;
}

void ua_destroy(ua_problem* p) {
    if (!p) return;
    cudaFree(p->d_err);
    cudaFree(p->d_ws);
    cudaFree(p->d_work);
    cudaFree(p->st_q);
    cudaFree(p->st_out);
    cudaFree(p->st_bt);
    cudaFree(p->st_cu);
    cudaFree(p->st_su);
    cudaFree(p->st_sinks);
    cudaFree(p->st_alibi);
    delete p;
}

int32_t ua_last_launch_count(const ua_problem* p) { return p ? p->last_launches : 0; }

const char* ua_last_path(const ua_problem* p) { return p ? p->last_path : "none"; }

ua_status ua_set_qq_bias(ua_problem* p, const float* bias, int64_t n, int64_t row_stride) {
    if (!p || !(p->desc.flags & UA_FLAG_QQ_BIAS)) return UA_ERR_INVALID_ARG;
    if (!bias) {
        p->qq_bias = nullptr;
        p->qq_n = p->qq_stride = 0;
        return UA_OK;
    }
    if (n < 1 || row_stride < n || (reinterpret_cast<uintptr_t>(bias) & 3u) != 0)
        return UA_ERR_INVALID_ARG;
    p->qq_bias = bias;
    p->qq_n = n;
    p->qq_stride = row_stride;
    return UA_OK;
}

ua_status ua_debug_stall_data_waits(ua_problem* p, int32_t enable, int64_t limit_ns) {
    if (!p) return UA_ERR_INVALID_ARG;
    if (enable && (limit_ns < 1000 || limit_ns > 1000000000)) return UA_ERR_INVALID_ARG;
    p->stall = enable ? 1 : 0;
    p->stall_ns = enable ? limit_ns : 0;
    return UA_OK;
}

ua_status ua_set_profile_events(ua_problem* p, void* ev_begin, void* ev_end) {
    if (!p || ((ev_begin == nullptr) != (ev_end == nullptr))) return UA_ERR_INVALID_ARG;
    p->prof_begin = reinterpret_cast<cudaEvent_t>(ev_begin);
    p->prof_end = reinterpret_cast<cudaEvent_t>(ev_end);
    return UA_OK;
}

}  // extern "C"

namespace {

// Host checks shared by the forward entry points, then the kernel parameters.
// Returns UA_OK with *skip set when the call has nothing to compute.
ua_status prepare_call(ua_problem* p, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* cu_seqlens_q,
                       const int32_t* seqused_k, int32_t num_seqs, int64_t total_q,
                       int32_t max_seqlen_q, int32_t max_seqlen_k, uint32_t flags,
                       const float* sinks, const float* alibi_slopes, void* out,
                       ua::FwdParams* fpp, bool* skip) {
    *skip = false;
    if (!p) return UA_ERR_INVALID_ARG;
    p->last_launches = 0;
    p->last_path = "none";
    const ua_problem_desc& d = p->desc;
    if (num_seqs < 0 || num_seqs > d.max_num_seqs || total_q < 0 || total_q > d.max_total_q)
        return UA_ERR_INVALID_ARG;
    if (max_seqlen_q < 0 || max_seqlen_k < 0 || max_seqlen_q > max_seqlen_k ||
        (int64_t)max_seqlen_k > (int64_t)d.max_blocks_per_seq * d.block_size)
        return UA_ERR_INVALID_ARG;
    if ((flags & ~d.flags) != 0) return UA_ERR_INVALID_ARG;
    if ((flags & UA_FLAG_WINDOW) && !(flags & UA_FLAG_CAUSAL)) return UA_ERR_INVALID_ARG;
    if (((flags & UA_FLAG_SINKS) != 0) != (sinks != nullptr)) return UA_ERR_INVALID_ARG;
    if (((flags & UA_FLAG_ALIBI) != 0) != (alibi_slopes != nullptr)) return UA_ERR_INVALID_ARG;
    if ((flags & UA_FLAG_QQ_BIAS) && (!p->qq_bias || (int64_t)max_seqlen_q > p->qq_n))
        return UA_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0) {
        *skip = true;
        return UA_OK;
    }
    if (num_seqs > 65535) return UA_ERR_UNSUPPORTED;   // grids index sequences on gridDim.z
    if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seqused_k || !out)
        return UA_ERR_INVALID_ARG;
    auto misaligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
    if (misaligned(q) || misaligned(out) || misaligned(k_cache) || misaligned(v_cache))
        return UA_ERR_INVALID_ARG;
    if (max_seqlen_k == 0) {
        // Only empty sequences can be well formed; nothing to compute.
        max_seqlen_k = 1;
        if (max_seqlen_q > 1) return UA_ERR_INVALID_ARG;
    }

    ua::FwdParams& fp = *fpp;
    std::memset(&fp, 0, sizeof fp);
    fp.q = static_cast<const __nv_bfloat16*>(q);
    fp.k_cache = k_cache;
    fp.v_cache = v_cache;
    fp.block_table = block_table;
    fp.cu_seqlens_q = cu_seqlens_q;
    fp.seqused_k = seqused_k;
    fp.sinks = sinks;
    fp.alibi = alibi_slopes;
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.err = p->d_err;
    fp.total_q = total_q;
    fp.num_blocks = d.num_blocks;
    fp.num_seqs = num_seqs;
    fp.bt_stride = d.max_blocks_per_seq;
    fp.max_seqlen_q = max_seqlen_q;
    fp.max_seqlen_k = max_seqlen_k;
    fp.hq = d.num_q_heads;
    fp.hk = d.num_kv_heads;
    fp.g = d.num_q_heads / d.num_kv_heads;
    fp.d = d.head_size;
    fp.b = d.block_size;
    fp.flags = flags;
    fp.scale = d.scale;
    fp.softcap = d.softcap;
    fp.window = d.window;
    fp.kv_fp8 = d.kv_dtype == UA_DTYPE_FP8_E4M3 ? 1 : 0;
    fp.k_scale = fp.kv_fp8 ? d.k_scale : 1.f;
    fp.v_scale = fp.kv_fp8 ? d.v_scale : 1.f;
    fp.part_bf16 = d.split_partials == UA_PARTIALS_BF16 ? 1 : 0;
    fp.work_list = static_cast<int2*>(p->d_work);
    fp.seq_prefix = reinterpret_cast<int32_t*>(fp.work_list + p->work_cap);
    fp.work_info = fp.seq_prefix + (d.max_num_seqs + 1);
    fp.work_cap = p->work_cap;
    fp.stall = p->stall;
    fp.stall_ns = p->stall_ns;
    if (flags & UA_FLAG_QQ_BIAS) {
        fp.qq_bias = p->qq_bias;
        fp.qq_stride = p->qq_stride;
    }
    return UA_OK;
}

}  // namespace

extern "C" {

ua_status ua_forward(ua_problem* p, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_table, const int32_t* cu_seqlens_q,
                     const int32_t* seqused_k, int32_t num_seqs, int64_t total_q,
                     int32_t max_seqlen_q, int32_t max_seqlen_k, uint32_t flags,
                     const float* sinks, const float* alibi_slopes, void* out, void* stream) {
    ua::FwdParams fp;
    bool skip = false;
    ua_status rs = prepare_call(p, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                                num_seqs, total_q, max_seqlen_q, max_seqlen_k, flags, sinks,
                                alibi_slopes, out, &fp, &skip);
    if (rs != UA_OK || skip) return rs;
    const ua_problem_desc& d = p->desc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int g = fp.g;
    max_seqlen_k = fp.max_seqlen_k;

    if (k_cache != p->map_k_ptr || v_cache != p->map_v_ptr) {
        if (!encode_cache_map(&p->map_k16, k_cache, d, 16) ||
            !encode_cache_map(&p->map_v16, v_cache, d, 16)) {
            p->map_k_ptr = p->map_v_ptr = nullptr;
            std::snprintf(g_cuda_err, sizeof g_cuda_err, "cuTensorMapEncodeTiled failed");
            return UA_ERR_CUDA;
        }
        p->map_k_ptr = k_cache;
        p->map_v_ptr = v_cache;
        p->map_p_rows = 0;
    }

    // ---- path choice ------------------------------------------------------
    const int64_t rows_per_kv = (int64_t)g * max_seqlen_q;
    const bool tc_ok = ua::prefill_shape_ok(fp);
    const bool dec_ok = ua::decode_tc_shape_ok(fp);
    bool use_dec = dec_ok;
    bool use_tc = !dec_ok && tc_ok && rows_per_kv > 16;
    if (d.path == UA_PATH_SPLIT_KV) use_dec = use_tc = false;
    if (d.path == UA_PATH_TENSOR_CORE) {
        if (!tc_ok) return UA_ERR_UNSUPPORTED;
        use_dec = false;
        use_tc = true;
    }
    if (d.path == UA_PATH_DECODE_TC || fp.kv_fp8) {
        if (!dec_ok) return UA_ERR_UNSUPPORTED;   // an fp8 cache is read by this kernel only
        use_dec = true;
        use_tc = false;
    }
    if (use_dec || use_tc) {
        // Both tensor-core kernels read the caches through boxes of b slots.
        if (p->map_p_rows != d.block_size) {
            if (!encode_cache_map(&p->map_kp, k_cache, d, d.block_size) ||
                !encode_cache_map(&p->map_vp, v_cache, d, d.block_size)) {
                std::snprintf(g_cuda_err, sizeof g_cuda_err, "cuTensorMapEncodeTiled failed");
                p->map_p_rows = 0;
                return UA_ERR_CUDA;
            }
            p->map_p_rows = d.block_size;
        }
    }
    if (use_dec) {
        ua::DecodePlan plan;
        ua::plan_decode_tc(fp, p->num_sms, p->ws_bytes, &plan);
        fp.splits = plan.splits;
        fp.chunk = plan.chunk;
        fp.part_o = p->d_ws;
        fp.part_ml = p->d_ws + (size_t)total_q * d.num_q_heads * plan.splits * d.head_size;
        prof_mark(p, true, st);
        cudaError_t e = ua::launch_decode_tc(plan, p->map_kp, p->map_vp, fp, st);
        prof_mark(p, false, st);
        if (e != cudaSuccess) {
            note_cuda(e, "decode kernel launch");
            return UA_ERR_CUDA;
        }
        if (plan.splits > 1) {
            e = ua::launch_combine(fp, st);
            if (e != cudaSuccess) {
                note_cuda(e, "combine kernel launch");
                return UA_ERR_CUDA;
            }
        }
        p->last_launches = plan.launches;
        p->last_path = plan.splits > 1 ? "decode_tc+combine" : "decode_tc";
        return UA_OK;
    }
    if (use_tc) {
        ua::PrefillPlan plan;
        ua::plan_prefill(fp, p->num_sms, p->ws_bytes, &plan);
        fp.splits = plan.splits;
        fp.chunk = plan.chunk;
        fp.part_o = p->d_ws;
        fp.part_ml = p->d_ws + (size_t)total_q * d.num_q_heads * plan.splits * d.head_size;
        prof_mark(p, true, st);
        cudaError_t e = ua::launch_prefill(plan, p->map_kp, p->map_vp, fp, st);
        prof_mark(p, false, st);
        if (e != cudaSuccess) {
            note_cuda(e, "prefill kernel launch");
            return UA_ERR_CUDA;
        }
        if (plan.splits > 1) {
            e = ua::launch_combine(fp, st);
            if (e != cudaSuccess) {
                note_cuda(e, "combine kernel launch");
                return UA_ERR_CUDA;
            }
        }
        p->last_launches = plan.launches;
        if (ua::prefill_pair_supported(fp.d) && plan.dense)
            p->last_path = plan.splits > 1 ? "tensor_core_grid+combine" : "tensor_core_grid";
        else if (ua::prefill_pair_supported(fp.d))
            p->last_path = plan.splits > 1 ? "tensor_core_pair+combine" : "tensor_core_pair";
        else
            p->last_path = plan.splits > 1 ? "tensor_core_cta2+combine" : "tensor_core_cta2";
        return UA_OK;
    }

    int rows = 1;
    int row_tiles = 1;
    if (rows_per_kv <= 16) {
        while (rows < rows_per_kv) rows <<= 1;
    } else {
        rows = 16;
        row_tiles = ceil_div(rows_per_kv, 16);
    }
    const int smem = ua::split_smem_bytes(d.head_size, rows);
    const int cps = std::max(1, std::min(8, (228 * 1024) / (smem + 1024)));
    const int64_t base = (int64_t)num_seqs * d.num_kv_heads * row_tiles;
    const int64_t slots = (int64_t)p->num_sms * cps;
    int splits = (int)std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, (4 * slots + base - 1) / base));
    splits = std::min(splits, std::max(1, ceil_div(max_seqlen_k, 256)));
    const size_t per_split = (size_t)total_q * d.num_q_heads * (d.head_size + 2) * sizeof(float);
    splits = (int)std::min<size_t>((size_t)splits, p->ws_bytes / per_split);
    if (splits < 1) splits = 1;
    int chunk = ceil_div(ceil_div(max_seqlen_k, splits), 64) * 64;
    splits = ceil_div(max_seqlen_k, chunk);
    if (row_tiles * (int64_t)d.num_kv_heads > 0x7fffffffLL || splits > 65535) return UA_ERR_UNSUPPORTED;
    fp.splits = splits;
    fp.chunk = chunk;
    fp.row_tiles = row_tiles;
    fp.part_o = p->d_ws;
    fp.part_ml = p->d_ws + (size_t)total_q * d.num_q_heads * splits * d.head_size;

    prof_mark(p, true, st);
    cudaError_t e = ua::launch_split(rows, p->map_k16, p->map_v16, fp, st);
    prof_mark(p, false, st);
    if (e != cudaSuccess) {
        note_cuda(e, "split kernel launch");
        return UA_ERR_CUDA;
    }
    p->last_launches = 1;
    if (splits > 1) {
        e = ua::launch_combine(fp, st);
        if (e != cudaSuccess) {
            note_cuda(e, "combine kernel launch");
            return UA_ERR_CUDA;
        }
        p->last_launches = 2;
        p->last_path = "split_kv+combine";
    } else {
        p->last_path = "split_kv_direct";
    }
    return UA_OK;
}

ua_status ua_forward_topk(ua_problem* p, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const int32_t* cu_seqlens_q,
                          const int32_t* seqused_k, int32_t num_seqs, int64_t total_q,
                          int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t* topk_idx,
                          const int32_t* topk_len, int32_t topk_stride, uint32_t flags,
                          const float* sinks, const float* alibi_slopes, void* out, void* stream) {
    ua::FwdParams fp;
    bool skip = false;
    ua_status rs = prepare_call(p, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                                num_seqs, total_q, max_seqlen_q, max_seqlen_k, flags, sinks,
                                alibi_slopes, out, &fp, &skip);
    if (rs != UA_OK) return rs;
    if (topk_stride < 1) return UA_ERR_INVALID_ARG;
    if (topk_stride > (1 << 30)) return UA_ERR_UNSUPPORTED;   // entry indices stay in int32
    if (skip) return UA_OK;
    if (!topk_idx || !topk_len) return UA_ERR_INVALID_ARG;
    const ua_problem_desc& d = p->desc;
    if (d.kv_dtype != UA_DTYPE_BF16) return UA_ERR_UNSUPPORTED;
    if (d.path != UA_PATH_AUTO && d.path != UA_PATH_DECODE_TC) return UA_ERR_UNSUPPORTED;
    fp.topk_idx = topk_idx;
    fp.topk_len = topk_len;
    fp.topk_stride = topk_stride;
    if (!ua::topk_shape_ok(fp)) return UA_ERR_UNSUPPORTED;
    if (k_cache != p->map_g_k_ptr || v_cache != p->map_g_v_ptr) {
        if (!ua::encode_gather_map(&p->map_kg, k_cache, d.num_blocks, d.block_size, d.num_kv_heads,
                                   d.head_size) ||
            !ua::encode_gather_map(&p->map_vg, v_cache, d.num_blocks, d.block_size, d.num_kv_heads,
                                   d.head_size)) {
            p->map_g_k_ptr = p->map_g_v_ptr = nullptr;
            // Either the cache's rows overflow the gather's 32-bit row index
            // or the encoder failed.
            if ((int64_t)d.num_blocks * d.block_size * d.num_kv_heads > 0x7fffffffLL)
                return UA_ERR_UNSUPPORTED;
            std::snprintf(g_cuda_err, sizeof g_cuda_err, "cuTensorMapEncodeTiled failed");
            return UA_ERR_CUDA;
        }
        p->map_g_k_ptr = k_cache;
        p->map_g_v_ptr = v_cache;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ua::TopkPlan plan;
    ua::plan_topk(fp, p->num_sms, p->ws_bytes, &plan);
    fp.splits = plan.splits;
    fp.chunk = plan.chunk;
    fp.part_o = p->d_ws;
    fp.part_ml = p->d_ws + (size_t)total_q * d.num_q_heads * plan.splits * d.head_size;
    prof_mark(p, true, st);
    cudaError_t e = ua::launch_topk(plan, p->map_kg, p->map_vg, fp, st);
    prof_mark(p, false, st);
    if (e != cudaSuccess) {
        note_cuda(e, "top-k kernel launch");
        return UA_ERR_CUDA;
    }
    if (plan.splits > 1) {
        e = ua::launch_combine(fp, st);
        if (e != cudaSuccess) {
            note_cuda(e, "combine kernel launch");
            return UA_ERR_CUDA;
        }
    }
    p->last_launches = plan.launches;
    p->last_path = plan.splits > 1 ? "topk_tc+combine" : "topk_tc";
    return UA_OK;
}

ua_status ua_forward_host(ua_problem* p, const void* q_host, const void* k_cache,
                          const void* v_cache, const int32_t* block_table_host,
                          const int32_t* cu_seqlens_q_host, const int32_t* seqused_k_host,
                          int32_t num_seqs, int64_t total_q, int32_t max_seqlen_q,
                          int32_t max_seqlen_k, uint32_t flags, const float* sinks_host,
                          const float* alibi_host, void* out_host, void* stream) {
    if (!p) return UA_ERR_INVALID_ARG;
    const ua_problem_desc& d = p->desc;
    if (num_seqs < 0 || num_seqs > d.max_num_seqs || total_q < 0 || total_q > d.max_total_q)
        return UA_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0) return UA_OK;
    if (!q_host || !block_table_host || !cu_seqlens_q_host || !seqused_k_host || !out_host)
        return UA_ERR_INVALID_ARG;
    const size_t qbytes_max = (size_t)d.max_total_q * d.num_q_heads * d.head_size * 2;
    if (!p->st_q) {
        bool ok = cudaMalloc(&p->st_q, qbytes_max) == cudaSuccess &&
                  cudaMalloc(&p->st_out, qbytes_max) == cudaSuccess &&
                  cudaMalloc(&p->st_bt, (size_t)d.max_num_seqs * d.max_blocks_per_seq * 4) == cudaSuccess &&
                  cudaMalloc(&p->st_cu, (size_t)(d.max_num_seqs + 1) * 4) == cudaSuccess &&
                  cudaMalloc(&p->st_su, (size_t)d.max_num_seqs * 4) == cudaSuccess &&
                  cudaMalloc(&p->st_sinks, (size_t)d.num_q_heads * 4) == cudaSuccess &&
                  cudaMalloc(&p->st_alibi, (size_t)d.num_q_heads * 4) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            cudaFree(p->st_q); cudaFree(p->st_out); cudaFree(p->st_bt); cudaFree(p->st_cu);
            cudaFree(p->st_su); cudaFree(p->st_sinks); cudaFree(p->st_alibi);
            p->st_q = p->st_out = nullptr;
            p->st_bt = p->st_cu = p->st_su = nullptr;
            p->st_sinks = p->st_alibi = nullptr;
            return UA_ERR_OUT_OF_MEMORY;
        }
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t qbytes = (size_t)total_q * d.num_q_heads * d.head_size * 2;
    cudaError_t e = cudaMemcpyAsync(p->st_q, q_host, qbytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->st_bt, block_table_host, (size_t)num_seqs * d.max_blocks_per_seq * 4,
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->st_cu, cu_seqlens_q_host, (size_t)(num_seqs + 1) * 4,
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->st_su, seqused_k_host, (size_t)num_seqs * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && sinks_host)
        e = cudaMemcpyAsync(p->st_sinks, sinks_host, (size_t)d.num_q_heads * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && alibi_host)
        e = cudaMemcpyAsync(p->st_alibi, alibi_host, (size_t)d.num_q_heads * 4, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) {
        note_cuda(e, "ua_forward_host upload");
        return UA_ERR_CUDA;
    }
    ua_status s = ua_forward(p, p->st_q, k_cache, v_cache, p->st_bt, p->st_cu, p->st_su, num_seqs,
                             total_q, max_seqlen_q, max_seqlen_k, flags,
                             sinks_host ? p->st_sinks : nullptr, alibi_host ? p->st_alibi : nullptr,
                             p->st_out, stream);
    if (s != UA_OK) return s;
    e = cudaMemcpyAsync(out_host, p->st_out, qbytes, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        note_cuda(e, "ua_forward_host download");
        return UA_ERR_CUDA;
    }
    return UA_OK;
}

ua_status ua_check_device_error(ua_problem* p, void* stream, int32_t* code) {
    if (!p || !code) return UA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t h = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpy(&h, p->d_err, sizeof h, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        note_cuda(e, "ua_check_device_error");
        return UA_ERR_CUDA;
    }
    *code = h;
    return h ? UA_ERR_DEVICE : UA_OK;
}

}  // extern "C"
