// ua_noalloc.cu -- ua_forward_noalloc: the split-KV forward pass for callers
// that cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is not an option -- inside
// a memory pool or arena that owns every byte of the device and forbids
// side allocations, inside a CUDA-graph or stream-capture region where an
// allocation would break the capture, in a plugin whose host framework hands
// it only the tensors of the call, or on a latency path where an allocator
// call (and its possible device synchronisation) is not acceptable.  Such a
// caller cannot create a ua_problem, because ua_problem_create allocates the
// split workspace and the error word.
//
// What it does instead: the fp32 split partials (m, l, o) and the device error
// word live in one file-scope __device__ array of fixed size, so the library
// itself owns that scratch from the moment it is loaded; every GPU that loads
// the library holds kScratchBytes of it until the process exits.  The caller
// passes only inputs and outputs.  The kernels are the same split kernel and
// combine kernel that ua_forward launches on its split path; only the
// partials' address differs.
//
// Rules that follow from a single shared array:
//  * The first call in a CUDA context resolves the array's device address in
//    that context with cudaGetSymbolAddress (once per context: the address
//    is cached under the context's process-unique id, so a caller that makes
//    another context current on the same device gets that context's own
//    address, never a stale one).  Make that first call before any stream
//    capture begins.
//  * Every call on a device uses the same array and leaves its contents
//    behind; the error word is cleared at the start of each call.  Calls whose
//    kernels overlap on the GPU (different streams, no ordering between them)
//    race on the array and corrupt each other's results: order them.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "ua_common.cuh"
#include "ua_split.h"
#include "ua_tmap.h"

namespace {

// Scratch capacity: 16 MiB of fp32 partials, plus the error word.
constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr int kMaxContexts = 64;
constexpr int kMaxSplitsNoAlloc = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes + 256];

// Driver entry points, reached through the runtime (no -lcuda link).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(ptr);
}

std::mutex g_setup_mutex;
struct ScratchEntry {
    unsigned long long ctx_id;
    void* addr;
};
ScratchEntry g_scratch_addr[kMaxContexts];
int g_num_scratch = 0;

// Id of the context current on this thread (0 and false if none or unknown).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch in the current context (the runtime makes the
// device's primary context current if no context is); resolved once per
// context.
cudaError_t scratch_address(void** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    if (have_id) {
        for (int i = 0; i < g_num_scratch; ++i)
            if (g_scratch_addr[i].ctx_id == id) {
                *out = g_scratch_addr[i].addr;
                return cudaSuccess;
            }
    }
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
    if (e != cudaSuccess) return e;
    // The runtime call above binds a context if none was current.
    if (!have_id) have_id = current_context_id(&id);
    if (have_id && g_num_scratch < kMaxContexts) g_scratch_addr[g_num_scratch++] = {id, ptr};
    *out = ptr;
    return cudaSuccess;
}

int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

}  // namespace

extern "C" ua_status ua_forward_noalloc(const ua_problem_desc* d, const void* q,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, const int32_t* cu_seqlens_q,
                                        const int32_t* seqused_k, int32_t num_seqs,
                                        int64_t total_q, int32_t max_seqlen_q,
                                        int32_t max_seqlen_k, uint32_t flags, const float* sinks,
                                        const float* alibi_slopes, void* out,
                                        int32_t* device_error, void* stream) {
    if (!d) return UA_ERR_INVALID_ARG;
    const uint32_t known = UA_FLAG_CAUSAL | UA_FLAG_SOFTCAP | UA_FLAG_ALIBI | UA_FLAG_WINDOW |
                           UA_FLAG_SINKS | UA_FLAG_QQ_BIAS;
    if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_q_heads % d->num_kv_heads != 0 ||
        d->num_blocks <= 0 || d->max_blocks_per_seq <= 0 || (d->flags & ~known) ||
        !(d->scale > 0.f) || !std::isfinite(d->scale))
        return UA_ERR_INVALID_ARG;
    if (d->path > UA_PATH_DECODE_TC) return UA_ERR_INVALID_ARG;
    // This entry point runs the split kernel only: a description that forces
    // another kernel family is refused rather than silently served by it.
    if (d->path != UA_PATH_AUTO && d->path != UA_PATH_SPLIT_KV) return UA_ERR_UNSUPPORTED;
    if (d->flags & UA_FLAG_QQ_BIAS) return UA_ERR_UNSUPPORTED;   // the bias is bound to a ua_problem
    if (d->split_partials != UA_PARTIALS_F32 && d->split_partials != UA_PARTIALS_BF16)
        return UA_ERR_INVALID_ARG;
    if ((d->flags & UA_FLAG_SOFTCAP) && !(d->softcap > 0.f && std::isfinite(d->softcap)))
        return UA_ERR_INVALID_ARG;
    if ((d->flags & UA_FLAG_WINDOW) && (d->window < 1 || !(d->flags & UA_FLAG_CAUSAL)))
        return UA_ERR_INVALID_ARG;
    if (d->dtype != UA_DTYPE_BF16 || d->kv_dtype != UA_DTYPE_BF16 || (d->head_size != 64 && d->head_size != 128 &&
                                      d->head_size != 256) ||
        (d->block_size != 16 && d->block_size != 32 && d->block_size != 64) ||
        d->num_blocks > (int64_t(1) << 31) - 1)
        return UA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        max_seqlen_q > max_seqlen_k ||
        (int64_t)max_seqlen_k > (int64_t)d->max_blocks_per_seq * d->block_size)
        return UA_ERR_INVALID_ARG;
    if ((flags & ~d->flags) || ((flags & UA_FLAG_WINDOW) && !(flags & UA_FLAG_CAUSAL)) ||
        (((flags & UA_FLAG_SINKS) != 0) != (sinks != nullptr)) ||
        (((flags & UA_FLAG_ALIBI) != 0) != (alibi_slopes != nullptr)))
        return UA_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0) return UA_OK;
    if (num_seqs > 65535) return UA_ERR_UNSUPPORTED;   // one grid row of CTAs per sequence
    if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seqused_k || !out)
        return UA_ERR_INVALID_ARG;
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(q) || misaligned(out) || misaligned(k_cache) || misaligned(v_cache))
        return UA_ERR_INVALID_ARG;
    // The scratch must hold at least two segments of fp32 partials per row.
    const size_t per_split = (size_t)total_q * d->num_q_heads * (d->head_size + 2) * sizeof(float);
    if (per_split > kScratchBytes / 2) return UA_ERR_UNSUPPORTED;
    if (max_seqlen_k == 0) {
        if (max_seqlen_q > 1) return UA_ERR_INVALID_ARG;
        max_seqlen_k = 1;
    }

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return UA_ERR_CUDA;
    int num_sms = 0;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return UA_ERR_CUDA;
    void* scratch = nullptr;
    e = scratch_address(&scratch);
    if (e != cudaSuccess) return UA_ERR_CUDA;

    CUtensorMap tk, tv;
    // 16-slot boxes with the 128-byte swizzle the split kernel reads.
    if (!ua::encode_cache_map(&tk, k_cache, d->head_size, d->num_kv_heads, d->block_size,
                              d->num_blocks, false, 16) ||
        !ua::encode_cache_map(&tv, v_cache, d->head_size, d->num_kv_heads, d->block_size,
                              d->num_blocks, false, 16))
        return UA_ERR_CUDA;

    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t* err = device_error ? device_error
                                : reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) +
                                                             kScratchBytes);
    if (!device_error) {
        e = cudaMemsetAsync(err, 0, sizeof(int32_t), st);
        if (e != cudaSuccess) return UA_ERR_CUDA;
    }

    // Launch shape: the planner rule of the split path (row tile of up to 16
    // packed rows, about four waves of CTAs), capped by the scratch capacity.
    const int g = d->num_q_heads / d->num_kv_heads;
    const int64_t rows_per_kv = (int64_t)g * max_seqlen_q;
    int rows = 1, row_tiles = 1;
    if (rows_per_kv <= 16) {
        while (rows < rows_per_kv) rows <<= 1;
    } else {
        rows = 16;
        row_tiles = cdiv(rows_per_kv, 16);
    }
    const int smem = ua::split_smem_bytes(d->head_size, rows);
    const int cps = std::max(1, std::min(8, (228 * 1024) / (smem + 1024)));
    const int64_t base = (int64_t)num_seqs * d->num_kv_heads * row_tiles;
    const int64_t slots = (int64_t)num_sms * cps;
    int splits = (int)std::min<int64_t>(kMaxSplitsNoAlloc,
                                        std::max<int64_t>(1, (4 * slots + base - 1) / base));
    splits = std::min(splits, std::max(1, cdiv(max_seqlen_k, 256)));
    splits = (int)std::min<size_t>((size_t)splits, kScratchBytes / per_split);
    if (splits < 1) splits = 1;
    const int chunk = cdiv(cdiv(max_seqlen_k, splits), 64) * 64;
    splits = cdiv(max_seqlen_k, chunk);
    if (row_tiles * (int64_t)d->num_kv_heads > 0x7fffffffLL || splits > 65535)
        return UA_ERR_UNSUPPORTED;

    ua::FwdParams fp;
    std::memset(&fp, 0, sizeof fp);
    fp.part_bf16 = d->split_partials == UA_PARTIALS_BF16 ? 1 : 0;
    fp.q = static_cast<const __nv_bfloat16*>(q);
    fp.block_table = block_table;
    fp.cu_seqlens_q = cu_seqlens_q;
    fp.seqused_k = seqused_k;
    fp.sinks = sinks;
    fp.alibi = alibi_slopes;
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.part_o = static_cast<float*>(scratch);
    fp.part_ml = fp.part_o + (size_t)total_q * d->num_q_heads * splits * d->head_size;
    fp.err = err;
    fp.total_q = total_q;
    fp.num_blocks = d->num_blocks;
    fp.num_seqs = num_seqs;
    fp.bt_stride = d->max_blocks_per_seq;
    fp.max_seqlen_q = max_seqlen_q;
    fp.max_seqlen_k = max_seqlen_k;
    fp.hq = d->num_q_heads;
    fp.hk = d->num_kv_heads;
    fp.g = g;
    fp.d = d->head_size;
    fp.b = d->block_size;
    fp.flags = flags;
    fp.scale = d->scale;
    fp.softcap = d->softcap;
    fp.window = d->window;
    fp.splits = splits;
    fp.chunk = chunk;
    fp.row_tiles = row_tiles;

    e = ua::launch_split(rows, tk, tv, fp, st);
    if (e == cudaSuccess && splits > 1) e = ua::launch_combine(fp, st);
    return e == cudaSuccess ? UA_OK : UA_ERR_CUDA;
}
