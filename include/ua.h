/*
 * ua.h -- C ABI of the unified paged varlen attention forward library
 * (libua.so, sm_103a).
 *
 * One forward call serves decode (S_q = 1), prefill (S_q = S_k) and chunked
 * prefill (1 < S_q < S_k) over a block-table-mapped bf16 KV cache.  For each
 * packed query row i of sequence s and query head h it computes
 *
 *     O_i = sum_j softmax(x)_j V_j   over the visible keys j of s,
 *
 * with the score transform applied in this fixed order (gfx950 "Unified paged
 * attention on gfx950, from the math up", section 1 "What unified attention
 * computes", steps 1-7):
 *
 *     x_j  = tau * <Q_i, K_j>                            scale
 *     x_j  = c * tanh(x_j / c)            UA_FLAG_SOFTCAP
 *     x_j += slope_h * (j - ctx)          UA_FLAG_ALIBI
 *     x_j += B[i][j - ctx] for j >= ctx   UA_FLAG_QQ_BIAS (see ua_set_qq_bias)
 *     drop j > i + ctx                    UA_FLAG_CAUSAL
 *     drop j < i + ctx - W + 1            UA_FLAG_WINDOW (requires CAUSAL)
 *     sink_h joins the denominator        UA_FLAG_SINKS (no value row)
 *
 * where ctx = S_k - S_q (the query chunk is the last S_q of the sequence's S_k
 * keys, and its K/V are already in the cache), GQA maps query head h to KV head
 * floor(h / g) with g = H_q / H_k (section 0, notation; section 4 on packing the
 * g heads of one KV head into one tile), and a row with an empty denominator
 * gets O_i = 0 (gfx1151 ALGORITHM.md section 6).
 *
 * Layouts (all row-major, contiguous, device memory owned by the caller):
 *   q, out        bf16  [total_q, H_q, d]        packed ragged batch
 *   k_cache,
 *   v_cache       bf16  [num_blocks, b, H_k, d]  paged cache (section 0)
 *   block_table   int32 [num_seqs, max_blocks_per_seq]; key j of sequence s
 *                       lives in block block_table[s][j / b], slot j % b
 *   cu_seqlens_q  int32 [num_seqs + 1]; sequence s owns rows
 *                       cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1, cu_seqlens_q[0] = 0
 *   seqused_k     int32 [num_seqs]; S_k of each sequence
 *   sinks         fp32  [H_q] natural-log sink logits (UA_FLAG_SINKS only)
 *   alibi_slopes  fp32  [H_q] (UA_FLAG_ALIBI only)
 * Block-table entries past ceil(S_k / b) are never read.
 *
 * Every call is asynchronous on the given stream and never synchronises the
 * host.  Errors the host can see are returned as ua_status before anything is
 * launched; errors only the device can see (bad lengths or block ids inside
 * the metadata arrays) are recorded in a problem-owned device error word that
 * ua_check_device_error() reads -- the kernels never trap.
 */
#ifndef UA_H_
#define UA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ua_status {
    UA_OK = 0,
    UA_ERR_INVALID_ARG = 1,   /* a null or malformed argument; nothing launched */
    UA_ERR_UNSUPPORTED = 2,   /* valid, but outside what this build implements */
    UA_ERR_CUDA = 3,          /* a CUDA runtime call failed (see ua_last_cuda_error) */
    UA_ERR_OUT_OF_MEMORY = 4, /* device workspace allocation failed */
    UA_ERR_DEVICE = 5         /* the device error word was non-zero */
} ua_status;

/* Score-transform flags (section 1 of the spec above).  A problem is created
 * with the set it may use; each call passes a subset of it. */
enum {
    UA_FLAG_CAUSAL = 1u << 0,
    UA_FLAG_SOFTCAP = 1u << 1,
    UA_FLAG_ALIBI = 1u << 2,
    UA_FLAG_WINDOW = 1u << 3,
    UA_FLAG_SINKS = 1u << 4,
    UA_FLAG_QQ_BIAS = 1u << 5
};

/* Bits of the device error word. */
enum {
    UA_DEVERR_CONTEXT = 1u << 0,  /* seqused_k[s] < S_q(s): rows of s are written as 0 */
    UA_DEVERR_BLOCK_ID = 1u << 1, /* a block id outside [0, num_blocks): those keys read as 0 */
    UA_DEVERR_CU_SEQLENS = 1u << 2, /* cu_seqlens_q decreasing or past total_q: s skipped */
    UA_DEVERR_BOUNDS = 1u << 3,   /* S_q > max_seqlen_q or S_k > max_seqlen_k or
                                     S_k > max_blocks_per_seq * b: rows of s written as 0
                                     where addressable */
    UA_DEVERR_TIMEOUT = 1u << 4   /* a bounded on-chip wait gave up; results unspecified */
};

/* Element types.  Q, O: bf16.  K/V caches: bf16, or fp8 e4m3 codes (one byte
 * each; OCP e4m3: bias 7, subnormals, no infinities, 0x7f / 0xff NaN) with one
 * scale per tensor, K = code * k_scale, V = code * v_scale (gfx950 page,
 * section 7.3 "fp8 KV cache (bf16-Q + fp8-KV)").  The fp8 cache is read by
 * the DECODE_TC path only. */
enum { UA_DTYPE_BF16 = 0, UA_DTYPE_FP8_E4M3 = 1 };

/* Execution path (gfx950 spec section 6: a path whose query-tile grid fills
 * the device versus split-KV segments plus a reduction).
 *   SPLIT_KV     CUDA-core split-KV kernel + combine, any shape.
 *   TENSOR_CORE  tcgen05 kernels over tiles of 128 packed (position, head)
 *                rows (floor(128 / g) positions of the g heads of one KV
 *                head): two tiles per CTA at d = 64 and 128, two tiles per
 *                cluster of two CTAs at d = 256; KV-split + combine when the
 *                tile grid is small; needs g <= 128.
 *   DECODE_TC    tcgen05 kernel with the keys on the MMA M dimension for
 *                calls with at most 16 packed rows per KV head: needs
 *                g * max_seqlen_q <= 16 (d = 64, 128 or 256; an fp8 cache
 *                needs d = 128).
 *   AUTO         DECODE_TC when it applies, else TENSOR_CORE when it applies
 *                and a KV head has more than 16 packed rows, else SPLIT_KV.
 * A forced path that does not apply returns UA_ERR_UNSUPPORTED. */
enum { UA_PATH_AUTO = 0, UA_PATH_SPLIT_KV = 1, UA_PATH_TENSOR_CORE = 2, UA_PATH_DECODE_TC = 3 };

/* Storage of the per-segment o partials that a KV-split call writes and the
 * combine kernel reads (gfx950 spec section 5; storing them in bf16 halves
 * their bytes and stores, as the pages' sparse decode kernel does).  m and l
 * stay fp32 either way; bf16 rounds each partial o element once (relative
 * error <= 2^-9 of that element). */
enum { UA_PARTIALS_F32 = 0, UA_PARTIALS_BF16 = 1 };

/*
 * Static description of a problem family (UnifiedAttentionProblem in the
 * gfx950 spec: one flag per bias/mask term, section 1 last paragraph and
 * section 6).  Validated by ua_problem_create.
 */
typedef struct ua_problem_desc {
    int32_t num_q_heads;        /* H_q > 0 */
    int32_t num_kv_heads;       /* H_k > 0, H_q % H_k == 0 */
    int32_t head_size;          /* d in {64, 128, 256} */
    int32_t block_size;         /* b in {16, 32, 64} */
    int64_t num_blocks;         /* physical blocks in each cache, > 0 */
    int32_t max_num_seqs;       /* upper bound on num_seqs per call, > 0 */
    int32_t max_blocks_per_seq; /* row stride of block_table, > 0 */
    int64_t max_total_q;        /* upper bound on total_q per call, > 0 */
    int32_t dtype;              /* UA_DTYPE_BF16 */
    uint32_t flags;             /* UA_FLAG_* the calls may use */
    float scale;                /* tau > 0 (usually 1/sqrt(d)) */
    float softcap;              /* c > 0 when UA_FLAG_SOFTCAP, else ignored */
    int32_t window;             /* W >= 1 when UA_FLAG_WINDOW, else ignored */
    uint32_t path;              /* UA_PATH_*: which kernel family serves the calls */
    int32_t kv_dtype;           /* UA_DTYPE_BF16, or UA_DTYPE_FP8_E4M3 (needs d = 128 and
                                   path AUTO or DECODE_TC; a call whose shape the
                                   decode kernel does not take returns
                                   UA_ERR_UNSUPPORTED) */
    float k_scale;              /* fp8 caches: K = code * k_scale, > 0; else ignored */
    float v_scale;              /* fp8 caches: V = code * v_scale, > 0; else ignored */
    int32_t split_partials;     /* UA_PARTIALS_F32 (0, the default) or UA_PARTIALS_BF16 */
} ua_problem_desc;

typedef struct ua_problem ua_problem;

/*
 * Validate *desc and create a problem bound to the current CUDA device.  The
 * problem owns a device workspace (split-KV partials of fp32 (m, l, o), the
 * device error word) that is allocated here, once; ua_forward allocates
 * nothing.  Returns UA_ERR_INVALID_ARG for malformed fields (e.g. H_q % H_k !=
 * 0, WINDOW without CAUSAL), UA_ERR_UNSUPPORTED for d or b outside the sets
 * above or a non-bf16 dtype, UA_ERR_OUT_OF_MEMORY if the workspace cannot be
 * allocated.  *out is set only on UA_OK; free it with ua_destroy.
 */
ua_status ua_problem_create(const ua_problem_desc *desc, ua_problem **out);

/*
 * Forward pass, enqueued on `stream` (a cudaStream_t; NULL = legacy default
 * stream), without host synchronisation.
 *
 * num_seqs <= max_num_seqs and num_seqs <= 65535 (else UA_ERR_UNSUPPORTED);
 * total_q = cu_seqlens_q[num_seqs] <= max_total_q;
 * max_seqlen_q / max_seqlen_k are host-side upper bounds on S_q(s) / S_k(s)
 * used to size the launch (the device checks them and reports
 * UA_DEVERR_BOUNDS).  `flags` must be a subset of the problem's flags;
 * `sinks` / `alibi_slopes` must be non-null exactly when their flag is set.
 * All array pointers are device pointers with the layouts above, `out` must
 * not alias any input, and q / out / caches must be 16-byte aligned.  `out` is
 * fully written for every row of every well-formed sequence.
 *
 * Returns UA_ERR_INVALID_ARG (nothing launched) on a contract violation the
 * host can see, UA_ERR_CUDA if a launch fails.
 */
ua_status ua_forward(ua_problem *p, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, const int32_t *cu_seqlens_q,
                     const int32_t *seqused_k, int32_t num_seqs, int64_t total_q,
                     int32_t max_seqlen_q, int32_t max_seqlen_k, uint32_t flags,
                     const float *sinks, const float *alibi_slopes, void *out,
                     void *stream);

/*
 * ua_forward_topk -- sparse top-k decode ("[Triton/Gluon] [GFX950] Sparse
 * paged attention and Sparse MLA", its token-granular top-k gather): each
 * query token t attends to its own list of key positions instead of to all
 * S_k keys of its sequence,
 *
 *     O_(t,h) = sum_e softmax(x)_e V_(j_e),  j_e = topk_idx[t][e], e < topk_len[t],
 *
 * where x_e is the score chain above evaluated for key j_e (the masks, ALiBi
 * and QQ-bias use the listed position j_e).  Entries outside [0, S_k) are
 * padding (-1 by convention) and are not keys; an entry listed twice counts
 * twice.  Same arguments as ua_forward plus:
 *   topk_idx     int32 [total_q, topk_stride] device, the lists (row t = token t)
 *   topk_len     int32 [total_q] device, list lengths in [0, topk_stride];
 *                a length outside it sets UA_DEVERR_BOUNDS and writes the
 *                token's rows as 0
 *   topk_stride  > 0, entries per list row (at most 2^30)
 * A listed key in a block whose id is out of range is dropped and sets
 * UA_DEVERR_BLOCK_ID.  Needs d = 128, g <= 16, a bf16 cache, path AUTO
 * or DECODE_TC and num_blocks * b * H_k < 2^31 (else UA_ERR_UNSUPPORTED).
 * The lists are split into segments of 128-entry tiles per token (one CTA
 * each, merged by the combine kernel), counted from each token's own length.
 */
ua_status ua_forward_topk(ua_problem *p, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_table, const int32_t *cu_seqlens_q,
                          const int32_t *seqused_k, int32_t num_seqs, int64_t total_q,
                          int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t *topk_idx,
                          const int32_t *topk_len, int32_t topk_stride, uint32_t flags,
                          const float *sinks, const float *alibi_slopes, void *out,
                          void *stream);

/*
 * Same computation with the per-step inputs and the output in HOST memory:
 * q_host, block_table_host, cu_seqlens_q_host, seqused_k_host, sinks_host and
 * alibi_host are copied to problem-owned device staging buffers (allocated on
 * first use, sized by the problem's maxima), the forward runs on `stream`, the
 * result is copied into out_host, and the call returns after `stream` has
 * drained.  The caches stay device-resident (k_cache / v_cache are device
 * pointers).  Pinned host memory makes the copies asynchronous DMA.
 */
ua_status ua_forward_host(ua_problem *p, const void *q_host, const void *k_cache,
                          const void *v_cache, const int32_t *block_table_host,
                          const int32_t *cu_seqlens_q_host, const int32_t *seqused_k_host,
                          int32_t num_seqs, int64_t total_q, int32_t max_seqlen_q,
                          int32_t max_seqlen_k, uint32_t flags, const float *sinks_host,
                          const float *alibi_host, void *out_host, void *stream);

/*
 * Synchronise `stream`, return the device error word (UA_DEVERR_* bits) in
 * *code and clear it.  Returns UA_ERR_DEVICE when *code != 0, UA_OK otherwise.
 */
ua_status ua_check_device_error(ua_problem *p, void *stream, int32_t *code);

/*
 * Number of kernel launches the most recent ua_forward / ua_forward_host call
 * enqueued (for launch accounting in benchmarks).
 */
int32_t ua_last_launch_count(const ua_problem *p);

/* Human-readable name of the execution path the last forward call took. */
const char *ua_last_path(const ua_problem *p);

/*
 * Query-query bias (gfx950 page, section 1, step 4): with UA_FLAG_QQ_BIAS a
 * call adds B[i][j - ctx] to the score of query row i (the row's index inside
 * its sequence's query chunk, 0 <= i < S_q) and key j, for the keys of the
 * query section (ctx <= j < S_k), after softcap and ALiBi and before the
 * masks.  Keys of the context (j < ctx) get no bias.  B is one fp32 matrix in
 * natural-log units, shared by every sequence and every query head; its
 * element (a, c) is bias[a * row_stride + c].
 *
 * bias: device pointer, owned by the caller, read by every later call that
 *       passes UA_FLAG_QQ_BIAS until it is replaced; NULL clears it.
 * n:    rows and columns of B that may be read; a call with the flag needs
 *       max_seqlen_q <= n (else UA_ERR_INVALID_ARG, nothing launched).
 * row_stride: elements between rows, >= n.
 * The problem must have been created with UA_FLAG_QQ_BIAS in its flags.
 * Returns UA_ERR_INVALID_ARG for n < 1 or row_stride < n with a non-NULL bias.
 */
ua_status ua_set_qq_bias(ua_problem *p, const float *bias, int64_t n, int64_t row_stride);

/*
 * Profiling hook: when both events are non-null, every later forward call
 * records `ev_begin` on its stream immediately before launching its dominant
 * kernel (the attention kernel, not the split combine) and `ev_end`
 * immediately after it, so the caller can time that kernel alone with
 * cudaEventElapsedTime.  The events (cudaEvent_t) stay owned by the caller;
 * pass NULL, NULL to switch the hook off.
 */
ua_status ua_set_profile_events(ua_problem *p, void *ev_begin, void *ev_end);

/*
 * Testing hook for the bounded-wait abort path; not for production use.
 * Every on-chip wait of the kernels is bounded (about one second); when one
 * gives up, the kernel sets UA_DEVERR_TIMEOUT, raises a CTA-wide abort flag so
 * that every role leaves its loop, waits (bounded) for the copies and
 * tensor-core operations it issued, frees its tensor memory and returns.
 * While this hook is enabled, the split, decode tensor-core, two-tile and
 * CTA-pair prefill kernels of later forward calls make their first
 * consumer-side K/V data wait wait on a barrier that nothing completes,
 * bounded by limit_ns instead: the wait gives up, the call returns,
 * ua_check_device_error reports UA_DEVERR_TIMEOUT, and the outputs of that
 * call are unspecified.  (In the CTA-pair kernel only the MMA-issuing CTA
 * stalls; its partner's waits give up on their normal bound.)  The waits
 * that drain a CTA's own copies and MMAs keep their normal bound.
 * enable = 0 restores normal calls.  limit_ns must lie in [1e3, 1e9] when
 * enabling (else UA_ERR_INVALID_ARG).
 */
ua_status ua_debug_stall_data_waits(ua_problem *p, int32_t enable, int64_t limit_ns);

/*
 * ua_forward_noalloc -- the split-KV forward pass without any allocation.
 * (An addition of this library; the paper has no counterpart.)
 *
 * For callers that cannot call cudaMalloc: code that lives inside a memory
 * arena owning the whole device, code running inside stream capture where an
 * allocation would break the capture, plugins that are handed only the
 * tensors of the call, and latency paths that must not enter an allocator.
 * Such callers cannot use ua_problem_create, which allocates the workspace.
 *
 * It takes the problem description by value-pointer (no ua_problem) plus the
 * same inputs and output as ua_forward, and runs the same split kernel and
 * combine kernel.  Their fp32 partials live in a 16 MiB array that the
 * library declares statically in device memory: every GPU that loads
 * libua.so holds those 16 MiB until the process exits.  Calls whose partials
 * (total_q * H_q * (d + 2) * 4 bytes per segment) do not fit twice in that
 * array return UA_ERR_UNSUPPORTED and launch nothing, as do descriptions
 * with an fp8 cache (kv_dtype != UA_DTYPE_BF16) or with UA_FLAG_QQ_BIAS
 * (the bias matrix is bound to a ua_problem).
 *
 * device_error: optional caller-owned device int32 that receives the
 * UA_DEVERR_* bits (OR-ed in; the caller clears it).  When NULL the bits go to
 * a word inside the static array, cleared at the start of each call, and are
 * not reported.
 *
 * The first call in a CUDA context resolves the array's address in that
 * context (once per context; a caller that switches contexts on one device
 * gets each context's own address); make that first call before any stream
 * capture.  All calls on a device share the array and leave their partials in
 * it: calls whose kernels may overlap on the GPU race on it and must be
 * ordered by the caller.
 *
 * desc->path must be UA_PATH_AUTO or UA_PATH_SPLIT_KV (this entry point runs
 * the split kernel only; TENSOR_CORE or DECODE_TC return UA_ERR_UNSUPPORTED,
 * a value past UA_PATH_DECODE_TC UA_ERR_INVALID_ARG); desc->max_num_seqs and
 * desc->max_total_q are not used.  num_seqs above 65535 returns
 * UA_ERR_UNSUPPORTED.
 */
ua_status ua_forward_noalloc(const ua_problem_desc *desc, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *block_table,
                             const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                             int32_t num_seqs, int64_t total_q, int32_t max_seqlen_q,
                             int32_t max_seqlen_k, uint32_t flags, const float *sinks,
                             const float *alibi_slopes, void *out, int32_t *device_error,
                             void *stream);

/* Free the workspace and the problem.  NULL is a no-op. */
void ua_destroy(ua_problem *p);

/* Static string for a status code. */
const char *ua_status_string(ua_status s);

/* Text of the last CUDA error seen by this thread inside the library. */
const char *ua_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* UA_H_ */
