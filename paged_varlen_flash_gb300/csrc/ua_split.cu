// ua_split.cu -- split-KV paged attention on CUDA cores (decode and small row
// tiles), plus the log-sum-exp combine kernel.
//
// Work unit: one CTA per (row tile of ROWS packed (position, head) rows of one
// KV head, KV segment, sequence).  Packing the g query heads that share a KV
// head into one tile follows the GQA packing of gfx950 "Unified paged
// attention on gfx950, from the math up", section 4; splitting the keys into
// segments whose partial (m, l, o) are merged afterwards is the 3D split-KV
// path of section 5.  Inside a CTA, each of the four warps streams its own
// 16-key subtiles through a 3-stage TMA ring (one 4-D tensor-map box per
// paged block slice, 128-byte swizzled so that both the key-per-lane score
// reads and the dim-per-lane value reads are free of bank conflicts), keeps
// its own online-softmax state (gfx1151 ALGORITHM.md section 3, in base 2 as
// in gfx950 section 2, with the lazy re-anchor threshold of 8 from
// attention_dense.py), and the warps are merged with the same associative
// rule at the end of the CTA.
#include <cfloat>
#include <cstdint>

#include "ua_common.cuh"
#include "ua_ptx.cuh"
#include "ua_split.h"

namespace ua {
namespace {

constexpr int kWarps = 4;
constexpr int kSub = 16;    // keys per warp subtile
constexpr int kStages = 3;  // TMA ring depth per warp
constexpr float kLazyThreshold = 8.0f;

template <int D, int ROWS>
struct SplitLayout {
    static constexpr int kPanels = D / 64;               // 128-byte swizzle panels per key row
    static constexpr int kPanelBytes = kSub * 128;       // one panel of one subtile
    static constexpr int kKvBytes = kPanels * kPanelBytes;  // K (or V) of one subtile
    static constexpr int kStageBytes = 2 * kKvBytes;
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kRingBytes = kWarps * kWarpBytes;
    static constexpr int kQBytes = ROWS * D * 4;         // q rows, fp32
    static constexpr int kPBytes = kWarps * kSub * ROWS * 4;
    static constexpr int kBarBytes = kWarps * kStages * 8 + 8;   // + one barrier nothing completes
    static constexpr int kMergeBytes = kWarps * ROWS * (D + 2) * 4;
    static_assert(kMergeBytes <= kRingBytes, "merge area must fit in the ring");
    static constexpr int kQOff = kRingBytes;
    static constexpr int kPOff = kQOff + kQBytes;
    static constexpr int kBarOff = kPOff + kPBytes;
    static constexpr int kMetaOff = kBarOff + kBarBytes;
    static constexpr int kMetaBytes = ROWS * 3 * 4 + 8 + ROWS * 8;
    static constexpr int kSmem = kMetaOff + kMetaBytes + 1024;  // + alignment slack
};

__device__ __forceinline__ float dot8(const float* q, uint4 k) {
    float a = q[0] * bf16_lo(k.x);
    a = fmaf(q[1], bf16_hi(k.x), a);
    a = fmaf(q[2], bf16_lo(k.y), a);
    a = fmaf(q[3], bf16_hi(k.y), a);
    a = fmaf(q[4], bf16_lo(k.z), a);
    a = fmaf(q[5], bf16_hi(k.z), a);
    a = fmaf(q[6], bf16_lo(k.w), a);
    a = fmaf(q[7], bf16_hi(k.w), a);
    return a;
}

template <int D, int ROWS, bool SPLIT>
__global__ void __launch_bounds__(kWarps * 32)
split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
             const FwdParams p) {
    using L = SplitLayout<D, ROWS>;
    constexpr int DPL = D / 32;   // output dims per lane in the value pass
    constexpr int NCH = D / 16;   // 8-element chunks per lane in the score pass

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* q_s = reinterpret_cast<float*>(smem + L::kQOff);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.z;
    const int seg = blockIdx.y;
    const int hkv = blockIdx.x % p.hk;
    const int rt = blockIdx.x / p.hk;

    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, s, sq, sk, q0);
    if (st && rt == 0 && hkv == 0 && seg == 0 && threadIdx.x == 0) atomicOr(p.err, (int)st);
    if (st & UA_DEVERR_CU_SEQLENS) return;
    const int g = p.g;
    const int nrows = g * sq;
    const int r0 = rt * ROWS;
    if (r0 >= nrows) return;
    const int nseg = seq_segments(p, st, sk);
    if (seg >= nseg) return;
    const int ctx = sk - sq;
    const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
    const bool window = (p.flags & UA_FLAG_WINDOW) != 0;

    // Row metadata: packed row r -> (position i, head h, token) and its visible
    // key range [lo, hi]; kept in shared memory so large row tiles do not spill.
    int* row_hi = reinterpret_cast<int*>(smem + L::kMetaOff);
    int* row_lo = row_hi + ROWS;
    int* row_h = row_lo + ROWS;
    long long* row_tok = reinterpret_cast<long long*>(row_h + ROWS + (ROWS & 1));
    int max_hi = -1, min_lo = 0x7fffffff;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int rg = r0 + r;
        const int i = rg / g;
        int hi = causal ? min(i + ctx, sk - 1) : sk - 1;
        int lo = window ? max(0, i + ctx - p.window + 1) : 0;
        if (rg >= nrows || st) { hi = -1; lo = 0x7fffffff; }
        max_hi = max(max_hi, hi);
        min_lo = min(min_lo, lo);
        if (threadIdx.x == r) {
            row_hi[r] = hi;
            row_lo[r] = lo;
            row_h[r] = hkv * g + rg % g;
            row_tok[r] = q0 + i;
        }
    }
    int kb = seg * p.chunk;
    int ke = min(kb + p.chunk, sk);
    ke = min(ke, max_hi + 1);
    kb = max(kb, min_lo & ~(kSub - 1));
    const int t0 = kb / kSub;
    const int n_sub = (kb < ke) ? (ke + kSub - 1) / kSub - t0 : 0;

    // Q rows -> shared memory as fp32 (rows outside the tile are zero).
    for (int e = threadIdx.x; e < ROWS * (D / 8); e += kWarps * 32) {
        const int r = e / (D / 8), c = e % (D / 8);
        float* dst = q_s + r * D + c * 8;
        if (r0 + r < nrows && !st) {
            const int rg = r0 + r;
            const int64_t tok = q0 + rg / g;
            const int hh = hkv * g + rg % g;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                p.q + (tok * p.hq + hh) * (int64_t)D + c * 8));
            dst[0] = bf16_lo(v.x); dst[1] = bf16_hi(v.x);
            dst[2] = bf16_lo(v.y); dst[3] = bf16_hi(v.y);
            dst[4] = bf16_lo(v.z); dst[5] = bf16_hi(v.z);
            dst[6] = bf16_lo(v.w); dst[7] = bf16_hi(v.w);
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) dst[t] = 0.f;
        }
    }
    // The testing hook's stall waits on this barrier; nothing ever arrives.
    const uint32_t never = smem_u32(&bars[kWarps * kStages]);
    if (lane == 0) {
        for (int stg = 0; stg < kStages; ++stg) mbar_init(smem_u32(&bars[warp * kStages + stg]), 1);
        if (warp == 0) mbar_init(never, 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    __syncthreads();

    // This warp's subtiles: t0 + warp, t0 + warp + kWarps, ...
    const int my_n = (n_sub > warp) ? (n_sub - warp + kWarps - 1) / kWarps : 0;
    uint8_t* ring = smem + warp * L::kWarpBytes;
    const int32_t* bt_row = p.block_table + (int64_t)s * p.bt_stride;

    auto issue = [&](int it) {
        // Called by lane 0 only.
        const int stg = it % kStages;
        const int key0 = (t0 + warp + it * kWarps) * kSub;
        const int32_t blk = __ldg(bt_row + key0 / p.b);
        if (blk < 0 || (int64_t)blk >= p.num_blocks) atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
        const uint32_t bar = smem_u32(&bars[warp * kStages + stg]);
        const uint32_t kdst = smem_u32(ring + stg * L::kStageBytes);
        const uint32_t vdst = kdst + L::kKvBytes;
        mbar_arrive_expect_tx(bar, L::kStageBytes);
#pragma unroll
        for (int pn = 0; pn < L::kPanels; ++pn) {
            tma_load_4d(kdst + pn * L::kPanelBytes, &tm_k, pn * 64, hkv, key0 % p.b, blk, bar);
            tma_load_4d(vdst + pn * L::kPanelBytes, &tm_v, pn * 64, hkv, key0 % p.b, blk, bar);
        }
    };

    if (lane == 0) {
        for (int it = 0; it < my_n && it < kStages; ++it) issue(it);
    }
    __syncwarp();

    // Online-softmax state (m in log2 units; l per lane, summed at the end).
    float m_r[ROWS], l_r[ROWS], o_r[ROWS][DPL];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        m_r[r] = -INFINITY;
        l_r[r] = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) o_r[r][t] = 0.f;
    }

    const int kk = lane & 15;  // key within the subtile (score pass)
    const int hf = lane >> 4;  // which half of the head dim (score pass)
    float* p_s = reinterpret_cast<float*>(smem + L::kPOff) + warp * kSub * ROWS;
    const bool softcap = (p.flags & UA_FLAG_SOFTCAP) != 0;
    const bool alibi = (p.flags & UA_FLAG_ALIBI) != 0;
    const bool qq = (p.flags & UA_FLAG_QQ_BIAS) != 0;
    const float qk_scale_log2 = p.scale * kLog2e;
    bool timed_out = false;
    int fail_it = 0;

    // Value-pass lane geometry: dims [DPL*lane, DPL*lane + DPL).
    const int v_e = DPL * lane;
    const int v_panel = v_e / 64;
    const int v_chunk = (v_e % 64) / 8;
    const int v_byte = (v_e % 8) * 2;

    for (int it = 0; it < my_n; ++it) {
        const int stg = it % kStages;
        const uint32_t bar = smem_u32(&bars[warp * kStages + stg]);
        const bool ok = (p.stall && it == 0) ? mbar_wait_bounded(never, 0, (uint64_t)p.stall_ns)
                                             : mbar_wait_bounded(bar, (it / kStages) & 1);
        if (__any_sync(0xffffffffu, !ok)) {
            timed_out = true;
            fail_it = it;
            break;
        }
        const uint8_t* Ks = ring + stg * L::kStageBytes;
        const uint8_t* Vs = Ks + L::kKvBytes;
        const int key0 = (t0 + warp + it * kWarps) * kSub;
        const int j = key0 + kk;

        // ---- scores: lane (kk, hf) owns key kk over half of the head dim ----
        float acc[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) acc[r] = 0.f;
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
            const int c = hf * NCH + ((cc + hf) % NCH);
            const int pn = c >> 3, cp = c & 7;
            const uint4 kv = *reinterpret_cast<const uint4*>(
                Ks + pn * L::kPanelBytes + kk * 128 + ((cp ^ (kk & 7)) << 4));
#pragma unroll
            for (int r = 0; r < ROWS; ++r) acc[r] += dot8(q_s + r * D + c * 8, kv);
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], 16);
            float x2;
            if (softcap || alibi || qq) {
                float t = acc[r] * p.scale;
                if (softcap) t = p.softcap * tanh_from_exp2(t / p.softcap);
                if (alibi) t += __ldg(p.alibi + row_h[r]) * (float)(j - ctx);
                // Query section only; row_hi < S_k keeps j - ctx < S_q, and
                // padding rows (row_hi = -1) read nothing.
                if (qq && j >= ctx && j <= row_hi[r])
                    t += __ldg(p.qq_bias + (row_tok[r] - q0) * p.qq_stride + (j - ctx));
                x2 = t * kLog2e;
            } else {
                x2 = acc[r] * qk_scale_log2;
            }
            const bool vis = (j <= row_hi[r]) && (j >= row_lo[r]);
            x2 = vis ? x2 : -INFINITY;
            float tm = x2;
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
            tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
            if (tm > m_r[r] + kLazyThreshold) {  // re-anchor (also the first finite tile)
                const float alpha = fast_exp2(m_r[r] - tm);
                m_r[r] = tm;
                l_r[r] *= alpha;
#pragma unroll
                for (int t = 0; t < DPL; ++t) o_r[r][t] *= alpha;
            }
            const float pr = vis ? fast_exp2(x2 - m_r[r]) : 0.f;
            if (hf == 0) {
                l_r[r] += pr;
                p_s[kk * ROWS + r] = pr;
            }
        }
        __syncwarp();

        // ---- values: lane owns DPL dims; keys past S_k are never touched ----
        const int nk = min(kSub, sk - key0);
        for (int k2 = 0; k2 < nk; ++k2) {
            const uint8_t* vp = Vs + v_panel * L::kPanelBytes + k2 * 128 +
                                ((v_chunk ^ (k2 & 7)) << 4) + v_byte;
            float v[DPL];
            if constexpr (DPL == 2) {
                const uint32_t u = *reinterpret_cast<const uint32_t*>(vp);
                v[0] = bf16_lo(u); v[1] = bf16_hi(u);
            } else if constexpr (DPL == 4) {
                const uint2 u = *reinterpret_cast<const uint2*>(vp);
                v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
                v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
            } else {
                const uint4 u = *reinterpret_cast<const uint4*>(vp);
                v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
                v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
                v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
                v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const float pr = p_s[k2 * ROWS + r];
#pragma unroll
                for (int t = 0; t < DPL; ++t) o_r[r][t] = fmaf(pr, v[t], o_r[r][t]);
            }
        }
        __syncwarp();
        if (lane == 0 && it + kStages < my_n) {
            fence_proxy_async_smem();
            issue(it + kStages);
        }
        __syncwarp();
    }

    if (timed_out) {
        if (lane == 0) atomicOr(p.err, (int)UA_DEVERR_TIMEOUT);
        // Drain this warp's copies that may still be in flight (issued for
        // iterations fail_it .. fail_it + kStages - 1) before the shared memory
        // is reused or released; these waits are bounded as well.
        for (int x = fail_it; x < my_n && x < fail_it + kStages; ++x)
            mbar_wait_bounded(smem_u32(&bars[warp * kStages + (x % kStages)]), (x / kStages) & 1);
    }

    // ---- merge the warps' states (associative (m, l, o) rule) ----
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], off);
    }
    __syncthreads();  // every warp is done with its ring; reuse it as the merge area
    float* mo = reinterpret_cast<float*>(smem);                  // [kWarps][ROWS][D]
    float* mm = mo + kWarps * ROWS * D;                          // [kWarps][ROWS]
    float* ml = mm + kWarps * ROWS;                              // [kWarps][ROWS]
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
#pragma unroll
        for (int t = 0; t < DPL; ++t) mo[(warp * ROWS + r) * D + v_e + t] = o_r[r][t];
        if (lane == 0) {
            mm[warp * ROWS + r] = m_r[r];
            ml[warp * ROWS + r] = l_r[r];
        }
    }
    __syncthreads();

    const bool sinks = (p.flags & UA_FLAG_SINKS) != 0;
    for (int e = threadIdx.x; e < ROWS * D; e += kWarps * 32) {
        const int r = e / D, dd = e % D;
        if (r0 + r >= nrows) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * ROWS + r]);
        float O = 0.f, Lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = mm[w * ROWS + r];
                if (mw == -INFINITY) continue;
                const float a = fast_exp2(mw - M);
                O = fmaf(a, mo[(w * ROWS + r) * D + dd], O);
                Lsum = fmaf(a, ml[w * ROWS + r], Lsum);
            }
        }
        const int64_t row_id = row_tok[r] * p.hq + row_h[r];
        if constexpr (SPLIT) {
            part_store(p, (row_id * p.splits + seg) * D + dd, O);
            if (dd == 0) {
                p.part_ml[(row_id * p.splits + seg) * 2 + 0] = M;
                p.part_ml[(row_id * p.splits + seg) * 2 + 1] = Lsum;
            }
        } else {
            float res = 0.f;
            bool zero = false;
            if (sinks) {
                const float s2 = __ldg(p.sinks + row_h[r]) * kLog2e;
                if (s2 == INFINITY) {
                    zero = true;
                } else if (s2 > M) {
                    const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - s2);
                    O *= a;
                    Lsum = Lsum * a + 1.0f;
                } else if (s2 != -INFINITY) {
                    Lsum += fast_exp2(s2 - M);
                }
            }
            if (!zero && Lsum > 0.f) res = O * __frcp_rn(Lsum);
            p.out[row_id * D + dd] = __float2bfloat16_rn(res);
        }
    }
}

// One warp per output row: merge the row's segment partials (gfx950
// section 5: re-base every segment to the global max, sum the denominators),
// fold the sink column, apply one reciprocal, cast to bf16.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const FwdParams p) {
    constexpr int DPL = D / 32;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.total_q * p.hq) return;
    const int64_t token = row / p.hq;
    const int h = (int)(row % p.hq);
    // Owning sequence: last s with cu_seqlens_q[s] <= token.
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(p.cu_seqlens_q + mid) <= token) lo = mid; else hi = mid - 1;
    }
    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, lo, sq, sk, q0);
    if (st & UA_DEVERR_CU_SEQLENS) return;
    if (token < q0 || token >= q0 + sq) return;
    const int n = p.topk_len ? topk_segments(p, st, token) : seq_segments(p, st, sk);
    const float* ml = p.part_ml + row * p.splits * 2;
    float M = -INFINITY;
    for (int k = 0; k < n; ++k) M = fmaxf(M, ml[2 * k]);
    float o[DPL];
#pragma unroll
    for (int t = 0; t < DPL; ++t) o[t] = 0.f;
    float Lsum = 0.f;
    if (M != -INFINITY) {
        for (int k = 0; k < n; ++k) {
            const float mk = ml[2 * k];
            if (mk == -INFINITY) continue;  // empty segment: its o is never read
            const float a = fast_exp2(mk - M);
            Lsum = fmaf(a, ml[2 * k + 1], Lsum);
            const int64_t po = (row * p.splits + k) * D + lane * DPL;
#pragma unroll
            for (int t = 0; t < DPL; ++t) o[t] = fmaf(a, part_load(p, po + t), o[t]);
        }
    }
    bool zero = false;
    if (p.flags & UA_FLAG_SINKS) {
        const float s2 = __ldg(p.sinks + h) * kLog2e;
        if (s2 == INFINITY) {
            zero = true;
        } else if (s2 > M) {
            const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - s2);
#pragma unroll
            for (int t = 0; t < DPL; ++t) o[t] *= a;
            Lsum = Lsum * a + 1.0f;
        } else if (s2 != -INFINITY) {
            Lsum += fast_exp2(s2 - M);
        }
    }
    const float inv = (!zero && Lsum > 0.f) ? __frcp_rn(Lsum) : 0.f;
    __nv_bfloat16* dst = p.out + row * D + lane * DPL;
#pragma unroll
    for (int t = 0; t < DPL; ++t) dst[t] = __float2bfloat16_rn(o[t] * inv);
}

template <int D, int ROWS, bool SPLIT>
cudaError_t launch_split_t(const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                           cudaStream_t stream) {
    using L = SplitLayout<D, ROWS>;
    auto kern = split_kernel<D, ROWS, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.row_tiles * p.hk), (unsigned)p.splits, (unsigned)p.num_seqs);
    kern<<<grid, kWarps * 32, L::kSmem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

template <int D, bool SPLIT>
cudaError_t launch_rows(int rows, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                        cudaStream_t st) {
    switch (rows) {
        case 1: return launch_split_t<D, 1, SPLIT>(tk, tv, p, st);
        case 2: return launch_split_t<D, 2, SPLIT>(tk, tv, p, st);
        case 4: return launch_split_t<D, 4, SPLIT>(tk, tv, p, st);
        case 8: return launch_split_t<D, 8, SPLIT>(tk, tv, p, st);
        case 16: return launch_split_t<D, 16, SPLIT>(tk, tv, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int split_smem_bytes(int d, int rows) {
#define UA_CASE(DD, RR) if (d == DD && rows == RR) return SplitLayout<DD, RR>::kSmem;
    UA_CASE(64, 1) UA_CASE(64, 2) UA_CASE(64, 4) UA_CASE(64, 8) UA_CASE(64, 16)
    UA_CASE(128, 1) UA_CASE(128, 2) UA_CASE(128, 4) UA_CASE(128, 8) UA_CASE(128, 16)
    UA_CASE(256, 1) UA_CASE(256, 2) UA_CASE(256, 4) UA_CASE(256, 8) UA_CASE(256, 16)
#undef UA_CASE
    return -1;
}

cudaError_t launch_split(int rows, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t stream) {
    const bool split = p.splits > 1;
    switch (p.d) {
        case 64: return split ? launch_rows<64, true>(rows, tk, tv, p, stream)
                              : launch_rows<64, false>(rows, tk, tv, p, stream);
        case 128: return split ? launch_rows<128, true>(rows, tk, tv, p, stream)
                               : launch_rows<128, false>(rows, tk, tv, p, stream);
        case 256: return split ? launch_rows<256, true>(rows, tk, tv, p, stream)
                               : launch_rows<256, false>(rows, tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const FwdParams& p, cudaStream_t stream) {
    const int64_t rows = p.total_q * p.hq;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    if (blocks == 0) return cudaSuccess;
    switch (p.d) {
        case 64: combine_kernel<64><<<blocks, 256, 0, stream>>>(p); break;
        case 128: combine_kernel<128><<<blocks, 256, 0, stream>>>(p); break;
        case 256: combine_kernel<256><<<blocks, 256, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace ua
