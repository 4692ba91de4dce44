// ua_decode_tc.cu -- decode and small-chunk attention on the tcgen05 tensor
// cores, with the keys on the MMA's M dimension.
//
// A decode step has only g * S_q <= 16 packed (position, head) rows per KV
// head, so the products are laid out transposed:
//
//     S^T [128 keys x 16 rows] = K_tile [128 x d]  *  Q^T [d x 16]
//     O^T [d x 16 rows]       += V_tile^T [d x 128] * P^T [128 x 16]
//
// Both are tcgen05.mma kind::f16 with M = 128, N = 16: K and V come straight
// from their paged TMA tiles (V read MN-major, no transpose copy), Q^T and P^T
// are 16-row K-major tiles in shared memory, S^T and O^T accumulate in tensor
// memory (64 columns).  Tensor-memory lane = key for S^T and lane = head-dim
// element for O^T, so each softmax thread owns one key of the tile; the
// per-row maxima are reduced across the 128 keys with warp shuffles plus one
// shared-memory exchange per tile.  The math is the same streaming (m, l, o)
// recurrence in base 2 with the lazy re-anchor (gfx1151 ALGORITHM.md section
// 3; gfx950 "Unified paged attention on gfx950, from the math up", section 2;
// attention_dense.py lazy_rescale), split into KV segments whose partials the
// combine kernel merges (gfx950 section 5).
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "ua_common.cuh"
#include "ua_decode_common.cuh"
#include "ua_decode_tc.h"
#include "ua_ptx.cuh"
#include "ua_tc.cuh"
#include "ua_tmap.h"

// One K and one V stage per CTA keeps the footprint at ~77 KB, so two CTAs
// share an SM and each one's waits hide behind the other's copies; measured
// on the 64-sequence decode batch this streams faster than one CTA with a
// three-deep ring (5.8 vs 4.8 TB/s).
#ifndef UA_DEC_NSK
#define UA_DEC_NSK 1
#endif
#ifndef UA_DEC_NSV
#define UA_DEC_NSV 1
#endif

namespace ua {
namespace {

constexpr int kN = 16;          // packed rows per tile (MMA N)
constexpr int kBN = 128;        // keys per KV tile (MMA M of S^T)
constexpr int kThreadsD = 224;  // 4 softmax warps, TMA warp, QK^T issuer, P.V issuer
constexpr int kThreadsF8 = 352; // fp8 caches: + 4 warps turning e4m3 tiles into f16
constexpr int kWarpTmaD = 4;
constexpr int kWarpMmaD = 5;    // QK^T issuer (also allocates tensor memory)
constexpr int kWarpPvD = 6;     // P.V issuer
constexpr float kLazyD = 8.0f;

// NSK / NSV: K and V ring depths (a K stage is free once its QK^T ran, a V
// stage only once its P.V ran, so they may differ).  F8: the rings hold e4m3
// tiles (128 keys x 128 one-byte dims); K is turned into f16 in tensor memory
// (the QK^T A operand), V into an f16 tile in shared memory.
// D: head size (64, 128 or 256; the fp8 cache D = 128 only).  O^T has M = D
// rows: one M = 128 MMA per 16 keys at D = 128, two (dims 0-127, 128-255 into
// two 16-column blocks of tensor memory) at D = 256, and at D = 64 one M = 128
// MMA whose descriptor reads the tile's single 64-dim panel for both halves
// of M (lanes 64-127 receive a copy of lanes 0-63 that nobody reads).
template <int D, int NSK, int NSV, bool F8>
struct DCfg {
    static_assert(D == 64 || D == 128 || D == 256, "head size");
    static_assert(!F8 || D == 128, "fp8 caches at d = 128 only");
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kN * 128;              // 16 rows x 64 dims
    static constexpr int kQBytes = kPanels * kQPanel;
    static constexpr int kKvPanel = kBN * 128;            // 128 keys x 64 dims (16-bit)
    static constexpr int kKvBytes = kPanels * kKvPanel;
    static constexpr int kStage = F8 ? kBN * 128 : kKvBytes;   // one TMA ring stage
    static constexpr int kPPanel = kN * 128;              // 16 rows x 64 keys
    static constexpr int kPBuf = (kBN / 64) * kPPanel;    // one P^T tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = F8 ? 4096 : (D == 64 ? 4096 : 8192);
    static constexpr int kOffV = kOffK + NSK * kStage;
    static constexpr int kOffV16 = kOffV + NSV * kStage;  // F8: the f16 V tile
    static constexpr int kOffP = kOffV16 + (F8 ? kKvBytes : 0);  // two P^T buffers
    static constexpr int kOffBar = kOffP + 2 * kPBuf;
    // q_full, k_full[NSK], v_full[NSV], k_empty[NSK], v_empty[NSV], s_full[2],
    // p_full[2], o_done[2], drain[2]; F8: kc_full, kc_empty, vc_full, vc_empty;
    // never (the testing hook's stall waits on it; nothing arrives)
    static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 8 + (F8 ? 4 : 0) + 1;
    static constexpr int kOffRed = kOffBar + kNumBars * 8;    // maxima [2][4][16] fp32
    static constexpr int kOffSum = kOffRed + 2 * 4 * kN * 4;  // row sums [4][16] fp32
    static constexpr int kOffMisc = kOffSum + 4 * kN * 4;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static constexpr int kTmemS = 0;    // S^T buffers: columns [0, 16) and [16, 32)
    static constexpr int kTmemO = 32;   // O^T: columns [32, 48) (D = 256: dims 128-255 in [48, 64))
    static constexpr int kTmemK = 64;   // F8: f16 K (lane = key, two dims per column)
    static constexpr uint32_t kTmemCols = F8 ? 128 : 64;
    static_assert(kQBytes <= kOffK, "Q tile");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// NR: packed rows the softmax threads track (4, 8 or 16 >= g * S_q); the MMAs
// always run N = 16 and ignore the padding columns.
// e4m3 codes -> f16 (exact): the four bytes of `w` become two f16x2 words
// (lower byte in the lower half).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// F8: K and V caches hold e4m3 codes (gfx950 page, section 7.3): the MMAs run
// in f16 (every e4m3 value is exact in f16, and so is a bf16 Q of moderate
// magnitude), k_scale is folded into tau and v_scale into the output scale.
template <int D, int NSK, int NSV, int NR, bool PLAIN, bool F8>
__global__ void __launch_bounds__(F8 ? kThreadsF8 : kThreadsD, F8 ? 2 : 1)   // two CTAs per SM
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = DCfg<D, NSK, NSV, F8>;
    constexpr int kThreads = F8 ? kThreadsF8 : kThreadsD;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.z;
    const int hkv = blockIdx.y;
    const int seg = blockIdx.x;
    const bool split = p.splits > 1;
    const int g = p.g;

    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, s, sq, sk, q0);
    if (st && hkv == 0 && seg == 0 && threadIdx.x == 0) atomicOr(p.err, (int)st);
    if (st & UA_DEVERR_CU_SEQLENS) return;
    const int nrows = min(g * sq, kN);   // the planner guarantees g * S_q <= 16
    if (nrows <= 0) return;
    if (seg >= (split ? seq_segments(p, st, sk) : 1)) return;
    const int ctx = sk - sq;
    const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
    const bool window = (p.flags & UA_FLAG_WINDOW) != 0;
    int k_end = causal ? min(sk, sq - 1 + ctx + 1) : sk;
    int k_beg = window ? max(0, ctx - p.window + 1) : 0;
    if (split) {
        k_beg = max(k_beg, seg * p.chunk);
        k_end = min(k_end, seg * p.chunk + p.chunk);
    }
    if (st || k_beg >= k_end) {
        // Malformed lengths (rows written as zeros) or a segment no row sees
        // (an empty partial, m = -inf).
        for (int e = threadIdx.x; e < nrows * D; e += kThreads) {
            const int r = e / D, c = e % D;
            const int64_t row = (q0 + r / g) * p.hq + hkv * g + r % g;
            if (split) {
                if (c == 0) {
                    p.part_ml[(row * p.splits + seg) * 2 + 0] = -INFINITY;
                    p.part_ml[(row * p.splits + seg) * 2 + 1] = 0.f;
                }
            } else {
                p.out[row * D + c] = __float2bfloat16_rn(0.f);
            }
        }
        return;
    }
    const int t_begin = k_beg / kBN;
    const int n_tiles = (k_end + kBN - 1) / kBN - t_begin;

    uint64_t* bm = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    const uint32_t q_full = smem_u32(&bm[0]);
    const uint32_t k_full0 = smem_u32(&bm[1]);
    const uint32_t v_full0 = smem_u32(&bm[1 + NSK]);
    const uint32_t k_empty0 = smem_u32(&bm[1 + NSK + NSV]);
    const uint32_t v_empty0 = smem_u32(&bm[1 + 2 * NSK + NSV]);
    const uint32_t s_full0 = smem_u32(&bm[1 + 2 * NSK + 2 * NSV]);
    const uint32_t p_full0 = s_full0 + 16;
    const uint32_t o_done0 = s_full0 + 32;
    const uint32_t drain = s_full0 + 48;
    // F8: the f16 K in tensor memory / the f16 V tile written (kc_full, vc_full)
    // and read by their MMA (kc_empty, vc_empty); single-buffered.
    const uint32_t kc_full = s_full0 + 64, kc_empty = s_full0 + 72;
    const uint32_t vc_full = s_full0 + 80, vc_empty = s_full0 + 88;
    const uint32_t never = s_full0 + (F8 ? 96 : 64);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    float* lsum = reinterpret_cast<float*>(smem + C::kOffSum);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        // A ring stage is released by its MMA (bf16) or by the 128 converting
        // threads (F8).
        for (int i = 0; i < NSK; ++i) {
            mbar_init(k_full0 + 8 * i, 1);
            mbar_init(k_empty0 + 8 * i, F8 ? 128 : 1);
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(v_full0 + 8 * i, 1);
            mbar_init(v_empty0 + 8 * i, F8 ? 128 : 1);
        }
        if (F8) {
            mbar_init(kc_full, 128);
            mbar_init(kc_empty, 1);
            mbar_init(vc_full, 128);
            mbar_init(vc_empty, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full0 + 8 * i, 1);
            mbar_init(p_full0 + 8 * i, 128);
            mbar_init(o_done0 + 8 * i, 1);
        }
        mbar_init(drain, 1);
        mbar_init(drain + 8, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMmaD) {
        tc::tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sK = smem_u32(smem + C::kOffK);
    const uint32_t sV = smem_u32(smem + C::kOffV);
    const uint32_t sP = smem_u32(smem + C::kOffP);

    if (warp == kWarpTmaD) {
        // ------------------------------ TMA producer ------------------------------
        // The whole warp issues: lane i owns paged block i of each KV tile (its
        // id load and its TMA boxes), so one tile's boxes go out in parallel
        // instead of one after another from a single thread.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            // g heads x floor(16 / g) positions per panel
            mbar_arrive_expect_tx(q_full, (uint32_t)(g * (kN / g)) * 128u * C::kPanels);
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_3d(sQ + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, (int)q0, q_full);
        }
        const int b = p.b;
        const int nblk_seq = (sk + b - 1) / b;
        const int32_t* bt = p.block_table + (int64_t)s * p.bt_stride;
        // Block ids are fetched one tile ahead so their load latency overlaps
        // the current tile's waits and copies.
        auto tile_id = [&](int j) -> int32_t {
            const int blk0 = (t_begin + j) * kBN / b;
            return lane < min(kBN / b, nblk_seq - blk0) ? __ldg(bt + blk0 + lane) : 0;
        };
        int issued = 0;
        int32_t id_next = n_tiles > 0 ? tile_id(0) : 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int sk_ = j % NSK, sv_ = j % NSV;
            const int key0 = (t_begin + j) * kBN;
            const int blk0 = key0 / b;
            const int nb = min(kBN / b, nblk_seq - blk0);
            constexpr int kBoxes = F8 ? 1 : C::kPanels;   // 128-byte panels per key row
            const uint32_t bytes = (uint32_t)nb * b * 128 * kBoxes;
            const int32_t id = id_next;
            if (j + 1 < n_tiles) id_next = tile_id(j + 1);
            if (lane < nb && (id < 0 || (int64_t)id >= p.num_blocks))
                atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
            if (j >= NSK && !__all_sync(0xffffffffu, dwait(k_empty0 + 8 * sk_, ((j / NSK) + 1) & 1,
                                                           abort_flag, p.err)))
                break;
            if (lane == 0) mbar_arrive_expect_tx(k_full0 + 8 * sk_, bytes);
            __syncwarp();
            if (lane < nb) {
#pragma unroll
                for (int pn = 0; pn < kBoxes; ++pn)
                    tma_load_4d(sK + sk_ * C::kStage + pn * C::kKvPanel + lane * b * 128, &tm_k,
                                pn * 64, hkv, 0, id, k_full0 + 8 * sk_);
            }
            if (j >= NSV && !__all_sync(0xffffffffu, dwait(v_empty0 + 8 * sv_, ((j / NSV) + 1) & 1,
                                                           abort_flag, p.err)))
                break;
            if (lane == 0) mbar_arrive_expect_tx(v_full0 + 8 * sv_, bytes);
            __syncwarp();
            if (lane < nb) {
#pragma unroll
                for (int pn = 0; pn < kBoxes; ++pn)
                    tma_load_4d(sV + sv_ * C::kStage + pn * C::kKvPanel + lane * b * 128, &tm_v,
                                pn * 64, hkv, 0, id, v_full0 + 8 * sv_);
            }
            issued = j + 1;
        }
        if (*abort_flag && lane == 0) {
            // Let every copy this warp issued land before the CTA ends.
            for (int j = max(0, issued - NSK); j < issued; ++j)
                mbar_wait_bounded(k_full0 + 8 * (j % NSK), (j / NSK) & 1);
            for (int j = max(0, issued - NSV); j < issued; ++j)
                mbar_wait_bounded(v_full0 + 8 * (j % NSV), (j / NSV) & 1);
        }
        __syncwarp();
    } else if (warp == kWarpMmaD || warp == kWarpPvD) {
        // ---------------------- MMA issuers (one thread each) ----------------------
        // Two warps, each blocking only on the barriers its own MMAs need, so
        // neither spins and neither holds the other back: warp 5 issues
        // S^T(j) = K(j) Q^T once K(j) has landed and the softmax has released
        // S^T buffer (j & 1) (P of tile j - 2 published); warp 6 issues
        // O^T += V(j)^T P^T(j) once P(j) and V(j) are ready.
        constexpr uint32_t idesc_qk = F8 ? tc::idesc_f16_f32(kBN, kN, false, false)
                                         : tc::idesc_bf16_f32(kBN, kN, false, false);
        constexpr uint32_t idesc_pv = F8 ? tc::idesc_f16_f32(128, kN, true, false)
                                         : tc::idesc_bf16_f32(128, kN, true, false);
        auto wwait = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, dwait(bar, par, abort_flag, p.err));
        };
        if (warp == kWarpMmaD) {
            bool ok = wwait(q_full, 0);
            if (F8 && ok) {
                // The MMAs run in f16: convert the bf16 Q tile in place (the
                // same swizzled positions; every word is two elements).
                uint32_t* qw = reinterpret_cast<uint32_t*>(smem + C::kOffQ);
                for (int e = lane; e < C::kQBytes / 4; e += 32) {
                    const uint32_t w = qw[e];
                    uint32_t h;
                    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(bf16_hi(w)), "f"(bf16_lo(w)));
                    qw[e] = h;
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j >= 2 && !wwait(p_full0 + 8 * (j & 1), ((j - 2) >> 1) & 1)) break;
                const int stg = j % NSK;
                if (p.stall && j == 0) {
                    // Testing hook: the first K wait waits on a barrier that
                    // nothing completes and gives up after stall_ns.
                    if (!__all_sync(0xffffffffu, dwait(never, 0, abort_flag, p.err, (uint64_t)p.stall_ns)))
                        break;
                }
                if constexpr (F8) {
                    if (!wwait(kc_full, j & 1)) break;
                } else {
                    if (!wwait(k_full0 + 8 * stg, (j / NSK) & 1)) break;
                }
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t kst = sK + stg * C::kStage;
                    const uint32_t dS = tmem + C::kTmemS + (j & 1) * kN;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const int pn = k >> 2, off = (k & 3) * 32;
                        const uint64_t bq = tc::smem_desc_sw128(sQ + pn * C::kQPanel + off, 16, 1024);
                        if constexpr (F8) {
                            // A = f16 K from tensor memory: 16 dims per MMA = 8 columns.
                            tc::mma_bf16_ts(dS, tmem + C::kTmemK + k * 8, bq, idesc_qk, k > 0 ? 1u : 0u);
                        } else {
                            const uint64_t a = tc::smem_desc_sw128(kst + pn * C::kKvPanel + off, 16, 1024);
                            tc::mma_bf16(dS, a, bq, idesc_qk, k > 0 ? 1u : 0u);
                        }
                    }
                    tc::commit(s_full0 + 8 * (j & 1));
                    tc::commit(F8 ? kc_empty : k_empty0 + 8 * stg);
                }
                __syncwarp();
            }
        } else {
            for (int j = 0; j < n_tiles; ++j) {
                const int stg = j % NSV;
                if (!wwait(p_full0 + 8 * (j & 1), (j >> 1) & 1)) break;
                if constexpr (F8) {
                    if (!wwait(vc_full, j & 1)) break;
                } else {
                    if (!wwait(v_full0 + 8 * stg, (j / NSV) & 1)) break;
                }
                tc::fence_after_sync();
                const int key0 = (t_begin + j) * kBN;
                const int nvalid = min(kBN, sk - key0);
                if (!F8 && nvalid < kBN) {
                    // Keys past S_k: their V rows become zeros so that whatever
                    // the slots hold cannot reach O (0 * NaN is NaN).
                    uint8_t* vgen = smem + C::kOffV + stg * C::kStage;
                    const int per_panel = (kBN - nvalid) * 8;
                    for (int e = lane; e < per_panel * C::kPanels; e += 32) {
                        const int pn = e / per_panel, rem = e % per_panel;
                        *reinterpret_cast<uint4*>(vgen + pn * C::kKvPanel + (nvalid + rem / 8) * 128 +
                                                  (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    const uint32_t vst = F8 ? smem_u32(smem + C::kOffV16) : sV + stg * C::kStage;
                    const uint32_t pbuf = sP + (j & 1) * C::kPBuf;
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint64_t bp =
                            tc::smem_desc_sw128(pbuf + (kk >> 2) * C::kPPanel + (kk & 3) * 32, 16, 1024);
                        // A = V^T, MN-major: the leading-dimension offset steps
                        // from dims 0-63 to 64-127 of the M = 128 block (0 at
                        // D = 64: both halves read the one panel).
                        constexpr uint32_t lbo = D == 64 ? 0u : (uint32_t)C::kKvPanel;
#pragma unroll
                        for (int h = 0; h < (D == 256 ? 2 : 1); ++h) {
                            const uint64_t a = tc::smem_desc_sw128(vst + h * 2 * C::kKvPanel + kk * 16 * 128,
                                                                   lbo, 1024);
                            tc::mma_bf16(tmem + C::kTmemO + h * kN, a, bp, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    tc::commit(o_done0 + 8 * (j & 1));
                    tc::commit(F8 ? vc_empty : v_empty0 + 8 * stg);
                }
                __syncwarp();
            }
        }
        if (*abort_flag) {
            // No MMA this thread issued may still run when tensor memory is freed.
            const uint32_t dr = drain + 8 * (warp - kWarpMmaD);
            if (lane == 0) tc::commit(dr);
            __syncwarp();
            mbar_wait_bounded(dr, 0);
        }
    } else if (F8 && warp >= 7) {
        // --------------------- e4m3 -> f16 converters (F8, warps 7-10) ---------------------
        // Thread (warp, lane) owns key row r of each tile, r = tensor-memory lane
        // 32 * (warp % 4) + lane: K row r goes to tensor memory (two dims per
        // column), V row r to the f16 V tile (the swizzled layout a TMA copy of
        // a bf16 tile would have), zeros for keys past S_k.
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t tk = tmem + ((uint32_t)(quarter * 32) << 16) + C::kTmemK;
        for (int j = 0; j < n_tiles; ++j) {
            const int sk_ = j % NSK, sv_ = j % NSV;
            if (!__all_sync(0xffffffffu, dwait(k_full0 + 8 * sk_, (j / NSK) & 1, abort_flag, p.err))) break;
            if (j > 0 && !__all_sync(0xffffffffu, dwait(kc_empty, (j - 1) & 1, abort_flag, p.err))) break;
            tc::fence_after_sync();
            {
                const uint8_t* row = smem + C::kOffK + sk_ * C::kStage + r * 128;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    uint32_t f[16];
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int c = qq * 2 + c2;   // 16-byte chunk = dims 16c .. 16c + 15
                        const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
                        e4m3x4_to_f16x2(w.x, f[c2 * 8 + 0], f[c2 * 8 + 1]);
                        e4m3x4_to_f16x2(w.y, f[c2 * 8 + 2], f[c2 * 8 + 3]);
                        e4m3x4_to_f16x2(w.z, f[c2 * 8 + 4], f[c2 * 8 + 5]);
                        e4m3x4_to_f16x2(w.w, f[c2 * 8 + 6], f[c2 * 8 + 7]);
                    }
                    tc::st16(tk + qq * 16, f);
                }
                tc::wait_st();
            }
            tc::fence_before_sync();
            mbar_arrive(kc_full);
            mbar_arrive(k_empty0 + 8 * sk_);
            if (!__all_sync(0xffffffffu, dwait(v_full0 + 8 * sv_, (j / NSV) & 1, abort_flag, p.err))) break;
            if (j > 0 && !__all_sync(0xffffffffu, dwait(vc_empty, (j - 1) & 1, abort_flag, p.err))) break;
            {
                const bool live_key = (t_begin + j) * kBN + r < sk;
                const uint8_t* row = smem + C::kOffV + sv_ * C::kStage + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                    if (live_key) {
                        const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
                        e4m3x4_to_f16x2(w.x, lo.x, lo.y);
                        e4m3x4_to_f16x2(w.y, lo.z, lo.w);
                        e4m3x4_to_f16x2(w.z, hi.x, hi.y);
                        e4m3x4_to_f16x2(w.w, hi.z, hi.w);
                    }
                    // dims 16c .. 16c + 15: panel c / 4, 16-byte chunks 2 (c % 4) and 2 (c % 4) + 1
                    uint8_t* dst = smem + C::kOffV16 + (c >> 2) * C::kKvPanel + r * 128;
                    const int cc = 2 * (c & 3);
                    *reinterpret_cast<uint4*>(dst + ((cc ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4*>(dst + (((cc + 1) ^ (r & 7)) << 4)) = hi;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(vc_full);
            mbar_arrive(v_empty0 + 8 * sv_);
        }
    } else {
        // --------------------------- softmax warps 0-3 ----------------------------
        // Thread t: key t of each KV tile (S^T lane t) and head-dim element t of
        // the output (O^T lane t).
        const int t = threadIdx.x;
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        const bool softcap = (p.flags & UA_FLAG_SOFTCAP) != 0;
        const bool alibi = (p.flags & UA_FLAG_ALIBI) != 0;
        const bool qq = (p.flags & UA_FLAG_QQ_BIAS) != 0;
        const float tau = F8 ? p.scale * p.k_scale : p.scale;   // F8: k_scale folded in
        const float sl2 = tau * kLog2e;
        float m[NR], l[NR];
        // Visible key range [lo, hi] of each packed row (constant per CTA);
        // padding rows get an empty range.
        int rlo[NR], rhi[NR];
        float rslope[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
            const int i = r / g;
            rhi[r] = r < nrows ? (causal ? min(i + ctx, sk - 1) : sk - 1) : -1;
            rlo[r] = window ? max(0, i + ctx - p.window + 1) : 0;
            rslope[r] = (!PLAIN && alibi && r < nrows) ? __ldg(p.alibi + hkv * g + r % g) : 0.f;
        }
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const bool got = __all_sync(0xffffffffu, dwait(s_full0 + 8 * (j & 1), (j >> 1) & 1,
                                                           abort_flag, p.err));
            const int key = (t_begin + j) * kBN + t;
            float x[NR];
            if (got) {
                tc::fence_after_sync();
                uint32_t sv[kN];
                ld16(tl + C::kTmemS + (j & 1) * kN, sv);
                tc::wait_ld();
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    float v;
                    if constexpr (PLAIN) {
                        v = __uint_as_float(sv[r]) * sl2;
                    } else {
                        float tt = __uint_as_float(sv[r]) * tau;
                        if (softcap) tt = p.softcap * tanh_from_exp2(tt / p.softcap);
                        if (alibi) tt += rslope[r] * (float)(key - ctx);
                        // Query section of row r (position r / g); keys past
                        // the row's last visible key read nothing.
                        if (qq && key >= ctx && key <= rhi[r])
                            tt += __ldg(p.qq_bias + (int64_t)(r / g) * p.qq_stride + (key - ctx));
                        v = tt * kLog2e;
                    }
                    x[r] = (key >= rlo[r] && key <= rhi[r]) ? v : -INFINITY;
                }
            } else {
#pragma unroll
                for (int r = 0; r < NR; ++r) x[r] = -INFINITY;
            }
            // Per-row maxima over this warp's 32 keys, then over the 4 warps.
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r < nrows) {
                    const float w = warp_max_f32(x[r]);
                    if (lane == 0) red[((j & 1) * 4 + warp) * kN + r] = w;
                }
            }
            if (!dbar_and(1, 128, got)) {
                ok = false;
                break;
            }
            float alpha[NR];
            bool any_re = false;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                alpha[r] = 1.f;
                if (r < nrows) {
                    const float* rr = red + (j & 1) * 4 * kN + r;
                    const float tmax = fmaxf(fmaxf(rr[0], rr[kN]), fmaxf(rr[2 * kN], rr[3 * kN]));
                    // Lazy re-anchor: only when the tile max exceeds m by > 8 (log2).
                    if (tmax > m[r] + kLazyD) {
                        alpha[r] = fast_exp2(m[r] - tmax);
                        m[r] = tmax;
                        any_re = true;
                    }
                }
            }
            // p = 2^(x - m) on the fp16x2 special-function path; per-thread
            // partial row sums stay fp32.
            uint32_t pb[NR / 2];
#pragma unroll
            for (int r = 0; r < NR; r += 2) {
                const float a0 = x[r] - (m[r] == -INFINITY ? 0.f : m[r]);
                const float a1 = x[r + 1] - (m[r + 1] == -INFINITY ? 0.f : m[r + 1]);
                uint32_t h, e;
                asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(a1), "f"(a0));
                asm("ex2.approx.f16x2 %0, %1;" : "=r"(e) : "r"(h));
                float p0, p1;
                asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\t"
                    "cvt.f32.f16 %1, hi;\n\t}"
                    : "=f"(p0), "=f"(p1)
                    : "r"(e));
                l[r] = l[r] * alpha[r] + p0;
                l[r + 1] = l[r + 1] * alpha[r + 1] + p1;
                pb[r / 2] = F8 ? e : pack_bf16x2(p0, p1);   // the P.V MMA's element type
            }
            // P^T buffer (j & 1) was read by the P.V of tile j - 2; rescaling O
            // needs the P.V of tile j - 1.
            bool go = true;
            if (j >= 2)
                go = __all_sync(0xffffffffu, dwait(o_done0 + 8 * (j & 1), ((j - 2) >> 1) & 1,
                                                   abort_flag, p.err));
            if (go && any_re && j > 0) {
                go = __all_sync(0xffffffffu, dwait(o_done0 + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1,
                                                   abort_flag, p.err));
                if (go) {
                    tc::fence_after_sync();
#pragma unroll
                    for (int h = 0; h < (D == 256 ? 2 : 1); ++h) {
                        uint32_t o[kN];
                        ld16(tl + C::kTmemO + h * kN, o);
                        tc::wait_ld();
#pragma unroll
                        for (int r = 0; r < NR; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
                        st16(tl + C::kTmemO + h * kN, o);
                    }
                    tc::wait_st();
                }
            }
            if (go) {
                // P^T row r, key t: K-major [16 rows][128 keys] in two 64-key
                // 128-byte-swizzled panels.
                uint8_t* pbase = smem + C::kOffP + (j & 1) * C::kPBuf + (t >> 6) * C::kPPanel;
                const int kin = t & 63;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r >= nrows) continue;  // padding columns of O^T are never read
                    const uint16_t v = (r & 1) ? (uint16_t)(pb[r / 2] >> 16) : (uint16_t)(pb[r / 2] & 0xffffu);
                    *reinterpret_cast<uint16_t*>(pbase + r * 128 + (((kin >> 3) ^ (r & 7)) << 4) +
                                                 (kin & 7) * 2) = v;
                }
                fence_proxy_async_smem();
                tc::fence_before_sync();
                mbar_arrive(p_full0 + 8 * (j & 1));
            }
        }
        // ------------------------------ epilogue ---------------------------------
        if (ok) {
            const bool done = __all_sync(0xffffffffu,
                                         dwait(o_done0 + 8 * ((n_tiles - 1) & 1),
                                               ((n_tiles - 1) >> 1) & 1, abort_flag, p.err));
            // Row sums over the 128 keys: warp shuffles, then the 4 warps.
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r < nrows) {
                    float w = l[r];
                    w += __shfl_xor_sync(0xffffffffu, w, 1);
                    w += __shfl_xor_sync(0xffffffffu, w, 2);
                    w += __shfl_xor_sync(0xffffffffu, w, 4);
                    w += __shfl_xor_sync(0xffffffffu, w, 8);
                    w += __shfl_xor_sync(0xffffffffu, w, 16);
                    if (lane == 0) lsum[warp * kN + r] = w;
                }
            }
            if (dbar_and(1, 128, done)) {
                tc::fence_after_sync();
                // Thread t: output dim t (and t + 128 at D = 256); at D = 64
                // threads 64-127 hold copies and store nothing.
                uint32_t o[kN], o2[kN];
                ld16(tl + C::kTmemO, o);
                if constexpr (D == 256) ld16(tl + C::kTmemO + kN, o2);
                tc::wait_ld();
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r >= nrows) continue;
                    const float L0 = lsum[r] + lsum[kN + r] + lsum[2 * kN + r] + lsum[3 * kN + r];
                    const int64_t row = (q0 + r / g) * p.hq + hkv * g + r % g;
                    const float ov = __uint_as_float(o[r]) * (F8 ? p.v_scale : 1.f);
                    const float ov2 = D == 256 ? __uint_as_float(o2[r]) : 0.f;
                    if (split) {
                        if (D != 64 || t < 64) part_store(p, (row * p.splits + seg) * D + t, ov);
                        if (D == 256) part_store(p, (row * p.splits + seg) * D + 128 + t, ov2);
                        if (t == 0) {
                            p.part_ml[(row * p.splits + seg) * 2 + 0] = m[r];
                            p.part_ml[(row * p.splits + seg) * 2 + 1] = L0;
                        }
                    } else {
                        float num = 1.f, L = L0;
                        bool zero = false;
                        if (p.flags & UA_FLAG_SINKS) {
                            const float s2 = __ldg(p.sinks + hkv * g + r % g) * kLog2e;
                            if (s2 == INFINITY) {
                                zero = true;
                            } else if (s2 > m[r]) {
                                const float a = (m[r] == -INFINITY) ? 0.f : fast_exp2(m[r] - s2);
                                num = a;
                                L = L * a + 1.0f;
                            } else if (s2 != -INFINITY) {
                                L += fast_exp2(s2 - m[r]);
                            }
                        }
                        const float inv = (!zero && L > 0.f) ? num * __frcp_rn(L) : 0.f;
                        if (D != 64 || t < 64) p.out[row * D + t] = __float2bfloat16_rn(ov * inv);
                        if (D == 256) p.out[row * D + 128 + t] = __float2bfloat16_rn(ov2 * inv);
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMmaD) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace

bool decode_tc_shape_ok(const FwdParams& p) {
    const bool d_ok = p.kv_fp8 ? p.d == 128 : (p.d == 64 || p.d == 128 || p.d == 256);
    return d_ok && p.g >= 1 && p.g <= kN && (int64_t)p.g * p.max_seqlen_q <= kN;
}

void plan_decode_tc(const FwdParams& p, int num_sms, size_t workspace_bytes, DecodePlan* plan) {
    *plan = DecodePlan();
    plan->kv_box_rows = p.b;
    // Segments of whole 128-key tiles, at least 8 tiles each, aiming at about
    // four waves of the two CTAs an SM holds (measured on the 64-sequence
    // decode batch: 3-4 segments per (sequence, KV head) beat 2 and 5+).
    const int64_t base = (int64_t)p.hk * p.num_seqs;
    const int64_t want = (8LL * num_sms + base - 1) / base;
    const int64_t by_len = std::max<int64_t>(1, p.max_seqlen_k / (8 * kBN));
    int splits = (int)std::min<int64_t>(std::min<int64_t>(want, by_len), 64);
    const size_t per_split = (size_t)p.total_q * p.hq * (p.d + 2) * sizeof(float);
    splits = (int)std::min<size_t>((size_t)splits, per_split ? workspace_bytes / per_split : 1);
    if (splits < 1) splits = 1;
    if (splits > 1) {
        const int per = (p.max_seqlen_k + splits - 1) / splits;
        plan->chunk = (per + kBN - 1) / kBN * kBN;
        splits = (p.max_seqlen_k + plan->chunk - 1) / plan->chunk;
    }
    plan->splits = splits;
    plan->launches = splits > 1 ? 2 : 1;
}

namespace {

template <int D, int NSK, int NSV, bool F8>
cudaError_t launch_decode_t(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                            const FwdParams& p, const DecodePlan& plan, cudaStream_t stream) {
    using C = DCfg<D, NSK, NSV, F8>;
    const bool plain = (p.flags & (UA_FLAG_SOFTCAP | UA_FLAG_ALIBI | UA_FLAG_QQ_BIAS)) == 0;
    const int rows = p.g * p.max_seqlen_q;
    auto kern = rows <= 4 ? (plain ? decode_tc_kernel<D, NSK, NSV, 4, true, F8>
                                   : decode_tc_kernel<D, NSK, NSV, 4, false, F8>)
              : rows <= 8 ? (plain ? decode_tc_kernel<D, NSK, NSV, 8, true, F8>
                                   : decode_tc_kernel<D, NSK, NSV, 8, false, F8>)
                          : (plain ? decode_tc_kernel<D, NSK, NSV, 16, true, F8>
                                   : decode_tc_kernel<D, NSK, NSV, 16, false, F8>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)plan.splits, (unsigned)p.hk, (unsigned)p.num_seqs);
    kern<<<grid, F8 ? kThreadsF8 : kThreadsD, C::kSmem, stream>>>(tq, tm_k, tm_v, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecodePlan& plan, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const FwdParams& p, cudaStream_t stream) {
    // Q map: [total_q, H_q, d]; box = 64 dims x g heads x floor(16/g) positions
    // (16 rows when g divides 16; the rows past g * S_q are padding).
    CUtensorMap tq;
    cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.hq, (cuuint64_t)p.total_q};
    cuuint64_t strides[2] = {2ull * p.d, 2ull * p.d * p.hq};
    cuuint32_t box[3] = {64, (cuuint32_t)p.g, (cuuint32_t)(kN / p.g)};
    if (!encode_bf16_sw128(&tq, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    constexpr int NSK = UA_DEC_NSK, NSV = UA_DEC_NSV;
    // fp8 tiles carry half the bytes, so each CTA needs twice the tiles in
    // flight to keep the same HBM rate: two staging stages per operand (the
    // e4m3 stages are half the size, so two CTAs still share an SM).
    if (p.kv_fp8) return launch_decode_t<128, 2, 2, true>(tq, tm_k, tm_v, p, plan, stream);
    switch (p.d) {
        // d = 64: 16 KB K/V tiles, three stages each and still two CTAs per
        // SM (measured on the 64-sequence batch at d = 64: 4.86 TB/s with
        // three stages, 4.73 with two, 4.59 with one and four CTAs per SM).
        case 64: return launch_decode_t<64, 3, 3, false>(tq, tm_k, tm_v, p, plan, stream);
        case 128: return launch_decode_t<128, NSK, NSV, false>(tq, tm_k, tm_v, p, plan, stream);
        // d = 256: 64 KB K/V tiles, one stage each (one CTA per SM).
        case 256: return launch_decode_t<256, 1, 1, false>(tq, tm_k, tm_v, p, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ua
