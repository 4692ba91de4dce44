// ua_prefill.cu -- prefill / chunked-prefill attention for head size 256 on
// the tcgen05 tensor cores of sm_103a (head sizes 64 and 128 use the two-tile
// kernel of ua_prefill_pair.cu), plus the prefill planner and launcher.
//
// Work unit: one CTA per (tile of 128 packed (position, head) rows of one KV
// head, sequence[, KV segment]).  The g query heads that share a KV head are
// packed into the tile's rows, so one QK^T MMA serves the whole group (gfx950
// "Unified paged attention on gfx950, from the math up", section 4, GQA
// packing).  The CTA walks its visible KV tiles with the streaming (m, l, o)
// recurrence of gfx1151 ALGORITHM.md section 3, in base 2 (gfx950 section 2),
// with the lazy re-anchor threshold of 8, mask-free interior tiles and the
// causal early exit and sliding-window start tile of attention_dense.py
// (section 8.1 of the gfx950 page).  Key tiles are visited from the diagonal
// backwards (the result does not depend on the order).
//
// Roles (11 warps):
//   warps 0-7  softmax + epilogue: two warpgroups share each row's BN key
//              columns (one shared-memory max exchange per tile); thread
//              (part, r) owns row r, which is tensor-memory lane r;
//   warp 8     TMA producer: Q tile once (a 3-D box of g heads x 128/g
//              positions), then K and V tiles through NK- and NV-stage rings,
//              one box per (paged block, 64-wide head-dim panel), block ids
//              read from the block table one tile ahead;
//   warp 9     tensor-memory allocator and QK^T issuer;
//   warp 10    P.V issuer (P bf16 from tensor memory, V MN-major straight
//              from its TMA tile).
//
// Tensor memory (512 columns): S0 [0, BN), S1 [BN, 2 BN), O [2 BN, 2 BN + D),
// three bf16 P buffers after O (the softmax writing P(j) waits only for the
// P.V of tile j - 3).
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "ua_common.cuh"
#include "ua_prefill.h"
#include "ua_prefill_common.cuh"
#include "ua_ptx.cuh"
#include "ua_tc.cuh"
#include "ua_tmap.h"

namespace ua {
namespace {

using namespace pf;

template <int D, int BN, int NK, int NV, int SPLIT>
struct PCfg {
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kRows * 128;
    static constexpr int kQBytes = kPanels * kQPanel;
    static constexpr int kKvPanel = BN * 128;
    static constexpr int kKvBytes = kPanels * kKvPanel;
    static constexpr int kPBytes = 0;   // P lives in tensor memory
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + NK * kKvBytes;
    static constexpr int kOffP = kOffV + NV * kKvBytes;
    static constexpr int kOffBar = kOffP + kPBytes;
    // q_full, k_full[NK], v_full[NV], k_empty[NK], v_empty[NV], s_full[2],
    // p_full[3], o_done[3] (per P buffer), drain[2]
    static constexpr int kNumBars = 1 + 2 * NK + 2 * NV + 2 + 3 + 3 + 2;
    static constexpr int kOffRed = kOffBar + kNumBars * 8;      // [2 parity][SPLIT][128] fp32
    static constexpr int kOffMisc = kOffRed + 2 * SPLIT * kRows * 4;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static constexpr int kTmemS = 0;
    static constexpr int kTmemO = 2 * BN;
    static constexpr int kTmemP = 2 * BN + D;   // three bf16 P buffers of BN / 2 columns
    static_assert(2 * BN + D + 3 * (BN / 2) <= (int)kTmemCols, "tensor memory budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// QQ: the query-query bias pass is compiled in (a separate instantiation, so
// that the score loop of the other non-plain calls keeps its registers).
template <int D, int BN, int NK, int NV, int SPLIT, bool PLAIN, bool QQ>
__global__ void __launch_bounds__(Roles<SPLIT>::kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = PCfg<D, BN, NK, NV, SPLIT>;
    using R = Roles<SPLIT>;
    constexpr int kThreads = R::kThreads;
    constexpr int kSmThreads = R::kSmThreads;
    constexpr int kWarpTma = R::kWarpTma;
    constexpr int kWarpMma = R::kWarpMma;
    constexpr int kWarpPv = R::kWarpPv;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.z;
    const int hkv = blockIdx.y;
    const bool split = p.splits > 1;             // write (m, l, o) partials per KV segment
    const int seg = blockIdx.x % p.splits;
    const int qt = (int)(gridDim.x / p.splits) - 1 - (int)(blockIdx.x / p.splits);  // heaviest first
    const int g = p.g;
    const int ppt = kRows / g;                  // positions per tile
    const int p0 = qt * ppt;

    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, s, sq, sk, q0);
    if (st && qt == 0 && hkv == 0 && seg == 0 && threadIdx.x == 0) atomicOr(p.err, (int)st);
    if (st & UA_DEVERR_CU_SEQLENS) return;
    if (p0 >= sq) return;
    if (seg >= (split ? seq_segments(p, st, sk) : 1)) return;
    const int p_last = min(p0 + ppt, sq) - 1;
    const int ctx = sk - sq;
    const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
    const bool window = (p.flags & UA_FLAG_WINDOW) != 0;
    int k_end = causal ? min(sk, p_last + ctx + 1) : sk;
    int k_beg = window ? max(0, p0 + ctx - p.window + 1) : 0;
    if (split) {  // this CTA's KV segment; segments are whole BN tiles
        k_beg = max(k_beg, seg * p.chunk);
        k_end = min(k_end, seg * p.chunk + p.chunk);
    }
    if (st || k_beg >= k_end) {
        // Malformed lengths (rows written as zeros) or a segment with no
        // visible key for any row of the tile (an empty partial, m = -inf).
        for (int e = threadIdx.x; e < kRows * (D / 8); e += kThreads) {
            const int r = e / (D / 8), c = e % (D / 8);
            const int i = p0 + r / g;
            if (i > p_last) continue;
            const int64_t row = (q0 + i) * p.hq + hkv * g + r % g;
            if (split) {
                if (c == 0) {
                    p.part_ml[(row * p.splits + seg) * 2 + 0] = -INFINITY;
                    p.part_ml[(row * p.splits + seg) * 2 + 1] = 0.f;
                }
            } else {
                *reinterpret_cast<uint4*>(p.out + row * D + c * 8) = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int t_begin = k_beg / BN;
    const int n_tiles = (k_end + BN - 1) / BN - t_begin;
    // Step j visits key tile t_last - j: from the diagonal backwards.  The
    // result does not depend on the order; with causal ALiBi the scores grow
    // toward the diagonal, so this order meets each row's largest scores
    // first and the running max (and O) rarely needs re-anchoring.
    const int t_last = t_begin + n_tiles - 1;

    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    Bars B;
    B.q_full = smem_u32(&bar_mem[0]);
    B.k_full0 = smem_u32(&bar_mem[1]);
    B.v_full0 = smem_u32(&bar_mem[1 + NK]);
    // A K stage is free once its QK^T has run, a V stage once its P.V has run,
    // so the next K tile can be requested a whole softmax earlier than V.
    B.k_empty0 = smem_u32(&bar_mem[1 + NK + NV]);
    B.v_empty0 = smem_u32(&bar_mem[1 + 2 * NK + NV]);
    constexpr int kBarS = 1 + 2 * NK + 2 * NV;
    B.s_full0 = smem_u32(&bar_mem[kBarS]);
    // Per-parity barriers: softmax warps may run one tile ahead of the MMA
    // warp, so P-ready and PV-done are tracked separately for even and odd
    // tiles (a single barrier could see arrivals of two tiles in one phase).
    B.p_full = smem_u32(&bar_mem[kBarS + 2]);   // P buffer j % 3 written
    B.o_done = smem_u32(&bar_mem[kBarS + 5]);   // the P.V reading buffer j % 3 done
    B.drain = smem_u32(&bar_mem[kBarS + 8]);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    if (threadIdx.x == 0) {
        mbar_init(B.q_full, 1);
        for (int i = 0; i < NK; ++i) {
            mbar_init(B.k_full0 + 8 * i, 1);
            mbar_init(B.k_empty0 + 8 * i, 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(B.v_full0 + 8 * i, 1);
            mbar_init(B.v_empty0 + 8 * i, 1);
        }
        mbar_init(B.s_full0, 1);
        mbar_init(B.s_full0 + 8, 1);
        for (int x = 0; x < 3; ++x) {
            mbar_init(B.p_full + 8 * x, kSmThreads);
            mbar_init(B.o_done + 8 * x, 1);
        }
        mbar_init(B.drain, 1);
        mbar_init(B.drain + 8, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sK = smem_u32(smem + C::kOffK);
    const uint32_t sV = smem_u32(smem + C::kOffV);

    if (warp == kWarpTma) {
        // ------------------------------ TMA producer ------------------------------
        // The whole warp issues: lane i owns paged block i of each KV tile (its
        // id load and its TMA boxes), so one tile's boxes go out in parallel
        // instead of one after another from a single thread.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            // g heads x ppt positions per panel (rows past g * ppt are padding)
            mbar_arrive_expect_tx(B.q_full, (uint32_t)(g * ppt) * 128u * C::kPanels);
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_3d(sQ + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, (int)(q0 + p0), B.q_full);
        }
        const int b = p.b;
        const int nblk_seq = (sk + b - 1) / b;
        const int32_t* bt = p.block_table + (int64_t)s * p.bt_stride;
        // Block ids are fetched one tile ahead so their load latency overlaps
        // the current tile's waits and copies.
        auto tile_id = [&](int j) -> int32_t {
            const int blk0 = (t_last - j) * BN / b;
            return lane < min(BN / b, nblk_seq - blk0) ? __ldg(bt + blk0 + lane) : 0;
        };
        int issued = 0;
        int32_t id_next = n_tiles > 0 ? tile_id(0) : 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int stk = j % NK, stv = j % NV;
            const int key0 = (t_last - j) * BN;
            const int blk0 = key0 / b;
            const int nb = min(BN / b, nblk_seq - blk0);
            const uint32_t bytes = (uint32_t)nb * b * 128 * C::kPanels;
            const int32_t id = id_next;
            if (j + 1 < n_tiles) id_next = tile_id(j + 1);
            if (lane < nb && (id < 0 || (int64_t)id >= p.num_blocks))
                atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
            if (j >= NK && !__all_sync(0xffffffffu, wait_or_abort(B.k_empty0 + 8 * stk, ((j / NK) + 1) & 1,
                                                                   abort_flag, p.err)))
                break;
            if (lane == 0) mbar_arrive_expect_tx(B.k_full0 + 8 * stk, bytes);
            __syncwarp();
            if (lane < nb) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_4d(sK + stk * C::kKvBytes + pn * C::kKvPanel + lane * b * 128, &tm_k,
                                pn * 64, hkv, 0, id, B.k_full0 + 8 * stk);
            }
            if (j >= NV && !__all_sync(0xffffffffu, wait_or_abort(B.v_empty0 + 8 * stv, ((j / NV) + 1) & 1,
                                                                   abort_flag, p.err)))
                break;
            if (lane == 0) mbar_arrive_expect_tx(B.v_full0 + 8 * stv, bytes);
            __syncwarp();
            if (lane < nb) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_4d(sV + stv * C::kKvBytes + pn * C::kKvPanel + lane * b * 128, &tm_v,
                                pn * 64, hkv, 0, id, B.v_full0 + 8 * stv);
            }
            issued = j + 1;
        }
        if (*abort_flag && lane == 0) {
            // Let every copy this warp issued land before the CTA ends.
            for (int j = max(0, issued - NK); j < issued; ++j)
                mbar_wait_bounded(B.k_full0 + 8 * (j % NK), (j / NK) & 1);
            for (int j = max(0, issued - NV); j < issued; ++j)
                mbar_wait_bounded(B.v_full0 + 8 * (j % NV), (j / NV) & 1);
        }
        __syncwarp();
    } else if (warp == kWarpMma || warp == kWarpPv) {
        // ---------------------- MMA issuers (one thread each) ----------------------
        // Two warps, each blocking only on the barriers its own MMAs need, so
        // neither spins and neither holds the other back: one issues
        // S(j) = Q K(j)^T once K(j) has landed and the softmax has released S
        // buffer (j & 1) (P of tile j - 2 published); the other issues
        // O += P(j) V(j) once P(j) and V(j) are ready.
        constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, BN, false, false);
        constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kRows, D, false, true);
        auto wwait = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_or_abort(bar, par, abort_flag, p.err));
        };
        if (warp == kWarpMma) {
            bool ok = wwait(B.q_full, 0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j >= 2 && !wwait(B.p_full + 8 * ((j - 2) % 3), ((j - 2) / 3) & 1)) break;
                const int stg = j % NK;
                if (!wwait(B.k_full0 + 8 * stg, (j / NK) & 1)) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t kst = sK + stg * C::kKvBytes;
                    const uint32_t dS = tmem + C::kTmemS + (j & 1) * BN;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const int pn = k >> 2, off = (k & 3) * 32;
                        const uint64_t a = tc::smem_desc_sw128(sQ + pn * C::kQPanel + off, 16, 1024);
                        const uint64_t bdesc = tc::smem_desc_sw128(kst + pn * C::kKvPanel + off, 16, 1024);
                        tc::mma_bf16(dS, a, bdesc, idesc_qk, k > 0 ? 1u : 0u);
                    }
                    tc::commit(B.s_full0 + 8 * (j & 1));
                    tc::commit(B.k_empty0 + 8 * stg);
                }
                __syncwarp();
            }
        } else {
            for (int j = 0; j < n_tiles; ++j) {
                const int stg = j % NV;
                if (!wwait(B.p_full + 8 * (j % 3), (j / 3) & 1)) break;
                if (!wwait(B.v_full0 + 8 * stg, (j / NV) & 1)) break;
                tc::fence_after_sync();
                const uint32_t vst = sV + stg * C::kKvBytes;
                const int key0 = (t_last - j) * BN;
                const int nvalid = min(BN, sk - key0);
                if (nvalid < BN) {
                    // Keys past S_k: whatever those slots hold must not reach O
                    // (0 * NaN is NaN), so their V rows become zeros.
                    uint8_t* vgen = smem + C::kOffV + stg * C::kKvBytes;
                    const int per_panel = (BN - nvalid) * 8;
                    for (int e = lane; e < per_panel * C::kPanels; e += 32) {
                        const int pn = e / per_panel, rem = e % per_panel;
                        *reinterpret_cast<uint4*>(vgen + pn * C::kKvPanel + (nvalid + rem / 8) * 128 +
                                                  (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    const uint32_t dO = tmem + C::kTmemO;
                    const uint32_t aP = tmem + C::kTmemP + (j % 3) * (BN / 2);
#pragma unroll
                    for (int k = 0; k < BN / 16; ++k) {
                        // A = P from tensor memory: 16 keys per MMA = 8 columns.
                        const uint64_t bdesc = tc::smem_desc_sw128(vst + k * 16 * 128, C::kKvPanel, 1024);
                        tc::mma_bf16_ts(dO, aP + k * 8, bdesc, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
                    }
                    tc::commit(B.o_done + 8 * (j % 3));
                    tc::commit(B.v_empty0 + 8 * stg);
                }
                __syncwarp();
            }
        }
        if (*abort_flag) {
            // No MMA this thread issued may still run when tensor memory is freed.
            const uint32_t dr = B.drain + 8 * (warp - kWarpMma);
            if (lane == 0) tc::commit(dr);
            __syncwarp();
            mbar_wait_bounded(dr, 0);
        }
    } else {
        // ------------------------- softmax + epilogue warps -----------------------
        // Thread (part, r): row r of the tile (tensor-memory lane r) and part
        // `part` of its BN key columns [part * CPT, part * CPT + CPT).  The
        // parts agree on the row max through shared memory once per tile.
        constexpr int CPT = BN / SPLIT;
        constexpr int OPT = D / SPLIT;   // output columns per thread
        static_assert(CPT % 32 == 0 && OPT % 32 == 0, "column split");
        const int r = threadIdx.x & (kRows - 1);
        const int half = threadIdx.x >> 7;   // part index
        const int i = p0 + r / g;
        const int head = hkv * g + r % g;
        const bool row_valid = i <= p_last;
        const int hi = causal ? min(i + ctx, sk - 1) : sk - 1;
        const int lo = window ? max(0, i + ctx - p.window + 1) : 0;
        const bool softcap = (p.flags & UA_FLAG_SOFTCAP) != 0;
        const bool alibi = (p.flags & UA_FLAG_ALIBI) != 0;
        const float sl2 = p.scale * kLog2e;
        const float slope = alibi ? __ldg(p.alibi + head) : 0.f;
        const float inv_cap = softcap ? 1.0f / p.softcap : 0.f;
        // The row's line of the query-query bias (none for padding rows).
        const float* qrow = (QQ && row_valid)
                                ? p.qq_bias + (int64_t)i * p.qq_stride
                                : nullptr;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float* red = reinterpret_cast<float*>(smem + C::kOffRed);
        // Keys every row of the tile sees: [kfree_lo, kfree_hi].
        const int kfree_hi = causal ? min(p0 + ctx, sk - 1) : sk - 1;
        const int kfree_lo = window ? max(0, p_last + ctx - p.window + 1) : 0;

        // Warps whose 32 rows are all padding (past the sequence's last
        // position) skip the score work; they still take part in every
        // barrier.
        const bool live = __any_sync(0xffffffffu, row_valid);
        float m = -INFINITY;  // running max, log2 units (identical in both halves)
        float l = 0.f;        // this half's share of the running denominator
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const bool got = __all_sync(0xffffffffu, wait_or_abort(B.s_full0 + 8 * (j & 1), (j >> 1) & 1,
                                                                   abort_flag, p.err));
            uint32_t sr[CPT / 32][32];
            const int key0 = (t_last - j) * BN + half * CPT;
            float pmax = -INFINITY;
            if (got && live) {
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < CPT / 32; ++c)
                    tc::ld32(trow + C::kTmemS + (j & 1) * BN + half * CPT + c * 32, sr[c]);
                tc::wait_ld();
                const bool mask_free = key0 >= kfree_lo && key0 + CPT - 1 <= kfree_hi;
                if constexpr (!PLAIN) {
                    // ALiBi: one int -> float conversion per tile; the per-key
                    // offsets are compile-time constants.
                    const float abias = slope * (float)(key0 - ctx);
#pragma unroll
                    for (int c = 0; c < CPT / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float t = __uint_as_float(sr[c][e]) * p.scale;
                            if (softcap) t = p.softcap * tanh_from_exp2(t * inv_cap);
                            if (alibi) t += abias + slope * (float)(c * 32 + e);
                            sr[c][e] = __float_as_uint(t * kLog2e);
                        }
                    // Query-query bias, in its own pass so that the loop above
                    // stays as lean without it: the query-section keys up to
                    // the row's last visible key (so j - ctx < S_q), in log2
                    // units like the scores it joins.
                    if (QQ && qrow != nullptr && key0 + CPT > ctx && key0 <= hi) {
#pragma unroll
                        for (int c = 0; c < CPT / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int kc = key0 - ctx + c * 32 + e;
                                if (kc >= 0 && kc <= hi - ctx)
                                    sr[c][e] = __float_as_uint(__uint_as_float(sr[c][e]) +
                                                               __ldg(qrow + kc) * kLog2e);
                            }
                    }
                }
                if (!mask_free) {
#pragma unroll
                    for (int c = 0; c < CPT / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int kj = key0 + c * 32 + e;
                            if (kj < lo || kj > hi) sr[c][e] = __float_as_uint(-INFINITY);
                        }
                }
                // Eight independent three-input max chains, then combined.
                float mx[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
#pragma unroll
                for (int c = 0; c < CPT / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 16)
#pragma unroll
                        for (int a = 0; a < 8; ++a)
                            mx[a] = fmax3(mx[a], __uint_as_float(sr[c][e + 2 * a]),
                                          __uint_as_float(sr[c][e + 2 * a + 1]));
                pmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7]));
            }
            red[((j & 1) * SPLIT + half) * kRows + r] = pmax;
            // Exchange the partial maxima; the same barrier votes on whether
            // every softmax thread got its scores (else all leave together).
            if (!bar_and_sync(1, kSmThreads, got)) {
                ok = false;
                break;
            }
            float tmax = pmax;
#pragma unroll
            for (int o = 1; o < SPLIT; ++o)
                tmax = fmaxf(tmax, red[((j & 1) * SPLIT + ((half + o) % SPLIT)) * kRows + r]);
            if constexpr (PLAIN) tmax *= sl2;
            // Lazy re-anchor: move the reference max only when the tile's max
            // exceeds it by more than 8 (log2), so P stays at most 2^8.
            float alpha = 1.f;
            const bool reanchor = tmax > m + kLazy;
            if (reanchor) {
                alpha = fast_exp2(m - tmax);
                m = tmax;
            }
            const float m_use = (m == -INFINITY) ? 0.f : m;
            const float xs = PLAIN ? sl2 : 1.0f;
            // P = 2^(x - m): the exponent argument in fp32 (packed pairs), the
            // power of two on the fp32 special-function path, row sums in fp32,
            // P rounded to bf16 for the MMA.
            float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            const float2 sc2 = make_float2(xs, xs);
            const float2 nm2 = make_float2(-m_use, -m_use);
            uint32_t pk[CPT / 2];
#pragma unroll
            for (int c = 0; c < CPT / 32; ++c)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 a = ffma2(make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])),
                                           sc2, nm2);
                    const float2 pr = exp2_pair_f32(a);
                    rs[(e >> 1) & 3] = fadd2(rs[(e >> 1) & 3], pr);
                    pk[(c * 32 + e) / 2] = pack_bf16x2(pr.x, pr.y);
                }
            const float2 rs01 = fadd2(rs[0], rs[1]), rs23 = fadd2(rs[2], rs[3]);
            l = l * alpha + ((rs01.x + rs01.y) + (rs23.x + rs23.y));
            // P buffer j % 3 in tensor memory was read by the P.V of tile
            // j - 3; rescaling O needs the P.V of tile j - 1 to have finished.
            bool go = true;
            if (j >= 3) {
                go = __all_sync(0xffffffffu, wait_or_abort(B.o_done + 8 * (j % 3),
                                                           ((j - 3) / 3) & 1, abort_flag, p.err));
                if (go) tc::fence_after_sync();
            }
            if (go && live && j > 0 && __any_sync(0xffffffffu, reanchor)) {
                go = __all_sync(0xffffffffu, wait_or_abort(B.o_done + 8 * ((j - 1) % 3),
                                                           ((j - 1) / 3) & 1, abort_flag, p.err));
                if (go) tc::fence_after_sync();
            }
            if (go && live && j > 0 && __any_sync(0xffffffffu, reanchor)) {
#pragma unroll 1
                for (int c = 0; c < OPT / 32; ++c) {
                    uint32_t o[32];
                    const uint32_t col = C::kTmemO + half * OPT + c * 32;
                    tc::ld32(trow + col, o);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc::st32(trow + col, o);
                }
                tc::wait_st();
            }
            if (go) {
                // This part's CPT keys of row r -> tensor-memory P buffer
                // j % 3: lane r, two bf16 keys per 32-bit column, the A
                // operand of the P.V MMA.  Padding-only warps leave their rows
                // stale; those output rows are never stored.
                if (live) {
                    const uint32_t pcol = C::kTmemP + (j % 3) * (BN / 2) + half * (CPT / 2);
                    if constexpr (CPT / 2 == 32) {
                        tc::st32(trow + pcol, pk);
                    } else {
                        static_assert(CPT / 2 == 16, "P columns per thread");
                        tc::st16(trow + pcol, pk);
                    }
                    tc::wait_st();
                }
                tc::fence_before_sync();
                mbar_arrive(B.p_full + 8 * (j % 3));
            }
        }
        // ------------------------------ epilogue ---------------------------------
        if (ok) {
            const bool done = __all_sync(0xffffffffu,
                                         wait_or_abort(B.o_done + 8 * ((n_tiles - 1) % 3),
                                                       ((n_tiles - 1) / 3) & 1, abort_flag, p.err));
            red[half * kRows + r] = l;
            const bool all_done = bar_and_sync(1, kSmThreads, done);
            if (all_done && live && split) {
                // Split partial: raw o (this part's columns), m in log2 units, l.
                tc::fence_after_sync();
                float L = l;
#pragma unroll
                for (int o = 1; o < SPLIT; ++o) L += red[((half + o) % SPLIT) * kRows + r];
                const int64_t row = (q0 + i) * p.hq + head;
                const int64_t po = (row * p.splits + seg) * D + half * OPT;
                if (row_valid && half == 0) {
                    p.part_ml[(row * p.splits + seg) * 2 + 0] = m;
                    p.part_ml[(row * p.splits + seg) * 2 + 1] = L;
                }
#pragma unroll 1
                for (int c = 0; c < OPT / 32; ++c) {
                    uint32_t o[32];
                    tc::ld32(trow + C::kTmemO + half * OPT + c * 32, o);
                    tc::wait_ld();
                    if (row_valid) part_store32(p, po + c * 32, o);
                }
            } else if (all_done && live && !split) {
                tc::fence_after_sync();
                float O_scale_num = 1.f;  // extra factor from the sink re-basing
                float L = l;
#pragma unroll
                for (int o = 1; o < SPLIT; ++o) L += red[((half + o) % SPLIT) * kRows + r];
                bool zero = false;
                if (p.flags & UA_FLAG_SINKS) {
                    const float s2 = __ldg(p.sinks + head) * kLog2e;
                    if (s2 == INFINITY) {
                        zero = true;
                    } else if (s2 > m) {
                        const float a = (m == -INFINITY) ? 0.f : fast_exp2(m - s2);
                        O_scale_num = a;
                        L = L * a + 1.0f;
                    } else if (s2 != -INFINITY) {
                        L += fast_exp2(s2 - m);
                    }
                }
                const float inv = (!zero && L > 0.f) ? O_scale_num * __frcp_rn(L) : 0.f;
                __nv_bfloat16* orow = p.out + ((q0 + i) * p.hq + head) * (int64_t)D + half * OPT;
#pragma unroll 1
                for (int c = 0; c < OPT / 32; ++c) {
                    uint32_t o[32];
                    tc::ld32(trow + C::kTmemO + half * OPT + c * 32, o);
                    tc::wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
                            v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                            v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                            v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                            *reinterpret_cast<uint4*>(orow + c * 32 + e) = v;
                        }
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int BN, int NK, int NV, int SPLIT, bool PLAIN, bool QQ = false>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const FwdParams& p, int tiles, cudaStream_t stream) {
    using C = PCfg<D, BN, NK, NV, SPLIT>;
    constexpr int kThreads = Roles<SPLIT>::kThreads;
    auto kern = prefill_kernel<D, BN, NK, NV, SPLIT, PLAIN, QQ>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(tiles * p.splits), (unsigned)p.hk, (unsigned)p.num_seqs);
    kern<<<grid, kThreads, C::kSmem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

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
    if (prefill_pair_supported(p.d))
        return plan.dense ? launch_prefill_grid(tq, tm_k, tm_v, p, (plan.num_tiles + 1) / 2, stream)
                          : launch_prefill_pair(tq, tm_k, tm_v, p, plan.ctas, stream);
    if (p.d != 256) return cudaErrorInvalidValue;
    return launch_prefill_cta2(tq, tm_k, tm_v, p, (plan.num_tiles + 1) / 2, stream);
}

}  // namespace ua
