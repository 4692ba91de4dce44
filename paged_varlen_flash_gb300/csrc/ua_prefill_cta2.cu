// ua_prefill_cta2.cu -- prefill / chunked-prefill attention for head size 256
// on CTA pairs: the two CTAs of a cluster run the tcgen05 MMAs of two query
// tiles together (cta_group::2, M = 256), so each CTA holds only half of every
// K and V tile in its shared memory and reads half of each MMA's B operand.
//
// Work unit: one cluster per (pair of adjacent tiles of 128 packed (position,
// head) rows of one KV head, sequence[, KV segment]).  CTA 0 of the pair
// owns the lower tile and issues the pair's MMAs; CTA 1 owns the upper tile.
// The g query heads that share a KV head are packed into a tile's rows
// (gfx950 "Unified paged attention on gfx950, from the math up", section 4,
// GQA packing).  Both CTAs walk the union of the two tiles' visible key
// tiles, 128 keys at a time, with the streaming (m, l, o) recurrence of
// gfx1151 ALGORITHM.md section 3 in base 2 (gfx950 section 2), the lazy
// re-anchor threshold of 8, mask-free interior tiles, the causal early exit
// and sliding-window start of attention_dense.py (gfx950 section 8.1); keys
// the lower tile cannot see in the pair's last tile are masked in its rows.
// Key tiles are visited from the diagonal backwards (the result does not
// depend on the order; with causal ALiBi the scores grow toward the diagonal,
// so the running max rarely needs re-anchoring).
//
// Per 128-key tile j (tensor memory of each CTA: S0 [0, 128), S1 [128, 256),
// O [256, 512); P(j) bf16 is written over the first 64 columns of S(j & 1)):
//   S(j) = Q K(j)^T    M = 256, N = 128 keys (64 held by each CTA), K = 256
//   O += P(j) V(j)     M = 256, N = 256 (128 of d held by each CTA), K = 128
// S(j + 2) = Q K(j + 2)^T overwrites the columns that hold P(j), so its
// issuer waits for P.V(j) to complete first.
//
// Roles (12 warps per CTA):
//   warps 0-7  softmax + epilogue: two warpgroups share each row's 128 key
//              columns (64 each; one shared-memory max exchange per tile);
//   warp 8     TMA producer of Q (once) and of this CTA's 64 keys of each K
//              tile, through a 2-stage ring; the copies complete on CTA 0's
//              barrier directly;
//   warp 9     tensor-memory allocation (both CTAs) and, in CTA 0, the QK^T
//              issuer;
//   warp 10    TMA producer of this CTA's 128 columns of d of each V tile
//              (2-stage ring, completing on a local barrier); zeroes the rows
//              past S_k of the sequence's last tile, then signals CTA 0;
//   warp 11    in CTA 0, the P.V issuer.
#include <algorithm>
#include <cstdint>

#include "ua_common.cuh"
#include "ua_prefill.h"
#include "ua_prefill_common.cuh"
#include "ua_ptx.cuh"
#include "ua_tc.cuh"

namespace ua {
namespace {

using namespace pf;

constexpr int kD = 256;
constexpr int kBN = 128;          // keys per tile
constexpr int kHalfKeys = 64;     // keys of a K tile held by each CTA
constexpr int kSplit = 2;         // softmax warpgroups sharing a row
constexpr int kCPT = kBN / kSplit;    // key columns per softmax thread
constexpr int kOPT = kD / kSplit;     // output columns per softmax thread
constexpr int kThreads2 = 128 * kSplit + 128;
constexpr int kSmThreads2 = 128 * kSplit;
constexpr int kWarpTma2 = 8, kWarpMma2 = 9, kWarpRel2 = 10, kWarpPv2 = 11;

template <int NK, int NV>
struct C2Cfg {
    static constexpr int kPanels = kD / 64;
    static constexpr int kQPanel = kRows * 128;          // 128 rows x 64 d
    static constexpr int kQBytes = kPanels * kQPanel;
    static constexpr int kKPanel = kHalfKeys * 128;      // 64 keys x 64 d
    static constexpr int kKBytes = kPanels * kKPanel;
    static constexpr int kVPanel = kBN * 128;            // 128 keys x 64 d
    static constexpr int kVBytes = 2 * kVPanel;          // this CTA's 128 columns of d
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + NK * kKBytes;
    static constexpr int kOffBar = kOffV + NV * kVBytes;
    // q_full, k_full[NK], k_empty[NK], v_land[NV], v_full[NV], v_empty[NV],
    // s_full[2], p_full[2], pv_done[2], drain[2], never (the testing hook's
    // stall waits on it; nothing arrives)
    static constexpr int kNumBars = 1 + 2 * NK + 3 * NV + 6 + 3;
    static constexpr int kOffRed = (kOffBar + kNumBars * 8 + 15) / 16 * 16;   // [2][kSplit][128] fp32
    static constexpr int kOffMisc = kOffRed + 2 * kSplit * kRows * 4;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static constexpr int kTmemO = 2 * kBN;
    static_assert(kTmemO + kD <= (int)kTmemCols, "tensor memory budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};

template <int NK, int NV, bool PLAIN, bool QQ>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads2, 1)
prefill_cta2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
    using C = C2Cfg<NK, NV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0: lower tile, MMA issuer
    const int s = blockIdx.z;
    const int hkv = blockIdx.y;
    const bool split = p.splits > 1;             // write (m, l, o) partials per KV segment
    const int unit = (int)(blockIdx.x >> 1);
    const int seg = unit % p.splits;
    const int npairs = (int)(gridDim.x >> 1) / p.splits;
    const int pair = npairs - 1 - unit / p.splits;   // heaviest first
    const int g = p.g;
    const int ppt = kRows / g;                  // positions per tile
    const int p0_pair = pair * 2 * ppt;
    const int p0 = p0_pair + (int)rank * ppt;   // this CTA's tile

    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, s, sq, sk, q0);
    if (st && pair == 0 && hkv == 0 && seg == 0 && rank == 0 && threadIdx.x == 0) atomicOr(p.err, (int)st);
    // Every exit before the pair's first cluster barrier depends on the pair
    // only, so both CTAs leave together.
    if (st & UA_DEVERR_CU_SEQLENS) return;
    if (p0_pair >= sq) return;
    if (seg >= (split ? seq_segments(p, st, sk) : 1)) return;
    const int p_last = min(p0 + ppt, sq) - 1;   // < p0 when the upper tile is past S_q
    const int last_pair = min(p0_pair + 2 * ppt, sq) - 1;
    const int ctx = sk - sq;
    const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
    const bool window = (p.flags & UA_FLAG_WINDOW) != 0;
    int k_end = causal ? min(sk, last_pair + ctx + 1) : sk;
    int k_beg = window ? max(0, p0_pair + ctx - p.window + 1) : 0;
    if (split) {  // this pair's KV segment; segments are whole tiles
        k_beg = max(k_beg, seg * p.chunk);
        k_end = min(k_end, seg * p.chunk + p.chunk);
    }
    if (st || k_beg >= k_end) {
        // Malformed lengths (rows written as zeros) or a segment with no
        // visible key for any row of the pair (an empty partial, m = -inf).
        for (int e = threadIdx.x; e < kRows * (kD / 8); e += kThreads2) {
            const int r = e / (kD / 8), c = e % (kD / 8);
            const int i = p0 + r / g;
            if (i > p_last) continue;
            const int64_t row = (q0 + i) * p.hq + hkv * g + r % g;
            if (split) {
                if (c == 0) {
                    p.part_ml[(row * p.splits + seg) * 2 + 0] = -INFINITY;
                    p.part_ml[(row * p.splits + seg) * 2 + 1] = 0.f;
                }
            } else {
                *reinterpret_cast<uint4*>(p.out + row * kD + c * 8) = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int t_begin = k_beg / kBN;
    const int n_tiles = (k_end + kBN - 1) / kBN - t_begin;
    const int t_last = t_begin + n_tiles - 1;   // step j visits tile t_last - j

    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    const uint32_t q_full = smem_u32(&bar_mem[0]);
    const uint32_t k_full0 = smem_u32(&bar_mem[1]);             // + 8 * stage (CTA 0's)
    const uint32_t k_empty0 = smem_u32(&bar_mem[1 + NK]);
    const uint32_t v_land0 = smem_u32(&bar_mem[1 + 2 * NK]);     // this CTA's V copy landed
    const uint32_t v_full0 = smem_u32(&bar_mem[1 + 2 * NK + NV]);   // both halves ready (CTA 0's)
    const uint32_t v_empty0 = smem_u32(&bar_mem[1 + 2 * NK + 2 * NV]);
    constexpr int kBarS = 1 + 2 * NK + 3 * NV;
    const uint32_t s_full0 = smem_u32(&bar_mem[kBarS]);         // + 8 * (j & 1)
    const uint32_t p_full0 = smem_u32(&bar_mem[kBarS + 2]);     // CTA 0's: 8 warps x 2 CTAs
    const uint32_t pv_done0 = smem_u32(&bar_mem[kBarS + 4]);
    const uint32_t drain0 = smem_u32(&bar_mem[kBarS + 6]);     // + 8 * issuer
    const uint32_t never = smem_u32(&bar_mem[kBarS + 8]);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < NK; ++i) {
            mbar_init(k_full0 + 8 * i, 1);
            mbar_init(k_empty0 + 8 * i, 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(v_land0 + 8 * i, 1);
            mbar_init(v_full0 + 8 * i, 2);
            mbar_init(v_empty0 + 8 * i, 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full0 + 8 * x, 1);
            mbar_init(p_full0 + 8 * x, 2 * kSmThreads2 / 32);
            mbar_init(pv_done0 + 8 * x, 1);
        }
        mbar_init(drain0, 1);
        mbar_init(drain0 + 8, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma2) {
        tc::tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish_pair();
    }
    // Both CTAs' barriers and tensor memory exist before either signals the other.
    tc::fence_before_sync();
    __syncwarp();
    cluster_sync_all();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sK = smem_u32(smem + C::kOffK);
    const uint32_t sV = smem_u32(smem + C::kOffV);
    const int b = p.b;
    const int nblk_seq = (sk + b - 1) / b;
    // Blocks of this CTA's share of tile t: its 64 keys of K, all 128 keys of V.
    auto k_blocks = [&](int key0, uint32_t r) {
        return max(0, min(kHalfKeys / b, nblk_seq - (key0 + (int)r * kHalfKeys) / b));
    };
    auto v_blocks = [&](int key0) { return max(0, min(kBN / b, nblk_seq - key0 / b)); };

    const int32_t* bt = p.block_table + (int64_t)s * p.bt_stride;
    if (warp == kWarpTma2) {
        // --------------------------- TMA producer: Q, K ---------------------------
        // Lane i owns paged block i of this CTA's 64 keys of each K tile (its
        // id load and its boxes), so a tile's boxes go out in parallel.  K runs
        // ahead of V on its own warp: the next K tile is requested as soon as
        // the QK^T two tiles back has read its stage.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            // g heads x ppt positions per panel and tile, both tiles of the pair
            if (rank == 0)
                mbar_arrive_expect_tx(q_full, 2u * (uint32_t)(g * ppt) * 128u * C::kPanels);
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_3d_pair(sQ + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, (int)(q0 + p0),
                                 mapa_shared(q_full, 0));
        }
        auto tile_id = [&](int j) -> int32_t {   // lane i: block i of this CTA's K keys
            const int blk0 = ((t_last - j) * kBN + (int)rank * kHalfKeys) / b;
            return lane < min(kHalfKeys / b, nblk_seq - blk0) ? __ldg(bt + blk0 + lane) : 0;
        };
        const uint32_t k_full_lead0 = mapa_shared(k_full0, 0);
        int32_t id_next = tile_id(0);
        for (int j = 0; j < n_tiles; ++j) {
            const int stk = j % NK;
            const int key0 = (t_last - j) * kBN;
            const int nbk = k_blocks(key0, rank);
            const int32_t id = id_next;
            if (j + 1 < n_tiles) id_next = tile_id(j + 1);
            if (j >= NK && !__all_sync(0xffffffffu, wait_or_abort(k_empty0 + 8 * stk, ((j / NK) + 1) & 1,
                                                                   abort_flag, p.err)))
                break;
            if (rank == 0 && lane == 0) {
                const uint32_t kb = (uint32_t)(k_blocks(key0, 0) + k_blocks(key0, 1)) * b * 128 * C::kPanels;
                mbar_arrive_expect_tx(k_full0 + 8 * stk, kb);
            }
            __syncwarp();
            if (lane < nbk) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_4d_pair(sK + stk * C::kKBytes + pn * C::kKPanel + lane * b * 128, &tm_k,
                                     pn * 64, hkv, 0, id, k_full_lead0 + 8 * stk);
            }
        }
        __syncwarp();
    } else if (warp == kWarpRel2) {
        // ------------------- V producer, zero fill and release --------------------
        // Lane i owns paged block i of each V tile's 128 keys (this CTA's 128
        // columns of d).  Keys past S_k: whatever their V slots hold must not
        // reach O (0 * NaN is NaN), so those rows become zeros before CTA 0 is
        // told the tile is ready.  V(j + NV) is requested once the P.V of
        // tile j has read its stage.
        if (lane == 0) tma_prefetch_desc(&tm_v);
        const uint32_t v_full_lead0 = mapa_shared(v_full0, 0);
        auto issue_v = [&](int j) -> bool {
            const int stv = j % NV;
            const int key0 = (t_last - j) * kBN;
            const int nbv = v_blocks(key0);
            const int blk0 = key0 / b;
            const int32_t id = lane < nbv ? __ldg(bt + blk0 + lane) : 0;
            if (lane < nbv && (id < 0 || (int64_t)id >= p.num_blocks))
                atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
            if (j >= NV && !__all_sync(0xffffffffu, wait_or_abort(v_empty0 + 8 * stv, ((j / NV) + 1) & 1,
                                                                   abort_flag, p.err)))
                return false;
            if (lane == 0) mbar_arrive_expect_tx(v_land0 + 8 * stv, (uint32_t)nbv * b * 128 * 2);
            __syncwarp();
            if (lane < nbv) {
#pragma unroll
                for (int pn = 0; pn < 2; ++pn)
                    tma_load_4d(sV + stv * C::kVBytes + pn * C::kVPanel + lane * b * 128, &tm_v,
                                ((int)rank * 2 + pn) * 64, hkv, 0, id, v_land0 + 8 * stv);
            }
            return true;
        };
        int issued = 0;
        bool ok = true;
        for (; ok && issued < min(NV, n_tiles); ++issued) ok = issue_v(issued);
        for (int j = 0; ok && j < n_tiles; ++j) {
            const int stv = j % NV;
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(v_land0 + 8 * stv, (j / NV) & 1, abort_flag, p.err))))
                break;
            const int key0 = (t_last - j) * kBN;
            const int nvalid = min(kBN, sk - key0);
            if (nvalid < kBN) {
                uint8_t* vgen = smem + C::kOffV + stv * C::kVBytes;
                const int per_panel = (kBN - nvalid) * 8;
                for (int e = lane; e < per_panel * 2; e += 32) {
                    const int pn = e / per_panel, rem = e % per_panel;
                    *reinterpret_cast<uint4*>(vgen + pn * C::kVPanel + (nvalid + rem / 8) * 128 +
                                              (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(v_full_lead0 + 8 * stv);
            if (issued < n_tiles && (ok = issue_v(issued))) ++issued;
        }
        if (*abort_flag && lane == 0) {
            // Let the V copies this warp issued land before the CTA ends (the
            // K copies complete on CTA 0's barrier and land within
            // microseconds; the pair leaves only after the final cluster
            // barrier, at least one wait limit later).
            for (int j = max(0, issued - NV); j < issued; ++j)
                mbar_wait_bounded(v_land0 + 8 * (j % NV), (j / NV) & 1);
        }
        __syncwarp();
    } else if (warp == kWarpMma2 || warp == kWarpPv2) {
        // (CTA 1's warps 9 and 11 have no MMA work: they go straight to the end.)
        if (rank == 0) {
        // --------------------- MMA issuers (CTA 0, two threads) ---------------------
        // Warp 9 issues every S(j) = Q K(j)^T, warp 11 every O += P(j) V(j), so
        // a P.V is queued as soon as its P is written instead of behind the
        // issue of the next QK^T (with one issuing thread the pipe idled
        // between them: an MMA issue returns only as the pipe drains).
        // S(j + 2) overwrites the columns that hold P(j), so its issuer first
        // waits for P.V(j) to complete.
        constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(2 * kRows, kBN, false, false);
        constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(2 * kRows, kD, false, true);
        const uint32_t peer = 1;
        const bool qk_role = warp == kWarpMma2;
        // Shared-memory descriptors as a base per operand buffer plus a
        // compile-time offset per MMA: the start-address field holds the byte
        // address >> 4 (below 2^14 for any shared-memory address), so adding
        // an offset never carries into the next field.
        const uint64_t q_desc = tc::smem_desc_sw128(sQ, 16, 1024);
        const uint64_t k_desc0 = tc::smem_desc_sw128(sK, 16, 1024);
        const uint64_t v_desc0 = tc::smem_desc_sw128(sV, C::kVPanel, 1024);
        auto wwait = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_or_abort(bar, par, abort_flag, p.err));
        };
        auto commit_both = [&](uint32_t bar) {
            tc::commit_pair(bar);
            tc::commit_pair(mapa_shared(bar, peer));
        };
        bool ok = true;
        if (qk_role) {
            ok = wwait(q_full, 0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int stg = j % NK;
                // Testing hook: the first K wait waits on a barrier that
                // nothing completes and gives up after stall_ns.
                if (p.stall && j == 0 &&
                    !(ok = __all_sync(0xffffffffu, wait_or_abort(never, 0, abort_flag, p.err,
                                                                 (uint64_t)p.stall_ns))))
                    break;
                if (j >= 2 && !(ok = wwait(pv_done0 + 8 * (j & 1), ((j - 2) >> 1) & 1))) break;
                if (!(ok = wwait(k_full0 + 8 * stg, (j / NK) & 1))) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t dS = tmem + (j & 1) * kBN;
                    const uint64_t kd_s = k_desc0 + (uint64_t)(((uint32_t)stg * C::kKBytes) >> 4);
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {
                        const uint32_t oq = ((k >> 2) * C::kQPanel + (k & 3) * 32) >> 4;
                        const uint32_t ok_ = ((k >> 2) * C::kKPanel + (k & 3) * 32) >> 4;
                        tc::mma_bf16_pair(dS, q_desc + oq, kd_s + ok_, idesc_qk, k > 0 ? 1u : 0u);
                    }
                    commit_both(s_full0 + 8 * (j & 1));
                    commit_both(k_empty0 + 8 * stg);
                }
                __syncwarp();
            }
        } else {
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int stv = j % NV;
                if (!(ok = wwait(p_full0 + 8 * (j & 1), (j >> 1) & 1))) break;
                if (!(ok = wwait(v_full0 + 8 * stv, (j / NV) & 1))) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint64_t vd_s = v_desc0 + (uint64_t)(((uint32_t)stv * C::kVBytes) >> 4);
                    const uint32_t aP = tmem + (j & 1) * kBN;
#pragma unroll
                    for (int k = 0; k < kBN / 16; ++k) {
                        // A = P from tensor memory: 16 keys per MMA = 8 columns.
                        tc::mma_bf16_ts_pair(tmem + C::kTmemO, aP + k * 8, vd_s + ((k * 16 * 128) >> 4), idesc_pv,
                                             (j > 0 || k > 0) ? 1u : 0u);
                    }
                    commit_both(v_empty0 + 8 * stv);
                    commit_both(pv_done0 + 8 * (j & 1));
                }
                __syncwarp();
            }
        }
        // No MMA of the pair may still run when either CTA frees its tensor
        // memory or leaves.
        const uint32_t dr = drain0 + (qk_role ? 0 : 8);
        if (lane == 0) tc::commit_pair(dr);
        __syncwarp();
        mbar_wait_bounded(dr, 0);
        }
    } else {
        // ------------------------- softmax + epilogue warps -----------------------
        // Thread (part, r): row r of this CTA's tile (tensor-memory lane r) and
        // key columns [part * 64, part * 64 + 64) of each tile.  The parts
        // agree on the row max through shared memory once per tile.
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
        const float* qrow = (QQ && row_valid) ? p.qq_bias + (int64_t)i * p.qq_stride : nullptr;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float* red = reinterpret_cast<float*>(smem + C::kOffRed);
        // Keys every row of this tile sees: [kfree_lo, kfree_hi].
        const int kfree_hi = causal ? min(p0 + ctx, sk - 1) : sk - 1;
        const int kfree_lo = window ? max(0, p_last + ctx - p.window + 1) : 0;
        const uint32_t p_full_lead0 = mapa_shared(p_full0, 0);

        // Warps whose 32 rows are all padding skip the score work; they
        // still take part in every barrier.
        const bool live = __any_sync(0xffffffffu, row_valid);
        float m = -INFINITY;  // running max, log2 units (identical in both parts)
        float l = 0.f;        // this part's share of the running denominator
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const uint32_t sbuf = (uint32_t)(j & 1) * kBN;
            const bool got = __all_sync(0xffffffffu, wait_or_abort(s_full0 + 8 * (j & 1), (j >> 1) & 1,
                                                                   abort_flag, p.err));
            uint32_t sr[kCPT / 32][32];
            const int key0 = (t_last - j) * kBN + half * kCPT;
            float pmax = -INFINITY;
            if (got && live) {
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < kCPT / 32; ++c) tc::ld32(trow + sbuf + half * kCPT + c * 32, sr[c]);
                tc::wait_ld();
                const bool mask_free = key0 >= kfree_lo && key0 + kCPT - 1 <= kfree_hi;
                if constexpr (!PLAIN) {
                    // ALiBi: one int -> float conversion per tile; the per-key
                    // offsets are compile-time constants.
                    const float abias = slope * (float)(key0 - ctx);
                    if (softcap) {
#pragma unroll
                        for (int c = 0; c < kCPT / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                float t = __uint_as_float(sr[c][e]) * p.scale;
                                t = p.softcap * tanh_from_exp2(t * inv_cap);
                                if (alibi) t += abias + slope * (float)(c * 32 + e);
                                sr[c][e] = __float_as_uint(t * kLog2e);
                            }
                    } else {
                        // No softcap: the score and the ALiBi term straight in
                        // log2 units, two FMAs per score (slope = 0 without
                        // ALiBi).
                        const float sc2 = p.scale * kLog2e, sl2a = slope * kLog2e, ab2 = abias * kLog2e;
#pragma unroll
                        for (int c = 0; c < kCPT / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                sr[c][e] = __float_as_uint(fmaf(__uint_as_float(sr[c][e]), sc2,
                                                                fmaf(sl2a, (float)(c * 32 + e), ab2)));
                    }
                    // Query-query bias, in its own pass: the query-section keys
                    // up to the row's last visible key (so j - ctx < S_q), in
                    // log2 units like the scores it joins.
                    if (QQ && qrow != nullptr && key0 + kCPT > ctx && key0 <= hi) {
#pragma unroll
                        for (int c = 0; c < kCPT / 32; ++c)
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
                    for (int c = 0; c < kCPT / 32; ++c)
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
                for (int c = 0; c < kCPT / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 16)
#pragma unroll
                        for (int a = 0; a < 8; ++a)
                            mx[a] = fmax3(mx[a], __uint_as_float(sr[c][e + 2 * a]),
                                          __uint_as_float(sr[c][e + 2 * a + 1]));
                pmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7]));
            }
            red[((j & 1) * kSplit + half) * kRows + r] = pmax;
            // Exchange the partial maxima.  The same barrier orders both
            // parts' reads of S(j) before either writes P(j) over its first
            // 64 columns, and votes on whether every softmax thread got its
            // scores (else all leave together).
            tc::fence_before_sync();
            if (!bar_and_sync(1, kSmThreads2, got)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float tmax = pmax;
#pragma unroll
            for (int o = 1; o < kSplit; ++o)
                tmax = fmaxf(tmax, red[((j & 1) * kSplit + ((half + o) % kSplit)) * kRows + r]);
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
            uint32_t pk[kCPT / 2];
#pragma unroll
            for (int c = 0; c < kCPT / 32; ++c)
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
            // Rescaling O needs the P.V of tile j - 1 to have finished.
            bool go = true;
            if (live && j > 0 && __any_sync(0xffffffffu, reanchor)) {
                go = __all_sync(0xffffffffu, wait_or_abort(pv_done0 + 8 * ((j - 1) & 1),
                                                           ((j - 1) >> 1) & 1, abort_flag, p.err));
                if (go) {
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < kOPT / 32; ++c) {
                        uint32_t o[32];
                        const uint32_t col = C::kTmemO + half * kOPT + c * 32;
                        tc::ld32(trow + col, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st32(trow + col, o);
                    }
                    tc::wait_st();
                }
            }
            if (!go) {
                ok = false;
                break;
            }
            // This part's 64 keys of row r -> P(j) over S(j & 1): lane r, two
            // bf16 keys per 32-bit column (part 0 in columns 0-31, part 1 in
            // 32-63), the A operand of the P.V MMA.  Padding-only warps leave
            // their rows stale; those output rows are never stored.
            if (live) {
                tc::st32(trow + sbuf + half * (kCPT / 2), pk);
                tc::wait_st();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(p_full_lead0 + 8 * (j & 1));
        }
        // ------------------------------ epilogue ---------------------------------
        if (ok) {
            const bool done = __all_sync(0xffffffffu,
                                         wait_or_abort(pv_done0 + 8 * ((n_tiles - 1) & 1),
                                                       ((n_tiles - 1) >> 1) & 1, abort_flag, p.err));
            red[half * kRows + r] = l;
            const bool all_done = bar_and_sync(1, kSmThreads2, done);
            if (all_done && live && split) {
                // Split partial: raw o (this part's columns), m in log2 units, l.
                tc::fence_after_sync();
                float L = l;
#pragma unroll
                for (int o = 1; o < kSplit; ++o) L += red[((half + o) % kSplit) * kRows + r];
                const int64_t row = (q0 + i) * p.hq + head;
                const int64_t po = (row * p.splits + seg) * kD + half * kOPT;
                if (row_valid && half == 0) {
                    p.part_ml[(row * p.splits + seg) * 2 + 0] = m;
                    p.part_ml[(row * p.splits + seg) * 2 + 1] = L;
                }
#pragma unroll 1
                for (int c = 0; c < kOPT / 32; ++c) {
                    uint32_t o[32];
                    tc::ld32(trow + C::kTmemO + half * kOPT + c * 32, o);
                    tc::wait_ld();
                    if (row_valid) part_store32(p, po + c * 32, o);
                }
            } else if (all_done && !split) {
                // A tile whose rows are all valid goes out through shared
                // memory (the K stages, free once the last MMA has run) and
                // one TMA store per 64-column panel: rows of a tile lie H_q * d
                // elements apart in the output, so per-thread row stores
                // would touch one sector per lane.  The last tile of a
                // sequence, whose padding rows must not be written, keeps
                // the per-thread stores.
                const bool staged = p_last - p0 + 1 == ppt;
                const uint32_t sO = smem_u32(smem + C::kOffK);
                static_assert(NK * C::kKBytes >= C::kPanels * C::kQPanel, "output staging");
                if (live) {
                    tc::fence_after_sync();
                    float O_scale_num = 1.f;  // extra factor from the sink re-basing
                    float L = l;
#pragma unroll
                    for (int o = 1; o < kSplit; ++o) L += red[((half + o) % kSplit) * kRows + r];
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
                    __nv_bfloat16* orow = p.out + ((q0 + i) * p.hq + head) * (int64_t)kD + half * kOPT;
#pragma unroll 1
                    for (int c = 0; c < kOPT / 32; ++c) {
                        uint32_t o[32];
                        tc::ld32(trow + C::kTmemO + half * kOPT + c * 32, o);
                        tc::wait_ld();
                        if (row_valid) {
#pragma unroll
                            for (int e = 0; e < 32; e += 8) {
                                uint4 v;
                                v.x = pack_bf16x2(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
                                v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                                v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                                v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                                if (staged) {
                                    // panel half * 2 + c / 2, 16-byte chunk (c % 2) * 4 + e / 8
                                    // of row r, 128-byte swizzled like the map's boxes
                                    const int chunk = (c & 1) * 4 + e / 8;
                                    *reinterpret_cast<uint4*>(smem + C::kOffK + (half * 2 + c / 2) * C::kQPanel +
                                                              r * 128 + ((chunk ^ (r & 7)) * 16)) = v;
                                } else {
                                    *reinterpret_cast<uint4*>(orow + c * 32 + e) = v;
                                }
                            }
                        }
                    }
                }
                if (staged) {
                    fence_proxy_async_smem();
                    bar_and_sync(1, kSmThreads2, true);
                    if (threadIdx.x == 0) {
#pragma unroll
                        for (int pn = 0; pn < C::kPanels; ++pn)
                            tma_store_3d(&tm_o, pn * 64, hkv * g, (int)(q0 + p0), sO + pn * C::kQPanel);
                        bulk_commit_and_wait_read();
                    }
                }
            }
        }
    }

    // Every role of both CTAs ends here: CTA 0 has drained its MMAs, so
    // neither CTA's shared or tensor memory is still read when it is freed.
    tc::fence_before_sync();
    __syncthreads();
    cluster_sync_all();   // (convergent: every thread arrives here once)
    if (warp == kWarpMma2) {
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem, kTmemCols);
    }
}

template <int NK, int NV, bool PLAIN, bool QQ = false>
cudaError_t launch_cta2_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& to, const FwdParams& p, int pairs, cudaStream_t stream) {
    using C = C2Cfg<NK, NV>;
    auto kern = prefill_cta2_kernel<NK, NV, PLAIN, QQ>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(2 * pairs * p.splits), (unsigned)p.hk, (unsigned)p.num_seqs);
    kern<<<grid, kThreads2, C::kSmem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_cta2(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& to, const FwdParams& p, int pairs, cudaStream_t stream) {
    if (p.d != kD || (p.b != 16 && p.b != 32 && p.b != 64)) return cudaErrorInvalidValue;
    const bool qq = (p.flags & UA_FLAG_QQ_BIAS) != 0;
    const bool plain = !qq && (p.flags & (UA_FLAG_SOFTCAP | UA_FLAG_ALIBI)) == 0;
    if (qq) return launch_cta2_t<2, 2, false, true>(tq, tm_k, tm_v, to, p, pairs, stream);
    return plain ? launch_cta2_t<2, 2, true>(tq, tm_k, tm_v, to, p, pairs, stream)
                 : launch_cta2_t<2, 2, false>(tq, tm_k, tm_v, to, p, pairs, stream);
}

}  // namespace ua
