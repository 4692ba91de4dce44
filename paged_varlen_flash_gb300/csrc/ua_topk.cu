// ua_topk.cu -- sparse top-k decode on the tcgen05 tensor cores: every query
// token attends to its own list of key positions in its sequence's paged
// cache (the token-granular top-k gather of "[Triton/Gluon] [GFX950] Sparse
// paged attention and Sparse MLA"), not to all of its S_k keys.
//
// One CTA serves one (query token, KV head, list segment); its rows are the g
// query heads of that KV head (g <= 16).  The products are laid out as in the
// decode kernel, keys on the MMA M dimension:
//
//     S^T [128 listed keys x 16 rows] = K_gathered [128 x d] * Q^T [d x 16]
//     O^T [d x 16 rows]              += V_gathered^T [d x 128] * P^T [128 x 16]
//
// The K and V tiles are gathered row by row into the same 128-byte-swizzled
// panels a paged TMA box would give.  Each cache is viewed as a 2-D tensor
// [num_blocks * b * H_k rows, d columns]; a lane maps four list entries
// through the block table to their cache rows.  By default K comes through
// TMA tile::gather4 (box = one 64-dim panel of one row, four rows per
// instruction) and V through 16-byte cp.async from a second loader warp (one
// warp instruction moves two 256-byte rows): the row requests an SM keeps in
// flight bound this kernel, and the two paths draw on separate capacity.
// Entries that are not keys of the row (padding, out of range, hidden by the
// causal mask or the window, or in a bad block) have their scores masked;
// their V rows are written as zeros (cp.async loader) or zeroed by the P.V
// issuer before the MMA (gather4 loader, which fetches row 0 for them), since
// a weight of 0 times stale data could still be NaN.
//
// The softmax is the decode kernel's: base 2, lazy re-anchor, fp32 (m, l),
// P in bf16, O^T rescaled in tensor memory; the score chain (scale, softcap,
// ALiBi, QQ-bias, masks) uses the listed position j of each key (gfx950
// "Unified paged attention on gfx950, from the math up", section 1).  Long
// lists are split into segments of whole 128-entry tiles whose partials the
// combine kernel merges (section 5); the number of segments is taken per
// token from its own list length, and surplus CTAs return at once.
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "ua_common.cuh"
#include "ua_decode_common.cuh"
#include "ua_ptx.cuh"
#include "ua_tc.cuh"
#include "ua_tmap.h"
#include "ua_topk.h"

// K and V ring depths (two CTAs per SM hold NSK + NSV <= 3 stages).
#ifndef UA_TOPK_NSK
#define UA_TOPK_NSK 1
#endif
#ifndef UA_TOPK_NSV
#define UA_TOPK_NSV 1
#endif
#ifndef UA_TOPK_MIN_TILES
#define UA_TOPK_MIN_TILES 4
#endif
// How each operand's rows are fetched: 1 = 16-byte cp.async from a loader
// warp (coalesced: one warp instruction moves two 256-byte rows), 0 = TMA
// tile::gather4 from the producer warp.
#ifndef UA_TOPK_K_LSU
#define UA_TOPK_K_LSU 0
#endif
#ifndef UA_TOPK_V_LSU
#define UA_TOPK_V_LSU 1
#endif
#define UA_TOPK_LSU (UA_TOPK_K_LSU || UA_TOPK_V_LSU)

namespace ua {
namespace {

constexpr int kN = 16;          // rows per tile (MMA N): the g heads of one token, padded
constexpr int kBN = 128;        // list entries per tile (MMA M of S^T)
constexpr int kD = 128;         // head size
// 4 softmax warps, K loader (also Q), QK^T issuer, P.V issuer, V loader (LSU)
constexpr int kThreads = UA_TOPK_LSU ? 256 : 224;
constexpr int kWarpTma = 4;
constexpr int kWarpLdV = 7;
constexpr int kWarpMma = 5;     // QK^T issuer (also allocates tensor memory)
constexpr int kWarpPv = 6;      // P.V issuer
constexpr float kLazy = 8.0f;

template <int NSK, int NSV>
struct TCfg {
    static constexpr int kPanels = kD / 64;
    static constexpr int kQPanel = kN * 128;              // 16 rows x 64 dims
    static constexpr int kQBytes = kPanels * kQPanel;
    static constexpr int kKvPanel = kBN * 128;            // 128 rows x 64 dims
    static constexpr int kKvBytes = kPanels * kKvPanel;
    static constexpr int kPPanel = kN * 128;              // 16 rows x 64 keys
    static constexpr int kPBuf = (kBN / 64) * kPPanel;    // one P^T tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = 4096;
    static constexpr int kOffV = kOffK + NSK * kKvBytes;
    static constexpr int kOffP = kOffV + NSV * kKvBytes;  // two P^T buffers
    static constexpr int kOffBar = kOffP + 2 * kPBuf;
    // q_full, k_full[NSK], v_full[NSV], k_empty[NSK], v_empty[NSV], s_full[2],
    // p_full[2], o_done[2], drain[2]
    static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 8;
    static constexpr int kOffRed = kOffBar + kNumBars * 8;    // maxima [2][4][16] fp32
    static constexpr int kOffSum = kOffRed + 2 * 4 * kN * 4;  // row sums [4][16] fp32
    static constexpr int kOffMask = kOffSum + 4 * kN * 4;     // key masks [2][4] words
    static constexpr int kOffMisc = kOffMask + 2 * 4 * 4;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static constexpr int kTmemS = 0;    // S^T buffers: columns [0, 16) and [16, 32)
    static constexpr int kTmemO = 32;   // O^T: columns [32, 48)
    static constexpr uint32_t kTmemCols = 64;
    static_assert(kQBytes <= kOffK, "Q tile");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// The cache row (2-D view [num_blocks * b * H_k, d]) of listed key j, or -1
// when j is not a key of the sequence or its block id is out of range.
__device__ __forceinline__ int32_t cache_row(const FwdParams& p, const int32_t* bt, int j, int sk,
                                             int hkv, bool& bad_block) {
    if (j < 0 || j >= sk) return -1;
    const int32_t blk = __ldg(bt + j / p.b);
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        bad_block = true;
        return -1;
    }
    return (int32_t)(((int64_t)blk * p.b + j % p.b) * p.hk + hkv);
}

// NR: rows the softmax threads track (4, 8 or 16 >= g); the MMAs always run
// N = 16 and ignore the padding columns.
template <int NSK, int NSV, int NR, bool PLAIN>
__global__ void __launch_bounds__(kThreads, 2)   // two CTAs per SM
topk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = TCfg<NSK, NSV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t token = blockIdx.x;
    const int hkv = blockIdx.y;
    const int seg = blockIdx.z;
    const bool split = p.splits > 1;
    const int g = p.g;
    const int nrows = g;

    // Owning sequence: the last s with cu_seqlens_q[s] <= token.
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(p.cu_seqlens_q + mid) <= token) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    int sq, sk;
    int64_t q0;
    uint32_t st = seq_status(p, s, sq, sk, q0);
    if (st && token == q0 && hkv == 0 && seg == 0 && threadIdx.x == 0) atomicOr(p.err, (int)st);
    if (st & UA_DEVERR_CU_SEQLENS) return;
    if (token < q0 || token >= q0 + sq) return;   // a row outside every sequence
    const int len = topk_length(p, token);
    if (len < 0) {
        if (hkv == 0 && seg == 0 && threadIdx.x == 0) atomicOr(p.err, (int)UA_DEVERR_BOUNDS);
        st |= UA_DEVERR_BOUNDS;
    }
    if (seg >= (split ? topk_segments(p, st, token) : 1)) return;
    const int i = (int)(token - q0);
    const int ctx = sk - sq;
    const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
    const bool window = (p.flags & UA_FLAG_WINDOW) != 0;
    const int e_beg = split ? seg * p.chunk : 0;
    const int e_end = split ? min(len, e_beg + p.chunk) : len;
    if (st || e_beg >= e_end) {
        // A malformed sequence or list (rows written as zeros), or an empty
        // list (no key, no value: O = 0; split: an empty partial, m = -inf).
        for (int e = threadIdx.x; e < nrows * kD; e += kThreads) {
            const int r = e / kD, c = e % kD;
            const int64_t row = token * p.hq + hkv * g + r;
            if (split) {
                if (c == 0) {
                    p.part_ml[(row * p.splits + seg) * 2 + 0] = -INFINITY;
                    p.part_ml[(row * p.splits + seg) * 2 + 1] = 0.f;
                }
            } else {
                p.out[row * kD + c] = __float2bfloat16_rn(0.f);
            }
        }
        return;
    }
    const int n_tiles = (e_end - e_beg + kBN - 1) / kBN;
    const int32_t* lst = p.topk_idx + token * p.topk_stride;
    const int32_t* bt = p.block_table + (int64_t)s * p.bt_stride;

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
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    float* lsum = reinterpret_cast<float*>(smem + C::kOffSum);
    uint32_t* kmask = reinterpret_cast<uint32_t*>(smem + C::kOffMask);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int k = 0; k < NSK; ++k) {
            mbar_init(k_full0 + 8 * k, 1);
            mbar_init(k_empty0 + 8 * k, 1);
        }
        for (int k = 0; k < NSV; ++k) {
            mbar_init(v_full0 + 8 * k, 1);
            mbar_init(v_empty0 + 8 * k, 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(s_full0 + 8 * k, 1);
            mbar_init(p_full0 + 8 * k, 128);
            mbar_init(o_done0 + 8 * k, 1);
        }
        mbar_init(drain, 1);
        mbar_init(drain + 8, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
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

    if ((UA_TOPK_K_LSU && warp == kWarpTma) || (UA_TOPK_V_LSU && warp == kWarpLdV)) {
        // ------------------------------ row loaders ------------------------------
        // Warp 4 copies the K tiles (and loads Q), warp 7 the V tiles.  Lane l
        // maps list entries 4l .. 4l+3 of a tile to cache rows (one tile ahead);
        // warp instruction n then moves rows n and n + 64: lanes 0-15 copy the
        // sixteen 16-byte chunks of row n, lanes 16-31 those of row n + 64, into
        // the 128-byte-swizzled panels the MMA reads.  Rows of entries that are
        // not keys of the sequence are skipped (K: their scores are masked) or
        // zeroed (V: their weight is 0, and 0 times stale data could be NaN).
        const bool is_k = warp == kWarpTma;
        if (is_k && lane == 0) {
            tma_prefetch_desc(&tm_q);
            mbar_arrive_expect_tx(q_full, (uint32_t)g * 128u * C::kPanels);   // the token's g rows
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_3d(sQ + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, (int)token, q_full);
        }
        const char* cache = static_cast<const char*>(is_k ? p.k_cache : p.v_cache);
        const uint32_t ring = is_k ? sK : sV;
        const uint32_t full0 = is_k ? k_full0 : v_full0;
        const uint32_t empty0 = is_k ? k_empty0 : v_empty0;
        bool bad_block = false;
        auto tile_rows = [&](int j, int32_t (&rw)[4]) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = e_beg + j * kBN + 4 * lane + k;
                rw[k] = e < e_end ? cache_row(p, bt, __ldg(lst + e), sk, hkv, bad_block) : -1;
            }
        };
        const int half = lane >> 4;           // 0: row n, 1: row n + 64
        const int c = lane & 15;              // 16-byte chunk of the 256-byte row
        const uint32_t chunk_off = (uint32_t)(c >> 3) * C::kKvPanel;
        const int src_base = half * 16;       // lanes holding rows 64 .. 127
        int32_t nxt[4];
        tile_rows(0, nxt);
        const int nst = is_k ? NSK : NSV;
        for (int j = 0; j < n_tiles; ++j) {
            const int stg = j % nst;
            int32_t cur[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) cur[k] = nxt[k];
            if (j >= nst && !__all_sync(0xffffffffu, dwait(empty0 + 8 * stg, ((j / nst) + 1) & 1,
                                                           abort_flag, p.err)))
                break;
            const uint32_t dst0 = ring + stg * C::kKvBytes + chunk_off;
#pragma unroll 4
            for (int n4 = 0; n4 < 64; n4 += 4) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int n = n4 + k;             // rows n (owned by lane n/4) and n + 64
                    const int32_t row = __shfl_sync(0xffffffffu, cur[k], src_base + (n >> 2));
                    const int r = n + half * 64;
                    const uint32_t dst = dst0 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
                    if (row >= 0)
                        cp_async16(dst, cache + (int64_t)row * (kD * 2) + c * 16);
                    else if (!is_k)
                        st_shared_zero16(dst);
                }
            }
            // The next tile's rows (a list load, then a dependent block-table
            // load) are looked up while this tile's copies are in flight.
            if (j + 1 < n_tiles) tile_rows(j + 1, nxt);
            cp_async_wait_all();
            fence_proxy_async_smem();   // the MMAs read these rows through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(full0 + 8 * stg);
        }
        if (__any_sync(0xffffffffu, bad_block) && lane == 0) atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
        __syncwarp();
    } else if (warp == (UA_TOPK_K_LSU ? kWarpLdV : kWarpTma)) {
        // ------------------------------ gather producer ------------------------------
        // Lane l owns list entries 4l .. 4l+3 of each tile: it maps them to cache
        // rows (one tile ahead, so the list and block-table loads overlap the
        // current tile's waits) and issues one four-row gather per panel.
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        if (!UA_TOPK_K_LSU && lane == 0) {
            tma_prefetch_desc(&tm_q);
            mbar_arrive_expect_tx(q_full, (uint32_t)g * 128u * C::kPanels);   // the token's g rows
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_3d(sQ + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, (int)token, q_full);
        }
        bool bad_block = false;
        auto tile_rows = [&](int j, int32_t (&rw)[4]) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = e_beg + j * kBN + 4 * lane + k;
                const int32_t r = e < e_end ? cache_row(p, bt, __ldg(lst + e), sk, hkv, bad_block) : -1;
                rw[k] = r < 0 ? 0 : r;
            }
        };
        int32_t nxt[4];
        tile_rows(0, nxt);
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int stk = j % NSK, stv = j % NSV;
            int32_t cur[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) cur[k] = nxt[k];
            if (!UA_TOPK_K_LSU) {
                if (j >= NSK && !__all_sync(0xffffffffu, dwait(k_empty0 + 8 * stk, ((j / NSK) + 1) & 1,
                                                               abort_flag, p.err)))
                    break;
                if (lane == 0) mbar_arrive_expect_tx(k_full0 + 8 * stk, C::kKvBytes);
                __syncwarp();
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_gather4(sK + stk * C::kKvBytes + pn * C::kKvPanel + lane * 4 * 128, &tm_k,
                                pn * 64, cur[0], cur[1], cur[2], cur[3], k_full0 + 8 * stk);
            }
            if (!UA_TOPK_V_LSU) {
                if (j >= NSV && !__all_sync(0xffffffffu, dwait(v_empty0 + 8 * stv, ((j / NSV) + 1) & 1,
                                                               abort_flag, p.err)))
                    break;
                if (lane == 0) mbar_arrive_expect_tx(v_full0 + 8 * stv, C::kKvBytes);
                __syncwarp();
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_gather4(sV + stv * C::kKvBytes + pn * C::kKvPanel + lane * 4 * 128, &tm_v,
                                pn * 64, cur[0], cur[1], cur[2], cur[3], v_full0 + 8 * stv);
            }
            issued = j + 1;
            // The next tile's rows are looked up after this tile's gathers
            // are on their way (in-order issue would otherwise hold them).
            if (j + 1 < n_tiles) tile_rows(j + 1, nxt);
        }
        if (__any_sync(0xffffffffu, bad_block) && lane == 0) atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
        if (*abort_flag && lane == 0) {
            // Let every copy this warp issued land before the CTA ends.
            for (int j = max(0, issued - NSK); j < issued && !UA_TOPK_K_LSU; ++j)
                mbar_wait_bounded(k_full0 + 8 * (j % NSK), (j / NSK) & 1);
            for (int j = max(0, issued - NSV); j < issued && !UA_TOPK_V_LSU; ++j)
                mbar_wait_bounded(v_full0 + 8 * (j % NSV), (j / NSV) & 1);
        }
        __syncwarp();
    } else if (warp == kWarpMma || warp == kWarpPv) {
        // ---------------------- MMA issuers (one thread each) ----------------------
        constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kBN, kN, false, false);
        constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kD, kN, true, false);
        auto wwait = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, dwait(bar, par, abort_flag, p.err));
        };
        if (warp == kWarpMma) {
            bool ok = wwait(q_full, 0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                // S^T buffer (j & 1) is free once P of tile j - 2 is published.
                if (j >= 2 && !wwait(p_full0 + 8 * (j & 1), ((j - 2) >> 1) & 1)) break;
                const int stg = j % NSK;
                if (!wwait(k_full0 + 8 * stg, (j / NSK) & 1)) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t kst = sK + stg * C::kKvBytes;
                    const uint32_t dS = tmem + C::kTmemS + (j & 1) * kN;
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {
                        const int pn = k >> 2, off = (k & 3) * 32;
                        const uint64_t bq = tc::smem_desc_sw128(sQ + pn * C::kQPanel + off, 16, 1024);
                        const uint64_t a = tc::smem_desc_sw128(kst + pn * C::kKvPanel + off, 16, 1024);
                        tc::mma_bf16(dS, a, bq, idesc_qk, k > 0 ? 1u : 0u);
                    }
                    tc::commit(s_full0 + 8 * (j & 1));
                    tc::commit(k_empty0 + 8 * stg);
                }
                __syncwarp();
            }
        } else {
            for (int j = 0; j < n_tiles; ++j) {
                const int stg = j % NSV;
                if (!wwait(p_full0 + 8 * (j & 1), (j >> 1) & 1)) break;
                if (!wwait(v_full0 + 8 * stg, (j / NSV) & 1)) break;
                tc::fence_after_sync();
                // V rows of entries that are not keys of the row become zeros
                // (their weight is 0, but 0 times a NaN in the gathered row is NaN).
                const uint32_t* mk = kmask + (j & 1) * 4;
                const uint32_t full = mk[0] & mk[1] & mk[2] & mk[3];
                if (!UA_TOPK_V_LSU && full != 0xffffffffu) {
                    uint8_t* vst = smem + C::kOffV + stg * C::kKvBytes;
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {
                        if ((mk[q] >> lane) & 1u) continue;
                        const int row = q * 32 + lane;
#pragma unroll
                        for (int pn = 0; pn < C::kPanels; ++pn) {
                            uint4* dst = reinterpret_cast<uint4*>(vst + pn * C::kKvPanel + row * 128);
#pragma unroll
                            for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    const uint32_t vst = sV + stg * C::kKvBytes;
                    const uint32_t pbuf = sP + (j & 1) * C::kPBuf;
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint64_t a = tc::smem_desc_sw128(vst + kk * 16 * 128, C::kKvPanel, 1024);
                        const uint64_t bp =
                            tc::smem_desc_sw128(pbuf + (kk >> 2) * C::kPPanel + (kk & 3) * 32, 16, 1024);
                        tc::mma_bf16(tmem + C::kTmemO, a, bp, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::commit(o_done0 + 8 * (j & 1));
                    tc::commit(v_empty0 + 8 * stg);
                }
                __syncwarp();
            }
        }
        if (*abort_flag) {
            // No MMA this thread issued may still run when tensor memory is freed.
            const uint32_t dr = drain + 8 * (warp - kWarpMma);
            if (lane == 0) tc::commit(dr);
            __syncwarp();
            mbar_wait_bounded(dr, 0);
        }
    } else {
        // --------------------------- softmax warps 0-3 ----------------------------
        // Thread t: list entry t of each tile (S^T lane t) and head-dim element t
        // of the output (O^T lane t).  Every row of the CTA is the same query
        // token, so an entry is a key of all rows or of none.
        const int t = threadIdx.x;
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        const bool softcap = (p.flags & UA_FLAG_SOFTCAP) != 0;
        const bool alibi = (p.flags & UA_FLAG_ALIBI) != 0;
        const float* qrow = (p.flags & UA_FLAG_QQ_BIAS) ? p.qq_bias + (int64_t)i * p.qq_stride : nullptr;
        const float sl2 = p.scale * kLog2e;
        const int khi = causal ? i + ctx : sk - 1;                 // last visible position
        const int klo = window ? i + ctx - p.window + 1 : 0;       // first visible position
        float m[NR], l[NR], rslope[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
            rslope[r] = (!PLAIN && alibi && r < nrows) ? __ldg(p.alibi + hkv * g + r) : 0.f;
        }
        bool ok = true;
        // The entry's listed position and whether it is a key of the row, one
        // tile ahead: looked up after P of the previous tile is published, so
        // the two dependent loads overlap the wait for the next S.
        auto lookup = [&](int j, int& jp, bool& valid) {
            const int e = e_beg + j * kBN + t;
            jp = -1;
            valid = false;
            if (e < e_end) {
                jp = __ldg(lst + e);
                bool bad = false;
                valid = cache_row(p, bt, jp, sk, hkv, bad) >= 0 && jp <= khi && jp >= klo;
            }
        };
        int jp_next;
        bool valid_next;
        lookup(0, jp_next, valid_next);
        for (int j = 0; j < n_tiles; ++j) {
            const int jp = jp_next;
            const bool valid = valid_next;
            const bool got = __all_sync(0xffffffffu, dwait(s_full0 + 8 * (j & 1), (j >> 1) & 1,
                                                           abort_flag, p.err));
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
                        float tt = __uint_as_float(sv[r]) * p.scale;
                        if (softcap) tt = p.softcap * tanh_from_exp2(tt / p.softcap);
                        if (alibi) tt += rslope[r] * (float)(jp - ctx);
                        if (qrow && valid && jp >= ctx) tt += __ldg(qrow + (jp - ctx));
                        v = tt * kLog2e;
                    }
                    x[r] = (valid && r < nrows) ? v : -INFINITY;
                }
            } else {
#pragma unroll
                for (int r = 0; r < NR; ++r) x[r] = -INFINITY;
            }
            // Per-row maxima over this warp's 32 entries, then over the 4 warps.
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r < nrows) {
                    const float w = warp_max_f32(x[r]);
                    if (lane == 0) red[((j & 1) * 4 + warp) * kN + r] = w;
                }
            }
            const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
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
                    if (tmax > m[r] + kLazy) {
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
                uint32_t h, ex;
                asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(a1), "f"(a0));
                asm("ex2.approx.f16x2 %0, %1;" : "=r"(ex) : "r"(h));
                float p0, p1;
                asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\t"
                    "cvt.f32.f16 %1, hi;\n\t}"
                    : "=f"(p0), "=f"(p1)
                    : "r"(ex));
                l[r] = l[r] * alpha[r] + p0;
                l[r + 1] = l[r + 1] * alpha[r + 1] + p1;
                pb[r / 2] = pack_bf16x2(p0, p1);
            }
            // P^T buffer (j & 1) and mask (j & 1) were read by the P.V of tile
            // j - 2; rescaling O needs the P.V of tile j - 1.
            bool go = true;
            if (j >= 2)
                go = __all_sync(0xffffffffu, dwait(o_done0 + 8 * (j & 1), ((j - 2) >> 1) & 1,
                                                   abort_flag, p.err));
            if (go && any_re && j > 0) {
                go = __all_sync(0xffffffffu, dwait(o_done0 + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1,
                                                   abort_flag, p.err));
                if (go) {
                    tc::fence_after_sync();
                    uint32_t o[kN];
                    ld16(tl + C::kTmemO, o);
                    tc::wait_ld();
#pragma unroll
                    for (int r = 0; r < NR; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
                    st16(tl + C::kTmemO, o);
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
                if (lane == 0) kmask[(j & 1) * 4 + warp] = vmask;
                fence_proxy_async_smem();
                tc::fence_before_sync();
                mbar_arrive(p_full0 + 8 * (j & 1));
            }
            if (j + 1 < n_tiles) lookup(j + 1, jp_next, valid_next);
        }
        // ------------------------------ epilogue ---------------------------------
        if (ok) {
            const bool done = __all_sync(0xffffffffu,
                                         dwait(o_done0 + 8 * ((n_tiles - 1) & 1),
                                               ((n_tiles - 1) >> 1) & 1, abort_flag, p.err));
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
                uint32_t o[kN];
                ld16(tl + C::kTmemO, o);
                tc::wait_ld();
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r >= nrows) continue;
                    const float L0 = lsum[r] + lsum[kN + r] + lsum[2 * kN + r] + lsum[3 * kN + r];
                    const int64_t row = token * p.hq + hkv * g + r;
                    const float ov = __uint_as_float(o[r]);
                    if (split) {
                        part_store(p, (row * p.splits + seg) * kD + t, ov);
                        if (t == 0) {
                            p.part_ml[(row * p.splits + seg) * 2 + 0] = m[r];
                            p.part_ml[(row * p.splits + seg) * 2 + 1] = L0;
                        }
                    } else {
                        float num = 1.f, L = L0;
                        bool zero = false;
                        if (p.flags & UA_FLAG_SINKS) {
                            const float s2 = __ldg(p.sinks + hkv * g + r) * kLog2e;
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
                        p.out[row * kD + t] = __float2bfloat16_rn(ov * inv);
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int NSK, int NSV>
cudaError_t launch_topk_t(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                          const FwdParams& p, const TopkPlan& plan, cudaStream_t stream) {
    using C = TCfg<NSK, NSV>;
    const bool plain = (p.flags & (UA_FLAG_SOFTCAP | UA_FLAG_ALIBI | UA_FLAG_QQ_BIAS)) == 0;
    auto kern = p.g <= 4 ? (plain ? topk_kernel<NSK, NSV, 4, true> : topk_kernel<NSK, NSV, 4, false>)
              : p.g <= 8 ? (plain ? topk_kernel<NSK, NSV, 8, true> : topk_kernel<NSK, NSV, 8, false>)
                         : (plain ? topk_kernel<NSK, NSV, 16, true> : topk_kernel<NSK, NSV, 16, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)p.total_q, (unsigned)p.hk, (unsigned)plan.splits);
    kern<<<grid, kThreads, C::kSmem, stream>>>(tq, tm_k, tm_v, p);
    return cudaGetLastError();
}

}  // namespace

bool topk_shape_ok(const FwdParams& p) {
    return p.d == kD && p.g >= 1 && p.g <= kN && p.topk_stride >= 1 &&
           p.total_q <= 0x7fffffffLL;
}

bool encode_gather_map(CUtensorMap* m, const void* cache, int64_t num_blocks, int b, int hk, int d) {
    // [num_blocks * b * H_k rows, d columns] (bf16), box = 64 columns x 1 row.
    const int64_t rows = num_blocks * b * hk;
    if (rows > 0x7fffffffLL) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {2ull * d};
    cuuint32_t box[2] = {64, 1};
    return encode_bf16_sw128(m, cache, 2, dims, strides, box);
}

void plan_topk(const FwdParams& p, int num_sms, size_t workspace_bytes, TopkPlan* plan) {
    *plan = TopkPlan();
    // Segments of whole 128-entry tiles, at least UA_TOPK_MIN_TILES each,
    // and no more CTAs than one wave of the two an SM holds: every extra
    // segment refills a pipeline and adds a combine.  Measured on 256
    // tokens x 2048 entries: one segment per token 3.26 TB/s, two 2.71.
    const int64_t base = (int64_t)p.hk * p.total_q;
    const int64_t want = std::max<int64_t>(1, (2LL * num_sms) / base);
    const int64_t by_len = std::max<int64_t>(1, p.topk_stride / (UA_TOPK_MIN_TILES * kBN));
    int splits = (int)std::min<int64_t>(std::min<int64_t>(want, by_len), 64);
    const size_t per_split = (size_t)p.total_q * p.hq * (p.d + 2) * sizeof(float);
    splits = (int)std::min<size_t>((size_t)splits, per_split ? workspace_bytes / per_split : 1);
    if (splits < 1) splits = 1;
    if (splits > 1) {
        const int per = (p.topk_stride + splits - 1) / splits;
        plan->chunk = (per + kBN - 1) / kBN * kBN;
        splits = (p.topk_stride + plan->chunk - 1) / plan->chunk;
    }
    plan->splits = splits;
    plan->launches = splits > 1 ? 2 : 1;
}

cudaError_t launch_topk(const TopkPlan& plan, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                        const FwdParams& p, cudaStream_t stream) {
    // Q map: [total_q, H_q, d]; box = 64 dims x g heads x 1 position (the
    // token's g rows; the other rows of the 16-row tile are padding that the
    // MMAs compute and nobody reads).
    CUtensorMap tq;
    cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.hq, (cuuint64_t)p.total_q};
    cuuint64_t strides[2] = {2ull * p.d, 2ull * p.d * p.hq};
    cuuint32_t box[3] = {64, (cuuint32_t)p.g, 1};
    if (!encode_bf16_sw128(&tq, p.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    return launch_topk_t<UA_TOPK_NSK, UA_TOPK_NSV>(tq, tm_k, tm_v, p, plan, stream);
}

}  // namespace ua
