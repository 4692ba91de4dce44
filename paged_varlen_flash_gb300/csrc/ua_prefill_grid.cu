// ua_prefill_grid.cu -- prefill attention for head sizes 64 and 128 on the
// tcgen05 tensor cores of sm_103a, one CTA per work unit over a dense grid:
// the form the planner picks when the batch's padded grid is nearly all real
// units and fills the GPU at least twice (a long prefill, equal-length
// sequences).  Ragged batches go to the persistent kernel of
// ua_prefill_pair.cu instead; the two share the unit, the roles and the math.
// Measured on the long causal prefill (8,192 x 8,192, 128/8 heads): 1.87 ms
// here against 2.06 ms for the persistent form, while the persistent form
// takes the chunked batch in 0.137 ms against 0.171 ms here.
//
// Work unit: one CTA per (pair of tiles of 128 packed (position, head) rows of
// one KV head, sequence[, KV segment]).  Tile A holds the earlier positions,
// tile B the next ones; the g query heads sharing the KV head are packed into
// the rows (gfx950 "Unified paged attention on gfx950, from the math up",
// section 4; floor(128 / g) positions per tile).  CTAs go out heaviest tile
// pair first with the KV heads of one pair adjacent.  Both tiles consume
// every K and V tile the CTA loads, so a paged K/V tile crosses the TMA unit
// once per 256 query rows -- on this cache layout (one 128-byte TMA row per
// key and 64-dim panel) the copy engine, not the tensor cores, is what a
// 128-row tile runs out of first.
//
// The math is the streaming (m, l, o) recurrence of gfx1151 ALGORITHM.md
// section 3 in base 2 (gfx950 section 2) with the lazy re-anchor threshold of
// 8, the mask-free / masked tile split and the causal early exit of
// attention_dense.py (gfx950 section 8.1), per tile.
//
// Roles (12 warps):
//   warps 0-3  softmax + epilogue of tile A, warps 4-7 of tile B: thread r
//              owns row r (tensor-memory lane r) and all 128 key columns of
//              each S tile, so the two warpgroups never wait for each other;
//   warp 8     TMA producer: Q_A and Q_B once, then K and V tiles through NK-
//              and NV-stage rings (one box per paged block and 64-wide
//              head-dim panel, one lane per block);
//   warp 9     MMA issuer of tile A (also owns tensor memory);
//   warp 10    MMA issuer of tile B;
//   warp 11    idle (completes the third warpgroup for register reallocation).
//
// Tensor memory (512 columns): S_A [0, 128), S_B [128, 256),
// O_A [256, 256 + D), O_B [256 + D, 256 + 2D).  P_X (bf16, two keys per
// column) is written over the first 64 columns of S_X once S_X has been read;
// the next QK^T into S_X is issued right behind the P.V that reads it, by the
// same thread.
//
// Schedule: each warpgroup runs its own chain S_x(j) -> softmax -> P_x(j) ->
// P.V -> S_x(j + 1); the two chains settle half a step apart, so while one
// warpgroup works on its scores the tensor cores run the other tile's P.V and
// next QK^T.
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "ua_common.cuh"
#include "ua_prefill.h"
#include "ua_prefill_common.cuh"
#include "ua_ptx.cuh"
#include "ua_tc.cuh"

namespace ua {
namespace {

using namespace pf;

constexpr int kBN = 128;   // keys per K/V tile (the QK^T MMA's N)

template <int D, int NK, int NV>
struct GridCfg {
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kRows * 128;        // 128 rows x 64 dims
    static constexpr int kQTile = kPanels * kQPanel;
    static constexpr int kKvPanel = kBN * 128;
    static constexpr int kKvBytes = kPanels * kKvPanel;
    static constexpr int kOffQ = 0;                     // Q_A then Q_B
    static constexpr int kOffK = kOffQ + 2 * kQTile;
    static constexpr int kOffV = kOffK + NK * kKvBytes;
    static constexpr int kOffBar = kOffV + NV * kKvBytes;
    // q_full, k_full[NK], v_full[NV], k_empty[NK], v_empty[NV], s_full[2],
    // p_full[2], o_done[2] (once, after a tile's last P.V), drain[2] (the
    // last four indexed by tile)
    static constexpr int kNumBars = 1 + 2 * NK + 2 * NV + 9;   // + never (testing hook)
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static constexpr int kTmemO = 2 * kBN;
    static_assert(2 * kBN + 2 * D <= (int)kTmemCols, "tensor memory budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// Two softmax warpgroups (one per tile), then a third warpgroup of the TMA
// warp, the two MMA-issuing warps and one idle warp (register reallocation
// works on whole warpgroups).
struct GR {
    static constexpr int kThreads = 384;
    static constexpr int kWarpTma = 8;
    static constexpr int kWarpMma = 9;    // MMA issuer of tile A, tensor-memory owner
    static constexpr int kWarpPv = 10;    // MMA issuer of tile B
    // Registers per thread after the split: 2 x 128 x 224 + 128 x 56 equals
    // the 384 x 168 the block is launched with.
    static constexpr uint32_t kRegsSoftmax = 224;
    static constexpr uint32_t kRegsOther = 56;
};

// QQ: the query-query bias pass is compiled in (a separate instantiation, so
// that the score loop of the other non-plain calls keeps its registers).
template <int D, int NK, int NV, bool PLAIN, bool QQ>
__global__ void __launch_bounds__(GR::kThreads, 1)
prefill_grid_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
    using C = GridCfg<D, NK, NV>;
    using R = GR;
    constexpr int kThreads = R::kThreads;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.z;
    const bool split = p.splits > 1;             // write (m, l, o) partials per KV segment
    // Launch order (x fastest, then y) -> heaviest tile pair first, the KV
    // heads of one pair (and its segments) adjacent.
    const int lin = (int)(blockIdx.y * gridDim.x + blockIdx.x);
    const int seg = lin % p.splits;
    const int hkv = (lin / p.splits) % p.hk;
    const int pairs = (int)(gridDim.x / p.splits);
    const int qp = pairs - 1 - lin / (p.splits * p.hk);
    const int g = p.g;
    const int ppt = kRows / g;                  // positions per tile
    const int p0 = qp * 2 * ppt;                // first position of tile A

    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, s, sq, sk, q0);
    if (st && qp == 0 && hkv == 0 && seg == 0 && threadIdx.x == 0) atomicOr(p.err, (int)st);
    if (st & UA_DEVERR_CU_SEQLENS) return;
    if (p0 >= sq) return;
    if (seg >= (split ? seq_segments(p, st, sk) : 1)) return;
    const bool has_b = p0 + ppt < sq;
    const int last_a = min(p0 + ppt, sq) - 1;
    const int last_b = has_b ? min(p0 + 2 * ppt, sq) - 1 : last_a;
    const int ctx = sk - sq;
    const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
    const bool window = (p.flags & UA_FLAG_WINDOW) != 0;
    int k_beg = window ? max(0, p0 + ctx - p.window + 1) : 0;
    int kend_a = causal ? min(sk, last_a + ctx + 1) : sk;
    int kend_b = causal ? min(sk, last_b + ctx + 1) : sk;
    if (split) {  // this CTA's KV segment; segments are whole tiles
        k_beg = max(k_beg, seg * p.chunk);
        kend_a = min(kend_a, seg * p.chunk + p.chunk);
        kend_b = min(kend_b, seg * p.chunk + p.chunk);
    }
    const int k_end = has_b ? kend_b : kend_a;
    if (st || k_beg >= k_end) {
        // Malformed lengths (rows written as zeros) or a segment with no
        // visible key for any row of either tile (an empty partial, m = -inf).
        for (int e = threadIdx.x; e < 2 * kRows * (D / 8); e += kThreads) {
            const int rr = e / (D / 8), c = e % (D / 8);
            const int x = rr / kRows, r = rr % kRows;
            const int i = p0 + x * ppt + r / g;
            if (i > (x ? last_b : last_a) || (x && !has_b)) continue;
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
    const int t_begin = k_beg / kBN;
    // Key tiles per query tile: A stops where its causal range (or the
    // segment) ends; B covers every tile.
    const int n_a = kend_a > k_beg ? (kend_a + kBN - 1) / kBN - t_begin : 0;
    const int n_b = has_b ? (kend_b + kBN - 1) / kBN - t_begin : 0;
    const int n_tiles = max(n_a, n_b);

    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    const uint32_t q_full = smem_u32(&bar_mem[0]);
    const uint32_t k_full0 = smem_u32(&bar_mem[1]);
    const uint32_t v_full0 = smem_u32(&bar_mem[1 + NK]);
    // A K stage is free once both tiles' QK^T ran, a V stage once both P.V ran.
    const uint32_t k_empty0 = smem_u32(&bar_mem[1 + NK + NV]);
    const uint32_t v_empty0 = smem_u32(&bar_mem[1 + 2 * NK + NV]);
    constexpr int kBarT = 1 + 2 * NK + 2 * NV;
    const uint32_t s_full0 = smem_u32(&bar_mem[kBarT]);       // + 8 * tile
    const uint32_t p_full0 = smem_u32(&bar_mem[kBarT + 2]);
    const uint32_t o_done0 = smem_u32(&bar_mem[kBarT + 4]);
    const uint32_t drain0 = smem_u32(&bar_mem[kBarT + 6]);
    const uint32_t never = smem_u32(&bar_mem[kBarT + 8]);   // the testing hook's stall
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < NK; ++i) {
            mbar_init(k_full0 + 8 * i, 1);
            mbar_init(k_empty0 + 8 * i, 2);   // one arrival per tile reading the stage
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(v_full0 + 8 * i, 1);
            mbar_init(v_empty0 + 8 * i, 2);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full0 + 8 * x, 1);
            mbar_init(p_full0 + 8 * x, kRows);   // tile x's warpgroup
            mbar_init(o_done0 + 8 * x, 1);
            mbar_init(drain0 + 8 * x, 1);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == R::kWarpMma) {
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

    if (warp >= 8) {
    // Registers move from this warpgroup (copies, MMA issue, one idle warp) to
    // the softmax warps, which hold a whole 128-key row of scores each.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(GR::kRegsOther));
    if (warp == R::kWarpTma) {
        // ------------------------------ TMA producer ------------------------------
        // Lane i owns paged block i of each KV tile (its id load and its TMA
        // boxes), so one tile's boxes go out in parallel.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            // One box per panel and tile: g heads x ppt positions = g * ppt
            // rows (128 when g divides 128; the rows past them are padding
            // whose outputs are never stored).
            mbar_arrive_expect_tx(q_full, (has_b ? 2u : 1u) * (uint32_t)(g * ppt) * 128u * C::kPanels);
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn) {
                tma_load_3d(sQ + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, (int)(q0 + p0), q_full);
                if (has_b)
                    tma_load_3d(sQ + C::kQTile + pn * C::kQPanel, &tm_q, pn * 64, hkv * g,
                                (int)(q0 + p0 + ppt), q_full);
            }
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
            const int stk = j % NK, stv = j % NV;
            const int blk0 = (t_begin + j) * kBN / b;
            const int nb = min(kBN / b, nblk_seq - blk0);
            const uint32_t bytes = (uint32_t)nb * b * 128 * C::kPanels;
            const int32_t id = id_next;
            if (j + 1 < n_tiles) id_next = tile_id(j + 1);
            if (lane < nb && (id < 0 || (int64_t)id >= p.num_blocks))
                atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
            if (j >= NK && !__all_sync(0xffffffffu, wait_or_abort(k_empty0 + 8 * stk, ((j / NK) + 1) & 1,
                                                                   abort_flag, p.err)))
                break;
            if (lane == 0) mbar_arrive_expect_tx(k_full0 + 8 * stk, bytes);
            __syncwarp();
            if (lane < nb) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_4d(sK + stk * C::kKvBytes + pn * C::kKvPanel + lane * b * 128, &tm_k,
                                pn * 64, hkv, 0, id, k_full0 + 8 * stk);
            }
            if (j >= NV && !__all_sync(0xffffffffu, wait_or_abort(v_empty0 + 8 * stv, ((j / NV) + 1) & 1,
                                                                   abort_flag, p.err)))
                break;
            if (lane == 0) mbar_arrive_expect_tx(v_full0 + 8 * stv, bytes);
            __syncwarp();
            if (lane < nb) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_4d(sV + stv * C::kKvBytes + pn * C::kKvPanel + lane * b * 128, &tm_v,
                                pn * 64, hkv, 0, id, v_full0 + 8 * stv);
            }
            issued = j + 1;
        }
        if (*abort_flag && lane == 0) {
            // Let every copy this warp issued land before the CTA ends.
            for (int j = max(0, issued - NK); j < issued; ++j)
                mbar_wait_bounded(k_full0 + 8 * (j % NK), (j / NK) & 1);
            for (int j = max(0, issued - NV); j < issued; ++j)
                mbar_wait_bounded(v_full0 + 8 * (j % NV), (j / NV) & 1);
        }
        __syncwarp();
    } else if (warp == R::kWarpMma || warp == R::kWarpPv) {
        // ---------------------- MMA issuers (one thread each) ----------------------
        // Warp kWarpMma issues for tile A, kWarpPv for tile B, so the two
        // tiles' chains never queue behind each other's waits.  Per key tile
        // j the issuer of tile x waits for P_x(j) and V(j), issues
        // O_x += P_x(j) V(j), then (K(j + 1) landed) S_x = Q_x K(j + 1)^T right
        // behind it: MMAs from one thread run in issue order, so the QK^T that
        // overwrites the columns holding P_x cannot overtake the P.V reading
        // them, and the issuer never blocks on its own MMAs (each such wait
        // would leave the tensor pipe idle).  A stage is released by two
        // arrivals, one per tile that reads it; a tile only one of them reads
        // gets both from that tile's issuer.
        constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, kBN, false, false);
        constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kRows, D, false, true);
        auto wwait = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_or_abort(bar, par, abort_flag, p.err));
        };
        const int x = warp - R::kWarpMma;
        const int nx = x ? n_b : n_a;
        const int n_other = x ? n_a : n_b;
        const uint32_t dS = tmem + x * kBN;
        const uint32_t dO = tmem + C::kTmemO + x * D;
        const uint32_t qst = sQ + x * C::kQTile;
        auto issue_qk = [&](int j) -> bool {
            const int stg = j % NK;
            // Testing hook: the first K wait waits on a barrier that nothing
            // completes and gives up after stall_ns.
            if (p.stall && j == 0 &&
                !__all_sync(0xffffffffu, wait_or_abort(never, 0, abort_flag, p.err, (uint64_t)p.stall_ns)))
                return false;
            if (!wwait(k_full0 + 8 * stg, (j / NK) & 1)) return false;
            tc::fence_after_sync();
            if (lane == 0) {
                const uint32_t kst = sK + stg * C::kKvBytes;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const int pn = k >> 2, off = (k & 3) * 32;
                    const uint64_t a = tc::smem_desc_sw128(qst + pn * C::kQPanel + off, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(kst + pn * C::kKvPanel + off, 16, 1024);
                    tc::mma_bf16(dS, a, bd, idesc_qk, k > 0 ? 1u : 0u);
                }
                tc::commit(s_full0 + 8 * x);
                tc::commit(k_empty0 + 8 * stg);
                if (j >= n_other) tc::commit(k_empty0 + 8 * stg);
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        if (nx > 0) ok = wwait(q_full, 0) && issue_qk(0);
        for (int j = 0; ok && j < nx; ++j) {
            const int stg = j % NV;
            if (!(ok = wwait(p_full0 + 8 * x, j & 1))) break;
            if (!(ok = wwait(v_full0 + 8 * stg, (j / NV) & 1))) break;
            tc::fence_after_sync();
            const uint32_t vst = sV + stg * C::kKvBytes;
            const int key0 = (t_begin + j) * kBN;
            const int nvalid = min(kBN, sk - key0);
            if (nvalid < kBN) {
                // Keys past S_k: whatever those slots hold must not reach O
                // (0 * NaN is NaN), so their V rows become zeros.  (Both
                // issuers may clear the same rows; each clears before its own
                // P.V and only zeros are ever written there.)
                uint8_t* vgen = smem + C::kOffV + stg * C::kKvBytes;
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
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k) {
                    // A = P_x from tensor memory: 16 keys per MMA = 8 columns.
                    const uint64_t bd = tc::smem_desc_sw128(vst + k * 16 * 128, C::kKvPanel, 1024);
                    tc::mma_bf16_ts(dO, dS + k * 8, bd, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
                }
                tc::commit(v_empty0 + 8 * stg);
                if (j >= n_other) tc::commit(v_empty0 + 8 * stg);
                if (j + 1 == nx) tc::commit(o_done0 + 8 * x);
            }
            __syncwarp();
            if (j + 1 < nx) ok = issue_qk(j + 1);
        }
        if (*abort_flag) {
            // No MMA this thread issued may still run when tensor memory is freed.
            const uint32_t dr = drain0 + 8 * x;
            if (lane == 0) tc::commit(dr);
            __syncwarp();
            mbar_wait_bounded(dr, 0);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(GR::kRegsSoftmax));
        // ------------------------- softmax + epilogue warps -----------------------
        // Warpgroup x owns tile x: thread r holds row r (tensor-memory lane r)
        // and all 128 key columns of each S_x tile, so a row's max and sum
        // need no exchange and the two warpgroups never wait for each other.
        const int x = threadIdx.x >> 7;
        const int r = threadIdx.x & (kRows - 1);
        const int head = hkv * g + r % g;
        const bool softcap = (p.flags & UA_FLAG_SOFTCAP) != 0;
        const bool alibi = (p.flags & UA_FLAG_ALIBI) != 0;
        const float sl2 = p.scale * kLog2e;
        const float slope = alibi ? __ldg(p.alibi + head) : 0.f;
        const float inv_cap = softcap ? 1.0f / p.softcap : 0.f;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = trow + x * kBN;
        const int first = p0 + x * ppt;
        const int last = x ? last_b : last_a;
        const int pos = first + r / g;
        const bool valid = (x == 0 || has_b) && pos <= last;
        const int hi = causal ? min(pos + ctx, sk - 1) : sk - 1;
        const int lo = window ? max(0, pos + ctx - p.window + 1) : 0;
        // The row's line of the query-query bias (none for padding rows).
        const float* qrow = (QQ && valid)
                                ? p.qq_bias + (int64_t)pos * p.qq_stride
                                : nullptr;
        // Keys every row of the tile sees: [kfree_lo, kfree_hi].
        const int kfree_hi = causal ? min(first + ctx, sk - 1) : sk - 1;
        const int kfree_lo = window ? max(0, last + ctx - p.window + 1) : 0;
        // Warps whose 32 rows are all padding skip the score work; they still
        // take part in every barrier.
        const bool live = __any_sync(0xffffffffu, valid);
        const int nx = x ? n_b : n_a;
        const uint32_t p_full = p_full0 + 8 * x;
        const uint32_t o_done = o_done0 + 8 * x;
        float m = -INFINITY;  // running max, log2 units
        float l = 0.f;        // running denominator
        bool ok = true;
        for (int j = 0; j < nx; ++j) {
            // Plain scores: take turns with the other warpgroup (A(j) after
            // B(j - 1), B(j) after A(j)), so each softmax has the
            // special-function pipe to itself while the tensor cores run the
            // other tile's MMAs, instead of both tiles computing, then both
            // waiting, in lockstep.  (With softcap / ALiBi the score work
            // outweighs the MMAs and the two warpgroups are better run side
            // by side.)
            const int turn = x == 0 ? j - 1 : j;          // the other tile's step to follow
            if (PLAIN && turn >= 0 && turn < (x == 0 ? n_b : n_a)) {
                if (!__all_sync(0xffffffffu, wait_or_abort(p_full0 + 8 * (1 - x), turn & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
            }
            if (!__all_sync(0xffffffffu, wait_or_abort(s_full0 + 8 * x, j & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            uint32_t sr[kBN / 32][32];
            const int key0 = (t_begin + j) * kBN;
            float tmax = -INFINITY;
            if (live) {
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) tc::ld32(s_col + c * 32, sr[c]);
                tc::wait_ld();
                const bool mask_free = key0 >= kfree_lo && key0 + kBN - 1 <= kfree_hi;
                if constexpr (!PLAIN) {
                    // ALiBi: one int -> float conversion per tile; the per-key
                    // offsets are compile-time constants.
                    const float abias = slope * (float)(key0 - ctx);
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c)
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
                    if (QQ && qrow != nullptr && key0 + kBN > ctx && key0 <= hi) {
#pragma unroll
                        for (int c = 0; c < kBN / 32; ++c)
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
                    for (int c = 0; c < kBN / 32; ++c)
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
                for (int c = 0; c < kBN / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 16)
#pragma unroll
                        for (int a = 0; a < 8; ++a)
                            mx[a] = fmax3(mx[a], __uint_as_float(sr[c][e + 2 * a]),
                                          __uint_as_float(sr[c][e + 2 * a + 1]));
                tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                if constexpr (PLAIN) tmax *= sl2;
            }
            // Lazy re-anchor: move the reference max only when the tile's max
            // exceeds it by more than 8 (log2), so P stays at most 2^8.
            float alpha = 1.f;
            const bool reanchor = tmax > m + kLazy;
            if (reanchor) {
                alpha = fast_exp2(m - tmax);
                m = tmax;
            }
            if (live) {
                const float m_use = (m == -INFINITY) ? 0.f : m;
                const float xs = PLAIN ? sl2 : 1.0f;
                // P = 2^(x - m): the exponent argument in fp32 (packed pairs),
                // the power of two on the fp32 special-function path (the
                // fp16x2 form gives the same results per clock but needs three
                // conversions per pair on the same pipe), row sums in fp32.  P goes
                // over the first 64 columns of S_x (lane r, two bf16 keys per
                // 32-bit column: the A operand of the P.V MMA); this thread has
                // already read all of its row's S.
                float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                const float2 sc2 = make_float2(xs, xs);
                const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 a = ffma2(make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])),
                                               sc2, nm2);
                        const float2 pr = exp2_pair_f32(a);
                        rs[(e >> 1) & 3] = fadd2(rs[(e >> 1) & 3], pr);
                        pk[e / 2] = pack_bf16x2(pr.x, pr.y);
                    }
                    tc::st16(s_col + c * 16, pk);
                }
                const float2 rs01 = fadd2(rs[0], rs[1]), rs23 = fadd2(rs[2], rs[3]);
                l = l * alpha + ((rs01.x + rs01.y) + (rs23.x + rs23.y));
                tc::wait_st();
            }
            if (live && j > 0 && __any_sync(0xffffffffu, reanchor)) {
                // Rescale O_x.  The P.V of tile j - 1 has finished: its issuer
                // issued it before this tile's QK^T, whose completion
                // (s_full, waited above) covers every MMA issued before it.
                {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        const uint32_t col = trow + C::kTmemO + x * D + c * 32;
                        tc::ld32(col, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st32(col, o);
                    }
                    tc::wait_st();
                }
            }
            tc::fence_before_sync();
            mbar_arrive(p_full);
        }
        // ------------------------------ epilogue ---------------------------------
        if (ok && nx > 0)
            ok = __all_sync(0xffffffffu, wait_or_abort(o_done, 0, abort_flag, p.err));   // after the last P.V
        if (ok && valid && split) {
            // Split partial: raw o (below), m in log2 units, l.
            const int64_t row = (q0 + pos) * p.hq + head;
            p.part_ml[(row * p.splits + seg) * 2 + 0] = nx > 0 ? m : -INFINITY;
            p.part_ml[(row * p.splits + seg) * 2 + 1] = nx > 0 ? l : 0.f;
        }
        // A tile whose rows are all valid goes out through shared memory --
        // its own Q buffer, free once its last QK^T has run, in the layout of
        // the map's boxes -- and one TMA store per 64-column panel: rows of a
        // tile lie H_q * d elements apart in the output, so per-thread row
        // stores touch one sector per lane.  A sequence's last tile, whose
        // padding rows must not be written, keeps the per-thread stores.
        const bool staged = !split && nx > 0 && (x == 0 || has_b) && last - first + 1 == ppt;
        uint8_t* stage = smem + C::kOffQ + x * C::kQTile;
        if (ok && live && nx > 0) {
            // tcgen05.ld is warp-collective: every lane of a live warp loads.
            tc::fence_after_sync();
            const int64_t row = (q0 + pos) * p.hq + head;
            const uint32_t ocol = trow + C::kTmemO + x * D;
            float inv = 0.f;
            if (!split) {
                float O_scale_num = 1.f;  // extra factor from the sink re-basing
                float L = l;
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
                inv = (!zero && L > 0.f) ? O_scale_num * __frcp_rn(L) : 0.f;
            }
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tc::ld32(ocol + c * 32, o);
                tc::wait_ld();
                if (!valid) continue;
                if (split) {
                    part_store32(p, (row * p.splits + seg) * D + c * 32, o);
                } else {
                    __nv_bfloat16* orow = p.out + row * (int64_t)D + c * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        if (staged) {
                            // panel c / 2, 16-byte chunk (c % 2) * 4 + e / 8 of
                            // row r, 128-byte swizzled
                            const int chunk = (c & 1) * 4 + e / 8;
                            *reinterpret_cast<uint4*>(stage + (c / 2) * C::kQPanel + r * 128 +
                                                      ((chunk ^ (r & 7)) * 16)) = v;
                        } else {
                            *reinterpret_cast<uint4*>(orow + e) = v;
                        }
                    }
                }
            }
        } else if (ok && valid && nx == 0 && !split) {
            // No visible key in this call (cannot happen without a split):
            // the row is zero.
            __nv_bfloat16* orow = p.out + ((q0 + pos) * p.hq + head) * (int64_t)D;
            for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
        }
        if (staged) {
            // Every thread of the warpgroup arrives (the vote carries whether
            // all of them got their output), then one thread stores.
            fence_proxy_async_smem();
            if (bar_and_sync(2 + x, kRows, ok) && r == 0) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_store_3d(&tm_o, pn * 64, hkv * g, (int)(q0 + first),
                                 smem_u32(stage + pn * C::kQPanel));
                bulk_commit_and_wait_read();
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == R::kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int NK, int NV, bool PLAIN, bool QQ = false>
cudaError_t launch_grid_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& to, const FwdParams& p, int pairs, cudaStream_t stream) {
    using C = GridCfg<D, NK, NV>;
    constexpr int kThreads = GR::kThreads;
    auto kern = prefill_grid_kernel<D, NK, NV, PLAIN, QQ>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(pairs * p.splits), (unsigned)p.hk, (unsigned)p.num_seqs);
    kern<<<grid, kThreads, C::kSmem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_grid(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const CUtensorMap& to, const FwdParams& p, int pairs, cudaStream_t stream) {
    const bool qq = (p.flags & UA_FLAG_QQ_BIAS) != 0;
    const bool plain = !qq && (p.flags & (UA_FLAG_SOFTCAP | UA_FLAG_ALIBI)) == 0;
    switch (p.d) {
        case 64:
            if (qq) return launch_grid_t<64, 4, 4, false, true>(tq, tm_k, tm_v, to, p, pairs, stream);
            return plain ? launch_grid_t<64, 4, 4, true>(tq, tm_k, tm_v, to, p, pairs, stream)
                         : launch_grid_t<64, 4, 4, false>(tq, tm_k, tm_v, to, p, pairs, stream);
        case 128:
            if (qq) return launch_grid_t<128, 2, 2, false, true>(tq, tm_k, tm_v, to, p, pairs, stream);
            return plain ? launch_grid_t<128, 2, 2, true>(tq, tm_k, tm_v, to, p, pairs, stream)
                         : launch_grid_t<128, 2, 2, false>(tq, tm_k, tm_v, to, p, pairs, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ua
