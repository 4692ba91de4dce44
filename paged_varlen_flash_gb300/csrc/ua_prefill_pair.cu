// ua_prefill_pair.cu -- prefill / chunked-prefill attention for head sizes 64
// and 128 on the tcgen05 tensor cores of sm_103a: a persistent kernel that
// works through a device-built, longest-first list of work units, two query
// tiles per unit.
//
// Work unit: (sequence, pair of tiles of 128 packed (position, head) rows of
// one KV head, KV segment).  Tile A holds the earlier positions, tile B the
// next ones; the g query heads sharing the KV head are packed into the rows
// (gfx950 "Unified paged attention on gfx950, from the math up", section 4;
// floor(128 / g) positions per tile).  Both tiles consume every K and V tile
// the unit loads, so a paged K/V tile crosses the TMA unit once per 256 query
// rows -- on this cache layout (one 128-byte TMA row per key and 64-dim
// panel) the copy engine, not the tensor cores, is what a 128-row tile runs
// out of first.
//
// Work decomposition (gfx950 page, section 8.2: a persistent grid-stride over
// a work list, longest items first; attention_dense.py, its persistent
// variant's work-item decode):
//   plan_pairs_kernel   one CTA: counts each sequence's (tile pair, segment)
//                       entries (a block scan over the sequences), bins the
//                       entries by the number of KV tiles their two tiles
//                       visit and writes them longest first into the work
//                       list, then resets the claim counter.  No host sync:
//                       the lengths are read on the device.
//   prefill_pair_kernel one CTA per SM (launched as a programmatic dependent
//                       of the planner, so its prologue -- barrier init,
//                       tensor-memory allocation -- overlaps the planner);
//                       the TMA warp claims units from the counter (unit u =
//                       entry u / H_k, KV head u % H_k) and publishes each
//                       unit's descriptor through a two-slot ring in shared
//                       memory.  Tensor memory, barriers and the K/V rings
//                       stay live across units: the next unit's Q and first
//                       K/V tiles load while the current one's epilogue reads
//                       O out of tensor memory.
//
// The math is the streaming (m, l, o) recurrence of gfx1151 ALGORITHM.md
// section 3 in base 2 (gfx950 section 2) with the lazy re-anchor threshold of
// 8, the mask-free / masked tile split and the causal early exit of
// attention_dense.py (gfx950 section 8.1), per tile.
//
// Roles (12 warps):
//   warps 0-3  softmax + epilogue of tile A, warps 4-7 of tile B: thread r
//              owns row r (tensor-memory lane r) and all 128 key columns of
//              each S tile, so the two warpgroups never exchange row data;
//   warp 8     work claims, unit descriptors, TMA producer: Q_A and Q_B per
//              unit, then K and V tiles through NK- and NV-stage rings (one
//              box per paged block and 64-wide head-dim panel, one lane per
//              block);
//   warp 9     MMA issuer of tile A (also owns tensor memory);
//   warp 10    MMA issuer of tile B;
//   warp 11    idle (completes the third warpgroup for register reallocation).
//
// Tensor memory (512 columns): S_A [0, 128), S_B [128, 256),
// O_A [256, 256 + D), O_B [256 + D, 256 + 2D).  P_X (bf16, two keys per
// column) is written over the first 64 columns of S_X once S_X has been read;
// the next QK^T into S_X is issued right behind the P.V that reads it, by the
// same thread.  A unit's first P.V into O_X waits until the previous unit's
// epilogue has read O_X (o_free).
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

constexpr int kBN = 128;            // keys per K/V tile (the QK^T MMA's N)
constexpr int kPlanThreads = 1024;  // planner CTA
constexpr int kCostBuckets = 2048;  // planner cost bins (KV tile-steps, clamped)

// Score transform variants, each its own instantiation so that the plain
// loop keeps its registers:
//   kPlain    scale only (the scale is folded into the exponent);
//   kSoftcap  scale + softcap: y = tanh(s * tau / c), the logit in log2 units
//             is y * c * log2(e), folded into the exponent the same way;
//   kGeneral  any mix of softcap, ALiBi and (QQ) the query-query bias.
enum { kPlain = 0, kSoftcap = 1, kGeneral = 2 };

// One work unit, written by the TMA warp into a two-slot ring and read by the
// MMA and softmax warps.
struct PairUnit {
    int32_t live;     // 0: the list is exhausted, leave
    int32_t zero;     // rows written as zeros (or empty partials); no MMA
    int32_t s, hkv, seg;
    int32_t q0, sq, sk;
    int32_t p0, has_b, last_a, last_b;
    int32_t t_begin, n_a, n_b;
    int32_t kv0;      // K/V tiles this CTA loaded before this unit
};
static_assert(sizeof(PairUnit) == 64, "unit descriptor");

// Key range a (sequence, tile pair, segment) visits: tile A stops where its
// causal range (or the segment) ends; tile B covers every tile of the range.
// n_a = n_b = 0 when no row of either tile sees a key in this segment.
struct PairRange {
    int p0, has_b, last_a, last_b, t_begin, n_a, n_b;
};

__device__ __forceinline__ PairRange pair_range(const FwdParams& p, int sq, int sk, int pair,
                                                int seg) {
    PairRange r;
    const int ppt = kRows / p.g;
    r.p0 = pair * 2 * ppt;
    r.has_b = r.p0 + ppt < sq;
    r.last_a = min(r.p0 + ppt, sq) - 1;
    r.last_b = r.has_b ? min(r.p0 + 2 * ppt, sq) - 1 : r.last_a;
    const int ctx = sk - sq;
    const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
    const bool window = (p.flags & UA_FLAG_WINDOW) != 0;
    int k_beg = window ? max(0, r.p0 + ctx - p.window + 1) : 0;
    int kend_a = causal ? min(sk, r.last_a + ctx + 1) : sk;
    int kend_b = causal ? min(sk, r.last_b + ctx + 1) : sk;
    if (p.splits > 1) {   // this unit's KV segment; segments are whole tiles
        k_beg = max(k_beg, seg * p.chunk);
        kend_a = min(kend_a, seg * p.chunk + p.chunk);
        kend_b = min(kend_b, seg * p.chunk + p.chunk);
    }
    const int k_end = r.has_b ? kend_b : kend_a;
    r.t_begin = k_beg / kBN;
    if (k_beg >= k_end) {
        r.n_a = r.n_b = 0;
    } else {
        r.n_a = kend_a > k_beg ? (kend_a + kBN - 1) / kBN - r.t_begin : 0;
        r.n_b = r.has_b ? (kend_b + kBN - 1) / kBN - r.t_begin : 0;
    }
    return r;
}

// Work-list entries of sequence s: its tile pairs times its KV segments
// (none for a sequence whose cu_seqlens_q is malformed).
__device__ __forceinline__ int seq_entries(const FwdParams& p, int s, uint32_t* st_out) {
    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, s, sq, sk, q0);
    *st_out = st;
    if ((st & UA_DEVERR_CU_SEQLENS) || sq <= 0) return 0;
    const int span = 2 * (kRows / p.g);
    const int nseg = p.splits > 1 ? seq_segments(p, st, sk) : 1;
    return (sq + span - 1) / span * nseg;
}

// Inclusive scan over the planner's 1024 threads (Hillis-Steele in shared
// memory); every thread of the CTA must call it.
__device__ __forceinline__ int block_scan(int v, int* tmp) {
    const int tid = threadIdx.x;
    tmp[tid] = v;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
        const int add = tid >= off ? tmp[tid - off] : 0;
        __syncthreads();
        tmp[tid] += add;
        __syncthreads();
    }
    const int r = tmp[tid];
    __syncthreads();
    return r;
}

// Decode list position e into (sequence, tile pair, segment) through the
// per-sequence prefix, and return the unit's cost bin (KV tile-steps of both
// tiles; malformed sequences cost 0 and go last).
__device__ __forceinline__ int entry_cost(const FwdParams& p, int e, int num_seqs, int& s,
                                          int& pair, int& seg) {
    int lo = 0, hi = num_seqs - 1;   // last s with seq_prefix[s] <= e
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seq_prefix[mid] <= e) lo = mid; else hi = mid - 1;
    }
    s = lo;
    int sq, sk;
    int64_t q0;
    const uint32_t st = seq_status(p, s, sq, sk, q0);
    const int nseg = p.splits > 1 ? seq_segments(p, st, sk) : 1;
    const int local = e - p.seq_prefix[s];
    pair = local / nseg;
    seg = local % nseg;
    if (st) return 0;
    const PairRange r = pair_range(p, sq, sk, pair, seg);
    return min(r.n_a + r.n_b, kCostBuckets - 1);
}

__global__ void __launch_bounds__(kPlanThreads) plan_pairs_kernel(const FwdParams p) {
    // The persistent kernel may start now; it waits for this grid to finish
    // before it reads the list.
    griddep_launch();
    __shared__ int hist[kCostBuckets];
    __shared__ int tmp[kPlanThreads];
    const int tid = threadIdx.x;
    const int n = p.num_seqs;
    // 1. entries per sequence (each thread a contiguous run of sequences),
    //    their exclusive prefix, and the status bits of malformed sequences
    const int per = (n + kPlanThreads - 1) / kPlanThreads;
    const int s0 = min(n, tid * per), s1 = min(n, s0 + per);
    int local = 0;
    for (int s = s0; s < s1; ++s) {
        uint32_t st;
        local += seq_entries(p, s, &st);
        if (st) atomicOr(p.err, (int)st);
    }
    const int incl = block_scan(local, tmp);
    int run = incl - local;
    for (int s = s0; s < s1; ++s) {
        uint32_t st;
        p.seq_prefix[s] = run;
        run += seq_entries(p, s, &st);
    }
    if (tid == kPlanThreads - 1) tmp[0] = incl;
    for (int b = tid; b < kCostBuckets; b += kPlanThreads) hist[b] = 0;
    __syncthreads();   // also orders the prefix writes before their reads below
    const int total = min(tmp[0], p.work_cap);
    // 2. histogram of the costs
    for (int e = tid; e < total; e += kPlanThreads) {
        int s, pair, seg;
        atomicAdd(&hist[entry_cost(p, e, n, s, pair, seg)], 1);
    }
    __syncthreads();
    // 3. bin offsets, highest cost first: thread t owns bins 2047 - 2t and
    //    2046 - 2t
    const int b0 = kCostBuckets - 1 - 2 * tid, b1 = b0 - 1;
    const int h0 = hist[b0], h1 = hist[b1];
    const int base = block_scan(h0 + h1, tmp) - (h0 + h1);
    hist[b0] = base;
    hist[b1] = base + h0;
    __syncthreads();
    // 4. scatter (the order inside one bin does not matter: every unit writes
    //    only its own rows)
    for (int e = tid; e < total; e += kPlanThreads) {
        int s, pair, seg;
        const int c = entry_cost(p, e, n, s, pair, seg);
        const int pos = atomicAdd(&hist[c], 1);
        p.work_list[pos] = make_int2(s, (pair << 7) | seg);
    }
    if (tid == 0) {
        p.work_info[0] = total;
        p.work_info[1] = 0;   // claim counter
    }
}

template <int D, int NK, int NV>
struct PairCfg {
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kRows * 128;        // 128 rows x 64 dims
    static constexpr int kQTile = kPanels * kQPanel;
    static constexpr int kKvPanel = kBN * 128;
    static constexpr int kKvBytes = kPanels * kKvPanel;
    static constexpr int kOffQ = 0;                     // Q_A then Q_B
    static constexpr int kOffK = kOffQ + 2 * kQTile;
    static constexpr int kOffV = kOffK + NK * kKvBytes;
    static constexpr int kOffBar = kOffV + NV * kKvBytes;
    // q_full, q_empty, k_full[NK], v_full[NV], k_empty[NK], v_empty[NV], then
    // per tile: s_full[2], p_full[2], o_done[2], o_free[2]; unit ring
    // u_full[2], u_empty[2]; drain[2]; softmax turns turn[2]; never (the
    // testing hook's stall waits on it; nothing arrives)
    static constexpr int kNumBars = 2 + 2 * NK + 2 * NV + 17;
    static constexpr int kOffUnit = (kOffBar + kNumBars * 8 + 63) / 64 * 64;
    static constexpr int kOffMisc = kOffUnit + 2 * (int)sizeof(PairUnit);
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static constexpr int kTmemO = 2 * kBN;
    static_assert(2 * kBN + 2 * D <= (int)kTmemCols, "tensor memory budget");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// Two softmax warpgroups (one per tile), then a third warpgroup of the TMA
// warp, the two MMA-issuing warps and one idle warp (register reallocation
// works on whole warpgroups).
struct PR {
    static constexpr int kThreads = 384;
    static constexpr int kWarpTma = 8;
    static constexpr int kWarpMma = 9;    // MMA issuer of tile A, tensor-memory owner
    static constexpr int kWarpPv = 10;    // MMA issuer of tile B
    // Registers per thread after the split: 2 x 128 x 216 + 128 x 72 equals
    // the 384 x 168 the block is launched with (the claim / descriptor /
    // issue loops of the third warpgroup spill at 56).
    static constexpr uint32_t kRegsSoftmax = 216;
    static constexpr uint32_t kRegsOther = 72;
    static constexpr int kUnitReaders = 2 + 256;   // MMA warps (one lane each) + softmax threads
};

template <int D, int NK, int NV, int MODE, bool QQ>
__global__ void __launch_bounds__(PR::kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = PairCfg<D, NK, NV>;
    using R = PR;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool split = p.splits > 1;             // write (m, l, o) partials per KV segment
    const int g = p.g;
    const int ppt = kRows / g;                  // positions per tile

    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    const uint32_t q_full = smem_u32(&bar_mem[0]);
    const uint32_t q_empty = smem_u32(&bar_mem[1]);   // both tiles' last QK^T of a unit done
    const uint32_t k_full0 = smem_u32(&bar_mem[2]);
    const uint32_t v_full0 = smem_u32(&bar_mem[2 + NK]);
    // A K stage is free once both tiles' QK^T ran, a V stage once both P.V ran.
    const uint32_t k_empty0 = smem_u32(&bar_mem[2 + NK + NV]);
    const uint32_t v_empty0 = smem_u32(&bar_mem[2 + 2 * NK + NV]);
    constexpr int kBarT = 2 + 2 * NK + 2 * NV;
    const uint32_t s_full0 = smem_u32(&bar_mem[kBarT]);        // + 8 * tile
    const uint32_t p_full0 = smem_u32(&bar_mem[kBarT + 2]);
    const uint32_t o_done0 = smem_u32(&bar_mem[kBarT + 4]);    // a unit's last P.V done
    const uint32_t o_free0 = smem_u32(&bar_mem[kBarT + 6]);    // its epilogue read O
    const uint32_t u_full0 = smem_u32(&bar_mem[kBarT + 8]);    // + 8 * slot
    const uint32_t u_empty0 = smem_u32(&bar_mem[kBarT + 10]);
    const uint32_t drain0 = smem_u32(&bar_mem[kBarT + 12]);
    const uint32_t turn0 = smem_u32(&bar_mem[kBarT + 14]);     // + 8 * tile
    const uint32_t never = smem_u32(&bar_mem[kBarT + 16]);
    PairUnit* units = reinterpret_cast<PairUnit*>(smem + C::kOffUnit);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 2);                // one arrival per tile
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
            mbar_init(o_free0 + 8 * x, kRows);
            mbar_init(u_full0 + 8 * x, 1);
            mbar_init(u_empty0 + 8 * x, R::kUnitReaders);
            mbar_init(drain0 + 8 * x, 1);
            mbar_init(turn0 + 8 * x, kRows);
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PR::kRegsOther));
    auto wwait = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xffffffffu, wait_or_abort(bar, par, abort_flag, p.err));
    };
    if (warp == R::kWarpTma) {
        // --------------------- work claims + TMA producer ---------------------
        // Lane i owns paged block i of each KV tile (its id load and its TMA
        // boxes), so one tile's boxes go out in parallel.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        griddep_wait();   // the planner's list, length and counter are ready
        const int num_units = *reinterpret_cast<volatile int32_t*>(p.work_info) * p.hk;
        const int b = p.b;
        int n = 0;        // units published
        int qn = 0;       // Q loads issued
        int kt = 0;       // K/V tiles issued (both operands)
        int k_extra = 0;  // 1 if a K copy went out without its V (abort)
        bool ok = true;
        for (;;) {
            int u = 0;
            if (lane == 0) u = atomicAdd(p.work_info + 1, 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            const int slot = n & 1;
            if (n >= 2 && !(ok = wwait(u_empty0 + 8 * slot, ((n >> 1) + 1) & 1))) break;
            if (lane == 0) {
                PairUnit w;
                std::memset(&w, 0, sizeof w);
                w.live = u < num_units;
                if (w.live) {
                    const int2 ent = p.work_list[u / p.hk];
                    w.s = ent.x;
                    w.hkv = u % p.hk;
                    w.seg = ent.y & 127;
                    int64_t q0;
                    const uint32_t st = seq_status(p, w.s, w.sq, w.sk, q0);
                    w.q0 = (int32_t)q0;
                    const PairRange r = pair_range(p, w.sq, w.sk, ent.y >> 7, w.seg);
                    w.p0 = r.p0;
                    w.has_b = r.has_b;
                    w.last_a = r.last_a;
                    w.last_b = r.last_b;
                    w.t_begin = r.t_begin;
                    w.n_a = st ? 0 : r.n_a;
                    w.n_b = st ? 0 : r.n_b;
                    w.zero = (st != 0) || (w.n_a + w.n_b == 0);
                    w.kv0 = kt;
                }
                units[slot] = w;
                mbar_arrive(u_full0 + 8 * slot);
            }
            __syncwarp();
            // Every lane takes the fields it needs into registers (the copy
            // asm statements clobber memory).
            const PairUnit& ud = units[slot];
            const int live = ud.live, zero = ud.zero, has_b = ud.has_b, hkv = ud.hkv;
            const int q_row = ud.q0 + ud.p0, t_begin = ud.t_begin, useq = ud.s, sk = ud.sk;
            const int n_tiles = max(ud.n_a, ud.n_b);
            ++n;
            if (!live) break;
            if (zero) continue;
            // Q_A and Q_B of this unit, once both tiles' last QK^T of the
            // previous unit has read the old ones.
            if (qn >= 1 && !(ok = wwait(q_empty, (qn - 1) & 1))) break;
            if (lane == 0) {
                // One box per panel and tile: g heads x ppt positions = g * ppt
                // rows (128 when g divides 128; the rows past them are padding
                // whose outputs are never stored).
                mbar_arrive_expect_tx(q_full, (has_b ? 2u : 1u) * (uint32_t)(g * ppt) * 128u * C::kPanels);
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn) {
                    tma_load_3d(sQ + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, q_row, q_full);
                    if (has_b)
                        tma_load_3d(sQ + C::kQTile + pn * C::kQPanel, &tm_q, pn * 64, hkv * g, q_row + ppt,
                                    q_full);
                }
            }
            ++qn;
            const int nblk_seq = (sk + b - 1) / b;
            const int32_t* bt = p.block_table + (int64_t)useq * p.bt_stride;
            // Block ids are fetched one tile ahead so their load latency
            // overlaps the current tile's waits and copies.
            auto tile_id = [&](int j) -> int32_t {
                const int blk0 = (t_begin + j) * kBN / b;
                return lane < min(kBN / b, nblk_seq - blk0) ? __ldg(bt + blk0 + lane) : 0;
            };
            int32_t id_next = tile_id(0);
            for (int j = 0; j < n_tiles; ++j, ++kt) {
                const int stk = kt % NK, stv = kt % NV;
                const int blk0 = (t_begin + j) * kBN / b;
                const int nb = min(kBN / b, nblk_seq - blk0);
                const uint32_t bytes = (uint32_t)nb * b * 128 * C::kPanels;
                const int32_t id = id_next;
                if (j + 1 < n_tiles) id_next = tile_id(j + 1);
                if (lane < nb && (id < 0 || (int64_t)id >= p.num_blocks))
                    atomicOr(p.err, (int)UA_DEVERR_BLOCK_ID);
                if (kt >= NK && !(ok = wwait(k_empty0 + 8 * stk, ((kt / NK) + 1) & 1))) break;
                if (lane == 0) mbar_arrive_expect_tx(k_full0 + 8 * stk, bytes);
                __syncwarp();
                if (lane < nb) {
#pragma unroll
                    for (int pn = 0; pn < C::kPanels; ++pn)
                        tma_load_4d(sK + stk * C::kKvBytes + pn * C::kKvPanel + lane * b * 128, &tm_k,
                                    pn * 64, hkv, 0, id, k_full0 + 8 * stk);
                }
                if (kt >= NV && !(ok = wwait(v_empty0 + 8 * stv, ((kt / NV) + 1) & 1))) {
                    k_extra = 1;   // this tile's K copy was issued, its V copy not
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(v_full0 + 8 * stv, bytes);
                __syncwarp();
                if (lane < nb) {
#pragma unroll
                    for (int pn = 0; pn < C::kPanels; ++pn)
                        tma_load_4d(sV + stv * C::kKvBytes + pn * C::kKvPanel + lane * b * 128, &tm_v,
                                    pn * 64, hkv, 0, id, v_full0 + 8 * stv);
                }
            }
            if (!ok) break;
        }
        if (*abort_flag && lane == 0) {
            // Let every copy this warp issued land before the CTA ends.
            if (qn > 0) mbar_wait_bounded(q_full, (qn - 1) & 1);
            for (int j = max(0, kt + k_extra - NK); j < kt + k_extra; ++j)
                mbar_wait_bounded(k_full0 + 8 * (j % NK), (j / NK) & 1);
            for (int j = max(0, kt - NV); j < kt; ++j)
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
        const int x = warp - R::kWarpMma;
        const uint32_t dS = tmem + x * kBN;
        const uint32_t dO = tmem + C::kTmemO + x * D;
        const uint32_t qst = sQ + x * C::kQTile;
        // Shared-memory descriptors as a base per operand buffer plus a
        // compile-time offset per MMA: the start-address field holds the byte
        // address >> 4 (below 2^14 for any shared-memory address), so adding
        // an offset never carries into the next field, and the issue loop
        // spends one add per descriptor instead of recomputing it.
        const uint64_t q_desc = tc::smem_desc_sw128(qst, 16, 1024);
        const uint64_t k_desc0 = tc::smem_desc_sw128(sK, 16, 1024);
        const uint64_t v_desc0 = tc::smem_desc_sw128(sV, C::kKvPanel, 1024);
        constexpr uint32_t kStageStep = (uint32_t)C::kKvBytes >> 4;   // one ring stage
        int n = 0, qn = 0;
        int sx = 0;   // S tiles of tile x issued before this unit
        int ux = 0;   // units with work for tile x before this one
        bool ok = true;
        for (;;) {
            const int slot = n & 1;
            if (!(ok = wwait(u_full0 + 8 * slot, (n >> 1) & 1))) break;
            // The fields this warp needs, in registers (the MMA asm statements
            // clobber memory, so fields read from shared memory inside the
            // issue loop would be reloaded after every MMA); the slot is
            // released at once.
            const PairUnit& ud = units[slot];
            const int live = ud.live, zero = ud.zero;
            const int nx = x ? ud.n_b : ud.n_a;
            const int n_other = x ? ud.n_a : ud.n_b;
            const int kv0 = ud.kv0, t_begin = ud.t_begin, sk = ud.sk;
            __syncwarp();
            if (lane == 0) mbar_arrive(u_empty0 + 8 * slot);
            ++n;
            if (!live) break;
            if (zero) continue;
            if (!(ok = wwait(q_full, qn & 1))) break;
            ++qn;
            if (nx == 0) {
                // This tile reads neither Q nor any K/V stage in this unit.
                if (lane == 0) mbar_arrive(q_empty);
                __syncwarp();
                continue;
            }
            auto issue_qk = [&](int j) -> bool {
                const int kt = kv0 + j;
                const int stg = kt % NK;
                // Testing hook: the first K wait of the CTA waits on a barrier
                // that nothing completes and gives up after stall_ns.
                if (p.stall && kt == 0 &&
                    !__all_sync(0xffffffffu, wait_or_abort(never, 0, abort_flag, p.err, (uint64_t)p.stall_ns)))
                    return false;
                if (!wwait(k_full0 + 8 * stg, (kt / NK) & 1)) return false;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint64_t kd_s = k_desc0 + (uint64_t)((uint32_t)stg * kStageStep);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t oq = ((k >> 2) * C::kQPanel + (k & 3) * 32) >> 4;
                        const uint32_t ok_ = ((k >> 2) * C::kKvPanel + (k & 3) * 32) >> 4;
                        tc::mma_bf16(dS, q_desc + oq, kd_s + ok_, idesc_qk, k > 0 ? 1u : 0u);
                    }
                    tc::commit(s_full0 + 8 * x);
                    tc::commit(k_empty0 + 8 * stg);
                    if (j >= n_other) tc::commit(k_empty0 + 8 * stg);
                    if (j + 1 == nx) tc::commit(q_empty);   // this tile's last read of Q_x
                }
                __syncwarp();
                return true;
            };
            ok = issue_qk(0);
            for (int j = 0; ok && j < nx; ++j) {
                const int kt = kv0 + j;
                const int stg = kt % NV;
                if (!(ok = wwait(p_full0 + 8 * x, (sx + j) & 1))) break;
                if (!(ok = wwait(v_full0 + 8 * stg, (kt / NV) & 1))) break;
                // The first P.V of a unit overwrites O_x: the previous unit's
                // epilogue must have read it.
                if (j == 0 && ux > 0 && !(ok = wwait(o_free0 + 8 * x, (ux - 1) & 1))) break;
                tc::fence_after_sync();
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
                    const uint64_t vd = v_desc0 + (uint64_t)((uint32_t)stg * kStageStep);
#pragma unroll
                    for (int k = 0; k < kBN / 16; ++k) {
                        // A = P_x from tensor memory: 16 keys per MMA = 8 columns.
                        tc::mma_bf16_ts(dO, dS + k * 8, vd + ((k * 16 * 128) >> 4), idesc_pv,
                                        (j > 0 || k > 0) ? 1u : 0u);
                    }
                    tc::commit(v_empty0 + 8 * stg);
                    if (j >= n_other) tc::commit(v_empty0 + 8 * stg);
                    if (j + 1 == nx) tc::commit(o_done0 + 8 * x);
                }
                __syncwarp();
                if (j + 1 < nx) ok = issue_qk(j + 1);
            }
            if (!ok) break;
            sx += nx;
            ++ux;
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
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PR::kRegsSoftmax));
        // ------------------------- softmax + epilogue warps -----------------------
        // Warpgroup x owns tile x: thread r holds row r (tensor-memory lane r)
        // and all 128 key columns of each S_x tile, so a row's max and sum
        // need no exchange and the two warpgroups never wait for each other.
        const int x = threadIdx.x >> 7;
        const int r = threadIdx.x & (kRows - 1);
        const bool causal = (p.flags & UA_FLAG_CAUSAL) != 0;
        const bool window = (p.flags & UA_FLAG_WINDOW) != 0;
        const bool softcap = (p.flags & UA_FLAG_SOFTCAP) != 0;
        const bool alibi = (p.flags & UA_FLAG_ALIBI) != 0;
        // Scale of the exponent argument: the logit in log2 units is
        // s * sl2 (plain) or y * cap_l2 with y = tanh(s * tau / c) (softcap).
        const float sl2 = p.scale * kLog2e;
        const float cap_l2 = softcap ? p.softcap * kLog2e : 0.f;
        const float cap_in = softcap ? p.scale / p.softcap : 0.f;
        const float xs = MODE == kPlain ? sl2 : MODE == kSoftcap ? cap_l2 : 1.0f;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = trow + x * kBN;
        const uint32_t ocol = trow + C::kTmemO + x * D;
        const uint32_t p_full = p_full0 + 8 * x;
        const uint32_t o_done = o_done0 + 8 * x;
        int n = 0;
        int sx = 0;           // S tiles of this tile before this unit
        int ux = 0;           // units with work for this tile before this one
        int tb = 0;           // turn rounds of either warpgroup before this unit
        bool ok = true;
        for (;;) {
            const int slot = n & 1;
            if (!(ok = __all_sync(0xffffffffu, wait_or_abort(u_full0 + 8 * slot, (n >> 1) & 1, abort_flag,
                                                             p.err))))
                break;
            const PairUnit un = units[slot];
            mbar_arrive(u_empty0 + 8 * slot);
            ++n;
            if (!un.live) break;
            const int first = un.p0 + x * ppt;
            const int last = x ? un.last_b : un.last_a;
            const int pos = first + r / g;
            const bool valid = (x == 0 || un.has_b) && pos <= last;
            const int head = un.hkv * g + r % g;
            const int64_t row = ((int64_t)un.q0 + pos) * p.hq + head;
            const int seg = un.seg;
            if (un.zero) {
                // Malformed lengths (rows written as zeros) or a segment with
                // no visible key for any row of either tile (an empty
                // partial, m = -inf).
                if (valid) {
                    if (split) {
                        p.part_ml[(row * p.splits + seg) * 2 + 0] = -INFINITY;
                        p.part_ml[(row * p.splits + seg) * 2 + 1] = 0.f;
                    } else {
                        uint4* orow = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll
                        for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            const int sk = un.sk;
            const int ctx = sk - un.sq;
            const int hi = causal ? min(pos + ctx, sk - 1) : sk - 1;
            const int lo = window ? max(0, pos + ctx - p.window + 1) : 0;
            const float slope = (MODE == kGeneral && alibi) ? __ldg(p.alibi + head) : 0.f;
            // The row's line of the query-query bias (none for padding rows).
            const float* qrow = (QQ && valid) ? p.qq_bias + (int64_t)pos * p.qq_stride : nullptr;
            // Keys every row of the tile sees: [kfree_lo, kfree_hi].
            const int kfree_hi = causal ? min(first + ctx, sk - 1) : sk - 1;
            const int kfree_lo = window ? max(0, last + ctx - p.window + 1) : 0;
            // Warps whose 32 rows are all padding skip the score work; they
            // still take part in every barrier.
            const bool live = __any_sync(0xffffffffu, valid);
            const int nx = x ? un.n_b : un.n_a;
            const int n_other = x ? un.n_a : un.n_b;
            // Light score work takes turns with the other warpgroup, so each
            // softmax has the issue slots and the special-function pipe to
            // itself while the tensor cores run the other tile's MMAs: round
            // j of A follows round j - 1 of B, round j of B follows round j
            // of A.  Both warpgroups run T = max(n_a, n_b) rounds per unit (a
            // tile with fewer key tiles passes through its extra rounds) and
            // A closes each unit by waiting for B's last round, so neither
            // can run ahead of the other by more than one round and the
            // parity waits on the turn barriers stay exact across units.
            // (With ALiBi or the query-query bias the two warpgroups run side
            // by side.)
            constexpr bool kTurns = MODE != kGeneral;
            const int rounds = kTurns ? max(nx, n_other) : nx;
            float m = -INFINITY;  // running max, log2 units
            float l = 0.f;        // running denominator
            for (int j = 0; j < rounds; ++j) {
                const int follow = x == 0 ? j - 1 : j;   // the other warpgroup's round to follow
                if (kTurns && follow >= 0 &&
                    !(ok = __all_sync(0xffffffffu, wait_or_abort(turn0 + 8 * (1 - x), (tb + follow) & 1,
                                                                 abort_flag, p.err))))
                    break;
                if (j >= nx) {
                    mbar_arrive(turn0 + 8 * x);   // a round this tile has no key tile for
                    continue;
                }
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(s_full0 + 8 * x, (sx + j) & 1, abort_flag,
                                                                 p.err))))
                    break;
                uint32_t sr[kBN / 32][32];
                const int key0 = (un.t_begin + j) * kBN;
                float tmax = -INFINITY;
                if (live) {
                    tc::fence_after_sync();
                    // With a transform: half of the row's scores first, the
                    // other half's loads in flight while the first half is
                    // transformed.  Plain scores: all four loads, one wait.
                    tc::ld32(s_col, sr[0]);
                    tc::ld32(s_col + 32, sr[1]);
                    if constexpr (MODE != kPlain) tc::wait_ld();
                    tc::ld32(s_col + 64, sr[2]);
                    tc::ld32(s_col + 96, sr[3]);
                    auto transform = [&](int c) {
                        if constexpr (MODE == kSoftcap) {
                            const float2 k2 = make_float2(cap_in, cap_in);
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float2 a = fmul2(make_float2(__uint_as_float(sr[c][e]),
                                                                   __uint_as_float(sr[c][e + 1])), k2);
                                sr[c][e] = __float_as_uint(tanh_fast(a.x));
                                sr[c][e + 1] = __float_as_uint(tanh_fast(a.y));
                            }
                        } else if constexpr (MODE == kGeneral) {
                            // ALiBi: one int -> float conversion per tile; the
                            // per-key offsets are compile-time constants.
                            const float abias = slope * (float)(key0 - ctx);
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                float t = __uint_as_float(sr[c][e]);
                                t = softcap ? p.softcap * tanh_fast(t * cap_in) : t * p.scale;
                                if (alibi) t += abias + slope * (float)(c * 32 + e);
                                sr[c][e] = __float_as_uint(t * kLog2e);
                            }
                        }
                    };
                    transform(0);
                    transform(1);
                    tc::wait_ld();
                    transform(2);
                    transform(3);
                    if constexpr (QQ) {
                        // Query-query bias, in its own pass: the query-section
                        // keys up to the row's last visible key (so j - ctx <
                        // S_q), in log2 units like the scores it joins.
                        if (qrow != nullptr && key0 + kBN > ctx && key0 <= hi) {
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
                    const bool mask_free = key0 >= kfree_lo && key0 + kBN - 1 <= kfree_hi;
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
                    tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7]));
                    tmax *= xs;   // to log2 units (xs > 0 keeps the order)
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
                    // P = 2^(x * xs - m): the exponent argument in fp32 (packed
                    // pairs), the power of two on the fp32 special-function
                    // path, row sums in fp32.  P goes over the first 64 columns
                    // of S_x (lane r, two bf16 keys per 32-bit column: the A
                    // operand of the P.V MMA); this thread has already read all
                    // of its row's S.
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
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        const uint32_t col = ocol + c * 32;
                        tc::ld32(col, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st32(col, o);
                    }
                    tc::wait_st();
                }
                tc::fence_before_sync();
                mbar_arrive(p_full);
                if (kTurns) mbar_arrive(turn0 + 8 * x);
            }
            if (!ok) break;
            // ------------------------------ epilogue ---------------------------------
            if (nx > 0 && !(ok = __all_sync(0xffffffffu, wait_or_abort(o_done, ux & 1, abort_flag, p.err))))
                break;   // after the last P.V
            if (valid && split) {
                // Split partial: raw o (below), m in log2 units, l.
                p.part_ml[(row * p.splits + seg) * 2 + 0] = nx > 0 ? m : -INFINITY;
                p.part_ml[(row * p.splits + seg) * 2 + 1] = nx > 0 ? l : 0.f;
            }
            if (live && nx > 0) {
                // tcgen05.ld is warp-collective: every lane of a live warp loads.
                tc::fence_after_sync();
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
                            *reinterpret_cast<uint4*>(orow + e) = v;
                        }
                    }
                }
            } else if (valid && nx == 0 && !split) {
                // No visible key in this call (cannot happen without a split):
                // the row is zero.
                __nv_bfloat16* orow = p.out + row * (int64_t)D;
                for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
            }
            if (nx > 0) {
                // O_x has been read: the next unit's first P.V may overwrite it.
                tc::fence_before_sync();
                mbar_arrive(o_free0 + 8 * x);
                ++ux;
            }
            // A's closing wait: B's last round of this unit.
            if (kTurns && x == 0 && rounds > 0 &&
                !(ok = __all_sync(0xffffffffu, wait_or_abort(turn0 + 8, (tb + rounds - 1) & 1, abort_flag,
                                                             p.err))))
                break;
            sx += nx;
            if (kTurns) tb += rounds;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == R::kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int NK, int NV, int MODE, bool QQ = false>
cudaError_t launch_pair_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdParams& p, int ctas, cudaStream_t stream) {
    using C = PairCfg<D, NK, NV>;
    auto kern = prefill_pair_kernel<D, NK, NV, MODE, QQ>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    // The planner first; the persistent kernel may start while it runs.
    plan_pairs_kernel<<<1, kPlanThreads, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(PR::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace

bool prefill_pair_supported(int d) { return d == 64 || d == 128; }

int64_t pair_work_entries_bound(const FwdParams& p, int splits) {
    // Entries = sum over sequences of ceil(S_q / (2 ppt)) x segments
    // <= (total_q / (2 ppt) + num_seqs) x splits.
    const int64_t span = 2 * (kRows / p.g);
    return (p.total_q / span + p.num_seqs) * splits;
}

cudaError_t launch_prefill_pair(const CUtensorMap& tq, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                const FwdParams& p, int ctas, cudaStream_t stream) {
    const bool qq = (p.flags & UA_FLAG_QQ_BIAS) != 0;
    const bool alibi = (p.flags & UA_FLAG_ALIBI) != 0;
    const bool softcap = (p.flags & UA_FLAG_SOFTCAP) != 0;
    const int mode = (qq || alibi) ? kGeneral : softcap ? kSoftcap : kPlain;
    switch (p.d) {
        case 64:
            if (qq) return launch_pair_t<64, 4, 4, kGeneral, true>(tq, tm_k, tm_v, p, ctas, stream);
            if (mode == kPlain) return launch_pair_t<64, 4, 4, kPlain>(tq, tm_k, tm_v, p, ctas, stream);
            if (mode == kSoftcap) return launch_pair_t<64, 4, 4, kSoftcap>(tq, tm_k, tm_v, p, ctas, stream);
            return launch_pair_t<64, 4, 4, kGeneral>(tq, tm_k, tm_v, p, ctas, stream);
        case 128:
            if (qq) return launch_pair_t<128, 2, 2, kGeneral, true>(tq, tm_k, tm_v, p, ctas, stream);
            if (mode == kPlain) return launch_pair_t<128, 2, 2, kPlain>(tq, tm_k, tm_v, p, ctas, stream);
            if (mode == kSoftcap) return launch_pair_t<128, 2, 2, kSoftcap>(tq, tm_k, tm_v, p, ctas, stream);
            return launch_pair_t<128, 2, 2, kGeneral>(tq, tm_k, tm_v, p, ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ua
