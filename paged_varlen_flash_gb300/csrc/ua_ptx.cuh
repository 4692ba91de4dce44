// ua_ptx.cuh -- small inline-PTX helpers for sm_103a: shared-memory addresses,
// mbarriers with bounded waits, TMA tensor loads, and bf16 unpacking.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ua {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA / tensor-core) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for an mbarrier phase, giving up after about one second of wall time
// (checked every 256 polls).  Returns false if it gave up.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_ns();
    for (;;) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - start > limit_ns) return false;
    }
}

// ---- CTA pairs (a cluster of two CTAs) ----------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the same shared-memory offset in CTA `rank`
// of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of any CTA of the cluster.  Default semantics
// (release at CTA scope): what the arrival publishes is tensor-memory data,
// which the writer orders with tcgen05.wait::st and
// tcgen05.fence::before_thread_sync before it arrives and the reader with
// tcgen05.fence::after_thread_sync after its wait; a cluster-scope release
// here costs a memory barrier per arrival (measured: 8 % of the CTA-pair
// prefill's time).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Every thread of both CTAs: release this CTA's prior writes, wait for the peer.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// ---- TMA ---------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 4-D tiled load into shared memory, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                            int32_t c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// The same loads for a CTA pair: the box lands in this CTA's shared memory
// and the byte count completes on `bar_cluster`, an mbarrier of either CTA
// of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                                 int32_t c2, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster)
        : "memory");
}

// 3-D tiled store from shared memory (the box at src, laid out with the
// map's swizzle) to global memory, tracked by the bulk async-group of the
// issuing thread.
__device__ __forceinline__ void tma_store_3d(const void* tmap, int32_t c0, int32_t c1, int32_t c2,
                                             uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(c0), "r"(c1), "r"(c2), "r"(src)
        : "memory");
}

// Close the thread's bulk async-group and wait until every store in it has
// read its shared-memory source.
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Row gather from a 2-D tensor map whose box is {cols, 1}: rows r0..r3 (each
// `cols` wide from column c0) land as four consecutive box rows at dst, with
// the map's swizzle, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap, int32_t c0, int32_t r0,
                                            int32_t r1, int32_t r2, int32_t r3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
        "r"(bar)
        : "memory");
}

// ---- per-thread asynchronous copies (LSU path) ---------------------------------
// 16 bytes global -> shared, cached in L2 only.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Wait until every cp.async this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t dst) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
}

// ---- bf16 ------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// tanh by the special-function unit's own approximation (tanh.approx.f32,
// one instruction; relative error about 2^-11 over the whole range).  Used by
// the compute-bound prefill kernel, where the softcap's two extra special-
// function operations per score (an exponential and a reciprocal) would make
// that unit, not the tensor cores, the bound.  A logit of magnitude |x| moves
// by at most ~5e-4 |x|, the same order as rounding P to bf16 for the MMA.
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the kernel before it in the
// stream still runs; griddep_wait() blocks the calling thread until that
// kernel has completed and its memory is visible, and griddep_launch() lets
// the dependent kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// tanh from its exponential form, tanh(x) = 1 - 2 / (e^{2x} + 1), with the
// hardware base-2 exponential and a fast reciprocal: relative error a few
// fp32 ulps away from 0 and absolute error ~1e-7 near 0 (far below the bf16
// output resolution); saturates to +-1 for large |x|.  Every kernel's softcap
// term calls this one definition.
__device__ __forceinline__ float tanh_from_exp2(float x) {
    const float e = fast_exp2(x * (2.0f * kLog2e));
    return 1.0f - __fdividef(2.0f, e + 1.0f);
}

}  // namespace ua
