// ua_prefill_common.cuh -- device helpers shared by the tensor-core prefill
// kernels: bounded mbarrier waits that honour the CTA's abort
// flag, packed fp32 arithmetic, the base-2 exponential of a pair, a named
// barrier with an AND vote.
#pragma once

#include <cstdint>

#include "ua_common.cuh"
#include "ua_ptx.cuh"

namespace ua {
namespace pf {

constexpr float kLazy = 8.0f;
constexpr int kRows = 128;
constexpr uint32_t kTmemCols = 512;

// Wait on an mbarrier phase; gives up (and raises the CTA's abort flag and the
// device error bit) after about a second, or as soon as another role aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* err,
                                              uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_ns();
    for (;;) {
        for (int i = 0; i < 128; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - start > limit_ns) {
            *abort_flag = 1;
            atomicOr(err, (int)UA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
          "l"(*reinterpret_cast<uint64_t*>(&c)));
    return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
    return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
    return *reinterpret_cast<float2*>(&d);
}

// 2^a for a pair on the fp32 special-function path.  -inf maps to 0.
__device__ __forceinline__ float2 exp2_pair_f32(float2 a) {
    return make_float2(fast_exp2(a.x), fast_exp2(a.y));
}

// Named barrier over `count` threads that also returns the AND of `pred`
// across them.
__device__ __forceinline__ bool bar_and_sync(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

}  // namespace pf
}  // namespace ua
