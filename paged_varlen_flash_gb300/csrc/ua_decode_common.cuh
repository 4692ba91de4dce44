// ua_decode_common.cuh -- device helpers shared by the transposed decode
// kernels (keys on the MMA M dimension, 16 packed rows on N): bounded mbarrier
// waits that honour the CTA abort flag, a vote barrier, 16-column tensor
// memory loads and stores and a warp max.
#pragma once

#include <cstdint>

#include "ua_common.cuh"
#include "ua_ptx.cuh"

namespace ua {

__device__ __forceinline__ bool dwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      int32_t* err, uint64_t limit_ns = kWaitLimitNs) {
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

__device__ __forceinline__ bool dbar_and(int id, int count, bool pred) {
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

__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// Warp-wide float max through the integer reduction unit: IEEE-754 floats
// compare like sign-magnitude integers, so flipping the magnitude bits of
// negative values gives an order-preserving signed-integer key; one
// redux.sync.max.s32 then replaces a five-step shuffle tree.
__device__ __forceinline__ float warp_max_f32(float v) {
    const int b = __float_as_int(v);
    int key = b >= 0 ? b : (b ^ 0x7fffffff);
    int r;
    asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(key));
    return __int_as_float(r >= 0 ? r : (r ^ 0x7fffffff));
}

}  // namespace ua
