// ua_tmap.h -- host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so that no -lcuda link is
// needed).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace ua {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// bf16 tensor map with 128-byte swizzle; dims / strides innermost first
// (strides in bytes, rank - 1 of them), box in elements.
inline bool encode_bf16_sw128(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                              const cuuint64_t* strides, const cuuint32_t* box) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// 4-D map over a paged cache [num_blocks, b, H_k, d] (innermost first: d,
// H_k, b, num_blocks) whose box is one 128-byte swizzle panel (64 bf16 or 128
// e4m3 elements) x 1 KV head x `box_rows` consecutive slots x 1 block.  The
// TMA unit forms addresses in 64 bits, so a cache beyond 2 GiB needs no other
// path (the offset overflow of gfx950 "Unified paged attention on gfx950,
// from the math up", section 7.2, cannot happen here).
inline bool encode_cache_map(CUtensorMap* m, const void* base, int d, int hk, int b,
                             int64_t num_blocks, bool fp8, int box_rows) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    const cuuint64_t es = fp8 ? 1 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)hk, (cuuint64_t)b, (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {es * d, es * d * hk, es * d * hk * b};
    cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ua
