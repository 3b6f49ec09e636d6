// Host-side encoding of tiled TMA tensor maps (bf16, 128-byte swizzle), through the
// runtime's driver entry point so the library does not link libcuda.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace harts {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// bf16 tensor of `rank` dims (innermost first), zero fill out of range; 128-byte swizzle
// unless `swizzle` is false (then the box lands row-major, unpadded).
inline bool encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                        const cuuint64_t *strides, const cuuint32_t *box, bool swizzle = true) {
    auto fn = encode_tiled();
    if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace harts
