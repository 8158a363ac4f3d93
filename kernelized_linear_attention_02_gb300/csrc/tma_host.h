// tma_host.h -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so that the library does
// not link against libcuda directly).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace la {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A tensor of up to 5 dimensions (dims[0] innermost, contiguous), strides in
// bytes for dims 1.., box in elements; out-of-range elements of a load read
// as zero and out-of-range elements of a store are skipped.
inline bool make_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                            const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                            CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t d[5];
    cuuint64_t s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i > 0) s[i - 1] = strides_bytes[i - 1];
    }
    CUresult r = enc(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A bf16 tensor of up to 3 dimensions (dims[0] innermost, contiguous),
// strides in bytes for dims 1 and 2, box in elements, 128-byte swizzle;
// out-of-range elements of a box read as zero.
inline bool make_tensor_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                                 const uint64_t* strides_bytes, const uint32_t* box) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t d[3] = {dims[0], rank > 1 ? dims[1] : 1, rank > 2 ? dims[2] : 1};
    cuuint64_t s[2] = {rank > 1 ? strides_bytes[0] : 0, rank > 2 ? strides_bytes[1] : 0};
    cuuint32_t b[3] = {box[0], rank > 1 ? box[1] : 1, rank > 2 ? box[2] : 1};
    cuuint32_t e[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace la
