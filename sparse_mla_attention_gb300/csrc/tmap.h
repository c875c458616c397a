// tmap.h -- host helper that encodes TMA tensor maps. The driver entry point
// is looked up through the runtime (cudaGetDriverEntryPointByVersion), so the
// library does not link against the driver library.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace smla {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// Row-major 2-D bf16 tensor [rows, cols] (cols contiguous, row stride
// `row_stride_elems`), box of box_rows x box_cols elements, 128-byte swizzle
// (box_cols * 2 must be 128) or none. Out-of-range boxes read zeros.
inline bool make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_cols,
                              bool swizzle128) {
    auto fn = encode_tiled_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_stride_elems * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Two row-major bf16 tensors of the same shape [T, H, 512] (rows of 512
// contiguous elements), a and b, seen as one 5-D tensor whose dimensions are,
// innermost first: column inside a 64-column block (64), head (H, stride one
// row), 64-column block (8, stride 128 bytes), which tensor (2, stride
// `pair_stride_bytes` = address of b minus address of a) and token (T, stride
// H rows). A box of `blocks` column blocks of both tensors for `tokens`
// consecutive tokens lands in shared memory as [token][tensor][block][head][64
// columns], 128-byte swizzled, the same bytes as separate [H x 64] boxes laid
// end to end (a token past T reads zeros). Returns false if the driver refuses
// the encoding (e.g. a stride of 2^40 bytes or more).
inline bool make_tmap_bf16_pair5d(CUtensorMap* m, const void* a, uint64_t pair_stride_bytes,
                                  uint64_t T, uint32_t H, uint32_t blocks, uint32_t tokens = 1) {
    auto fn = encode_tiled_fn();
    if (!fn) return false;
    if (pair_stride_bytes == 0 || pair_stride_bytes % 16 != 0 || pair_stride_bytes >= (uint64_t(1) << 40))
        return false;
    cuuint64_t dims[5] = {64, H, 8, 2, T};
    cuuint64_t strides[4] = {1024, 128, pair_stride_bytes, uint64_t(H) * 1024};
    cuuint32_t box[5] = {64, H, blocks, 2, tokens};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(a), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace smla
