// Host side of the TMA tile copies: tensor maps of the bf16 [BH][T][cols]
// arrays the tensor-core kernels stream in 128-row boxes, and of the fp32
// accumulation rows they reduce into.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace kata {
namespace tc {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda); null if unavailable.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess && qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map of a bf16 [BH][T][cols] array read as 128-row x 64-column boxes
// (128-byte rows, 128-byte swizzle: the layout the kernel's operand tiles
// use; columns past `cols` and rows past T are filled with zeros).
inline bool rows_map(CUtensorMap* m, const void* base, int cols, int T, int BH) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)T * cols * 2};
    cuuint32_t box[3] = {64, 128u, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of transposed keys, bf16 [BH][chunks][P][row] (row d of a chunk
// = dimension d over its 128 tokens, then `row` - 128 pad elements), read as
// boxes of P rows x 64 tokens (128-byte rows, 128-byte swizzle): two boxes
// per chunk.
inline bool kt_map(CUtensorMap* m, const void* base, int P, int chunks, int BH, int row) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)row, (cuuint64_t)chunks * P, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)row * 2, (cuuint64_t)chunks * P * row * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)P, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same transposed keys read as one box per chunk: P rows x `row`
// elements, no swizzle (the rows land in shared memory `row` * 2 bytes apart,
// pad included).
inline bool kt_rows_map(CUtensorMap* m, const void* base, int P, int chunks, int BH, int row) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)row, (cuuint64_t)chunks * P, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)row * 2, (cuuint64_t)chunks * P * row * 2};
    cuuint32_t box[3] = {(cuuint32_t)row, (cuuint32_t)P, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of an fp32 [BH][Tc][cols] accumulation array written by boxes
// of 128 rows x w columns (w = 32: 128-byte rows, 128-byte swizzle; w = 16:
// 64-byte rows, no swizzle); cols is a multiple of w.
inline bool acc_map(CUtensorMap* m, const void* base, int cols, int w, int Tc, int BH) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)Tc, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)Tc * cols * 4};
    cuuint32_t box[3] = {(cuuint32_t)w, 128u, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, w == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace kata
