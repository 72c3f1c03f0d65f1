// Device helpers shared by the SIMT kernels of libkata: dtype conversion,
// row loads with the unit-sphere projection, and the packed lift index.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace kata {

constexpr float kSqrt2 = 1.41421356237309504880f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_as(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Rows [r0, r0 + rows) of a [T][P] matrix, each put on the unit sphere
// (x / ||x||, zero stays zero), into dst[r * ld + i] as fp32.  Rows at or
// past T are written as zeros.  Whole block participates, one warp per row.
template <typename Tin, int P>
__device__ __forceinline__ void load_rows_unit(const Tin* __restrict__ src, int r0, int rows, int T,
                                               float* dst, int ld) {
    constexpr int PER_LANE = (P + 31) / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int r = warp; r < rows; r += nwarps) {
        const int t = r0 + r;
        float x[PER_LANE];
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < PER_LANE; ++m) {
            const int i = lane + 32 * m;
            x[m] = (t < T && i < P) ? to_f32(src[(int64_t)t * P + i]) : 0.f;
            ss = fmaf(x[m], x[m], ss);
        }
        ss = warp_sum(ss);
        const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
        for (int m = 0; m < PER_LANE; ++m) {
            const int i = lane + 32 * m;
            if (i < P) dst[r * ld + i] = x[m] * inv;
        }
    }
}

// Rows [r0, r0 + rows) of a [T][DV] matrix as fp32 into dst[r * ld + c];
// rows at or past T become zeros.
template <typename Tin, int DV>
__device__ __forceinline__ void load_rows_plain(const Tin* __restrict__ src, int r0, int rows, int T,
                                                float* dst, int ld) {
    for (int e = threadIdx.x; e < rows * DV; e += blockDim.x) {
        const int r = e / DV, c = e - r * DV, t = r0 + r;
        dst[r * ld + c] = t < T ? to_f32(src[(int64_t)t * DV + c]) : 0.f;
    }
}

// Inverse of the packed index idx(i, j) = i*P - i*(i-1)/2 + (j - i), i <= j.
__device__ __forceinline__ void unpack_index(int a, int P, int& i, int& j) {
    int row = 0, start = 0;
    while (a >= start + (P - row)) {
        start += P - row;
        ++row;
    }
    i = row;
    j = row + (a - start);
}

}  // namespace kata
