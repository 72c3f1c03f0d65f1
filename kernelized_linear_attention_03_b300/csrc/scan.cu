// Inter-chunk prefix of chunk states (the cumulative pass of the paper's
// chunked-scan paragraph).  (S_loc, Z_loc) add as vectors, so the exclusive
// prefix over the chunk axis can be taken
//   * sequentially: one thread per 4 state elements walks the N_C chunks
//     (depth N_C, every element's walk independent), or
//   * as a log-depth scan: a block stages an [N_C x 16] slab of one head's
//     state in shared memory and runs ceil(log2 N_C) rounds in which every
//     chunk adds the chunk 2^d before it (N_C-wide work per round), then
//     writes the exclusive prefix.  Chunk counts above the slab window are
//     walked window by window with a carry.
// Both read every element once and write it once: the pass is HBM-bound.
#include <cstdint>

#include "kata_internal.h"

namespace kata {
namespace {

constexpr int kSeqThreads = 256;

template <int VEC>
struct Vec;
template <>
struct Vec<4> {
    using T = float4;
    static __device__ __forceinline__ float4 zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ float4 add(float4 a, float4 b) {
        return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    }
};
template <>
struct Vec<1> {
    using T = float;
    static __device__ __forceinline__ float zero() { return 0.f; }
    static __device__ __forceinline__ float add(float a, float b) { return a + b; }
};

// x and y may be the same buffer: every element's loads precede its stores.
template <int VEC>
__global__ void __launch_bounds__(kSeqThreads)
scan_sequential_kernel(const float* x, float* y, const float* init, float* fin, int64_t heads,
                       int64_t NC, int64_t W) {
    using V = Vec<VEC>;
    using T = typename V::T;
    const int64_t per_head = W / VEC;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= heads * per_head) return;
    const int64_t h = gid / per_head, e = (gid - h * per_head) * VEC;
    T run = init ? *reinterpret_cast<const T*>(init + h * W + e) : V::zero();
    const float* src = x + h * NC * W + e;
    float* dst = y + h * NC * W + e;
    int64_t c = 0;
    for (; c + 4 <= NC; c += 4) {
        T a0 = *reinterpret_cast<const T*>(src + (c + 0) * W);
        T a1 = *reinterpret_cast<const T*>(src + (c + 1) * W);
        T a2 = *reinterpret_cast<const T*>(src + (c + 2) * W);
        T a3 = *reinterpret_cast<const T*>(src + (c + 3) * W);
        *reinterpret_cast<T*>(dst + (c + 0) * W) = run;
        run = V::add(run, a0);
        *reinterpret_cast<T*>(dst + (c + 1) * W) = run;
        run = V::add(run, a1);
        *reinterpret_cast<T*>(dst + (c + 2) * W) = run;
        run = V::add(run, a2);
        *reinterpret_cast<T*>(dst + (c + 3) * W) = run;
        run = V::add(run, a3);
    }
    for (; c < NC; ++c) {
        T a = *reinterpret_cast<const T*>(src + c * W);
        *reinterpret_cast<T*>(dst + c * W) = run;
        run = V::add(run, a);
    }
    if (fin) *reinterpret_cast<T*>(fin + h * W + e) = run;
}

constexpr int kTreeThreads = 256;
constexpr int kTreeE = 16;       // state elements per slab column group
constexpr int kTreeWin = 1024;   // chunks per shared-memory window
constexpr int kTreePer = kTreeWin * kTreeE / kTreeThreads;

// Block = (element group g of head h).  Slab sx[c][e] for the current window.
__global__ void __launch_bounds__(kTreeThreads)
scan_tree_kernel(const float* x, float* y, const float* init, float* fin, int64_t NC, int64_t W,
                 int64_t groups) {
    extern __shared__ float sx[];  // [kTreeWin][kTreeE]
    __shared__ float carry[kTreeE];
    const int64_t h = blockIdx.x / groups, g = blockIdx.x - h * groups;
    const int64_t e0 = g * kTreeE;
    const int tid = threadIdx.x;
    if (tid < kTreeE) carry[tid] = (init && e0 + tid < W) ? init[h * W + e0 + tid] : 0.f;
    for (int64_t w0 = 0; w0 < NC; w0 += kTreeWin) {
        const int len = (int)((NC - w0) < kTreeWin ? (NC - w0) : kTreeWin);
        __syncthreads();
        for (int idx = tid; idx < len * kTreeE; idx += kTreeThreads) {
            const int c = idx / kTreeE, e = idx - c * kTreeE;
            sx[idx] = (e0 + e < W) ? x[(h * NC + w0 + c) * W + e0 + e] : 0.f;
        }
        __syncthreads();
        for (int d = 1; d < len; d <<= 1) {
            float tmp[kTreePer];
#pragma unroll
            for (int m = 0; m < kTreePer; ++m) {
                const int idx = tid + m * kTreeThreads;
                tmp[m] = (idx < len * kTreeE && idx / kTreeE >= d) ? sx[idx - d * kTreeE] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int m = 0; m < kTreePer; ++m) {
                const int idx = tid + m * kTreeThreads;
                if (idx < len * kTreeE) sx[idx] += tmp[m];
            }
            __syncthreads();
        }
        for (int idx = tid; idx < len * kTreeE; idx += kTreeThreads) {
            const int c = idx / kTreeE, e = idx - c * kTreeE;
            if (e0 + e < W) y[(h * NC + w0 + c) * W + e0 + e] = carry[e] + (c > 0 ? sx[idx - kTreeE] : 0.f);
        }
        __syncthreads();
        if (tid < kTreeE) carry[tid] += sx[(len - 1) * kTreeE + tid];
    }
    __syncthreads();
    if (fin && tid < kTreeE && e0 + tid < W) fin[h * W + e0 + tid] = carry[tid];
}

__global__ void copy_or_zero_kernel(const float* src, float* dst, int64_t count) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) dst[i] = src ? src[i] : 0.f;
}

}  // namespace

cudaError_t launch_scan(int mode, const float* x, float* y, const float* init, float* fin,
                        int64_t heads, int64_t NC, int64_t W, cudaStream_t s) {
    if (heads <= 0 || W <= 0) return cudaSuccess;
    if (mode == 0) {
        const bool vec4 = (W % 4 == 0);
        const int64_t threads = heads * (vec4 ? W / 4 : W);
        const int64_t blocks = (threads + kSeqThreads - 1) / kSeqThreads;
        if (vec4)
            KATA_TRACED("scan_sequential", s,
                        scan_sequential_kernel<4><<<(unsigned)blocks, kSeqThreads, 0, s>>>(x, y, init, fin,
                                                                                          heads, NC, W));
        else
            KATA_TRACED("scan_sequential", s,
                        scan_sequential_kernel<1><<<(unsigned)blocks, kSeqThreads, 0, s>>>(x, y, init, fin,
                                                                                          heads, NC, W));
        return cudaGetLastError();
    }
    const size_t smem = sizeof(float) * kTreeWin * kTreeE;
    cudaError_t e = cudaFuncSetAttribute(scan_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t groups = (W + kTreeE - 1) / kTreeE;
    KATA_TRACED("scan_tree", s,
                scan_tree_kernel<<<(unsigned)(heads * groups), kTreeThreads, smem, s>>>(x, y, init, fin, NC, W,
                                                                                         groups));
    return cudaGetLastError();
}

cudaError_t launch_copy_or_zero(const float* src, float* dst, int64_t count, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    KATA_TRACED("copy_or_zero", s, copy_or_zero_kernel<<<(unsigned)((count + 255) / 256), 256, 0, s>>>(src, dst, count));
    return cudaGetLastError();
}

}  // namespace kata
