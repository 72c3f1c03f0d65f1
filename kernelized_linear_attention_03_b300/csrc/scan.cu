// Inter-chunk prefix of chunk states (the cumulative pass of the paper's
// chunked-scan paragraph).  (S_loc, Z_loc) add as vectors, so the exclusive
// prefix over the chunk axis can be taken
//   * sequentially: one thread per 4 state elements walks the N_C chunks
//     (depth N_C, every element's walk independent), or
//   * as a log-depth tree: per 16-byte column vector, a work-efficient
//     up-sweep / down-sweep over runs of 8 or 16 chunks held in registers around
//     a Kogge-Stone scan of the run totals in shared memory (depth log2 of
//     the 256-chunk window plus log2 of the run).  Longer sequences continue
//     window by window from a carry.
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

// Log-depth scan.  A block owns a tile of kTreeTPR x VEC state columns of
// one head and a window of GROUPS x CPT consecutive chunks; thread (g, cc)
// holds the CPT chunks CPT g .. CPT g + CPT - 1 of column group cc in
// registers.
//   1. up-sweep inside the thread: pairwise partial sums, log2 CPT levels;
//   2. inclusive Kogge-Stone over the GROUPS group totals in shared memory,
//      log2(GROUPS) rounds, each GROUPS-wide;
//   3. down-sweep inside the thread, giving each chunk its exclusive prefix
//      within the group, then the group's offset is added.
// Depth log2(CPT) + log2(GROUPS) + log2(CPT) = log2(window) + log2(CPT).
// Windows beyond the first continue from a carry.  Loads
// and stores are full 16-byte vectors along the columns, all CPT of a thread
// in flight at once.
constexpr int kTreeTPR = 4;  // threads across a tile row

template <int VEC, int GROUPS, int CPT>
__global__ void __launch_bounds__(GROUPS * kTreeTPR)
scan_tree_kernel(const float* x, float* y, const float* init, float* fin, int64_t NC, int64_t W,
                 int64_t tiles) {
    using V = Vec<VEC>;
    using T = typename V::T;
    constexpr int kWin = GROUPS * CPT;
    __shared__ T part[2][GROUPS][kTreeTPR];
    const int64_t h = blockIdx.x / tiles, tile = blockIdx.x - h * tiles;
    const int g = threadIdx.x / kTreeTPR, cc = threadIdx.x % kTreeTPR;
    const int64_t e = (tile * kTreeTPR + cc) * VEC;
    const bool col_ok = e < W;  // VEC = 4 only when W % 4 == 0
    T carry = (init && col_ok) ? *reinterpret_cast<const T*>(init + h * W + e) : V::zero();
    const float* src = x + h * NC * W + e;
    float* dst = y + h * NC * W + e;
    for (int64_t w0 = 0; w0 < NC; w0 += kWin) {
        const int64_t c0 = w0 + (int64_t)g * CPT;
        T a[CPT];
#pragma unroll
        for (int m = 0; m < CPT; ++m)
            a[m] = (col_ok && c0 + m < NC) ? *reinterpret_cast<const T*>(src + (c0 + m) * W) : V::zero();
        // up-sweep
#pragma unroll
        for (int st = 1; st < CPT; st <<= 1)
#pragma unroll
            for (int i = 2 * st - 1; i < CPT; i += 2 * st) a[i] = V::add(a[i - st], a[i]);
        // group totals
        int buf = 0;
        part[0][g][cc] = a[CPT - 1];
        __syncthreads();
#pragma unroll
        for (int d = 1; d < GROUPS; d <<= 1) {
            T v = part[buf][g][cc];
            if (g >= d) v = V::add(part[buf][g - d][cc], v);
            part[buf ^ 1][g][cc] = v;
            buf ^= 1;
            __syncthreads();
        }
        const T offset = V::add(carry, g > 0 ? part[buf][g - 1][cc] : V::zero());
        const T wtotal = part[buf][GROUPS - 1][cc];
        // down-sweep: exclusive prefixes within the thread
        a[CPT - 1] = V::zero();
#pragma unroll
        for (int st = CPT / 2; st >= 1; st >>= 1)
#pragma unroll
            for (int i = 2 * st - 1; i < CPT; i += 2 * st) {
                const T left = a[i - st];
                a[i - st] = a[i];
                a[i] = V::add(a[i], left);
            }
#pragma unroll
        for (int m = 0; m < CPT; ++m)
            if (col_ok && c0 + m < NC) *reinterpret_cast<T*>(dst + (c0 + m) * W) = V::add(offset, a[m]);
        carry = V::add(carry, wtotal);
        __syncthreads();  // part[] is rewritten by the next window
    }
    if (fin && col_ok) *reinterpret_cast<T*>(fin + h * W + e) = carry;
}

template <int VEC, int GROUPS, int CPT>
cudaError_t launch_tree(const float* x, float* y, const float* init, float* fin, int64_t heads, int64_t NC,
                        int64_t W, cudaStream_t s) {
    const int64_t tiles = (W + kTreeTPR * VEC - 1) / (kTreeTPR * VEC);
    KATA_TRACED("scan_tree", s,
                (scan_tree_kernel<VEC, GROUPS, CPT><<<(unsigned)(heads * tiles), GROUPS * kTreeTPR, 0, s>>>(
                    x, y, init, fin, NC, W, tiles)));
    return cudaGetLastError();
}

template <int VEC>
cudaError_t launch_tree_vec(const float* x, float* y, const float* init, float* fin, int64_t heads, int64_t NC,
                            int64_t W, cudaStream_t s) {
    // small blocks keep the most copies in flight per SM; sequences past 256
    // chunks chain 256-chunk windows
    if (NC <= 64) return launch_tree<VEC, 8, 8>(x, y, init, fin, heads, NC, W, s);
    if (NC <= 256) return launch_tree<VEC, 32, 8>(x, y, init, fin, heads, NC, W, s);
    return launch_tree<VEC, 16, 16>(x, y, init, fin, heads, NC, W, s);
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

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
    const bool vec4 = W % 4 == 0 && aligned16(x) && aligned16(y) && aligned16(init) && aligned16(fin);
    if (vec4) return launch_tree_vec<4>(x, y, init, fin, heads, NC, W, s);
    return launch_tree_vec<1>(x, y, init, fin, heads, NC, W, s);
}

cudaError_t launch_copy_or_zero(const float* src, float* dst, int64_t count, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    KATA_TRACED("copy_or_zero", s, copy_or_zero_kernel<<<(unsigned)((count + 255) / 256), 256, 0, s>>>(src, dst, count));
    return cudaGetLastError();
}

}  // namespace kata
