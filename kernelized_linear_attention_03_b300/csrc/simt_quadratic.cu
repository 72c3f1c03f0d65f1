// Flash-style O(T^2) KATA forward on CUDA cores (fp32 arithmetic, any input
// dtype): the flash-attention-style forward of the paper's abstract,
// o_t = sum_{s<=t} (qh_t.kh_s)^2 v_s / sum_{s<=t} (qh_t.kh_s)^2.
// Scores of unit vectors lie in [0, 1], so no running maximum or rescale
// is needed.  Serves the fp32 inputs and shapes the tensor-core path does
// not take.
#include "kata_device.cuh"
#include "kata_internal.h"

namespace kata {
namespace {

constexpr int kBQ = 64;        // queries per block
constexpr int kBK = 64;        // keys per tile
constexpr int kThreads = 256;  // 64 rows x 4 column groups

template <int P, int DV>
constexpr size_t quad_smem_bytes() {
    return sizeof(float) * (kBQ * (P + 1) + kBK * (P + 1) + kBK * DV + kBQ * (kBK + 1));
}

template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
quadratic_simt_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                      const Tin* __restrict__ v, Tin* __restrict__ o, int T) {
    constexpr int LDP = P + 1, LDS = kBK + 1, CPT = DV / 4;
    extern __shared__ float smem[];
    float* Qs = smem;               // [kBQ][LDP] unit queries
    float* Ks = Qs + kBQ * LDP;     // [kBK][LDP] unit keys
    float* Vs = Ks + kBK * LDP;     // [kBK][DV]
    float* Ss = Vs + kBK * DV;      // [kBQ][LDS] masked squared scores

    const int qt = gridDim.x - 1 - blockIdx.x;  // heaviest query tiles first
    const int64_t bh = blockIdx.y;
    const Tin* qh = q + bh * T * P;
    const Tin* kh = k + bh * T * P;
    const Tin* vh = v + bh * T * DV;
    load_rows_unit<Tin, P>(qh, qt * kBQ, kBQ, T, Qs, LDP);

    const int r = threadIdx.x >> 2, cg = threadIdx.x & 3;
    const int qi = qt * kBQ + r;
    float acc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) acc[c] = 0.f;
    float den = 0.f;

    for (int kt = 0; kt <= qt; ++kt) {
        __syncthreads();
        load_rows_unit<Tin, P>(kh, kt * kBK, kBK, T, Ks, LDP);
        load_rows_plain<Tin, DV>(vh, kt * kBK, kBK, T, Vs, DV);
        __syncthreads();
#pragma unroll 4
        for (int m = 0; m < kBK / 4; ++m) {
            const int j = cg + 4 * m, kj = kt * kBK + j;
            float d = 0.f;
#pragma unroll
            for (int i = 0; i < P; ++i) d = fmaf(Qs[r * LDP + i], Ks[j * LDP + i], d);
            Ss[r * LDS + j] = (kj <= qi && kj < T) ? d * d : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < kBK; ++j) {
            const float s = Ss[r * LDS + j];
            den += s;
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[c] = fmaf(s, Vs[j * DV + cg * CPT + c], acc[c]);
        }
    }
    if (qi < T) {
        Tin* oh = o + (bh * T + qi) * DV + cg * CPT;
#pragma unroll
        for (int c = 0; c < CPT; ++c) store_as(oh + c, den > 0.f ? acc[c] / den : 0.f);
    }
}

template <typename Tin, int P, int DV>
cudaError_t launch_typed(const void* q, const void* k, const void* v, void* o, int BH, int T,
                         cudaStream_t s) {
    constexpr size_t smem = quad_smem_bytes<P, DV>();
    auto kern = quadratic_simt_kernel<Tin, P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((T + kBQ - 1) / kBQ, BH);
    KATA_TRACED("quadratic_simt", s,
                kern<<<grid, kThreads, smem, s>>>(static_cast<const Tin*>(q), static_cast<const Tin*>(k),
                                                  static_cast<const Tin*>(v), static_cast<Tin*>(o), T));
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t dispatch(int p, int dv, const void* q, const void* k, const void* v, void* o, int BH,
                     int T, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return launch_typed<Tin, P_, DV_>(q, k, v, o, BH, T, s);
    KATA_CASE(16, 16) KATA_CASE(16, 32) KATA_CASE(16, 64)
    KATA_CASE(32, 16) KATA_CASE(32, 32) KATA_CASE(32, 64)
    KATA_CASE(64, 16) KATA_CASE(64, 32) KATA_CASE(64, 64)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_quadratic_simt(int dtype, const void* q, const void* k, const void* v, void* o,
                                  int BH, int T, int p, int dv, cudaStream_t s) {
    return dtype == 0 ? dispatch<float>(p, dv, q, k, v, o, BH, T, s)
                      : dispatch<__nv_bfloat16>(p, dv, q, k, v, o, BH, T, s);
}

}  // namespace kata
