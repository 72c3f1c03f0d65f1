// Chunked-state KATA forward on CUDA cores, in the three phases of the
// paper's chunked-scan paragraph: a per-chunk state kernel (one block per
// chunk and packed-row tile), the cumulative pass (scan.cu), and a per-chunk
// output kernel that adds the prefix readout psi(Q_c) [P_c | Pz_c] to the
// local C x C causal part.  fp32 arithmetic for any input dtype; this is the
// path for fp32 inputs and the per-chunk state producer of
// kata_chunk_state_scan.
#include "kata_device.cuh"
#include "kata_internal.h"
#include "simt_output.cuh"

namespace kata {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxC = 128;

// ---------------------------------------------------------------- chunk states
// Block (chunk c, row tile of 64 packed indices, head bh): thread owns one
// packed row a = (i, j) and DV/4 value columns; z is written by column group 0.
constexpr int kRowsPerBlock = 64;

template <int P, int DV>
constexpr size_t state_smem_bytes() {
    return sizeof(float) * (kMaxC * (P + 1) + kMaxC * DV);
}

template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
chunk_states_simt_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v,
                         float* __restrict__ S_loc, float* __restrict__ z_loc, int T, int C, int NC) {
    constexpr int LDP = P + 1, CPT = DV / 4, N = P * (P + 1) / 2;
    extern __shared__ float smem[];
    float* Ks = smem;               // [C][LDP] unit keys
    float* Vs = Ks + kMaxC * LDP;   // [C][DV]
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.z;
    const int t0 = c * C, len = min(C, T - t0);
    load_rows_unit<Tin, P>(k + bh * T * P, t0, len, T, Ks, LDP);
    load_rows_plain<Tin, DV>(v + bh * T * DV, t0, len, T, Vs, DV);
    __syncthreads();

    const int a = blockIdx.y * kRowsPerBlock + (threadIdx.x >> 2), cg = threadIdx.x & 3;
    if (a >= N) return;
    int i, j;
    unpack_index(a, P, i, j);
    const float scale = (i == j) ? 1.f : kSqrt2;
    float acc[CPT];
#pragma unroll
    for (int m = 0; m < CPT; ++m) acc[m] = 0.f;
    float zacc = 0.f;
    for (int s = 0; s < len; ++s) {
        const float psi = Ks[s * LDP + i] * Ks[s * LDP + j] * scale;
        zacc += psi;
#pragma unroll
        for (int m = 0; m < CPT; ++m) acc[m] = fmaf(psi, Vs[s * DV + cg * CPT + m], acc[m]);
    }
    float* dst = S_loc + ((bh * NC + c) * N + a) * DV + cg * CPT;
#pragma unroll
    for (int m = 0; m < CPT; ++m) dst[m] = acc[m];
    if (cg == 0) z_loc[(bh * NC + c) * N + a] = zacc;
}

template <typename Tin, int P, int DV>
cudaError_t states_typed(const void* k, const void* v, float* S, float* z, int BH, int T, int C,
                         cudaStream_t s) {
    constexpr size_t smem = state_smem_bytes<P, DV>();
    constexpr int N = P * (P + 1) / 2;
    auto kern = chunk_states_simt_kernel<Tin, P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int NC = (T + C - 1) / C;
    dim3 grid(NC, (N + kRowsPerBlock - 1) / kRowsPerBlock, BH);
    KATA_TRACED("chunk_states_simt", s,
                kern<<<grid, kThreads, smem, s>>>(static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                                                  S, z, T, C, NC));
    return cudaGetLastError();
}

template <typename Tin, int P, int DV>
cudaError_t output_typed(const void* q, const void* k, const void* v, const float* Pre,
                         const float* Prez, void* o, int BH, int T, int C, cudaStream_t s) {
    constexpr size_t smem = chunk_out::output_smem_bytes<P, DV>();
    auto kern = chunk_out::chunk_output_kernel<Tin, P, DV, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int NC = (T + C - 1) / C;
    dim3 grid(NC, BH);
    KATA_TRACED("chunk_output_simt", s,
                kern<<<grid, chunk_out::kThreads, smem, s>>>(static_cast<const Tin*>(q), static_cast<const Tin*>(k),
                                                             static_cast<const Tin*>(v), nullptr, Pre, Prez,
                                                             static_cast<Tin*>(o), T, C, NC));
    return cudaGetLastError();
}

#define KATA_FOR_SHAPES(X)                                            \
    X(16, 16) X(16, 32) X(16, 64) X(32, 16) X(32, 32) X(32, 64) X(64, 16) \
    X(64, 32) X(64, 64)

template <typename Tin>
cudaError_t states_dispatch(int p, int dv, const void* k, const void* v, float* S, float* z, int BH,
                            int T, int C, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return states_typed<Tin, P_, DV_>(k, v, S, z, BH, T, C, s);
    KATA_FOR_SHAPES(KATA_CASE)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t output_dispatch(int p, int dv, const void* q, const void* k, const void* v,
                            const float* Pre, const float* Prez, void* o, int BH, int T, int C,
                            cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return output_typed<Tin, P_, DV_>(q, k, v, Pre, Prez, o, BH, T, C, s);
    KATA_FOR_SHAPES(KATA_CASE)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunk_states_simt(int dtype, const void* k, const void* v, float* S_loc,
                                     float* z_loc, int BH, int T, int p, int dv, int C,
                                     cudaStream_t s) {
    return dtype == 0 ? states_dispatch<float>(p, dv, k, v, S_loc, z_loc, BH, T, C, s)
                      : states_dispatch<__nv_bfloat16>(p, dv, k, v, S_loc, z_loc, BH, T, C, s);
}

cudaError_t launch_chunk_output_simt(int dtype, const void* q, const void* k, const void* v,
                                     const float* P, const float* Pz, void* o, int BH, int T,
                                     int p, int dv, int C, cudaStream_t s) {
    return dtype == 0 ? output_dispatch<float>(p, dv, q, k, v, P, Pz, o, BH, T, C, s)
                      : output_dispatch<__nv_bfloat16>(p, dv, q, k, v, P, Pz, o, BH, T, C, s);
}

}  // namespace kata
