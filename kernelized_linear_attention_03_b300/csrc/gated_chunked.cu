// Gated chunked forward (fp32 accumulation, any input dtype; for bf16 inputs
// the local states run on the tensor cores, the rest on CUDA cores).
// One scalar gate gamma_t in [0, 1] per head and token scales the running
// state before the token's own term is added,
//   S_t = gamma_t S_{t-1} + psi(kh_t) v_t^T,   z_t = gamma_t z_{t-1} + psi(kh_t),
// and the readout is unchanged.  The three phases of the chunked form carry
// decays (all as direct products of gates, so a zero gate is exact):
//   local state  X_c = sum_{s in c} (prod_{r=s+1..end_c} gamma_r) psi(kh_s) v_s^T,
//   chunk decay  a_c = prod_{r in c} gamma_r,
//   prefix       P_0 = S0,  P_{c+1} = a_c P_c + X_c   (one step per chunk),
//   output       num_t = (prod_{r=c C..t} gamma_r) psi(qh_t)^T P_c
//                        + sum_{s in c, s<=t} (prod_{r=s+1..t} gamma_r) (qh_t.kh_s)^2 v_s,
//                den_t likewise with 1 for v_s.
// Local states: bf16, the tensor-core chunk-state kernel with each token's key
// lift weighted by its decay to the chunk's end (gate_decay_kernel); fp32, a
// CUDA-core kernel.  Output: the register-tiled kernel of simt_output.cuh.
#include <type_traits>

#include "kata_device.cuh"
#include "kata_internal.h"
#include "simt_output.cuh"

namespace kata {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxC = 128;
constexpr int kRowsPerBlock = 64;

// ---------------------------------------------------------------- chunk states
template <int P, int DV>
constexpr size_t state_smem_bytes() {
    return sizeof(float) * (kMaxC * (P + 1) + kMaxC * DV + kMaxC);
}

// Block (chunk c, tile of 64 packed rows, head bh); also writes the chunk
// decay a_c (block y = 0, thread 0).
template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
gated_states_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v, const float* __restrict__ gate,
                    float* __restrict__ X, float* __restrict__ Xz, float* __restrict__ a, int T, int C, int NC) {
    constexpr int LDP = P + 1, CPT = DV / 4, N = P * (P + 1) / 2;
    extern __shared__ float smem[];
    float* Ks = smem;              // [C][LDP] unit keys
    float* Vs = Ks + kMaxC * LDP;  // [C][DV]
    float* dec = Vs + kMaxC * DV;  // [C] decay from token s to the chunk's end
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.z;
    const int t0 = c * C, len = min(C, T - t0);
    load_rows_unit<Tin, P>(k + bh * T * P, t0, len, T, Ks, LDP);
    load_rows_plain<Tin, DV>(v + bh * T * DV, t0, len, T, Vs, DV);
    if (threadIdx.x == 0) {
        const float* g = gate + bh * T + t0;
        float d = 1.f;
        for (int s = len - 1; s >= 0; --s) {
            dec[s] = d;  // prod_{r=s+1..len-1} gamma
            d *= g[s];
        }
        if (blockIdx.y == 0) a[bh * NC + c] = d;  // prod over the whole chunk
    }
    __syncthreads();

    const int r = blockIdx.y * kRowsPerBlock + (threadIdx.x >> 2), cg = threadIdx.x & 3;
    if (r >= N) return;
    int i, j;
    unpack_index(r, P, i, j);
    const float scale = (i == j) ? 1.f : kSqrt2;
    float acc[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x) acc[x] = 0.f;
    float zacc = 0.f;
    for (int s = 0; s < len; ++s) {
        const float psi = dec[s] * Ks[s * LDP + i] * Ks[s * LDP + j] * scale;
        zacc += psi;
#pragma unroll
        for (int x = 0; x < CPT; ++x) acc[x] = fmaf(psi, Vs[s * DV + cg * CPT + x], acc[x]);
    }
    float* dst = X + ((bh * NC + c) * N + r) * DV + cg * CPT;
#pragma unroll
    for (int x = 0; x < CPT; ++x) dst[x] = acc[x];
    if (cg == 0) Xz[(bh * NC + c) * N + r] = zacc;
}

// ---------------------------------------------------------------- gated prefix
// x [heads][NC][W] -> exclusive gated prefix in place: y_c = P_c with P_0 =
// init (or 0) and P_{c+1} = a_c P_c + x_c; fin (or null) receives P_NC.
// One thread per VEC consecutive columns, one step per chunk; the values of
// kBatch chunks are loaded before any of them is overwritten, so that the
// loads of a batch are in flight together (each step's store would otherwise
// hold back the next chunk's load).
constexpr int kBatch = 8;

template <int VEC>
__global__ void gated_scan_kernel(float* __restrict__ x, const float* __restrict__ a, const float* __restrict__ init,
                                  float* __restrict__ fin, int64_t heads, int64_t NC, int64_t W) {
    const int64_t per_head = W / VEC;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= heads * per_head) return;
    const int64_t h = gid / per_head, e = (gid - h * per_head) * VEC;
    float run[VEC];
#pragma unroll
    for (int u = 0; u < VEC; ++u) run[u] = init ? init[h * W + e + u] : 0.f;
    float* col = x + h * NC * W + e;
    const float* ah = a + h * NC;
    for (int64_t c0 = 0; c0 < NC; c0 += kBatch) {
        float xv[kBatch][VEC], av[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const bool live = c0 + b < NC;
            av[b] = live ? ah[c0 + b] : 0.f;
            if (VEC == 4) {
                const float4 t = live ? *reinterpret_cast<const float4*>(col + (c0 + b) * W) : make_float4(0.f, 0.f, 0.f, 0.f);
                xv[b][0] = t.x;
                xv[b][VEC > 1 ? 1 : 0] = t.y;
                xv[b][VEC > 2 ? 2 : 0] = t.z;
                xv[b][VEC > 3 ? 3 : 0] = t.w;
            } else {
#pragma unroll
                for (int u = 0; u < VEC; ++u) xv[b][u] = live ? col[(c0 + b) * W + u] : 0.f;
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            if (c0 + b >= NC) break;
            if (VEC == 4) {
                *reinterpret_cast<float4*>(col + (c0 + b) * W) =
                    make_float4(run[0], run[VEC > 1 ? 1 : 0], run[VEC > 2 ? 2 : 0], run[VEC > 3 ? 3 : 0]);
            } else {
#pragma unroll
                for (int u = 0; u < VEC; ++u) col[(c0 + b) * W + u] = run[u];
            }
#pragma unroll
            for (int u = 0; u < VEC; ++u) run[u] = fmaf(av[b], run[u], xv[b][u]);
        }
    }
    if (fin) {
#pragma unroll
        for (int u = 0; u < VEC; ++u) fin[h * W + e + u] = run[u];
    }
}

// ---------------------------------------------------------------- decays for the tensor-core chunk states
// One warp per (chunk c, head bh): dec[t] = prod_{r=t+1..end_c} gamma_r for the
// chunk's tokens and a[c] = prod over the chunk (fp32 products; a zero gate
// gives exact zeros).  Each lane takes up to kMaxC / 32 consecutive tokens; the
// lanes' products are combined by a suffix product across the warp.
__global__ void __launch_bounds__(32)
gate_decay_kernel(const float* __restrict__ gate, float* __restrict__ dec, float* __restrict__ a, int T, int C, int NC) {
    constexpr int kPer = kMaxC / 32;
    const int c = blockIdx.x, lane = threadIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * C, len = min(C, T - t0), per = (C + 31) / 32;
    float gl[kPer];
    float tot = 1.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int s = lane * per + i;
        gl[i] = (i < per && s < len) ? gate[bh * T + t0 + s] : 1.f;
        tot *= gl[i];
    }
    float incl = tot;  // product of this lane's gates and every later lane's
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float later = __shfl_down_sync(0xffffffffu, incl, d);
        if (lane + d < 32) incl *= later;
    }
    float run = __shfl_down_sync(0xffffffffu, incl, 1);
    if (lane == 31) run = 1.f;
#pragma unroll
    for (int i = kPer - 1; i >= 0; --i) {
        const int s = lane * per + i;
        if (i < per && s < len) dec[bh * T + t0 + s] = run;
        run *= gl[i];
    }
    if (lane == 0) a[bh * NC + c] = incl;
}

template <typename Tin, int P, int DV>
cudaError_t gated_typed(const void* q, const void* k, const void* v, const float* gate, void* o, float* X, float* Xz,
                        float* a, float* dec, const float* S0, const float* z0, float* S_final, float* z_final, int BH,
                        int T, int C, cudaStream_t s) {
    constexpr int N = P * (P + 1) / 2;
    const int NC = (T + C - 1) / C;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        // bf16: the chunk states on the tensor cores (the chunk-state kernel,
        // each token's key lift weighted by its decay to the chunk's end)
        KATA_TRACED("gate_decay", s, (gate_decay_kernel<<<dim3(NC, BH), 32, 0, s>>>(gate, dec, a, T, C, NC)));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if ((e = launch_states_tc(k, v, X, Xz, BH, T, P, DV, C, NC, NC, 0, 1, s, dec)) != cudaSuccess) return e;
    } else {
        constexpr size_t smem = state_smem_bytes<P, DV>();
        auto kern = gated_states_kernel<Tin, P, DV>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        KATA_TRACED("gated_states_simt", s,
                    kern<<<dim3(NC, (N + kRowsPerBlock - 1) / kRowsPerBlock, BH), kThreads, smem, s>>>(
                        static_cast<const Tin*>(k), static_cast<const Tin*>(v), gate, X, Xz, a, T, C, NC));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    for (int part = 0; part < 2; ++part) {
        const int64_t W = part == 0 ? (int64_t)N * DV : N;
        float* xs = part == 0 ? X : Xz;
        const float* init = part == 0 ? S0 : z0;
        float* fin = part == 0 ? S_final : z_final;
        auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
        if (W % 4 == 0 && a16(xs)) {
            const int64_t threads = (int64_t)BH * (W / 4);
            KATA_TRACED("gated_scan", s,
                        (gated_scan_kernel<4><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(xs, a, init, fin, BH, NC, W)));
        } else {
            const int64_t threads = (int64_t)BH * W;
            KATA_TRACED("gated_scan", s,
                        (gated_scan_kernel<1><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(xs, a, init, fin, BH, NC, W)));
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    constexpr size_t smem = chunk_out::output_smem_bytes<P, DV>();
    auto kern = chunk_out::chunk_output_kernel<Tin, P, DV, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    KATA_TRACED("gated_output_simt", s,
                kern<<<dim3(NC, BH), chunk_out::kThreads, smem, s>>>(static_cast<const Tin*>(q), static_cast<const Tin*>(k),
                                                          static_cast<const Tin*>(v), gate, X, Xz,
                                                          static_cast<Tin*>(o), T, C, NC));
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t gated_dispatch(int p, int dv, const void* q, const void* k, const void* v, const float* gate, void* o,
                           float* X, float* Xz, float* a, float* dec, const float* S0, const float* z0, float* S_final,
                           float* z_final, int BH, int T, int C, cudaStream_t s) {
#define KATA_CASE(P_, DV_)                                                                                      \
    if (p == P_ && dv == DV_)                                                                                   \
        return gated_typed<Tin, P_, DV_>(q, k, v, gate, o, X, Xz, a, dec, S0, z0, S_final, z_final, BH, T, C, s);
    KATA_CASE(16, 16) KATA_CASE(16, 32) KATA_CASE(16, 64)
    KATA_CASE(32, 16) KATA_CASE(32, 32) KATA_CASE(32, 64)
    KATA_CASE(64, 16) KATA_CASE(64, 32) KATA_CASE(64, 64)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunked_gated(int dtype, const void* q, const void* k, const void* v, const float* gate, void* o,
                                 float* X, float* Xz, float* a, float* dec, const float* S0, const float* z0,
                                 float* S_final, float* z_final, int BH, int T, int p, int dv, int C, cudaStream_t s) {
    return dtype == 0 ? gated_dispatch<float>(p, dv, q, k, v, gate, o, X, Xz, a, dec, S0, z0, S_final, z_final, BH, T,
                                              C, s)
                      : gated_dispatch<__nv_bfloat16>(p, dv, q, k, v, gate, o, X, Xz, a, dec, S0, z0, S_final, z_final,
                                                      BH, T, C, s);
}

}  // namespace kata
