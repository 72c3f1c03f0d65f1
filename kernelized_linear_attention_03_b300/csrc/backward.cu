// Backward of the KATA forward on CUDA cores (fp32 arithmetic, any input
// dtype), by the chain rule through the definition
//   o_t = N_t / D_t,  N_t = sum_{s<=t} w_ts v_s,  D_t = sum_{s<=t} w_ts,
//   w_ts = c_ts^2,  c_ts = qh_t . kh_s,  qh = q/||q||,  kh = k/||k||.
// With G_t = dL/do_t and delta_t = G_t . o_t:
//   dv_s  = sum_{t>=s} (w_ts / D_t) G_t
//   dc_ts = 2 c_ts (G_t . v_s - delta_t) / D_t
//   dqh_t = sum_{s<=t} dc_ts kh_s,   dkh_s = sum_{t>=s} dc_ts qh_t
//   dq_t  = (dqh_t - (qh_t . dqh_t) qh_t) / ||q_t||   (k likewise).
// Rows with D_t = 0 pass no gradient; zero q or k vectors receive none.
// Flash-style, O(T^2): a row pass per query tile (D_t and delta_t, then
// dq_t) and a column pass per key tile (dv_s, dk_s), each walking the tiles
// of the causal triangle.
#include "kata_device.cuh"
#include "kata_internal.h"

namespace kata {
namespace {

constexpr int kBT = 64;        // rows per tile (queries or keys)
constexpr int kThreads = 256;  // 64 rows x 4 column groups

// Rows [r0, r0 + kBT) of a [T][P] matrix on the unit sphere into dst (ld
// P + 1) and their norms into nrm; rows past T are zero.  One warp per row.
template <typename Tin, int P>
__device__ __forceinline__ void load_unit_rows_norm(const Tin* __restrict__ src, int r0, int T, float* dst,
                                                    float* nrm) {
    constexpr int PER_LANE = (P + 31) / 32, LDP = P + 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int r = warp; r < kBT; r += nwarps) {
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
        const float n = ss > 0.f ? sqrtf(ss) : 0.f;
        const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
        for (int m = 0; m < PER_LANE; ++m) {
            const int i = lane + 32 * m;
            if (i < P) dst[r * LDP + i] = x[m] * inv;
        }
        if (lane == 0) nrm[r] = n;
    }
}

template <int P, int DV>
constexpr size_t rows_smem_bytes() {
    // Qs, Ks [kBT][P+1]; Vs, Gs [kBT][DV]; Cs, Xs [kBT][kBT+1]; qn, Dsh, dsh [kBT]
    return sizeof(float) * (2 * kBT * (P + 1) + 2 * kBT * DV + 2 * kBT * (kBT + 1) + 3 * kBT);
}

// Row pass.  Block (query tile qt, head bh); thread (r, cg) owns query r of
// the tile, value columns [cg DV/4, (cg+1) DV/4) and lift coordinates
// [cg P/4, (cg+1) P/4).
template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_rows_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                const Tin* __restrict__ dO, Tin* __restrict__ dq, float* __restrict__ Dout,
                float* __restrict__ delta_out, int T) {
    constexpr int LDP = P + 1, LDS = kBT + 1, CV = DV / 4, CP = P / 4;
    extern __shared__ float smem[];
    float* Qs = smem;
    float* Ks = Qs + kBT * LDP;
    float* Vs = Ks + kBT * LDP;
    float* Gs = Vs + kBT * DV;
    float* Cs = Gs + kBT * DV;
    float* Xs = Cs + kBT * LDS;
    float* qn = Xs + kBT * LDS;
    float* Dsh = qn + kBT;
    float* dsh = Dsh + kBT;

    const int qt = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const Tin* qh = q + bh * T * P;
    const Tin* kh = k + bh * T * P;
    const Tin* vh = v + bh * T * DV;
    const int r = threadIdx.x >> 2, cg = threadIdx.x & 3;
    const int qi = qt * kBT + r;
    load_unit_rows_norm<Tin, P>(qh, qt * kBT, T, Qs, qn);
    load_rows_plain<Tin, DV>(dO + bh * T * DV, qt * kBT, kBT, T, Gs, DV);

    // ---- pass A: D_t and o_t, then delta_t = G_t . o_t
    float num[CV];
#pragma unroll
    for (int x = 0; x < CV; ++x) num[x] = 0.f;
    float den = 0.f;
    for (int kt = 0; kt <= qt; ++kt) {
        __syncthreads();
        load_rows_unit<Tin, P>(kh, kt * kBT, kBT, T, Ks, LDP);
        load_rows_plain<Tin, DV>(vh, kt * kBT, kBT, T, Vs, DV);
        __syncthreads();
        for (int m = 0; m < kBT / 4; ++m) {
            const int j = cg + 4 * m, kj = kt * kBT + j;
            float c = 0.f;
#pragma unroll
            for (int i = 0; i < P; ++i) c = fmaf(Qs[r * LDP + i], Ks[j * LDP + i], c);
            Cs[r * LDS + j] = (kj <= qi && kj < T) ? c : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < kBT; ++j) {
            const float c = Cs[r * LDS + j], w = c * c;
            den += w;
#pragma unroll
            for (int x = 0; x < CV; ++x) num[x] = fmaf(w, Vs[j * DV + cg * CV + x], num[x]);
        }
    }
    float dpart = 0.f;
    if (den > 0.f) {
        const float inv = 1.f / den;
#pragma unroll
        for (int x = 0; x < CV; ++x) dpart = fmaf(Gs[r * DV + cg * CV + x], num[x] * inv, dpart);
    }
    // the four column groups of a query are lanes 4r .. 4r + 3 of one warp
    dpart += __shfl_xor_sync(0xffffffffu, dpart, 1);
    dpart += __shfl_xor_sync(0xffffffffu, dpart, 2);
    if (cg == 0) {
        Dsh[r] = den;
        dsh[r] = dpart;
        if (qi < T) {
            Dout[bh * T + qi] = den;
            delta_out[bh * T + qi] = dpart;
        }
    }

    // ---- pass B: dqh_t = sum_s dc_ts kh_s
    float gq[CP];
#pragma unroll
    for (int x = 0; x < CP; ++x) gq[x] = 0.f;
    for (int kt = 0; kt <= qt; ++kt) {
        __syncthreads();
        load_rows_unit<Tin, P>(kh, kt * kBT, kBT, T, Ks, LDP);
        load_rows_plain<Tin, DV>(vh, kt * kBT, kBT, T, Vs, DV);
        __syncthreads();
        for (int m = 0; m < kBT / 4; ++m) {
            const int j = cg + 4 * m, kj = kt * kBT + j;
            float c = 0.f, gv = 0.f;
#pragma unroll
            for (int i = 0; i < P; ++i) c = fmaf(Qs[r * LDP + i], Ks[j * LDP + i], c);
#pragma unroll
            for (int x = 0; x < DV; ++x) gv = fmaf(Gs[r * DV + x], Vs[j * DV + x], gv);
            const bool live = kj <= qi && kj < T;
            Cs[r * LDS + j] = live ? c : 0.f;
            Xs[r * LDS + j] = live ? gv : 0.f;
        }
        __syncthreads();
        const float D = Dsh[r];
        if (D > 0.f) {
            const float invD = 1.f / D, dl = dsh[r];
            for (int j = 0; j < kBT; ++j) {
                const float c = Cs[r * LDS + j];
                const float dc = 2.f * c * (Xs[r * LDS + j] - dl) * invD;
#pragma unroll
                for (int x = 0; x < CP; ++x) gq[x] = fmaf(dc, Ks[j * LDP + cg * CP + x], gq[x]);
            }
        }
    }
    // through the projection: dq = (dqh - (qh . dqh) qh) / ||q||
    float ug = 0.f;
#pragma unroll
    for (int x = 0; x < CP; ++x) ug = fmaf(Qs[r * LDP + cg * CP + x], gq[x], ug);
    ug += __shfl_xor_sync(0xffffffffu, ug, 1);
    ug += __shfl_xor_sync(0xffffffffu, ug, 2);
    if (qi < T) {
        const float n = qn[r];
        const float inv = n > 0.f ? 1.f / n : 0.f;
        Tin* out = dq + (bh * T + qi) * P + cg * CP;
#pragma unroll
        for (int x = 0; x < CP; ++x) store_as(out + x, (gq[x] - ug * Qs[r * LDP + cg * CP + x]) * inv);
    }
}

template <int P, int DV>
constexpr size_t cols_smem_bytes() {
    // Ks, Qs [kBT][P+1]; Vs, Gs [kBT][DV]; Cs, Xs [kBT][kBT+1] (key-major); kn, Dq, dq_ [kBT]
    return sizeof(float) * (2 * kBT * (P + 1) + 2 * kBT * DV + 2 * kBT * (kBT + 1) + 3 * kBT);
}

// Column pass.  Block (key tile kt, head bh); thread (j, cg) owns key j of the
// tile, value columns [cg DV/4, ...) of dv and lift coordinates [cg P/4, ...)
// of dk; it walks the query tiles qt >= kt.
template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_cols_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                const Tin* __restrict__ dO, Tin* __restrict__ dk, Tin* __restrict__ dvo,
                const float* __restrict__ Din, const float* __restrict__ delta_in, int T) {
    constexpr int LDP = P + 1, LDS = kBT + 1, CV = DV / 4, CP = P / 4;
    extern __shared__ float smem[];
    float* Ks = smem;
    float* Qs = Ks + kBT * LDP;
    float* Vs = Qs + kBT * LDP;
    float* Gs = Vs + kBT * DV;
    float* Cs = Gs + kBT * DV;  // [key j][query i]
    float* Xs = Cs + kBT * LDS;
    float* kn = Xs + kBT * LDS;
    float* Dq = kn + kBT;
    float* dl = Dq + kBT;

    const int nt = (T + kBT - 1) / kBT;
    const int kt = nt - 1 - blockIdx.x;  // longest column walks first
    const int64_t bh = blockIdx.y;
    const Tin* qh = q + bh * T * P;
    const Tin* Gh = dO + bh * T * DV;
    const int j = threadIdx.x >> 2, cg = threadIdx.x & 3;
    const int kj = kt * kBT + j;
    load_unit_rows_norm<Tin, P>(k + bh * T * P, kt * kBT, T, Ks, kn);
    load_rows_plain<Tin, DV>(v + bh * T * DV, kt * kBT, kBT, T, Vs, DV);

    float gk[CP], gv[CV];
#pragma unroll
    for (int x = 0; x < CP; ++x) gk[x] = 0.f;
#pragma unroll
    for (int x = 0; x < CV; ++x) gv[x] = 0.f;
    for (int qt = kt; qt < nt; ++qt) {
        __syncthreads();
        load_rows_unit<Tin, P>(qh, qt * kBT, kBT, T, Qs, LDP);
        load_rows_plain<Tin, DV>(Gh, qt * kBT, kBT, T, Gs, DV);
        for (int i = threadIdx.x; i < kBT; i += blockDim.x) {
            const int t = qt * kBT + i;
            Dq[i] = t < T ? Din[bh * T + t] : 0.f;
            dl[i] = t < T ? delta_in[bh * T + t] : 0.f;
        }
        __syncthreads();
        // thread (j, cg): queries i = cg + 4 m
        for (int m = 0; m < kBT / 4; ++m) {
            const int i = cg + 4 * m, t = qt * kBT + i;
            float c = 0.f, x = 0.f;
#pragma unroll
            for (int a = 0; a < P; ++a) c = fmaf(Qs[i * LDP + a], Ks[j * LDP + a], c);
#pragma unroll
            for (int a = 0; a < DV; ++a) x = fmaf(Gs[i * DV + a], Vs[j * DV + a], x);
            const bool live = kj <= t && t < T && kj < T;
            Cs[j * LDS + i] = live ? c : 0.f;
            Xs[j * LDS + i] = live ? x : 0.f;
        }
        __syncthreads();
        for (int i = 0; i < kBT; ++i) {
            const float D = Dq[i];
            if (!(D > 0.f)) continue;
            const float invD = 1.f / D, c = Cs[j * LDS + i];
            const float w = c * c * invD;
            const float dc = 2.f * c * (Xs[j * LDS + i] - dl[i]) * invD;
#pragma unroll
            for (int x = 0; x < CV; ++x) gv[x] = fmaf(w, Gs[i * DV + cg * CV + x], gv[x]);
#pragma unroll
            for (int x = 0; x < CP; ++x) gk[x] = fmaf(dc, Qs[i * LDP + cg * CP + x], gk[x]);
        }
    }
    float ug = 0.f;
#pragma unroll
    for (int x = 0; x < CP; ++x) ug = fmaf(Ks[j * LDP + cg * CP + x], gk[x], ug);
    ug += __shfl_xor_sync(0xffffffffu, ug, 1);
    ug += __shfl_xor_sync(0xffffffffu, ug, 2);
    if (kj < T) {
        const float n = kn[j];
        const float inv = n > 0.f ? 1.f / n : 0.f;
        Tin* ok = dk + (bh * T + kj) * P + cg * CP;
#pragma unroll
        for (int x = 0; x < CP; ++x) store_as(ok + x, (gk[x] - ug * Ks[j * LDP + cg * CP + x]) * inv);
        Tin* ov = dvo + (bh * T + kj) * DV + cg * CV;
#pragma unroll
        for (int x = 0; x < CV; ++x) store_as(ov + x, gv[x]);
    }
}

template <typename Tin, int P, int DV>
cudaError_t backward_typed(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk, void* dv,
                           float* Dws, float* deltaws, int BH, int T, cudaStream_t s) {
    const int nt = (T + kBT - 1) / kBT;
    {
        constexpr size_t smem = rows_smem_bytes<P, DV>();
        auto kern = bwd_rows_kernel<Tin, P, DV>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        KATA_TRACED("backward_rows_simt", s,
                    kern<<<dim3(nt, BH), kThreads, smem, s>>>(
                        static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                        static_cast<const Tin*>(dO), static_cast<Tin*>(dq), Dws, deltaws, T));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    constexpr size_t smem = cols_smem_bytes<P, DV>();
    auto kern = bwd_cols_kernel<Tin, P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    KATA_TRACED("backward_cols_simt", s,
                kern<<<dim3(nt, BH), kThreads, smem, s>>>(
                    static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                    static_cast<const Tin*>(dO), static_cast<Tin*>(dk), static_cast<Tin*>(dv), Dws, deltaws, T));
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t dispatch(int p, int dv_, const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk,
                     void* dv, float* Dws, float* deltaws, int BH, int T, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv_ == DV_) return backward_typed<Tin, P_, DV_>(q, k, v, dO, dq, dk, dv, Dws, deltaws, BH, T, s);
    KATA_CASE(16, 16) KATA_CASE(16, 32) KATA_CASE(16, 64)
    KATA_CASE(32, 16) KATA_CASE(32, 32) KATA_CASE(32, 64)
    KATA_CASE(64, 16) KATA_CASE(64, 32) KATA_CASE(64, 64)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_backward(int dtype, const void* q, const void* k, const void* v, const void* dO, void* dq,
                            void* dk, void* dv, float* D_ws, float* delta_ws, int BH, int T, int p, int dv_dim,
                            cudaStream_t s) {
    return dtype == 0 ? dispatch<float>(p, dv_dim, q, k, v, dO, dq, dk, dv, D_ws, delta_ws, BH, T, s)
                      : dispatch<__nv_bfloat16>(p, dv_dim, q, k, v, dO, dq, dk, dv, D_ws, delta_ws, BH, T, s);
}

}  // namespace kata
