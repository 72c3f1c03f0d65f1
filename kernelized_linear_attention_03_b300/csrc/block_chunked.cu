// KATA-Sigma-g and KATA-M-g forwards on CUDA cores ("two reduced PSD
// families" paragraph): the chunked form in the three phases of the
// chunked-scan paragraph (per-chunk states in the block lift, the cumulative
// pass of scan.cu, a per-chunk output adding the prefix readout to the local
// C x C causal part) and the flash-style quadratic form.  fp32 arithmetic for
// any input dtype.  The lift's packed row r is described by block_row(); the
// local scores come from block dot products (block_score()), not through the
// lift.
#include "block_lift.cuh"
#include "kata_internal.h"

namespace kata {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxC = 128;
constexpr int kRowsPerBlock = 64;  // packed rows per block of the state kernel
constexpr int kTile = 32;          // packed rows / keys per tile of the output kernel

// ---------------------------------------------------------------- chunk states
// Block (chunk c, tile of 64 packed rows, head bh): thread owns one packed row
// and DV/4 value columns; z is written by column group 0.
template <int P, int DV>
constexpr size_t state_smem_bytes() {
    return sizeof(float) * (kMaxC * (P + 1) + kMaxC * DV);
}

template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
block_states_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v, float* __restrict__ S_loc,
                    float* __restrict__ z_loc, int T, int C, int NC, int family, int g, int N) {
    constexpr int LDP = P + 1, CPT = DV / 4;
    extern __shared__ float smem[];
    float* Ks = smem;              // [C][LDP] unit keys
    float* Vs = Ks + kMaxC * LDP;  // [C][DV]
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.z;
    const int t0 = c * C, len = min(C, T - t0);
    load_rows_unit<Tin, P>(k + bh * T * P, t0, len, T, Ks, LDP);
    load_rows_plain<Tin, DV>(v + bh * T * DV, t0, len, T, Vs, DV);
    __syncthreads();

    const int a = blockIdx.y * kRowsPerBlock + (threadIdx.x >> 2), cg = threadIdx.x & 3;
    if (a >= N) return;
    const int m = P / g;
    const BlockRow d = block_row(a, family, m);
    float acc[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x) acc[x] = 0.f;
    float zacc = 0.f;
    for (int s = 0; s < len; ++s) {
        const float psi = block_coord(Ks + s * LDP, d, g, m);
        zacc += psi;
#pragma unroll
        for (int x = 0; x < CPT; ++x) acc[x] = fmaf(psi, Vs[s * DV + cg * CPT + x], acc[x]);
    }
    float* dst = S_loc + ((bh * NC + c) * N + a) * DV + cg * CPT;
#pragma unroll
    for (int x = 0; x < CPT; ++x) dst[x] = acc[x];
    if (cg == 0) z_loc[(bh * NC + c) * N + a] = zacc;
}

// ---------------------------------------------------------------- chunk output
// Block (chunk c, head bh): thread owns token tid/2 of the chunk and half of
// the value columns.  The prefix readout walks the packed rows in tiles of 32
// (lifted queries and prefix rows staged in shared memory); the local part
// walks the chunk's keys in tiles of 32 with masked block scores.
template <int P, int DV>
constexpr size_t output_smem_bytes() {
    return sizeof(float) * (2 * kMaxC * (P + 1) + kMaxC * DV + kMaxC * (kTile + 1) + kTile * DV + kTile +
                            kMaxC * (kTile + 1)) +
           sizeof(int) * 3 * kTile;
}

template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
block_output_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                    const float* __restrict__ Pre, const float* __restrict__ Prez, Tin* __restrict__ o, int T,
                    int C, int NC, int family, int g, int N) {
    constexpr int LDP = P + 1, LDT = kTile + 1, CPT = DV / 2;
    extern __shared__ float smem[];
    float* Qs = smem;              // [C][LDP]
    float* Ks = Qs + kMaxC * LDP;  // [C][LDP]
    float* Vs = Ks + kMaxC * LDP;  // [C][DV]
    float* Ps = Vs + kMaxC * DV;   // [C][LDT] lifted-query tile
    float* St = Ps + kMaxC * LDT;  // [kTile][DV] prefix state tile
    float* Zt = St + kTile * DV;   // [kTile]
    float* Sc = Zt + kTile;        // [C][LDT] local score tile
    int* Ii = reinterpret_cast<int*>(Sc + kMaxC * LDT);
    int* Jj = Ii + kTile;
    int* Bk = Jj + kTile;

    const int m = P / g;
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * C, len = min(C, T - t0);
    load_rows_unit<Tin, P>(q + bh * T * P, t0, len, T, Qs, LDP);
    load_rows_unit<Tin, P>(k + bh * T * P, t0, len, T, Ks, LDP);
    load_rows_plain<Tin, DV>(v + bh * T * DV, t0, len, T, Vs, DV);

    const int t = threadIdx.x >> 1, half = threadIdx.x & 1;
    float acc[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x) acc[x] = 0.f;
    float den = 0.f;

    const float* Pc = Pre + (bh * NC + c) * (int64_t)N * DV;
    const float* Pzc = Prez + (bh * NC + c) * (int64_t)N;
    for (int a0 = 0; a0 < N; a0 += kTile) {
        __syncthreads();
        if (threadIdx.x < kTile) {
            BlockRow d{0, 0, -1, 0.f};
            if (a0 + threadIdx.x < N) d = block_row(a0 + threadIdx.x, family, m);
            Ii[threadIdx.x] = d.i;
            Jj[threadIdx.x] = d.j;
            Bk[threadIdx.x] = d.blk;
            Zt[threadIdx.x] = a0 + threadIdx.x < N ? Pzc[a0 + threadIdx.x] : 0.f;
        }
        for (int e = threadIdx.x; e < kTile * DV; e += blockDim.x) {
            const int aa = e / DV;
            St[e] = a0 + aa < N ? Pc[(int64_t)a0 * DV + e] : 0.f;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < len * kTile; e += blockDim.x) {
            const int tt = e / kTile, aa = e - tt * kTile;
            BlockRow d;
            d.i = Ii[aa];
            d.j = Jj[aa];
            d.blk = Bk[aa];
            d.scale = d.i == d.j ? 1.f : kSqrt2;
            Ps[tt * LDT + aa] = a0 + aa < N ? block_coord(Qs + tt * LDP, d, g, m) : 0.f;
        }
        __syncthreads();
        if (t < len) {
            for (int aa = 0; aa < kTile; ++aa) {
                const float ps = Ps[t * LDT + aa];
                den = fmaf(ps, Zt[aa], den);
#pragma unroll
                for (int x = 0; x < CPT; ++x) acc[x] = fmaf(ps, St[aa * DV + half * CPT + x], acc[x]);
            }
        }
    }
    for (int s0 = 0; s0 < len; s0 += kTile) {
        __syncthreads();
        for (int e = threadIdx.x; e < len * kTile; e += blockDim.x) {
            const int tt = e / kTile, ss = e - tt * kTile, s = s0 + ss;
            const bool live = s <= tt && s < len;
            Sc[tt * LDT + ss] = live ? block_score(Qs + tt * LDP, Ks + s * LDP, family, g, m) : 0.f;
        }
        __syncthreads();
        if (t < len) {
            for (int ss = 0; ss < kTile && s0 + ss < len; ++ss) {
                const float sc = Sc[t * LDT + ss];
                den += sc;
#pragma unroll
                for (int x = 0; x < CPT; ++x) acc[x] = fmaf(sc, Vs[(s0 + ss) * DV + half * CPT + x], acc[x]);
            }
        }
    }
    if (t < len) {
        Tin* ot = o + (bh * T + t0 + t) * DV + half * CPT;
#pragma unroll
        for (int x = 0; x < CPT; ++x) store_as(ot + x, den > 0.f ? acc[x] / den : 0.f);
    }
}

// ---------------------------------------------------------------- quadratic form
// Flash-style: block of 64 queries, key tiles of 64 up to the diagonal; the
// masked block scores of a tile in shared memory, then accumulated against V
// (scores of unit vectors are bounded, so no running maximum is needed).
constexpr int kBQ = 64, kBK = 64;

template <int P, int DV>
constexpr size_t quad_smem_bytes() {
    return sizeof(float) * (kBQ * (P + 1) + kBK * (P + 1) + kBK * DV + kBQ * (kBK + 1));
}

template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads)
block_quadratic_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                       Tin* __restrict__ o, int T, int family, int g) {
    constexpr int LDP = P + 1, LDS = kBK + 1, CPT = DV / 4;
    extern __shared__ float smem[];
    float* Qs = smem;            // [kBQ][LDP] unit queries
    float* Ks = Qs + kBQ * LDP;  // [kBK][LDP] unit keys
    float* Vs = Ks + kBK * LDP;  // [kBK][DV]
    float* Ss = Vs + kBK * DV;   // [kBQ][LDS] masked scores

    const int m = P / g;
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
    for (int x = 0; x < CPT; ++x) acc[x] = 0.f;
    float den = 0.f;

    for (int kt = 0; kt <= qt; ++kt) {
        __syncthreads();
        load_rows_unit<Tin, P>(kh, kt * kBK, kBK, T, Ks, LDP);
        load_rows_plain<Tin, DV>(vh, kt * kBK, kBK, T, Vs, DV);
        __syncthreads();
        for (int x = 0; x < kBK / 4; ++x) {
            const int j = cg + 4 * x, kj = kt * kBK + j;
            Ss[r * LDS + j] = (kj <= qi && kj < T) ? block_score(Qs + r * LDP, Ks + j * LDP, family, g, m) : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < kBK; ++j) {
            const float s = Ss[r * LDS + j];
            den += s;
#pragma unroll
            for (int x = 0; x < CPT; ++x) acc[x] = fmaf(s, Vs[j * DV + cg * CPT + x], acc[x]);
        }
    }
    if (qi < T) {
        Tin* oh = o + (bh * T + qi) * DV + cg * CPT;
#pragma unroll
        for (int x = 0; x < CPT; ++x) store_as(oh + x, den > 0.f ? acc[x] / den : 0.f);
    }
}

// ---------------------------------------------------------------- launchers
struct Lift {
    int family, g, N;
};

template <typename Tin, int P, int DV>
cudaError_t states_typed(const void* k, const void* v, float* S, float* z, int BH, int T, int C, Lift L,
                         cudaStream_t s) {
    constexpr size_t smem = state_smem_bytes<P, DV>();
    auto kern = block_states_kernel<Tin, P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int NC = (T + C - 1) / C;
    const dim3 grid(NC, (L.N + kRowsPerBlock - 1) / kRowsPerBlock, BH);
    KATA_TRACED("block_states_simt", s,
                kern<<<grid, kThreads, smem, s>>>(static_cast<const Tin*>(k), static_cast<const Tin*>(v), S, z, T,
                                                  C, NC, L.family, L.g, L.N));
    return cudaGetLastError();
}

template <typename Tin, int P, int DV>
cudaError_t output_typed(const void* q, const void* k, const void* v, const float* Pre, const float* Prez, void* o,
                         int BH, int T, int C, Lift L, cudaStream_t s) {
    constexpr size_t smem = output_smem_bytes<P, DV>();
    auto kern = block_output_kernel<Tin, P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int NC = (T + C - 1) / C;
    KATA_TRACED("block_output_simt", s,
                kern<<<dim3(NC, BH), kThreads, smem, s>>>(static_cast<const Tin*>(q), static_cast<const Tin*>(k),
                                                          static_cast<const Tin*>(v), Pre, Prez, static_cast<Tin*>(o),
                                                          T, C, NC, L.family, L.g, L.N));
    return cudaGetLastError();
}

template <typename Tin, int P, int DV>
cudaError_t quadratic_typed(const void* q, const void* k, const void* v, void* o, int BH, int T, Lift L,
                            cudaStream_t s) {
    constexpr size_t smem = quad_smem_bytes<P, DV>();
    auto kern = block_quadratic_kernel<Tin, P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    KATA_TRACED("block_quadratic_simt", s,
                kern<<<dim3((T + kBQ - 1) / kBQ, BH), kThreads, smem, s>>>(
                    static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                    static_cast<Tin*>(o), T, L.family, L.g));
    return cudaGetLastError();
}

#define KATA_BLOCK_SHAPES(X) \
    X(16, 16) X(16, 32) X(16, 64) X(32, 16) X(32, 32) X(32, 64) X(64, 16) X(64, 32) X(64, 64)

template <typename Tin>
cudaError_t states_dispatch(int p, int dv, const void* k, const void* v, float* S, float* z, int BH, int T, int C,
                            Lift L, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return states_typed<Tin, P_, DV_>(k, v, S, z, BH, T, C, L, s);
    KATA_BLOCK_SHAPES(KATA_CASE)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t output_dispatch(int p, int dv, const void* q, const void* k, const void* v, const float* Pre,
                            const float* Prez, void* o, int BH, int T, int C, Lift L, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return output_typed<Tin, P_, DV_>(q, k, v, Pre, Prez, o, BH, T, C, L, s);
    KATA_BLOCK_SHAPES(KATA_CASE)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t quadratic_dispatch(int p, int dv, const void* q, const void* k, const void* v, void* o, int BH, int T,
                               Lift L, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return quadratic_typed<Tin, P_, DV_>(q, k, v, o, BH, T, L, s);
    KATA_BLOCK_SHAPES(KATA_CASE)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

Lift make_lift(int family, int p, int g) { return Lift{family, g, block_lift_dim(family, p, g)}; }

}  // namespace

cudaError_t launch_block_states(int dtype, const void* k, const void* v, float* S_loc, float* z_loc, int BH, int T,
                                int p, int dv, int C, int family, int g, cudaStream_t s) {
    const Lift L = make_lift(family, p, g);
    if (L.N <= 0) return cudaErrorInvalidValue;
    return dtype == 0 ? states_dispatch<float>(p, dv, k, v, S_loc, z_loc, BH, T, C, L, s)
                      : states_dispatch<__nv_bfloat16>(p, dv, k, v, S_loc, z_loc, BH, T, C, L, s);
}

cudaError_t launch_block_output(int dtype, const void* q, const void* k, const void* v, const float* P,
                                const float* Pz, void* o, int BH, int T, int p, int dv, int C, int family, int g,
                                cudaStream_t s) {
    const Lift L = make_lift(family, p, g);
    if (L.N <= 0) return cudaErrorInvalidValue;
    return dtype == 0 ? output_dispatch<float>(p, dv, q, k, v, P, Pz, o, BH, T, C, L, s)
                      : output_dispatch<__nv_bfloat16>(p, dv, q, k, v, P, Pz, o, BH, T, C, L, s);
}

cudaError_t launch_block_quadratic(int dtype, const void* q, const void* k, const void* v, void* o, int BH, int T,
                                   int p, int dv, int family, int g, cudaStream_t s) {
    const Lift L = make_lift(family, p, g);
    if (L.N <= 0) return cudaErrorInvalidValue;
    return dtype == 0 ? quadratic_dispatch<float>(p, dv, q, k, v, o, BH, T, L, s)
                      : quadratic_dispatch<__nv_bfloat16>(p, dv, q, k, v, o, BH, T, L, s);
}

}  // namespace kata
