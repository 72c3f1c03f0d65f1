// O(T) backward of the KATA forward in the chunked form, on CUDA cores
// (fp32 arithmetic, any input dtype).  With G_t = dL/do_t, the forward's row
// normaliser D_t and delta_t = G_t . o_t, write gN_t = G_t / D_t and
// gD_t = -delta_t / D_t (both 0 where D_t = 0).  Per chunk c of kBC tokens:
//   query side  dpsi(qh_t) = P_c gN_t + Pz_c gD_t  (P_c, Pz_c: the forward's
//               exclusive prefix states) and, inside the chunk,
//               dc_ts = 2 c_ts (gN_t . v_s + gD_t) for s <= t, c_ts = qh_t . kh_s;
//               dqh_t = 2 Gamma(dpsi(qh_t)) qh_t + sum_s dc_ts kh_s;
//   gradient states R_c = sum_{t in c} psi(qh_t) [gN_t | gD_t]^T, and their
//               reverse exclusive prefix dS_c = sum_{c' > c} R_c';
//   key side    dpsi(kh_s) = dS_c v_s + dSz_c,  dv_s = dS_c^T psi(kh_s)
//               + sum_{t in c, t >= s} c_ts^2 gN_t,
//               dkh_s = 2 Gamma(dpsi(kh_s)) kh_s + sum_t dc_ts qh_t;
// where Gamma(gamma) is the symmetric p x p matrix of a packed coordinate
// vector (diagonal gamma_ii, off-diagonal gamma_ij / sqrt 2), so that
// 2 Gamma(gamma) u is the gradient of gamma . psi(u).  Finally dq, dk go back
// through the unit-sphere projections.  The chunk length of the backward is
// its own (kBC), independent of the forward's.
#include "kata_device.cuh"
#include "kata_internal.h"

namespace kata {
namespace {

constexpr int kBC = 64;         // tokens per backward chunk
constexpr int kQThreads = 128;  // two threads per token
constexpr int kTile = 32;       // packed rows / tokens per tile
constexpr int kSThreads = 256;
constexpr int kRowsPerBlock = 64;

// Rows [r0, r0 + rows) of a [T][P] matrix on the unit sphere into dst (ld
// P + 1) and their norms into nrm (zero vectors stay zero); rows past T are
// zero.  One warp per row.
template <typename Tin, int P>
__device__ __forceinline__ void load_unit_norm(const Tin* __restrict__ src, int r0, int rows, int T, float* dst,
                                               float* nrm) {
    constexpr int PER_LANE = (P + 31) / 32, LDP = P + 1;
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
            if (i < P) dst[r * LDP + i] = x[m] * inv;
        }
        if (lane == 0) nrm[r] = ss > 0.f ? sqrtf(ss) : 0.f;
    }
}

// dst[r][i] += 2 Gamma(gamma) u restricted to packed row (i, j): the
// gradient of gamma_(ij) psi_(ij)(u) with respect to u.
__device__ __forceinline__ void scatter_lift_grad(float* dst, const float* u, int i, int j, float gam) {
    if (i == j) {
        dst[i] = fmaf(2.f * gam, u[i], dst[i]);
    } else {
        dst[i] = fmaf(kSqrt2 * gam, u[j], dst[i]);
        dst[j] = fmaf(kSqrt2 * gam, u[i], dst[j]);
    }
}

// ---------------------------------------------------------------- query side
template <int P, int DV>
constexpr size_t query_smem_floats() {
    return 2 * kBC * (P + 1) + 2 * kBC * DV + 2 * kBC * (kTile + 1) + kTile * DV + kTile + kBC * (P + 1) + 3 * kBC +
           2 * kTile;
}

// Block (chunk c, head bh); thread (t, half) owns token t and value columns
// [half DV/2, ...).  Recomputes the forward row (D_t, o_t), writes D_t and
// delta_t, and writes dq_t.
template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kQThreads)
cbwd_query_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                  const Tin* __restrict__ dO, const float* __restrict__ Pre, const float* __restrict__ Prez,
                  Tin* __restrict__ dq, float* __restrict__ Dout, float* __restrict__ dlout, int T, int NC) {
    constexpr int LDP = P + 1, LDT = kTile + 1, CPT = DV / 2, HP = P / 2, N = P * (P + 1) / 2;
    extern __shared__ float smem[];
    float* Qs = smem;             // [kBC][LDP] unit queries
    float* Ks = Qs + kBC * LDP;   // [kBC][LDP] unit keys
    float* Vs = Ks + kBC * LDP;   // [kBC][DV]
    float* Gs = Vs + kBC * DV;    // [kBC][DV] dO rows
    float* Pt = Gs + kBC * DV;    // [kBC][LDT] lifted queries / scores
    float* Xs = Pt + kBC * LDT;   // [kBC][LDT] dO_t . v_s
    float* St = Xs + kBC * LDT;   // [kTile][DV] prefix rows
    float* Zt = St + kTile * DV;  // [kTile]
    float* dQ = Zt + kTile;       // [kBC][LDP] gradient of the unit query
    float* qn = dQ + kBC * LDP;   // [kBC]
    float* Dsh = qn + kBC;        // [kBC]
    float* dsh = Dsh + kBC;       // [kBC]
    int* Ii = reinterpret_cast<int*>(dsh + kBC);
    int* Jj = Ii + kTile;

    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kBC, len = min(kBC, T - t0);
    load_unit_norm<Tin, P>(q + bh * T * P, t0, kBC, T, Qs, qn);
    load_rows_unit<Tin, P>(k + bh * T * P, t0, kBC, T, Ks, LDP);
    load_rows_plain<Tin, DV>(v + bh * T * DV, t0, kBC, T, Vs, DV);
    load_rows_plain<Tin, DV>(dO + bh * T * DV, t0, kBC, T, Gs, DV);
    for (int e = threadIdx.x; e < kBC * LDP; e += blockDim.x) dQ[e] = 0.f;

    const int t = threadIdx.x >> 1, half = threadIdx.x & 1;
    const bool live_t = t < len;
    const float* Pc = Pre + (bh * NC + c) * (int64_t)N * DV;
    const float* Pzc = Prez + (bh * NC + c) * (int64_t)N;

    auto load_prefix_tile = [&](int a0) {
        if (threadIdx.x < kTile) {
            int i = 0, j = 0;
            if (a0 + threadIdx.x < N) unpack_index(a0 + threadIdx.x, P, i, j);
            Ii[threadIdx.x] = i;
            Jj[threadIdx.x] = j;
            Zt[threadIdx.x] = a0 + threadIdx.x < N ? Pzc[a0 + threadIdx.x] : 0.f;
        }
        for (int e = threadIdx.x; e < kTile * DV; e += blockDim.x) {
            const int aa = e / DV;
            St[e] = a0 + aa < N ? Pc[(int64_t)a0 * DV + e] : 0.f;
        }
    };

    // ---- forward row: prefix readout plus the local causal part
    float acc[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x) acc[x] = 0.f;
    float den = 0.f;
    for (int a0 = 0; a0 < N; a0 += kTile) {
        __syncthreads();
        load_prefix_tile(a0);
        __syncthreads();
        for (int e = threadIdx.x; e < kBC * kTile; e += blockDim.x) {
            const int tt = e / kTile, aa = e - tt * kTile;
            const int i = Ii[aa], j = Jj[aa];
            const float scale = (i == j) ? 1.f : kSqrt2;
            Pt[tt * LDT + aa] = a0 + aa < N ? Qs[tt * LDP + i] * Qs[tt * LDP + j] * scale : 0.f;
        }
        __syncthreads();
        for (int aa = 0; aa < kTile; ++aa) {
            const float ps = Pt[t * LDT + aa];
            den = fmaf(ps, Zt[aa], den);
#pragma unroll
            for (int x = 0; x < CPT; ++x) acc[x] = fmaf(ps, St[aa * DV + half * CPT + x], acc[x]);
        }
    }
    for (int s0 = 0; s0 < kBC; s0 += kTile) {
        __syncthreads();
        for (int e = threadIdx.x; e < kBC * kTile; e += blockDim.x) {
            const int tt = e / kTile, ss = e - tt * kTile, s = s0 + ss;
            float d = 0.f;
            if (s <= tt && s < len) {
#pragma unroll 16
                for (int i = 0; i < P; ++i) d = fmaf(Qs[tt * LDP + i], Ks[s * LDP + i], d);
            }
            Pt[tt * LDT + ss] = d * d;
        }
        __syncthreads();
        for (int ss = 0; ss < kTile; ++ss) {
            const float sc = Pt[t * LDT + ss];
            den += sc;
#pragma unroll
            for (int x = 0; x < CPT; ++x) acc[x] = fmaf(sc, Vs[(s0 + ss) * DV + half * CPT + x], acc[x]);
        }
    }
    const bool has = live_t && den > 0.f;
    const float invD = has ? 1.f / den : 0.f;
    float dpart = 0.f;
#pragma unroll
    for (int x = 0; x < CPT; ++x) dpart = fmaf(Gs[t * DV + half * CPT + x], acc[x] * invD, dpart);
    const float delta = dpart + __shfl_xor_sync(0xffffffffu, dpart, 1);
    if (half == 0) {
        Dsh[t] = has ? den : 0.f;
        dsh[t] = has ? delta : 0.f;
        if (live_t) {
            Dout[bh * T + t0 + t] = den;
            dlout[bh * T + t0 + t] = delta;
        }
    }
    float gN[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x) gN[x] = Gs[t * DV + half * CPT + x] * invD;
    const float gD = -delta * invD;

    // ---- dqh from the prefix: 2 Gamma(P_c gN + Pz_c gD) qh
    for (int a0 = 0; a0 < N; a0 += kTile) {
        __syncthreads();
        load_prefix_tile(a0);
        __syncthreads();
        for (int aa = 0; aa < kTile; ++aa) {
            float g = half == 0 ? Zt[aa] * gD : 0.f;
#pragma unroll
            for (int x = 0; x < CPT; ++x) g = fmaf(St[aa * DV + half * CPT + x], gN[x], g);
            g += __shfl_xor_sync(0xffffffffu, g, 1);
            if (half == 0 && has && a0 + aa < N) scatter_lift_grad(dQ + t * LDP, Qs + t * LDP, Ii[aa], Jj[aa], g);
        }
    }
    // ---- dqh from the chunk's own keys: sum_s dc_ts kh_s
    for (int s0 = 0; s0 < kBC; s0 += kTile) {
        __syncthreads();
        for (int e = threadIdx.x; e < kBC * kTile; e += blockDim.x) {
            const int tt = e / kTile, ss = e - tt * kTile, s = s0 + ss;
            float d = 0.f, x = 0.f;
            if (s <= tt && s < len) {
#pragma unroll 16
                for (int i = 0; i < P; ++i) d = fmaf(Qs[tt * LDP + i], Ks[s * LDP + i], d);
#pragma unroll 16
                for (int i = 0; i < DV; ++i) x = fmaf(Gs[tt * DV + i], Vs[s * DV + i], x);
            }
            Pt[tt * LDT + ss] = d;
            Xs[tt * LDT + ss] = x;
        }
        __syncthreads();
        if (has) {
            const float dl = dsh[t];
            for (int ss = 0; ss < kTile; ++ss) {
                const float cc = Pt[t * LDT + ss];
                const float dc = 2.f * cc * (Xs[t * LDT + ss] - dl) * invD;
#pragma unroll
                for (int x = 0; x < HP; ++x)
                    dQ[t * LDP + half * HP + x] = fmaf(dc, Ks[(s0 + ss) * LDP + half * HP + x],
                                                        dQ[t * LDP + half * HP + x]);
            }
        }
    }
    __syncthreads();
    // ---- back through the projection: dq = (dqh - (qh . dqh) qh) / ||q||
    float ug = 0.f;
#pragma unroll
    for (int x = 0; x < HP; ++x) ug = fmaf(Qs[t * LDP + half * HP + x], dQ[t * LDP + half * HP + x], ug);
    ug += __shfl_xor_sync(0xffffffffu, ug, 1);
    if (live_t) {
        const float inv = qn[t] > 0.f ? 1.f / qn[t] : 0.f;
        Tin* out = dq + (bh * T + t0 + t) * P + half * HP;
#pragma unroll
        for (int x = 0; x < HP; ++x)
            store_as(out + x, (dQ[t * LDP + half * HP + x] - ug * Qs[t * LDP + half * HP + x]) * inv);
    }
}

// ---------------------------------------------------------------- gradient states
// Block (chunk c, tile of 64 packed rows, head bh): thread owns one packed row
// and DV/4 columns of R_c = sum_t psi(qh_t) [gN_t | gD_t]^T.
template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kSThreads)
cbwd_gstates_kernel(const Tin* __restrict__ q, const Tin* __restrict__ dO, const float* __restrict__ Din,
                    const float* __restrict__ dlin, float* __restrict__ R, float* __restrict__ Rz, int T, int NC) {
    constexpr int LDP = P + 1, CPT = DV / 4, N = P * (P + 1) / 2;
    extern __shared__ float smem[];
    float* Qs = smem;            // [kBC][LDP]
    float* Gn = Qs + kBC * LDP;  // [kBC][DV]  dO / D
    float* gD = Gn + kBC * DV;   // [kBC]      -delta / D
    const int c = blockIdx.x;
    const int64_t bh = blockIdx.z;
    const int t0 = c * kBC, len = min(kBC, T - t0);
    load_rows_unit<Tin, P>(q + bh * T * P, t0, kBC, T, Qs, LDP);
    load_rows_plain<Tin, DV>(dO + bh * T * DV, t0, kBC, T, Gn, DV);
    __syncthreads();
    for (int e = threadIdx.x; e < kBC * DV; e += blockDim.x) {
        const int tt = e / DV;
        const float D = tt < len ? Din[bh * T + t0 + tt] : 0.f;
        Gn[e] = D > 0.f ? Gn[e] / D : 0.f;
    }
    for (int tt = threadIdx.x; tt < kBC; tt += blockDim.x) {
        const float D = tt < len ? Din[bh * T + t0 + tt] : 0.f;
        gD[tt] = D > 0.f ? -dlin[bh * T + t0 + tt] / D : 0.f;
    }
    __syncthreads();
    const int a = blockIdx.y * kRowsPerBlock + (threadIdx.x >> 2), cg = threadIdx.x & 3;
    if (a >= N) return;
    int i, j;
    unpack_index(a, P, i, j);
    const float scale = (i == j) ? 1.f : kSqrt2;
    float acc[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x) acc[x] = 0.f;
    float zacc = 0.f;
    for (int tt = 0; tt < len; ++tt) {
        const float psi = Qs[tt * LDP + i] * Qs[tt * LDP + j] * scale;
        zacc = fmaf(psi, gD[tt], zacc);
#pragma unroll
        for (int x = 0; x < CPT; ++x) acc[x] = fmaf(psi, Gn[tt * DV + cg * CPT + x], acc[x]);
    }
    float* dst = R + ((bh * NC + c) * N + a) * DV + cg * CPT;
#pragma unroll
    for (int x = 0; x < CPT; ++x) dst[x] = acc[x];
    if (cg == 0) Rz[(bh * NC + c) * N + a] = zacc;
}

// Reverse exclusive prefix over the chunk axis, in place: x_c <- sum_{c' > c} x_c'.
// One thread per VEC consecutive columns; the values of kRevBatch chunks are
// loaded before any of them is overwritten, so that a batch's loads are in
// flight together (each step's store would otherwise hold back the next load).
constexpr int kRevBatch = 8;

template <int VEC>
__global__ void reverse_exclusive_kernel(float* __restrict__ x, int64_t heads, int64_t NC, int64_t W) {
    const int64_t per_head = W / VEC;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= heads * per_head) return;
    const int64_t h = gid / per_head, e = (gid - h * per_head) * VEC;
    float* col = x + h * NC * W + e;
    float run[VEC];
#pragma unroll
    for (int u = 0; u < VEC; ++u) run[u] = 0.f;
    for (int64_t c1 = NC - 1; c1 >= 0; c1 -= kRevBatch) {
        float xv[kRevBatch][VEC];
#pragma unroll
        for (int b = 0; b < kRevBatch; ++b) {
            const int64_t c = c1 - b;
            if (VEC == 4) {
                const float4 t = c >= 0 ? *reinterpret_cast<const float4*>(col + c * W) : make_float4(0.f, 0.f, 0.f, 0.f);
                xv[b][0] = t.x;
                xv[b][VEC > 1 ? 1 : 0] = t.y;
                xv[b][VEC > 2 ? 2 : 0] = t.z;
                xv[b][VEC > 3 ? 3 : 0] = t.w;
            } else {
#pragma unroll
                for (int u = 0; u < VEC; ++u) xv[b][u] = c >= 0 ? col[c * W + u] : 0.f;
            }
        }
#pragma unroll
        for (int b = 0; b < kRevBatch; ++b) {
            const int64_t c = c1 - b;
            if (c < 0) break;
            if (VEC == 4) {
                *reinterpret_cast<float4*>(col + c * W) =
                    make_float4(run[0], run[VEC > 1 ? 1 : 0], run[VEC > 2 ? 2 : 0], run[VEC > 3 ? 3 : 0]);
            } else {
#pragma unroll
                for (int u = 0; u < VEC; ++u) col[c * W + u] = run[u];
            }
#pragma unroll
            for (int u = 0; u < VEC; ++u) run[u] += xv[b][u];
        }
    }
}

// ---------------------------------------------------------------- key side
template <int P, int DV>
constexpr size_t key_smem_floats() {
    return 2 * kBC * (P + 1) + 2 * kBC * DV + 2 * kBC * (kTile + 1) + kTile * DV + kTile + kBC * (P + 1) + 3 * kBC +
           2 * kTile;
}

// Block (chunk c, head bh); thread (s, half) owns key s of the chunk, value
// columns [half DV/2, ...) of dv and lift coordinates [half P/2, ...) of dk.
template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kQThreads)
cbwd_key_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                const Tin* __restrict__ dO, const float* __restrict__ Din, const float* __restrict__ dlin,
                const float* __restrict__ dS, const float* __restrict__ dSz, Tin* __restrict__ dk,
                Tin* __restrict__ dvo, int T, int NC) {
    constexpr int LDP = P + 1, LDT = kTile + 1, CPT = DV / 2, HP = P / 2, N = P * (P + 1) / 2;
    extern __shared__ float smem[];
    float* Ks = smem;             // [kBC][LDP] unit keys
    float* Qs = Ks + kBC * LDP;   // [kBC][LDP] unit queries
    float* Vs = Qs + kBC * LDP;   // [kBC][DV]
    float* Gs = Vs + kBC * DV;    // [kBC][DV] dO rows
    float* Pt = Gs + kBC * DV;    // [kBC][LDT] lifted keys / scores (key-major)
    float* Xs = Pt + kBC * LDT;   // [kBC][LDT] dO_t . v_s (key-major)
    float* St = Xs + kBC * LDT;   // [kTile][DV] dS rows
    float* Zt = St + kTile * DV;  // [kTile]
    float* dK = Zt + kTile;       // [kBC][LDP]
    float* kn = dK + kBC * LDP;   // [kBC]
    float* Dsh = kn + kBC;        // [kBC]
    float* dsh = Dsh + kBC;       // [kBC]
    int* Ii = reinterpret_cast<int*>(dsh + kBC);
    int* Jj = Ii + kTile;

    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kBC, len = min(kBC, T - t0);
    load_unit_norm<Tin, P>(k + bh * T * P, t0, kBC, T, Ks, kn);
    load_rows_unit<Tin, P>(q + bh * T * P, t0, kBC, T, Qs, LDP);
    load_rows_plain<Tin, DV>(v + bh * T * DV, t0, kBC, T, Vs, DV);
    load_rows_plain<Tin, DV>(dO + bh * T * DV, t0, kBC, T, Gs, DV);
    for (int e = threadIdx.x; e < kBC * LDP; e += blockDim.x) dK[e] = 0.f;
    for (int tt = threadIdx.x; tt < kBC; tt += blockDim.x) {
        Dsh[tt] = tt < len ? Din[bh * T + t0 + tt] : 0.f;
        dsh[tt] = tt < len ? dlin[bh * T + t0 + tt] : 0.f;
    }

    const int s = threadIdx.x >> 1, half = threadIdx.x & 1;
    const bool live_s = s < len;
    const float* dSc = dS + (bh * NC + c) * (int64_t)N * DV;
    const float* dSzc = dSz + (bh * NC + c) * (int64_t)N;
    float gv[CPT];
#pragma unroll
    for (int x = 0; x < CPT; ++x) gv[x] = 0.f;

    // ---- from later chunks: dv_s = dS_c^T psi(kh_s), dkh_s = 2 Gamma(dS_c v_s + dSz_c) kh_s
    for (int a0 = 0; a0 < N; a0 += kTile) {
        __syncthreads();
        if (threadIdx.x < kTile) {
            int i = 0, j = 0;
            if (a0 + threadIdx.x < N) unpack_index(a0 + threadIdx.x, P, i, j);
            Ii[threadIdx.x] = i;
            Jj[threadIdx.x] = j;
            Zt[threadIdx.x] = a0 + threadIdx.x < N ? dSzc[a0 + threadIdx.x] : 0.f;
        }
        for (int e = threadIdx.x; e < kTile * DV; e += blockDim.x) {
            const int aa = e / DV;
            St[e] = a0 + aa < N ? dSc[(int64_t)a0 * DV + e] : 0.f;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kBC * kTile; e += blockDim.x) {
            const int ss = e / kTile, aa = e - ss * kTile;
            const int i = Ii[aa], j = Jj[aa];
            const float scale = (i == j) ? 1.f : kSqrt2;
            Pt[ss * LDT + aa] = a0 + aa < N ? Ks[ss * LDP + i] * Ks[ss * LDP + j] * scale : 0.f;
        }
        __syncthreads();
        for (int aa = 0; aa < kTile; ++aa) {
            const float pk = Pt[s * LDT + aa];
            float g = half == 0 ? Zt[aa] : 0.f;
#pragma unroll
            for (int x = 0; x < CPT; ++x) {
                const float sv = St[aa * DV + half * CPT + x];
                gv[x] = fmaf(pk, sv, gv[x]);
                g = fmaf(sv, Vs[s * DV + half * CPT + x], g);
            }
            g += __shfl_xor_sync(0xffffffffu, g, 1);
            if (half == 0 && live_s && a0 + aa < N) scatter_lift_grad(dK + s * LDP, Ks + s * LDP, Ii[aa], Jj[aa], g);
        }
    }
    // ---- from the chunk's own later queries t >= s
    for (int q0 = 0; q0 < kBC; q0 += kTile) {
        __syncthreads();
        for (int e = threadIdx.x; e < kBC * kTile; e += blockDim.x) {
            const int ss = e / kTile, tt = e - ss * kTile, t = q0 + tt;
            float d = 0.f, x = 0.f;
            if (t >= ss && t < len && ss < len) {
#pragma unroll 16
                for (int i = 0; i < P; ++i) d = fmaf(Qs[t * LDP + i], Ks[ss * LDP + i], d);
#pragma unroll 16
                for (int i = 0; i < DV; ++i) x = fmaf(Gs[t * DV + i], Vs[ss * DV + i], x);
            }
            Pt[ss * LDT + tt] = d;
            Xs[ss * LDT + tt] = x;
        }
        __syncthreads();
        if (live_s) {
            for (int tt = 0; tt < kTile; ++tt) {
                const int t = q0 + tt;
                const float D = Dsh[t];
                if (!(D > 0.f)) continue;
                const float invD = 1.f / D, cc = Pt[s * LDT + tt];
                const float w = cc * cc * invD;
                const float dc = 2.f * cc * (Xs[s * LDT + tt] - dsh[t]) * invD;
#pragma unroll
                for (int x = 0; x < CPT; ++x) gv[x] = fmaf(w, Gs[t * DV + half * CPT + x], gv[x]);
#pragma unroll
                for (int x = 0; x < HP; ++x)
                    dK[s * LDP + half * HP + x] = fmaf(dc, Qs[t * LDP + half * HP + x], dK[s * LDP + half * HP + x]);
            }
        }
    }
    __syncthreads();
    float ug = 0.f;
#pragma unroll
    for (int x = 0; x < HP; ++x) ug = fmaf(Ks[s * LDP + half * HP + x], dK[s * LDP + half * HP + x], ug);
    ug += __shfl_xor_sync(0xffffffffu, ug, 1);
    if (live_s) {
        const float inv = kn[s] > 0.f ? 1.f / kn[s] : 0.f;
        Tin* ok = dk + (bh * T + t0 + s) * P + half * HP;
#pragma unroll
        for (int x = 0; x < HP; ++x)
            store_as(ok + x, (dK[s * LDP + half * HP + x] - ug * Ks[s * LDP + half * HP + x]) * inv);
        Tin* ov = dvo + (bh * T + t0 + s) * DV + half * CPT;
#pragma unroll
        for (int x = 0; x < CPT; ++x) store_as(ov + x, gv[x]);
    }
}

template <typename Tin, int P, int DV>
cudaError_t typed(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk, void* dv, float* S,
                  float* z, float* D, float* dl, int BH, int T, cudaStream_t s) {
    constexpr int N = P * (P + 1) / 2;
    const int NC = (T + kBC - 1) / kBC;
    const int dtype = sizeof(Tin) == 4 ? 0 : 1;
    // forward prefix states at the backward's chunk length (bf16: the
    // tensor-core chunk-state kernel writes every chunk's exclusive prefix in
    // one pass, as the forward's own states are built)
    cudaError_t e;
    if (dtype == 1) {
        e = launch_states_tc(k, v, S, z, BH, T, P, DV, kBC, NC, NC, 1, 1, s);
    } else {
        e = launch_chunk_states_simt(dtype, k, v, S, z, BH, T, P, DV, kBC, s);
        if (e == cudaSuccess) e = launch_scan(0, S, S, nullptr, nullptr, BH, NC, (int64_t)N * DV, s);
        if (e == cudaSuccess) e = launch_scan(0, z, z, nullptr, nullptr, BH, NC, N, s);
    }
    if (e != cudaSuccess) return e;
    {
        constexpr size_t smem = sizeof(float) * query_smem_floats<P, DV>();
        auto kern = cbwd_query_kernel<Tin, P, DV>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        KATA_TRACED("backward_query_simt", s,
                    kern<<<dim3(NC, BH), kQThreads, smem, s>>>(
                        static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                        static_cast<const Tin*>(dO), S, z, static_cast<Tin*>(dq), D, dl, T, NC));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        constexpr size_t smem = sizeof(float) * (kBC * (P + 1) + kBC * DV + kBC);
        auto kern = cbwd_gstates_kernel<Tin, P, DV>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        KATA_TRACED("backward_gstates_simt", s,
                    kern<<<dim3(NC, (N + kRowsPerBlock - 1) / kRowsPerBlock, BH), kSThreads, smem, s>>>(
                        static_cast<const Tin*>(q), static_cast<const Tin*>(dO), D, dl, S, z, T, NC));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    for (int part = 0; part < 2; ++part) {
        const int64_t W = part == 0 ? (int64_t)N * DV : N;
        float* xs = part == 0 ? S : z;
        if (W % 4 == 0 && (reinterpret_cast<uintptr_t>(xs) & 15u) == 0) {
            const int64_t threads = (int64_t)BH * (W / 4);
            KATA_TRACED("backward_reverse_scan", s,
                        (reverse_exclusive_kernel<4><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(xs, BH, NC, W)));
        } else {
            const int64_t threads = (int64_t)BH * W;
            KATA_TRACED("backward_reverse_scan", s,
                        (reverse_exclusive_kernel<1><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(xs, BH, NC, W)));
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    constexpr size_t smem = sizeof(float) * key_smem_floats<P, DV>();
    auto kern = cbwd_key_kernel<Tin, P, DV>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    KATA_TRACED("backward_key_simt", s,
                kern<<<dim3(NC, BH), kQThreads, smem, s>>>(
                    static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                    static_cast<const Tin*>(dO), D, dl, S, z, static_cast<Tin*>(dk), static_cast<Tin*>(dv), T, NC));
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t dispatch(int p, int dv_, const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk,
                     void* dv, float* S, float* z, float* D, float* dl, int BH, int T, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv_ == DV_) return typed<Tin, P_, DV_>(q, k, v, dO, dq, dk, dv, S, z, D, dl, BH, T, s);
    KATA_CASE(16, 16) KATA_CASE(16, 32) KATA_CASE(16, 64)
    KATA_CASE(32, 16) KATA_CASE(32, 32) KATA_CASE(32, 64)
    KATA_CASE(64, 16) KATA_CASE(64, 32) KATA_CASE(64, 64)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

int backward_chunk_len() { return kBC; }

cudaError_t launch_backward_chunked(int dtype, const void* q, const void* k, const void* v, const void* dO, void* dq,
                                    void* dk, void* dv, float* S_ws, float* z_ws, float* D_ws, float* delta_ws, int BH,
                                    int T, int p, int dv_dim, cudaStream_t s) {
    return dtype == 0
               ? dispatch<float>(p, dv_dim, q, k, v, dO, dq, dk, dv, S_ws, z_ws, D_ws, delta_ws, BH, T, s)
               : dispatch<__nv_bfloat16>(p, dv_dim, q, k, v, dO, dq, dk, dv, S_ws, z_ws, D_ws, delta_ws, BH, T, s);
}

}  // namespace kata
