// Per-chunk output of the chunked form on CUDA cores (fp32 arithmetic, any
// input dtype), for the plain and the gated prefix: per chunk c and head, the
// prefix readout psi(qh_t)^T [P_c | Pz_c] of the exclusive prefix state plus
// the local causal part sum_{s in c, s <= t} (qh_t.kh_s)^2 [v_s | 1], then the
// division (0 where the denominator is not positive).  The gated form
// (GATED) scales the readout by prod_{r=cC..t} gamma_r and each local term by
// prod_{r=s+1..t} gamma_r, all as direct products of gates.  Each including
// translation unit instantiates its own variant (internal linkage).
#pragma once

#include <cstdint>
#include <type_traits>

#include "kata_device.cuh"
#include "tc_primitives.cuh"

namespace kata {
namespace {
namespace chunk_out {

constexpr int kThreads = 256;  // threads per block
constexpr int kMaxC = 128;     // longest chunk
constexpr int kSlotTile = 64;  // packed rows of the prefix state per pass
constexpr int kKeyTile = 32;   // keys of the chunk per pass of the local part

template <int P, int DV>
__host__ __device__ constexpr int output_union_floats() {
    constexpr int LDP = P + 1, LDT = kMaxC + 4;
    constexpr int readout = kSlotTile * LDT + 2 * (kSlotTile * DV + kSlotTile);
    constexpr int local = kKeyTile * LDP + kKeyTile * DV + kKeyTile * LDT;
    return readout > local ? readout : local;
}

template <int P, int DV>
constexpr size_t output_smem_bytes() {
    return sizeof(float) * ((size_t)kMaxC * (P + 1) + kMaxC + output_union_floats<P, DV>()) +
           sizeof(int) * 2 * kSlotTile;
}

// Block (chunk c, head bh), kThreads threads: thread (tg, cg) holds tokens
// 4 tg .. 4 tg + 3 (and the same of KT - 1 further token groups when one
// pass of the block does not cover the chunk) times value columns
// 4 cg .. 4 cg + 3 in registers.
//   prefix readout  per tile of kSlotTile packed rows: the chunk's query
//                   lifts (rows x tokens) and the prefix state rows in shared
//                   memory (the next tile's rows copied asynchronously into a
//                   second buffer meanwhile), each thread accumulating its
//                   4 x 4 products (two 16-byte loads per 16 multiply-adds);
//                   GATED: then scaled by the decay from the chunk's start,
//                   prod_{r=cC..t} gamma_r
//   local part      per tile of kKeyTile keys: the squared scores
//                   (qh_t.kh_s)^2 of keys s <= t (GATED: times
//                   prod_{r=s+1..t} gamma_r; keys x tokens) and the values,
//                   accumulated the same way
// Each (token, column) sum runs over the packed rows, then over the keys, in
// order.  The denominators' products are shared out over the CG threads of a
// token group (thread cg takes rows cg, cg + CG, ...) and summed by shuffles
// at the end.
template <typename Tin, int P, int DV, bool GATED>
__global__ void __launch_bounds__(kThreads, 2)
chunk_output_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                    const float* __restrict__ gate, const float* __restrict__ Pre, const float* __restrict__ Prez,
                    Tin* __restrict__ o, int T, int C, int NC) {
    constexpr int LDP = P + 1, LDT = kMaxC + 4, N = P * (P + 1) / 2;
    constexpr int CG = DV / 4, TGT = kThreads / CG, KT = (kMaxC / 4 + TGT - 1) / TGT;
    static_assert(kSlotTile % CG == 0 && kKeyTile % CG == 0 && CG <= 32, "column groups");
    extern __shared__ float smem[];
    float* Qs = smem;              // [C][LDP] unit queries
    float* gs = Qs + kMaxC * LDP;  // [C] gates of the chunk
    float* Ru = gs + kMaxC;        // the readout's and the local part's tiles share this
    float* Pt = Ru;                                // [kSlotTile][LDT] query lifts, row-major by packed row
    float* Sb = Pt + kSlotTile * LDT;              // two buffers of [kSlotTile][DV] prefix state rows
    float* Zb = Sb + 2 * kSlotTile * DV;           // and of [kSlotTile] prefix normaliser rows
    float* Ks = Ru;                                // [kKeyTile][LDP] unit keys
    float* Vs = Ks + kKeyTile * LDP;               // [kKeyTile][DV]
    float* Sc = Vs + kKeyTile * DV;                // [kKeyTile][LDT] decayed squared scores, by key
    int* Ii = reinterpret_cast<int*>(Ru + output_union_floats<P, DV>());
    int* Jj = Ii + kSlotTile;

    const int c = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * C, len = min(C, T - t0);
    const int ngroups = (len + 3) / 4, nt = 4 * ngroups;
    load_rows_unit<Tin, P>(q + bh * T * P, t0, len, T, Qs, LDP);
    if constexpr (GATED)
        for (int s = threadIdx.x; s < kMaxC; s += blockDim.x) gs[s] = s < len ? gate[bh * T + t0 + s] : 0.f;

    const int cg = threadIdx.x % CG, tg0 = threadIdx.x / CG;
    float acc[KT][4][4], den[KT][4];
#pragma unroll
    for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            den[kt][i] = 0.f;
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[kt][i][x] = 0.f;
        }
    // the 4 x 4 products of row `row` of A (tokens) and B (columns): 16 multiply-adds per token group
    auto accumulate = [&](const float* A, const float* B, int row) {
        const float4 b = *reinterpret_cast<const float4*>(B + row * DV + 4 * cg);
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            const int tg = tg0 + kt * TGT;
            if (tg < ngroups) {
                const float4 a = *reinterpret_cast<const float4*>(A + row * LDT + 4 * tg);
                const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int x = 0; x < 4; ++x) acc[kt][i][x] = fmaf(av[i], bv[x], acc[kt][i][x]);
            }
        }
    };
    // this thread's share of the denominator: row `row` of A times w
    auto accumulate_den = [&](const float* A, int row, float w) {
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            const int tg = tg0 + kt * TGT;
            if (tg < ngroups) {
                const float4 a = *reinterpret_cast<const float4*>(A + row * LDT + 4 * tg);
                den[kt][0] = fmaf(a.x, w, den[kt][0]);
                den[kt][1] = fmaf(a.y, w, den[kt][1]);
                den[kt][2] = fmaf(a.z, w, den[kt][2]);
                den[kt][3] = fmaf(a.w, w, den[kt][3]);
            }
        }
    };

    // prefix readout psi(qh_t)^T P_c
    const float* Pc = Pre + (bh * NC + c) * (int64_t)N * DV;
    const float* Pzc = Prez + (bh * NC + c) * (int64_t)N;
    // packed rows a0 .. a0 + kSlotTile - 1 of the prefix state into buffer b (rows past N zero-filled)
    auto copy_tile = [&](int a0, int b) {
        float* St = Sb + b * kSlotTile * DV;
        for (int e = threadIdx.x; e < kSlotTile * (DV / 4); e += blockDim.x) {
            const bool in = a0 + e / (DV / 4) < N;
            tc::cp_async16(St + 4 * e, in ? Pc + (int64_t)a0 * DV + 4 * e : Pc, in ? 16u : 0u);
        }
        for (int e = threadIdx.x; e < kSlotTile / 4; e += blockDim.x) {
            const bool in = a0 + 4 * e < N;  // N - a0 rows are left; a partial vector is read as scalars below
            if (in && a0 + 4 * e + 4 <= N)
                tc::cp_async16(Zb + b * kSlotTile + 4 * e, Pzc + a0 + 4 * e, 16u);
            else
                for (int u = 0; u < 4; ++u) Zb[b * kSlotTile + 4 * e + u] = a0 + 4 * e + u < N ? Pzc[a0 + 4 * e + u] : 0.f;
        }
        tc::cp_async_commit();
    };
    // the chunk's query lifts of packed rows a0 .. into Pt; (aa, tt) from e by
    // shifts when the token count is a power of two (every full chunk)
    auto lift_tile = [&](int a0, auto pow2) {
        constexpr bool POW2 = decltype(pow2)::value;
        const int sh = __ffs(nt) - 1;
        for (int e = threadIdx.x; e < kSlotTile * nt; e += blockDim.x) {
            const int aa = POW2 ? e >> sh : e / nt, tt = POW2 ? e & (nt - 1) : e - aa * nt;
            const int i = Ii[aa], j = Jj[aa];
            const float scale = (i == j) ? 1.f : kSqrt2;
            Pt[aa * LDT + tt] = (tt < len && a0 + aa < N) ? Qs[tt * LDP + i] * Qs[tt * LDP + j] * scale : 0.f;
        }
    };
    const bool pow2 = (nt & (nt - 1)) == 0;
    copy_tile(0, 0);
    for (int a0 = 0, b = 0; a0 < N; a0 += kSlotTile, b ^= 1) {
        __syncthreads();  // the previous tile's readers are done (with Pt and with buffer b ^ 1)
        if (a0 + kSlotTile < N)
            copy_tile(a0 + kSlotTile, b ^ 1);
        else
            tc::cp_async_commit();  // (an empty group keeps the count of groups in flight fixed)
        if (threadIdx.x < kSlotTile) {
            int i = 0, j = 0;
            if (a0 + threadIdx.x < N) unpack_index(a0 + threadIdx.x, P, i, j);
            Ii[threadIdx.x] = i;
            Jj[threadIdx.x] = j;
        }
        tc::cp_async_wait<1>();  // this thread's copies of tile b have landed
        __syncthreads();         // everyone's, and the row indices
        if (pow2)
            lift_tile(a0, std::true_type{});
        else
            lift_tile(a0, std::false_type{});
        __syncthreads();
        const float* St = Sb + b * kSlotTile * DV;
        const float* Zt = Zb + b * kSlotTile;
        for (int r0 = 0; r0 < kSlotTile; r0 += CG) {
            accumulate_den(Pt, r0 + cg, Zt[r0 + cg]);
#pragma unroll
            for (int u = 0; u < CG; ++u) accumulate(Pt, St, r0 + u);
        }
    }
    tc::cp_async_wait<0>();
    // GATED: scaled by prod_{r=cC..t} gamma_r
    if constexpr (GATED) {
#pragma unroll
        for (int kt = 0; kt < KT; ++kt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * (tg0 + kt * TGT) + i;
                if (t < len) {
                    float h = 1.f;
                    for (int r = 0; r <= t; ++r) h *= gs[r];
                    den[kt][i] *= h;
#pragma unroll
                    for (int x = 0; x < 4; ++x) acc[kt][i][x] *= h;
                }
            }
    }
    // local part: sum_{s in c, s <= t} (GATED: prod_{r=s+1..t} gamma_r) (qh_t.kh_s)^2 [v_s | 1]
    for (int s0 = 0; s0 < len; s0 += kKeyTile) {
        __syncthreads();  // the previous tile's readers are done
        load_rows_unit<Tin, P>(k + bh * T * P, t0 + s0, kKeyTile, T, Ks, LDP);
        load_rows_plain<Tin, DV>(v + bh * T * DV, t0 + s0, kKeyTile, T, Vs, DV);
        __syncthreads();
        for (int e = threadIdx.x; e < kKeyTile * nt; e += blockDim.x) {
            const int ss = e / nt, tt = e - ss * nt, s = s0 + ss;
            float val = 0.f;
            if (tt < len && s <= tt) {
                float d = 0.f;
#pragma unroll 16
                for (int i = 0; i < P; ++i) d = fmaf(Qs[tt * LDP + i], Ks[ss * LDP + i], d);
                val = d * d;
                if constexpr (GATED) {
                    float decay = 1.f;
                    for (int r = tt; r > s; --r) decay *= gs[r];
                    val = decay * val;
                }
            }
            Sc[ss * LDT + tt] = val;
        }
        __syncthreads();
        for (int r0 = 0; r0 < kKeyTile; r0 += CG) {
            accumulate_den(Sc, r0 + cg, 1.f);
#pragma unroll
            for (int u = 0; u < CG; ++u) accumulate(Sc, Vs, r0 + u);
        }
    }
    // denominators: the CG threads of a token group are neighbouring lanes
#pragma unroll
    for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int off = 1; off < CG; off <<= 1) den[kt][i] += __shfl_xor_sync(0xffffffffu, den[kt][i], off);
#pragma unroll
    for (int kt = 0; kt < KT; ++kt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = 4 * (tg0 + kt * TGT) + i;
            if (t < len) {
                Tin* ot = o + (bh * T + t0 + t) * DV + 4 * cg;
#pragma unroll
                for (int x = 0; x < 4; ++x) store_as(ot + x, den[kt][i] > 0.f ? acc[kt][i][x] / den[kt][i] : 0.f);
            }
        }
}

}  // namespace chunk_out
}  // namespace
}  // namespace kata
