// Gated chunked forward on CUDA cores (fp32 arithmetic, any input dtype).
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
#include <type_traits>

#include "kata_device.cuh"
#include "kata_internal.h"
#include "tc_primitives.cuh"

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

// ---------------------------------------------------------------- chunk output
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
//                   then scaled by the decay from the chunk's start,
//                   prod_{r=cC..t} gamma_r
//   local part      per tile of kKeyTile keys: the decayed squared scores
//                   prod_{r=s+1..t} gamma_r (qh_t.kh_s)^2 (keys x tokens) and
//                   the values, accumulated the same way
// Each (token, column) sum runs over the packed rows, then over the keys, in
// order.  The denominators' products are shared out over the CG threads of a
// token group (thread cg takes rows cg, cg + CG, ...) and summed by shuffles
// at the end.
template <typename Tin, int P, int DV>
__global__ void __launch_bounds__(kThreads, 2)
gated_output_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
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
    // scaled by prod_{r=cC..t} gamma_r
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
    // local part: sum_{s in c, s <= t} prod_{r=s+1..t} gamma_r (qh_t.kh_s)^2 [v_s | 1]
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
                float decay = 1.f;
                for (int r = tt; r > s; --r) decay *= gs[r];
                val = decay * (d * d);
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
    constexpr size_t smem = output_smem_bytes<P, DV>();
    auto kern = gated_output_kernel<Tin, P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    KATA_TRACED("gated_output_simt", s,
                kern<<<dim3(NC, BH), kThreads, smem, s>>>(static_cast<const Tin*>(q), static_cast<const Tin*>(k),
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
