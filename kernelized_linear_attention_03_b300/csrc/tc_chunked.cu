// Exact O(T) chunked-state KATA forward on the tcgen05 tensor cores (bf16
// inputs, fp32 accumulation): the chunked-scan paragraph's decomposition
// fused into one kernel per (head, segment), with the running state kept on
// chip instead of being written to memory per chunk.
//
// Per chunk of 128 tokens, with S the state before the chunk, Z = sum k k^T
// over the same tokens (the p x p form of the normaliser z: psi(q)^T z =
// q^T Z q) and M the causal mask s <= t inside the chunk:
//   numerator   Y = psiQ(Q) S + ((Q Kh^T) o (Q Kh^T) o M) V
//   denominator d = rowdot(Q, Q Z) + rowsum((Q Kh^T) o (Q Kh^T) o M)
//   o = Y / d;   S += psiK(Kh)^T V;   Z += Kh^T Kh
// Q is used as given (its norm cancels between Y and d); Kh are the unit keys.
//
// The state of one head (n x dv fp32, n = p(p+1)/2) is spread over a
// thread-block cluster.  Each "tile CTA" owns two 128-slot tiles of the
// packed lift; it keeps its state rows in tensor memory (fp32, accumulated
// by the update MMA) and a bf16 copy in shared memory (B operand of the
// readout MMA).  Its query lift goes to tensor memory (A operand of the
// readout), its key lift to shared memory (A operand of the update).  The
// "extra CTA" owns the last, partly filled tile, the intra-chunk part and Z.
// Each CTA's partial Y (128 x dv fp32) is summed in distributed shared
// memory: CTA r owns rows [r*R, r*R + R) of the chunk, receives the partials
// of those rows from every CTA of the cluster (double-buffered by chunk
// parity), adds them, divides by d and stores o.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "kata_internal.h"
#include "tc_lift.cuh"
#include "tc_primitives.cuh"

namespace kata {
namespace {

using namespace tc;
namespace cg = cooperative_groups;

__device__ unsigned int g_chunked_tc_status = 0;

constexpr int kThreads = 128;
constexpr int kChunk = 128;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kAtom = 128 * 128;  // 128 rows x 128 bytes
constexpr float kSqrt2f = 1.41421356237309504880f;
constexpr float kInvSqrt2f = 0.70710678118654752440f;

__host__ __device__ constexpr uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

template <int P, int DV>
struct Cfg {
    static constexpr int n = lift::packed_n(P);
    static constexpr int NT = n / 128;                 // full tiles
    static constexpr int TAIL = n - 128 * NT;          // slots of the last tile (8, 16 or 32)
    static constexpr int TPC = NT >= 2 ? 2 : 1;        // tiles per tile CTA
    static constexpr int NTC = NT / TPC;               // tile CTAs
    static constexpr int CS = NTC + 1;                 // cluster size
    static constexpr int R = (kChunk + CS - 1) / CS;   // output rows owned per CTA
    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr uint32_t ak_off = 0;              // key lift, TPC tiles x 2 atoms
    static constexpr uint32_t q_off = 2 * kAtom;       // extra CTA: queries (K-major)
    static constexpr uint32_t kh_off = 3 * kAtom;      // extra CTA: unit keys (K-major)
    static constexpr uint32_t bv_off = 4 * kAtom;      // values (MN-major, N = dv)
    static constexpr uint32_t s16_off = 5 * kAtom;     // bf16 state rows, TPC tiles
    static constexpr uint32_t z16_off = 6 * kAtom;     // extra CTA: bf16 Z (K-major, P rows)
    static constexpr uint32_t recv_off = 7 * kAtom;
    static constexpr uint32_t recv_part = R * DV * 4;  // one CTA's partial rows
    static constexpr uint32_t recv_den = CS * recv_part;
    static constexpr uint32_t recv_buf = round16(recv_den + R * 4);
    static constexpr uint32_t total = recv_off + 2 * recv_buf;
    static constexpr size_t smem = total + 1024;
    // tensor memory columns
    static constexpr uint32_t tm_s = 0;                // tile CTA: TPC x 64 state columns
    static constexpr uint32_t tm_aq = 128;             // tile CTA: TPC x 64 query-lift columns
    static constexpr uint32_t tm_y = 256;              // tile CTA: partial Y
    static constexpr uint32_t tx_s = 0;                // extra CTA: tail state
    static constexpr uint32_t tx_aq = 64;              // extra CTA: tail query lift
    static constexpr uint32_t tx_y = 128;              // extra CTA: partial Y
    static constexpr uint32_t tx_sc = 192;             // extra CTA: scores (128 cols), P in place
    static constexpr uint32_t tx_w = 320;              // extra CTA: Q Z
    static constexpr uint32_t tx_z = 384;              // extra CTA: Z
    static_assert(NT % TPC == 0, "tiles must split evenly");
    static_assert(total + 1024 <= 232448, "shared memory");
};

// ---------------------------------------------------------------- lifts per tile
template <int P, int TAU>
__device__ __forceinline__ void key_tile(const uint32_t (&u)[P / 2], uint8_t* As, int row) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint4 val;
        val.x = lift::lift_word<P, false>(u, u, 64 * TAU + 4 * c + 0);
        val.y = lift::lift_word<P, false>(u, u, 64 * TAU + 4 * c + 1);
        val.z = lift::lift_word<P, false>(u, u, 64 * TAU + 4 * c + 2);
        val.w = lift::lift_word<P, false>(u, u, 64 * TAU + 4 * c + 3);
        *reinterpret_cast<uint4*>(As + mn_sw128_chunk(8 * c, row, kAtom)) = val;
    }
}

template <int P, int TAU>
__device__ __forceinline__ void query_tile(const uint32_t (&u)[P / 2], const uint32_t (&u2)[P / 2],
                                           uint32_t taddr) {
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = lift::lift_word<P, true>(u, u2, 64 * TAU + c0 + i);
        tmem_st16(taddr + c0, w);
    }
}

template <int P, int TAU = 0>
__device__ __forceinline__ void lift_tile(int tau, const uint32_t (&uk)[P / 2], const uint32_t (&uq)[P / 2],
                                          const uint32_t (&uq2)[P / 2], uint8_t* As, int row, uint32_t taddr) {
    if constexpr (TAU < lift::tiles_of(P)) {
        if (tau == TAU) {
            key_tile<P, TAU>(uk, As, row);
            query_tile<P, TAU>(uq, uq2, taddr);
        } else {
            lift_tile<P, TAU + 1>(tau, uk, uq, uq2, As, row, taddr);
        }
    }
}

// ---------------------------------------------------------------- state rows
// Thread t holds lane t of a 128-slot tile: load its start row (C ABI packed
// order, sqrt(2) removed) into tensor memory and the bf16 copy.
template <int P, int DV>
__device__ __forceinline__ void load_state_tile(const float* S_start, int tau, uint32_t taddr, uint8_t* S16,
                                                int t) {
    constexpr int n = lift::packed_n(P);
    const int slot = tau * 128 + t;
    float x[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) x[c] = 0.f;
    if (S_start != nullptr && slot < n) {
        int i = 0, j = 0;
        lift::slot_coord(P, slot, i, j);
        const float f = i < j ? kInvSqrt2f : 1.f;
        const float4* src = reinterpret_cast<const float4*>(S_start + (int64_t)lift::canonical_index(P, i, j) * DV);
#pragma unroll
        for (int c = 0; c < DV / 4; ++c) {
            const float4 a = src[c];
            x[4 * c] = a.x * f;
            x[4 * c + 1] = a.y * f;
            x[4 * c + 2] = a.z * f;
            x[4 * c + 3] = a.w * f;
        }
    }
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 16) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(x[c0 + i]);
        tmem_st16(taddr + c0, r);
    }
#pragma unroll
    for (int c = 0; c < DV / 8; ++c) {
        uint4 w;
        w.x = pack_bf16x2(x[8 * c], x[8 * c + 1]);
        w.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
        w.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
        w.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
        *reinterpret_cast<uint4*>(S16 + mn_sw128_chunk(8 * c, t, kAtom)) = w;
    }
}

// Refresh the bf16 copy of lane t of a state tile from tensor memory.
template <int DV>
__device__ __forceinline__ void refresh_state_tile(uint32_t taddr, uint8_t* S16, int t) {
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + c0, r);
        tmem_wait_ld();
        uint4 a, b;
        a.x = pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1]));
        a.y = pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3]));
        a.z = pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5]));
        a.w = pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7]));
        b.x = pack_bf16x2(__uint_as_float(r[8]), __uint_as_float(r[9]));
        b.y = pack_bf16x2(__uint_as_float(r[10]), __uint_as_float(r[11]));
        b.z = pack_bf16x2(__uint_as_float(r[12]), __uint_as_float(r[13]));
        b.w = pack_bf16x2(__uint_as_float(r[14]), __uint_as_float(r[15]));
        *reinterpret_cast<uint4*>(S16 + mn_sw128_chunk(c0, t, kAtom)) = a;
        *reinterpret_cast<uint4*>(S16 + mn_sw128_chunk(c0 + 8, t, kAtom)) = b;
    }
}

// Write lane t of a state tile to the C ABI's packed order (sqrt(2) restored).
template <int P, int DV>
__device__ __forceinline__ void store_state_tile(float* S_out, int tau, uint32_t taddr, int t) {
    constexpr int n = lift::packed_n(P);
    const int slot = tau * 128 + t;
    uint32_t r[DV];
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 16) {
        uint32_t q[16];
        tmem_ld16(taddr + c0, q);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[c0 + i] = q[i];
    }
    tmem_wait_ld();
    if (slot < n) {
        int i = 0, j = 0;
        lift::slot_coord(P, slot, i, j);
        const float f = i < j ? kSqrt2f : 1.f;
        float4* dst = reinterpret_cast<float4*>(S_out + (int64_t)lift::canonical_index(P, i, j) * DV);
#pragma unroll
        for (int c = 0; c < DV / 4; ++c)
            dst[c] = make_float4(f * __uint_as_float(r[4 * c]), f * __uint_as_float(r[4 * c + 1]),
                                 f * __uint_as_float(r[4 * c + 2]), f * __uint_as_float(r[4 * c + 3]));
    }
}

// ---------------------------------------------------------------- kernel
template <int P, int DV>
__global__ void __launch_bounds__(kThreads, 1)
chunked_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, __nv_bfloat16* __restrict__ o,
                  const float* __restrict__ S_start, const float* __restrict__ z_start, int start_groups,
                  float* __restrict__ S_final, float* __restrict__ z_final, int T, int seg_chunks) {
    using K = Cfg<P, DV>;
    constexpr int n = K::n;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int t = threadIdx.x, warp = t >> 5;
    const int rank = (int)cluster.block_rank();
    const bool extra = rank == K::NTC;
    const int g = blockIdx.x / K::CS;
    const int G = gridDim.x / K::CS;
    const int64_t bh = blockIdx.y;
    const int NCH = (T + kChunk - 1) / kChunk;
    const int c_begin = g * seg_chunks, c_end = min(NCH, c_begin + seg_chunks);
    const __nv_bfloat16* qh = q + bh * (int64_t)T * P;
    const __nv_bfloat16* kh = k + bh * (int64_t)T * P;
    const __nv_bfloat16* vh = v + bh * (int64_t)T * DV;
    __nv_bfloat16* oh = o + bh * (int64_t)T * DV;

    if (t == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t lane0 = (uint32_t)(warp * 32);
    auto tm = [&](uint32_t col) { return tmem_addr(tb, lane0, col); };

    // ---- start state of this segment
    const int sg = start_groups > 1 ? g : 0;
    const float* S0 = S_start ? S_start + (bh * start_groups + sg) * (int64_t)n * DV : nullptr;
    const float* z0 = z_start ? z_start + (bh * start_groups + sg) * (int64_t)n : nullptr;
    if (!extra) {
#pragma unroll
        for (int tl = 0; tl < K::TPC; ++tl)
            load_state_tile<P, DV>(S0, rank * K::TPC + tl, tm(K::tm_s + 64 * tl), sm + K::s16_off + tl * kAtom, t);
    } else {
        load_state_tile<P, DV>(S0, K::NT, tm(K::tx_s), sm + K::s16_off, t);
        // Z row t (t < P) from the packed normaliser: Z_ij = z_idx(i,j) / (sqrt2 if i != j)
        float zr[P];
#pragma unroll
        for (int j = 0; j < P; ++j) {
            float val = 0.f;
            if (z0 != nullptr && t < P) {
                const int a = t < j ? t : j, b = t < j ? j : t;
                val = z0[lift::canonical_index(P, a, b)] * (a == b ? 1.f : kInvSqrt2f);
            }
            zr[j] = val;
        }
#pragma unroll
        for (int c0 = 0; c0 < P; c0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(zr[c0 + i]);
            tmem_st16(tm(K::tx_z + c0), r);
        }
        if (t < P) {
#pragma unroll
            for (int c = 0; c < P / 8; ++c) {
                uint4 w;
                w.x = pack_bf16x2(zr[8 * c], zr[8 * c + 1]);
                w.y = pack_bf16x2(zr[8 * c + 2], zr[8 * c + 3]);
                w.z = pack_bf16x2(zr[8 * c + 4], zr[8 * c + 5]);
                w.w = pack_bf16x2(zr[8 * c + 6], zr[8 * c + 7]);
                *reinterpret_cast<uint4*>(sm + K::z16_off + sw128_chunk(t, 8 * c, P)) = w;
            }
        }
    }
    tmem_wait_st();

    uint32_t phase = 0;
    bool ok = true;
    const int owner = t / K::R, orow = t % K::R;

    for (int c = c_begin; c < c_end; ++c) {
        const int tok = c * kChunk + t;
        const bool valid = tok < T;
        const int buf = (c - c_begin) & 1;
        uint8_t* recv = sm + K::recv_off + buf * K::recv_buf;
        // ---- this token's rows
        uint4 qraw[P / 8], kraw[P / 8];
        uint32_t uq[P / 2], uq2[P / 2], uk[P / 2];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < P / 8; ++i) {
            qraw[i] = valid ? *reinterpret_cast<const uint4*>(qh + (int64_t)tok * P + 8 * i) : make_uint4(0, 0, 0, 0);
            kraw[i] = valid ? *reinterpret_cast<const uint4*>(kh + (int64_t)tok * P + 8 * i) : make_uint4(0, 0, 0, 0);
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(&qraw[i]);
            const __nv_bfloat16* ke = reinterpret_cast<const __nv_bfloat16*>(&kraw[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uq[4 * i + j] = qw[j];
                uq2[4 * i + j] = lift::bf16x2_mul(qw[j], 0x40004000u);  // 2q, exact
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = __bfloat162float(ke[j]);
                ss = fmaf(x, x, ss);
            }
        }
        const float kinv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
        for (int i = 0; i < P / 8; ++i) {
            const __nv_bfloat16* ke = reinterpret_cast<const __nv_bfloat16*>(&kraw[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                uk[4 * i + j] = pack_bf16x2(__bfloat162float(ke[2 * j]) * kinv, __bfloat162float(ke[2 * j + 1]) * kinv);
        }
        // ---- lifts (query -> tensor memory, key -> shared memory)
        if (!extra) {
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl)
                lift_tile<P>(rank * K::TPC + tl, uk, uq, uq2, sm + K::ak_off + 2 * tl * kAtom, t,
                             tm(K::tm_aq + 64 * tl));
        } else {
            lift_tile<P>(K::NT, uk, uq, uq2, sm + K::ak_off, t, tm(K::tx_aq));
#pragma unroll
            for (int i = 0; i < P / 8; ++i) {
                *reinterpret_cast<uint4*>(sm + K::q_off + sw128_chunk(t, 8 * i, kChunk)) = qraw[i];
                *reinterpret_cast<uint4*>(sm + K::kh_off + sw128_chunk(t, 8 * i, kChunk)) =
                    make_uint4(uk[4 * i], uk[4 * i + 1], uk[4 * i + 2], uk[4 * i + 3]);
            }
        }
#pragma unroll
        for (int i = 0; i < DV / 8; ++i) {
            const uint4 val = valid ? *reinterpret_cast<const uint4*>(vh + (int64_t)tok * DV + 8 * i)
                                    : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sm + K::bv_off + mn_sw128_chunk(8 * i, t, kAtom)) = val;
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA group 1
        if (t == 0 && ok) {
            tc_fence_after();
            const uint32_t sb = smem_u32(sm);
            constexpr uint32_t id_read = idesc_bf16_f32_major(128, DV, false, true);
            constexpr uint32_t id_upd = idesc_bf16_f32_major(128, DV, true, true);
            const uint64_t bv0 = sdesc_mnmajor_sw128(sb + K::bv_off, kAtom);
            if (!extra) {
#pragma unroll 1
                for (int tl = 0; tl < K::TPC; ++tl)
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts(tb + K::tm_y, tb + K::tm_aq + 64 * tl + 8 * ks,
                               sdesc_mnmajor_sw128(sb + K::s16_off + tl * kAtom + ks * 2048, kAtom), id_read,
                               (tl > 0 || ks > 0) ? 1u : 0u);
#pragma unroll 1
                for (int tl = 0; tl < K::TPC; ++tl)
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss(tb + K::tm_s + 64 * tl,
                               sdesc_mnmajor_sw128(sb + K::ak_off + 2 * tl * kAtom + ks * 2048, kAtom),
                               bv0 + (uint64_t)((ks * 2048) >> 4), id_upd, 1u);
            } else {
                // tail tile: readout over its TAIL slots, update
                for (int ks = 0; ks < (K::TAIL + 15) / 16; ++ks)
                    mma_ts(tb + K::tx_y, tb + K::tx_aq + 8 * ks,
                           sdesc_mnmajor_sw128(sb + K::s16_off + ks * 2048, kAtom), id_read, ks > 0 ? 1u : 0u);
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tb + K::tx_s, sdesc_mnmajor_sw128(sb + K::ak_off + ks * 2048, kAtom),
                           bv0 + (uint64_t)((ks * 2048) >> 4), id_upd, 1u);
                // intra scores Q Kh^T and Q Z
                constexpr uint32_t id_sc = idesc_bf16_f32(128, 128);
                constexpr uint32_t id_w = idesc_bf16_f32(128, P);
                for (int ks = 0; ks < P / 16; ++ks) {
                    const uint64_t qd = sdesc_kmajor_sw128(sb + K::q_off + ks * 32);
                    mma_ss(tb + K::tx_sc, qd, sdesc_kmajor_sw128(sb + K::kh_off + ks * 32), id_sc, ks > 0 ? 1u : 0u);
                    mma_ss(tb + K::tx_w, qd, sdesc_kmajor_sw128(sb + K::z16_off + ks * 32), id_w, ks > 0 ? 1u : 0u);
                }
                // Z += Kh^T Kh (A: unit keys viewed MN-major, both M atoms on the same data)
                constexpr uint32_t id_z = idesc_bf16_f32_major(128, P, true, true);
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tb + K::tx_z, sdesc_mnmajor_sw128(sb + K::kh_off + ks * 2048, 0),
                           sdesc_mnmajor_sw128(sb + K::kh_off + ks * 2048, kAtom), id_z, 1u);
            }
            mma_commit(&bar);
        }
        if (ok) {
            ok = mbar_wait(&bar, phase, &abort_flag, kWaitNs);
            phase ^= 1;
            if (!ok) abort_flag = 1;
        }
        ok = __syncthreads_and(ok);
        tc_fence_after();

        float den = 0.f;
        if (extra) {
            // ---- P = (Q Kh^T)^2 masked, in place as bf16; intra denominator
            float dsum = 0.f;
            if (ok) {
#pragma unroll 1
                for (int c0 = 0; c0 < kChunk; c0 += 32) {
                    uint32_t s0[16], s1[16], pk[16];
                    tmem_ld16(tm(K::tx_sc + c0), s0);
                    tmem_ld16(tm(K::tx_sc + c0 + 16), s1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float a = __uint_as_float(s0[2 * i]), b = __uint_as_float(s0[2 * i + 1]);
                        float cc = __uint_as_float(s1[2 * i]), d = __uint_as_float(s1[2 * i + 1]);
                        a = (c0 + 2 * i <= t) ? a * a : 0.f;
                        b = (c0 + 2 * i + 1 <= t) ? b * b : 0.f;
                        cc = (c0 + 16 + 2 * i <= t) ? cc * cc : 0.f;
                        d = (c0 + 16 + 2 * i + 1 <= t) ? d * d : 0.f;
                        pk[i] = pack_bf16x2(a, b);
                        pk[8 + i] = pack_bf16x2(cc, d);
                        const __nv_bfloat162 h0 = *reinterpret_cast<const __nv_bfloat162*>(&pk[i]);
                        const __nv_bfloat162 h1 = *reinterpret_cast<const __nv_bfloat162*>(&pk[8 + i]);
                        dsum += (__low2float(h0) + __high2float(h0)) + (__low2float(h1) + __high2float(h1));
                    }
                    tmem_st16(tm(K::tx_sc + c0 / 2), pk);
                }
                // inter denominator q^T Z q from W = Q Z
                float dint = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < P; c0 += 16) {
                    uint32_t w[16];
                    tmem_ld16(tm(K::tx_w + c0), w);
                    tmem_wait_ld();
                    const __nv_bfloat16* qe = reinterpret_cast<const __nv_bfloat16*>(qraw) + c0;
#pragma unroll
                    for (int i = 0; i < 16; ++i) dint = fmaf(__bfloat162float(qe[i]), __uint_as_float(w[i]), dint);
                }
                den = dsum + dint;
            }
            tmem_wait_st();
            tc_fence_before();
            __syncthreads();
            // ---- MMA group 2: Y += P V
            if (t == 0 && ok) {
                tc_fence_after();
                const uint32_t sb = smem_u32(sm);
                constexpr uint32_t id_pv = idesc_bf16_f32_major(128, DV, false, true);
                for (int ks = 0; ks < 8; ++ks)
                    mma_ts(tb + K::tx_y, tb + K::tx_sc + 8 * ks,
                           sdesc_mnmajor_sw128(sb + K::bv_off + ks * 2048, kAtom), id_pv, 1u);
                mma_commit(&bar);
            }
            // ---- meanwhile: bf16 copies of Z and of the tail state
            {
                uint32_t zr[P];
#pragma unroll
                for (int c0 = 0; c0 < P; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tx_z + c0), r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) zr[c0 + i] = r[i];
                }
                tmem_wait_ld();
                if (t < P) {
#pragma unroll
                    for (int c8 = 0; c8 < P / 8; ++c8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(zr[8 * c8]), __uint_as_float(zr[8 * c8 + 1]));
                        w.y = pack_bf16x2(__uint_as_float(zr[8 * c8 + 2]), __uint_as_float(zr[8 * c8 + 3]));
                        w.z = pack_bf16x2(__uint_as_float(zr[8 * c8 + 4]), __uint_as_float(zr[8 * c8 + 5]));
                        w.w = pack_bf16x2(__uint_as_float(zr[8 * c8 + 6]), __uint_as_float(zr[8 * c8 + 7]));
                        *reinterpret_cast<uint4*>(sm + K::z16_off + sw128_chunk(t, 8 * c8, P)) = w;
                    }
                }
            }
            refresh_state_tile<DV>(tm(K::tx_s), sm + K::s16_off, t);
            if (ok) {
                ok = mbar_wait(&bar, phase, &abort_flag, kWaitNs);
                phase ^= 1;
                if (!ok) abort_flag = 1;
            }
            ok = __syncthreads_and(ok);
            tc_fence_after();
        } else {
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl)
                refresh_state_tile<DV>(tm(K::tm_s + 64 * tl), sm + K::s16_off + tl * kAtom, t);
        }

        // ---- partial Y (and d) to the owner of this row
        {
            const uint32_t ycol = extra ? K::tx_y : K::tm_y;
            float* dst = cluster.map_shared_rank(
                reinterpret_cast<float*>(recv + rank * K::recv_part + orow * DV * 4), owner);
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tm(ycol + c0), r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    reinterpret_cast<float4*>(dst + c0)[i] =
                        make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                    __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
            }
            if (extra) {
                float* ddst = cluster.map_shared_rank(reinterpret_cast<float*>(recv + K::recv_den + orow * 4), owner);
                *ddst = den;
            }
        }
        tc_fence_before();
        cluster.sync();
        tc_fence_after();

        // ---- owned rows: sum the partials, divide, store
        {
            const int r0 = rank * K::R;
            const int rows = min(K::R, kChunk - r0);
            for (int e = t; e < rows * (DV / 2); e += kThreads) {
                const int lr = e / (DV / 2), col = 2 * (e % (DV / 2));
                float a = 0.f, b = 0.f;
#pragma unroll
                for (int src = 0; src < K::CS; ++src) {
                    const float2 x = *reinterpret_cast<const float2*>(recv + src * K::recv_part + (lr * DV + col) * 4);
                    a += x.x;
                    b += x.y;
                }
                const float d = *reinterpret_cast<const float*>(recv + K::recv_den + lr * 4);
                const float inv = d > 0.f ? 1.f / d : 0.f;
                const int otok = c * kChunk + r0 + lr;
                if (otok < T)
                    *reinterpret_cast<__nv_bfloat162*>(oh + (int64_t)otok * DV + col) =
                        __floats2bfloat162_rn(a * inv, b * inv);
            }
        }
    }

    // ---- final state of the last segment
    if (S_final != nullptr && g == G - 1) {
        const int64_t head_s = bh * (int64_t)n * DV, head_z = bh * (int64_t)n;
        if (!extra) {
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl)
                store_state_tile<P, DV>(S_final + head_s, rank * K::TPC + tl, tm(K::tm_s + 64 * tl), t);
        } else {
            store_state_tile<P, DV>(S_final + head_s, K::NT, tm(K::tx_s), t);
            uint32_t zr[P];
#pragma unroll
            for (int c0 = 0; c0 < P; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tm(K::tx_z + c0), r);
#pragma unroll
                for (int i = 0; i < 16; ++i) zr[c0 + i] = r[i];
            }
            tmem_wait_ld();
            if (t < P) {
#pragma unroll
                for (int j = 0; j < P; ++j)
                    if (j >= t)
                        z_final[head_z + lift::canonical_index(P, t, j)] =
                            __uint_as_float(zr[j]) * (j == t ? 1.f : kSqrt2f);
            }
        }
    }
    if (!ok && t == 0) atomicOr(&g_chunked_tc_status, kStatusTimeout);
    if (!ok) mbar_wait_quiet(&bar, phase ^ 1, kWaitNs / 4);
    tc_fence_before();
    cluster.sync();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------- host side
template <int P, int DV>
cudaError_t configure(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int G, int BH, cudaStream_t s) {
    using K = Cfg<P, DV>;
    auto kern = chunked_tc_kernel<P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K::smem);
    if (e == cudaSuccess && K::CS > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(K::CS * G, BH, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = K::smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = K::CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaSuccess;
}

template <int P, int DV>
int max_clusters() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[1];
        int m = 0;
        if (configure<P, DV>(cfg, attr, 1, 1, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&m, chunked_tc_kernel<P, DV>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cached[dev] = m > 0 ? m : -1;
    }
    return cached[dev] > 0 ? cached[dev] : 0;
}

template <int P, int DV>
cudaError_t launch_typed(const void* q, const void* k, const void* v, void* o, const float* S_start,
                         const float* z_start, int start_groups, float* S_final, float* z_final, int BH, int T,
                         int seg_chunks, int G, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    cudaError_t e = configure<P, DV>(cfg, attr, G, BH, s);
    if (e != cudaSuccess) return e;
    KATA_TRACED("chunked_tc", s,
                e = cudaLaunchKernelEx(&cfg, chunked_tc_kernel<P, DV>, static_cast<const __nv_bfloat16*>(q),
                                       static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                                       static_cast<__nv_bfloat16*>(o), S_start, z_start, start_groups, S_final,
                                       z_final, T, seg_chunks));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

#define KATA_DISPATCH(...)                                              \
    do {                                                                 \
        if (p == 16 && dv == 16) { constexpr int P = 16, DV = 16; __VA_ARGS__; } \
        if (p == 16 && dv == 32) { constexpr int P = 16, DV = 32; __VA_ARGS__; } \
        if (p == 16 && dv == 64) { constexpr int P = 16, DV = 64; __VA_ARGS__; } \
        if (p == 32 && dv == 16) { constexpr int P = 32, DV = 16; __VA_ARGS__; } \
        if (p == 32 && dv == 32) { constexpr int P = 32, DV = 32; __VA_ARGS__; } \
        if (p == 32 && dv == 64) { constexpr int P = 32, DV = 64; __VA_ARGS__; } \
        if (p == 64 && dv == 16) { constexpr int P = 64, DV = 16; __VA_ARGS__; } \
        if (p == 64 && dv == 32) { constexpr int P = 64, DV = 32; __VA_ARGS__; } \
        if (p == 64 && dv == 64) { constexpr int P = 64, DV = 64; __VA_ARGS__; } \
    } while (0)

int chunked_tc_segments(int p, int dv, int BH, int T) {
    const int nch = (T + kChunk - 1) / kChunk;
    int m = 0;
    KATA_DISPATCH(m = max_clusters<P, DV>());
    if (m <= 0) return 0;
    if (nch <= 0) return 1;
    int G = m / (BH > 0 ? BH : 1);
    if (G < 1) G = 1;
    if (G > nch) G = nch;
    const int per = (nch + G - 1) / G;
    return (nch + per - 1) / per;
}

int chunked_tc_segment_chunks(int T, int G) {
    const int nch = (T + kChunk - 1) / kChunk;
    return (nch + G - 1) / G;
}

cudaError_t launch_chunked_tc(const void* q, const void* k, const void* v, void* o, const float* S_start,
                              const float* z_start, int start_groups, float* S_final, float* z_final, int BH,
                              int T, int p, int dv, int G, cudaStream_t s) {
    const int seg_chunks = chunked_tc_segment_chunks(T, G);
    KATA_DISPATCH(return launch_typed<P, DV>(q, k, v, o, S_start, z_start, start_groups, S_final, z_final, BH, T,
                                             seg_chunks, G, s));
    return cudaErrorInvalidValue;
}

unsigned int chunked_tc_take_status() {
    unsigned int val = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&val, g_chunked_tc_status, sizeof(val)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_chunked_tc_status, &zero, sizeof(zero));
    return val;
}

}  // namespace kata
