// Exact O(T) chunked-state KATA forward on the tcgen05 tensor cores (bf16
// inputs, fp32 accumulation): the chunked-scan paragraph's decomposition with
// the running state kept on chip instead of being written to memory per
// chunk.
//
// Per chunk of 128 tokens, with S the state before the chunk, Z = sum k k^T
// over the same tokens (the p x p form of the normaliser z: psi(q)^T z =
// q^T Z q) and M the causal mask s <= t inside the chunk:
//   numerator   Y = psiQ(Q) S + ((Q Kh^T) o (Q Kh^T) o M) V
//   denominator d = rowdot(Q, Q Z) + rowsum((Q Kh^T) o (Q Kh^T) o M)
//   o = Y / d;   S += psiK(Kh)^T V;   Z += Kh^T Kh
// Q is used as given (its norm cancels between Y and d); Kh are the unit keys.
//
// Three kernels.  The intra-chunk kernel computes every chunk's local part
// (the masked squared scores times V, and their row sums) into fp32
// accumulation rows Y[BH][Tc][dv], d[BH][Tc], and the chunk's unit keys
// transposed for the key lift.  The state kernel then runs one CTA per
// (head, segment, 128-slot tile of the packed lift): the CTA keeps its tile
// of the state (128 x dv fp32) in tensor memory and a bf16 copy in shared
// memory, lifts the chunk's keys and queries for its slots into tensor
// memory, updates its state rows and adds its partial readout psiQ(Q) S_tile
// to Y with a TMA reduce-add.  One more CTA per (head, segment) keeps Z and
// adds the inter-chunk denominators to d.  The CTAs of a head
// share nothing but the accumulation rows, so they need no cluster and fill
// the GPU independently.  A last pass writes o = Y / d.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "kata_internal.h"
#include "tc_lift.cuh"
#include "tc_primitives.cuh"
#include "tc_tma.cuh"

namespace kata {
namespace {

using namespace tc;

__device__ unsigned int g_chunked_tc_status = 0;

constexpr int kThreads = 512;  // warpgroups: query lift and output, state epilogue, key lift, MMA and loads
// Register split between the warpgroups after launch (setmaxnreg): the MMA
// warpgroup gives back registers that the query warpgroup takes.
// 128 * (kRegsLift + kRegsState + kRegsLaunch + kRegsMma) must not exceed
// 512 * (registers per thread at launch); the launcher checks that.
constexpr uint32_t kRegsLift = 168, kRegsState = 128, kRegsLaunch = 128, kRegsMma = 88;
constexpr int kChunk = 128;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kAtom = 128 * 128;  // 128 rows x 128 bytes
// transposed unit keys of a chunk in memory: P rows of 128 tokens (bf16) and
// a 16-byte pad
constexpr int kKtCols = kChunk + 8;
constexpr uint32_t kKtRow = kKtCols * 2;
constexpr float kSqrt2f = 1.41421356237309504880f;
constexpr float kInvSqrt2f = 0.70710678118654752440f;

// P: width of q and k; LG: blocks of the lift (1: the full lift; g > 1: the
// KATA-Sigma-g lift, the sum of the g block lifts of width M = P / g).
template <int P, int DV, int LG>
struct Cfg {
    static constexpr int M = P / LG;                   // width of the lifted blocks
    static constexpr int n = lift::packed_n(M);
    static constexpr int NT = n / 128;                 // full tiles
    static constexpr int TAIL = n - 128 * NT;          // slots of the last tile (8, 16 or 32)
    static constexpr int CS = NT + 2;                  // CTAs per head and segment: one per tile, one for Z
    // transposed unit keys of a chunk: in a tile CTA one bulk copy of the
    // padded rows (P x kKtRow bytes); in the normaliser CTA two 64-token boxes
    // of P rows x 128 bytes (128-byte swizzle, the MMA operand layout)
    static constexpr uint32_t kt_box = P * 128;
    static constexpr uint32_t kt_bytes = 2 * kt_box;
    static constexpr uint32_t kt_rows_bytes = P * kKtRow;
    // partial readout staged for the reduce-add: YH boxes of 128 rows x YW
    // fp32 columns (128-byte rows for YW = 32)
    static constexpr int YW = DV < 32 ? DV : 32;
    static constexpr int YH = DV / YW;
    static constexpr uint32_t y_box = 128 * YW * 4;
    static constexpr uint32_t y_stage = YH * y_box;
    // shared memory, in 16 KB atoms from a 1024-byte aligned base: V x2,
    // bf16 state, query stages x2, bf16 Z (normaliser CTA), transposed-key
    // stages (three atoms: two padded stages in a tile CTA; two swizzled
    // stages and a spare atom in the normaliser CTA, whose M = 128 reads of
    // the Z update run past the last stage), then two partial-readout stages
    static constexpr uint32_t o_v = 0, o_s16 = 2 * kAtom, o_q = 3 * kAtom, o_z16 = 5 * kAtom, o_kt = 6 * kAtom,
                              o_y = 9 * kAtom;
    static constexpr uint32_t total = o_y + 2 * y_stage;
    static constexpr size_t smem = total + 1024;
    // tensor memory columns
    static constexpr uint32_t tm_s = 0;      // 64: fp32 state tile
    // key-lift buffers: two, so that the lift of the next chunk overlaps this
    // chunk's update (with the readouts issued by a warp of their own: 2-4%
    // faster than one buffer at p = 64)
    static constexpr int AKB = 2;
    static constexpr uint32_t tm_ak = 64;    // AKB slots x 64: key lift (bf16 pairs of tokens); the last tile's lanes past the tail hold zeros
    static constexpr uint32_t tm_aq = 64 + 64 * AKB;  // 2 slots x 64: query lift (bf16 pairs of slots)
    static constexpr uint32_t tm_y = tm_aq + 128;    // 2 slots x 64: partial readout
    static constexpr uint32_t tm_w = 384;    // normaliser CTA (which has no tile): Q Z
    static constexpr uint32_t tm_z = 448;    // normaliser CTA: Z
    static_assert(TAIL > 0 && TAIL <= 32, "tail tile");
    static_assert(tm_y + 128 <= 512, "tensor memory columns");
    static_assert(total + 4096 <= 232448, "shared memory");
    static_assert(kt_bytes <= kAtom && 2 * kt_rows_bytes <= 3 * kAtom, "transposed-key stages");
    static_assert(DV % YW == 0 && DV <= 64, "value width");
};

// ---------------------------------------------------------------- key lift, one slot per thread
// The key lift of internal slot (i, j) for the 128 tokens of a chunk comes
// from the chunk's transposed unit keys `kts` (row d = dimension d over the
// tokens, kKtRow bytes apart: 128 tokens and a 16-byte pad, so that rows
// d, d+1, ... start in consecutive 16-byte bank groups and a warp reading one
// 16-byte piece of 32 consecutive rows is conflict-free): k_i k_j for the
// full lift, sum_a k_{aM+i} k_{aM+j} over the LG blocks of width M for
// KATA-Sigma-g.  Consecutive tokens sit side by side in both rows, so the 16
// bytes of tokens [8g, 8g + 8) are four bf16x2 multiplies of two 16-byte
// loads at compile-time offsets from the two rows.
// 16 bytes at shared address a + OFF.
template <int OFF>
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4 + %5];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(a), "n"(OFF)
                 : "memory");
    return r;
}

template <int LG, int G>
__device__ __forceinline__ uint4 key_words(const uint32_t (&ri)[LG], const uint32_t (&rj)[LG]) {
    uint4 r;
#pragma unroll
    for (int blk = 0; blk < LG; ++blk) {
        const uint4 a = lds128<16 * G>(ri[blk]);
        const uint4 b = lds128<16 * G>(rj[blk]);
        if (blk == 0) {
            r.x = hmul2_bf16(a.x, b.x);
            r.y = hmul2_bf16(a.y, b.y);
            r.z = hmul2_bf16(a.z, b.z);
            r.w = hmul2_bf16(a.w, b.w);
        } else {
            r.x = hfma2_bf16(a.x, b.x, r.x);
            r.y = hfma2_bf16(a.y, b.y, r.y);
            r.z = hfma2_bf16(a.z, b.z, r.z);
            r.w = hfma2_bf16(a.w, b.w, r.w);
        }
    }
    return r;
}

// Lane `slot % 128` of a tensor-memory operand (64 columns, column c = the
// bf16 pair of tokens 2c, 2c+1) receives the key lift of slot `slot`, a
// quarter of the chunk (32 tokens) per tensor-memory store; slots past n
// give zeros.
template <int P, int LG>
__device__ __forceinline__ void key_row_tmem(const uint8_t* kts, int slot, uint32_t taddr) {
    constexpr int M = P / LG;
    constexpr int n = lift::packed_n(M);
    const bool live = slot < n;
    int i = 0, j = 0;
    if (live) lift::slot_coord(M, slot, i, j);
    uint32_t ri[LG], rj[LG];  // shared addresses of the factor rows
#pragma unroll
    for (int blk = 0; blk < LG; ++blk) {
        ri[blk] = smem_u32(kts) + (uint32_t)(blk * M + i) * kKtRow;
        rj[blk] = smem_u32(kts) + (uint32_t)(blk * M + j) * kKtRow;
    }
    // one quarter (32 tokens) at a time: a rolled loop keeps the loads of one
    // quarter in flight, within the warpgroup's registers
#pragma unroll 1
    for (int qt = 0; qt < 4; ++qt) {
        uint32_t w[16];
        uint4 r[4];
        if (live) {
            r[0] = key_words<LG, 0>(ri, rj);
            r[1] = key_words<LG, 1>(ri, rj);
            r[2] = key_words<LG, 2>(ri, rj);
            r[3] = key_words<LG, 3>(ri, rj);
        } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) r[cc] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            w[4 * cc] = r[cc].x;
            w[4 * cc + 1] = r[cc].y;
            w[4 * cc + 2] = r[cc].z;
            w[4 * cc + 3] = r[cc].w;
        }
        tmem_st16(taddr + 16 * qt, w);
#pragma unroll
        for (int blk = 0; blk < LG; ++blk) {
            ri[blk] += 64;
            rj[blk] += 64;
        }
    }
}

// ---------------------------------------------------------------- query lifts per tile
// Query lift word w (slots 2w, 2w+1 of the lift of width M): for KATA-Sigma-g
// the sum of the LG block lifts (bf16x2 additions).
template <int P, int LG>
__device__ __forceinline__ uint32_t query_word(const uint32_t (&u)[P / 2], int w) {
    constexpr int M = P / LG;
    uint32_t x = lift::lift_word<M, true>(u, w);
#pragma unroll
    for (int blk = 1; blk < LG; ++blk) x = hadd2_bf16(x, lift::lift_word<M, true>(u + blk * (M / 2), w));
    return x;
}

template <int P, int LG, int TAU>
__device__ __forceinline__ void query_tile(const uint32_t (&u)[P / 2], uint32_t taddr) {
    uint32_t w[64];  // the tile's 64 words, stored by one tensor-memory instruction
#pragma unroll
    for (int i = 0; i < 64; ++i) w[i] = query_word<P, LG>(u, 64 * TAU + i);
    tmem_st64(taddr, w);
}

template <int P, int LG, int TAU = 0>
__device__ __forceinline__ void query_dispatch(int tau, const uint32_t (&uq)[P / 2], uint32_t taddr) {
    if constexpr (TAU < lift::tiles_of(P / LG)) {
        if (tau == TAU)
            query_tile<P, LG, TAU>(uq, taddr);
        else
            query_dispatch<P, LG, TAU + 1>(tau, uq, taddr);
    }
}

// Query lift of the last (partly filled) tile: its first 16 words (32 slots).
template <int P, int LG>
__device__ __forceinline__ void query_tail(const uint32_t (&uq)[P / 2], uint32_t taddr) {
    constexpr int TAU = lift::tiles_of(P / LG) - 1;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = query_word<P, LG>(uq, 64 * TAU + i);
    tmem_st16(taddr, w);
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


// ---------------------------------------------------------------- state kernel
// CTA kinds, by tile index tau: tau < NT a full 128-slot tile of the lift;
// tau = NT the last, partly filled tile (TAIL slots); tau = NT + 1 the
// normaliser CTA, which keeps Z and adds the inter-chunk denominators
// q^T Z q to d (no state tile).
// Warp roles (512 threads, four warpgroups); thread e of a warpgroup is
// tensor-memory lane e:
//   warps 0-3   query:    lane = token; lifts its staged query row for this
//                         CTA's slots into tensor memory (A operand of the
//                         readout); one chunk behind, reads the token's
//                         partial readout, stages it in shared memory and
//                         (one thread) adds the chunk's rows to Y by TMA
//   warps 4-7   state:    lane = slot; after each update reads the state row
//                         and releases it to the next update, then refreshes
//                         the bf16 copy the next readout reads (normaliser
//                         CTA: the same for Z, and the denominators)
//   warps 8-11  key lift: lane = slot; multiplies two rows of the chunk's
//                         transposed unit keys into the update's A operand
//   warp 12     MMA:      per chunk the update (state += lift(K)^T V)
//                         (normaliser CTA: Z += Kh^T Kh and W = Q Z); the
//                         whole warp runs the loop, one elected lane issues
//   warp 13     loads:    lane 0 issues the TMA loads (transposed keys, values,
//                         queries)
//   warp 14     MMA:      per chunk the readout (Y = lift(Q) S) of the state
//                         before the chunk (tile CTAs)
template <int P, int DV, int LG>
__global__ void __launch_bounds__(kThreads, 1)
chunked_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmkt,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmy,
                  const __grid_constant__ CUtensorMap tmktr, float* __restrict__ dacc,
                  const float* __restrict__ S_start, const float* __restrict__ z_start,
                  int start_groups, int start_stride, float* __restrict__ S_final, float* __restrict__ z_final, int T,
                  int seg_chunks) {
    using K = Cfg<P, DV, LG>;
    constexpr int n = K::n, M = K::M;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t qs_full[2], qs_free[2], kts_full[2], kts_free[2], v_full[2], v_free[2];
    __shared__ uint64_t qlift_full[2], aq_free[2], y_part[2], y_free[2], ys_full[2], ys_free[2];
    __shared__ uint64_t klift_full[2], ak_free[2], upd_done, state_read, s16_ready, drain, drain2;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int t = threadIdx.x, warp = t >> 5;
    // grid: x = head, y = (segment, tile): neighbouring CTAs (which share an
    // SM pair and its instruction fetch) run the same tile of different heads
    const int tau = blockIdx.y % K::CS;  // tile of the packed lift (NT + 1: the normaliser CTA)
    const int g = blockIdx.y / K::CS;    // segment
    const int G = gridDim.y / K::CS;
    const bool tail = tau == K::NT;      // the last, partly filled tile
    const bool zc = tau == K::NT + 1;    // Z and the denominators
    const int64_t bh = blockIdx.x;
    const int NCH = (T + kChunk - 1) / kChunk;
    const int64_t head_prow = bh * (int64_t)NCH * kChunk;  // accumulation rows: whole chunks per head
    const int c0 = g * seg_chunks, c1 = min(NCH, c0 + seg_chunks);
    const int nk = c1 - c0;
    uint8_t* const s_s16 = sm + K::o_s16;
    uint8_t* const s_z16 = sm + K::o_z16;
    auto v_buf = [&](int kk) { return sm + K::o_v + (kk & 1) * kAtom; };
    auto q_buf = [&](int kk) { return sm + K::o_q + (kk & 1) * kAtom; };
    // transposed-key stage of chunk kk: padded rows (tile CTAs) or swizzled boxes (normaliser)
    auto kt_buf = [&](int kk) { return sm + K::o_kt + (kk & 1) * (zc ? kAtom : K::kt_rows_bytes); };
    auto y_buf = [&](int kk) { return sm + K::o_y + (kk & 1) * K::y_stage; };

    if (t == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&qs_full[b], 1);
            // the staged queries are read by the query warps (tiles) or by the
            // state warps after the Q Z product that reads them too (normaliser)
            mbar_init(&qs_free[b], 128);
            mbar_init(&kts_full[b], 1);
            // the staged keys are read by the key-lift warps (tiles) or by the
            // Z update (normaliser, one commit)
            mbar_init(&kts_free[b], zc ? 1 : 128);
            mbar_init(&v_full[b], 1);
            mbar_init(&v_free[b], 1);
            mbar_init(&qlift_full[b], 128);
            mbar_init(&aq_free[b], 1);
            mbar_init(&y_part[b], 1);
            mbar_init(&y_free[b], 128);
            mbar_init(&ys_full[b], 128);
            mbar_init(&ys_free[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&klift_full[b], 128);
            mbar_init(&ak_free[b], 1);
        }
        mbar_init(&upd_done, 1);
        mbar_init(&state_read, 128);
        mbar_init(&s16_ready, 128);
        mbar_init(&drain, 1);
        mbar_init(&drain2, 1);
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
    const uint32_t lane0 = (uint32_t)((warp & 3) * 32);
    auto tm = [&](uint32_t col) { return tmem_addr(tb, lane0, col); };
    auto fail = [&]() {
        abort_flag = 1;
        atomicOr(&g_chunked_tc_status, kStatusTimeout);
    };
    // Bounded waits whose outcome is the same for every lane of the warp (the
    // warp-collective tensor-memory instructions that follow need that).
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, &abort_flag, kWaitNs));
    };

    // ---- start state of this segment (state warps: lane = slot / dimension)
    if (warp >= 4 && warp < 8) {
        const int e = t - 128;
        const int sg = start_groups > 1 ? g * start_stride : 0;  // this segment's start state
        if (!zc) {
            const float* S0 = S_start ? S_start + (bh * start_groups + sg) * (int64_t)n * DV : nullptr;
            load_state_tile<M, DV>(S0, tau, tm(K::tm_s), s_s16, e);
        } else {
            const float* z0 = z_start ? z_start + (bh * start_groups + sg) * (int64_t)n : nullptr;
            float zr[M];
#pragma unroll
            for (int j = 0; j < M; ++j) {
                float val = 0.f;
                if (z0 != nullptr && e < M) {
                    const int a = e < j ? e : j, b = e < j ? j : e;
                    val = z0[lift::canonical_index(M, a, b)] * (a == b ? 1.f : kInvSqrt2f);
                }
                zr[j] = val;
            }
#pragma unroll
            for (int c = 0; c < M; c += 16) {
                uint32_t r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(zr[c + i]);
                tmem_st16(tm(K::tm_z + c), r);
            }
            if (e < M) {
#pragma unroll
                for (int c = 0; c < M / 8; ++c)
                    *reinterpret_cast<uint4*>(s_z16 + sw128_chunk(e, 8 * c, M)) =
                        make_uint4(pack_bf16x2(zr[8 * c], zr[8 * c + 1]), pack_bf16x2(zr[8 * c + 2], zr[8 * c + 3]),
                                   pack_bf16x2(zr[8 * c + 4], zr[8 * c + 5]), pack_bf16x2(zr[8 * c + 6], zr[8 * c + 7]));
            }
        }
        tmem_wait_st();
    }
    // the last tile's key lift fills lanes [0, 32) of its operand; the other
    // lanes are read by its M = 128 update into state rows nothing reads, and
    // are kept at zero
    if (tail && warp >= 9 && warp < 12) {
        uint32_t zw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) zw[i] = 0u;
#pragma unroll
        for (int c = 0; c < 64 * K::AKB; c += 16) tmem_st16(tm(K::tm_ak + c), zw);
        tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();  // barriers initialised and start state in place
    tc_fence_after();

    if (warp < 4) {
        // =============================================================== query warps
        regs_inc<kRegsLift>();
        const int e = t;
        // query lift of chunk kk into its tensor-memory slot (double-buffered:
        // overlaps the previous chunk's readout)
        auto lift_q = [&](int kk) -> bool {
            const int slot = kk & 1, use = kk >> 1;
            if (!wait(&qs_full[slot], use & 1)) return false;
            const uint8_t* my_q = q_buf(kk) + t * 128;
            uint32_t uq[P / 2];
#pragma unroll
            for (int i = 0; i < P / 8; ++i) {
                const uint4 a = *reinterpret_cast<const uint4*>(my_q + ((i ^ (t & 7)) << 4));
                uq[4 * i] = a.x;
                uq[4 * i + 1] = a.y;
                uq[4 * i + 2] = a.z;
                uq[4 * i + 3] = a.w;
            }
            mbar_arrive(&qs_free[slot]);
            if (kk >= 2 && !wait(&aq_free[slot], (use - 1) & 1)) return false;
            tc_fence_after();
            if (!tail)
                query_dispatch<P, LG>(tau, uq, tm(K::tm_aq + 64 * slot));
            else
                query_tail<P, LG>(uq, tm(K::tm_aq + 64 * slot));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&qlift_full[slot]);
            return true;
        };
        // this lane's partial readout of chunk c0 + kc -> the stage; thread 0
        // adds the stage to the chunk's accumulation rows
        auto out = [&](int kc) -> bool {
            const int slot = kc & 1, use = kc >> 1;
            if (!wait(&y_part[slot], use & 1)) return false;
            tc_fence_after();
            uint32_t y[DV];
#pragma unroll
            for (int c = 0; c < DV; c += 16) tmem_ld16(tm(K::tm_y + 64 * slot + c), *reinterpret_cast<uint32_t(*)[16]>(y + c));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&y_free[slot]);
            // the stage's previous contents (chunk kc - 2) have been read by the TMA
            if (kc >= 2 && !wait(&ys_free[slot], (use - 1) & 1)) return false;
            uint8_t* stg = y_buf(kc);
#pragma unroll
            for (int hh = 0; hh < K::YH; ++hh) {
#pragma unroll
                for (int c = 0; c < K::YW / 4; ++c) {
                    const uint32_t off = K::YW == 32 ? (uint32_t)e * 128u + ((uint32_t)(c ^ (e & 7)) << 4)
                                                     : (uint32_t)e * (K::YW * 4) + (uint32_t)c * 16u;
                    *reinterpret_cast<uint4*>(stg + hh * K::y_box + off) =
                        make_uint4(y[hh * K::YW + 4 * c], y[hh * K::YW + 4 * c + 1], y[hh * K::YW + 4 * c + 2],
                                   y[hh * K::YW + 4 * c + 3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&ys_full[slot]);
            if (t == 0) {
                if (!mbar_wait(&ys_full[slot], use & 1, &abort_flag, kWaitNs)) return false;
                const int row0 = (c0 + kc) * kChunk;
#pragma unroll
                for (int hh = 0; hh < K::YH; ++hh)
                    tma_reduce_add_3d(&tmy, hh * K::YW, row0, (int)bh, stg + hh * K::y_box);
                bulk_commit();
                // the previous chunk's stage has been read: it may be rewritten
                bulk_wait_read<1>();
                if (kc >= 1) mbar_arrive(&ys_free[(kc - 1) & 1]);
            }
            return true;
        };
        if (!zc) {
            for (int kk = 0; kk <= nk; ++kk) {
                if (kk < nk && !lift_q(kk)) { fail(); break; }
                if (kk >= 1 && !out(kk - 1)) { fail(); break; }
            }
            // no reduce-add may still be reading shared memory when the CTA exits
            if (t == 0) bulk_wait<0>();
        }
    } else if (warp < 8) {
        // =============================================================== state warps
        regs_inc<kRegsState>();
        const int e = t - 128;
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            // state (Z) after this chunk's update
            if (!wait(&upd_done, kk & 1)) { fail(); break; }
            tc_fence_after();
            uint32_t sreg[(M > DV ? M : DV) / 2];  // bf16 pairs of this lane's state (Z) row
            if (!zc) {
#pragma unroll
                for (int c32 = 0; c32 < DV; c32 += 32) {
                    uint32_t r[2][16];  // two loads in flight per wait
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (c32 + 16 * h < DV) tmem_ld16(tm(K::tm_s + c32 + 16 * h), r[h]);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (c32 + 16 * h < DV)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                sreg[(c32 + 16 * h) / 2 + i] = pack_bf16x2(__uint_as_float(r[h][2 * i]), __uint_as_float(r[h][2 * i + 1]));
                }
            } else {
#pragma unroll
                for (int c16 = 0; c16 < M; c16 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tm_z + c16), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        sreg[c16 / 2 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                }
            }
            tc_fence_before();
            mbar_arrive(&state_read);
            // this chunk's readout (W) is done: its bf16 state (Z) copy may be replaced
            if (!wait(&y_part[slot], use & 1)) { fail(); break; }
            tc_fence_after();
            if (!zc) {
#pragma unroll
                for (int c8 = 0; c8 < DV / 8; ++c8)
                    *reinterpret_cast<uint4*>(s_s16 + mn_sw128_chunk(8 * c8, e, kAtom)) =
                        make_uint4(sreg[4 * c8], sreg[4 * c8 + 1], sreg[4 * c8 + 2], sreg[4 * c8 + 3]);
            } else {
                // inter-chunk denominator q^T Z q from W = Q Z (Z before this chunk)
                uint4 qrow[P / 8];
                const uint8_t* sq = q_buf(kk);  // this chunk's staged queries
#pragma unroll
                for (int i = 0; i < P / 8; ++i) qrow[i] = *reinterpret_cast<const uint4*>(sq + sw128_chunk(e, 8 * i, kChunk));
                const __nv_bfloat16* qe = reinterpret_cast<const __nv_bfloat16*>(qrow);
                float dint = 0.f;
#pragma unroll
                for (int c16 = 0; c16 < P; c16 += 16) {
                    uint32_t w[16];
                    tmem_ld16(tm(K::tm_w + c16), w);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) dint = fmaf(__bfloat162float(qe[c16 + i]), __uint_as_float(w[i]), dint);
                }
                tc_fence_before();
                mbar_arrive(&qs_free[slot]);  // this chunk's staged queries and W have been read
                atomicAdd(dacc + head_prow + (int64_t)(c0 + kk) * kChunk + e, dint);
                if (e < M) {
#pragma unroll
                    for (int c8 = 0; c8 < M / 8; ++c8)
                        *reinterpret_cast<uint4*>(s_z16 + sw128_chunk(e, 8 * c8, M)) =
                            make_uint4(sreg[4 * c8], sreg[4 * c8 + 1], sreg[4 * c8 + 2], sreg[4 * c8 + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s16_ready);
        }
        // final state of the last segment
        if (S_final != nullptr && g == G - 1 && !abort_flag) {
            const int64_t head_s = bh * (int64_t)n * DV, head_z = bh * (int64_t)n;
            if (!zc) {
                store_state_tile<M, DV>(S_final + head_s, tau, tm(K::tm_s), e);
            } else {
                uint32_t zr[M];
#pragma unroll
                for (int c16 = 0; c16 < M; c16 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tm_z + c16), r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) zr[c16 + i] = r[i];
                }
                tmem_wait_ld();
                if (e < M) {
#pragma unroll
                    for (int j = 0; j < M; ++j)
                        if (j >= e)
                            z_final[head_z + lift::canonical_index(M, e, j)] = __uint_as_float(zr[j]) * (j == e ? 1.f : kSqrt2f);
                }
            }
        }
    } else if (warp < 12) {
        // =============================================================== key-lift warps
        const int e = t - 256;
        if (!zc) {
            for (int kk = 0; kk < nk; ++kk) {
                const int stg = kk & 1, use = kk >> 1;
                if (!wait(&kts_full[stg], use & 1)) { fail(); break; }
                // the key-lift buffer's previous chunk (kk - AKB) has been read by its update
                const int ab = kk % K::AKB, ause = kk / K::AKB;
                if (kk >= K::AKB && !wait(&ak_free[ab], (ause - 1) & 1)) { fail(); break; }
                tc_fence_after();
                if (!tail || warp == 8) key_row_tmem<P, LG>(kt_buf(kk), tau * 128 + e, tm(K::tm_ak + 64 * ab));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&klift_full[ab]);
                mbar_arrive(&kts_free[stg]);
            }
        }
    } else {
        regs_dec<kRegsMma>();
    }
    if (t == 416) {
        // =============================================================== TMA producer
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmkt);
        tma_prefetch_desc(&tmktr);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmy);
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            const int row = (c0 + kk) * kChunk;
            // transposed unit keys of chunk kk into its stage
            if (kk >= 2 && !mbar_wait(&kts_free[slot], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            if (!zc) {
                mbar_arrive_expect_tx(&kts_full[slot], K::kt_rows_bytes);
                tma_load_3d(kt_buf(kk), &tmktr, 0, (c0 + kk) * P, (int)bh, &kts_full[slot]);
            } else {
                mbar_arrive_expect_tx(&kts_full[slot], K::kt_bytes);
                tma_load_3d(kt_buf(kk), &tmkt, 0, (c0 + kk) * P, (int)bh, &kts_full[slot]);
                tma_load_3d(kt_buf(kk) + K::kt_box, &tmkt, 64, (c0 + kk) * P, (int)bh, &kts_full[slot]);
            }
            // value tile of chunk kk into its buffer (state tiles only)
            if (!zc) {
                if (kk >= 2 && !mbar_wait(&v_free[slot], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
                mbar_arrive_expect_tx(&v_full[slot], kAtom);
                tma_load_3d(v_buf(kk), &tmv, 0, row, (int)bh, &v_full[slot]);
            }
            // query rows of chunk kk into its stage
            if (kk >= 2 && !mbar_wait(&qs_free[slot], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&qs_full[slot], kAtom);
            tma_load_3d(q_buf(kk), &tmq, 0, row, (int)bh, &qs_full[slot]);
        }
    }
    if (warp == 12 || (warp == 14 && !zc)) {
        // =============================================================== MMA issuers
        // Tile CTAs: warp 12 issues the updates, warp 14 the readouts (the two
        // chains share no operand, and neither issuer's waits hold up the
        // other's MMAs); the normaliser CTA: warp 12 issues both of its products.
        // The whole warp runs the issue loop (waits, descriptors) and one
        // elected lane issues each instruction: the operands stay warp-uniform,
        // which keeps the issue of back-to-back MMAs as cheap as a loop of
        // constants (a single lane in a divergent branch issues them at about
        // two thirds of that rate).  Every descriptor is built once; the loop
        // adds compile-time offsets (a step moves the start-address field, in
        // 16-byte units).
        constexpr uint32_t id_mn = idesc_bf16_f32_major(128, DV, false, true);
        constexpr uint32_t id_z = idesc_bf16_f32(128, M);
        constexpr uint32_t id_w = idesc_bf16_f32(128, M);
        constexpr uint64_t kStepMN = 2048 >> 4, kStepK = 32 >> 4, kBoxD = K::kt_box >> 4;
        // K step ks of a K-major operand whose 64-element K atoms are `atom` (16-byte units) apart
        auto kstep = [](uint64_t atom, int ks) { return (uint64_t)(ks >> 2) * atom + (uint64_t)(ks & 3) * kStepK; };
        const uint64_t d_s16 = sdesc_mnmajor_sw128(smem_u32(s_s16), kAtom);
        const uint64_t d_v[2] = {sdesc_mnmajor_sw128(smem_u32(v_buf(0)), kAtom),
                                 sdesc_mnmajor_sw128(smem_u32(v_buf(1)), kAtom)};
        // normaliser CTA: staged transposed keys (both operands of the Z update), staged Q, Z
        const uint64_t d_kt[2] = {sdesc_kmajor_sw128(smem_u32(kt_buf(0))), sdesc_kmajor_sw128(smem_u32(kt_buf(1)))};
        const uint64_t d_q[2] = {sdesc_kmajor_sw128(smem_u32(q_buf(0))), sdesc_kmajor_sw128(smem_u32(q_buf(1)))};
        const uint64_t d_z16 = sdesc_kmajor_sw128(smem_u32(s_z16));
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            if (!zc) {
                if (warp == 12) {
                    const int ab = kk % K::AKB, ause = kk / K::AKB;
                    if (!wait(&v_full[slot], use & 1) || !wait(&klift_full[ab], ause & 1) ||
                        (kk >= 1 && !wait(&state_read, (kk - 1) & 1))) {
                        fail();
                        break;
                    }
                    tc_fence_after();
                    // ---- update: state += lift(K)^T V
                    const uint64_t dv = d_v[slot];
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts_w(tb + K::tm_s, tb + K::tm_ak + 64 * ab + 8 * ks, dv + ks * kStepMN, id_mn, 1u);
                    mma_commit_w(&ak_free[ab]);
                    mma_commit_w(&upd_done);
                    mma_commit_w(&v_free[slot]);
                } else {
                    // ---- readout of the state before this chunk
                    if (!wait(&qlift_full[slot], use & 1) || (kk >= 1 && !wait(&s16_ready, (kk - 1) & 1)) ||
                        (kk >= 2 && !wait(&y_free[slot], (use - 1) & 1))) {
                        fail();
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dy = tb + K::tm_y + 64 * slot, aq = tb + K::tm_aq + 64 * slot;
                    if (!tail) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_ts_w(dy, aq + 8 * ks, d_s16 + ks * kStepMN, id_mn, ks > 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < (K::TAIL + 15) / 16; ++ks)
                            mma_ts_w(dy, aq + 8 * ks, d_s16 + ks * kStepMN, id_mn, ks > 0 ? 1u : 0u);
                    }
                    mma_commit_w(&y_part[slot]);
                    mma_commit_w(&aq_free[slot]);
                }
            } else {
                if (!wait(&kts_full[slot], use & 1) || (kk >= 1 && !wait(&state_read, (kk - 1) & 1))) {
                    fail();
                    break;
                }
                tc_fence_after();
                // ---- Z += sum over the blocks of Kh_b^T Kh_b
#pragma unroll
                for (int blk = 0; blk < LG; ++blk)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss_w(tb + K::tm_z, d_kt[slot] + (uint64_t)(blk * M * 8) + kstep(kBoxD, ks),
                                 d_kt[slot] + (uint64_t)(blk * M * 8) + kstep(kBoxD, ks), id_z, 1u);
                mma_commit_w(&kts_free[slot]);
                mma_commit_w(&upd_done);
                // ---- W = [Q_0 Z | Q_1 Z | ...] with Z before this chunk, one block of columns per block of the queries
                if (!wait(&qs_full[slot], use & 1) || (kk >= 1 && !wait(&s16_ready, (kk - 1) & 1))) {
                    fail();
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int blk = 0; blk < LG; ++blk)
#pragma unroll
                    for (int ks = 0; ks < M / 16; ++ks)
                        mma_ss_w(tb + K::tm_w + blk * M, d_q[slot] + (blk * (M / 16) + ks) * kStepK, d_z16 + ks * kStepK,
                                 id_w, ks > 0 ? 1u : 0u);
                mma_commit_w(&y_part[slot]);
            }
        }
        // every issued MMA has completed before tensor memory is released
        mma_commit_w(warp == 12 ? &drain : &drain2);
        mbar_wait_quiet(warp == 12 ? &drain : &drain2, 0, kWaitNs);
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------- output
// o = Y / d for the rows t < T (0 where d = 0); one thread per 8 columns.
template <int DV>
__global__ void __launch_bounds__(256)
normalize_kernel(const float* __restrict__ yacc, const float* __restrict__ dacc, __nv_bfloat16* __restrict__ o, int T,
                 int Tc, int64_t BH) {
    constexpr int per = DV / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BH * T * per) return;
    const int64_t row = i / per;
    const int c = (int)(i % per);
    const int64_t bh = row / T, tt = row % T;
    const int64_t arow = bh * Tc + tt;
    const float4 a = *reinterpret_cast<const float4*>(yacc + arow * DV + 8 * c);
    const float4 b = *reinterpret_cast<const float4*>(yacc + arow * DV + 8 * c + 4);
    const float d = dacc[arow];
    const float inv = d > 0.f ? 1.f / d : 0.f;
    *reinterpret_cast<uint4*>(o + row * DV + 8 * c) =
        make_uint4(pack_bf16x2(a.x * inv, a.y * inv), pack_bf16x2(a.z * inv, a.w * inv), pack_bf16x2(b.x * inv, b.y * inv),
                   pack_bf16x2(b.z * inv, b.w * inv));
}


// ---------------------------------------------------------------- intra-chunk part
// Every chunk on its own (no state): for the 128 queries of a chunk,
//   P = (Q Kh^T) o (Q Kh^T) o M   (bf16, M the causal mask s <= t)
//   Y = P V,  d = rowsum(P)       (fp32 accumulation)
// Y and d, the rows' intra-chunk normaliser, initialise the forward's fp32
// accumulation rows [BH][Tc][DV] and [BH][Tc] (Tc = T rounded up to whole
// chunks; rows past T are not written): the state kernel adds the
// inter-chunk parts to them.  The chunk's unit keys also go out transposed, kT
// [BH][chunks][P][kKtCols] bf16 (128 tokens, zeros past T, and a pad): the
// state kernel's key lift reads them.  d sums exactly the rounded weights Y
// is built from, which keeps the intra-chunk weights a convex combination.
// One CTA per (chunk, head), 128 columns of tensor memory and about 66 KB of
// shared memory, so several chunks are in flight per SM; thread t owns query
// / key / value row t.
template <int P, int DV, int LG>
__global__ void __launch_bounds__(128)
intra_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, __nv_bfloat16* __restrict__ kt_out,
                const __grid_constant__ CUtensorMap tmy, float* __restrict__ d_out, int T) {
    constexpr int YW = DV < 32 ? DV : 32, YH = DV / YW;  // fp32 output boxes of 128 rows x YW columns
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar, drain, ld_full;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* Qs = sm;              // K-major, 128 rows x 128 B (TMA, zeros past T and past P)
    uint8_t* Ks = sm + kAtom;      // keys, normalised in place: unit keys, K-major
    uint8_t* Vs = sm + 2 * kAtom;  // V, MN-major (TMA)
    uint8_t* KTs = sm + 3 * kAtom; // transposed unit keys: P rows of kKtRow bytes
    uint8_t* Ys = sm;              // fp32 rows for the output boxes (over Q and K once the scores are read)
    const int t = threadIdx.x, warp = t >> 5;
    const int64_t bh = blockIdx.y;
    const int row = blockIdx.x * kChunk + t;
    const bool valid = row < T;
    // y and d rows: T rounded up to whole chunks per head
    const int64_t prow = bh * (int64_t)(gridDim.x * kChunk) + row;
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_init(&drain, 1);
        mbar_init(&ld_full, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    __syncthreads();
    // q, k, v rows of the chunk by TMA (rows past T read as zeros)
    if (t == 0) {
        mbar_arrive_expect_tx(&ld_full, 3 * kAtom);
        tma_load_3d(Qs, &tmq, 0, blockIdx.x * kChunk, (int)bh, &ld_full);
        tma_load_3d(Ks, &tmk, 0, blockIdx.x * kChunk, (int)bh, &ld_full);
        tma_load_3d(Vs, &tmv, 0, blockIdx.x * kChunk, (int)bh, &ld_full);
    }
    const bool loaded = __all_sync(0xffffffffu, mbar_wait(&ld_full, 0, &abort_flag, kWaitNs));
    // thread t normalises key row t in place and writes it transposed into the staging boxes
    if (loaded) {
        uint4 kr[P / 8];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < P / 8; ++i) {
            kr[i] = *reinterpret_cast<const uint4*>(Ks + sw128_chunk(t, 8 * i, kChunk));
            const __nv_bfloat16* ke = reinterpret_cast<const __nv_bfloat16*>(&kr[i]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = __bfloat162float(ke[j]);
                ss = fmaf(x, x, ss);
            }
        }
        const float kinv = ss > 0.f ? rsqrtf(ss) : 0.f;
        // the pad of row t (never read; written so that the copy out is defined)
        if (t < P) *reinterpret_cast<uint4*>(KTs + t * kKtRow + 2 * kChunk) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < P / 8; ++i) {
            const __nv_bfloat16* ke = reinterpret_cast<const __nv_bfloat16*>(&kr[i]);
            uint4 w;
            w.x = pack_bf16x2(__bfloat162float(ke[0]) * kinv, __bfloat162float(ke[1]) * kinv);
            w.y = pack_bf16x2(__bfloat162float(ke[2]) * kinv, __bfloat162float(ke[3]) * kinv);
            w.z = pack_bf16x2(__bfloat162float(ke[4]) * kinv, __bfloat162float(ke[5]) * kinv);
            w.w = pack_bf16x2(__bfloat162float(ke[6]) * kinv, __bfloat162float(ke[7]) * kinv);
            *reinterpret_cast<uint4*>(Ks + sw128_chunk(t, 8 * i, kChunk)) = w;
            // dimensions 8i .. 8i+7 of this token: rows of the transposed keys, column t
            const uint16_t* we = reinterpret_cast<const uint16_t*>(&w);
#pragma unroll
            for (int j = 0; j < 8; ++j) *reinterpret_cast<uint16_t*>(KTs + (8 * i + j) * kKtRow + t * 2) = we[j];
        }
    }
    fence_proxy_async_smem();
    __syncthreads();
    // the transposed unit keys of the chunk out in one bulk copy (read before the CTA exits)
    if (t == 0 && loaded) {
        bulk_store(kt_out + ((int64_t)bh * gridDim.x + blockIdx.x) * (P * kKtCols), KTs, P * kKtRow);
        bulk_commit();
    }
    if (!loaded && t == 0) {
        abort_flag = 1;
        atomicOr(&g_chunked_tc_status, kStatusTimeout);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t lane0 = (uint32_t)(warp * 32);
    // P = scores^2 masked, bf16, in place (columns 0..63), and its row sum;
    // quarters past this warp's rows are all masked.  Full lift: the scores
    // are (q . kh)^2.  KATA-Sigma-g: sum over the block pairs (a, b) of
    // (q_a . kh_b)^2, one product per pair into columns 0..127, whose squares
    // are summed in registers.
    float den = 0.f;
    bool ok = true;
    const uint64_t dq = sdesc_kmajor_sw128(smem_u32(Qs)), dk = sdesc_kmajor_sw128(smem_u32(Ks));
    constexpr uint32_t id_sc = idesc_bf16_f32(128, 128);
    if constexpr (LG == 1) {
        // scores (q . kh); P = scores^2
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < P / 16; ++ks) mma_ss(tb, dq + 2 * ks, dk + 2 * ks, id_sc, ks > 0 ? 1u : 0u);
            mma_commit(&bar);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&bar, 0, &abort_flag, kWaitNs));
        if (!ok) abort_flag = 1;
        tc_fence_after();
        if (ok) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t pk[16];
                if (q4 <= warp) {
                    uint32_t sc[32];
                    tmem_ld16(tmem_addr(tb, lane0, 32 * q4), *reinterpret_cast<uint32_t(*)[16]>(sc));
                    tmem_ld16(tmem_addr(tb, lane0, 32 * q4 + 16), *reinterpret_cast<uint32_t(*)[16]>(sc + 16));
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int col = 32 * q4 + 2 * i;
                        float a = __uint_as_float(sc[2 * i]), b = __uint_as_float(sc[2 * i + 1]);
                        a = col <= t ? a * a : 0.f;
                        b = col + 1 <= t ? b * b : 0.f;
                        pk[i] = pack_bf16x2(a, b);
                        const __nv_bfloat162 hp = *reinterpret_cast<const __nv_bfloat162*>(&pk[i]);
                        den += __low2float(hp) + __high2float(hp);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[i] = 0u;
                }
                tmem_st16(tmem_addr(tb, lane0, 16 * q4), pk);
            }
            tmem_wait_st();
        }
    } else {
        constexpr int M = P / LG;
        float acc[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) acc[c] = 0.f;
        // every thread runs every iteration (the block barrier below is reached
        // by all of them even after a wait gave up)
        for (int pr = 0; pr < LG * LG; ++pr) {
            const int a = pr / LG, b = pr % LG;
            if (t == 0 && ok) {
#pragma unroll
                for (int ks = 0; ks < M / 16; ++ks)
                    mma_ss(tb, dq + 2 * (a * (M / 16) + ks), dk + 2 * (b * (M / 16) + ks), id_sc, ks > 0 ? 1u : 0u);
                mma_commit(&bar);
            }
            ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar, pr & 1, &abort_flag, kWaitNs));
            if (!ok) abort_flag = 1;
            tc_fence_after();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                if (ok && q4 <= warp) {
                    uint32_t sc[32];
                    tmem_ld16(tmem_addr(tb, lane0, 32 * q4), *reinterpret_cast<uint32_t(*)[16]>(sc));
                    tmem_ld16(tmem_addr(tb, lane0, 32 * q4 + 16), *reinterpret_cast<uint32_t(*)[16]>(sc + 16));
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float x = __uint_as_float(sc[i]);
                        acc[32 * q4 + i] = fmaf(x, x, acc[32 * q4 + i]);
                    }
                }
            }
            // every lane has read this pair's scores before the next pair overwrites them
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
        if (ok) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int col = 32 * q4 + 2 * i;
                    const float x0 = (q4 <= warp && col <= t) ? acc[col] : 0.f;
                    const float x1 = (q4 <= warp && col + 1 <= t) ? acc[col + 1] : 0.f;
                    pk[i] = pack_bf16x2(x0, x1);
                    const __nv_bfloat162 hp = *reinterpret_cast<const __nv_bfloat162*>(&pk[i]);
                    den += __low2float(hp) + __high2float(hp);
                }
                tmem_st16(tmem_addr(tb, lane0, 16 * q4), pk);
            }
            tmem_wait_st();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Y into columns 64.. (the scores there have been read)
    if (t == 0 && !abort_flag) {
        const uint64_t dv = sdesc_mnmajor_sw128(smem_u32(Vs), kAtom);
        constexpr uint32_t id_pv = idesc_bf16_f32_major(128, DV, false, true);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_ts(tb + 64, tb + 8 * ks, dv + ks * (2048 >> 4), id_pv, ks > 0 ? 1u : 0u);
        mma_commit(&bar);
    }
    ok = !abort_flag && __all_sync(0xffffffffu, mbar_wait(&bar, (LG * LG) & 1, &abort_flag, kWaitNs));
    tc_fence_after();
    if (ok) {
        // row t of Y into the output boxes (over the query and key tiles, whose
        // products are done), the normaliser straight out
        uint32_t y[DV];
#pragma unroll
        for (int c = 0; c < DV; c += 16) tmem_ld16(tmem_addr(tb, lane0, 64 + c), *reinterpret_cast<uint32_t(*)[16]>(y + c));
        tmem_wait_ld();
#pragma unroll
        for (int hh = 0; hh < YH; ++hh)
#pragma unroll
            for (int c = 0; c < YW / 4; ++c) {
                const uint32_t off = YW == 32 ? (uint32_t)t * 128u + ((uint32_t)(c ^ (t & 7)) << 4)
                                              : (uint32_t)t * (YW * 4) + (uint32_t)c * 16u;
                *reinterpret_cast<uint4*>(Ys + hh * (128 * YW * 4) + off) =
                    make_uint4(y[hh * YW + 4 * c], y[hh * YW + 4 * c + 1], y[hh * YW + 4 * c + 2], y[hh * YW + 4 * c + 3]);
            }
        if (valid) d_out[prow] = den;
    } else if (t == 0) {
        atomicOr(&g_chunked_tc_status, kStatusTimeout);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0) {
        if (ok) {
#pragma unroll
            for (int hh = 0; hh < YH; ++hh)
                tma_store_3d(&tmy, hh * YW, blockIdx.x * kChunk, (int)bh, Ys + hh * (128 * YW * 4));
            bulk_commit();
        }
        // no store may still be reading shared memory when the CTA exits
        bulk_wait_read<0>();
        // every issued MMA has completed before the tensor memory is released
        mma_commit(&drain);
        mbar_wait_quiet(&drain, 0, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 128);
}

// o = (numerator + intra rows) / (denominator + intra normaliser), in place

// ---------------------------------------------------------------- host side
// The register split of the kernel fits in its launch allocation.
template <int P, int DV, int LG>
bool register_split_fits() {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, chunked_tc_kernel<P, DV, LG>) != cudaSuccess) return false;
    return (uint32_t)kThreads * (uint32_t)fa.numRegs >= 128u * (kRegsLift + kRegsState + kRegsLaunch + kRegsMma);
}

// CTAs of the state kernel resident at once on the current device (one per
// SM when it fits), 0 if the kernel cannot run there.
template <int P, int DV, int LG>
int resident_ctas() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        using K = Cfg<P, DV, LG>;
        int per_sm = 0, sms = 0;
        if (!register_split_fits<P, DV, LG>() ||
            cudaFuncSetAttribute(chunked_tc_kernel<P, DV, LG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K::smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunked_tc_kernel<P, DV, LG>, kThreads, K::smem) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cached[dev] = per_sm * sms > 0 ? per_sm * sms : -1;
    }
    return cached[dev] > 0 ? cached[dev] : 0;
}

// Workspace of the forward: fp32 accumulation rows Y [BH][Tc][dv] and d
// [BH][Tc] (Tc = T rounded up to whole chunks), transposed unit keys
// [BH][chunks][p][128] bf16.
struct IntraWs {
    size_t y_off, d_off, kt_off, total;
};
IntraWs intra_ws(int BH, int T, int p, int dv) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t nch = (size_t)(T + kChunk - 1) / kChunk;
    IntraWs w;
    w.y_off = 0;
    w.d_off = up((size_t)BH * nch * kChunk * dv * 4);
    w.kt_off = w.d_off + up((size_t)BH * nch * kChunk * 4);
    w.total = w.kt_off + up((size_t)BH * nch * p * kKtCols * 2);
    return w;
}

template <int P, int DV, int LG>
cudaError_t launch_typed(const void* q, const void* k, const void* v, void* o, void* intra,
                         const float* S_start, const float* z_start, int start_groups, int start_stride,
                         float* S_final, float* z_final, int BH, int T, int seg_chunks, int G, cudaStream_t s) {
    using K = Cfg<P, DV, LG>;
    if (!register_split_fits<P, DV, LG>()) return cudaErrorInvalidConfiguration;
    const IntraWs w = intra_ws(BH, T, P, DV);
    auto* yacc = reinterpret_cast<float*>(static_cast<char*>(intra) + w.y_off);
    auto* dacc = reinterpret_cast<float*>(static_cast<char*>(intra) + w.d_off);
    auto* kt = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(intra) + w.kt_off);
    const int nch = (T + kChunk - 1) / kChunk;
    // the intra-chunk part (initialises the accumulation rows) and the
    // transposed unit keys of every chunk first
    CUtensorMap tq, tk, tkt, tktr, tv, ty;
    if (!rows_map(&tq, q, P, T, BH) || !rows_map(&tk, k, P, T, BH) || !kt_map(&tkt, kt, P, nch, BH, kKtCols) || !kt_rows_map(&tktr, kt, P, nch, BH, kKtCols) ||
        !rows_map(&tv, v, DV, T, BH) || !acc_map(&ty, yacc, DV, K::YW, nch * kChunk, BH))
        return cudaErrorInvalidValue;
    constexpr size_t intra_smem = 3 * kAtom + P * kKtRow + 1024;
    cudaError_t e = cudaFuncSetAttribute(intra_tc_kernel<P, DV, LG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)intra_smem);
    if (e != cudaSuccess) return e;
    KATA_TRACED("intra_tc", s,
                (intra_tc_kernel<P, DV, LG><<<dim3((unsigned)nch, (unsigned)BH), 128, intra_smem, s>>>(
                    tq, tk, tv, kt, ty, dacc, T)));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(chunked_tc_kernel<P, DV, LG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)K::smem)) != cudaSuccess)
        return e;
    KATA_TRACED("chunked_tc", s,
                (chunked_tc_kernel<P, DV, LG><<<dim3((unsigned)BH, (unsigned)(K::CS * G)), kThreads, K::smem, s>>>(
                    tq, tkt, tv, ty, tktr, dacc, S_start, z_start, start_groups, start_stride, S_final, z_final, T,
                    seg_chunks)));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t items = (int64_t)BH * T * (DV / 8);
    if (items > 0)
        KATA_TRACED("normalize", s,
                    (normalize_kernel<DV><<<(unsigned)((items + 255) / 256), 256, 0, s>>>(
                        yacc, dacc, static_cast<__nv_bfloat16*>(o), T, nch * kChunk, (int64_t)BH)));
    return cudaGetLastError();
}

}  // namespace

// (p, dv, lift blocks): the full lift (1 block) at p = 16, 32, 64 and the
// KATA-Sigma-g lift with blocks of 16 or 32 (p = 32 with g = 2; p = 64 with
// g = 2 or 4).
#define KATA_DISPATCH_DV(P_, LG_, ...)                                                   \
    do {                                                                                 \
        if (dv == 16) { constexpr int P = P_, DV = 16, LG = LG_; __VA_ARGS__; }          \
        if (dv == 32) { constexpr int P = P_, DV = 32, LG = LG_; __VA_ARGS__; }          \
        if (dv == 64) { constexpr int P = P_, DV = 64, LG = LG_; __VA_ARGS__; }          \
    } while (0)
#define KATA_DISPATCH(...)                                                   \
    do {                                                                     \
        if (p == 16 && lg == 1) KATA_DISPATCH_DV(16, 1, __VA_ARGS__);        \
        if (p == 32 && lg == 1) KATA_DISPATCH_DV(32, 1, __VA_ARGS__);        \
        if (p == 64 && lg == 1) KATA_DISPATCH_DV(64, 1, __VA_ARGS__);        \
        if (p == 32 && lg == 2) KATA_DISPATCH_DV(32, 2, __VA_ARGS__);        \
        if (p == 64 && lg == 2) KATA_DISPATCH_DV(64, 2, __VA_ARGS__);        \
        if (p == 64 && lg == 4) KATA_DISPATCH_DV(64, 4, __VA_ARGS__);        \
    } while (0)

bool chunked_tc_supports(int p, int dv, int lg) {
    bool ok = false;
    KATA_DISPATCH(ok = true);
    return ok;
}

int chunked_tc_segments(int p, int dv, int lg, int BH, int T) {
    const int nch = (T + kChunk - 1) / kChunk;
    int m = 0, cs = 1;
    KATA_DISPATCH(m = resident_ctas<P, DV, LG>(); cs = Cfg<P, DV, LG>::CS);
    if (m <= 0) return 0;
    if (nch <= 0) return 1;
    // as many segments per head as keep every resident CTA busy in one wave
    int G = (m / cs) / (BH > 0 ? BH : 1);
    if (G < 1) G = 1;
    if (G > nch) G = nch;
    const int per = (nch + G - 1) / G;
    return (nch + per - 1) / per;
}

int chunked_tc_segment_chunks(int T, int G) {
    const int nch = (T + kChunk - 1) / kChunk;
    return (nch + G - 1) / G;
}

size_t chunked_tc_intra_bytes(int BH, int T, int p, int dv) { return intra_ws(BH, T, p, dv).total; }

cudaError_t launch_chunked_tc(const void* q, const void* k, const void* v, void* o, void* intra,
                              const float* S_start, const float* z_start, int start_groups, int start_stride,
                              float* S_final, float* z_final, int BH, int T, int p, int dv, int lg, int G,
                              cudaStream_t s) {
    const int seg_chunks = chunked_tc_segment_chunks(T, G);
    KATA_DISPATCH(return launch_typed<P, DV, LG>(q, k, v, o, intra, S_start, z_start, start_groups, start_stride, S_final,
                                                 z_final, BH, T, seg_chunks, G, s));
    return cudaErrorInvalidValue;
}

unsigned int chunked_tc_take_status() {
    unsigned int val = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&val, g_chunked_tc_status, sizeof(val)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_chunked_tc_status, &zero, sizeof(zero));
    return val;
}

}  // namespace kata
