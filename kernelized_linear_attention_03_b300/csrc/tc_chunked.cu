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
// "extra CTA" owns the last, partly filled tile and Z (the inter-chunk
// denominator).  Each CTA's partial Y (128 x dv, sent as bf16) is summed in
// distributed shared memory: tile CTA r owns rows [r*R, r*R + R) of the
// chunk, receives the partials of those rows from every CTA of the cluster
// (a ring of RS chunks) and stores their sum and the rows' inter-chunk
// denominator.  The intra-chunk part of every chunk is computed by a separate
// kernel on a second stream, beside the clusters (which leave SMs free); a
// combine pass then adds it and divides.
#include <cooperative_groups.h>
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
namespace cg = cooperative_groups;

__device__ unsigned int g_chunked_tc_status = 0;


constexpr int kThreads = 512;  // warpgroups: lift, state epilogue, readout epilogue, MMA
// Register split between the warpgroups after launch (setmaxnreg): the MMA
// warpgroup gives back registers that the lift and state warpgroups take.
// 128 * (kRegsLift + kRegsState + kRegsLaunch + kRegsMma) must not exceed
// 512 * (registers per thread at launch); the launcher checks that.
constexpr uint32_t kRegsLift = 168, kRegsState = 128, kRegsLaunch = 128, kRegsMma = 88;
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
    static constexpr int R = kChunk / NTC;             // output rows owned per tile CTA (the extra CTA owns none)
    // shared memory, in 16 KB atoms from a 1024-byte aligned base
    //   tile CTA : key lift [0, 2 TPC), V (slot 0), bf16 state [TPC], query/key staging, V (slot 1)
    //   extra CTA: tail key lift, unit keys [2], bf16 Z, V (slot 0), bf16 tail state, staging [2], V (slot 1)
    static constexpr uint32_t t_ak = 0, t_v = (2 * TPC) * kAtom, t_s16 = (2 * TPC + 1) * kAtom,
                              t_stage = (3 * TPC + 1) * kAtom, t_v2 = (3 * TPC + 3) * kAtom;
    static constexpr uint32_t x_ak = 0, x_kh = 1 * kAtom, x_z16 = 3 * kAtom, x_v = 4 * kAtom,
                              x_s16 = 5 * kAtom, x_stage = 6 * kAtom, x_v2 = 10 * kAtom;  // extra: V slots x_v, x_v2,
                                                                                           // unit-key slots x_kh, x_kh + 1
    // query / key row staging, (Q tile, K tile) per stage, filled by TMA: one
    // stage in a tile CTA (its lift warps copy the rows out at once), two in
    // the extra CTA (its MMAs read the queries in place)
    static constexpr uint32_t atoms = 11, atoms_tile = 3 * TPC + 4;
    // partial readouts received by a tile CTA: one part per (source CTA,
    // receive slot) = R rows of bf16 laid out [DV/8][R] x 16 bytes (a warp's
    // store of one column group is contiguous per owner), then R fp32
    // denominators (extra CTA's part only)
    static constexpr uint32_t part_y = R * DV * 2;
    static constexpr uint32_t recv_part = part_y + round16(R * 4);
    static constexpr uint32_t recv_buf = CS * recv_part;
    static constexpr uint32_t recv_off = atoms_tile * kAtom;
    // receive slots (chunks in flight): three where they fit
    static constexpr int RS = recv_off + 3 * recv_buf + 1024 + 4096 <= 232448 ? 3 : 2;
    static constexpr uint32_t total = (recv_off + RS * recv_buf) > atoms * kAtom ? recv_off + RS * recv_buf : atoms * kAtom;
    static constexpr size_t smem = total + 1024;
    // tensor memory columns, tile CTA
    static constexpr uint32_t tm_s = 0;      // TPC x 64: fp32 state
    static constexpr uint32_t tm_aq = 128;   // 2 slots x 128: query lift
    static constexpr uint32_t tm_y = 384;    // 2 slots x 64: partial readout
    // tensor memory columns, extra CTA
    static constexpr uint32_t tx_s = 0;      // tail state
    static constexpr uint32_t tx_aq = 64;    // 2 slots x 32: tail query lift
    static constexpr uint32_t tx_y = 128;    // 2 slots x 64: partial readout
    static constexpr uint32_t tx_w = 384;    // Q Z
    static constexpr uint32_t tx_z = 448;    // Z
    static_assert(NT % TPC == 0, "tiles must split evenly");
    static_assert(TAIL > 0 && TAIL <= 32, "tail tile");
    static_assert(total + 1024 <= 232448, "shared memory");
    static_assert(atoms_tile <= atoms, "tile CTA layout");
    static_assert(R * NTC == kChunk, "owned rows");
};

// ---------------------------------------------------------------- lifts per tile
template <int P, int TAU>
__device__ __forceinline__ void key_tile(const uint32_t (&u)[P / 2], uint8_t* As, int row) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint4 val;
        val.x = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 0);
        val.y = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 1);
        val.z = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 2);
        val.w = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 3);
        *reinterpret_cast<uint4*>(As + mn_sw128_chunk(8 * c, row, kAtom)) = val;
    }
}

template <int P, int TAU>
__device__ __forceinline__ void query_tile(const uint32_t (&u)[P / 2], uint32_t taddr) {
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = lift::lift_word<P, true>(u, 64 * TAU + c0 + i);
        tmem_st16(taddr + c0, w);
    }
}

template <int P, int TAU = 0>
__device__ __forceinline__ void query_dispatch(int tau, const uint32_t (&uq)[P / 2], uint32_t taddr) {
    if constexpr (TAU < lift::tiles_of(P)) {
        if (tau == TAU)
            query_tile<P, TAU>(uq, taddr);
        else
            query_dispatch<P, TAU + 1>(tau, uq, taddr);
    }
}

template <int P, int TAU = 0>
__device__ __forceinline__ void key_dispatch(int tau, const uint32_t (&uk)[P / 2], uint8_t* As, int row) {
    if constexpr (TAU < lift::tiles_of(P)) {
        if (tau == TAU)
            key_tile<P, TAU>(uk, As, row);
        else
            key_dispatch<P, TAU + 1>(tau, uk, As, row);
    }
}

// Key lift of the last (partly filled) tile into its first 64-slot atom, up
// to the next multiple of 16 slots (slots past n are written as zeros).
template <int P>
__device__ __forceinline__ void key_tail(const uint32_t (&u)[P / 2], uint8_t* As, int row) {
    constexpr int TAU = lift::tiles_of(P) - 1;
    constexpr int tail = lift::packed_n(P) - 128 * TAU;
    constexpr int chunks = 2 * ((tail + 15) / 16);
#pragma unroll
    for (int c = 0; c < chunks; ++c) {
        uint4 val;
        val.x = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 0);
        val.y = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 1);
        val.z = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 2);
        val.w = lift::lift_word<P, false>(u, 64 * TAU + 4 * c + 3);
        *reinterpret_cast<uint4*>(As + mn_sw128_chunk(8 * c, row, kAtom)) = val;
    }
}

// Query lift of the last (partly filled) tile: its first 16 words (32 slots).
template <int P>
__device__ __forceinline__ void query_tail(const uint32_t (&uq)[P / 2], uint32_t taddr) {
    constexpr int TAU = lift::tiles_of(P) - 1;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = lift::lift_word<P, true>(uq, 64 * TAU + i);
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
// Warp roles (512 threads, four warpgroups):
//   warps 0-3   lift:     thread t = token t of the chunk; reads its staged
//                         query and key rows, puts the key on the unit sphere,
//                         writes the query lift (tensor memory) and the key
//                         lift (shared memory; extra CTA: also the unit keys)
//   warps 4-7   state:    thread e = tensor-memory lane e; reads the state
//                         after each update and releases it to the next update,
//                         refreshes the bf16 copy for the next readout (extra
//                         CTA: also Z and the rows' inter-chunk denominators)
//   warps 8-11  readout:  thread e = lane e; reads the partial readout and
//                         sends each row to the tile CTA that owns it
//   warps 12-15 warp 12 lane 0 issues every tcgen05.mma, warp 13 lane 0 the
//                         TMA loads; warps 14-15 reduce the owned rows and
//                         store their numerators and denominators
// Per chunk the MMAs run update (state += lift(K)^T V) then readout
// (Y = lift(Q) S), so the next update starts as soon as the state warps have
// read the state.
template <int P, int DV>
__global__ void __launch_bounds__(kThreads, 1)
chunked_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, __nv_bfloat16* __restrict__ o,
                  float* __restrict__ den_out, const float* __restrict__ S_start, const float* __restrict__ z_start, int start_groups,
                  float* __restrict__ S_final, float* __restrict__ z_final, int T, int seg_chunks) {
    using K = Cfg<P, DV>;
    constexpr int n = K::n;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t lift_full[2], aq_free[2], y_part[2], y_free[2], den_ready[2], v_free[2];
    __shared__ uint64_t recv_full[K::RS], peer_free[K::RS];
    __shared__ uint64_t local_full[K::RS];  // this CTA's own partial rows written (one arrival per row)
    __shared__ float dens[2][kChunk];  // extra CTA: denominators of the chunk rows
    __shared__ uint64_t ak_free, upd_done, state_read, s16_ready, drain;
    __shared__ uint64_t rd_sync;  // bounded group barrier of the reduce warps
    __shared__ uint64_t stage_full[2], stage_free[2], v_full[2], kh_free[2];
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
    const int c0 = g * seg_chunks, c1 = min(NCH, c0 + seg_chunks);
    const int nk = c1 - c0;
    const int my_rows = extra ? 0 : K::R;
    // bytes of partial rows (and the extra CTA's denominators) other CTAs
    // deliver per chunk
    const uint32_t rx_bytes = (K::CS - 1) * my_rows * DV * 2 + my_rows * 4;
    // shared memory of this CTA's role
    uint8_t* const s_ak = sm + (extra ? K::x_ak : K::t_ak);
    // value buffer of chunk kk (two, so the next chunk's values load while the
    // update, or in the extra CTA the one-chunk-late intra part, reads these)
    auto v_buf = [&](int kk) { return sm + ((kk & 1) ? (extra ? K::x_v2 : K::t_v2) : (extra ? K::x_v : K::t_v)); };
    // staging stages and the stage of chunk kk
    const int nstg = extra ? 2 : 1;
    uint8_t* const s_s16 = sm + (extra ? K::x_s16 : K::t_s16);
    uint8_t* const s_stage = sm + (extra ? K::x_stage : K::t_stage);
    auto s_kh = [&](int kk) { return sm + K::x_kh + (kk & 1) * kAtom; };
    uint8_t* const s_z16 = sm + K::x_z16;
    uint8_t* const s_recv = sm + K::recv_off;

    if (t == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&lift_full[b], 128);
            mbar_init(&aq_free[b], 1);
            mbar_init(&y_part[b], 1);
            mbar_init(&y_free[b], 128);

            mbar_init(&den_ready[b], 128);
            mbar_init(&v_free[b], 1);
        }
        mbar_init(&rd_sync, 64);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&stage_full[b], 1);
            // the staged rows are read by the lift warps and, in the extra CTA,
            // also by the state warps (its Q operand lives there)
            mbar_init(&stage_free[b], extra ? 256 : 128);
            mbar_init(&kh_free[b], 1);
            mbar_init(&v_full[b], 1);
        }
        mbar_init(&ak_free, 1);
        mbar_init(&upd_done, 1);
        mbar_init(&state_read, 128);
        mbar_init(&s16_ready, 128);
        mbar_init(&drain, 1);
        fence_mbar_init();
        for (int b = 0; b < K::RS; ++b) {
            mbar_init(&recv_full[b], 1);
            mbar_init(&peer_free[b], K::NTC);  // one arrival per owner
            mbar_init(&local_full[b], my_rows > 0 ? my_rows : 1);
        }
        fence_mbar_init();
        // the first RS chunks' partial rows may arrive as soon as the cluster starts
        if (my_rows > 0)
            for (int b = 0; b < K::RS && b < nk; ++b) mbar_arrive_expect_tx(&recv_full[b], rx_bytes);
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
    auto wait_cluster = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, &abort_flag, kWaitNs));
    };
    // Group barrier of 128 threads on an mbarrier (bounded, unlike bar.sync):
    // every thread arrives, then waits for the phase of use number `n`.
    auto group_sync = [&](uint64_t* bar, uint32_t n) {
        mbar_arrive(bar);
        return wait(bar, n & 1);
    };

    // ---- start state of this segment (epilogue warps: lane = slot / dim)
    if (warp >= 4 && warp < 8) {
        const int e = t - 128;
        const int sg = start_groups > 1 ? g : 0;
        const float* S0 = S_start ? S_start + (bh * start_groups + sg) * (int64_t)n * DV : nullptr;
        const float* z0 = z_start ? z_start + (bh * start_groups + sg) * (int64_t)n : nullptr;
        if (!extra) {
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl)
                load_state_tile<P, DV>(S0, rank * K::TPC + tl, tm(K::tm_s + 64 * tl), s_s16 + tl * kAtom, e);
        } else {
            load_state_tile<P, DV>(S0, K::NT, tm(K::tx_s), s_s16, e);
            float zr[P];
#pragma unroll
            for (int j = 0; j < P; ++j) {
                float val = 0.f;
                if (z0 != nullptr && e < P) {
                    const int a = e < j ? e : j, b = e < j ? j : e;
                    val = z0[lift::canonical_index(P, a, b)] * (a == b ? 1.f : kInvSqrt2f);
                }
                zr[j] = val;
            }
#pragma unroll
            for (int c = 0; c < P; c += 16) {
                uint32_t r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(zr[c + i]);
                tmem_st16(tm(K::tx_z + c), r);
            }
            if (e < P) {
#pragma unroll
                for (int c = 0; c < P / 8; ++c)
                    *reinterpret_cast<uint4*>(s_z16 + sw128_chunk(e, 8 * c, P)) =
                        make_uint4(pack_bf16x2(zr[8 * c], zr[8 * c + 1]), pack_bf16x2(zr[8 * c + 2], zr[8 * c + 3]),
                                   pack_bf16x2(zr[8 * c + 4], zr[8 * c + 5]), pack_bf16x2(zr[8 * c + 6], zr[8 * c + 7]));
            }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
    }
    tc_fence_before();
    cluster.sync();  // barriers initialised and start state in place cluster-wide
    tc_fence_after();

    if (warp < 4) {
        // =============================================================== lift warps
        regs_inc<kRegsLift>();
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            const int stg = kk % nstg, stg_use = kk / nstg;
            // this token's query and key rows (128-byte swizzled, staged by TMA)
            if (!wait(&stage_full[stg], stg_use & 1)) { fail(); break; }
            const uint8_t* my_q = s_stage + stg * 2 * kAtom + t * 128;
            const uint8_t* my_k = my_q + kAtom;
            uint32_t uq[P / 2];
            uint4 kraw[P / 8];
#pragma unroll
            for (int i = 0; i < P / 8; ++i) {
                const uint4 a = *reinterpret_cast<const uint4*>(my_q + ((i ^ (t & 7)) << 4));
                uq[4 * i] = a.x;
                uq[4 * i + 1] = a.y;
                uq[4 * i + 2] = a.z;
                uq[4 * i + 3] = a.w;
                kraw[i] = *reinterpret_cast<const uint4*>(my_k + ((i ^ (t & 7)) << 4));
            }
            mbar_arrive(&stage_free[stg]);
            // unit key
            uint32_t uk[P / 2];
            {
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < P / 8; ++i) {
                    const __nv_bfloat16* ke = reinterpret_cast<const __nv_bfloat16*>(&kraw[i]);
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
            }
            // query lift -> tensor memory slot (double-buffered: overlaps the
            // previous chunk's update)
            if (kk >= 2 && !wait(&aq_free[slot], (use - 1) & 1)) { fail(); break; }
            tc_fence_after();
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
                    query_dispatch<P>(rank * K::TPC + tl, uq, tm(K::tm_aq + 128 * slot + 64 * tl));
            } else {
                query_tail<P>(uq, tm(K::tx_aq + 32 * slot));
            }
            // key lift -> shared memory (single buffer)
            if (kk >= 1 && !wait(&ak_free, (kk - 1) & 1)) { fail(); break; }
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
                    key_dispatch<P>(rank * K::TPC + tl, uk, s_ak + 2 * tl * kAtom, t);
            } else {
                key_tail<P>(uk, s_ak, t);
                if (kk >= 2 && !wait(&kh_free[slot], (use - 1) & 1)) { fail(); break; }
#pragma unroll
                for (int i = 0; i < P / 8; ++i)
                    *reinterpret_cast<uint4*>(s_kh(kk) + sw128_chunk(t, 8 * i, kChunk)) =
                        make_uint4(uk[4 * i], uk[4 * i + 1], uk[4 * i + 2], uk[4 * i + 3]);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&lift_full[slot]);
        }
    } else if (warp < 8) {
        // =============================================================== state warps
        regs_inc<kRegsState>();
        const int e = t - 128;
        bool ok = true;
        for (int kk = 0; kk < nk && ok; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            // state after this chunk's update
            if (!wait(&upd_done, kk & 1)) { fail(); break; }
            tc_fence_after();
            uint32_t sreg[K::TPC][DV / 2];  // bf16 pairs of this lane's state rows
            uint32_t zreg[P / 2];           // extra CTA: bf16 pairs of this lane's Z row
            float den = 0.f;
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
#pragma unroll
                    for (int c16 = 0; c16 < DV; c16 += 16) {
                        uint32_t r[16];
                        tmem_ld16(tm(K::tm_s + 64 * tl + c16), r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            sreg[tl][c16 / 2 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    }
                tc_fence_before();
                mbar_arrive(&state_read);
            } else {
#pragma unroll
                for (int c16 = 0; c16 < DV; c16 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tx_s + c16), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        sreg[0][c16 / 2 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                }
#pragma unroll
                for (int c16 = 0; c16 < P; c16 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tx_z + c16), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        zreg[c16 / 2 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                }
                tc_fence_before();
                mbar_arrive(&state_read);
            }
            // this chunk's readout is done: its bf16 state copy may be replaced
            if (!wait(&y_part[slot], use & 1)) { fail(); break; }
            tc_fence_after();
            if (extra) {
                // inter-chunk denominator q^T Z q from W = Q Z (Z before this chunk)
                uint4 qrow[P / 8];
                const uint8_t* sq = s_stage + slot * 2 * kAtom;  // this chunk's staged queries
#pragma unroll
                for (int i = 0; i < P / 8; ++i) qrow[i] = *reinterpret_cast<const uint4*>(sq + sw128_chunk(e, 8 * i, kChunk));
                const __nv_bfloat16* qe = reinterpret_cast<const __nv_bfloat16*>(qrow);
                float dint = 0.f;
#pragma unroll
                for (int c16 = 0; c16 < P; c16 += 16) {
                    uint32_t w[16];
                    tmem_ld16(tm(K::tx_w + c16), w);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) dint = fmaf(__bfloat162float(qe[c16 + i]), __uint_as_float(w[i]), dint);
                }
                den += dint;
                tc_fence_before();
                mbar_arrive(&stage_free[slot]);  // this chunk's staged queries and W have been read
            }
            auto write_s16 = [&](const uint32_t (&x)[DV / 2], int tl) {
#pragma unroll
                for (int c8 = 0; c8 < DV / 8; ++c8)
                    *reinterpret_cast<uint4*>(s_s16 + tl * kAtom + mn_sw128_chunk(8 * c8, e, kAtom)) =
                        make_uint4(x[4 * c8], x[4 * c8 + 1], x[4 * c8 + 2], x[4 * c8 + 3]);
            };
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl) write_s16(sreg[tl], tl);
            } else {
                write_s16(sreg[0], 0);
                if (e < P) {
#pragma unroll
                    for (int c8 = 0; c8 < P / 8; ++c8)
                        *reinterpret_cast<uint4*>(s_z16 + sw128_chunk(e, 8 * c8, P)) =
                            make_uint4(zreg[4 * c8], zreg[4 * c8 + 1], zreg[4 * c8 + 2], zreg[4 * c8 + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s16_ready);
            if (extra) {
                dens[slot][e] = den;
                mbar_arrive(&den_ready[slot]);
            }
        }
        // final state of the last segment
        if (S_final != nullptr && g == G - 1 && !abort_flag) {
            const int64_t head_s = bh * (int64_t)n * DV, head_z = bh * (int64_t)n;
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
                    store_state_tile<P, DV>(S_final + head_s, rank * K::TPC + tl, tm(K::tm_s + 64 * tl), e);
            } else {
                store_state_tile<P, DV>(S_final + head_s, K::NT, tm(K::tx_s), e);
                uint32_t zr[P];
#pragma unroll
                for (int c16 = 0; c16 < P; c16 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tx_z + c16), r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) zr[c16 + i] = r[i];
                }
                tmem_wait_ld();
                if (e < P) {
#pragma unroll
                    for (int j = 0; j < P; ++j)
                        if (j >= e)
                            z_final[head_z + lift::canonical_index(P, e, j)] = __uint_as_float(zr[j]) * (j == e ? 1.f : kSqrt2f);
                }
            }
        }
    } else if (warp < 12) {
        // =============================================================== readout warps
        const int e = t - 256;
        const int owner = e / K::R, orow = e % K::R;
        // this lane's partial readout of chunk c0 + kc -> its owner (the extra
        // CTA adds the row's inter-chunk denominator)
        auto send = [&](int kc) -> bool {
            const int slot = kc & 1, use = kc >> 1;
            const int rs = kc % K::RS, ruse = kc / K::RS;
            if (!wait(&y_part[slot], use & 1)) return false;
            tc_fence_after();
            float den = 0.f;
            if (extra) {
                if (!wait(&den_ready[slot], use & 1)) return false;
                den = dens[slot][e];
            }
            uint32_t ypk[DV / 2];
            const uint32_t ycol = (extra ? K::tx_y : K::tm_y) + 64 * slot;
#pragma unroll
            for (int c16 = 0; c16 < DV; c16 += 16) {
                uint32_t r[16];
                tmem_ld16(tm(ycol + c16), r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) ypk[c16 / 2 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            }
            tc_fence_before();
            mbar_arrive(&y_free[slot]);
            // the owners have consumed what this receive slot held RS chunks ago
            if (kc >= K::RS && !wait_cluster(&peer_free[rs], (ruse - 1) & 1)) return false;
            uint8_t* recv = s_recv + rs * K::recv_buf;
            uint8_t* dst = recv + rank * K::recv_part + orow * 16;
            if (owner == rank) {
#pragma unroll
                for (int i = 0; i < DV / 8; ++i)
                    *reinterpret_cast<uint4*>(dst + i * K::R * 16) = make_uint4(ypk[4 * i], ypk[4 * i + 1], ypk[4 * i + 2], ypk[4 * i + 3]);
                if (extra) *reinterpret_cast<float*>(recv + rank * K::recv_part + K::part_y + orow * 4) = den;
                mbar_arrive(&local_full[rs]);
            } else {
                const uint32_t rdst = cluster_addr(dst, owner);
                const uint32_t rbar = cluster_addr(&recv_full[rs], owner);
#pragma unroll
                for (int i = 0; i < DV / 8; ++i)
                    st_async_v4_b32(rdst + i * K::R * 16, ypk[4 * i], ypk[4 * i + 1], ypk[4 * i + 2], ypk[4 * i + 3], rbar);
                if (extra) st_async_f32(cluster_addr(recv + rank * K::recv_part + K::part_y + orow * 4, owner), den, rbar);
            }
            return true;
        };
        for (int kk = 0; kk < nk; ++kk)
            if (!send(kk)) { fail(); break; }
    } else {
        regs_dec<kRegsMma>();
    }
    if (warp >= 14 && my_rows > 0) {
        // =============================================================== reduce warps
        // owner side, chunk by chunk as the partial rows land: sum them, store
        // the rows' inter-chunk numerator and denominator, then hand the
        // receive slot back to every sender (its next use is RS chunks later)
        constexpr int kRedIt = (K::R * (DV / 8) + 63) / 64;
        const int er = t - 448;
        const int r0 = rank * K::R;
        const int items = my_rows * (DV / 8);
        __nv_bfloat16* oh = o + bh * (int64_t)T * DV;
        float* dh = den_out + bh * (int64_t)T;
        for (int kr = 0; kr < nk; ++kr) {
            const int r = kr % K::RS;
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(&recv_full[r], (kr / K::RS) & 1, &abort_flag, kWaitNs) &&
                                             mbar_wait(&local_full[r], (kr / K::RS) & 1, &abort_flag, kWaitNs))) {
                fail();
                break;
            }
            const uint8_t* recv = s_recv + r * K::recv_buf;
#pragma unroll
            for (int it = 0; it < kRedIt; ++it) {
                const int idx = er + 64 * it;
                if (idx >= items) break;
                const int lr = idx % my_rows, i = idx / my_rows;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int src = 0; src < K::CS; ++src) {
                    const uint4 x = *reinterpret_cast<const uint4*>(recv + src * K::recv_part + (i * K::R + lr) * 16);
                    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[2 * j] += __low2float(h[j]);
                        acc[2 * j + 1] += __high2float(h[j]);
                    }
                }
                const int otok = (c0 + kr) * kChunk + r0 + lr;
                if (otok < T) {
                    // the inter-chunk numerator and denominator of the row; the
                    // combine pass adds the intra-chunk part and divides
                    *reinterpret_cast<uint4*>(oh + (int64_t)otok * DV + 8 * i) =
                        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                                   pack_bf16x2(acc[6], acc[7]));
                    if (i == 0) dh[otok] = *reinterpret_cast<const float*>(recv + K::NTC * K::recv_part + K::part_y + lr * 4);
                }
            }
            mbar_arrive(&rd_sync);
            if (!__all_sync(0xffffffffu, mbar_wait(&rd_sync, kr & 1, &abort_flag, kWaitNs))) {
                fail();
                break;
            }
            if (er == 0 && kr + K::RS < nk) mbar_arrive_expect_tx(&recv_full[r], rx_bytes);
            if (er < K::CS) mbar_arrive_remote(cluster_addr(&peer_free[r], er));
        }
    }
    if (t == 416) {
        // =============================================================== TMA producer
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            const int stg = kk % nstg, stg_use = kk / nstg;
            const int row = (c0 + kk) * kChunk;
            // query and key rows of chunk kk into its stage
            if (kk >= nstg && !mbar_wait(&stage_free[stg], (stg_use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&stage_full[stg], 2 * kAtom);
            tma_load_3d(s_stage + stg * 2 * kAtom, &tmq, 0, row, (int)bh, &stage_full[stg]);
            tma_load_3d(s_stage + stg * 2 * kAtom + kAtom, &tmk, 0, row, (int)bh, &stage_full[stg]);
            // value tile of chunk kk into its buffer
            if (kk >= 2 && !mbar_wait(&v_free[slot], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&v_full[slot], kAtom);
            tma_load_3d(v_buf(kk), &tmv, 0, row, (int)bh, &v_full[slot]);
        }
    }
    if (t == 384) {
        // =============================================================== MMA issuer
        // Every descriptor is built once: one thread issues all MMAs, so the
        // issue loop carries no descriptor arithmetic beyond one add per
        // K step (a step moves the start-address field, in 16-byte units).
        constexpr uint32_t id_read = idesc_bf16_f32_major(128, DV, false, true);
        constexpr uint32_t id_upd = idesc_bf16_f32_major(128, DV, true, true);
        constexpr uint32_t id_z = idesc_bf16_f32_major(128, P, true, true);
        constexpr uint32_t id_w = idesc_bf16_f32(128, P);
        constexpr uint64_t kStepMN = 2048 >> 4, kStepK = 32 >> 4, kAtomD = kAtom >> 4;
        // key lift (A of the update): tile CTA two 64-slot atoms per tile; the
        // extra CTA's tail tile one atom that the second M atom aliases (its
        // rows past the tail are never read)
        const uint64_t d_ak = sdesc_mnmajor_sw128(smem_u32(s_ak), extra ? 0u : kAtom);
        const uint64_t d_s16 = sdesc_mnmajor_sw128(smem_u32(s_s16), kAtom);
        const uint64_t d_v[2] = {sdesc_mnmajor_sw128(smem_u32(v_buf(0)), kAtom),
                                 sdesc_mnmajor_sw128(smem_u32(v_buf(1)), kAtom)};
        // extra CTA: unit keys as M (aliased atoms) and as N; staged Q; Z
        const uint64_t d_khm[2] = {sdesc_mnmajor_sw128(smem_u32(s_kh(0)), 0), sdesc_mnmajor_sw128(smem_u32(s_kh(1)), 0)};
        const uint64_t d_khn[2] = {sdesc_mnmajor_sw128(smem_u32(s_kh(0)), kAtom),
                                   sdesc_mnmajor_sw128(smem_u32(s_kh(1)), kAtom)};
        const uint64_t d_q[2] = {sdesc_kmajor_sw128(smem_u32(s_stage)), sdesc_kmajor_sw128(smem_u32(s_stage + 2 * kAtom))};
        const uint64_t d_z16 = sdesc_kmajor_sw128(smem_u32(s_z16));
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            if (!mbar_wait(&lift_full[slot], use & 1, &abort_flag, kWaitNs)) { fail(); break; }
            if (!mbar_wait(&v_full[slot], use & 1, &abort_flag, kWaitNs)) { fail(); break; }
            if (kk >= 1 && !mbar_wait(&state_read, (kk - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            tc_fence_after();
            const uint64_t dv = d_v[slot];
            // ---- group U: state updates (extra CTA: tail state and Z)
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss(tb + K::tm_s + 64 * tl, d_ak + 2 * tl * kAtomD + ks * kStepMN, dv + ks * kStepMN, id_upd, 1u);
                mma_commit(&upd_done);
                mma_commit(&ak_free);
                mma_commit(&v_free[slot]);
            } else {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) mma_ss(tb + K::tx_s, d_ak + ks * kStepMN, dv + ks * kStepMN, id_upd, 1u);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tb + K::tx_z, d_khm[slot] + ks * kStepMN, d_khn[slot] + ks * kStepMN, id_z, 1u);
                mma_commit(&upd_done);
                mma_commit(&ak_free);
                mma_commit(&v_free[slot]);
                mma_commit(&kh_free[slot]);
            }
            // ---- group R: readout of the state before this chunk
            if (kk >= 1 && !mbar_wait(&s16_ready, (kk - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            if (kk >= 2 && !mbar_wait(&y_free[slot], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            tc_fence_after();
            if (!extra) {
                const uint32_t dy = tb + K::tm_y + 64 * slot, aq = tb + K::tm_aq + 128 * slot;
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts(dy, aq + 64 * tl + 8 * ks, d_s16 + tl * kAtomD + ks * kStepMN, id_read,
                               (tl > 0 || ks > 0) ? 1u : 0u);
                mma_commit(&y_part[slot]);
                mma_commit(&aq_free[slot]);
            } else {
                const uint32_t dy = tb + K::tx_y + 64 * slot, aq = tb + K::tx_aq + 32 * slot;
#pragma unroll
                for (int ks = 0; ks < (K::TAIL + 15) / 16; ++ks)
                    mma_ts(dy, aq + 8 * ks, d_s16 + ks * kStepMN, id_read, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < P / 16; ++ks)
                    mma_ss(tb + K::tx_w, d_q[slot] + ks * kStepK, d_z16 + ks * kStepK, id_w, ks > 0 ? 1u : 0u);
                mma_commit(&y_part[slot]);
                mma_commit(&aq_free[slot]);
            }
        }
        // every issued MMA has completed before tensor memory is released
        mma_commit(&drain);
        mbar_wait_quiet(&drain, 0, kWaitNs);
    }

    tc_fence_before();
    __syncwarp();
    cluster.sync();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------- intra-chunk part
// Every chunk on its own (no state): for the 128 queries of a chunk,
//   P = (Q Kh^T) o (Q Kh^T) o M   (bf16, M the causal mask s <= t)
//   Y = P V,  d = rowsum(P)       (fp32 accumulation)
// Y goes out as bf16 rows [BH][T][DV] and d, the rows' intra-chunk
// normaliser, as fp32 [BH][T]; the fused forward adds both when it combines
// a chunk's rows.  d sums exactly the rounded weights Y is built from, which
// keeps the intra-chunk weights a convex combination.  One CTA per (chunk,
// head), 128 columns of tensor memory and 48 KB of shared memory, so several
// chunks are in flight per SM; thread t owns query / key / value row t.
template <int P, int DV>
__global__ void __launch_bounds__(128)
intra_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                const __nv_bfloat16* __restrict__ v, __nv_bfloat16* __restrict__ y_out, float* __restrict__ d_out,
                int T) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar, drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* Qs = sm;              // K-major, 128 rows x 128 B
    uint8_t* Ks = sm + kAtom;      // unit keys, K-major
    uint8_t* Vs = sm + 2 * kAtom;  // V, MN-major
    const int t = threadIdx.x, warp = t >> 5;
    const int64_t bh = blockIdx.y;
    const int row = blockIdx.x * kChunk + t;
    const bool valid = row < T;
    const int64_t grow = bh * T + (valid ? row : 0);
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_init(&drain, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    // rows -> shared memory (zeros past T)
    {
        const uint4* gq = reinterpret_cast<const uint4*>(q + grow * P);
        const uint4* gk = reinterpret_cast<const uint4*>(k + grow * P);
        const uint4* gv = reinterpret_cast<const uint4*>(v + grow * DV);
        uint4 kr[P / 8];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < P / 8; ++i) {
            const uint4 a = valid ? gq[i] : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(Qs + sw128_chunk(t, 8 * i, kChunk)) = a;
            kr[i] = valid ? gk[i] : make_uint4(0, 0, 0, 0);
            const __nv_bfloat16* ke = reinterpret_cast<const __nv_bfloat16*>(&kr[i]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = __bfloat162float(ke[j]);
                ss = fmaf(x, x, ss);
            }
        }
        const float kinv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
        for (int i = 0; i < P / 8; ++i) {
            const __nv_bfloat16* ke = reinterpret_cast<const __nv_bfloat16*>(&kr[i]);
            uint4 w;
            w.x = pack_bf16x2(__bfloat162float(ke[0]) * kinv, __bfloat162float(ke[1]) * kinv);
            w.y = pack_bf16x2(__bfloat162float(ke[2]) * kinv, __bfloat162float(ke[3]) * kinv);
            w.z = pack_bf16x2(__bfloat162float(ke[4]) * kinv, __bfloat162float(ke[5]) * kinv);
            w.w = pack_bf16x2(__bfloat162float(ke[6]) * kinv, __bfloat162float(ke[7]) * kinv);
            *reinterpret_cast<uint4*>(Ks + sw128_chunk(t, 8 * i, kChunk)) = w;
        }
#pragma unroll
        for (int i = 0; i < DV / 8; ++i)
            *reinterpret_cast<uint4*>(Vs + mn_sw128_chunk(8 * i, t, kAtom)) = valid ? gv[i] : make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t lane0 = (uint32_t)(warp * 32);
    if (t == 0) {
        const uint64_t dq = sdesc_kmajor_sw128(smem_u32(Qs)), dk = sdesc_kmajor_sw128(smem_u32(Ks));
        constexpr uint32_t id_sc = idesc_bf16_f32(128, 128);
#pragma unroll
        for (int ks = 0; ks < P / 16; ++ks) mma_ss(tb, dq + 2 * ks, dk + 2 * ks, id_sc, ks > 0 ? 1u : 0u);
        mma_commit(&bar);
    }
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bar, 0, &abort_flag, kWaitNs));
    if (!ok) abort_flag = 1;
    tc_fence_after();
    // P = scores^2 masked, bf16, in place (columns 0..63), and its row sum;
    // quarters past this warp's rows are all masked
    float den = 0.f;
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
    ok = !abort_flag && __all_sync(0xffffffffu, mbar_wait(&bar, 1, &abort_flag, kWaitNs));
    tc_fence_after();
    if (ok) {
        uint32_t y[DV];
#pragma unroll
        for (int c = 0; c < DV; c += 16) tmem_ld16(tmem_addr(tb, lane0, 64 + c), *reinterpret_cast<uint32_t(*)[16]>(y + c));
        tmem_wait_ld();
        if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(y_out + grow * DV);
#pragma unroll
            for (int i = 0; i < DV / 8; ++i)
                dst[i] = make_uint4(pack_bf16x2(__uint_as_float(y[8 * i]), __uint_as_float(y[8 * i + 1])),
                                    pack_bf16x2(__uint_as_float(y[8 * i + 2]), __uint_as_float(y[8 * i + 3])),
                                    pack_bf16x2(__uint_as_float(y[8 * i + 4]), __uint_as_float(y[8 * i + 5])),
                                    pack_bf16x2(__uint_as_float(y[8 * i + 6]), __uint_as_float(y[8 * i + 7])));
            d_out[grow] = den;
        }
    } else if (t == 0) {
        atomicOr(&g_chunked_tc_status, kStatusTimeout);
    }
    // every issued MMA has completed before the tensor memory is released
    if (t == 0) {
        mma_commit(&drain);
        mbar_wait_quiet(&drain, 0, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 128);
}

// o = (numerator + intra rows) / (denominator + intra normaliser), in place
// over the fused kernel's bf16 numerators; thread = 8 columns of one row.
template <int DV>
__global__ void __launch_bounds__(256)
combine_kernel(__nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ y_intra,
               const float* __restrict__ d_intra, const float* __restrict__ d_inter, int64_t rows) {
    const int64_t total = rows * (DV / 8);
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = idx / (DV / 8);
        const uint4 a = reinterpret_cast<const uint4*>(o)[idx];
        const uint4 b = reinterpret_cast<const uint4*>(y_intra)[idx];
        const float d = d_inter[row] + d_intra[row];
        const float inv = d > 0.f ? 1.f / d : 0.f;
        const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
        uint4 r;
        uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = pack_bf16x2((__low2float(ha[j]) + __low2float(hb[j])) * inv,
                               (__high2float(ha[j]) + __high2float(hb[j])) * inv);
        reinterpret_cast<uint4*>(o)[idx] = r;
    }
}

// ---------------------------------------------------------------- host side
// The register split of the kernel fits in its launch allocation.
template <int P, int DV>
bool register_split_fits() {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, chunked_tc_kernel<P, DV>) != cudaSuccess) return false;
    return (uint32_t)kThreads * (uint32_t)fa.numRegs >= 128u * (kRegsLift + kRegsState + kRegsLaunch + kRegsMma);
}

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
        if (!register_split_fits<P, DV>() || configure<P, DV>(cfg, attr, 1, 1, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&m, chunked_tc_kernel<P, DV>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cached[dev] = m > 0 ? m : -1;
    }
    return cached[dev] > 0 ? cached[dev] : 0;
}

// A second stream of the current device, and two events, for running the
// intra-chunk kernel beside the fused kernel (created once per device).
struct AuxStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex mu;  // held across one call's fork ... join, so calls from several host threads do not interleave
};
cudaError_t aux_stream(AuxStream** out) {
    static AuxStream aux[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    AuxStream& a = aux[dev];
    if (a.s == nullptr) {
        if ((e = cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &a;
    return cudaSuccess;
}

template <int P, int DV>
cudaError_t launch_typed(const void* q, const void* k, const void* v, void* o, void* y_intra, float* d_intra,
                         float* d_inter, const float* S_start, const float* z_start, int start_groups,
                         float* S_final, float* z_final, int BH, int T, int seg_chunks, int G, cudaStream_t s) {
    if (!register_split_fits<P, DV>()) return cudaErrorInvalidConfiguration;
    AuxStream* aux = nullptr;
    cudaError_t e = aux_stream(&aux);
    if (e != cudaSuccess) return e;
    // the intra-chunk rows of every chunk, on a second stream: the fused
    // kernel's clusters leave SMs free, and it does not read these rows
    constexpr size_t intra_smem = 3 * kAtom + 1024;
    if ((e = cudaFuncSetAttribute(intra_tc_kernel<P, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)intra_smem)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    if ((e = configure<P, DV>(cfg, attr, G, BH, s)) != cudaSuccess) return e;
    CUtensorMap tq, tk, tv;
    if (!rows_map(&tq, q, P, T, BH) || !rows_map(&tk, k, P, T, BH) || !rows_map(&tv, v, DV, T, BH))
        return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lk(aux->mu);
    if ((e = cudaEventRecord(aux->fork, s)) != cudaSuccess || (e = cudaStreamWaitEvent(aux->s, aux->fork, 0)) != cudaSuccess)
        return e;
    // the fused kernel first, so its clusters are placed before the intra CTAs fill the device
    KATA_TRACED("chunked_tc", s,
                e = cudaLaunchKernelEx(&cfg, chunked_tc_kernel<P, DV>, tq, tk, tv, static_cast<__nv_bfloat16*>(o),
                                       d_inter, S_start, z_start, start_groups, S_final, z_final, T, seg_chunks));
    if (e != cudaSuccess) return e;
    const dim3 igrid((unsigned)((T + kChunk - 1) / kChunk), (unsigned)BH);
    KATA_TRACED("intra_tc", aux->s,
                (intra_tc_kernel<P, DV><<<igrid, 128, intra_smem, aux->s>>>(
                    static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                    static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(y_intra), d_intra, T)));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaEventRecord(aux->join, aux->s)) != cudaSuccess || (e = cudaStreamWaitEvent(s, aux->join, 0)) != cudaSuccess)
        return e;
    const int64_t rows = (int64_t)BH * T;
    const int64_t work = rows * (DV / 8);
    const unsigned blocks = (unsigned)std::min<int64_t>((work + 255) / 256, 148 * 16);
    KATA_TRACED("combine", s,
                (combine_kernel<DV><<<blocks, 256, 0, s>>>(static_cast<__nv_bfloat16*>(o),
                                                             static_cast<const __nv_bfloat16*>(y_intra), d_intra,
                                                             d_inter, rows)));
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

size_t chunked_tc_intra_bytes(int BH, int T, int dv) {
    return (size_t)BH * (size_t)T * ((size_t)dv * 2 + 8);
}

cudaError_t launch_chunked_tc(const void* q, const void* k, const void* v, void* o, void* intra,
                              const float* S_start, const float* z_start, int start_groups, float* S_final,
                              float* z_final, int BH, int T, int p, int dv, int G, cudaStream_t s) {
    const int seg_chunks = chunked_tc_segment_chunks(T, G);
    // intra-chunk rows: bf16 [BH][T][dv], then fp32 intra-chunk normalisers
    // [BH][T], then the fused kernel's inter-chunk denominators [BH][T]
    void* y_intra = intra;
    float* d_intra = reinterpret_cast<float*>(static_cast<char*>(intra) + (size_t)BH * T * dv * 2);
    float* d_inter = d_intra + (size_t)BH * T;
    KATA_DISPATCH(return launch_typed<P, DV>(q, k, v, o, y_intra, d_intra, d_inter, S_start, z_start, start_groups,
                                             S_final, z_final, BH, T, seg_chunks, G, s));
    return cudaErrorInvalidValue;
}

unsigned int chunked_tc_take_status() {
    unsigned int val = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&val, g_chunked_tc_status, sizeof(val)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_chunked_tc_status, &zero, sizeof(zero));
    return val;
}

}  // namespace kata

