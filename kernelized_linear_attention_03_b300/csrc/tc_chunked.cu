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
// thread-block cluster.  Each "tile CTA" owns one or two 128-slot tiles of
// the packed lift; it keeps its state rows in tensor memory (fp32,
// accumulated by the update MMA) and a bf16 copy in shared memory (B operand
// of the readout MMA).  Its query lift goes to tensor memory (A operand of
// the readout), its key lift (A operand of the update, built one slot per
// thread from the chunk's transposed unit keys) to tensor memory as well
// where the columns allow (one tile per CTA), else to shared memory.  The
// "extra CTA" owns the last, partly filled tile and Z (the inter-chunk
// denominator).  Each CTA's partial Y (128 x dv, sent as bf16) is summed in
// distributed shared memory: tile CTA r owns rows [r*R, r*R + R) of the
// chunk, receives the partials of those rows from every CTA of the cluster
// (a ring of RS chunks), adds the rows' intra-chunk part and writes the
// outputs.  The intra-chunk part of every chunk, and the transposed unit
// keys the key lift reads, come from a kernel that runs first.
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


constexpr int kThreads = 512;  // warpgroups: query lift and readout, state epilogue, key lift, MMA
// Register split between the warpgroups after launch (setmaxnreg): the MMA
// warpgroup gives back registers that the query warpgroup takes.
// 128 * (kRegsLift + kRegsState + kRegsLaunch + kRegsMma) must not exceed
// 512 * (registers per thread at launch); the launcher checks that.
constexpr uint32_t kRegsLift = 152, kRegsState = 128, kRegsLaunch = 128, kRegsMma = 104;
constexpr int kChunk = 128;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kAtom = 128 * 128;  // 128 rows x 128 bytes
constexpr float kSqrt2f = 1.41421356237309504880f;
constexpr float kInvSqrt2f = 0.70710678118654752440f;

__host__ __device__ constexpr uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

// P: width of q and k; LG: blocks of the lift (1: the full lift; g > 1: the
// KATA-Sigma-g lift, the sum of the g block lifts of width M = P / g).
template <int P, int DV, int LG>
struct Cfg {
    static constexpr int M = P / LG;                   // width of the lifted blocks
    static constexpr int n = lift::packed_n(M);
    static constexpr int NT = n / 128;                 // full tiles
    static constexpr int TAIL = n - 128 * NT;          // slots of the last tile (8, 16 or 32)
    static constexpr int TPC = M == 64 ? 2 : 1;        // tiles per tile CTA
    static constexpr int NTC = NT / TPC;               // tile CTAs
    static constexpr int CS = NTC + 1;                 // cluster size
    static constexpr int R = kChunk / NTC;             // output rows owned per tile CTA (the extra CTA owns none)
    // transposed unit keys of a chunk: two 64-token boxes of P rows x 128 bytes
    static constexpr uint32_t kt_box = P * 128;
    static constexpr uint32_t kt_bytes = 2 * kt_box;
    // the tile CTA's key lift: tensor memory with one tile per CTA, shared
    // memory with two (their state, query lift double buffer and partial
    // readouts leave no columns for it)
    static constexpr bool AKT = TPC == 1;
    // shared memory, in 16 KB atoms from a 1024-byte aligned base
    //   tile CTA : [key lift, two 64-token atoms per tile, unless AKT], V x2,
    //              bf16 state [TPC], query stage, transposed-key stages x2
    //   extra CTA: V x2, bf16 tail state, bf16 Z, query stages x2,
    //              transposed-key stages x2, one spare atom (the M = 128
    //              reads of the Z update run past the last stage)
    static constexpr uint32_t ak_atoms = AKT ? 0 : 2 * TPC;
    static constexpr uint32_t t_ak = 0, t_v = ak_atoms * kAtom, t_s16 = t_v + 2 * kAtom, t_q = t_s16 + TPC * kAtom,
                              t_kt = t_q + kAtom;
    static constexpr uint32_t x_v = 0, x_s16 = 2 * kAtom, x_z16 = 3 * kAtom, x_q = 4 * kAtom, x_kt = 6 * kAtom;
    static constexpr uint32_t atoms_tile = ak_atoms + TPC + 5, atoms_extra = 9;
    // partial readouts received by a tile CTA: one part per (source CTA,
    // receive slot) = R rows of bf16 laid out [DV/8][R] x 16 bytes (a warp's
    // store of one column group is contiguous per owner), then R fp32
    // denominators (extra CTA's part only)
    static constexpr uint32_t part_y = R * DV * 2;
    static constexpr uint32_t recv_part = part_y + round16(R * 4);
    static constexpr uint32_t recv_buf = CS * recv_part;
    static constexpr uint32_t recv_off = atoms_tile * kAtom;
    // the owned rows' intra-chunk part, staged by a bulk copy per chunk: R
    // rows of bf16, then R fp32 normalisers
    static constexpr uint32_t intra_slot = R * DV * 2 + round16(R * 4);
    // receive slots (chunks in flight, each with its intra-chunk stage):
    // three where they fit beside the static shared memory
    static constexpr uint32_t kStaticReserve = 1024 + 3072;
    static constexpr int RS = recv_off + 3 * (recv_buf + intra_slot) + kStaticReserve <= 232448 ? 3 : 2;
    static constexpr uint32_t intra_off = recv_off + RS * recv_buf;
    static constexpr uint32_t tile_end = intra_off + RS * intra_slot;
    static constexpr uint32_t total = tile_end > atoms_extra * kAtom ? tile_end : atoms_extra * kAtom;
    static constexpr size_t smem = total + 1024;
    // tensor memory columns, tile CTA
    static constexpr uint32_t tm_s = 0;                                // TPC x 64: fp32 state
    static constexpr uint32_t tm_ak = 64 * TPC;                        // AKT: 64, key lift (bf16 pairs of tokens)
    static constexpr uint32_t tm_aq = AKT ? 128 * TPC : 64 * TPC;      // 2 slots x TPC x 64: query lift
    static constexpr uint32_t tm_y = tm_aq + 128 * TPC;                // 2 slots x 64: partial readout
    // tensor memory columns, extra CTA
    static constexpr uint32_t tx_s = 0;      // tail state
    static constexpr uint32_t tx_aq = 64;    // 2 slots x 32: tail query lift
    static constexpr uint32_t tx_y = 128;    // 2 slots x 64: partial readout
    static constexpr uint32_t tx_ak = 256;   // 64: tail key lift (lanes past the tail hold zeros)
    static constexpr uint32_t tx_w = 384;    // Q Z
    static constexpr uint32_t tx_z = 448;    // Z
    static_assert(NT % TPC == 0, "tiles must split evenly");
    static_assert(tm_y + 128 <= 512, "tensor memory columns");
    static_assert(TAIL > 0 && TAIL <= 32, "tail tile");
    static_assert(total + kStaticReserve <= 232448, "shared memory");
    static_assert(R * NTC == kChunk, "owned rows");
    static_assert(kt_bytes <= kAtom, "transposed-key stage");
    static_assert((R * DV * 2) % 16 == 0 && (R * 4) % 16 == 0 && intra_off % 16 == 0, "bulk copy sizes");
};

// ---------------------------------------------------------------- key lift, one slot per thread
// The key lift of internal slot (i, j) for the 128 tokens of a chunk comes
// from the chunk's transposed unit keys `kts` (row d = dimension d over the
// tokens, two 64-token boxes of P rows, 128-byte swizzle): k_i k_j for the
// full lift, sum_a k_{aM+i} k_{aM+j} over the LG blocks of width M for
// KATA-Sigma-g.  Consecutive tokens sit side by side in both, so the 16
// bytes of tokens [64h + 8c, 64h + 8c + 8) are four bf16x2 multiplies of two
// 16-byte loads.
template <int P, int LG>
__device__ __forceinline__ uint4 key_words(const uint8_t* kts, int i, int j, int h, int c) {
    constexpr int M = P / LG;
    uint4 r;
#pragma unroll
    for (int blk = 0; blk < LG; ++blk) {
        const int bi = blk * M + i, bj = blk * M + j;  // rows of this block's two factors
        const uint4 a = *reinterpret_cast<const uint4*>(kts + h * (P * 128) + bi * 128 + ((c ^ (bi & 7)) << 4));
        const uint4 b = *reinterpret_cast<const uint4*>(kts + h * (P * 128) + bj * 128 + ((c ^ (bj & 7)) << 4));
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

// Row `row` of a K-major shared-memory operand tile (two 64-token atoms of
// 128 rows x 128 bytes, 128-byte swizzle) receives the key lift of slot
// `slot`; slots past n give zeros.
template <int P, int LG>
__device__ __forceinline__ void key_row_smem(const uint8_t* kts, int slot, uint8_t* ak, int row) {
    constexpr int n = lift::packed_n(P / LG);
    uint8_t* dst0 = ak + (row >> 3) * 1024 + (row & 7) * 128;
    const bool live = slot < n;
    int i = 0, j = 0;
    if (live) lift::slot_coord(P / LG, slot, i, j);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(dst0 + h * kAtom + ((c ^ (row & 7)) << 4)) =
                live ? key_words<P, LG>(kts, i, j, h, c) : make_uint4(0, 0, 0, 0);
}

// Lane `slot % 128` of a tensor-memory operand (64 columns, column c = the
// bf16 pair of tokens 2c, 2c+1) receives the key lift of slot `slot`, a
// quarter of the chunk (32 tokens) per tensor-memory store; slots past n
// give zeros.
template <int P, int LG>
__device__ __forceinline__ void key_row_tmem(const uint8_t* kts, int slot, uint32_t taddr) {
    constexpr int n = lift::packed_n(P / LG);
    const bool live = slot < n;
    int i = 0, j = 0;
    if (live) lift::slot_coord(P / LG, slot, i, j);
#pragma unroll
    for (int qt = 0; qt < 4; ++qt) {
        uint32_t w[16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const uint4 r = live ? key_words<P, LG>(kts, i, j, qt >> 1, (qt & 1) * 4 + cc) : make_uint4(0, 0, 0, 0);
            w[4 * cc] = r.x;
            w[4 * cc + 1] = r.y;
            w[4 * cc + 2] = r.z;
            w[4 * cc + 3] = r.w;
        }
        tmem_st16(taddr + 16 * qt, w);
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
//   warps 0-3   query:    thread t = token t of the chunk; reads its staged
//                         query row, writes the query lift (tensor memory,
//                         the A operand of the readout); then, one chunk
//                         behind, reads lane t of the partial readout and
//                         sends the row to the tile CTA that owns it
//   warps 4-7   state:    thread e = tensor-memory lane e; reads the state
//                         after each update and releases it to the next update,
//                         refreshes the bf16 copy for the next readout (extra
//                         CTA: also Z and the rows' inter-chunk denominators)
//   warps 8-11  key lift: thread e = slot e of each tile; multiplies two rows
//                         of the chunk's transposed unit keys into row e of
//                         the update's A operand (shared memory, K-major)
//   warps 12-15 warp 12 lane 0 issues every tcgen05.mma, warp 13 lane 0 the
//                         TMA loads; warps 14-15 reduce the owned rows, add
//                         the intra-chunk part and store the outputs
// Per chunk the MMAs run update tile by tile (state += lift(K)^T V; each
// tile's key-lift rows are released as soon as its MMAs are done, so the
// next chunk's lift of that tile overlaps the rest) and then the readout
// (Y = lift(Q) S) of the state before the chunk.
template <int P, int DV, int LG>
__global__ void __launch_bounds__(kThreads, 1)
chunked_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmkt,
                  const __grid_constant__ CUtensorMap tmv, __nv_bfloat16* __restrict__ o,
                  const __nv_bfloat16* __restrict__ y_intra, const float* __restrict__ d_intra,
                  const float* __restrict__ S_start, const float* __restrict__ z_start, int start_groups,
                  float* __restrict__ S_final, float* __restrict__ z_final, int T, int seg_chunks) {
    using K = Cfg<P, DV, LG>;
    constexpr int n = K::n, M = K::M;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t qs_full[2], qs_free[2], kts_full[2], kts_free[2], v_full[2], v_free[2];
    __shared__ uint64_t klift_full[2], ak_free[2], qlift_full[2], aq_free[2];
    __shared__ uint64_t y_part[2], y_free[2], den_ready[2];
    __shared__ uint64_t upd_done, state_read, s16_ready, drain, rd_sync;
    __shared__ uint64_t recv_full[K::RS], peer_free[K::RS];
    __shared__ uint64_t local_full[K::RS];  // this CTA's own partial rows written (one arrival per row)
    __shared__ uint64_t intra_full[K::RS];  // the owned rows' intra-chunk part staged
    __shared__ float dens[2][kChunk];       // extra CTA: inter-chunk denominators of the chunk rows
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
    const int nq = extra ? 2 : 1;  // query stages (the extra CTA's MMAs read the queries in place)
    uint8_t* const s_ak = sm + K::t_ak;  // tile CTA key lift, when it lives in shared memory
    uint8_t* const s_s16 = sm + (extra ? K::x_s16 : K::t_s16);
    uint8_t* const s_z16 = sm + K::x_z16;
    uint8_t* const s_recv = sm + K::recv_off;
    auto v_buf = [&](int kk) { return sm + (extra ? K::x_v : K::t_v) + (kk & 1) * kAtom; };
    auto q_buf = [&](int s) { return sm + (extra ? K::x_q : K::t_q) + s * kAtom; };
    auto kt_buf = [&](int s) { return sm + (extra ? K::x_kt : K::t_kt) + s * kAtom; };

    if (t == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&qs_full[b], 1);
            // the staged queries are read by the query warps and, in the extra
            // CTA, by the state warps (after the Q Z product that reads them too)
            mbar_init(&qs_free[b], extra ? 256 : 128);
            mbar_init(&kts_full[b], 1);
            // the staged keys are read by the key-lift warps and, in the extra
            // CTA, by the Z update (one commit)
            mbar_init(&kts_free[b], extra ? 129 : 128);
            mbar_init(&v_full[b], 1);
            mbar_init(&v_free[b], 1);
            mbar_init(&klift_full[b], 128);
            mbar_init(&ak_free[b], 1);
            mbar_init(&qlift_full[b], 128);
            mbar_init(&aq_free[b], 1);
            mbar_init(&y_part[b], 1);
            mbar_init(&y_free[b], 128);
            mbar_init(&den_ready[b], 128);
        }
        mbar_init(&upd_done, 1);
        mbar_init(&state_read, 128);
        mbar_init(&s16_ready, 128);
        mbar_init(&drain, 1);
        mbar_init(&rd_sync, 64);
        for (int b = 0; b < K::RS; ++b) {
            mbar_init(&recv_full[b], 1);
            mbar_init(&peer_free[b], K::NTC);  // one arrival per owner
            mbar_init(&local_full[b], my_rows > 0 ? my_rows : 1);
            mbar_init(&intra_full[b], 1);
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

    // ---- start state of this segment (state warps: lane = slot / dim)
    if (warp >= 4 && warp < 8) {
        const int e = t - 128;
        const int sg = start_groups > 1 ? g : 0;
        const float* S0 = S_start ? S_start + (bh * start_groups + sg) * (int64_t)n * DV : nullptr;
        const float* z0 = z_start ? z_start + (bh * start_groups + sg) * (int64_t)n : nullptr;
        if (!extra) {
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl)
                load_state_tile<M, DV>(S0, rank * K::TPC + tl, tm(K::tm_s + 64 * tl), s_s16 + tl * kAtom, e);
        } else {
            load_state_tile<M, DV>(S0, K::NT, tm(K::tx_s), s_s16, e);
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
                tmem_st16(tm(K::tx_z + c), r);
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
    // the extra CTA's tail key lift fills lanes [0, 32) of its operand; the
    // other lanes are read by the tail update's M = 128 MMAs into state rows
    // nothing reads, and are kept at zero
    if (extra && warp >= 9 && warp < 12) {
        uint32_t zw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) zw[i] = 0u;
#pragma unroll
        for (int c = 0; c < 64; c += 16) tmem_st16(tm(K::tx_ak + c), zw);
        tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    cluster.sync();  // barriers initialised and start state in place cluster-wide
    tc_fence_after();

    if (warp < 4) {
        // =============================================================== query warps
        regs_inc<kRegsLift>();
        const int e = t;
        const int owner = e / K::R, orow = e % K::R;
        // query lift of chunk kk into its tensor-memory slot (double-buffered:
        // overlaps the previous chunk's readout)
        auto lift_q = [&](int kk) -> bool {
            const int slot = kk & 1, use = kk >> 1;
            const int stg = kk % nq, stg_use = kk / nq;
            if (!wait(&qs_full[stg], stg_use & 1)) return false;
            const uint8_t* my_q = q_buf(stg) + t * 128;
            uint32_t uq[P / 2];
#pragma unroll
            for (int i = 0; i < P / 8; ++i) {
                const uint4 a = *reinterpret_cast<const uint4*>(my_q + ((i ^ (t & 7)) << 4));
                uq[4 * i] = a.x;
                uq[4 * i + 1] = a.y;
                uq[4 * i + 2] = a.z;
                uq[4 * i + 3] = a.w;
            }
            mbar_arrive(&qs_free[stg]);
            if (kk >= 2 && !wait(&aq_free[slot], (use - 1) & 1)) return false;
            tc_fence_after();
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
                    query_dispatch<P, LG>(rank * K::TPC + tl, uq, tm(K::tm_aq + 64 * K::TPC * slot + 64 * tl));
            } else {
                query_tail<P, LG>(uq, tm(K::tx_aq + 32 * slot));
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&qlift_full[slot]);
            return true;
        };
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
            {
                uint32_t r[DV / 16][16];  // all loads in flight, one wait
#pragma unroll
                for (int c = 0; c < DV / 16; ++c) tmem_ld16(tm(ycol + 16 * c), r[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < DV / 16; ++c)
#pragma unroll
                    for (int i = 0; i < 8; ++i) ypk[8 * c + i] = pack_bf16x2(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1]));
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
        for (int kk = 0; kk <= nk; ++kk) {
            if (kk < nk && !lift_q(kk)) { fail(); break; }
            if (kk >= 1 && !send(kk - 1)) { fail(); break; }
        }
    } else if (warp < 8) {
        // =============================================================== state warps
        regs_inc<kRegsState>();
        const int e = t - 128;
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            // state after this chunk's update
            if (!wait(&upd_done, kk & 1)) { fail(); break; }
            tc_fence_after();
            uint32_t sreg[K::TPC][DV / 2];  // bf16 pairs of this lane's state rows
            uint32_t zreg[M / 2];           // extra CTA: bf16 pairs of this lane's Z row
            const int ntl = extra ? 1 : K::TPC;
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl) {
                if (tl >= ntl) break;
                const uint32_t scol = extra ? K::tx_s : K::tm_s + 64 * tl;
#pragma unroll
                for (int c32 = 0; c32 < DV; c32 += 32) {
                    uint32_t r[2][16];  // two loads in flight per wait
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (c32 + 16 * h < DV) tmem_ld16(tm(scol + c32 + 16 * h), r[h]);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (c32 + 16 * h < DV)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                sreg[tl][(c32 + 16 * h) / 2 + i] =
                                    pack_bf16x2(__uint_as_float(r[h][2 * i]), __uint_as_float(r[h][2 * i + 1]));
                }
            }
            if (extra) {
#pragma unroll
                for (int c16 = 0; c16 < M; c16 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tx_z + c16), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        zreg[c16 / 2 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                }
            }
            tc_fence_before();
            mbar_arrive(&state_read);
            // this chunk's readout is done: its bf16 state copy may be replaced
            if (!wait(&y_part[slot], use & 1)) { fail(); break; }
            tc_fence_after();
            float den = 0.f;
            if (extra) {
                // inter-chunk denominator q^T Z q from W = Q Z (Z before this chunk)
                uint4 qrow[P / 8];
                const uint8_t* sq = q_buf(kk % nq);  // this chunk's staged queries
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
                den = dint;
                tc_fence_before();
                mbar_arrive(&qs_free[kk % nq]);  // this chunk's staged queries and W have been read
            }
            auto write_s16 = [&](const uint32_t (&x)[DV / 2], int tl) {
#pragma unroll
                for (int c8 = 0; c8 < DV / 8; ++c8)
                    *reinterpret_cast<uint4*>(s_s16 + tl * kAtom + mn_sw128_chunk(8 * c8, e, kAtom)) =
                        make_uint4(x[4 * c8], x[4 * c8 + 1], x[4 * c8 + 2], x[4 * c8 + 3]);
            };
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl)
                if (tl < ntl) write_s16(sreg[tl], tl);
            if (extra && e < M) {
#pragma unroll
                for (int c8 = 0; c8 < M / 8; ++c8)
                    *reinterpret_cast<uint4*>(s_z16 + sw128_chunk(e, 8 * c8, M)) =
                        make_uint4(zreg[4 * c8], zreg[4 * c8 + 1], zreg[4 * c8 + 2], zreg[4 * c8 + 3]);
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
                    store_state_tile<M, DV>(S_final + head_s, rank * K::TPC + tl, tm(K::tm_s + 64 * tl), e);
            } else {
                store_state_tile<M, DV>(S_final + head_s, K::NT, tm(K::tx_s), e);
                uint32_t zr[M];
#pragma unroll
                for (int c16 = 0; c16 < M; c16 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tm(K::tx_z + c16), r);
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
        for (int kk = 0; kk < nk; ++kk) {
            const int stg = kk & 1, use = kk >> 1;
            if (!wait(&kts_full[stg], use & 1)) { fail(); break; }
            const uint8_t* kts = kt_buf(stg);
            bool ok = true;
            const int ntl = extra ? 1 : K::TPC;
#pragma unroll
            for (int tl = 0; tl < K::TPC; ++tl) {
                if (tl >= ntl) break;
                if (kk >= 1 && !wait(&ak_free[tl], (kk - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (extra) {
                    if (warp == 8) key_row_tmem<P, LG>(kts, K::NT * 128 + e, tm(K::tx_ak));
                } else if constexpr (K::AKT) {
                    key_row_tmem<P, LG>(kts, (rank * K::TPC + tl) * 128 + e, tm(K::tm_ak + 64 * tl));
                } else {
                    key_row_smem<P, LG>(kts, (rank * K::TPC + tl) * 128 + e, s_ak + 2 * tl * kAtom, e);
                }
                fence_proxy_async_smem();
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&klift_full[tl]);
            }
            if (!ok) { fail(); break; }
            mbar_arrive(&kts_free[stg]);
        }
    } else {
        regs_dec<kRegsMma>();
    }
    if (warp >= 14 && my_rows > 0) {
        // =============================================================== reduce warps
        // owner side, chunk by chunk as the partial rows land: sum them and
        // the intra-chunk rows (staged by a bulk copy RS chunks ahead), hand
        // the receive slot back to every sender (its next use is RS chunks
        // later), then divide and store the outputs
        constexpr int kRedIt = (K::R * (DV / 8) + 63) / 64;
        constexpr uint32_t kIntraY = K::R * DV * 2, kIntraBytes = kIntraY + K::R * 4;
        const int er = t - 448;
        const int r0 = rank * K::R;
        const int items = my_rows * (DV / 8);
        const int64_t head_row = bh * (int64_t)T;                // output rows
        const int64_t head_prow = bh * (int64_t)NCH * kChunk;    // intra-chunk rows: whole chunks per head
        uint8_t* const s_intra = sm + K::intra_off;
        int staged = 0, consumed = 0;  // bulk copies issued / waited for
        auto stage_intra = [&](int kr) {
            ++staged;
            const int r = kr % K::RS;
            const int64_t row = head_prow + (int64_t)(c0 + kr) * kChunk + r0;
            uint8_t* dst = s_intra + r * K::intra_slot;
            mbar_arrive_expect_tx(&intra_full[r], kIntraBytes);
            bulk_load(dst, y_intra + row * DV, kIntraY, &intra_full[r]);
            bulk_load(dst + kIntraY, d_intra + row, K::R * 4, &intra_full[r]);
        };
        if (er == 0)
            for (int kr = 0; kr < K::RS && kr < nk; ++kr) stage_intra(kr);
        for (int kr = 0; kr < nk; ++kr) {
            const int r = kr % K::RS;
            const uint32_t par = (kr / K::RS) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(&recv_full[r], par, &abort_flag, kWaitNs) &&
                                             mbar_wait(&local_full[r], par, &abort_flag, kWaitNs) &&
                                             mbar_wait(&intra_full[r], par, &abort_flag, kWaitNs))) {
                fail();
                break;
            }
            consumed = kr + 1;
            const uint8_t* recv = s_recv + r * K::recv_buf;
            const uint8_t* sin = s_intra + r * K::intra_slot;
            float acc[kRedIt][8], den[kRedIt];
#pragma unroll
            for (int it = 0; it < kRedIt; ++it) {
                const int idx = er + 64 * it;
                const int lr = idx % my_rows, i = idx / my_rows;
                if (idx >= items) continue;
                const uint4 yin = *reinterpret_cast<const uint4*>(sin + lr * (DV * 2) + i * 16);
                const __nv_bfloat162* hy = reinterpret_cast<const __nv_bfloat162*>(&yin);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[it][2 * j] = __low2float(hy[j]);
                    acc[it][2 * j + 1] = __high2float(hy[j]);
                }
                den[it] = *reinterpret_cast<const float*>(sin + kIntraY + lr * 4);
#pragma unroll
                for (int src = 0; src < K::CS; ++src) {
                    const uint4 x = *reinterpret_cast<const uint4*>(recv + src * K::recv_part + (i * K::R + lr) * 16);
                    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[it][2 * j] += __low2float(h[j]);
                        acc[it][2 * j + 1] += __high2float(h[j]);
                    }
                }
                den[it] += *reinterpret_cast<const float*>(recv + K::NTC * K::recv_part + K::part_y + lr * 4);
            }
            // every reader of slot r is past its last read once rd_sync completes
            mbar_arrive(&rd_sync);
            if (!__all_sync(0xffffffffu, mbar_wait(&rd_sync, kr & 1, &abort_flag, kWaitNs))) {
                fail();
                break;
            }
            if (er == 0 && kr + K::RS < nk) {
                mbar_arrive_expect_tx(&recv_full[r], rx_bytes);
                fence_proxy_async_smem();
                stage_intra(kr + K::RS);
            }
            if (er < K::CS) mbar_arrive_remote_relaxed(cluster_addr(&peer_free[r], er));
#pragma unroll
            for (int it = 0; it < kRedIt; ++it) {
                const int idx = er + 64 * it;
                const int lr = idx % my_rows, i = idx / my_rows;
                const int otok = (c0 + kr) * kChunk + r0 + lr;
                if (idx < items && otok < T) {
                    const float inv = den[it] > 0.f ? 1.f / den[it] : 0.f;
                    const float* a = acc[it];
                    *reinterpret_cast<uint4*>(o + (head_row + otok) * DV + 8 * i) =
                        make_uint4(pack_bf16x2(a[0] * inv, a[1] * inv), pack_bf16x2(a[2] * inv, a[3] * inv),
                                   pack_bf16x2(a[4] * inv, a[5] * inv), pack_bf16x2(a[6] * inv, a[7] * inv));
                }
            }
        }
        // no bulk copy may still be landing in shared memory when the CTA exits
        if (er == 0)
            for (int kr = consumed; kr < staged; ++kr) mbar_wait_quiet(&intra_full[kr % K::RS], (kr / K::RS) & 1, kWaitNs);
    }
    if (t == 416) {
        // =============================================================== TMA producer
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmkt);
        tma_prefetch_desc(&tmv);
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            const int stg = kk % nq, stg_use = kk / nq;
            const int row = (c0 + kk) * kChunk;
            // transposed unit keys of chunk kk into its stage
            if (kk >= 2 && !mbar_wait(&kts_free[slot], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&kts_full[slot], K::kt_bytes);
            tma_load_3d(kt_buf(slot), &tmkt, 0, (c0 + kk) * P, (int)bh, &kts_full[slot]);
            tma_load_3d(kt_buf(slot) + K::kt_box, &tmkt, 64, (c0 + kk) * P, (int)bh, &kts_full[slot]);
            // value tile of chunk kk into its buffer
            if (kk >= 2 && !mbar_wait(&v_free[slot], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&v_full[slot], kAtom);
            tma_load_3d(v_buf(kk), &tmv, 0, row, (int)bh, &v_full[slot]);
            // query rows of chunk kk into its stage
            if (kk >= nq && !mbar_wait(&qs_free[stg], (stg_use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&qs_full[stg], kAtom);
            tma_load_3d(q_buf(stg), &tmq, 0, row, (int)bh, &qs_full[stg]);
        }
    }
    if (warp == 12) {
        // =============================================================== MMA issuer
        // The whole warp runs the issue loop (waits, descriptors) and one
        // elected lane issues each instruction: the operands stay warp-uniform,
        // which keeps the issue of back-to-back MMAs as cheap as a loop of
        // constants (a single lane in a divergent branch issues them at about
        // two thirds of that rate).  Every descriptor is built once; the loop
        // adds compile-time offsets (a step moves the start-address field, in
        // 16-byte units).
        constexpr uint32_t id_read = idesc_bf16_f32_major(128, DV, false, true);
        constexpr uint32_t id_upd = idesc_bf16_f32_major(128, DV, false, true);
        constexpr uint32_t id_z = idesc_bf16_f32(128, M);
        constexpr uint32_t id_w = idesc_bf16_f32(128, M);
        constexpr uint64_t kStepMN = 2048 >> 4, kStepK = 32 >> 4, kAtomD = kAtom >> 4, kBoxD = K::kt_box >> 4;
        // K step ks of a K-major operand whose 64-element K atoms are `atom` (16-byte units) apart
        auto kstep = [](uint64_t atom, int ks) { return (uint64_t)(ks >> 2) * atom + (uint64_t)(ks & 3) * kStepK; };
        const uint64_t d_ak = sdesc_kmajor_sw128(smem_u32(s_ak));
        const uint64_t d_s16 = sdesc_mnmajor_sw128(smem_u32(s_s16), kAtom);
        const uint64_t d_v[2] = {sdesc_mnmajor_sw128(smem_u32(v_buf(0)), kAtom),
                                 sdesc_mnmajor_sw128(smem_u32(v_buf(1)), kAtom)};
        // extra CTA: staged transposed keys (both operands of the Z update), staged Q, Z
        const uint64_t d_kt[2] = {sdesc_kmajor_sw128(smem_u32(kt_buf(0))), sdesc_kmajor_sw128(smem_u32(kt_buf(1)))};
        const uint64_t d_q[2] = {sdesc_kmajor_sw128(smem_u32(q_buf(0))), sdesc_kmajor_sw128(smem_u32(q_buf(extra ? 1 : 0)))};
        const uint64_t d_z16 = sdesc_kmajor_sw128(smem_u32(s_z16));
        for (int kk = 0; kk < nk; ++kk) {
            const int slot = kk & 1, use = kk >> 1;
            if (!wait(&v_full[slot], use & 1)) { fail(); break; }
            const uint64_t dv = d_v[slot];
            // ---- group U: state updates, tile by tile (extra CTA: tail state and Z)
            bool ok = true;
            if (!extra) {
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl) {
                    if (!wait(&klift_full[tl], kk & 1)) { ok = false; break; }
                    if (tl == 0 && kk >= 1 && !wait(&state_read, (kk - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        if constexpr (K::AKT)
                            mma_ts_w(tb + K::tm_s + 64 * tl, tb + K::tm_ak + 64 * tl + 8 * ks, dv + ks * kStepMN, id_upd, 1u);
                        else
                            mma_ss_w(tb + K::tm_s + 64 * tl, d_ak + 2 * tl * kAtomD + kstep(kAtomD, ks), dv + ks * kStepMN,
                                     id_upd, 1u);
                    }
                    mma_commit_w(&ak_free[tl]);
                }
                if (!ok) { fail(); break; }
                mma_commit_w(&upd_done);
                mma_commit_w(&v_free[slot]);
            } else {
                if (!wait(&klift_full[0], kk & 1) ||
                    !wait(&kts_full[slot], use & 1) ||
                    (kk >= 1 && !wait(&state_read, (kk - 1) & 1))) { fail(); break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) mma_ts_w(tb + K::tx_s, tb + K::tx_ak + 8 * ks, dv + ks * kStepMN, id_upd, 1u);
                // Z += sum over the blocks of (rows of the block)^T (rows of the block)
#pragma unroll
                for (int blk = 0; blk < LG; ++blk)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss_w(tb + K::tx_z, d_kt[slot] + (uint64_t)(blk * M * 8) + kstep(kBoxD, ks),
                               d_kt[slot] + (uint64_t)(blk * M * 8) + kstep(kBoxD, ks), id_z, 1u);
                mma_commit_w(&ak_free[0]);
                mma_commit_w(&upd_done);
                mma_commit_w(&v_free[slot]);
                mma_commit_w(&kts_free[slot]);
            }
            // ---- group R: readout of the state before this chunk
            if (!wait(&qlift_full[slot], use & 1)) { fail(); break; }
            if (kk >= 1 && !wait(&s16_ready, (kk - 1) & 1)) { fail(); break; }
            if (kk >= 2 && !wait(&y_free[slot], (use - 1) & 1)) { fail(); break; }
            if (extra && !wait(&qs_full[kk % nq], (kk / nq) & 1)) { fail(); break; }
            tc_fence_after();
            if (!extra) {
                const uint32_t dy = tb + K::tm_y + 64 * slot, aq = tb + K::tm_aq + 64 * K::TPC * slot;
#pragma unroll
                for (int tl = 0; tl < K::TPC; ++tl)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts_w(dy, aq + 64 * tl + 8 * ks, d_s16 + tl * kAtomD + ks * kStepMN, id_read,
                               (tl > 0 || ks > 0) ? 1u : 0u);
            } else {
                const uint32_t dy = tb + K::tx_y + 64 * slot, aq = tb + K::tx_aq + 32 * slot;
#pragma unroll
                for (int ks = 0; ks < (K::TAIL + 15) / 16; ++ks)
                    mma_ts_w(dy, aq + 8 * ks, d_s16 + ks * kStepMN, id_read, ks > 0 ? 1u : 0u);
                // W = [Q_0 Z | Q_1 Z | ...], one block of columns per block of the queries
#pragma unroll
                for (int blk = 0; blk < LG; ++blk)
#pragma unroll
                    for (int ks = 0; ks < M / 16; ++ks)
                        mma_ss_w(tb + K::tx_w + blk * M, d_q[kk % nq] + (blk * (M / 16) + ks) * kStepK,
                               d_z16 + ks * kStepK, id_w, ks > 0 ? 1u : 0u);
            }
            mma_commit_w(&y_part[slot]);
            mma_commit_w(&aq_free[slot]);
        }
        // every issued MMA has completed before tensor memory is released
        mma_commit_w(&drain);
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
// Y goes out as bf16 rows [BH][Tc][DV] and d, the rows' intra-chunk
// normaliser, as fp32 [BH][Tc] (Tc = T rounded up to whole chunks; rows past
// T are not written); the fused forward adds both when it writes a chunk's
// outputs.  The chunk's unit keys also go out transposed, kT
// [BH][chunks][P][128] bf16 (zeros past T): the fused forward's key lift
// reads them.  d sums exactly the rounded weights Y is built from, which
// keeps the intra-chunk weights a convex combination.  One CTA per (chunk,
// head), 128 columns of tensor memory and 48 KB of shared memory, so several
// chunks are in flight per SM; thread t owns query / key / value row t.
template <int P, int DV, int LG>
__global__ void __launch_bounds__(128)
intra_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                const __nv_bfloat16* __restrict__ v, __nv_bfloat16* __restrict__ y_out, float* __restrict__ d_out,
                __nv_bfloat16* __restrict__ kt_out, int T) {
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
    // y and d rows: T rounded up to whole chunks per head
    const int64_t prow = bh * (int64_t)(gridDim.x * kChunk) + row;
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
            // dimensions 8i .. 8i+7 of this token into the transposed keys
            const __nv_bfloat16* we = reinterpret_cast<const __nv_bfloat16*>(&w);
            __nv_bfloat16* kt = kt_out + ((bh * gridDim.x + blockIdx.x) * P + 8 * i) * kChunk + t;
#pragma unroll
            for (int j = 0; j < 8; ++j) kt[j * kChunk] = we[j];
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
        uint32_t y[DV];
#pragma unroll
        for (int c = 0; c < DV; c += 16) tmem_ld16(tmem_addr(tb, lane0, 64 + c), *reinterpret_cast<uint32_t(*)[16]>(y + c));
        tmem_wait_ld();
        if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(y_out + prow * DV);
#pragma unroll
            for (int i = 0; i < DV / 8; ++i)
                dst[i] = make_uint4(pack_bf16x2(__uint_as_float(y[8 * i]), __uint_as_float(y[8 * i + 1])),
                                    pack_bf16x2(__uint_as_float(y[8 * i + 2]), __uint_as_float(y[8 * i + 3])),
                                    pack_bf16x2(__uint_as_float(y[8 * i + 4]), __uint_as_float(y[8 * i + 5])),
                                    pack_bf16x2(__uint_as_float(y[8 * i + 6]), __uint_as_float(y[8 * i + 7])));
            d_out[prow] = den;
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

// ---------------------------------------------------------------- host side
// The register split of the kernel fits in its launch allocation.
template <int P, int DV, int LG>
bool register_split_fits() {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, chunked_tc_kernel<P, DV, LG>) != cudaSuccess) return false;
    return (uint32_t)kThreads * (uint32_t)fa.numRegs >= 128u * (kRegsLift + kRegsState + kRegsLaunch + kRegsMma);
}

template <int P, int DV, int LG>
cudaError_t configure(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int G, int BH, cudaStream_t s) {
    using K = Cfg<P, DV, LG>;
    auto kern = chunked_tc_kernel<P, DV, LG>;
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

template <int P, int DV, int LG>
int max_clusters() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[1];
        int m = 0;
        if (!register_split_fits<P, DV, LG>() || configure<P, DV, LG>(cfg, attr, 1, 1, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&m, chunked_tc_kernel<P, DV, LG>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cached[dev] = m > 0 ? m : -1;
    }
    return cached[dev] > 0 ? cached[dev] : 0;
}

// Workspace of the forward's intra-chunk kernel: bf16 rows [BH][T][dv],
// fp32 normalisers [BH][T], transposed unit keys [BH][chunks][p][128] bf16.
struct IntraWs {
    size_t y_off, d_off, kt_off, total;
};
IntraWs intra_ws(int BH, int T, int p, int dv) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t nch = (size_t)(T + kChunk - 1) / kChunk;
    IntraWs w;
    w.y_off = 0;
    w.d_off = up((size_t)BH * nch * kChunk * dv * 2);
    w.kt_off = w.d_off + up((size_t)BH * nch * kChunk * 4);
    w.total = w.kt_off + up((size_t)BH * nch * p * kChunk * 2);
    return w;
}

template <int P, int DV, int LG>
cudaError_t launch_typed(const void* q, const void* k, const void* v, void* o, void* intra,
                         const float* S_start, const float* z_start, int start_groups, float* S_final,
                         float* z_final, int BH, int T, int seg_chunks, int G, cudaStream_t s) {
    if (!register_split_fits<P, DV, LG>()) return cudaErrorInvalidConfiguration;
    const IntraWs w = intra_ws(BH, T, P, DV);
    auto* y_intra = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(intra) + w.y_off);
    auto* d_intra = reinterpret_cast<float*>(static_cast<char*>(intra) + w.d_off);
    auto* kt = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(intra) + w.kt_off);
    const int nch = (T + kChunk - 1) / kChunk;
    // the intra-chunk rows and the transposed unit keys of every chunk first
    constexpr size_t intra_smem = 3 * kAtom + 1024;
    cudaError_t e = cudaFuncSetAttribute(intra_tc_kernel<P, DV, LG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)intra_smem);
    if (e != cudaSuccess) return e;
    KATA_TRACED("intra_tc", s,
                (intra_tc_kernel<P, DV, LG><<<dim3((unsigned)nch, (unsigned)BH), 128, intra_smem, s>>>(
                    static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                    static_cast<const __nv_bfloat16*>(v), y_intra, d_intra, kt, T)));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    if ((e = configure<P, DV, LG>(cfg, attr, G, BH, s)) != cudaSuccess) return e;
    CUtensorMap tq, tkt, tv;
    if (!rows_map(&tq, q, P, T, BH) || !kt_map(&tkt, kt, P, nch, BH) || !rows_map(&tv, v, DV, T, BH))
        return cudaErrorInvalidValue;
    KATA_TRACED("chunked_tc", s,
                e = cudaLaunchKernelEx(&cfg, chunked_tc_kernel<P, DV, LG>, tq, tkt, tv, static_cast<__nv_bfloat16*>(o),
                                       static_cast<const __nv_bfloat16*>(y_intra), static_cast<const float*>(d_intra),
                                       S_start, z_start, start_groups, S_final, z_final, T, seg_chunks));
    if (e != cudaSuccess) return e;
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
    int m = 0;
    KATA_DISPATCH(m = max_clusters<P, DV, LG>());
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

size_t chunked_tc_intra_bytes(int BH, int T, int p, int dv) { return intra_ws(BH, T, p, dv).total; }

cudaError_t launch_chunked_tc(const void* q, const void* k, const void* v, void* o, void* intra,
                              const float* S_start, const float* z_start, int start_groups, float* S_final,
                              float* z_final, int BH, int T, int p, int dv, int lg, int G, cudaStream_t s) {
    const int seg_chunks = chunked_tc_segment_chunks(T, G);
    KATA_DISPATCH(return launch_typed<P, DV, LG>(q, k, v, o, intra, S_start, z_start, start_groups, S_final, z_final, BH, T,
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
