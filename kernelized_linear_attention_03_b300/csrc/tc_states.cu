// Segment states on the tcgen05 tensor cores (bf16 inputs, fp32 accumulate):
// for each head and each segment of L consecutive tokens,
//   S_seg = sum_{t in seg} psi(kh_t) v_t^T,   z_seg = sum_{t in seg} psi(kh_t)
// (the state S_t = Psi(K_{1:t})^T V_{1:t} of the state-size paragraph
// restricted to one segment; with L = C these are the local chunk states of
// the chunked-scan paragraph's state kernel).
//
// One CTA owns one 128-slot tile of the packed lift for a run of segments
// of one head; blocks of up to 128 tokens stream through a pipeline
// (384 threads):
//   warp 0 lane 0   TMA: key and value rows of each block into a ring of
//                   kStages stages
//   warp 1 lane 0   issues D[slots x 80] += psiK(K)^T [V | 1] per block (K =
//                   tokens; B = the value tile and a constant ones atom), two
//                   accumulators in tensor memory alternating by segment
//   warps 4-7       thread = token: unit key, the tile's lifted coordinates
//                   into a token-major (MN-major for the MMA) swizzled tile,
//                   double-buffered
//   warps 8-11      at each segment end, thread = slot: the accumulator row
//                   out in the C ABI's sqrt(2)-packed order
#include <cuda_bf16.h>

#include <cstdint>

#include "kata_internal.h"
#include "tc_lift.cuh"
#include "tc_primitives.cuh"
#include "tc_tma.cuh"

namespace kata {
namespace {

using namespace tc;

__device__ unsigned int g_states_tc_status = 0;

constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr float kSqrt2f = 1.41421356237309504880f;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kAtom = 128 * 128;  // one MN atom: 128 K-rows (tokens) x 128 bytes
constexpr uint32_t kNB = 80;           // B columns: 64 value slots, the ones column, pad
// shared memory from a 1024-byte aligned base: A[2] (two 64-slot atoms
// each), K[kStages], V[kStages], the ones atom (last: every value stage
// reaches it with a positive atom stride), then the output staging (128
// rows of 64 fp32, each row padded by 16 bytes)
constexpr uint32_t kAOff = 0, kKOff = 4 * kAtom, kVOff = (4 + kStages) * kAtom,
                   kOnesOff = (4 + 2 * kStages) * kAtom, kOutOff = (5 + 2 * kStages) * kAtom;
constexpr uint32_t kOutRow = 64 * 4 + 16;
constexpr size_t kSmem = kOutOff + 128 * kOutRow + 1024;

// Key lift word w (slots 2w, 2w+1) of the lift of width M = P / LG: the full
// lift (LG = 1) or KATA-Sigma-g, the sum of the LG block lifts (products
// accumulated by bf16x2 multiply-adds in block order, as the fused forward's
// key lift does).
template <int P, int LG>
__device__ __forceinline__ uint32_t key_word(const uint32_t (&u)[P / 2], int w) {
    constexpr int M = P / LG;
    if constexpr (LG == 1) {
        return lift::lift_word<M, false>(u, w);
    } else {
        constexpr int n = lift::packed_n(M);
        const int s0 = 2 * w, s1 = 2 * w + 1;
        if (s0 >= n) return 0u;
        int i0 = 0, j0 = 0, i1 = 0, j1 = 0;
        lift::slot_coord(M, s0, i0, j0);
        if (s1 < n) {
            lift::slot_coord(M, s1, i1, j1);
        } else {
            i1 = i0;
            j1 = j0;
        }
        uint32_t r = 0u;
#pragma unroll
        for (int blk = 0; blk < LG; ++blk) {
            const uint32_t* ub = u + blk * (M / 2);
            const uint32_t x = lift::u_pair(ub, i0, i1), y = lift::u_pair(ub, j0, j1);
            r = blk == 0 ? hmul2_bf16(x, y) : hfma2_bf16(x, y, r);
        }
        return s1 < n ? r : (r & 0xFFFFu);
    }
}

// Lifted key coordinates of tile TAU for this thread's token into row `row`
// of the token-major A tile.
// SCALE: every word times the bf16 pair dd (a per-token weight of the lift).
template <int P, int LG, int TAU, bool SCALE>
__device__ __forceinline__ void key_tile_to_smem(const uint32_t (&u)[P / 2], uint8_t* As, int row, uint32_t dd) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint4 val;
        val.x = key_word<P, LG>(u, 64 * TAU + 4 * c + 0);
        val.y = key_word<P, LG>(u, 64 * TAU + 4 * c + 1);
        val.z = key_word<P, LG>(u, 64 * TAU + 4 * c + 2);
        val.w = key_word<P, LG>(u, 64 * TAU + 4 * c + 3);
        if (SCALE) {
            val.x = hmul2_bf16(val.x, dd);
            val.y = hmul2_bf16(val.y, dd);
            val.z = hmul2_bf16(val.z, dd);
            val.w = hmul2_bf16(val.w, dd);
        }
        *reinterpret_cast<uint4*>(As + mn_sw128_chunk(8 * c, row, kAtom)) = val;
    }
}

template <int P, int LG, bool SCALE, int TAU = 0>
__device__ __forceinline__ void key_tile_dispatch(int tau, const uint32_t (&u)[P / 2], uint8_t* As, int row,
                                                  uint32_t dd) {
    if constexpr (TAU < lift::tiles_of(P / LG)) {
        if (tau == TAU)
            key_tile_to_smem<P, LG, TAU, SCALE>(u, As, row, dd);
        else
            key_tile_dispatch<P, LG, SCALE, TAU + 1>(tau, u, As, row, dd);
    }
}

template <int P, int DV, int LG>
__global__ void __launch_bounds__(kThreads, 1)
states_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 float* __restrict__ S_out, float* __restrict__ z_out, int T, int L, int NS, int NS_out,
                 int segs_per_cta, int prefix, const float* __restrict__ dec) {
    // dec (or null; full lift only): a weight per token, the key lift of token
    // t taken times dec[bh][t] (the gated form's decay to its chunk's end)
    // prefix != 0 (one CTA per tile and head, all segments): each segment's
    // row is the exclusive running sum of the segments before it, summed in
    // segment order in the epilogue's registers, instead of the segment's own total
    // T: tokens per head; segments 0..NS-1 of L tokens (L a multiple of 128,
    // or L <= 128) are computed into rows of a [BH, NS_out, n] layout.
    constexpr int M = P / LG;  // width of the lifted blocks (P for the full lift)
    constexpr int n = lift::packed_n(M);
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t k_full[kStages], v_full[kStages], kv_free[kStages], a_full[2], a_free[2];
    __shared__ uint64_t acc_full[2], acc_free[2], drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int t = threadIdx.x, warp = t >> 5;
    const int tau = blockIdx.x;
    const int64_t bh = blockIdx.z;
    const int seg0 = blockIdx.y * segs_per_cta;
    const int seg1 = min(NS, seg0 + segs_per_cta);
    const int bl = L < 128 ? L : 128;  // tokens per block
    const int tok0 = seg0 * L, tok1 = min(T, seg1 * L);
    const int nblk = tok1 > tok0 ? (tok1 - tok0 + bl - 1) / bl : 0;
    // block i: tokens [b0, b1) of segment seg
    auto block = [&](int i, int& b0, int& b1, int& seg) {
        b0 = tok0 + i * bl;
        seg = b0 / L;
        b1 = min(min(T, (seg + 1) * L), b0 + bl);
    };

    if (t == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&k_full[st], 1);
            mbar_init(&v_full[st], 1);
            mbar_init(&kv_free[st], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&a_full[b], 128);
            mbar_init(&a_free[b], 1);
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_free[b], 128);
        }
        mbar_init(&drain, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    for (int r = t; r < 128; r += kThreads)
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sm + kOnesOff + mn_sw128_chunk(8 * c, r, kAtom)) =
                make_uint4(c == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    auto fail = [&]() {
        abort_flag = 1;
        atomicOr(&g_states_tc_status, kStatusTimeout);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, &abort_flag, kWaitNs));
    };

    if (t == 0) {
        // =============================================================== TMA producer
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        int issued = 0;
        for (int i = 0; i < nblk; ++i) {
            const int st = i % kStages, use = i / kStages;
            int b0, b1, seg;
            block(i, b0, b1, seg);
            if (i >= kStages && !mbar_wait(&kv_free[st], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&k_full[st], kAtom);
            tma_load_3d(sm + kKOff + st * kAtom, &tmk, 0, b0, (int)bh, &k_full[st]);
            mbar_arrive_expect_tx(&v_full[st], kAtom);
            tma_load_3d(sm + kVOff + st * kAtom, &tmv, 0, b0, (int)bh, &v_full[st]);
            issued = i + 1;
        }
        // no copy may still be landing in shared memory when the CTA exits
        for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
            mbar_wait_quiet(&k_full[i % kStages], (i / kStages) & 1, kWaitNs);
            mbar_wait_quiet(&v_full[i % kStages], (i / kStages) & 1, kWaitNs);
        }
    } else if (warp == 1) {
        // =============================================================== MMA issuer
        // (the whole warp runs the loop; one elected lane issues each instruction)
        constexpr uint32_t idesc = idesc_bf16_f32_major(128, kNB, true, true);
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            const int st = i % kStages, ab = i & 1;
            int b0, b1, seg;
            block(i, b0, b1, seg);
            const int sl = seg - seg0, acb = sl & 1;
            const bool first = b0 == seg * L, last = b1 == min(T, (seg + 1) * L);
            if (!wait(&a_full[ab], (i >> 1) & 1) ||
                !wait(&v_full[st], (i / kStages) & 1) ||
                (first && sl >= 2 && !wait(&acc_free[acb], ((sl - 2) >> 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t d_a = sdesc_mnmajor_sw128(smem_u32(sm + kAOff + 2 * ab * kAtom), kAtom);
            const uint64_t d_b = sdesc_mnmajor_sw128(smem_u32(sm + kVOff + st * kAtom),
                                                     (uint32_t)(kOnesOff - (kVOff + st * kAtom)));
            const int steps = (b1 - b0 + 15) / 16;
            for (int ks = 0; ks < steps; ++ks)
                mma_ss_w(tb + 128 * acb, d_a + ks * (2048 >> 4), d_b + ks * (2048 >> 4), idesc,
                       (first && ks == 0) ? 0u : 1u);
            mma_commit_w(&a_free[ab]);
            mma_commit_w(&kv_free[st]);
            if (last) mma_commit_w(&acc_full[acb]);
        }
        if (!ok) fail();
        mma_commit_w(&drain);
        mbar_wait_quiet(&drain, 0, kWaitNs);
    } else if (warp >= 4 && warp < 8) {
        // =============================================================== lift warps
        const int lt = t - 128;
        for (int i = 0; i < nblk; ++i) {
            const int st = i % kStages, ab = i & 1;
            int b0, b1, seg;
            block(i, b0, b1, seg);
            const bool valid = b0 + lt < b1;
            if (!wait(&k_full[st], (i / kStages) & 1)) { fail(); break; }
            if (i >= 2 && !wait(&a_free[ab], ((i - 2) >> 1) & 1)) { fail(); break; }
            const uint8_t* kb = sm + kKOff + st * kAtom;
            uint32_t u[P / 2];
            {
                uint4 raw[P / 8];
                float ss = 0.f;
#pragma unroll
                for (int c = 0; c < P / 8; ++c) {
                    raw[c] = valid ? *reinterpret_cast<const uint4*>(kb + sw128_chunk(lt, 8 * c, 128)) : make_uint4(0, 0, 0, 0);
                    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[c]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float x = __bfloat162float(e[j]);
                        ss = fmaf(x, x, ss);
                    }
                }
                const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
                for (int c = 0; c < P / 8; ++c) {
                    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[c]);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        u[4 * c + j] = pack_bf16x2(__bfloat162float(e[2 * j]) * inv, __bfloat162float(e[2 * j + 1]) * inv);
                }
            }
            if constexpr (LG == 1) {
                if (dec != nullptr) {
                    const float w = valid ? dec[bh * (int64_t)T + b0 + lt] : 0.f;
                    key_tile_dispatch<P, LG, true>(tau, u, sm + kAOff + 2 * ab * kAtom, lt, pack_bf16x2(w, w));
                } else {
                    key_tile_dispatch<P, LG, false>(tau, u, sm + kAOff + 2 * ab * kAtom, lt, 0u);
                }
            } else {
                key_tile_dispatch<P, LG, false>(tau, u, sm + kAOff + 2 * ab * kAtom, lt, 0u);
            }
            fence_proxy_async_smem();
            mbar_arrive(&a_full[ab]);
        }
    } else if (warp >= 8) {
        // =============================================================== epilogue warps
        // thread e reads accumulator row e (slot tau*128 + e); the rows go out
        // through shared memory so that each canonical row (DV contiguous
        // floats) is written by one warp store
        const int e = t - 256, ew = e >> 5, lane = e & 31;
        const uint32_t lane0 = (uint32_t)((warp & 3) * 32);
        const int slot = tau * 128 + e;
        int ci = 0, cj = 0;
        if (slot < n) lift::slot_coord(M, slot, ci, cj);
        const float f = ci < cj ? kSqrt2f : 1.f;
        const int my_canon = slot < n ? lift::canonical_index(M, ci, cj) : -1;
        uint8_t* stage = sm + kOutOff;
        float run[DV + 1];  // running sum of the segment totals (prefix mode)
#pragma unroll
        for (int c = 0; c <= DV; ++c) run[c] = 0.f;
        for (int seg = seg0; seg < seg1; ++seg) {
            if (seg * L >= T) break;
            const int sl = seg - seg0, acb = sl & 1;
            if (!wait(&acc_full[acb], (sl >> 1) & 1)) { fail(); break; }
            tc_fence_after();
            const int64_t base = (bh * NS_out + seg) * (int64_t)n;
            // 32 columns per tensor-memory wait (the last wait also brings the
            // ones column, z): out = the segment's total, or (prefix mode) the
            // sum before it, into the staging row
            __syncwarp();  // this warp's previous rows have left the staging
            uint32_t zr = 0;
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
                uint32_t r[2][16];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    if (c0 + 16 * hh < DV) tmem_ld16(tmem_addr(tb + 128 * acb, lane0, c0 + 16 * hh), r[hh]);
                if (c0 + 32 >= DV) zr = tmem_ld1(tmem_addr(tb + 128 * acb, lane0, 64));  // the ones column: z
                tmem_wait_ld();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (c0 + 16 * hh >= DV) continue;
                    float out[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float tot = __uint_as_float(r[hh][i]);
                        out[i] = prefix ? run[c0 + 16 * hh + i] : tot;
                        run[c0 + 16 * hh + i] += tot;
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<float4*>(stage + e * kOutRow + 4 * (c0 + 16 * hh + 4 * c)) =
                            make_float4(f * out[4 * c], f * out[4 * c + 1], f * out[4 * c + 2], f * out[4 * c + 3]);
                }
            }
            {
                const float tot = __uint_as_float(zr);
                const float zo = prefix ? run[DV] : tot;
                run[DV] += tot;
                if (slot < n) z_out[base + my_canon] = f * zo;
            }
            tc_fence_before();
            mbar_arrive(&acc_free[acb]);
            __syncwarp();
            if (DV == 64) {
                // two rows per store instruction (16 bytes a lane), unrolled so
                // that the staging loads and the stores of several rows are in
                // flight at once
                const int half = lane >> 4, c16 = lane & 15;
#pragma unroll 4
                for (int rr = 0; rr < 32; rr += 2) {
                    const int row = rr + half;
                    const int canon = __shfl_sync(0xffffffffu, my_canon, row);
                    if (canon >= 0) {
                        const float4 val = *reinterpret_cast<const float4*>(stage + (32 * ew + row) * kOutRow + 16 * c16);
                        *reinterpret_cast<float4*>(S_out + (base + canon) * DV + 4 * c16) = val;
                    }
                }
            } else {
                for (int rr = 0; rr < 32; ++rr) {
                    const int canon = __shfl_sync(0xffffffffu, my_canon, rr);
                    if (canon < 0) continue;
                    const uint8_t* src = stage + (32 * ew + rr) * kOutRow;
                    float* dst = S_out + (base + canon) * DV;
                    if (lane < DV) dst[lane] = *reinterpret_cast<const float*>(src + 4 * lane);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 256);
}

template <int P, int DV, int LG>
cudaError_t launch_typed(const void* k, const void* v, float* S_out, float* z_out, int BH, int T, int L,
                         int NS, int NS_out, int prefix, const float* dec, cudaStream_t s) {
    auto kern = states_tc_kernel<P, DV, LG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    CUtensorMap tk, tv;
    if (!rows_map(&tk, k, P, T, BH) || !rows_map(&tv, v, DV, T, BH)) return cudaErrorInvalidValue;
    const int tiles = lift::tiles_of(P / LG);
    // about two CTAs per SM in total, each a run of segments
    const int64_t units = (int64_t)tiles * BH;
    int groups = prefix ? 1 : (int)((2 * 148) / (units > 0 ? units : 1));
    groups = groups < 1 ? 1 : (groups > NS ? NS : groups);
    const int per = (NS + groups - 1) / groups;
    groups = (NS + per - 1) / per;
    dim3 grid(tiles, groups, BH);
    KATA_TRACED("states_tc", s,
                kern<<<grid, kThreads, kSmem, s>>>(tk, tv, S_out, z_out, T, L, NS, NS_out, per, prefix, dec));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_states_tc(const void* k, const void* v, float* S_out, float* z_out, int BH, int T,
                             int p, int dv, int L, int NS, int NS_out, int prefix, int lg, cudaStream_t s,
                             const float* dec) {
    if (NS <= 0) return cudaSuccess;
    if (dec != nullptr && lg != 1) return cudaErrorInvalidValue;
#define KATA_CASE(P_, DV_, LG_)                  \
    if (p == P_ && dv == DV_ && lg == LG_) \
        return launch_typed<P_, DV_, LG_>(k, v, S_out, z_out, BH, T, L, NS, NS_out, prefix, dec, s);
    KATA_CASE(16, 16, 1) KATA_CASE(16, 32, 1) KATA_CASE(16, 64, 1)
    KATA_CASE(32, 16, 1) KATA_CASE(32, 32, 1) KATA_CASE(32, 64, 1)
    KATA_CASE(64, 16, 1) KATA_CASE(64, 32, 1) KATA_CASE(64, 64, 1)
    // KATA-Sigma-g: the block widths of the fused forward (p = 32, g = 2; p = 64, g = 2 or 4)
    KATA_CASE(32, 16, 2) KATA_CASE(32, 32, 2) KATA_CASE(32, 64, 2)
    KATA_CASE(64, 16, 2) KATA_CASE(64, 32, 2) KATA_CASE(64, 64, 2)
    KATA_CASE(64, 16, 4) KATA_CASE(64, 32, 4) KATA_CASE(64, 64, 4)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

unsigned int states_tc_take_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_states_tc_status, sizeof(v)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_states_tc_status, &zero, sizeof(zero));
    return v;
}

}  // namespace kata
