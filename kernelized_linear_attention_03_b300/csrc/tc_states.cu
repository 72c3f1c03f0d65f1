// Segment states on the tcgen05 tensor cores (bf16 inputs, fp32 accumulate):
// for each head and each segment of L consecutive tokens,
//   S_seg = sum_{t in seg} psi(kh_t) v_t^T,   z_seg = sum_{t in seg} psi(kh_t)
// (the state S_t = Psi(K_{1:t})^T V_{1:t} of the state-size paragraph
// restricted to one segment; with L = C these are the local chunk states of
// the chunked-scan paragraph's state kernel).
//
// One CTA owns one 128-slot tile of the packed lift for a run of segments
// of one head.  Per block of up to 128 tokens: every thread puts its key on
// the unit sphere, writes its 128 lifted coordinates of the tile into a
// token-major (MN-major for the MMA) swizzled tile, and its value row with a
// trailing ones column into a token-major [V | 1] tile; one thread issues
//   D[slots x (dv+16)] += psiK(K)^T [V | 1]     (tcgen05, D in TMEM)
// with K = tokens.  At the end of a segment the tile's rows are written out
// in the C ABI's sqrt(2)-packed order.
#include <cuda_bf16.h>

#include <cstdint>

#include "kata_internal.h"
#include "tc_lift.cuh"
#include "tc_primitives.cuh"

namespace kata {
namespace {

using namespace tc;

__device__ unsigned int g_states_tc_status = 0;

constexpr int kThreads = 128;
constexpr float kSqrt2f = 1.41421356237309504880f;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kAtom = 128 * 128;  // one MN atom: 128 K-rows (tokens) x 128 bytes

template <int DV>
struct StatesLayout {
    static constexpr int NB = DV + 16;                       // [V | 1 | 0 pad] columns
    static constexpr int b_atoms = (NB + 63) / 64;
    static constexpr uint32_t a_off = 0, b_off = 2 * kAtom;  // A: two 64-slot atoms
    static constexpr uint32_t total = b_off + b_atoms * kAtom;
    static constexpr size_t smem = total + 1024;
};

// Lifted key coordinates of tile TAU for this thread's token into row `row`
// of the token-major A tile.
template <int P, int TAU>
__device__ __forceinline__ void key_tile_to_smem(const uint32_t (&u)[P / 2], uint8_t* As, int row) {
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

template <int P, int TAU = 0>
__device__ __forceinline__ void key_tile_dispatch(int tau, const uint32_t (&u)[P / 2], uint8_t* As, int row) {
    if constexpr (TAU < lift::tiles_of(P)) {
        if (tau == TAU)
            key_tile_to_smem<P, TAU>(u, As, row);
        else
            key_tile_dispatch<P, TAU + 1>(tau, u, As, row);
    }
}

template <int P, int DV>
__global__ void __launch_bounds__(kThreads)
states_tc_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                 float* __restrict__ S_out, float* __restrict__ z_out, int T, int L, int NS,
                 int NS_out, int segs_per_cta) {
    // T: tokens per head (row stride and bound); segments 0..NS-1 of L tokens
    // are computed (NS may cover fewer than all T tokens) into rows of a
    // [BH, NS_out, n] layout.
    using Lay = StatesLayout<DV>;
    constexpr int NB = Lay::NB;
    constexpr int n = lift::packed_n(P);
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* As = sm + Lay::a_off;
    uint8_t* Bs = sm + Lay::b_off;

    const int t = threadIdx.x, warp = t >> 5;
    const int tau = blockIdx.x;
    const int64_t bh = blockIdx.z;
    const int seg0 = blockIdx.y * segs_per_cta;
    const int seg1 = min(NS, seg0 + segs_per_cta);
    const __nv_bfloat16* kh = k + bh * (int64_t)T * P;
    const __nv_bfloat16* vh = v + bh * (int64_t)T * DV;

    if (t == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t d_tm = tmem_base;
    const uint32_t lane0 = (uint32_t)(warp * 32);
    uint32_t phase = 0;
    bool ok = true;

    for (int seg = seg0; seg < seg1 && ok; ++seg) {
        const int s_begin = seg * L, s_end = min(T, s_begin + L);
        bool first = true;
        for (int b0 = s_begin; b0 < s_end; b0 += 128) {
            const int b1 = min(s_end, b0 + 128);
            const int tok = b0 + t;
            const bool valid = tok < b1;
            // ---- unit key, lifted tile coordinates -> A (token-major)
            uint32_t u[P / 2];
            {
                uint4 raw[P / 8];
                float ss = 0.f;
#pragma unroll
                for (int c = 0; c < P / 8; ++c) {
                    raw[c] = valid ? *reinterpret_cast<const uint4*>(kh + (int64_t)tok * P + 8 * c)
                                   : make_uint4(0, 0, 0, 0);
                    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[c]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float x = __bfloat162float(e[i]);
                        ss = fmaf(x, x, ss);
                    }
                }
                const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
                for (int c = 0; c < P / 8; ++c) {
                    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[c]);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        u[4 * c + i] = pack_bf16x2(__bfloat162float(e[2 * i]) * inv,
                                                   __bfloat162float(e[2 * i + 1]) * inv);
                }
            }
            key_tile_dispatch<P>(tau, u, As, t);
            // ---- [V | 1 | 0] row -> B (token-major)
#pragma unroll
            for (int c = 0; c < DV / 8; ++c) {
                const uint4 val = valid ? *reinterpret_cast<const uint4*>(vh + (int64_t)tok * DV + 8 * c)
                                        : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(Bs + mn_sw128_chunk(8 * c, t, kAtom)) = val;
            }
            *reinterpret_cast<uint4*>(Bs + mn_sw128_chunk(DV, t, kAtom)) =
                make_uint4(valid ? pack_bf16x2(1.f, 0.f) : 0u, 0, 0, 0);
            *reinterpret_cast<uint4*>(Bs + mn_sw128_chunk(DV + 8, t, kAtom)) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            // ---- D += psiK^T [V | 1] over this block's tokens
            if (t == 0) {
                tc_fence_after();
                constexpr uint32_t idesc = idesc_bf16_f32_major(128, NB, true, true);
                const int steps = (b1 - b0 + 15) / 16;
                for (int ks = 0; ks < steps; ++ks)
                    mma_ss(d_tm, sdesc_mnmajor_sw128(smem_u32(As) + ks * 2048, kAtom),
                           sdesc_mnmajor_sw128(smem_u32(Bs) + ks * 2048, kAtom), idesc,
                           (first && ks == 0) ? 0u : 1u);
                mma_commit(&bar);
            }
            first = false;
            ok = mbar_wait(&bar, phase, &abort_flag, kWaitNs);
            phase ^= 1;
            if (!ok) abort_flag = 1;
            if (!__syncthreads_and(ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        if (!ok) break;
        // ---- write the segment's tile rows in the sqrt(2)-packed order
        const int slot = tau * 128 + t;
        uint32_t r[NB];
#pragma unroll
        for (int c0 = 0; c0 < NB; c0 += 16) {
            uint32_t q[16];
            tmem_ld16(tmem_addr(d_tm, lane0, c0), q);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[c0 + i] = q[i];
        }
        tmem_wait_ld();
        if (slot < n) {
            int i = 0, j = 0;
            lift::slot_coord(P, slot, i, j);
            const float f = i < j ? kSqrt2f : 1.f;
            const int64_t row = (bh * NS_out + seg) * (int64_t)n + lift::canonical_index(P, i, j);
            float4* dst = reinterpret_cast<float4*>(S_out + row * DV);
#pragma unroll
            for (int c = 0; c < DV / 4; ++c)
                dst[c] = make_float4(f * __uint_as_float(r[4 * c]), f * __uint_as_float(r[4 * c + 1]),
                                     f * __uint_as_float(r[4 * c + 2]), f * __uint_as_float(r[4 * c + 3]));
            z_out[row] = f * __uint_as_float(r[DV]);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (!ok) {
        if (t == 0) atomicOr(&g_states_tc_status, kStatusTimeout);
        mbar_wait_quiet(&bar, phase ^ 1, kWaitNs / 4);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(d_tm, 128);
}

template <int P, int DV>
cudaError_t launch_typed(const void* k, const void* v, float* S_out, float* z_out, int BH, int T, int L,
                         int NS, int NS_out, cudaStream_t s) {
    constexpr size_t smem = StatesLayout<DV>::smem;
    auto kern = states_tc_kernel<P, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int tiles = lift::tiles_of(P);
    // a few segments per CTA, enough CTAs for several waves
    const int64_t work = (int64_t)tiles * NS * BH;
    int per = (int)((work + 148 * 8 - 1) / (148 * 8));
    per = per < 1 ? 1 : (per > 64 ? 64 : per);
    const int groups = (NS + per - 1) / per;
    dim3 grid(tiles, groups, BH);
    KATA_TRACED("states_tc", s,
                kern<<<grid, kThreads, smem, s>>>(static_cast<const __nv_bfloat16*>(k),
                                                  static_cast<const __nv_bfloat16*>(v), S_out, z_out, T,
                                                  L, NS, NS_out, per));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_states_tc(const void* k, const void* v, float* S_out, float* z_out, int BH, int T,
                             int p, int dv, int L, int NS, int NS_out, cudaStream_t s) {
    if (NS <= 0) return cudaSuccess;
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return launch_typed<P_, DV_>(k, v, S_out, z_out, BH, T, L, NS, NS_out, s);
    KATA_CASE(16, 16) KATA_CASE(16, 32) KATA_CASE(16, 64)
    KATA_CASE(32, 16) KATA_CASE(32, 32) KATA_CASE(32, 64)
    KATA_CASE(64, 16) KATA_CASE(64, 32) KATA_CASE(64, 64)
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
