// Self-test of libkata's tcgen05 building blocks (test infrastructure): one
// CTA computes D[128 x N] = A[128 x K] * B[N x K]^T with bf16 operands and an
// fp32 TMEM accumulator, A taken from shared memory (mode 0) or from tensor
// memory (mode 1), B from shared memory, both in the K-major 128B-swizzled
// layout.  The test compares D with a host matmul.
#include <cuda_bf16.h>
#include <cstdint>

#include "../../kernelized_linear_attention_03_b300/csrc/tc_primitives.cuh"

using namespace kata::tc;

namespace {

__global__ void __launch_bounds__(128) gemm_probe(const __nv_bfloat16* __restrict__ A,
                                                  const __nv_bfloat16* __restrict__ B,
                                                  float* __restrict__ D, int K, int N, int mode,
                                                  int* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int kblocks = (K + 63) / 64;     // 128-byte rows, 64 elements per column block
    uint8_t* As = smem;                    // 128 rows x kblocks blocks
    uint8_t* Bs = smem + 128 * 128 * kblocks;  // N rows x kblocks blocks (N multiple of 8)
    const int t = threadIdx.x, warp = t >> 5;
    if (t == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    // operands into the swizzled layout, 8 elements (16 B) at a time
    for (int e = t; e < 128 * (K / 8); e += 128) {
        const int r = e / (K / 8), k = (e % (K / 8)) * 8;
        *reinterpret_cast<uint4*>(As + sw128_chunk(r, k, 128)) =
            *reinterpret_cast<const uint4*>(A + (size_t)r * K + k);
    }
    for (int e = t; e < N * (K / 8); e += 128) {
        const int r = e / (K / 8), k = (e % (K / 8)) * 8;
        *reinterpret_cast<uint4*>(Bs + sw128_chunk(r, k, N)) =
            *reinterpret_cast<const uint4*>(B + (size_t)r * K + k);
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t d_tmem = tb, a_tmem = tb + 128;  // D: cols 0..N-1, A: cols 128..128+K/2-1
    if (mode == 1) {
        // row t of A into lane t, column c holding elements (2c, 2c+1)
        const uint32_t lane0 = (uint32_t)(warp * 32);
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t r[16];
            for (int i = 0; i < 16; ++i) {
                const int k = 2 * (c0 + i);
                r[i] = pack_bf16x2(__bfloat162float(A[(size_t)t * K + k]),
                                   __bfloat162float(A[(size_t)t * K + k + 1]));
            }
            tmem_st16(tmem_addr(a_tmem, lane0, c0), r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t == 0) {
        const uint32_t idesc = idesc_bf16_f32(128, N);
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint32_t koff = (ks & 3) * 32;
            const uint64_t ad = sdesc_kmajor_sw128(smem_u32(As) + (ks >> 2) * 128 * 128 + koff);
            const uint64_t bd = sdesc_kmajor_sw128(smem_u32(Bs) + (ks >> 2) * N * 128 + koff);
            if (mode == 0)
                mma_ss(d_tmem, ad, bd, idesc, ks > 0);
            else
                mma_ts(d_tmem, a_tmem + ks * 8, bd, idesc, ks > 0);
        }
        mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0, &abort_flag, 1000000000ull);
    if (!ok) {
        abort_flag = 1;
        atomicExch(status, 1);
    }
    tc_fence_after();
    if (ok) {
        const uint32_t lane0 = (uint32_t)(warp * 32);
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tmem_addr(d_tmem, lane0, c0), r);
            tmem_wait_ld();
            for (int i = 0; i < 16; ++i) D[(size_t)t * N + c0 + i] = __uint_as_float(r[i]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 256);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int kata_tc_selftest(const void* A, const void* B,
                                                                     float* D, int K, int N, int mode,
                                                                     int* status, cudaStream_t s) {
    if (K < 16 || K > 128 || K % 16 || N < 16 || N > 128 || N % 16 || (mode != 0 && mode != 1)) return 1;
    const int smem = 1024 + (128 + N) * 128 * ((K + 63) / 64);
    if (cudaFuncSetAttribute(gemm_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 2;
    gemm_probe<<<1, 128, smem, s>>>(static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B),
                                    D, K, N, mode, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
