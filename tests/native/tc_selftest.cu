// Self-test of libkata's tcgen05 building blocks (test infrastructure): one
// CTA computes D[128 x N] = A[128 x K] * B[N x K]^T with bf16 operands and an
// fp32 TMEM accumulator, A taken from shared memory or from tensor memory,
// B from shared memory, shared-memory operands in the K-major or MN-major
// 128B-swizzled layouts.  The test compares D with a host matmul.
#include <cuda_bf16.h>
#include <cstdint>

#include "../../kernelized_linear_attention_03_b300/csrc/tc_primitives.cuh"

using namespace kata::tc;

namespace {

// mode 0: A smem K-major,  B smem K-major
// mode 1: A tmem,           B smem K-major
// mode 2: A smem MN-major,  B smem K-major
// mode 3: A tmem,           B smem MN-major
// mode 4: A smem MN-major,  B smem MN-major
__global__ void __launch_bounds__(128) gemm_probe(const __nv_bfloat16* __restrict__ A,
                                                  const __nv_bfloat16* __restrict__ B,
                                                  float* __restrict__ D, int K, int N, int mode,
                                                  int* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const bool a_mn = (mode == 2 || mode == 4), b_mn = (mode == 3 || mode == 4);
    const uint32_t a_atom = (uint32_t)K * 128u;  // MN-major atom: K rows of 128 bytes
    const uint32_t b_atom = (uint32_t)K * 128u;
    uint8_t* As = smem;                                        // 32 KB at most
    uint8_t* Bs = smem + 128 * 128 * 2;                        // up to 128 x 128 elements
    const int t = threadIdx.x, warp = t >> 5;
    if (t == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    // operands into the swizzled layouts, one element at a time
    for (int e = t; e < 128 * K; e += 128) {
        const int m = e / K, k = e % K;
        const uint32_t off = a_mn ? mn_sw128_offset(m, k, a_atom) : sw128_offset(m, k, 128);
        *reinterpret_cast<__nv_bfloat16*>(As + off) = A[(size_t)m * K + k];
    }
    for (int e = t; e < N * K; e += 128) {
        const int n = e / K, k = e % K;
        const uint32_t off = b_mn ? mn_sw128_offset(n, k, b_atom) : sw128_offset(n, k, N);
        *reinterpret_cast<__nv_bfloat16*>(Bs + off) = B[(size_t)n * K + k];
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
    const bool a_tm = (mode == 1 || mode == 3);
    if (a_tm) {
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
        const uint32_t idesc = idesc_bf16_f32_major(128, N, a_mn, b_mn);
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint32_t koff = (ks & 3) * 32;
            const uint64_t ad = a_mn ? sdesc_mnmajor_sw128(smem_u32(As) + ks * 2048, a_atom)
                                     : sdesc_kmajor_sw128(smem_u32(As) + (ks >> 2) * 128 * 128 + koff);
            const uint64_t bd = b_mn ? sdesc_mnmajor_sw128(smem_u32(Bs) + ks * 2048, b_atom)
                                     : sdesc_kmajor_sw128(smem_u32(Bs) + (ks >> 2) * N * 128 + koff);
            if (a_tm)
                mma_ts(d_tmem, a_tmem + ks * 8, bd, idesc, ks > 0);
            else
                mma_ss(d_tmem, ad, bd, idesc, ks > 0);
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
    if (K < 16 || K > 128 || K % 16 || N < 16 || N > 128 || N % 16 || mode < 0 || mode > 4) return 1;
    const int smem = 1024 + 2 * 128 * 128 * 2;
    if (cudaFuncSetAttribute(gemm_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 2;
    gemm_probe<<<1, 128, smem, s>>>(static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B),
                                    D, K, N, mode, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// ---------------------------------------------------------------- bounded waits
// A warp waits on an mbarrier that nothing ever arrives on, with a budget of
// `budget_ns`; the wait must give up, and the kernel must report it and return
// (the same bounded wait every tensor-core kernel of the library uses).
namespace {

__global__ void wait_probe(int* status, unsigned long long* elapsed_ns, unsigned long long budget_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        kata::tc::mbar_init(&bar, 1);
        kata::tc::fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    const unsigned long long t0 = kata::tc::globaltimer_ns();
    const bool ok = kata::tc::mbar_wait(&bar, 0, &abort_flag, budget_ns);
    const unsigned long long t1 = kata::tc::globaltimer_ns();
    if (threadIdx.x == 0) {
        status[0] = ok ? 0 : 1;  // 1: the wait gave up, as it must
        elapsed_ns[0] = t1 - t0;
    }
}

__global__ void after_probe(int* status) {
    if (threadIdx.x == 0) status[1] = 42;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int kata_wait_selftest(int* status,
                                                                       unsigned long long* elapsed_ns,
                                                                       unsigned long long budget_ns,
                                                                       cudaStream_t s) {
    wait_probe<<<1, 32, 0, s>>>(status, elapsed_ns, budget_ns);
    after_probe<<<1, 32, 0, s>>>(status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
