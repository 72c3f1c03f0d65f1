// Recurrent decode step (the constant-time recurrent inference of the
// abstract; the state recurrence S_t = S_{t-1} + psi(kh_t) v_t^T of the
// state-size paragraph taken one token at a time):
//   S += psi(kh) v^T,  z += psi(kh),  o = psi(qh)^T S / psi(qh)^T z
// with the updated state (causality s <= t).  The step reads and writes every
// state element once and does two FMAs per element: HBM-bound.
//
// One cluster per head.  Its NSPLIT CTAs split the head's n packed rows;
// each CTA updates its rows with 16-byte loads and stores (a state row of dv
// floats is dv/4 threads wide) and forms a partial readout [num | den].  The
// cluster's rank-0 CTA sums the NSPLIT partials out of the other CTAs' shared
// memory, in rank order, and divides.  The same kernel serves the block lifts
// (KATA-Sigma-g, KATA-M-g; BLOCK = true) with the lift's packed rows.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstdint>

#include "block_lift.cuh"
#include "kata_internal.h"

namespace kata {
namespace {

namespace cg = cooperative_groups;

constexpr int kDecThreads = 256;
constexpr int kDecUnroll = 4;  // state rows of a thread in flight at once
constexpr int kDecMaxSplit = 8;

template <typename Tin, int P, int DV, bool BLOCK, bool GATED = false>
__global__ void __launch_bounds__(kDecThreads)
decode_step_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                   Tin* __restrict__ o, float* __restrict__ S, float* __restrict__ z, int family, int g,
                   int n_block, const float* __restrict__ gate = nullptr) {
    // full lift: N = p(p+1)/2; block lift (family, g): N = n_block
    const int N = BLOCK ? n_block : P * (P + 1) / 2;
    const int m = BLOCK ? P / g : P, nm = m * (m + 1) / 2;
    constexpr int CPR = DV / 4;            // 16-byte columns of a state row
    constexpr int RP = kDecThreads / CPR;  // state rows per pass of the block
    constexpr int NW = kDecThreads / 32;
    static_assert(CPR <= 32 && 32 % CPR == 0, "a warp holds whole state rows");
    __shared__ float qh[P], kh[P];
    __shared__ __align__(16) float vv[DV];
    __shared__ __align__(16) float red[NW][DV];
    __shared__ float red_den[NW];
    __shared__ float part[DV + 1];
    __shared__ float tot[DV + 1];

    cg::cluster_group cluster = cg::this_cluster();
    const int nsplit = (int)cluster.num_blocks();
    const int split = (int)cluster.block_rank();
    const int64_t bh = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    load_rows_unit<Tin, P>(q + bh * P, 0, 1, 1, qh, P);
    load_rows_unit<Tin, P>(k + bh * P, 0, 1, 1, kh, P);
    load_rows_plain<Tin, DV>(v + bh * DV, 0, 1, 1, vv, DV);
    __syncthreads();

    // this CTA's packed rows [r0, r1)
    const int per = (N + nsplit - 1) / nsplit;
    const int r0 = split * per, r1 = min(N, r0 + per);
    const int c4 = tid % CPR, rr = tid / CPR;
    const float4 v4 = reinterpret_cast<const float4*>(vv)[c4];
    // gated step: the state is scaled by the head's gate before the token is added
    const float gam = GATED ? gate[bh] : 1.f;
    float4* Srow = reinterpret_cast<float4*>(S + bh * (int64_t)N * DV) + c4;
    float* zh = z + bh * (int64_t)N;

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    // (i, start): the lift row i holding packed row r, start = idx(i, i)
    // (inside block blk, whose first packed row is bstart, for M-g); r only
    // grows along a thread's walk, so i and blk only move forward.
    int i = 0, start = 0, blk = 0, bstart = 0;
    for (int rb = r0 + rr; rb < r1; rb += RP * kDecUnroll) {
        float4 s[kDecUnroll];
        float zr[kDecUnroll];
#pragma unroll
        for (int u = 0; u < kDecUnroll; ++u) {
            const int r = rb + u * RP;
            s[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            zr[u] = 0.f;
            if (r < r1) {
                s[u] = Srow[(int64_t)r * CPR];
                if (c4 == 0) zr[u] = zh[r];
            }
        }
#pragma unroll
        for (int u = 0; u < kDecUnroll; ++u) {
            const int r = rb + u * RP;
            if (r < r1) {
                float fk, fq;
                if constexpr (!BLOCK) {
                    while (r >= start + (P - i)) {
                        start += P - i;
                        ++i;
                    }
                    const int j = i + (r - start);
                    const float w = i == j ? 1.f : kSqrt2;
                    fk = w * kh[i] * kh[j];
                    fq = w * qh[i] * qh[j];
                } else {
                    if (family == kLiftMulti)
                        while (r >= bstart + nm) {
                            bstart += nm;
                            ++blk;
                            i = 0;
                            start = 0;
                        }
                    const int rl = r - bstart;
                    while (rl >= start + (m - i)) {
                        start += m - i;
                        ++i;
                    }
                    const int j = i + (rl - start);
                    const float w = i == j ? 1.f : kSqrt2;
                    if (family == kLiftMulti) {
                        fk = w * kh[blk * m + i] * kh[blk * m + j];
                        fq = w * qh[blk * m + i] * qh[blk * m + j];
                    } else {
                        float sk = 0.f, sq = 0.f;
                        for (int a = 0; a < g; ++a) {
                            sk = fmaf(kh[a * m + i], kh[a * m + j], sk);
                            sq = fmaf(qh[a * m + i], qh[a * m + j], sq);
                        }
                        fk = w * sk;
                        fq = w * sq;
                    }
                }
                float4 t = s[u];
                if constexpr (GATED) {
                    t.x *= gam;
                    t.y *= gam;
                    t.z *= gam;
                    t.w *= gam;
                }
                t.x = fmaf(fk, v4.x, t.x);
                t.y = fmaf(fk, v4.y, t.y);
                t.z = fmaf(fk, v4.z, t.z);
                t.w = fmaf(fk, v4.w, t.w);
                Srow[(int64_t)r * CPR] = t;
                acc.x = fmaf(fq, t.x, acc.x);
                acc.y = fmaf(fq, t.y, acc.y);
                acc.z = fmaf(fq, t.z, acc.z);
                acc.w = fmaf(fq, t.w, acc.w);
                if (c4 == 0) {
                    const float zn = (GATED ? gam * zr[u] : zr[u]) + fk;
                    zh[r] = zn;
                    den = fmaf(fq, zn, den);
                }
            }
        }
    }

    // block partial: sum over the rows each warp holds, then over warps
#pragma unroll
    for (int off = CPR; off < 32; off <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    den = warp_sum(den);
    if (lane < CPR) reinterpret_cast<float4*>(red[warp])[lane] = acc;
    if (lane == 0) red_den[warp] = den;
    __syncthreads();
    if (tid < DV) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) a += red[w][tid];
        part[tid] = a;
    } else if (tid == DV) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) a += red_den[w];
        part[DV] = a;
    }

    // head total on the rank-0 CTA; every CTA stays until it has been read
    cluster.sync();
    if (split == 0) {
        if (tid <= DV) {
            float a = 0.f;
            for (int c = 0; c < nsplit; ++c) a += cluster.map_shared_rank(part, c)[tid];
            tot[tid] = a;
        }
        __syncthreads();
        if (tid < DV) {
            const float d = tot[DV];
            store_as(o + bh * DV + tid, d > 0.f ? tot[tid] / d : 0.f);
        }
    }
    cluster.sync();
}

template <typename Tin, int P, int DV>
cudaError_t launch_typed(const void* q, const void* k, const void* v, void* o, float* S, float* z, int BH,
                         int family, int g, const float* gate, cudaStream_t s) {
    const bool block = family != kLiftFull;
    const int N = block ? block_lift_dim(family, P, g) : P * (P + 1) / 2;
    if (N <= 0) return cudaErrorInvalidValue;
    constexpr int RP = kDecThreads / (DV / 4);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // enough CTAs for two per SM, each with at least one full pass of rows
    int nsplit = (2 * sms + BH - 1) / BH;
    nsplit = std::max(1, std::min({nsplit, kDecMaxSplit, N / RP}));
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)nsplit, (unsigned)BH, 1);
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (gate)
        KATA_TRACED("decode_step_gated", s,
                    e = cudaLaunchKernelEx(&cfg, decode_step_kernel<Tin, P, DV, false, true>,
                                           static_cast<const Tin*>(q), static_cast<const Tin*>(k),
                                           static_cast<const Tin*>(v), static_cast<Tin*>(o), S, z, family, g, N,
                                           gate));
    else if (block)
        KATA_TRACED("decode_step_block", s,
                    e = cudaLaunchKernelEx(&cfg, decode_step_kernel<Tin, P, DV, true>, static_cast<const Tin*>(q),
                                           static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                                           static_cast<Tin*>(o), S, z, family, g, N, nullptr));
    else
        KATA_TRACED("decode_step", s,
                    e = cudaLaunchKernelEx(&cfg, decode_step_kernel<Tin, P, DV, false>, static_cast<const Tin*>(q),
                                           static_cast<const Tin*>(k), static_cast<const Tin*>(v),
                                           static_cast<Tin*>(o), S, z, family, g, N, nullptr));
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename Tin, int P>
cudaError_t by_dv(const void* q, const void* k, const void* v, void* o, float* S, float* z, int BH, int dv,
                  int family, int g, const float* gate, cudaStream_t s) {
    switch (dv) {
        case 16: return launch_typed<Tin, P, 16>(q, k, v, o, S, z, BH, family, g, gate, s);
        case 32: return launch_typed<Tin, P, 32>(q, k, v, o, S, z, BH, family, g, gate, s);
        case 64: return launch_typed<Tin, P, 64>(q, k, v, o, S, z, BH, family, g, gate, s);
    }
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t by_p(const void* q, const void* k, const void* v, void* o, float* S, float* z, int BH, int p, int dv,
                 int family, int g, const float* gate, cudaStream_t s) {
    switch (p) {
        case 16: return by_dv<Tin, 16>(q, k, v, o, S, z, BH, dv, family, g, gate, s);
        case 32: return by_dv<Tin, 32>(q, k, v, o, S, z, BH, dv, family, g, gate, s);
        case 64: return by_dv<Tin, 64>(q, k, v, o, S, z, BH, dv, family, g, gate, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_step(int dtype, const void* q, const void* k, const void* v, void* o, float* S,
                               float* z, int BH, int p, int dv, int family, int g, const float* gate,
                               cudaStream_t s) {
    return dtype == 0 ? by_p<float>(q, k, v, o, S, z, BH, p, dv, family, g, gate, s)
                      : by_p<__nv_bfloat16>(q, k, v, o, S, z, BH, p, dv, family, g, gate, s);
}

}  // namespace kata
