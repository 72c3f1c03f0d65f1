// Block lifts of the "two reduced PSD families" paragraph, on the device.
// g divides p, m = p/g; a unit vector u is cut into g contiguous blocks
// u_a = u[a m .. a m + m - 1].
//   family 1, KATA-Sigma-g: psi(u) = sum_a u_a u_a^T, packed m(m+1)/2;
//     <psi(q), psi(k)> = sum_{a,b} (q_a.k_b)^2.
//   family 2, KATA-M-g: psi(u) = (u_1 u_1^T, ..., u_g u_g^T), the g packed
//     m x m blocks one after another, g m(m+1)/2 coordinates;
//     <psi(q), psi(k)> = sum_a (q_a.k_a)^2.
//   family 0: the full rank-one lift (g = 1, m = p).
// Inside a block the packing of the full lift: upper triangle row by row,
// off-diagonal coordinates times sqrt 2.
#pragma once

#include "kata_device.cuh"

namespace kata {

constexpr int kLiftFull = 0, kLiftSigma = 1, kLiftMulti = 2;

// Width of the lift; -1 if (family, g) does not fit p.
__host__ __device__ inline int block_lift_dim(int family, int p, int g) {
    if (p <= 0 || g <= 0 || p % g != 0) return -1;
    const int m = p / g, nm = m * (m + 1) / 2;
    if (family == kLiftFull) return g == 1 ? nm : -1;
    if (family == kLiftSigma) return nm;
    if (family == kLiftMulti) return g * nm;
    return -1;
}

// Packed row r of a block lift: the pair (i, j), i <= j < m, inside block
// `blk` (-1: the g blocks summed, families 0 and 1) and its scale.
struct BlockRow {
    int i, j, blk;
    float scale;
};

__device__ __forceinline__ BlockRow block_row(int r, int family, int m) {
    BlockRow d;
    d.blk = -1;
    if (family == kLiftMulti) {
        const int nm = m * (m + 1) / 2;
        d.blk = r / nm;
        r -= d.blk * nm;
    }
    unpack_index(r, m, d.i, d.j);
    d.scale = d.i == d.j ? 1.f : kSqrt2;
    return d;
}

// psi_r(u) for the row described by d; u is a unit vector in shared memory.
__device__ __forceinline__ float block_coord(const float* u, const BlockRow& d, int g, int m) {
    if (d.blk >= 0) return d.scale * u[d.blk * m + d.i] * u[d.blk * m + d.j];
    float s = 0.f;
    for (int a = 0; a < g; ++a) s = fmaf(u[a * m + d.i], u[a * m + d.j], s);
    return d.scale * s;
}

// <psi(qu), psi(ku)> from block dot products: every block pair for
// Sigma-g, equal blocks otherwise.
__device__ __forceinline__ float block_score(const float* qu, const float* ku, int family, int g, int m) {
    float w = 0.f;
    for (int a = 0; a < g; ++a)
        for (int b = 0; b < g; ++b) {
            if (family != kLiftSigma && a != b) continue;
            float c = 0.f;
            for (int i = 0; i < m; ++i) c = fmaf(qu[a * m + i], ku[b * m + i], c);
            w = fmaf(c, c, w);
        }
    return w;
}

}  // namespace kata
