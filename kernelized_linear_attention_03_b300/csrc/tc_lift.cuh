// The rank-one lift psi(u) = u u^T of the tensor-core kernels, in the slot
// order they keep internally (the rank-one lift paragraph after Eq. 8; the
// packed width n = p(p+1)/2 of Eq. 8).
//
// Internal slot order.  With h = p/2, the n = h(2h+1) coordinates (i <= j)
// of the upper triangle are laid out as 2h+1 rows of h slots, slot s in row
// R = s / h at column l = s % h.  Even rows R = 2r < 2h are the "rectangle"
// (r, h + l); odd rows R = 2r + 1 and the last row R = 2h (r = h) fold the
// two triangles together:
//   l >= r -> (r, l)          (upper-left triangle)
//   l <  r -> (h + l, h-1+r)  (lower-right triangle)
// Two consecutive slots (l even) nearly always share one factor and take the
// other from an aligned pair of u: one bf16x2 multiply per pair.  Rectangle
// and fold rows alternate so that every 128-slot tile of the tensor-core
// kernels (a run of whole rows for p >= 16) holds as many of each: the fold
// rows' lift costs a little more, and the slowest tile sets the pace.
//
// Internal scaling.  Keys are lifted without the sqrt(2) of the packed
// Frobenius form: psiK(k)_(i,j) = k_i k_j.  Queries carry the whole factor 2
// of the off-diagonal terms: psiQ(q)_(i,j) = q_i q_j (i = j), 2 q_i q_j
// (i < j).  Then <psiQ(q), psiK(k)> = (q.k)^2 exactly as in the lift
// identity, every scaling is a power of two (exact in bf16), and a state
// built from psiK differs from the sqrt(2)-packed state of the C ABI only by
// a factor sqrt(2) on its off-diagonal rows.
#pragma once

#include <cstdint>

namespace kata {
namespace lift {

__host__ __device__ constexpr int packed_n(int P) { return P * (P + 1) / 2; }
__host__ __device__ constexpr int tiles_of(int P) { return (packed_n(P) + 127) / 128; }

// Coordinates (i, j), i <= j, of internal slot s < n.
__host__ __device__ constexpr void slot_coord(int P, int s, int& i, int& j) {
    const int h = P / 2;
    const int R = s / h, l = s % h;
    if (R < 2 * h && (R & 1) == 0) {
        i = R / 2;
        j = h + l;
    } else {
        const int r = R < 2 * h ? R / 2 : h;
        if (l >= r) {
            i = r;
            j = l;
        } else {
            i = h + l;
            j = h - 1 + r;
        }
    }
}

// Row of (i, j) in the C ABI's packed order idx(i,j) = i*P - i(i-1)/2 + (j-i).
__host__ __device__ constexpr int canonical_index(int P, int i, int j) { return i * P - i * (i - 1) / 2 + (j - i); }

// bf16 pair with element a of ua in the low half and element b of ub in the
// high half (arrays of packed bf16x2 words; a, b compile-time after unrolling).
__device__ __forceinline__ uint32_t bf16_pair(const uint32_t* ua, int a, const uint32_t* ub, int b) {
    const uint32_t sel = ((a & 1) ? 0x32u : 0x10u) | ((b & 1) ? 0x7600u : 0x5400u);
    return __byte_perm(ua[a >> 1], ub[b >> 1], sel);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// bf16 pair (u_a, u_b) of the vector u (P/2 packed words; a, b compile-time
// after unrolling): an aligned pair is the word itself, a repeated element one
// byte permute (shared by every word that repeats it), anything else a
// permute of two words.
__device__ __forceinline__ uint32_t u_pair(const uint32_t* u, int a, int b) {
    if ((a & 1) == 0 && b == a + 1) return u[a >> 1];
    if (a == b) return __byte_perm(u[a >> 1], 0u, (a & 1) ? 0x3232u : 0x1010u);
    return bf16_pair(u, a, u, b);
}

// Packed bf16x2 word holding the lift at slots (2w, 2w+1) of the vector u
// (P/2 packed words).  QUERY applies the query's factor 2 to off-diagonal
// slots (exact in bf16).  Slots at or past n give 0.  The word is the product
// of two pairs, (u_i0, u_i1) and (u_j0, u_j1); in every tile of the slot order
// one of them repeats a single element over a run of words, and the factor
// goes onto that one, so that it is computed once per run and each word costs
// one multiply.
template <int P, bool QUERY>
__device__ __forceinline__ uint32_t lift_word(const uint32_t* u, int w) {
    constexpr int n = packed_n(P);
    const int s0 = 2 * w, s1 = 2 * w + 1;
    if (s0 >= n) return 0u;
    int i0 = 0, j0 = 0, i1 = 0, j1 = 0;
    slot_coord(P, s0, i0, j0);
    if (s1 < n) {
        slot_coord(P, s1, i1, j1);
    } else {
        i1 = i0;
        j1 = j0;
    }
    uint32_t x = u_pair(u, i0, i1);
    uint32_t y = u_pair(u, j0, j1);
    if (QUERY) {
        const uint32_t f = (i0 < j0 ? 0x4000u : 0x3F80u) | ((i1 < j1 ? 0x4000u : 0x3F80u) << 16);  // (2|1, 2|1)
        if (f != 0x3F803F80u) {
            if (i0 == i1 || j0 != j1)
                x = bf16x2_mul(x, f);
            else
                y = bf16x2_mul(y, f);
        }
    }
    const uint32_t r = bf16x2_mul(x, y);
    return s1 < n ? r : (r & 0xFFFFu);
}

}  // namespace lift
}  // namespace kata
