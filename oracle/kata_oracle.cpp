// KATA oracle: a plain, slow, fp64 CPU restatement of the causal normalised
// linear-attention forward of "Kernelized Linear Attention: Breaking the
// Capacity Wall with Symmetric Cones" (arXiv 2607.17419).
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
// load this file; only the test suite, the smoke check and the benchmark's
// CPU-baseline leg use it.  It shares no code, header or constant with the
// CUDA library.
//
// Every function works on fp64 arrays in the layout the library documents:
//   q, k : [B, H, T, p]      v, o : [B, H, T, dv]
//   packed state S : [n, dv] with n = p(p+1)/2, z : [n]
//   packed index of (i, j), i <= j : row-major upper triangle
//        idx(i, j) = i*p - i*(i-1)/2 + (j - i)
// Plain loops, no BLAS, no blocking; threads only split independent heads.
//
// Citations are to the arXiv HTML page of the paper (section / equation):
//   * unit-sphere projection and the rank-one lift psi(u) = u u^T with
//     ||u u^T||_F = 1 and <u u^T, v v^T>_F = (u.v)^2: the "rank-one lift"
//     paragraph after Eq. 8;
//   * packed width n = p(p+1)/2: Eq. 8 and the state-size paragraph
//     ("n = d(d+1)/2 unique coordinates after symmetry packing");
//   * state S_t = Psi(K_{1:t})^T V_{1:t}: state-size paragraph;
//   * normalised readout psi(q_t)^T S_t / psi(q_t)^T Z_t: the discussion of
//     Assumption 1 (denominator psi(q_t)^T Z_t) and the convex output gate;
//   * chunked form: per-chunk local states, an associative prefix over the
//     N_C chunks (sequential, or a scan in ceil(log2 N_C) rounds of
//     N_C-wide work) and a per-chunk output that adds the local C x C
//     causal part: the chunked-scan paragraph (the one introducing the
//     three kernels and the wall-clock model).
//
// Readings where the pages are silent:
//   * off-diagonal packed coordinates carry a factor sqrt(2), diagonal 1, so
//     the packed dot product is the Frobenius product;
//   * q and k are normalised inside the forward; a zero vector stays zero;
//   * causality is inclusive (s <= t, "K_{1:t}");
//   * a zero denominator gives a zero output row (no epsilon);
//   * the chunk output uses the exclusive prefix of earlier chunks plus the
//     inclusive causal part of its own chunk; a ragged last chunk is shorter.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

inline int64_t packed_dim_i(int p) { return (int64_t)p * (p + 1) / 2; }

inline int64_t pidx(int p, int i, int j) {  // requires i <= j
    return (int64_t)i * p - (int64_t)i * (i - 1) / 2 + (j - i);
}

// u = x / ||x||; the zero vector maps to zero.
void normalize(const double* x, int p, double* u) {
    double ss = 0.0;
    for (int i = 0; i < p; ++i) ss += x[i] * x[i];
    double nrm = std::sqrt(ss);
    for (int i = 0; i < p; ++i) u[i] = nrm > 0.0 ? x[i] / nrm : 0.0;
}

// psi(u) = u u^T packed: diagonal u_i^2, off-diagonal sqrt(2) u_i u_j.
void lift(const double* u, int p, double* psi) {
    const double r2 = std::sqrt(2.0);
    for (int i = 0; i < p; ++i)
        for (int j = i; j < p; ++j)
            psi[pidx(p, i, j)] = (i == j) ? u[i] * u[i] : r2 * u[i] * u[j];
}

double dot(const double* a, const double* b, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

// Run f(head) for head in [0, heads) on up to nthreads threads.
template <class F>
void for_heads(int64_t heads, int nthreads, F f) {
    if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
    nthreads = (int)std::min<int64_t>(nthreads, std::max<int64_t>(heads, 1));
    if (nthreads <= 1) {
        for (int64_t h = 0; h < heads; ++h) f(h);
        return;
    }
    std::vector<std::thread> pool;
    for (int w = 0; w < nthreads; ++w)
        pool.emplace_back([&, w] {
            for (int64_t h = w; h < heads; h += nthreads) f(h);
        });
    for (auto& th : pool) th.join();
}

// Normalise every row of a [rows, p] block.
std::vector<double> normalized_rows(const double* x, int64_t rows, int p) {
    std::vector<double> u((size_t)(rows * p));
    for (int64_t r = 0; r < rows; ++r) normalize(x + r * p, p, u.data() + r * p);
    return u;
}

// Exclusive prefix over `nc` items of width `w`, sequential: one step per item.
void exclusive_sequential(const double* x, int64_t nc, int64_t w, double* out) {
    std::vector<double> run((size_t)w, 0.0);
    for (int64_t c = 0; c < nc; ++c) {
        for (int64_t e = 0; e < w; ++e) out[c * w + e] = run[e];
        for (int64_t e = 0; e < w; ++e) run[e] += x[c * w + e];
    }
}

// Exclusive prefix by a log-depth scan: ceil(log2 nc) rounds, each round adds
// to every item the item 2^d places earlier (read from the previous round),
// giving the inclusive prefix; the exclusive prefix is that shifted by one.
// Returns the number of rounds.
int exclusive_tree(const double* x, int64_t nc, int64_t w, double* out) {
    std::vector<double> cur(x, x + nc * w), nxt((size_t)(nc * w));
    int rounds = 0;
    for (int64_t d = 1; d < nc; d <<= 1) {
        for (int64_t c = 0; c < nc; ++c)
            for (int64_t e = 0; e < w; ++e)
                nxt[c * w + e] = cur[c * w + e] + (c >= d ? cur[(c - d) * w + e] : 0.0);
        cur.swap(nxt);
        ++rounds;
    }
    for (int64_t e = 0; e < w; ++e) out[e] = 0.0;
    for (int64_t c = 1; c < nc; ++c)
        for (int64_t e = 0; e < w; ++e) out[c * w + e] = cur[(c - 1) * w + e];
    return rounds;
}

}  // namespace

extern "C" {

int kor_packed_dim(int p) { return (int)packed_dim_i(p); }

void kor_normalize(const double* x, int p, double* u) { normalize(x, p, u); }

void kor_lift(const double* u, int p, double* psi) { lift(u, p, psi); }

// The plain definition, every row:
//   o_t = sum_{s<=t} (qh_t . kh_s)^2 v_s / sum_{s<=t} (qh_t . kh_s)^2.
int kor_forward_plain(const double* q, const double* k, const double* v, int B, int H, int T,
                      int p, int dv, double* o, int nthreads) {
    const int64_t heads = (int64_t)B * H;
    for_heads(heads, nthreads, [&](int64_t bh) {
        const double* qh = q + bh * T * p;
        const double* kh = k + bh * T * p;
        const double* vh = v + bh * T * dv;
        double* oh = o + bh * T * dv;
        std::vector<double> qu = normalized_rows(qh, T, p), ku = normalized_rows(kh, T, p);
        std::vector<double> num((size_t)dv);
        for (int t = 0; t < T; ++t) {
            std::fill(num.begin(), num.end(), 0.0);
            double den = 0.0;
            for (int s = 0; s <= t; ++s) {
                double c = dot(&qu[(size_t)t * p], &ku[(size_t)s * p], p);
                double w = c * c;
                den += w;
                for (int j = 0; j < dv; ++j) num[j] += w * vh[(int64_t)s * dv + j];
            }
            for (int j = 0; j < dv; ++j) oh[(int64_t)t * dv + j] = den > 0.0 ? num[j] / den : 0.0;
        }
    });
    return 0;
}

// The plain definition for selected rows only: row r is head bh[r] (= b*H + h),
// position t[r]; its dv outputs go to out[r*dv ...].  Cost O(t (p + dv)) per row.
int kor_forward_plain_rows(const double* q, const double* k, const double* v, int B, int H,
                           int T, int p, int dv, const int64_t* bh, const int64_t* t, int64_t nrows,
                           double* out, int nthreads) {
    for_heads(nrows, nthreads, [&](int64_t r) {
        const double* qh = q + bh[r] * T * p;
        const double* kh = k + bh[r] * T * p;
        const double* vh = v + bh[r] * T * dv;
        std::vector<double> qu((size_t)p), ku((size_t)p), num((size_t)dv, 0.0);
        normalize(qh + t[r] * p, p, qu.data());
        double den = 0.0;
        for (int64_t s = 0; s <= t[r]; ++s) {
            normalize(kh + s * p, p, ku.data());
            double c = dot(qu.data(), ku.data(), p);
            double w = c * c;
            den += w;
            for (int j = 0; j < dv; ++j) num[j] += w * vh[s * dv + j];
        }
        for (int j = 0; j < dv; ++j) out[r * dv + j] = den > 0.0 ? num[j] / den : 0.0;
    });
    (void)B;
    (void)H;
    return 0;
}

// Token-recurrent form in the explicit packed lift:
//   S += psi(kh_t) v_t^T,  z += psi(kh_t),  o_t = psi(qh_t)^T S / psi(qh_t)^T z.
// S0 [B,H,n,dv] / z0 [B,H,n] are the optional initial state (NULL = zero);
// S_final / z_final receive the state after the last token (NULL = skipped).
int kor_forward_recurrent(const double* q, const double* k, const double* v, int B, int H, int T,
                          int p, int dv, const double* S0, const double* z0, double* o,
                          double* S_final, double* z_final, int nthreads) {
    const int64_t heads = (int64_t)B * H, n = packed_dim_i(p);
    for_heads(heads, nthreads, [&](int64_t bh) {
        std::vector<double> S((size_t)(n * dv), 0.0), z((size_t)n, 0.0);
        if (S0) std::copy(S0 + bh * n * dv, S0 + (bh + 1) * n * dv, S.begin());
        if (z0) std::copy(z0 + bh * n, z0 + (bh + 1) * n, z.begin());
        std::vector<double> u((size_t)p), pk((size_t)n), pq((size_t)n), num((size_t)dv);
        for (int t = 0; t < T; ++t) {
            const double* kt = k + (bh * T + t) * p;
            const double* qt = q + (bh * T + t) * p;
            const double* vt = v + (bh * T + t) * dv;
            normalize(kt, p, u.data());
            lift(u.data(), p, pk.data());
            for (int64_t a = 0; a < n; ++a) {
                for (int j = 0; j < dv; ++j) S[a * dv + j] += pk[a] * vt[j];
                z[a] += pk[a];
            }
            normalize(qt, p, u.data());
            lift(u.data(), p, pq.data());
            std::fill(num.begin(), num.end(), 0.0);
            for (int64_t a = 0; a < n; ++a)
                for (int j = 0; j < dv; ++j) num[j] += pq[a] * S[a * dv + j];
            double den = dot(pq.data(), z.data(), n);
            double* ot = o + (bh * T + t) * dv;
            for (int j = 0; j < dv; ++j) ot[j] = den > 0.0 ? num[j] / den : 0.0;
        }
        if (S_final) std::copy(S.begin(), S.end(), S_final + bh * n * dv);
        if (z_final) std::copy(z.begin(), z.end(), z_final + bh * n);
    });
    return 0;
}

// Per-chunk local states of chunk length C (the last chunk may be shorter):
//   S_loc[c] = sum_{s in chunk c} psi(kh_s) v_s^T,  z_loc[c] = sum psi(kh_s).
// Outputs S_loc [B,H,NC,n,dv], z_loc [B,H,NC,n], NC = ceil(T / C).
int kor_chunk_states(const double* k, const double* v, int B, int H, int T, int p, int dv, int C,
                     double* S_loc, double* z_loc, int nthreads) {
    const int64_t heads = (int64_t)B * H, n = packed_dim_i(p);
    const int64_t NC = (T + C - 1) / C;
    for_heads(heads, nthreads, [&](int64_t bh) {
        std::vector<double> u((size_t)p), pk((size_t)n);
        for (int64_t c = 0; c < NC; ++c) {
            double* S = S_loc + (bh * NC + c) * n * dv;
            double* z = z_loc + (bh * NC + c) * n;
            std::fill(S, S + n * dv, 0.0);
            std::fill(z, z + n, 0.0);
            for (int64_t s = c * C; s < std::min<int64_t>((c + 1) * C, T); ++s) {
                normalize(k + (bh * T + s) * p, p, u.data());
                lift(u.data(), p, pk.data());
                const double* vs = v + (bh * T + s) * dv;
                for (int64_t a = 0; a < n; ++a) {
                    for (int j = 0; j < dv; ++j) S[a * dv + j] += pk[a] * vs[j];
                    z[a] += pk[a];
                }
            }
        }
    });
    return 0;
}

// Exclusive prefix of chunk states over the chunk axis, mode 0 = sequential
// (N_C steps), mode 1 = log-depth scan (ceil(log2 N_C) rounds).
// Returns the number of rounds (steps) taken for one head.
int kor_scan_exclusive(const double* S_loc, const double* z_loc, int B, int H, int NC, int n,
                       int dv, int mode, double* S_prefix, double* z_prefix, int nthreads) {
    const int64_t heads = (int64_t)B * H;
    std::vector<int> rounds((size_t)std::max<int64_t>(heads, 1), 0);
    for_heads(heads, nthreads, [&](int64_t bh) {
        const int64_t ws = (int64_t)n * dv;
        if (mode == 0) {
            exclusive_sequential(S_loc + bh * NC * ws, NC, ws, S_prefix + bh * NC * ws);
            exclusive_sequential(z_loc + bh * NC * n, NC, n, z_prefix + bh * NC * n);
            rounds[bh] = NC;
        } else {
            rounds[bh] = exclusive_tree(S_loc + bh * NC * ws, NC, ws, S_prefix + bh * NC * ws);
            exclusive_tree(z_loc + bh * NC * n, NC, n, z_prefix + bh * NC * n);
        }
    });
    return heads > 0 ? rounds[0] : 0;
}

// Chunked form: local chunk states, exclusive prefix over chunks (mode as in
// kor_scan_exclusive) seeded with the optional initial state, then for each
// token t of chunk c
//   num = psi(qh_t)^T P_c + sum_{s in c, s<=t} <psi(qh_t), psi(kh_s)> v_s
//   den = psi(qh_t)^T Pz_c + sum_{s in c, s<=t} <psi(qh_t), psi(kh_s)>
//   o_t = num / den.
// The intra-chunk scores use the lifted features, as the chunk output
// combines the prefix with the local C x C causal pattern.
int kor_forward_chunked(const double* q, const double* k, const double* v, int B, int H, int T,
                        int p, int dv, int C, int mode, const double* S0, const double* z0,
                        double* o, double* S_final, double* z_final, int nthreads) {
    const int64_t heads = (int64_t)B * H, n = packed_dim_i(p);
    const int64_t NC = (T + C - 1) / C, ws = n * dv;
    if (T <= 0) {
        for (int64_t bh = 0; bh < heads; ++bh) {
            if (S_final)
                for (int64_t e = 0; e < ws; ++e) S_final[bh * ws + e] = S0 ? S0[bh * ws + e] : 0.0;
            if (z_final)
                for (int64_t e = 0; e < n; ++e) z_final[bh * n + e] = z0 ? z0[bh * n + e] : 0.0;
        }
        return 0;
    }
    for_heads(heads, nthreads, [&](int64_t bh) {
        // 1. local chunk states
        std::vector<double> Sl((size_t)(NC * ws)), zl((size_t)(NC * n));
        kor_chunk_states(k + bh * T * p, v + bh * T * dv, 1, 1, T, p, dv, C, Sl.data(), zl.data(), 1);
        // 2. exclusive prefix, then add the initial state
        std::vector<double> P((size_t)(NC * ws)), Pz((size_t)(NC * n));
        kor_scan_exclusive(Sl.data(), zl.data(), 1, 1, (int)NC, (int)n, dv, mode, P.data(), Pz.data(), 1);
        if (S0)
            for (int64_t c = 0; c < NC; ++c)
                for (int64_t e = 0; e < ws; ++e) P[c * ws + e] += S0[bh * ws + e];
        if (z0)
            for (int64_t c = 0; c < NC; ++c)
                for (int64_t e = 0; e < n; ++e) Pz[c * n + e] += z0[bh * n + e];
        // 3. per-chunk output: prefix readout + local causal part
        std::vector<double> u((size_t)p), pq((size_t)n), num((size_t)dv);
        std::vector<double> pk((size_t)(C * n));
        for (int64_t c = 0; c < NC; ++c) {
            const int64_t t0 = c * C, t1 = std::min<int64_t>(t0 + C, T);
            for (int64_t s = t0; s < t1; ++s) {
                normalize(k + (bh * T + s) * p, p, u.data());
                lift(u.data(), p, &pk[(size_t)((s - t0) * n)]);
            }
            for (int64_t t = t0; t < t1; ++t) {
                normalize(q + (bh * T + t) * p, p, u.data());
                lift(u.data(), p, pq.data());
                std::fill(num.begin(), num.end(), 0.0);
                for (int64_t a = 0; a < n; ++a)
                    for (int j = 0; j < dv; ++j) num[j] += pq[a] * P[c * ws + a * dv + j];
                double den = dot(pq.data(), &Pz[(size_t)(c * n)], n);
                for (int64_t s = t0; s <= t; ++s) {
                    double w = dot(pq.data(), &pk[(size_t)((s - t0) * n)], n);
                    den += w;
                    for (int j = 0; j < dv; ++j) num[j] += w * v[(bh * T + s) * dv + j];
                }
                double* ot = o + (bh * T + t) * dv;
                for (int j = 0; j < dv; ++j) ot[j] = den > 0.0 ? num[j] / den : 0.0;
            }
        }
        // 4. final state = last prefix + last local state (+ initial state, already in P)
        if (S_final)
            for (int64_t e = 0; e < ws; ++e)
                S_final[bh * ws + e] = P[(NC - 1) * ws + e] + Sl[(NC - 1) * ws + e];
        if (z_final)
            for (int64_t e = 0; e < n; ++e)
                z_final[bh * n + e] = Pz[(NC - 1) * n + e] + zl[(NC - 1) * n + e];
    });
    return 0;
}

}  // extern "C"

namespace {

// ---------------------------------------------------------------- block lifts
// The two reduced PSD families ("two reduced PSD families" paragraph, after
// the state-size discussion): g divides p, m = p/g, and each unit vector u
// (the projected query or key) is cut into g blocks u_1..u_g of length m,
// u_a = (u[a m], ..., u[a m + m - 1]).
//   family 1, KATA-Sigma-g: psi(u) = sum_a u_a u_a^T, one m x m PSD matrix
//     packed in m(m+1)/2 coordinates; <psi(q), psi(k)>_F = sum_{a,b} (q_a.k_b)^2.
//   family 2, KATA-M-g: psi(u) = (u_1 u_1^T, ..., u_g u_g^T), g packed m x m
//     matrices one after another, g m(m+1)/2 coordinates;
//     <psi(q), psi(k)> = sum_a (q_a.k_a)^2.
//   family 0: the full rank-one lift (g must be 1).
// Packing inside an m x m block as for the full lift (upper triangle row by
// row, off-diagonal coordinates times sqrt 2).

// Width of the lift, or -1 if (family, g) does not fit p.
int block_dim_i(int p, int family, int g) {
    if (p <= 0 || g <= 0 || p % g != 0) return -1;
    const int m = p / g;
    if (family == 0) return g == 1 ? (int)packed_dim_i(p) : -1;
    if (family == 1) return (int)packed_dim_i(m);
    if (family == 2) return g * (int)packed_dim_i(m);
    return -1;
}

void lift_block(const double* u, int p, int family, int g, double* psi) {
    const int m = p / g;
    const double r2 = std::sqrt(2.0);
    if (family == 2) {
        for (int a = 0; a < g; ++a) lift(u + a * m, m, psi + a * packed_dim_i(m));
        return;
    }
    // family 0 (g = 1) and family 1: the block outer products summed
    for (int i = 0; i < m; ++i)
        for (int j = i; j < m; ++j) {
            double sum = 0.0;
            for (int a = 0; a < g; ++a) sum += u[a * m + i] * u[a * m + j];
            psi[pidx(m, i, j)] = (i == j) ? sum : r2 * sum;
        }
}

// The kernel of two unit vectors written from its definition (block dot
// products squared), not through the lift.
double block_kernel(const double* qu, const double* ku, int p, int family, int g) {
    const int m = p / g;
    double w = 0.0;
    for (int a = 0; a < g; ++a)
        for (int b = 0; b < g; ++b) {
            if (family != 1 && a != b) continue;
            const double c = dot(qu + a * m, ku + b * m, m);
            w += c * c;
        }
    return w;
}

}  // namespace

extern "C" {

int kor_block_dim(int p, int family, int g) { return block_dim_i(p, family, g); }

void kor_lift_block(const double* u, int p, int family, int g, double* psi) {
    lift_block(u, p, family, g, psi);
}

// The plain definition with a block lift, every row:
//   o_t = sum_{s<=t} w(qh_t, kh_s) v_s / sum_{s<=t} w(qh_t, kh_s),
//   w = sum_{a,b} (q_a.k_b)^2 (Sigma-g) or sum_a (q_a.k_a)^2 (M-g).
// Returns -1 if (family, g) does not fit p.
int kor_forward_plain_block(const double* q, const double* k, const double* v, int B, int H, int T,
                            int p, int dv, int family, int g, double* o, int nthreads) {
    if (block_dim_i(p, family, g) < 0) return -1;
    const int64_t heads = (int64_t)B * H;
    for_heads(heads, nthreads, [&](int64_t bh) {
        const double* vh = v + bh * T * dv;
        double* oh = o + bh * T * dv;
        std::vector<double> qu = normalized_rows(q + bh * T * p, T, p), ku = normalized_rows(k + bh * T * p, T, p);
        std::vector<double> num((size_t)dv);
        for (int t = 0; t < T; ++t) {
            std::fill(num.begin(), num.end(), 0.0);
            double den = 0.0;
            for (int s = 0; s <= t; ++s) {
                const double w = block_kernel(&qu[(size_t)t * p], &ku[(size_t)s * p], p, family, g);
                den += w;
                for (int j = 0; j < dv; ++j) num[j] += w * vh[(int64_t)s * dv + j];
            }
            for (int j = 0; j < dv; ++j) oh[(int64_t)t * dv + j] = den > 0.0 ? num[j] / den : 0.0;
        }
    });
    return 0;
}

// Token recurrence in the packed block lift (state [n_psi, dv], z [n_psi]):
//   S += psi(kh_t) v_t^T,  z += psi(kh_t),  o_t = psi(qh_t)^T S / psi(qh_t)^T z,
// optional initial / final state as in kor_forward_recurrent.  Returns -1 if
// (family, g) does not fit p.
int kor_forward_recurrent_block(const double* q, const double* k, const double* v, int B, int H, int T,
                                int p, int dv, int family, int g, const double* S0, const double* z0,
                                double* o, double* S_final, double* z_final, int nthreads) {
    const int64_t n = block_dim_i(p, family, g);
    if (n < 0) return -1;
    const int64_t heads = (int64_t)B * H;
    for_heads(heads, nthreads, [&](int64_t bh) {
        std::vector<double> S((size_t)(n * dv), 0.0), z((size_t)n, 0.0);
        if (S0) std::copy(S0 + bh * n * dv, S0 + (bh + 1) * n * dv, S.begin());
        if (z0) std::copy(z0 + bh * n, z0 + (bh + 1) * n, z.begin());
        std::vector<double> u((size_t)p), pk((size_t)n), pq((size_t)n), num((size_t)dv);
        for (int t = 0; t < T; ++t) {
            const double* vt = v + (bh * T + t) * dv;
            normalize(k + (bh * T + t) * p, p, u.data());
            lift_block(u.data(), p, family, g, pk.data());
            for (int64_t a = 0; a < n; ++a) {
                for (int j = 0; j < dv; ++j) S[a * dv + j] += pk[a] * vt[j];
                z[a] += pk[a];
            }
            normalize(q + (bh * T + t) * p, p, u.data());
            lift_block(u.data(), p, family, g, pq.data());
            std::fill(num.begin(), num.end(), 0.0);
            for (int64_t a = 0; a < n; ++a)
                for (int j = 0; j < dv; ++j) num[j] += pq[a] * S[a * dv + j];
            const double den = dot(pq.data(), z.data(), n);
            double* ot = o + (bh * T + t) * dv;
            for (int j = 0; j < dv; ++j) ot[j] = den > 0.0 ? num[j] / den : 0.0;
        }
        if (S_final) std::copy(S.begin(), S.end(), S_final + bh * n * dv);
        if (z_final) std::copy(z.begin(), z.end(), z_final + bh * n);
    });
    return 0;
}

// ---------------------------------------------------------------- backward
// Gradient of the plain definition.  The pages give no backward algorithm
// (the training use of the forward is named in the abstract); this is the
// chain rule through the definition
//   o_t = N_t / D_t,  N_t = sum_{s<=t} w_ts v_s,  D_t = sum_{s<=t} w_ts,
//   w_ts = c_ts^2,  c_ts = qh_t . kh_s,  qh = q / ||q||,  kh = k / ||k||.
// With G_t = dL/do_t:
//   dL/dv_s  = sum_{t>=s} (w_ts / D_t) G_t
//   dL/dw_ts = G_t . (v_s - o_t) / D_t
//   dL/dc_ts = 2 c_ts dL/dw_ts
//   dL/dqh_t = sum_{s<=t} dL/dc_ts kh_s,   dL/dkh_s = sum_{t>=s} dL/dc_ts qh_t
//   dL/dq_t  = (dL/dqh_t - (qh_t . dL/dqh_t) qh_t) / ||q_t||   (k likewise).
// A row with D_t = 0 (its output is fixed at zero) passes no gradient, and a
// zero q or k vector (where the projection has no derivative) receives none.
int kor_backward_plain(const double* q, const double* k, const double* v, const double* dO, int B, int H,
                       int T, int p, int dv, double* dq, double* dk, double* dvv, int nthreads) {
    const int64_t heads = (int64_t)B * H;
    for_heads(heads, nthreads, [&](int64_t bh) {
        const double* qh = q + bh * T * p;
        const double* kh = k + bh * T * p;
        const double* vh = v + bh * T * dv;
        const double* Gh = dO + bh * T * dv;
        std::vector<double> qu = normalized_rows(qh, T, p), ku = normalized_rows(kh, T, p);
        std::vector<double> gq((size_t)T * p, 0.0), gk((size_t)T * p, 0.0), gv((size_t)T * dv, 0.0);
        std::vector<double> o((size_t)dv);
        for (int t = 0; t < T; ++t) {
            // forward row t
            double den = 0.0;
            std::fill(o.begin(), o.end(), 0.0);
            for (int s = 0; s <= t; ++s) {
                const double c = dot(&qu[(size_t)t * p], &ku[(size_t)s * p], p);
                den += c * c;
                for (int j = 0; j < dv; ++j) o[j] += c * c * vh[(int64_t)s * dv + j];
            }
            if (!(den > 0.0)) continue;
            for (int j = 0; j < dv; ++j) o[j] /= den;
            // backward row t
            const double* G = Gh + (int64_t)t * dv;
            for (int s = 0; s <= t; ++s) {
                const double c = dot(&qu[(size_t)t * p], &ku[(size_t)s * p], p);
                const double w = c * c;
                double gw = 0.0;
                for (int j = 0; j < dv; ++j) {
                    gv[(size_t)s * dv + j] += w / den * G[j];
                    gw += G[j] * (vh[(int64_t)s * dv + j] - o[j]);
                }
                gw /= den;
                const double gc = 2.0 * c * gw;
                for (int i = 0; i < p; ++i) {
                    gq[(size_t)t * p + i] += gc * ku[(size_t)s * p + i];
                    gk[(size_t)s * p + i] += gc * qu[(size_t)t * p + i];
                }
            }
        }
        // through the unit-sphere projections
        auto project = [&](const double* x, const double* u, const double* gu, double* gx) {
            double nrm = 0.0;
            for (int i = 0; i < p; ++i) nrm += x[i] * x[i];
            nrm = std::sqrt(nrm);
            if (!(nrm > 0.0)) {
                for (int i = 0; i < p; ++i) gx[i] = 0.0;
                return;
            }
            const double ug = dot(u, gu, p);
            for (int i = 0; i < p; ++i) gx[i] = (gu[i] - ug * u[i]) / nrm;
        };
        for (int t = 0; t < T; ++t) {
            project(qh + (int64_t)t * p, &qu[(size_t)t * p], &gq[(size_t)t * p], dq + (bh * T + t) * p);
            project(kh + (int64_t)t * p, &ku[(size_t)t * p], &gk[(size_t)t * p], dk + (bh * T + t) * p);
        }
        std::copy(gv.begin(), gv.end(), dvv + bh * T * dv);
    });
    return 0;
}

// ---------------------------------------------------------------- gated prefix
// The Gated variant ("a Gated prefix adds the learned gate"; its recurrence
// is in an appendix the pages do not contain).  Reading: one scalar gate
// gamma_t in [0, 1] per head and token scales the running state before the
// token's own term is added,
//   S_t = gamma_t S_{t-1} + psi(kh_t) v_t^T,   z_t = gamma_t z_{t-1} + psi(kh_t),
// read out as before, o_t = psi(qh_t)^T S_t / psi(qh_t)^T z_t.  gamma = 1 is the
// ungated forward; gamma_t = 0 forgets everything before t.  The gate is an
// input, [B, H, T].

// The definition: o_t = sum_{s<=t} d_ts w_ts v_s / sum_{s<=t} d_ts w_ts with
// w_ts = (qh_t . kh_s)^2 and d_ts = prod_{r=s+1..t} gamma_r (d_tt = 1).
int kor_forward_plain_gated(const double* q, const double* k, const double* v, const double* gate, int B, int H,
                            int T, int p, int dv, double* o, int nthreads) {
    const int64_t heads = (int64_t)B * H;
    for_heads(heads, nthreads, [&](int64_t bh) {
        const double* vh = v + bh * T * dv;
        const double* gh = gate + bh * T;
        std::vector<double> qu = normalized_rows(q + bh * T * p, T, p), ku = normalized_rows(k + bh * T * p, T, p);
        std::vector<double> num((size_t)dv);
        for (int t = 0; t < T; ++t) {
            std::fill(num.begin(), num.end(), 0.0);
            double den = 0.0, decay = 1.0;
            for (int s = t; s >= 0; --s) {
                if (s < t) decay *= gh[s + 1];
                const double c = dot(&qu[(size_t)t * p], &ku[(size_t)s * p], p);
                const double w = decay * c * c;
                den += w;
                for (int j = 0; j < dv; ++j) num[j] += w * vh[(int64_t)s * dv + j];
            }
            for (int j = 0; j < dv; ++j) o[(bh * T + t) * dv + j] = den > 0.0 ? num[j] / den : 0.0;
        }
    });
    return 0;
}

// The gated token recurrence, with optional initial / final state as in
// kor_forward_recurrent (the initial state is scaled by gamma_0 too).
int kor_forward_recurrent_gated(const double* q, const double* k, const double* v, const double* gate, int B, int H,
                                int T, int p, int dv, const double* S0, const double* z0, double* o,
                                double* S_final, double* z_final, int nthreads) {
    const int64_t heads = (int64_t)B * H, n = packed_dim_i(p);
    for_heads(heads, nthreads, [&](int64_t bh) {
        std::vector<double> S((size_t)(n * dv), 0.0), z((size_t)n, 0.0);
        if (S0) std::copy(S0 + bh * n * dv, S0 + (bh + 1) * n * dv, S.begin());
        if (z0) std::copy(z0 + bh * n, z0 + (bh + 1) * n, z.begin());
        std::vector<double> u((size_t)p), pk((size_t)n), pq((size_t)n), num((size_t)dv);
        for (int t = 0; t < T; ++t) {
            const double gam = gate[bh * T + t];
            const double* vt = v + (bh * T + t) * dv;
            normalize(k + (bh * T + t) * p, p, u.data());
            lift(u.data(), p, pk.data());
            for (int64_t a = 0; a < n; ++a) {
                for (int j = 0; j < dv; ++j) S[a * dv + j] = gam * S[a * dv + j] + pk[a] * vt[j];
                z[a] = gam * z[a] + pk[a];
            }
            normalize(q + (bh * T + t) * p, p, u.data());
            lift(u.data(), p, pq.data());
            std::fill(num.begin(), num.end(), 0.0);
            for (int64_t a = 0; a < n; ++a)
                for (int j = 0; j < dv; ++j) num[j] += pq[a] * S[a * dv + j];
            const double den = dot(pq.data(), z.data(), n);
            for (int j = 0; j < dv; ++j) o[(bh * T + t) * dv + j] = den > 0.0 ? num[j] / den : 0.0;
        }
        if (S_final) std::copy(S.begin(), S.end(), S_final + bh * n * dv);
        if (z_final) std::copy(z.begin(), z.end(), z_final + bh * n);
    });
    return 0;
}

// Exclusive gated prefix over `nc` items of width `w`: item c carries the
// pair (a_c, x_c), and prefix_0 = 0, prefix_{c+1} = a_c prefix_c + x_c.  Pairs
// compose associatively: (a1, x1) then (a2, x2) = (a1 a2, a2 x1 + x2).
// mode 0: one step per item; mode 1: ceil(log2 nc) rounds, each combining
// every item with the item 2^d places earlier (Hillis-Steele on the pairs),
// giving inclusive prefixes that are shifted by one.  Returns the rounds.
static int gated_exclusive(const double* a, const double* x, int64_t nc, int64_t w, int mode, double* out) {
    if (mode == 0) {
        std::vector<double> run((size_t)w, 0.0);
        for (int64_t c = 0; c < nc; ++c) {
            for (int64_t e = 0; e < w; ++e) out[c * w + e] = run[e];
            for (int64_t e = 0; e < w; ++e) run[e] = a[c] * run[e] + x[c * w + e];
        }
        return (int)nc;
    }
    std::vector<double> ca(a, a + nc), cx(x, x + nc * w), na((size_t)nc), nx((size_t)(nc * w));
    int rounds = 0;
    for (int64_t d = 1; d < nc; d <<= 1) {
        for (int64_t c = 0; c < nc; ++c) {
            if (c >= d) {
                // (ca[c-d], cx[c-d]) then (ca[c], cx[c])
                na[c] = ca[c - d] * ca[c];
                for (int64_t e = 0; e < w; ++e) nx[c * w + e] = ca[c] * cx[(c - d) * w + e] + cx[c * w + e];
            } else {
                na[c] = ca[c];
                for (int64_t e = 0; e < w; ++e) nx[c * w + e] = cx[c * w + e];
            }
        }
        ca.swap(na);
        cx.swap(nx);
        ++rounds;
    }
    for (int64_t e = 0; e < w; ++e) out[e] = 0.0;
    for (int64_t c = 1; c < nc; ++c)
        for (int64_t e = 0; e < w; ++e) out[c * w + e] = cx[(c - 1) * w + e];
    return rounds;
}

int kor_scan_exclusive_gated(const double* a, const double* x, int heads, int nc, int w, int mode, double* out,
                             int nthreads) {
    std::vector<int> rounds((size_t)std::max(heads, 1), 0);
    for_heads(heads, nthreads, [&](int64_t h) {
        rounds[h] = gated_exclusive(a + h * nc, x + h * (int64_t)nc * w, nc, w, mode, out + h * (int64_t)nc * w);
    });
    return heads > 0 ? rounds[0] : 0;
}

// Gated chunked form.  Chunk c covers tokens [c C, min(c C + C, T)):
//   local state  S_loc_c = sum_{s in c} (prod_{r=s+1..end_c} gamma_r) psi(kh_s) v_s^T  (z likewise),
//   chunk decay  a_c = prod_{r in c} gamma_r,
//   prefix       P_0 = S0, P_{c+1} = a_c P_c + S_loc_c (gated scan, `mode`),
//   output       num_t = (prod_{r=c C..t} gamma_r) psi(qh_t)^T P_c
//                        + sum_{s in c, s<=t} (prod_{r=s+1..t} gamma_r) w_ts v_s,  den likewise.
int kor_forward_chunked_gated(const double* q, const double* k, const double* v, const double* gate, int B, int H,
                              int T, int p, int dv, int C, int mode, const double* S0, const double* z0, double* o,
                              double* S_final, double* z_final, int nthreads) {
    const int64_t heads = (int64_t)B * H, n = packed_dim_i(p), ws = n * dv;
    const int64_t NC = (T + C - 1) / C;
    for_heads(heads, nthreads, [&](int64_t bh) {
        const double* gh = gate + bh * T;
        // 1. local states and chunk decays; the initial state enters as an
        //    extra leading item (decay 1) so the scan adds it to every prefix
        const int64_t items = NC + 1;
        std::vector<double> a((size_t)items, 1.0), X((size_t)(items * ws), 0.0), Z((size_t)(items * n), 0.0);
        if (S0) std::copy(S0 + bh * ws, S0 + (bh + 1) * ws, X.begin());
        if (z0) std::copy(z0 + bh * n, z0 + (bh + 1) * n, Z.begin());
        std::vector<double> u((size_t)p), pk((size_t)n);
        for (int64_t c = 0; c < NC; ++c) {
            const int64_t t0 = c * C, t1 = std::min<int64_t>(t0 + C, T);
            double* Xc = &X[(size_t)((c + 1) * ws)];
            double* Zc = &Z[(size_t)((c + 1) * n)];
            double chunk_decay = 1.0;
            for (int64_t s = t0; s < t1; ++s) chunk_decay *= gh[s];
            a[(size_t)(c + 1)] = chunk_decay;
            for (int64_t s = t0; s < t1; ++s) {
                double decay = 1.0;  // prod_{r=s+1..t1-1} gamma_r
                for (int64_t r = s + 1; r < t1; ++r) decay *= gh[r];
                normalize(k + (bh * T + s) * p, p, u.data());
                lift(u.data(), p, pk.data());
                for (int64_t e = 0; e < n; ++e) {
                    for (int j = 0; j < dv; ++j) Xc[e * dv + j] += decay * pk[e] * v[(bh * T + s) * dv + j];
                    Zc[e] += decay * pk[e];
                }
            }
        }
        // 2. gated exclusive prefix over [initial state, chunk 0, ..., chunk NC-1]:
        //    item c+1's prefix is the state entering chunk c
        std::vector<double> PX((size_t)(items * ws)), PZ((size_t)(items * n));
        gated_exclusive(a.data(), X.data(), items, ws, mode, PX.data());
        gated_exclusive(a.data(), Z.data(), items, n, mode, PZ.data());
        // 3. per-chunk output
        std::vector<double> pq((size_t)n), num((size_t)dv), qu((size_t)p), ku((size_t)p);
        for (int64_t c = 0; c < NC; ++c) {
            const int64_t t0 = c * C, t1 = std::min<int64_t>(t0 + C, T);
            const double* Pc = &PX[(size_t)((c + 1) * ws)];
            const double* Pzc = &PZ[(size_t)((c + 1) * n)];
            double head_decay = 1.0;  // prod_{r=t0..t} gamma_r
            for (int64_t t = t0; t < t1; ++t) {
                head_decay *= gh[t];
                normalize(q + (bh * T + t) * p, p, qu.data());
                lift(qu.data(), p, pq.data());
                std::fill(num.begin(), num.end(), 0.0);
                for (int64_t e = 0; e < n; ++e)
                    for (int j = 0; j < dv; ++j) num[j] += head_decay * pq[e] * Pc[e * dv + j];
                double den = head_decay * dot(pq.data(), Pzc, n);
                for (int64_t s = t0; s <= t; ++s) {
                    double decay = 1.0;
                    for (int64_t r = s + 1; r <= t; ++r) decay *= gh[r];
                    normalize(k + (bh * T + s) * p, p, ku.data());
                    const double cc = dot(qu.data(), ku.data(), p);
                    const double w = decay * cc * cc;
                    den += w;
                    for (int j = 0; j < dv; ++j) num[j] += w * v[(bh * T + s) * dv + j];
                }
                for (int j = 0; j < dv; ++j) o[(bh * T + t) * dv + j] = den > 0.0 ? num[j] / den : 0.0;
            }
        }
        // 4. final state: the prefix after the last chunk
        if (S_final || z_final) {
            std::vector<double> Sf((size_t)ws), zf((size_t)n);
            const double al = a[(size_t)NC];
            for (int64_t e = 0; e < ws; ++e) Sf[e] = al * PX[(size_t)(NC * ws + e)] + X[(size_t)(NC * ws + e)];
            for (int64_t e = 0; e < n; ++e) zf[e] = al * PZ[(size_t)(NC * n + e)] + Z[(size_t)(NC * n + e)];
            if (S_final) std::copy(Sf.begin(), Sf.end(), S_final + bh * ws);
            if (z_final) std::copy(zf.begin(), zf.end(), z_final + bh * n);
        }
    });
    return 0;
}

// ---------------------------------------------------------------- sampled rows
// The block-lift and gated definitions for selected rows only (row r: head
// bh[r] = b*H + h, position t[r]), O(t (p + dv)) per row, for checks at sizes
// where every row would be too slow.  Outputs [nrows, dv].
int kor_forward_plain_block_rows(const double* q, const double* k, const double* v, int B, int H, int T, int p, int dv,
                                 int family, int g, const int64_t* bh, const int64_t* t, int64_t nrows, double* out,
                                 int nthreads) {
    if (block_dim_i(p, family, g) < 0) return -1;
    for_heads(nrows, nthreads, [&](int64_t r) {
        std::vector<double> qu((size_t)p), ku((size_t)p), num((size_t)dv, 0.0);
        normalize(q + (bh[r] * T + t[r]) * p, p, qu.data());
        double den = 0.0;
        for (int64_t s = 0; s <= t[r]; ++s) {
            normalize(k + (bh[r] * T + s) * p, p, ku.data());
            const double w = block_kernel(qu.data(), ku.data(), p, family, g);
            den += w;
            for (int j = 0; j < dv; ++j) num[j] += w * v[(bh[r] * T + s) * dv + j];
        }
        for (int j = 0; j < dv; ++j) out[r * dv + j] = den > 0.0 ? num[j] / den : 0.0;
    });
    (void)B;
    (void)H;
    return 0;
}

int kor_forward_plain_gated_rows(const double* q, const double* k, const double* v, const double* gate, int B, int H,
                                 int T, int p, int dv, const int64_t* bh, const int64_t* t, int64_t nrows, double* out,
                                 int nthreads) {
    for_heads(nrows, nthreads, [&](int64_t r) {
        std::vector<double> qu((size_t)p), ku((size_t)p), num((size_t)dv, 0.0);
        const double* gh = gate + bh[r] * T;
        normalize(q + (bh[r] * T + t[r]) * p, p, qu.data());
        double den = 0.0, decay = 1.0;
        for (int64_t s = t[r]; s >= 0; --s) {
            if (s < t[r]) decay *= gh[s + 1];
            normalize(k + (bh[r] * T + s) * p, p, ku.data());
            const double c = dot(qu.data(), ku.data(), p);
            const double w = decay * c * c;
            den += w;
            for (int j = 0; j < dv; ++j) num[j] += w * v[(bh[r] * T + s) * dv + j];
        }
        for (int j = 0; j < dv; ++j) out[r * dv + j] = den > 0.0 ? num[j] / den : 0.0;
    });
    (void)B;
    (void)H;
    return 0;
}

}  // extern "C"
