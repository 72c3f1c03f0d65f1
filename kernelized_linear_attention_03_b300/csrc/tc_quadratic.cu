// Flash-style O(T^2) KATA forward on the tcgen05 tensor cores (bf16 inputs,
// fp32 accumulation): the flash-attention-style operating point of the
// paper's abstract.  For one head and a tile of 128 queries, over key tiles
// of 128 up to the diagonal:
//   S = Q Kh^T            (tcgen05, A = raw queries, B = unit keys, D in TMEM)
//   P = S o S, masked     (CUDA cores: squared scores, causal mask s <= t,
//                          packed to bf16 in place in TMEM)
//   O += P [V | 1]        (tcgen05, A = P from TMEM, B = the value tile and a
//                          constant ones column, D in TMEM)
//   o = O[:, :dv] / O[:, 64]
// Only keys are put on the unit sphere: a query's norm scales numerator and
// denominator alike and cancels.  Scores of unit keys with a fixed query are
// bounded, so no running maximum or rescale is needed.
//
// Gated form (GATED): every weight also carries the decay of the gates after
// its key, G(t, s) = prod_{r=s+1..t} gamma_r.  With L_t the sum of log gamma_r
// since the last zero gate z_t <= t (both from gate_prefix_kernel),
// G(t, s) = [z_t <= s] exp(L_t - L_s).  A factor of a whole row cancels between
// numerator and denominator, so when the CTA's query rows share their last
// zero gate (none inside its tiles) and their decay is moderate (L at the
// first row minus L at the last below kSpanMax), each weight takes the key's
// factor exp(R - L_s) alone, R = L at the CTA's last row (at most 1 for gates
// in [0, 1]; 0 for keys before the zero gate): the key warps scale each unit
// key by the square root of its factor, and the scores and their squares are
// then those of the ungated form.  Other CTAs take exp(L_t - L_s) per weight.
//
// Pipeline (one CTA per pair of query tiles A = 2m, B = 2m + 1, sharing
// every key / value tile they both need; 512 threads):
//   warp 0 lane 0   TMA: both query tiles once, key and value tiles into a
//                   ring of kStages stages
//   warp 1 lane 0   issues every MMA, alternating the two query tiles:
//                   O_A(j), S_A(j+1), O_B(j), S_B(j+1), ... so that the
//                   squaring of one tile's scores overlaps the other tile's
//                   products
//   warps 4-7       squaring group of query tile A (and its o at the end)
//   warps 8-11      squaring group of query tile B (and its o at the end)
//   warps 12-15     put the keys of each staged tile on the unit sphere, in
//                   place (thread = key row)
//
// Short sequences (two CTAs a pair fit in one wave): clusters of two CTAs split a pair's
// key tiles, rank 0 taking tiles 0..m and rank 1 the rest (2m + 2 and 2m + 1
// tile products).  The weights need no running maximum, so the two partial
// sums of O simply add: rank 1 leaves its O (numerators and denominator,
// fp32) in its own shared memory, and rank 0 adds it through distributed
// shared memory before the division.
#include <cuda_bf16.h>

#include <cooperative_groups.h>

#include <cstdint>
#include <type_traits>

#include "kata_internal.h"
#include "tc_primitives.cuh"
#include "tc_tma.cuh"

namespace kata {
namespace {

using namespace tc;

__device__ unsigned int g_quad_tc_status = 0;

constexpr int kTile = 128;        // queries per tile, keys per tile
constexpr int kThreads = 512;
constexpr int kStages = 4;        // key / value ring
constexpr uint32_t kAtom = 128 * 128;
constexpr uint32_t kNV = 80;      // B columns of the value product: 64 value slots, the ones column, pad
constexpr uint64_t kWaitNs = 2000000000ull;  // bound of every device-side wait
constexpr float kSpanMax = 80.f;  // decay span of a query tile (natural log) below which its weights take key factors
constexpr float kLog2e = 1.44269504088896340736f;
constexpr int64_t kSplitMax = 148;  // CTAs of the split grid (two per pair) up to which pairs are split: one wave

// shared memory, 16 KB atoms from a 1024-byte aligned base: Q_A, Q_B,
// K[kStages], V[kStages], the ones atom (last, so every value stage reaches
// it with a positive atom stride)
constexpr uint32_t kQOff = 0, kKOff = 2 * kAtom, kVOff = (2 + kStages) * kAtom, kOnesOff = (2 + 2 * kStages) * kAtom;
// gated form, after the ones atom: per key stage, L_s of the tile's keys (fp32)
constexpr uint32_t kGateOff = (3 + 2 * kStages) * kAtom, kGateStage = kTile * 4;
constexpr size_t kSmem = (3 + 2 * kStages) * kAtom + 1024;
constexpr size_t kSmemGated = kSmem + kStages * kGateStage;
// tensor memory: scores (then squared weights, in place) and O per query tile
constexpr uint32_t kTmS = 0, kTmO = 256;  // tile g: S at 128 g, O at 256 + 128 g

// Per head, for every token t: L_t = sum of log gamma_r over r in (z_t, t]
// (fp32 logs summed in fp64) and z_t, the position of the last zero gate at or
// before t (-1 if none).  One block of kPrefixThreads per head: each thread
// takes a run of consecutive tokens, the runs' (sum, last zero) pairs are
// combined by a scan (a later zero restarts the sum), then every thread walks
// its run again from its prefix.
constexpr int kPrefixThreads = 1024;

__global__ void __launch_bounds__(kPrefixThreads)
gate_prefix_kernel(const float* __restrict__ gate, float* __restrict__ Lc, int* __restrict__ zid, int T) {
    __shared__ double ssum[kPrefixThreads];
    __shared__ int szero[kPrefixThreads];
    const int t = threadIdx.x;
    const int64_t base = (int64_t)blockIdx.x * T;
    const int run = (T + kPrefixThreads - 1) / kPrefixThreads;
    const int a = min(T, t * run), b = min(T, a + run);
    double sum = 0.0;
    int zero = -1;
    for (int r = a; r < b; ++r) {
        const float gm = gate[base + r];
        if (gm == 0.f) {
            zero = r;
            sum = 0.0;
        } else {
            sum += (double)logf(gm);
        }
    }
    ssum[t] = sum;
    szero[t] = zero;
    __syncthreads();
    // inclusive scan of the runs: (s1, z1) then (s2, z2) -> z2 >= 0 ? (s2, z2) : (s1 + s2, z1)
    for (int d = 1; d < kPrefixThreads; d <<= 1) {
        double ps = 0.0;
        int pz = -1;
        const bool has = t >= d;
        if (has) {
            ps = ssum[t - d];
            pz = szero[t - d];
        }
        __syncthreads();
        if (has && szero[t] < 0) {
            ssum[t] = ps + ssum[t];
            szero[t] = pz;
        }
        __syncthreads();
    }
    double cur = t > 0 ? ssum[t - 1] : 0.0;
    int cz = t > 0 ? szero[t - 1] : -1;
    for (int r = a; r < b; ++r) {
        const float gm = gate[base + r];
        if (gm == 0.f) {
            cz = r;
            cur = 0.0;
        } else {
            cur += (double)logf(gm);
        }
        Lc[base + r] = (float)cur;
        zid[base + r] = cz;
    }
}

template <int P, int DV, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
quadratic_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, __nv_bfloat16* __restrict__ o, int T,
                    const float* __restrict__ Lc, const int* __restrict__ zid, int split) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t q_full, k_full[kStages], v_full[kStages], k_ready[kStages], kv_free[kStages];
    __shared__ uint64_t s_full[2], p_full[2], o_done, drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int t = threadIdx.x, warp = t >> 5;
    // heaviest pairs first; with split, the two CTAs of a cluster take parts
    // 0 and 1 of one pair's key tiles
    const int part = split ? (int)(blockIdx.x & 1) : 0;
    const int m = (split ? (int)(gridDim.x >> 1) - 1 - (int)(blockIdx.x >> 1) : (int)gridDim.x - 1 - (int)blockIdx.x);
    const int64_t bh = blockIdx.y;
    const int ntiles = (T + kTile - 1) / kTile;
    const int qa = 2 * m, qb = 2 * m + 1;
    const bool has_b = qb < ntiles;
    // last key tile of query tile g (its diagonal; -1: no tile B)
    auto last = [&](int g) { return g ? (has_b ? qb : -1) : qa; };
    const int nj_all = has_b ? qb + 1 : qa + 1;
    // key tiles [j0, j1) of this CTA; query tile g takes j0 .. jend(g) of them
    const int j0 = split && part == 1 ? m + 1 : 0, j1 = split && part == 0 ? m + 1 : nj_all;
    const int nj = j1 - j0;
    auto jend = [&](int g) { return min(last(g), j1 - 1); };
    // gated form: whether the weights of this CTA's rows take key factors, the
    // reference R and the rows' common last zero gate
    bool gfast = false;
    float gref = 0.f;
    int gzero = -1;
    if (GATED) {
        const int r0 = qa * kTile, r1 = min(T, nj_all * kTile) - 1;
        const float l0 = Lc[bh * T + r0], l1 = Lc[bh * T + r1];
        gref = l1;
        gzero = zid[bh * T + r1];
        gfast = gzero < r0 && l0 - l1 < kSpanMax && l0 - l1 >= 0.f;
    }

    if (t == 0) {
        mbar_init(&q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&k_ready[s], 128);
            mbar_init(&kv_free[s], 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&s_full[g], 1);
            mbar_init(&p_full[g], 128);
        }
        mbar_init(&o_done, 1);
        mbar_init(&drain, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    // the ones atom: B rows = keys, column 64 of the value product = 1
    for (int r = t; r < kTile; r += kThreads)
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
        atomicOr(&g_quad_tc_status, kStatusTimeout);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, &abort_flag, kWaitNs));
    };

    if (t == 0) {
        // =============================================================== TMA producer
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        mbar_arrive_expect_tx(&q_full, (has_b ? 2 : 1) * kAtom);
        tma_load_3d(sm + kQOff, &tmq, 0, qa * kTile, (int)bh, &q_full);
        if (has_b) tma_load_3d(sm + kQOff + kAtom, &tmq, 0, qb * kTile, (int)bh, &q_full);
        int issued = 0;
        for (int jl = 0; jl < nj; ++jl) {
            const int st = jl % kStages, use = jl / kStages, j = j0 + jl;
            if (jl >= kStages && !mbar_wait(&kv_free[st], (use - 1) & 1, &abort_flag, kWaitNs)) { fail(); break; }
            mbar_arrive_expect_tx(&k_full[st], kAtom);
            tma_load_3d(sm + kKOff + st * kAtom, &tmk, 0, j * kTile, (int)bh, &k_full[st]);
            mbar_arrive_expect_tx(&v_full[st], kAtom);
            tma_load_3d(sm + kVOff + st * kAtom, &tmv, 0, j * kTile, (int)bh, &v_full[st]);
            issued = jl + 1;
        }
        // no copy may still be landing in shared memory when the CTA exits
        mbar_wait_quiet(&q_full, 0, kWaitNs);
        for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
            mbar_wait_quiet(&k_full[j % kStages], (j / kStages) & 1, kWaitNs);
            mbar_wait_quiet(&v_full[j % kStages], (j / kStages) & 1, kWaitNs);
        }
    } else if (warp == 1) {
        // =============================================================== MMA issuer
        // (the whole warp runs the loop; one elected lane issues each instruction)
        constexpr uint32_t id_s = idesc_bf16_f32(kTile, kTile);
        constexpr uint32_t id_o = idesc_bf16_f32_major(kTile, kNV, false, true);
        // scores of query tile g against key tile j (P in place of S afterwards)
        auto issue_s = [&](int g, int j) -> bool {
            const int jl = j - j0, st = jl % kStages;
            if (!wait(&k_ready[st], (jl / kStages) & 1)) return false;
            tc_fence_after();
            const uint64_t d_q = sdesc_kmajor_sw128(smem_u32(sm + kQOff + g * kAtom));
            const uint64_t d_k = sdesc_kmajor_sw128(smem_u32(sm + kKOff + st * kAtom));
#pragma unroll
            for (int ks = 0; ks < P / 16; ++ks)
                mma_ss_w(tb + kTmS + 128 * g, d_q + 2 * ks, d_k + 2 * ks, id_s, ks > 0 ? 1u : 0u);
            mma_commit_w(&s_full[g]);
            return true;
        };
        // O_g += P_g [V_j | 1]; then the next scores of tile g (they overwrite P_g)
        auto issue_o = [&](int g, int j) -> bool {
            const int jl = j - j0, st = jl % kStages;
            if (!wait(&p_full[g], jl & 1) ||
                !wait(&v_full[st], (jl / kStages) & 1))
                return false;
            tc_fence_after();
            // B = [value tile | ones]: two MN atoms, the ones atom kOnesOff - value stage bytes away
            const uint32_t vaddr = smem_u32(sm + kVOff + st * kAtom);
            const uint64_t d_v = sdesc_mnmajor_sw128(vaddr, (uint32_t)(kOnesOff - (kVOff + st * kAtom)));
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
                mma_ts_w(tb + kTmO + 128 * g, tb + kTmS + 128 * g + 8 * ks, d_v + ks * (2048 >> 4), id_o,
                       (j > j0 || ks > 0) ? 1u : 0u);
            if (j + 1 <= jend(g)) return issue_s(g, j + 1);
            return true;
        };
        bool ok = wait(&q_full, 0) && (jend(0) < j0 || issue_s(0, j0)) && (jend(1) < j0 || issue_s(1, j0));
        for (int j = j0; ok && j < j1; ++j) {
            if (j <= jend(0) && !issue_o(0, j)) { ok = false; break; }
            if (j <= jend(1) && !issue_o(1, j)) { ok = false; break; }
            mma_commit_w(&kv_free[(j - j0) % kStages]);  // both tiles' products with key / value tile j are issued
        }
        if (!ok) fail();
        mma_commit_w(&o_done);
        mma_commit_w(&drain);
        mbar_wait_quiet(&drain, 0, kWaitNs);
    } else if (warp >= 12) {
        // =============================================================== key normalisation
        const int r = t - 384;
        // gated form: L of this thread's key in the next tile, loaded one tile
        // ahead so that its latency overlaps the wait for the tile
        float lk_next = (GATED && j0 * kTile + r < T) ? Lc[bh * T + j0 * kTile + r] : 0.f;
        for (int j = j0; j < j1; ++j) {
            const int jl = j - j0, st = jl % kStages;
            const float lk = lk_next;
            if (GATED) {
                const int nk = (j + 1) * kTile + r;
                lk_next = (j + 1 < j1 && nk < T) ? Lc[bh * T + nk] : 0.f;
            }
            if (!wait(&k_full[st], (jl / kStages) & 1)) { fail(); break; }
            uint8_t* kb = sm + kKOff + st * kAtom;
            uint4 raw[P / 8];
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < P / 8; ++c) {
                raw[c] = *reinterpret_cast<const uint4*>(kb + sw128_chunk(r, 8 * c, kTile));
                const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[c]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float x = __bfloat162float(e[i]);
                    ss = fmaf(x, x, ss);
                }
            }
            float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
            if (GATED) {
                // the key's L (exact weights), or the unit key scaled by the
                // square root of its factor (0 before the zero gate and past T)
                const int key = j * kTile + r;
                reinterpret_cast<float*>(sm + kGateOff + st * kGateStage)[r] = lk;
                if (gfast) inv = (key < T && key >= gzero) ? inv * exp2f(0.5f * (gref - lk) * kLog2e) : 0.f;
            }
#pragma unroll
            for (int c = 0; c < P / 8; ++c) {
                const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&raw[c]);
                uint4 w;
                w.x = pack_bf16x2(__bfloat162float(e[0]) * inv, __bfloat162float(e[1]) * inv);
                w.y = pack_bf16x2(__bfloat162float(e[2]) * inv, __bfloat162float(e[3]) * inv);
                w.z = pack_bf16x2(__bfloat162float(e[4]) * inv, __bfloat162float(e[5]) * inv);
                w.w = pack_bf16x2(__bfloat162float(e[6]) * inv, __bfloat162float(e[7]) * inv);
                *reinterpret_cast<uint4*>(kb + sw128_chunk(r, 8 * c, kTile)) = w;
            }
            fence_proxy_async_smem();
            mbar_arrive(&k_ready[st]);
        }
    } else if (warp >= 4) {
        // =============================================================== squaring groups
        const int g = warp >= 8 ? 1 : 0;  // query tile A or B
        const int e = t & 127;            // query row = tensor-memory lane
        const int wq = (warp & 3);        // this warp's rows are 32 wq .. 32 wq + 31
        const uint32_t lane0 = (uint32_t)(wq * 32);
        const uint32_t sb = tb + kTmS + 128 * g;
        // gated form: this row's L and last zero gate (exact weights)
        float lrow = 0.f;
        int zrow = -1;
        if (GATED) {
            const int row = min(T - 1, last(g) * kTile + e);
            lrow = Lc[bh * T + row];
            zrow = zid[bh * T + row];
        }
        // P of key tile j in place of its scores; EXACT: every weight with its
        // own decay exp(L_t - L_s) (gated CTAs outside the key-factor range),
        // otherwise the squares as they are (the ungated form, and gated CTAs
        // whose key factors are already in the unit keys).  Two compiled loops,
        // chosen once per CTA, so the squaring of the common case stays lean.
        auto square = [&](auto exact_tag) -> bool {
            constexpr bool EXACT = decltype(exact_tag)::value;
            for (int j = j0; j <= jend(g); ++j) {
                const int jl = j - j0;
                if (!wait(&s_full[g], jl & 1)) return false;
                // the key tile's L values are in shared memory (its staging completed before the scores' MMA)
                if (EXACT && !wait(&k_ready[jl % kStages], (jl / kStages) & 1)) return false;
                tc_fence_after();
                const bool diag = j == last(g);  // keys past the query are masked only on the diagonal tile
                const float* gs = reinterpret_cast<const float*>(sm + kGateOff + (jl % kStages) * kGateStage);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[16];
                    if (!diag || q4 <= wq) {
                        uint32_t sc[32];
                        tmem_ld16(tmem_addr(sb, lane0, 32 * q4), *reinterpret_cast<uint32_t(*)[16]>(sc));
                        tmem_ld16(tmem_addr(sb, lane0, 32 * q4 + 16), *reinterpret_cast<uint32_t(*)[16]>(sc + 16));
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int col = 32 * q4 + 2 * i;
                            float a = __uint_as_float(sc[2 * i]), c = __uint_as_float(sc[2 * i + 1]);
                            a *= a;
                            c *= c;
                            if (EXACT) {
                                const float2 lk = *reinterpret_cast<const float2*>(gs + col);
                                const int key = j * kTile + col;
                                a = zrow <= key ? a * exp2f((lrow - lk.x) * kLog2e) : 0.f;
                                c = zrow <= key + 1 ? c * exp2f((lrow - lk.y) * kLog2e) : 0.f;
                            }
                            if (diag) {
                                a = col <= e ? a : 0.f;
                                c = col + 1 <= e ? c : 0.f;
                            }
                            pk[i] = pack_bf16x2(a, c);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = 0u;
                    }
                    tmem_st16(tmem_addr(sb, lane0, 16 * q4), pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[g]);
            }
            return true;
        };
        bool sq_ok;
        if constexpr (GATED) {
            sq_ok = gfast ? square(std::false_type{}) : square(std::true_type{});
        } else {
            sq_ok = square(std::false_type{});
        }
        if (!sq_ok) fail();
        // ---- o = O[:, :DV] / O[:, 64] (split: after the exchange below)
        const bool ok = wait(&o_done, 0) && !abort_flag;
        tc_fence_after();
        const int qi = (g == 0 ? qa : qb) * kTile + e;
        if (!split && ok && last(g) >= 0) {
            const uint32_t ob = tb + kTmO + 128 * g;
            uint32_t r[16];
            tmem_ld16(tmem_addr(ob, lane0, 64), r);
            tmem_wait_ld();
            const float den = __uint_as_float(r[0]);
            const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 16) {
                tmem_ld16(tmem_addr(ob, lane0, c0), r);
                tmem_wait_ld();
                if (qi < T) {
                    uint4 out[2];
                    uint32_t* w = reinterpret_cast<uint32_t*>(out);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
                    __nv_bfloat16* dst = o + (bh * T + qi) * (int64_t)DV + c0;
                    reinterpret_cast<uint4*>(dst)[0] = out[0];
                    reinterpret_cast<uint4*>(dst)[1] = out[1];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (split) {
        // every copy has landed and every MMA completed (the producer and the
        // MMA warp waited for them): the stage memory is free for the exchange,
        // x[g][c][row] = O_g[row][c] of rank 1 (c = DV: the denominator)
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        float* x = reinterpret_cast<float*>(sm);
        const bool sq = warp >= 4 && warp < 12;
        const int g = warp >= 8 ? 1 : 0, e = t & 127;
        const uint32_t lane0 = (uint32_t)((warp & 3) * 32), ob = tb + kTmO + 128 * g;
        const bool live = !abort_flag && jend(g) >= j0;  // this tile has products in this CTA
        if (sq && part == 1) {
            uint32_t r[16];
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 16) {
                if (live) {
                    tmem_ld16(tmem_addr(ob, lane0, c0), r);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) x[(g * (DV + 1) + c0 + i) * kTile + e] = live ? __uint_as_float(r[i]) : 0.f;
            }
            if (live) {
                tmem_ld16(tmem_addr(ob, lane0, 64), r);
                tmem_wait_ld();
            }
            x[(g * (DV + 1) + DV) * kTile + e] = live ? __uint_as_float(r[0]) : 0.f;
        }
        cluster_barrier();
        const int qi = (g == 0 ? qa : qb) * kTile + e;
        // (the tensor-memory loads are warp-wide: rows past T load and skip the store)
        if (sq && part == 0 && live) {
            const float* xr = cluster.map_shared_rank(x, 1);
            uint32_t r[16];
            tmem_ld16(tmem_addr(ob, lane0, 64), r);
            tmem_wait_ld();
            const float den = __uint_as_float(r[0]) + xr[(g * (DV + 1) + DV) * kTile + e];
            const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 16) {
                tmem_ld16(tmem_addr(ob, lane0, c0), r);
                tmem_wait_ld();
                uint4 out[2];
                uint32_t* w = reinterpret_cast<uint32_t*>(out);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float a = __uint_as_float(r[2 * i]) + xr[(g * (DV + 1) + c0 + 2 * i) * kTile + e];
                    const float b = __uint_as_float(r[2 * i + 1]) + xr[(g * (DV + 1) + c0 + 2 * i + 1) * kTile + e];
                    w[i] = pack_bf16x2(a * inv, b * inv);
                }
                if (qi < T) {
                    __nv_bfloat16* dst = o + (bh * T + qi) * (int64_t)DV + c0;
                    reinterpret_cast<uint4*>(dst)[0] = out[0];
                    reinterpret_cast<uint4*>(dst)[1] = out[1];
                }
            }
        }
        cluster_barrier();  // rank 1's shared memory stays until rank 0 has read it
    }
    if (warp == 0) tmem_dealloc(tb, 512);
}

template <int P, int DV, bool GATED>
cudaError_t launch_typed(const void* q, const void* k, const void* v, void* o, int BH, int T, const float* Lc,
                         const int* zid, cudaStream_t s) {
    auto kern = quadratic_tc_kernel<P, DV, GATED>;
    const size_t smem = GATED ? kSmemGated : kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk, tv;
    if (!rows_map(&tq, q, P, T, BH) || !rows_map(&tk, k, P, T, BH) || !rows_map(&tv, v, DV, T, BH))
        return cudaErrorInvalidValue;
    const int ntiles = (T + kTile - 1) / kTile, pairs = (ntiles + 1) / 2;
    // when even two CTAs a pair fit in one wave, split each pair's key tiles
    // over a cluster of two (a second wave costs more than the split saves)
    const int split = ntiles >= 2 && 2 * (int64_t)pairs * BH <= kSplitMax ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pairs * (1 + split)), (unsigned)BH, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1 + split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = split ? 1 : 0;
    KATA_TRACED(GATED ? "quadratic_gated_tc" : "quadratic_tc", s,
                (e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, static_cast<__nv_bfloat16*>(o), T, Lc, zid, split)));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quadratic_tc(const void* q, const void* k, const void* v, void* o, int BH, int T,
                                int p, int dv, cudaStream_t s) {
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return launch_typed<P_, DV_, false>(q, k, v, o, BH, T, nullptr, nullptr, s);
    KATA_CASE(16, 16) KATA_CASE(16, 32) KATA_CASE(16, 64)
    KATA_CASE(32, 16) KATA_CASE(32, 32) KATA_CASE(32, 64)
    KATA_CASE(64, 16) KATA_CASE(64, 32) KATA_CASE(64, 64)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

size_t quadratic_gated_tc_workspace(int BH, int T) {
    const size_t n = (size_t)BH * T;
    return ((n * sizeof(float) + 255) / 256) * 256 + ((n * sizeof(int) + 255) / 256) * 256;
}

cudaError_t launch_quadratic_gated_tc(const void* q, const void* k, const void* v, const float* gate, void* o,
                                      void* ws, int BH, int T, int p, int dv, cudaStream_t s) {
    const size_t n = (size_t)BH * T;
    float* Lc = static_cast<float*>(ws);
    int* zid = reinterpret_cast<int*>(static_cast<char*>(ws) + ((n * sizeof(float) + 255) / 256) * 256);
    KATA_TRACED("gate_prefix", s, (gate_prefix_kernel<<<(unsigned)BH, kPrefixThreads, 0, s>>>(gate, Lc, zid, T)));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
#define KATA_CASE(P_, DV_) \
    if (p == P_ && dv == DV_) return launch_typed<P_, DV_, true>(q, k, v, o, BH, T, Lc, zid, s);
    KATA_CASE(16, 16) KATA_CASE(16, 32) KATA_CASE(16, 64)
    KATA_CASE(32, 16) KATA_CASE(32, 32) KATA_CASE(32, 64)
    KATA_CASE(64, 16) KATA_CASE(64, 32) KATA_CASE(64, 64)
#undef KATA_CASE
    return cudaErrorInvalidValue;
}

unsigned int quadratic_tc_take_status() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_quad_tc_status, sizeof(v)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_quad_tc_status, &zero, sizeof(zero));
    return v;
}

}  // namespace kata
