// C ABI of libkata (declared in include/kata.h): argument checks, workspace
// sizing and dispatch to the kernels.  No device memory is allocated here.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/kata.h"
#include "kata_internal.h"

namespace {

constexpr int64_t kMaxT = int64_t(1) << 30;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool p_ok(int p) { return p == 16 || p == 32 || p == 64; }
bool dv_ok(int dv) { return dv == 16 || dv == 32 || dv == 64; }
bool c_ok(int C) { return C == 32 || C == 64 || C == 128; }
int64_t packed(int p) { return (int64_t)p * (p + 1) / 2; }
kata_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KATA_OK : KATA_ERR_CUDA; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shape checks shared by the forwards.  Returns KATA_OK or the error.
kata_status check_shapes(kata_dtype dt, int B, int H, int T, int p, int dv) {
    if (dt != KATA_FP32 && dt != KATA_BF16) return KATA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || T < 0) return KATA_ERR_INVALID_ARG;
    if (!p_ok(p) || !dv_ok(dv)) return KATA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 65535 || T > kMaxT) return KATA_ERR_UNSUPPORTED;
    return KATA_OK;
}

// cuMemGetAddressRange through the runtime's driver entry point (no link
// dependency on libcuda); null if unavailable.
PFN_cuMemGetAddressRange_v3020 mem_range_fn() {
    static PFN_cuMemGetAddressRange_v3020 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// A buffer the kernels may touch: non-null, 16-byte aligned, device memory of
// the current device (or managed memory), and -- where the driver can tell
// the allocation's extent -- at least `bytes` long from `ptr`.
kata_status check_buffer(const void* ptr, size_t bytes) {
    if (ptr == nullptr || !aligned16(ptr)) return KATA_ERR_INVALID_ARG;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_INVALID_ARG;
    }
    if (a.type == cudaMemoryTypeDevice) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || a.device != dev) return KATA_ERR_INVALID_ARG;
        if (PFN_cuMemGetAddressRange_v3020 fn = mem_range_fn()) {
            CUdeviceptr base = 0;
            size_t size = 0;
            if (fn(&base, &size, reinterpret_cast<CUdeviceptr>(ptr)) == CUDA_SUCCESS &&
                reinterpret_cast<uintptr_t>(ptr) + bytes > (uintptr_t)base + size)
                return KATA_ERR_INVALID_ARG;
        }
        return KATA_OK;
    }
    return a.type == cudaMemoryTypeManaged ? KATA_OK : KATA_ERR_INVALID_ARG;
}

size_t elem_bytes(kata_dtype dt) { return dt == KATA_FP32 ? 4 : 2; }

// Workspace of the chunked forward: per-chunk states [BH, NC, n, dv] and
// [BH, NC, n] in fp32, each 256-byte aligned.
struct ChunkedWs {
    size_t s_off, z_off, total;
    size_t i_off;  // tensor-core path: intra-chunk rows
};

ChunkedWs chunked_ws(int B, int H, int T, int p, int dv, int C, int64_t n_lift = 0) {
    const int64_t BH = (int64_t)B * H, NC = (T + C - 1) / C, n = n_lift > 0 ? n_lift : packed(p);
    ChunkedWs w;
    w.s_off = 0;
    w.i_off = 0;
    w.z_off = round_up(sizeof(float) * (size_t)(BH * NC * n * dv), 256);
    w.total = w.z_off + round_up(sizeof(float) * (size_t)(BH * NC * n), 256);
    return w;
}

// bf16 inputs take the tensor-core forward when its kernels can run on the
// current device; its workspace holds one start state per
// segment when the sequence is cut into G > 1 segments.  The segment totals
// are built over `sub` equal parts of each segment (more CTAs for the
// chunk-state kernel when few heads leave most of the GPU to it); their
// exclusive prefix at every sub-th part is a segment's start state.
struct TcPlan {
    bool use = false;
    int G = 1;
    int sub = 1;
    ChunkedWs ws{0, 0, 0, 0};
};

// lg: blocks of the lift (1: the full lift; g > 1: KATA-Sigma-g, whose state
// has the width of the lift of one block, p/g).
TcPlan tc_plan(kata_dtype dt, int B, int H, int T, int p, int dv, int lg = 1) {
    TcPlan pl;
    if (dt != KATA_BF16 || !kata::chunked_tc_supports(p, dv, lg)) return pl;
    const int64_t BH = (int64_t)B * H, n = packed(p / lg);
    int G = kata::chunked_tc_segments(p, dv, lg, (int)BH, T);
    if (G <= 0) return pl;
    pl.use = true;
    pl.G = G;
    size_t off = 0;
    if (G > 1) {
        // parts per segment: about two chunk-state CTAs per SM (148 SMs), a
        // divisor of the segment's chunks so that parts tile the segments
        const int seg_chunks = kata::chunked_tc_segment_chunks(T, G);
        const int64_t units = ((n + 127) / 128) * BH * (G - 1);
        const int want = (int)((2 * 148 + units - 1) / units);
        for (int d = want < seg_chunks ? want : seg_chunks; d >= 1; --d)
            if (seg_chunks % d == 0) {
                pl.sub = d;
                break;
            }
        const int64_t entries = (int64_t)G * pl.sub;
        pl.ws.s_off = 0;
        pl.ws.z_off = round_up(sizeof(float) * (size_t)(BH * entries * n * dv), 256);
        off = pl.ws.z_off + round_up(sizeof(float) * (size_t)(BH * entries * n), 256);
    }
    pl.ws.i_off = off;
    pl.ws.total = off + round_up(kata::chunked_tc_intra_bytes((int)BH, T, p, dv), 256);
    return pl;
}

// The tensor-core forward of a plan: one launch of the fused kernels when the
// sequence is one segment per head; otherwise the totals of the parts of
// segments 0..G-2 (chunk-state kernel), their exclusive prefixes seeded with
// the initial state (at every sub-th part: the start state of a segment),
// then the fused kernels with a start state per segment.  lg: blocks of the
// lift.
cudaError_t launch_tc_forward(const TcPlan& pl, const void* q, const void* k, const void* v, void* o, void* ws,
                              const float* S0, const float* z0, float* S_final, float* z_final, int64_t BH, int T,
                              int p, int dv, int lg, kata_scan_mode mode, cudaStream_t stream) {
    const ChunkedWs& w = pl.ws;
    void* intra = static_cast<char*>(ws) + w.i_off;
    if (pl.G == 1)
        return kata::launch_chunked_tc(q, k, v, o, intra, S0, z0, 1, 1, S_final, z_final, (int)BH, T, p, dv, lg, 1,
                                       stream);
    const int G = pl.G, sub = pl.sub, E = G * sub;  // E prefix entries per head
    const int64_t n = packed(p / lg);
    const int L = kata::chunked_tc_segment_chunks(T, G) * 128 / sub;  // tokens per part
    float* Sg = reinterpret_cast<float*>(static_cast<char*>(ws) + w.s_off);
    float* zg = reinterpret_cast<float*>(static_cast<char*>(ws) + w.z_off);
    cudaError_t e = kata::launch_states_tc(k, v, Sg, zg, (int)BH, T, p, dv, L, E - sub, E, 0, lg, stream);
    // the last segment's parts are not summed: zero them, so the scan reads defined values
    if (e == cudaSuccess)
        e = cudaMemset2DAsync(Sg + (size_t)(E - sub) * n * dv, sizeof(float) * (size_t)E * n * dv, 0,
                              sizeof(float) * (size_t)sub * n * dv, (size_t)BH, stream);
    if (e == cudaSuccess)
        e = cudaMemset2DAsync(zg + (size_t)(E - sub) * n, sizeof(float) * (size_t)E * n, 0,
                              sizeof(float) * (size_t)sub * n, (size_t)BH, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, Sg, Sg, S0, nullptr, BH, E, n * dv, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, zg, zg, z0, nullptr, BH, E, n, stream);
    if (e == cudaSuccess)
        e = kata::launch_chunked_tc(q, k, v, o, intra, Sg, zg, E, sub, S_final, z_final, (int)BH, T, p, dv, lg, G,
                                    stream);
    return e;
}

// Width of a lift (full, Sigma-g, M-g); -1 if (family, g) does not fit p.
int lift_dim(int family, int p, int g) {
    if (p <= 0 || g <= 0 || p % g != 0) return -1;
    const int64_t m = p / g, nm = m * (m + 1) / 2;
    if (family == KATA_LIFT_FULL) return g == 1 ? (int)nm : -1;
    if (family == KATA_LIFT_SIGMA) return (int)nm;
    if (family == KATA_LIFT_MULTI) return (int)(g * nm);
    return -1;
}

kata_status check_lift(kata_lift_family family, int p, int g) {
    if (family != KATA_LIFT_FULL && family != KATA_LIFT_SIGMA && family != KATA_LIFT_MULTI) return KATA_ERR_INVALID_ARG;
    if (g < 1) return KATA_ERR_INVALID_ARG;
    return lift_dim(family, p, g) > 0 ? KATA_OK : KATA_ERR_UNSUPPORTED;
}

// Shared body of the decode steps (shapes and lift already checked).
kata_status decode_common(const void* q, const void* k, const void* v, void* o, kata_dtype dt, int B, int H, int p,
                          int dv, int family, int g, float* S, float* z, cudaStream_t stream,
                          const float* gate = nullptr) {
    kata_status st = KATA_OK;
    const int64_t BH = (int64_t)B * H, n = lift_dim(family, p, g);
    if (BH == 0) return KATA_OK;
    const size_t qk_bytes = elem_bytes(dt) * BH * p, v_bytes = elem_bytes(dt) * BH * dv;
    const size_t sb = sizeof(float) * (size_t)(BH * n * dv), zb = sizeof(float) * (size_t)(BH * n);
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(o, v_bytes)) != KATA_OK ||
        (st = check_buffer(S, sb)) != KATA_OK || (st = check_buffer(z, zb)) != KATA_OK)
        return st;
    if (gate && (st = check_buffer(gate, sizeof(float) * (size_t)BH)) != KATA_OK) return st;
    // S and z are updated in place by different threads: they must not overlap.
    const char* sp = reinterpret_cast<const char*>(S);
    const char* zp = reinterpret_cast<const char*>(z);
    if (sp < zp + zb && zp < sp + sb) return KATA_ERR_INVALID_ARG;
    return cuda_status(kata::launch_decode_step(dt, q, k, v, o, S, z, (int)BH, p, dv, family, g, gate, stream));
}

}  // namespace

extern "C" {

int kata_packed_dim(int p) { return p < 0 ? -1 : (int)packed(p); }

const char* kata_status_string(kata_status s) {
    switch (s) {
        case KATA_OK: return "KATA_OK";
        case KATA_ERR_INVALID_ARG: return "KATA_ERR_INVALID_ARG: null or misaligned pointer, negative size or bad enum";
        case KATA_ERR_UNSUPPORTED: return "KATA_ERR_UNSUPPORTED: p, dv or C outside the supported set, or sizes too large";
        case KATA_ERR_WORKSPACE: return "KATA_ERR_WORKSPACE: workspace missing or too small";
        case KATA_ERR_CUDA: return "KATA_ERR_CUDA: a CUDA call or kernel launch failed";
        case KATA_ERR_TIMEOUT: return "KATA_ERR_TIMEOUT: a bounded device-side wait expired";
    }
    return "KATA_ERR_UNKNOWN";
}

kata_status kata_forward_quadratic(const void* q, const void* k, const void* v, void* o,
                                   kata_dtype dt, int B, int H, int T, int p, int dv, int C,
                                   cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv);
    if (st != KATA_OK) return st;
    if (C != 0 && !c_ok(C)) return KATA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * T;
    if (rows == 0) return KATA_OK;
    const size_t qk_bytes = elem_bytes(dt) * rows * p, v_bytes = elem_bytes(dt) * rows * dv;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(o, v_bytes)) != KATA_OK)
        return st;
    if (dt == KATA_BF16) return cuda_status(kata::launch_quadratic_tc(q, k, v, o, B * H, T, p, dv, stream));
    return cuda_status(kata::launch_quadratic_simt(dt, q, k, v, o, B * H, T, p, dv, stream));
}

size_t kata_quadratic_gated_workspace_bytes(kata_dtype dt, int B, int H, int T) {
    if (dt != KATA_BF16 || B < 0 || H < 0 || T < 0) return 0;
    if ((int64_t)B * H * T == 0) return 0;
    return kata::quadratic_gated_tc_workspace(B * H, T);
}

kata_status kata_forward_quadratic_gated(const void* q, const void* k, const void* v, const float* gate, void* o,
                                         kata_dtype dt, int B, int H, int T, int p, int dv, void* ws,
                                         size_t ws_bytes, cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv);
    if (st != KATA_OK) return st;
    if (dt != KATA_BF16) return KATA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * H * T;
    if (rows == 0) return KATA_OK;
    const size_t qk_bytes = elem_bytes(dt) * rows * p, v_bytes = elem_bytes(dt) * rows * dv;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(o, v_bytes)) != KATA_OK ||
        (st = check_buffer(gate, sizeof(float) * rows)) != KATA_OK)
        return st;
    const size_t need = kata::quadratic_gated_tc_workspace(B * H, T);
    if (ws == nullptr || ws_bytes < need) return KATA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KATA_ERR_INVALID_ARG;
    if ((st = check_buffer(ws, need)) != KATA_OK) return st;
    return cuda_status(kata::launch_quadratic_gated_tc(q, k, v, gate, o, ws, B * H, T, p, dv, stream));
}

size_t kata_chunked_workspace_bytes(kata_dtype dt, int B, int H, int T, int p, int dv, int C) {
    if (check_shapes(dt, B, H, T, p, dv) != KATA_OK || !c_ok(C)) return 0;
    if ((int64_t)B * H * T == 0) return 0;
    const TcPlan pl = tc_plan(dt, B, H, T, p, dv);
    return pl.use ? pl.ws.total : chunked_ws(B, H, T, p, dv, C).total;
}

kata_status kata_forward_chunked(const void* q, const void* k, const void* v, void* o,
                                 kata_dtype dt, int B, int H, int T, int p, int dv, int C,
                                 kata_scan_mode mode, const float* S0, const float* z0,
                                 float* S_final, float* z_final, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv);
    if (st != KATA_OK) return st;
    if (!c_ok(C)) return KATA_ERR_UNSUPPORTED;
    if (mode != KATA_SCAN_SEQUENTIAL && mode != KATA_SCAN_TREE) return KATA_ERR_INVALID_ARG;
    if ((S0 == nullptr) != (z0 == nullptr)) return KATA_ERR_INVALID_ARG;
    if ((S_final == nullptr) != (z_final == nullptr)) return KATA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H, n = packed(p);
    if (BH == 0) return KATA_OK;
    const size_t s_bytes = sizeof(float) * BH * n * dv, z_bytes = sizeof(float) * BH * n;
    if (S0 && ((st = check_buffer(S0, s_bytes)) != KATA_OK || (st = check_buffer(z0, z_bytes)) != KATA_OK))
        return st;
    if (S_final &&
        ((st = check_buffer(S_final, s_bytes)) != KATA_OK || (st = check_buffer(z_final, z_bytes)) != KATA_OK))
        return st;
    if (T == 0) {
        if (S_final == nullptr) return KATA_OK;
        cudaError_t e = kata::launch_copy_or_zero(S0, S_final, BH * n * dv, stream);
        if (e == cudaSuccess) e = kata::launch_copy_or_zero(z0, z_final, BH * n, stream);
        return cuda_status(e);
    }
    const size_t qk_bytes = elem_bytes(dt) * BH * T * p, v_bytes = elem_bytes(dt) * BH * T * dv;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(o, v_bytes)) != KATA_OK)
        return st;
    const TcPlan pl = tc_plan(dt, B, H, T, p, dv);
    const ChunkedWs w = pl.use ? pl.ws : chunked_ws(B, H, T, p, dv, C);
    if (w.total > 0) {
        if (ws == nullptr || ws_bytes < w.total) return KATA_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KATA_ERR_INVALID_ARG;
        if ((st = check_buffer(ws, w.total)) != KATA_OK) return st;
    }
    if (pl.use)
        return cuda_status(launch_tc_forward(pl, q, k, v, o, ws, S0, z0, S_final, z_final, BH, T, p, dv, 1, mode, stream));

    const int64_t NC = (T + C - 1) / C;
    float* S_loc = reinterpret_cast<float*>(static_cast<char*>(ws) + w.s_off);
    float* z_loc = reinterpret_cast<float*>(static_cast<char*>(ws) + w.z_off);
    cudaError_t e = kata::launch_chunk_states_simt(dt, k, v, S_loc, z_loc, (int)BH, T, p, dv, C, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, S_loc, S_loc, S0, S_final, BH, NC, n * dv, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, z_loc, z_loc, z0, z_final, BH, NC, n, stream);
    if (e == cudaSuccess)
        e = kata::launch_chunk_output_simt(dt, q, k, v, S_loc, z_loc, o, (int)BH, T, p, dv, C, stream);
    return cuda_status(e);
}

kata_status kata_chunk_state_scan(const void* k, const void* v, kata_dtype dt, int B, int H, int T,
                                  int p, int dv, int C, kata_scan_mode mode, float* S_prefix,
                                  float* z_prefix, cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv);
    if (st != KATA_OK) return st;
    if (!c_ok(C)) return KATA_ERR_UNSUPPORTED;
    if (mode != KATA_SCAN_SEQUENTIAL && mode != KATA_SCAN_TREE) return KATA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H, n = packed(p), NC = (T + C - 1) / C;
    if (BH * T == 0) return KATA_OK;
    const size_t qk_bytes = elem_bytes(dt) * BH * T * p, v_bytes = elem_bytes(dt) * BH * T * dv;
    if ((st = check_buffer(k, qk_bytes)) != KATA_OK || (st = check_buffer(v, v_bytes)) != KATA_OK ||
        (st = check_buffer(S_prefix, sizeof(float) * BH * NC * n * dv)) != KATA_OK ||
        (st = check_buffer(z_prefix, sizeof(float) * BH * NC * n)) != KATA_OK)
        return st;
    // bf16, sequential prefix: the state kernel sums the chunk states in chunk
    // order as it goes and writes the exclusive prefixes directly (one pass)
    if (dt == KATA_BF16 && mode == KATA_SCAN_SEQUENTIAL)
        return cuda_status(
            kata::launch_states_tc(k, v, S_prefix, z_prefix, (int)BH, T, p, dv, C, (int)NC, (int)NC, 1, 1, stream));
    cudaError_t e = dt == KATA_BF16
                        ? kata::launch_states_tc(k, v, S_prefix, z_prefix, (int)BH, T, p, dv, C, (int)NC, (int)NC, 0, 1, stream)
                        : kata::launch_chunk_states_simt(dt, k, v, S_prefix, z_prefix, (int)BH, T, p, dv, C, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, S_prefix, S_prefix, nullptr, nullptr, BH, NC, n * dv, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, z_prefix, z_prefix, nullptr, nullptr, BH, NC, n, stream);
    return cuda_status(e);
}

kata_status kata_scan_states(const float* S_loc, const float* z_loc, float* S_prefix,
                             float* z_prefix, int B, int H, int NC, int n, int dv,
                             kata_scan_mode mode, cudaStream_t stream) {
    if (B < 0 || H < 0 || NC < 0 || n < 0 || dv < 0) return KATA_ERR_INVALID_ARG;
    if (mode != KATA_SCAN_SEQUENTIAL && mode != KATA_SCAN_TREE) return KATA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H;
    if (BH * NC * n * dv == 0 && BH * NC * n == 0) return KATA_OK;
    const size_t sb = sizeof(float) * (size_t)(BH * NC * n * dv), zb = sizeof(float) * (size_t)(BH * NC * n);
    kata_status st;
    if ((st = check_buffer(S_loc, sb)) != KATA_OK || (st = check_buffer(z_loc, zb)) != KATA_OK ||
        (st = check_buffer(S_prefix, sb)) != KATA_OK || (st = check_buffer(z_prefix, zb)) != KATA_OK)
        return st;
    // Partial overlap of input and output would race; exact aliasing is fine.
    auto overlaps = [](const void* a, const void* b, size_t bytes) {
        const char* x = static_cast<const char*>(a);
        const char* y = static_cast<const char*>(b);
        return x != y && x < y + bytes && y < x + bytes;
    };
    if (overlaps(S_loc, S_prefix, sb) || overlaps(z_loc, z_prefix, zb)) return KATA_ERR_INVALID_ARG;
    cudaError_t e = kata::launch_scan(mode, S_loc, S_prefix, nullptr, nullptr, BH, NC, (int64_t)n * dv, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, z_loc, z_prefix, nullptr, nullptr, BH, NC, n, stream);
    return cuda_status(e);
}

kata_status kata_decode_step(const void* q, const void* k, const void* v, void* o, kata_dtype dt, int B, int H,
                             int p, int dv, float* S, float* z, cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, 1, p, dv);
    if (st != KATA_OK) return st;
    return decode_common(q, k, v, o, dt, B, H, p, dv, KATA_LIFT_FULL, 1, S, z, stream);
}


int kata_lift_dim(kata_lift_family family, int p, int g) {
    if (family != KATA_LIFT_FULL && family != KATA_LIFT_SIGMA && family != KATA_LIFT_MULTI) return -1;
    return lift_dim(family, p, g);
}

// bf16 KATA-Sigma-g forwards run on the tensor cores where the fused kernel
// has the block width; every other block lift on the CUDA cores.
TcPlan block_tc_plan(kata_dtype dt, kata_lift_family family, int g, int B, int H, int T, int p, int dv) {
    if (family != KATA_LIFT_SIGMA || g < 2) return TcPlan{};
    return tc_plan(dt, B, H, T, p, dv, g);
}

size_t kata_chunked_block_workspace_bytes(kata_dtype dt, kata_lift_family family, int g, int B, int H, int T, int p,
                                          int dv, int C) {
    if (check_shapes(dt, B, H, T, p, dv) != KATA_OK || !c_ok(C) || check_lift(family, p, g) != KATA_OK) return 0;
    if ((int64_t)B * H * T == 0) return 0;
    const TcPlan pl = block_tc_plan(dt, family, g, B, H, T, p, dv);
    return pl.use ? pl.ws.total : chunked_ws(B, H, T, p, dv, C, lift_dim(family, p, g)).total;
}

kata_status kata_forward_chunked_block(const void* q, const void* k, const void* v, void* o, kata_dtype dt, int B,
                                       int H, int T, int p, int dv, int C, kata_lift_family family, int g,
                                       kata_scan_mode mode, const float* S0, const float* z0, float* S_final,
                                       float* z_final, void* ws, size_t ws_bytes, cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv);
    if (st != KATA_OK) return st;
    if ((st = check_lift(family, p, g)) != KATA_OK) return st;
    if (!c_ok(C)) return KATA_ERR_UNSUPPORTED;
    if (mode != KATA_SCAN_SEQUENTIAL && mode != KATA_SCAN_TREE) return KATA_ERR_INVALID_ARG;
    if ((S0 == nullptr) != (z0 == nullptr)) return KATA_ERR_INVALID_ARG;
    if ((S_final == nullptr) != (z_final == nullptr)) return KATA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H, n = lift_dim(family, p, g);
    if (BH == 0) return KATA_OK;
    const size_t s_bytes = sizeof(float) * BH * n * dv, z_bytes = sizeof(float) * BH * n;
    if (S0 && ((st = check_buffer(S0, s_bytes)) != KATA_OK || (st = check_buffer(z0, z_bytes)) != KATA_OK))
        return st;
    if (S_final &&
        ((st = check_buffer(S_final, s_bytes)) != KATA_OK || (st = check_buffer(z_final, z_bytes)) != KATA_OK))
        return st;
    if (T == 0) {
        if (S_final == nullptr) return KATA_OK;
        cudaError_t e = kata::launch_copy_or_zero(S0, S_final, BH * n * dv, stream);
        if (e == cudaSuccess) e = kata::launch_copy_or_zero(z0, z_final, BH * n, stream);
        return cuda_status(e);
    }
    const size_t qk_bytes = elem_bytes(dt) * BH * T * p, v_bytes = elem_bytes(dt) * BH * T * dv;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(o, v_bytes)) != KATA_OK)
        return st;
    const TcPlan pl = block_tc_plan(dt, family, g, B, H, T, p, dv);
    const ChunkedWs w = pl.use ? pl.ws : chunked_ws(B, H, T, p, dv, C, n);
    if (ws == nullptr || ws_bytes < w.total) return KATA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KATA_ERR_INVALID_ARG;
    if ((st = check_buffer(ws, w.total)) != KATA_OK) return st;
    if (pl.use)
        return cuda_status(launch_tc_forward(pl, q, k, v, o, ws, S0, z0, S_final, z_final, BH, T, p, dv, g, mode, stream));
    const int64_t NC = (T + C - 1) / C;
    float* S_loc = reinterpret_cast<float*>(static_cast<char*>(ws) + w.s_off);
    float* z_loc = reinterpret_cast<float*>(static_cast<char*>(ws) + w.z_off);
    cudaError_t e = kata::launch_block_states(dt, k, v, S_loc, z_loc, (int)BH, T, p, dv, C, family, g, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, S_loc, S_loc, S0, S_final, BH, NC, n * dv, stream);
    if (e == cudaSuccess) e = kata::launch_scan(mode, z_loc, z_loc, z0, z_final, BH, NC, n, stream);
    if (e == cudaSuccess)
        e = kata::launch_block_output(dt, q, k, v, S_loc, z_loc, o, (int)BH, T, p, dv, C, family, g, stream);
    return cuda_status(e);
}

kata_status kata_forward_quadratic_block(const void* q, const void* k, const void* v, void* o, kata_dtype dt, int B,
                                         int H, int T, int p, int dv, kata_lift_family family, int g,
                                         cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv);
    if (st != KATA_OK) return st;
    if ((st = check_lift(family, p, g)) != KATA_OK) return st;
    const int64_t rows = (int64_t)B * H * T;
    if (rows == 0) return KATA_OK;
    const size_t qk_bytes = elem_bytes(dt) * rows * p, v_bytes = elem_bytes(dt) * rows * dv;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(o, v_bytes)) != KATA_OK)
        return st;
    return cuda_status(kata::launch_block_quadratic(dt, q, k, v, o, B * H, T, p, dv, family, g, stream));
}

kata_status kata_decode_step_block(const void* q, const void* k, const void* v, void* o, kata_dtype dt, int B, int H,
                                   int p, int dv, kata_lift_family family, int g, float* S, float* z,
                                   cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, 1, p, dv);
    if (st != KATA_OK) return st;
    if ((st = check_lift(family, p, g)) != KATA_OK) return st;
    return decode_common(q, k, v, o, dt, B, H, p, dv, family, g, S, z, stream);
}

size_t kata_backward_quadratic_workspace_bytes(int B, int H, int T) {
    if (B < 0 || H < 0 || T < 0) return 0;
    const int64_t rows = (int64_t)B * H * T;
    return rows == 0 ? 0 : 2 * round_up(sizeof(float) * (size_t)rows, 256);
}

kata_status kata_backward_quadratic(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk,
                                    void* dv, kata_dtype dt, int B, int H, int T, int p, int dv_dim, void* ws,
                                    size_t ws_bytes, cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv_dim);
    if (st != KATA_OK) return st;
    const int64_t rows = (int64_t)B * H * T;
    if (rows == 0) return KATA_OK;
    const size_t qk_bytes = elem_bytes(dt) * rows * p, v_bytes = elem_bytes(dt) * rows * dv_dim;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(dO, v_bytes)) != KATA_OK ||
        (st = check_buffer(dq, qk_bytes)) != KATA_OK || (st = check_buffer(dk, qk_bytes)) != KATA_OK ||
        (st = check_buffer(dv, v_bytes)) != KATA_OK)
        return st;
    const size_t need = kata_backward_quadratic_workspace_bytes(B, H, T);
    if (ws == nullptr || ws_bytes < need) return KATA_ERR_WORKSPACE;
    if ((st = check_buffer(ws, need)) != KATA_OK) return st;
    float* D_ws = static_cast<float*>(ws);
    float* delta_ws = reinterpret_cast<float*>(static_cast<char*>(ws) + need / 2);
    return cuda_status(kata::launch_backward(dt, q, k, v, dO, dq, dk, dv, D_ws, delta_ws, B * H, T, p, dv_dim,
                                             stream));
}

kata_status kata_decode_step_gated(const void* q, const void* k, const void* v, const float* gate, void* o,
                                   kata_dtype dt, int B, int H, int p, int dv, float* S, float* z,
                                   cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, 1, p, dv);
    if (st != KATA_OK) return st;
    if ((int64_t)B * H > 0 && gate == nullptr) return KATA_ERR_INVALID_ARG;
    return decode_common(q, k, v, o, dt, B, H, p, dv, KATA_LIFT_FULL, 1, S, z, stream, gate);
}

size_t kata_chunked_gated_workspace_bytes(kata_dtype dt, int B, int H, int T, int p, int dv, int C) {
    if (check_shapes(dt, B, H, T, p, dv) != KATA_OK || !c_ok(C)) return 0;
    const int64_t BH = (int64_t)B * H, NC = (T + C - 1) / C;
    if (BH * T == 0) return 0;
    const ChunkedWs w = chunked_ws(B, H, T, p, dv, C);
    // chunk decays a [BH,NC], then the per-token decays dec [BH,T]
    return w.total + round_up(sizeof(float) * (size_t)(BH * NC), 256) + round_up(sizeof(float) * (size_t)(BH * T), 256);
}

kata_status kata_forward_chunked_gated(const void* q, const void* k, const void* v, const float* gate, void* o,
                                       kata_dtype dt, int B, int H, int T, int p, int dv, int C, const float* S0,
                                       const float* z0, float* S_final, float* z_final, void* ws, size_t ws_bytes,
                                       cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv);
    if (st != KATA_OK) return st;
    if (!c_ok(C)) return KATA_ERR_UNSUPPORTED;
    if ((S0 == nullptr) != (z0 == nullptr)) return KATA_ERR_INVALID_ARG;
    if ((S_final == nullptr) != (z_final == nullptr)) return KATA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H, n = packed(p);
    if (BH == 0) return KATA_OK;
    const size_t s_bytes = sizeof(float) * BH * n * dv, z_bytes = sizeof(float) * BH * n;
    if (S0 && ((st = check_buffer(S0, s_bytes)) != KATA_OK || (st = check_buffer(z0, z_bytes)) != KATA_OK))
        return st;
    if (S_final &&
        ((st = check_buffer(S_final, s_bytes)) != KATA_OK || (st = check_buffer(z_final, z_bytes)) != KATA_OK))
        return st;
    if (T == 0) {
        if (S_final == nullptr) return KATA_OK;
        cudaError_t e = kata::launch_copy_or_zero(S0, S_final, BH * n * dv, stream);
        if (e == cudaSuccess) e = kata::launch_copy_or_zero(z0, z_final, BH * n, stream);
        return cuda_status(e);
    }
    const size_t qk_bytes = elem_bytes(dt) * BH * T * p, v_bytes = elem_bytes(dt) * BH * T * dv;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(o, v_bytes)) != KATA_OK ||
        (st = check_buffer(gate, sizeof(float) * (size_t)(BH * T))) != KATA_OK)
        return st;
    const size_t need = kata_chunked_gated_workspace_bytes(dt, B, H, T, p, dv, C);
    if (ws == nullptr || ws_bytes < need) return KATA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KATA_ERR_INVALID_ARG;
    if ((st = check_buffer(ws, need)) != KATA_OK) return st;
    const ChunkedWs w = chunked_ws(B, H, T, p, dv, C);
    float* X = reinterpret_cast<float*>(static_cast<char*>(ws) + w.s_off);
    float* Xz = reinterpret_cast<float*>(static_cast<char*>(ws) + w.z_off);
    float* a = reinterpret_cast<float*>(static_cast<char*>(ws) + w.total);
    float* dec = reinterpret_cast<float*>(static_cast<char*>(ws) + w.total +
                                          round_up(sizeof(float) * (size_t)(BH * ((T + C - 1) / C)), 256));
    return cuda_status(kata::launch_chunked_gated(dt, q, k, v, gate, o, X, Xz, a, dec, S0, z0, S_final, z_final,
                                                  (int)BH, T, p, dv, C, stream));
}

size_t kata_backward_chunked_workspace_bytes(int B, int H, int T, int p, int dv_dim) {
    if (B < 0 || H < 0 || T < 0 || !p_ok(p) || !dv_ok(dv_dim)) return 0;
    const int64_t rows = (int64_t)B * H * T;
    if (rows == 0) return 0;
    const ChunkedWs w = chunked_ws(B, H, T, p, dv_dim, kata::backward_chunk_len());
    return w.total + 2 * round_up(sizeof(float) * (size_t)rows, 256);
}

kata_status kata_backward_chunked(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk,
                                  void* dv, kata_dtype dt, int B, int H, int T, int p, int dv_dim, void* ws,
                                  size_t ws_bytes, cudaStream_t stream) {
    kata_status st = check_shapes(dt, B, H, T, p, dv_dim);
    if (st != KATA_OK) return st;
    const int64_t rows = (int64_t)B * H * T;
    if (rows == 0) return KATA_OK;
    const size_t qk_bytes = elem_bytes(dt) * rows * p, v_bytes = elem_bytes(dt) * rows * dv_dim;
    if ((st = check_buffer(q, qk_bytes)) != KATA_OK || (st = check_buffer(k, qk_bytes)) != KATA_OK ||
        (st = check_buffer(v, v_bytes)) != KATA_OK || (st = check_buffer(dO, v_bytes)) != KATA_OK ||
        (st = check_buffer(dq, qk_bytes)) != KATA_OK || (st = check_buffer(dk, qk_bytes)) != KATA_OK ||
        (st = check_buffer(dv, v_bytes)) != KATA_OK)
        return st;
    const size_t need = kata_backward_chunked_workspace_bytes(B, H, T, p, dv_dim);
    if (ws == nullptr || ws_bytes < need) return KATA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KATA_ERR_INVALID_ARG;
    if ((st = check_buffer(ws, need)) != KATA_OK) return st;
    const ChunkedWs w = chunked_ws(B, H, T, p, dv_dim, kata::backward_chunk_len());
    char* base = static_cast<char*>(ws);
    float* S_ws = reinterpret_cast<float*>(base + w.s_off);
    float* z_ws = reinterpret_cast<float*>(base + w.z_off);
    float* D_ws = reinterpret_cast<float*>(base + w.total);
    float* dl_ws = reinterpret_cast<float*>(base + w.total + round_up(sizeof(float) * (size_t)rows, 256));
    return cuda_status(kata::launch_backward_chunked(dt, q, k, v, dO, dq, dk, dv, S_ws, z_ws, D_ws, dl_ws, (int)(B * H),
                                                     T, p, dv_dim, stream));
}

kata_status kata_get_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KATA_ERR_CUDA;
    unsigned int word = kata::quadratic_tc_take_status();
    word |= kata::states_tc_take_status();
    word |= kata::chunked_tc_take_status();
    return word ? KATA_ERR_TIMEOUT : KATA_OK;
}

}  // extern "C"
