/*
 * kata.h -- C ABI of libkata.so: the KATA causal normalised linear-attention
 * forward ("Kernelized Linear Attention: Breaking the Capacity Wall with
 * Symmetric Cones", arXiv 2607.17419) on NVIDIA B300 (sm_103a).
 *
 * What every forward computes, per batch b, head h, position t (0-based):
 *   qh_t = q_t / ||q_t||, kh_s = k_s / ||k_s||      (unit-sphere projection,
 *        rank-one lift paragraph after Eq. 8; a zero vector stays zero)
 *   psi(u) = u u^T packed into n = p(p+1)/2 coordinates (Eq. 8), diagonal
 *        u_i^2, off-diagonal sqrt(2) u_i u_j, so <psi(a), psi(b)> = (a.b)^2
 *   S_t = S0 + sum_{s<=t} psi(kh_s) v_s^T,  z_t = z0 + sum_{s<=t} psi(kh_s)
 *        (state-size paragraph: S_t = Psi(K_{1:t})^T V_{1:t})
 *   o_t = psi(qh_t)^T S_t / psi(qh_t)^T z_t   (normalised readout with the
 *        denominator psi(q_t)^T Z_t of the Assumption 1 discussion; a zero
 *        denominator gives a zero row).  With S0 = z0 = 0 this equals
 *        o_t = sum_{s<=t} (qh_t.kh_s)^2 v_s / sum_{s<=t} (qh_t.kh_s)^2.
 *
 * Conventions shared by all calls
 *   Layouts   q, k: [B][H][T][p]; v, o: [B][H][T][dv]; all dense row-major.
 *             Packed state S: [B][H][n][dv] fp32, z: [B][H][n] fp32, with
 *             packed index idx(i,j) = i*p - i*(i-1)/2 + (j-i) for i <= j.
 *   Dtypes    KATA_FP32: q, k, v, o are float.  KATA_BF16: q, k, v, o are
 *             bfloat16 (o has the input dtype); accumulation is fp32.
 *   Shapes    p in {16, 32, 64}; dv in {16, 32, 64}; C in {32, 64, 128}
 *             (chunk length; quadratic form also accepts 0 = automatic);
 *             B, H, T >= 0 with B*H <= 65535; T <= 2^30.  Empty inputs
 *             (B*H*T == 0) launch nothing and return KATA_OK (pointers may
 *             then be NULL), except that a forward with T == 0 still writes
 *             S_final = S0 and z_final = z0 when asked.
 *   Pointers  Device pointers (or managed), 16-byte aligned; violations give
 *             KATA_ERR_INVALID_ARG before anything is launched.  The caller
 *             owns all memory; the library allocates no device memory.
 *   Streams   Every call is asynchronous on `stream` (0 = legacy default).
 *             Launch failures return KATA_ERR_CUDA.  Kernels never trap:
 *             a bounded device wait that expires records KATA_ERR_TIMEOUT in
 *             a device status word read by kata_get_device_status().
 *   Threads   Calls on different streams may run concurrently as long as
 *             their output and workspace buffers do not overlap.
 */
#ifndef KATA_H
#define KATA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KATA_API __attribute__((visibility("default")))
#else
#define KATA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KATA_OK = 0,
    KATA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad enum */
    KATA_ERR_UNSUPPORTED = 2,  /* p, dv or C outside the supported set, too large */
    KATA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    KATA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    KATA_ERR_TIMEOUT = 5       /* a bounded device-side wait expired */
} kata_status;

typedef enum { KATA_FP32 = 0, KATA_BF16 = 1 } kata_dtype;

/* Inter-chunk prefix: one step per chunk, or a log-depth tree scan
 * (chunked-scan paragraph): ceil(log2 N_C) levels for N_C up to 256 chunks;
 * longer sequences run one such tree per 256-chunk window, each window
 * starting from the previous one's total. */
typedef enum { KATA_SCAN_SEQUENTIAL = 0, KATA_SCAN_TREE = 1 } kata_scan_mode;

/* n = p(p+1)/2, the packed width of the rank-one lift (Eq. 8); -1 if p < 0. */
KATA_API int kata_packed_dim(int p);

/* Static, human-readable name of a status code; never NULL. */
KATA_API const char* kata_status_string(kata_status status);

/*
 * Flash-style O(T^2) form (the flash-attention-style forward of the
 * abstract): for each query tile, over key tiles up to the diagonal,
 * scores (qh.kh)^2 with the causal mask s <= t, accumulated against [V | 1]
 * and divided by the accumulated row sum.  Needs no workspace.
 *   q, k [B,H,T,p], v [B,H,T,dv] in; o [B,H,T,dv] out (input dtype).
 *   C: query/key tile hint (0, 32, 64 or 128); it does not change results.
 */
KATA_API kata_status kata_forward_quadratic(const void* q, const void* k, const void* v, void* o,
                                   kata_dtype dtype, int B, int H, int T, int p, int dv, int C,
                                   cudaStream_t stream);

/* Bytes of workspace kata_forward_chunked needs for these sizes (0 if none). */
KATA_API size_t kata_chunked_workspace_bytes(kata_dtype dtype, int B, int H, int T, int p, int dv, int C);

/*
 * Exact O(T) chunked-state form (chunked-scan paragraph): local chunk
 * states psi(K_c)^T [V_c | 1], an exclusive prefix over chunks (`mode`),
 * and per chunk the prefix readout psi(Q_c) [S | z] plus the local C x C
 * causal part (Q_c K_c^T)^2 masked times [V_c | 1], then the division.
 *   S0 [B,H,n,dv], z0 [B,H,n]: optional initial state (NULL = zero; give
 *     both or neither).
 *   S_final, z_final: optional state after the last token (NULL = not
 *     written; give both or neither).  May alias S0 / z0.
 *   workspace: device scratch of at least kata_chunked_workspace_bytes(),
 *     256-byte aligned; contents on entry are ignored.  The call owns it
 *     until the stream reaches the end of the call.
 * bf16 inputs run on the tensor cores: a first kernel computes every
 * chunk's local C x C part (into fp32 accumulation rows of the workspace)
 * and the chunk's transposed unit keys, then a state kernel carries each
 * 128-slot tile of the running state on chip and adds the tile's share of
 * every readout to the accumulation rows, and a last pass divides and
 * writes the outputs.  Every kernel of the call runs on `stream`.
 * Results do not depend on C or mode beyond fp32 rounding.
 */
KATA_API kata_status kata_forward_chunked(const void* q, const void* k, const void* v, void* o,
                                 kata_dtype dtype, int B, int H, int T, int p, int dv, int C,
                                 kata_scan_mode mode, const float* S0, const float* z0,
                                 float* S_final, float* z_final, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * Chunk states and their inter-chunk scan (the state kernel and the
 * cumulative pass of the chunked-scan paragraph): with N_C = ceil(T/C),
 *   S_prefix[b,h,c] = sum_{c' < c} psi(K_c')^T V_c'   [B,H,N_C,n,dv] fp32
 *   z_prefix[b,h,c] = sum_{c' < c} psi(K_c')^T 1       [B,H,N_C,n]    fp32
 * (exclusive prefixes: chunk 0 gets zeros).  The per-chunk states are built
 * in the output buffers and scanned in place, so no workspace is needed.
 */
KATA_API kata_status kata_chunk_state_scan(const void* k, const void* v, kata_dtype dtype, int B, int H,
                                  int T, int p, int dv, int C, kata_scan_mode mode,
                                  float* S_prefix, float* z_prefix, cudaStream_t stream);

/*
 * Exclusive prefix over the chunk axis of given chunk states (the
 * cumulative pass alone):
 *   S_prefix[b,h,c] = sum_{c'<c} S_loc[b,h,c'],  z likewise.
 *   S_loc/S_prefix [B,H,NC,n,dv], z_loc/z_prefix [B,H,NC,n], fp32.  Any
 *   n, dv >= 1.  In place (S_prefix == S_loc, z_prefix == z_loc) is allowed;
 *   partial overlap is not.
 */
KATA_API kata_status kata_scan_states(const float* S_loc, const float* z_loc, float* S_prefix,
                             float* z_prefix, int B, int H, int NC, int n, int dv,
                             kata_scan_mode mode, cudaStream_t stream);

/*
 * Recurrent decode step (the constant-time recurrent inference of the
 * abstract: the state recurrence of the state-size paragraph taken one
 * token at a time).  For each b, h, with the new token's q, k [B,H,p] and
 * v [B,H,dv]:
 *   S += psi(kh) v^T,  z += psi(kh)    S [B,H,n,dv], z [B,H,n] fp32, in the
 *                                      packed order above, updated in place
 *   o = psi(qh)^T S / psi(qh)^T z      o [B,H,dv] in the input dtype, read
 *                                      from the updated state (s <= t), a
 *                                      zero denominator giving a zero row.
 * Stepping from S = z = 0 through tokens 0..T-1 gives the forward's rows; a
 * forward's S_final, z_final continue as decode states, and a decode state
 * seeds a forward as S0, z0.  S and z must not overlap each other or q, k,
 * v, o (KATA_ERR_INVALID_ARG if S and z overlap).  Needs no workspace.
 */
KATA_API kata_status kata_decode_step(const void* q, const void* k, const void* v, void* o,
                                      kata_dtype dtype, int B, int H, int p, int dv, float* S,
                                      float* z, cudaStream_t stream);

/*
 * Block lifts: the two reduced PSD families of the paragraph that follows
 * the state-size discussion.  g divides p, m = p/g, and each unit query or
 * key u is cut into g contiguous blocks u_a = (u[a m], ..., u[a m + m - 1]):
 *   KATA_LIFT_SIGMA (KATA-Sigma-g): psi(u) = sum_a u_a u_a^T, one m x m PSD
 *     matrix, n = m(m+1)/2; kernel <psi(q), psi(k)> = sum_{a,b} (q_a.k_b)^2.
 *   KATA_LIFT_MULTI (KATA-M-g): psi(u) = (u_1 u_1^T, ..., u_g u_g^T), the g
 *     packed blocks one after another, n = g m(m+1)/2; kernel
 *     sum_a (q_a.k_a)^2.
 *   KATA_LIFT_FULL: the rank-one lift of Eq. 8 (g must be 1).
 * Inside a block the packing above (idx with m for p, off-diagonals times
 * sqrt 2).  Both families are the full lift at g = 1.  The *_block calls
 * compute the forwards above with this kernel in place of (qh.kh)^2 and
 * this lift in place of psi; states are [B,H,n,dv] / [B,H,n] with the
 * lift's n.  They run on CUDA cores in fp32 for either dtype.
 */
typedef enum { KATA_LIFT_FULL = 0, KATA_LIFT_SIGMA = 1, KATA_LIFT_MULTI = 2 } kata_lift_family;

/* n of a lift for head dimension p; -1 if g < 1, g does not divide p, the
 * family is unknown, or family is KATA_LIFT_FULL with g != 1. */
KATA_API int kata_lift_dim(kata_lift_family family, int p, int g);

/* Bytes of workspace kata_forward_chunked_block needs (0 if none or invalid). */
KATA_API size_t kata_chunked_block_workspace_bytes(kata_dtype dtype, kata_lift_family family, int g, int B,
                                                   int H, int T, int p, int dv, int C);

/*
 * Chunked-state form with a block lift: the three phases of
 * kata_forward_chunked (local chunk states in the lift, exclusive prefix
 * over chunks by `mode`, per chunk the prefix readout plus the local causal
 * part, here from block dot products).  Arguments, state and workspace
 * rules as for kata_forward_chunked, with n = kata_lift_dim(family, p, g).
 * KATA_ERR_INVALID_ARG for an unknown family or g < 1, KATA_ERR_UNSUPPORTED
 * if g does not fit p.
 */
KATA_API kata_status kata_forward_chunked_block(const void* q, const void* k, const void* v, void* o,
                                                kata_dtype dtype, int B, int H, int T, int p, int dv,
                                                int C, kata_lift_family family, int g,
                                                kata_scan_mode mode, const float* S0, const float* z0,
                                                float* S_final, float* z_final, void* workspace,
                                                size_t workspace_bytes, cudaStream_t stream);

/* Flash-style form with a block lift's kernel; as kata_forward_quadratic
 * (no tile hint), errors as kata_forward_chunked_block. */
KATA_API kata_status kata_forward_quadratic_block(const void* q, const void* k, const void* v, void* o,
                                                  kata_dtype dtype, int B, int H, int T, int p,
                                                  int dv, kata_lift_family family, int g,
                                                  cudaStream_t stream);

/* Decode step with a block lift; as kata_decode_step, with S [B,H,n,dv] and
 * z [B,H,n] for n = kata_lift_dim(family, p, g). */
KATA_API kata_status kata_decode_step_block(const void* q, const void* k, const void* v, void* o,
                                            kata_dtype dtype, int B, int H, int p, int dv,
                                            kata_lift_family family, int g, float* S, float* z,
                                            cudaStream_t stream);

/*
 * Gated prefix (the Gated variant: "a Gated prefix adds the learned gate";
 * its recurrence is in an appendix the pages do not contain).  Reading: one
 * scalar gate per head and token, gate [B,H,T] fp32 (values in [0, 1] keep
 * every weight nonnegative; others are used as given), scales the running
 * state before the token's own term is added,
 *   S_t = gate_t S_{t-1} + psi(kh_t) v_t^T,  z_t = gate_t z_{t-1} + psi(kh_t),
 * and the readout is unchanged.  A zero gate forgets everything before its
 * token; all-one gates give kata_forward_chunked.  The chunked form carries
 * per-chunk decays and a one-step-per-chunk gated prefix.  Other arguments,
 * states and errors as for kata_forward_chunked (S0 is scaled by gate_0).
 */
KATA_API size_t kata_chunked_gated_workspace_bytes(kata_dtype dtype, int B, int H, int T, int p, int dv,
                                                   int C);
KATA_API kata_status kata_forward_chunked_gated(const void* q, const void* k, const void* v,
                                                const float* gate, void* o, kata_dtype dtype, int B,
                                                int H, int T, int p, int dv, int C, const float* S0,
                                                const float* z0, float* S_final, float* z_final,
                                                void* workspace, size_t workspace_bytes,
                                                cudaStream_t stream);

/*
 * Gated prefix, flash-style form: the same output as kata_forward_chunked_gated
 * by the O(T^2) route of kata_forward_quadratic, each weight
 * (qh_t.kh_s)^2 carrying the decay prod_{r=s+1..t} gate_r (the gated readout
 * written out over all earlier tokens).  bf16 only (KATA_ERR_UNSUPPORTED for
 * fp32 inputs); gates in [0, 1] (a zero gate forgets everything before its
 * token; values outside [0, 1] are not supported by this form).  The decays
 * are taken from per-token sums of log gates (fp64, stored fp32) in the
 * workspace: at least kata_quadratic_gated_workspace_bytes() bytes, 256-byte
 * aligned.  q, k, v, o, gate and errors as kata_forward_chunked_gated.
 */
KATA_API size_t kata_quadratic_gated_workspace_bytes(kata_dtype dtype, int B, int H, int T);
KATA_API kata_status kata_forward_quadratic_gated(const void* q, const void* k, const void* v,
                                                  const float* gate, void* o, kata_dtype dtype, int B,
                                                  int H, int T, int p, int dv, void* workspace,
                                                  size_t workspace_bytes, cudaStream_t stream);

/* Gated decode step: as kata_decode_step with the state scaled by the head's
 * gate [B,H] fp32 first (S = gate S + psi(kh) v^T, z likewise). */
KATA_API kata_status kata_decode_step_gated(const void* q, const void* k, const void* v,
                                            const float* gate, void* o, kata_dtype dtype, int B, int H,
                                            int p, int dv, float* S, float* z, cudaStream_t stream);

/*
 * Backward: the gradients of L = sum(dO * o) for the forward above (every
 * form computes the same o), by the chain rule through the definition --
 * the pages give no backward algorithm:
 *   dv_s = sum_{t>=s} (w_ts / D_t) dO_t,  w_ts = (qh_t.kh_s)^2, D_t = sum_{s<=t} w_ts
 *   dc_ts = 2 (qh_t.kh_s) (dO_t.v_s - dO_t.o_t) / D_t
 *   dq_t, dk_s: sum_s dc_ts kh_s and sum_t dc_ts qh_t taken back through the
 *   unit-sphere projections (the component along q_t or k_s removed, divided
 *   by its norm).
 * A row with a zero denominator passes no gradient; a zero q or k vector
 * receives none.  q, k, dq, dk [B,H,T,p]; v, dO, dv [B,H,T,dv], all of
 * `dtype` (gradients in the input dtype, fp32 arithmetic).
 * kata_backward_quadratic: O(T^2) work per head (flash-style row and column
 * passes over the causal triangle); workspace at least
 * kata_backward_quadratic_workspace_bytes() bytes, 16-byte aligned.
 */
KATA_API size_t kata_backward_quadratic_workspace_bytes(int B, int H, int T);
KATA_API kata_status kata_backward_quadratic(const void* q, const void* k, const void* v, const void* dO,
                                             void* dq, void* dk, void* dv, kata_dtype dtype, int B, int H,
                                             int T, int p, int dv_dim, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/*
 * The same gradients in O(T) through the chunked form (chunks of 64 tokens,
 * whatever the forward's C): the forward's exclusive prefix states are
 * rebuilt; a query-side pass recomputes each row's normaliser D_t and
 * dO_t . o_t and takes dq from the prefix and the chunk's own keys; the
 * per-chunk gradient states sum_t psi(qh_t) [dO_t / D_t | -dO_t.o_t / D_t]
 * are summed over later chunks (a reverse exclusive prefix); a key-side
 * pass takes dk and dv from them and from the chunk's own later queries.
 * Arguments as kata_backward_quadratic; workspace: at least
 * kata_backward_chunked_workspace_bytes() bytes, 256-byte aligned.
 */
KATA_API size_t kata_backward_chunked_workspace_bytes(int B, int H, int T, int p, int dv_dim);
KATA_API kata_status kata_backward_chunked(const void* q, const void* k, const void* v, const void* dO,
                                           void* dq, void* dk, void* dv, kata_dtype dtype, int B, int H,
                                           int T, int p, int dv_dim, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: KATA_OK, or KATA_ERR_TIMEOUT if a bounded device-side
 * wait expired in an earlier call (that call's outputs are then invalid).
 * KATA_ERR_CUDA if the synchronisation itself fails.
 */
KATA_API kata_status kata_get_device_status(cudaStream_t stream);

/*
 * Chunked forward that allocates nothing (no counterpart in the paper; it
 * exists for callers that cannot call cudaMalloc: a plugin inside a runtime
 * that owns all device allocations, code under a fixed start-up memory
 * budget, or a real-time loop that must not enter the allocator).  Same
 * arguments, results and errors as kata_forward_chunked except that the
 * workspace is a fixed array of KATA_NOALLOC_SCRATCH_BYTES compiled into
 * the library, held by every GPU that loads it until the process exits.
 *   Sizes whose kata_chunked_workspace_bytes() exceeds that limit are
 *   refused with KATA_ERR_UNSUPPORTED before anything is launched.
 *   The first call on a device looks up the array's device address with
 *   that device current (cudaGetSymbolAddress); make that first call before
 *   any stream capture on the device.
 *   Every call shares the one array (its contents are overwritten and need
 *   no clearing): calls that may overlap on the GPU -- on different streams,
 *   or from different threads -- race on it and must be serialised by the
 *   caller, e.g. by issuing them on one stream.
 *   Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define KATA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
KATA_API kata_status kata_forward_chunked_noalloc(const void* q, const void* k, const void* v,
                                                  void* o, kata_dtype dtype, int B, int H, int T,
                                                  int p, int dv, int C, kata_scan_mode mode,
                                                  const float* S0, const float* z0,
                                                  float* S_final, float* z_final,
                                                  cudaStream_t stream);

/*
 * Launch tracing (instrumentation for benchmarks; not part of the method).
 * kata_trace_start(capacity) creates 2*capacity CUDA events and, until
 * kata_trace_stop(), brackets each kernel the library launches (from any
 * thread, on the call's stream) with an event pair.  Launches beyond the
 * capacity are not recorded.  kata_trace_stop() synchronises the recorded
 * events and returns how many launches were recorded (negative on a CUDA
 * error); kata_trace_get(i, &name, &ms) then gives the i-th launch's kernel
 * name (static string) and its device duration in milliseconds.  Starting a
 * new trace discards the previous one.  KATA_ERR_INVALID_ARG for a bad index
 * or capacity.
 */
KATA_API kata_status kata_trace_start(int capacity);
KATA_API int kata_trace_stop(void);
KATA_API kata_status kata_trace_get(int index, const char** name, float* ms);

#ifdef __cplusplus
}
#endif

#endif /* KATA_H */
