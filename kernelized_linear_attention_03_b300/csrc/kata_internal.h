// Internal launchers of libkata (host side).  Every launcher enqueues work on
// `stream` and returns cudaGetLastError() of its launches; argument checking
// happens before, in kata_api.cu.
#pragma once

#include <cuda_runtime_api.h>
#include <cstddef>
#include <cstdint>

namespace kata {

// SIMT flash-style quadratic form, any dtype: o = causal sum (qh.kh)^2 v / sum.
cudaError_t launch_quadratic_simt(int dtype, const void* q, const void* k, const void* v, void* o,
                                  int BH, int T, int p, int dv, cudaStream_t s);

// tcgen05 flash-style quadratic form, bf16 inputs and output.
cudaError_t launch_quadratic_tc(const void* q, const void* k, const void* v, void* o, int BH, int T,
                                int p, int dv, cudaStream_t s);
// Read and clear the device status word of the tensor-core quadratic kernel.
// Gated flash-style form (bf16): per-token log-gate sums and last zero gates
// into ws (quadratic_gated_tc_workspace bytes, 256-byte aligned), then the
// tensor-core kernel with the decays in its weights.
size_t quadratic_gated_tc_workspace(int BH, int T);
cudaError_t launch_quadratic_gated_tc(const void* q, const void* k, const void* v, const float* gate, void* o,
                                      void* ws, int BH, int T, int p, int dv, cudaStream_t s);
unsigned int quadratic_tc_take_status();

// Segment states on the tensor cores (bf16 k, v): for each head and each
// of the first NS segments of L tokens, into S_out [BH, NS_out, n, dv] and
// z_out [BH, NS_out, n] (fp32, sqrt(2)-packed order), for the full lift
// (lg = 1) or KATA-Sigma-g (lg = g > 1, n the lift width of one block).
// NS <= NS_out and NS <= ceil(T / L).  dec (or null; lg = 1 only): [BH, T]
// fp32, a weight on each token's key lift (the gated form's decays).
cudaError_t launch_states_tc(const void* k, const void* v, float* S_out, float* z_out, int BH, int T,
                             int p, int dv, int L, int NS, int NS_out, int prefix, int lg, cudaStream_t s,
                             const float* dec = nullptr);
unsigned int states_tc_take_status();

// Chunked forward on the tensor cores (bf16): one CTA per (head, segment,
// 128-slot tile of the lift).  chunked_tc_segments() gives the number of
// segments G the sequence is cut into on the current device (0 if the
// kernel cannot run there); chunked_tc_segment_chunks() the 128-token
// chunks per segment.  S_start/z_start: [BH, start_groups, n, dv] / [.., n]
// start states (sqrt(2)-packed order; NULL = zero); segment g starts from
// entry g * start_stride (start_groups 1: every segment from entry 0).
// `intra` is chunked_tc_intra_bytes() of device scratch (256-byte aligned)
// for the fp32 accumulation rows of the numerators and denominators and
// the transposed unit keys: the intra-chunk kernel initialises them, the
// state kernel adds to them, a last pass divides.
// lg: blocks of the lift (1: the full lift; 2 or 4: KATA-Sigma-g with
// blocks of p / lg); chunked_tc_supports() tells which (p, dv, lg) exist.
bool chunked_tc_supports(int p, int dv, int lg);
int chunked_tc_segments(int p, int dv, int lg, int BH, int T);
int chunked_tc_segment_chunks(int T, int G);
size_t chunked_tc_intra_bytes(int BH, int T, int p, int dv);
cudaError_t launch_chunked_tc(const void* q, const void* k, const void* v, void* o, void* intra,
                              const float* S_start, const float* z_start, int start_groups, int start_stride,
                              float* S_final, float* z_final, int BH, int T, int p, int dv, int lg, int G,
                              cudaStream_t s);
unsigned int chunked_tc_take_status();

// Per-chunk local states S_loc [BH,NC,n,dv], z_loc [BH,NC,n] (fp32, SIMT).
cudaError_t launch_chunk_states_simt(int dtype, const void* k, const void* v, float* S_loc,
                                     float* z_loc, int BH, int T, int p, int dv, int C,
                                     cudaStream_t s);

// Per-chunk output from exclusive prefixes P [BH,NC,n,dv], Pz [BH,NC,n] (SIMT).
cudaError_t launch_chunk_output_simt(int dtype, const void* q, const void* k, const void* v,
                                     const float* P, const float* Pz, void* o, int BH, int T,
                                     int p, int dv, int C, cudaStream_t s);

// Exclusive prefix over the chunk axis of x [heads, NC, W] into y (y may be
// x).  init [heads, W] (or null) seeds the prefix; fin [heads, W] (or null)
// receives init + total.  mode 0: one step per chunk; 1: log-depth scan.
cudaError_t launch_scan(int mode, const float* x, float* y, const float* init, float* fin,
                        int64_t heads, int64_t NC, int64_t W, cudaStream_t s);

// Recurrent decode step, any dtype: S += psi(kh) v^T, z += psi(kh) in place
// (S [BH,n,dv], z [BH,n] fp32), o = psi(qh)^T S / psi(qh)^T z [BH,dv].
// family 0 (g = 1): the full lift; 1 / 2: KATA-Sigma-g / KATA-M-g
// (block_lift.cuh), n = block_lift_dim(family, p, g).
// gate (or null): [BH] fp32, the gated step S = gate S + psi(kh) v^T (full lift only).
cudaError_t launch_decode_step(int dtype, const void* q, const void* k, const void* v, void* o, float* S,
                               float* z, int BH, int p, int dv, int family, int g, const float* gate,
                               cudaStream_t s);

// Gated chunked forward (any dtype; bf16 chunk states on the tensor cores):
// gate [BH,T] fp32; X [BH,NC,n,dv], Xz [BH,NC,n], a [BH,NC], dec [BH,T] fp32
// scratch; optional S0/z0 and S_final/z_final.
cudaError_t launch_chunked_gated(int dtype, const void* q, const void* k, const void* v, const float* gate, void* o,
                                 float* X, float* Xz, float* a, float* dec, const float* S0, const float* z0,
                                 float* S_final, float* z_final, int BH, int T, int p, int dv, int C, cudaStream_t s);

// Block-lift forwards on CUDA cores (family 1 Sigma-g, 2 M-g; block_lift.cuh),
// any dtype: per-chunk states S_loc [BH,NC,n,dv], z_loc [BH,NC,n] in the
// block lift; per-chunk output from their exclusive prefixes; the
// flash-style quadratic form.
cudaError_t launch_block_states(int dtype, const void* k, const void* v, float* S_loc, float* z_loc, int BH, int T,
                                int p, int dv, int C, int family, int g, cudaStream_t s);
cudaError_t launch_block_output(int dtype, const void* q, const void* k, const void* v, const float* P,
                                const float* Pz, void* o, int BH, int T, int p, int dv, int C, int family, int g,
                                cudaStream_t s);
cudaError_t launch_block_quadratic(int dtype, const void* q, const void* k, const void* v, void* o, int BH, int T,
                                   int p, int dv, int family, int g, cudaStream_t s);

// Backward of the forward (CUDA cores, any dtype): dq, dk [BH,T,p] and dv
// [BH,T,dv] in the input dtype from dO [BH,T,dv]; D_ws and delta_ws are
// [BH,T] fp32 scratch (row normalisers and dO . o).
// O(T) backward through the chunked form; S_ws [BH,NC,n,dv], z_ws [BH,NC,n]
// (NC = ceil(T / backward_chunk_len())), D_ws, delta_ws [BH,T], all fp32.
int backward_chunk_len();
cudaError_t launch_backward_chunked(int dtype, const void* q, const void* k, const void* v, const void* dO, void* dq,
                                    void* dk, void* dv, float* S_ws, float* z_ws, float* D_ws, float* delta_ws, int BH,
                                    int T, int p, int dv_dim, cudaStream_t s);

cudaError_t launch_backward(int dtype, const void* q, const void* k, const void* v, const void* dO, void* dq,
                            void* dk, void* dv, float* D_ws, float* delta_ws, int BH, int T, int p, int dv_dim,
                            cudaStream_t s);

// dst[i] = src ? src[i] : 0 for i < count (fp32), used for pass-through states.
cudaError_t launch_copy_or_zero(const float* src, float* dst, int64_t count, cudaStream_t s);

// Launch tracing (trace.cu): trace_begin returns a slot (or -1 when no trace
// is active) and records its start event; trace_end records the stop event.
int trace_begin(const char* name, cudaStream_t s);
void trace_end(int slot, cudaStream_t s);

// Brackets one kernel launch statement with trace events.
#define KATA_TRACED(name, stream, ...)                            \
    do {                                                          \
        const int kata_slot_ = ::kata::trace_begin(name, stream); \
        __VA_ARGS__;                                              \
        ::kata::trace_end(kata_slot_, stream);                    \
    } while (0)

}  // namespace kata
