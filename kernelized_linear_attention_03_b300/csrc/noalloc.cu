// kata_forward_chunked_noalloc: the chunked forward for callers that cannot
// allocate device memory.  Some callers may not call cudaMalloc at all: a
// plugin inside an inference runtime that owns every device allocation, code
// running under a fixed memory budget decided at start-up, or a real-time
// loop that must not hit the allocator's latency or its implicit
// synchronisation.  They still pass their inputs and outputs; the scratch the
// forward needs comes from one fixed array compiled into this library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  In host
// code its name is only a host-side stand-in, never a device address: the
// device address is looked up once per device with cudaGetSymbolAddress (with
// that device current) on the first call made on that device, and cached.
#include <mutex>

#include "../../include/kata.h"
#include "kata_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = KATA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 128;

}  // namespace

static __device__ __align__(256) unsigned char kata_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call per device, then cached).
cudaError_t scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, kata_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kata_status kata_forward_chunked_noalloc(const void* q, const void* k, const void* v,
                                                    void* o, kata_dtype dtype, int B, int H, int T,
                                                    int p, int dv, int C, kata_scan_mode mode,
                                                    const float* S0, const float* z0,
                                                    float* S_final, float* z_final,
                                                    cudaStream_t stream) {
    const size_t need = kata_chunked_workspace_bytes(dtype, B, H, T, p, dv, C);
    if (need > kNoAllocScratchBytes) return KATA_ERR_UNSUPPORTED;
    void* ws = nullptr;
    if (need > 0 && scratch_on_current_device(&ws) != cudaSuccess) {
        cudaGetLastError();
        return KATA_ERR_CUDA;
    }
    return kata_forward_chunked(q, k, v, o, dtype, B, H, T, p, dv, C, mode, S0, z0, S_final, z_final,
                                ws, need > 0 ? kNoAllocScratchBytes : 0, stream);
}
