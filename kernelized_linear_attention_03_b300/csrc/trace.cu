// Launch tracing for benchmarks: CUDA event pairs around every kernel launch
// of the library while a trace is active (kata_trace_* in include/kata.h).
#include <mutex>
#include <vector>

#include "../../include/kata.h"
#include "kata_internal.h"

namespace kata {
namespace {

struct Entry {
    const char* name;
    cudaEvent_t start, stop;
    float ms;
};

std::mutex g_mu;
bool g_on = false;
int g_used = 0;
std::vector<Entry> g_entries;

void destroy_all() {
    for (auto& e : g_entries) {
        cudaEventDestroy(e.start);
        cudaEventDestroy(e.stop);
    }
    g_entries.clear();
    g_used = 0;
}

}  // namespace

int trace_begin(const char* name, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on || g_used >= (int)g_entries.size()) return -1;
    const int slot = g_used++;
    g_entries[slot].name = name;
    cudaEventRecord(g_entries[slot].start, s);
    return slot;
}

void trace_end(int slot, cudaStream_t s) {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEventRecord(g_entries[slot].stop, s);
}

}  // namespace kata

extern "C" {

kata_status kata_trace_start(int capacity) {
    if (capacity <= 0 || capacity > (1 << 20)) return KATA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(kata::g_mu);
    kata::destroy_all();
    kata::g_entries.resize(capacity);
    for (auto& e : kata::g_entries) {
        e.name = nullptr;
        e.ms = 0.f;
        if (cudaEventCreate(&e.start) != cudaSuccess || cudaEventCreate(&e.stop) != cudaSuccess) {
            kata::g_entries.clear();
            return KATA_ERR_CUDA;
        }
    }
    kata::g_on = true;
    return KATA_OK;
}

int kata_trace_stop(void) {
    std::lock_guard<std::mutex> lk(kata::g_mu);
    kata::g_on = false;
    for (int i = 0; i < kata::g_used; ++i) {
        auto& e = kata::g_entries[i];
        if (cudaEventSynchronize(e.stop) != cudaSuccess ||
            cudaEventElapsedTime(&e.ms, e.start, e.stop) != cudaSuccess)
            return -1;
    }
    return kata::g_used;
}

kata_status kata_trace_get(int index, const char** name, float* ms) {
    std::lock_guard<std::mutex> lk(kata::g_mu);
    if (index < 0 || index >= kata::g_used || name == nullptr || ms == nullptr) return KATA_ERR_INVALID_ARG;
    *name = kata::g_entries[index].name;
    *ms = kata::g_entries[index].ms;
    return KATA_OK;
}

}  // extern "C"
