// kda_prefill_noalloc: the window-scheduled prefill for callers that cannot allocate
// device memory.
//
// kda_prefill_ex needs a caller-owned workspace when the (sequence, head) chains are too
// few to fill the GPU. Some callers cannot provide one: code embedded in a host
// application that owns every device allocation through its own pool and forbids raw
// cudaMalloc, or a latency-critical path where the synchronisation and cost of an
// allocation are not acceptable. This entry point gives them the same schedule with the
// scratch held in a fixed-size array inside the library image instead.
//
// The array lives for as long as the library is loaded, on every GPU that loads it, and
// all calls share it. Nothing in it needs to start at zero: every call writes each part
// of the scratch it later reads (window end states and maps, then window start states)
// before reading it, so the last call's leftovers are never used. Two calls whose GPU
// work overlaps (different streams, or different host threads on one device) race on
// the array and must be serialised by the caller.
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

// Scratch of the window schedule: 32 MiB. A plan on a GPU with `sms` multiprocessors windows
// the last `tail` chains (tail <= sms / 3) into W <= sms / tail + 1 windows each, and each
// windowed chain needs 3W - 5 FP32 states of 64 KiB, plus one int32 flag per window. So a
// plan needs at most tail (3W - 5) <= 3 sms - 2 tail <= 3 sms - 2 states (454 states,
// 28.4 MiB, on GB300's 152 SMs) and tail W <= sms + tail flags (under 1 KiB); the 512 states
// of this array cover every plan up to 171 SMs.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
// The array's name is a host-side stand-in in host code, so the runtime supplies the
// address the kernels may use.
int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KDA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" int kda_prefill_noalloc(const void *q, const void *k, const void *v, const void *g_raw,
                                   const float *beta, const int32_t *cu_seqlens, const float *init_state,
                                   void *out, float *final_state, int32_t num_seqs, int32_t total_tokens,
                                   int32_t num_heads, float scale, float lower_bound, int32_t gate_mode,
                                   kda_stream_t stream) {
    const int64_t need = kda_prefill_workspace_size(num_seqs, total_tokens, num_heads, 0);
    if (need < 0) return (int)need;
    if (need > (int64_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int st = kda::noalloc_scratch(&scratch);
    if (st != KDA_OK) return st;
    return kda_prefill_ex(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final_state, num_seqs, total_tokens,
                          num_heads, scale, lower_bound, gate_mode, nullptr, nullptr, 0, 0, scratch,
                          (int64_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}
