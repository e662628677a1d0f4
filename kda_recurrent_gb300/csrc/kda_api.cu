// C ABI of the KDA library: argument checks on the host, the device status word,
// and dispatch to the kernels. See include/kda.h for the contract of each call.
#include <math.h>
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

__device__ DeviceStatus g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
DeviceStatus *g_status_ptr[kMaxDevices] = {};

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

bool valid_gate(int32_t gate_mode, float lower_bound) {
    if (gate_mode < KDA_GATE_LOWER_BOUND || gate_mode > KDA_GATE_LOG_DECAY) return false;
    if (gate_mode == KDA_GATE_LOWER_BOUND && !(isfinite(lower_bound) && lower_bound <= 0.0f)) return false;
    return true;
}

}  // namespace

cudaError_t device_status_ptr(DeviceStatus **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (g_status_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) return e;
        g_status_ptr[dev] = static_cast<DeviceStatus *>(p);
    }
    *out = g_status_ptr[dev];
    return cudaSuccess;
}

}  // namespace kda

using namespace kda;

extern "C" {

int kda_abi_version(void) { return (1 << 16) | 0; }

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported request";
        case KDA_ERR_MISALIGNED: return "misaligned pointer";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case KDA_ERR_DEVICE_INPUT: return "invalid device-resident index data";
        default: return "unknown status";
    }
}

namespace {

int sm_count_of_current_device(int32_t *sms) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KDA_ERR_CUDA;
    *sms = n;
    return KDA_OK;
}

int prefill_common(const void *q, const void *k, const void *v, const void *g_raw, const float *beta,
                   const int32_t *cu_seqlens, const float *init_state, void *out, float *final_state,
                   int32_t num_seqs, int32_t total_tokens, int32_t num_heads, float scale, float lower_bound,
                   int32_t gate_mode, float *ckpt, const int32_t *ckpt_offsets, int64_t ckpt_rows,
                   int32_t ckpt_every, void *workspace, int64_t workspace_bytes, cudaStream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARG;
    if (!isfinite(scale) || !valid_gate(gate_mode, lower_bound)) return KDA_ERR_INVALID_ARG;
    if ((int64_t)total_tokens * num_heads * kHeadDim > (int64_t)1 << 40) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * num_heads > 0x7fffffffLL / 64) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !g_raw || !beta || !out)) return KDA_ERR_INVALID_ARG;
    if (total_tokens == 0 && final_state == nullptr) return KDA_OK;
    const void *p16[] = {q, k, v, g_raw, out, init_state, final_state, workspace};
    for (const void *p : p16)
        if (p && !aligned(p, 16)) return KDA_ERR_MISALIGNED;
    if (!aligned(beta, 4) || !aligned(cu_seqlens, 4)) return KDA_ERR_MISALIGNED;
    if (workspace != nullptr && workspace_bytes < 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_every < 0 || ckpt_every % kChunk != 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_every > 0) {
        if (!ckpt || !ckpt_offsets || ckpt_rows < 1) return KDA_ERR_INVALID_ARG;
        if (!aligned(ckpt, 16) || !aligned(ckpt_offsets, 4)) return KDA_ERR_MISALIGNED;
    }

    PrefillArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.g_raw = static_cast<const __nv_bfloat16 *>(g_raw);
    a.beta = beta;
    a.cu_seqlens = cu_seqlens;
    a.init_state = init_state;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.final_state = final_state;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.num_heads = num_heads;
    a.gate_mode = gate_mode;
    a.scale = scale;
    a.lower_bound = lower_bound;
    a.wins = 1;
    a.ws = nullptr;
    a.seq_chains = 0;
    a.seq_ctas = 0;
    a.win_first = 0;
    a.win_count = 1;
    a.ckpt = ckpt_every > 0 ? ckpt : nullptr;
    a.ckpt_offsets = ckpt_every > 0 ? ckpt_offsets : nullptr;
    a.ckpt_rows = ckpt_every > 0 ? ckpt_rows : 0;
    a.ckpt_every = ckpt_every;
    if (workspace != nullptr) {
        int32_t sms = 0;
        const int st = sm_count_of_current_device(&sms);
        if (st != KDA_OK) return st;
        const WindowPlan plan = plan_windows(num_seqs, total_tokens, num_heads, sms);
        if (plan.wins > 1) {
            if (workspace_bytes < plan.ws_bytes) return KDA_ERR_INVALID_ARG;
            a.wins = plan.wins;
            a.ws = static_cast<float *>(workspace);
            a.seq_chains = plan.seq_chains;
        }
    }
    cudaError_t e = device_status_ptr(&a.status);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    return from_cuda(launch_prefill_tc(a, stream));
}

}  // namespace

int kda_prefill(const void *q, const void *k, const void *v, const void *g_raw, const float *beta,
                const int32_t *cu_seqlens, const float *init_state, void *out, float *final_state,
                int32_t num_seqs, int32_t total_tokens, int32_t num_heads, float scale,
                float lower_bound, int32_t gate_mode, kda_stream_t stream) {
    return prefill_common(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final_state, num_seqs, total_tokens,
                          num_heads, scale, lower_bound, gate_mode, nullptr, nullptr, 0, 0, nullptr, 0,
                          reinterpret_cast<cudaStream_t>(stream));
}

int kda_prefill_ex(const void *q, const void *k, const void *v, const void *g_raw, const float *beta,
                   const int32_t *cu_seqlens, const float *init_state, void *out, float *final_state,
                   int32_t num_seqs, int32_t total_tokens, int32_t num_heads, float scale, float lower_bound,
                   int32_t gate_mode, float *checkpoints, const int32_t *ckpt_offsets, int64_t ckpt_rows,
                   int32_t ckpt_every, void *workspace, int64_t workspace_bytes, kda_stream_t stream) {
    return prefill_common(q, k, v, g_raw, beta, cu_seqlens, init_state, out, final_state, num_seqs, total_tokens,
                          num_heads, scale, lower_bound, gate_mode, checkpoints, ckpt_offsets, ckpt_rows, ckpt_every,
                          workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int64_t kda_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t num_heads, int32_t sm_count) {
    if (num_seqs < 0 || total_tokens < 0 || num_heads < 1 || sm_count < 0) return KDA_ERR_INVALID_ARG;
    if (sm_count == 0) {
        const int st = sm_count_of_current_device(&sm_count);
        if (st != KDA_OK) return st;
    }
    return plan_windows(num_seqs, total_tokens, num_heads, sm_count).ws_bytes;
}

int kda_decode_ex(const void *q, const void *k, const void *v, const void *g_raw, const float *beta,
                  const int32_t *slot_idx, void *state_pool, int64_t num_slots, int32_t state_dtype, void *out,
                  int32_t rows, int32_t tokens_per_row, int32_t num_heads, float scale, float lower_bound,
                  int32_t gate_mode, int32_t flags, float norm_eps, kda_stream_t stream) {
    if (rows < 0 || num_heads < 1 || num_slots < 1 || tokens_per_row < 1) return KDA_ERR_INVALID_ARG;
    if (tokens_per_row > KDA_DECODE_MAX_TOKENS) return KDA_ERR_UNSUPPORTED;
    if (state_dtype != KDA_STATE_F32 && state_dtype != KDA_STATE_BF16) return KDA_ERR_INVALID_ARG;
    if (!isfinite(scale) || !valid_gate(gate_mode, lower_bound)) return KDA_ERR_INVALID_ARG;
    if ((flags & ~(KDA_DECODE_L2NORM_QK | KDA_DECODE_BETA_LOGITS)) != 0) return KDA_ERR_INVALID_ARG;
    if ((flags & KDA_DECODE_L2NORM_QK) && !(isfinite(norm_eps) && norm_eps >= 0.0f)) return KDA_ERR_INVALID_ARG;
    if ((int64_t)rows * tokens_per_row * num_heads * 4 > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    if (num_slots > ((int64_t)1 << 62) / ((int64_t)num_heads * kHeadDim * kHeadDim * 4))
        return KDA_ERR_UNSUPPORTED;
    if (rows == 0) return KDA_OK;
    if (!q || !k || !v || !g_raw || !beta || !slot_idx || !state_pool || !out) return KDA_ERR_INVALID_ARG;
    const void *p16[] = {q, k, v, g_raw, out, state_pool};
    for (const void *p : p16)
        if (!aligned(p, 16)) return KDA_ERR_MISALIGNED;
    if (!aligned(beta, 4) || !aligned(slot_idx, 4)) return KDA_ERR_MISALIGNED;

    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.g_raw = static_cast<const __nv_bfloat16 *>(g_raw);
    a.beta = beta;
    a.slot_idx = slot_idx;
    a.state_pool = state_pool;
    a.num_slots = num_slots;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.rows = rows;
    a.num_heads = num_heads;
    a.gate_mode = gate_mode;
    a.state_dtype = state_dtype;
    a.scale = scale;
    a.lower_bound = lower_bound;
    a.flags = flags;
    a.norm_eps = (flags & KDA_DECODE_L2NORM_QK) ? norm_eps : 0.0f;
    a.tokens = tokens_per_row;
    cudaError_t e = device_status_ptr(&a.status);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    return from_cuda(launch_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

int kda_decode(const void *q, const void *k, const void *v, const void *g_raw, const float *beta,
               const int32_t *slot_idx, void *state_pool, int64_t num_slots, int32_t state_dtype,
               void *out, int32_t rows, int32_t num_heads, float scale, float lower_bound,
               int32_t gate_mode, kda_stream_t stream) {
    return kda_decode_ex(q, k, v, g_raw, beta, slot_idx, state_pool, num_slots, state_dtype, out, rows, 1,
                         num_heads, scale, lower_bound, gate_mode, 0, 0.0f, stream);
}

int kda_device_status(kda_stream_t stream, int32_t *detail) {
    DeviceStatus *dptr = nullptr;
    if (device_status_ptr(&dptr) != cudaSuccess) return KDA_ERR_CUDA;
    DeviceStatus host = {0, 0};
    const DeviceStatus zero = {0, 0};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&host, dptr, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaMemcpyAsync(dptr, &zero, sizeof(zero), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (detail) *detail = host.detail;
    return host.code;
}

}  // extern "C"
