// Internal declarations shared by the translation units of the KDA library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kHeadDim = KDA_HEAD_DIM;  // dk = dv = 128
constexpr int kChunk = KDA_CHUNK;       // prefill chunk length
constexpr int kMaxTokensPerRow = KDA_DECODE_MAX_TOKENS;

// Device status word: [0] = first kda_status error code recorded, [1] = its detail.
struct DeviceStatus {
    int32_t code;
    int32_t detail;
};

// Records `code` (if no earlier error is pending) and its detail. Device side.
__device__ __forceinline__ void report_error(DeviceStatus *st, int32_t code, int32_t detail) {
    if (st != nullptr && atomicCAS(&st->code, 0, code) == 0) {
        st->detail = detail;
    }
}

// Address of the device status word of the current device (set up on first use).
cudaError_t device_status_ptr(DeviceStatus **out);

struct DecodeArgs {
    const __nv_bfloat16 *q, *k, *v, *g_raw;
    const float *beta;
    const int32_t *slot_idx;
    void *state_pool;
    int64_t num_slots;
    __nv_bfloat16 *out;
    int32_t rows, num_heads, gate_mode, state_dtype;
    float scale, lower_bound;
    DeviceStatus *status;
    int32_t flags;   // KDA_DECODE_* input options
    float norm_eps;  // with KDA_DECODE_L2NORM_QK
    int32_t tokens;  // tokens per row (>= 1); token rows are laid out [rows][tokens][heads]
};

struct PrefillArgs {
    const __nv_bfloat16 *q, *k, *v, *g_raw;
    const float *beta;
    const int32_t *cu_seqlens;
    const float *init_state;
    __nv_bfloat16 *out;
    float *final_state;
    int32_t num_seqs, total_tokens, num_heads, gate_mode;
    float scale, lower_bound;
    DeviceStatus *status;
    // Window schedule: the chains from launch position `seq_chains` on have their chunks cut
    // into up to `wins` windows of equal length (wins = 1: no windows). Window 0 runs from
    // the initial state like a whole chain and leaves its end state as window 1's start; a
    // window pass computes the end state E (from a zero start) and the linear map M
    // (S_end = M S_start + E) of windows 1 .. wins - 2; the carry chains the start states of
    // windows 2 .. wins - 1; an output pass reruns windows 1 .. wins - 1 from them. `ws`
    // holds these FP32 128 x 128 slots per windowed chain (window_slot).
    int32_t wins;
    float *ws;
    int32_t seq_chains;
    // Per launch: CTAs [0, seq_ctas) run whole chains (positions 0 .. seq_ctas - 1); each later
    // group of win_count CTAs runs windows win_first .. win_first + win_count - 1 of the next
    // windowed chain.
    int32_t seq_ctas, win_first, win_count;
    // Optional intermediate states: every `ckpt_every` tokens (a multiple of the chunk),
    // the state after (j+1) * ckpt_every tokens of sequence n goes to row
    // ckpt_offsets[n] + j of ckpt [ckpt_rows][H][128][128] (ckpt_every = 0: none).
    float *ckpt;
    const int32_t *ckpt_offsets;
    int64_t ckpt_rows;
    int32_t ckpt_every;
};

// Window plan of a prefill call on a device with `sms` multiprocessors.
struct WindowPlan {
    int32_t wins;
    int64_t ws_bytes;
    int32_t seq_chains;  // chains before the windowed ones (0: all chains are windowed)
};
WindowPlan plan_windows(int32_t num_seqs, int32_t total_tokens, int32_t num_heads, int32_t sms);
constexpr int64_t kStateBytes = 128LL * 128 * 4;
// Slots of one windowed chain with `wins` windows: start states of windows 1 .. wins - 1, and
// E and M of windows 1 .. wins - 2.
__host__ __device__ constexpr int64_t window_slots(int64_t wins) { return 3 * wins - 5; }
// After the state slots of all windowed chains: one int32 per (windowed chain, window), set by
// the window pass to whether the window's map M has a nonzero entry, padded to 256 bytes.
__host__ __device__ constexpr int64_t window_flag_bytes(int64_t chains, int64_t wins) {
    return (chains * wins * 4 + 255) / 256 * 256;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream);  // windows when a.wins > 1

}  // namespace kda
