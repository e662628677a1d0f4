/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention hot path.
 *
 * KDA is a gated delta rule with a per-channel log decay. Per head it carries
 * an FP32 state S[dk = 128][dv = 128] and, token by token,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * Two entry points run it on the GPU:
 *   kda_prefill -- varlen sequences, computed chunk by chunk (32 tokens) in the
 *                  chunked form of "FlashInfer PR #4262: CAKE KDA Prefill
 *                  Highlights", section 2 (gate prefix sums, causal Mqk, 32 x 32
 *                  lower-triangular inverse, state decay and projection,
 *                  residual/beta transform, fused state + output update, output
 *                  store);
 *   kda_decode  -- one token per row against a slot-indexed state pool, updated
 *                  in place (FlashInfer PR #5551, "Kimi K3 TP12 H=8 fused KDA
 *                  decode": state pool + slot indices, lower-bound or softplus
 *                  gate, caller-owned outputs).
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless stated, owned by the caller. The
 *     library allocates nothing per call; its only global memory is a small
 *     device status word in the library image (see kda_device_status).
 *   - Every tensor is dense and row-major in the layout given. BF16 means IEEE
 *     bfloat16 bit patterns (uint16 storage). Tensor base addresses must be
 *     16-byte aligned (beta, cu_seqlens and slot_idx: 4-byte), else
 *     KDA_ERR_MISALIGNED.
 *   - The head dimension is fixed: dk = dv = KDA_HEAD_DIM = 128.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream),
 *     never synchronise, and return a kda_status. Argument errors are found on
 *     the host before anything is launched. A failed launch returns
 *     KDA_ERR_CUDA. Errors in device-resident index data are recorded in the
 *     device status word, never by a trap.
 *   - Gate modes: g is a per-channel natural-log decay computed from the raw
 *     gate a (g_raw) as
 *       KDA_GATE_LOWER_BOUND  g = lower_bound * sigmoid(a)   (lower_bound <= 0;
 *                             the "bounded lb" gate of PR #5551/#5565)
 *       KDA_GATE_SOFTPLUS     g = -softplus(a)               (the unbounded
 *                             "Kimi-Linear softplus" gate of PR #5565)
 *       KDA_GATE_LOG_DECAY    g = a                          (a <= 0 supplied
 *                             directly; positive values are not checked and
 *                             make the state grow)
 *   - beta is post-sigmoid, FP32, in [0, 1].
 */
#ifndef KDA_H
#define KDA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* Same type as cudaStream_t; declared here so callers need no CUDA header. */
typedef struct CUstream_st *kda_stream_t;

#define KDA_HEAD_DIM 128
#define KDA_CHUNK 32

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,    /* bad size, NULL pointer, bad mode or scalar        */
    KDA_ERR_UNSUPPORTED = -2,    /* a valid request this build does not run           */
    KDA_ERR_MISALIGNED = -3,     /* a pointer breaks the alignment rule above         */
    KDA_ERR_CUDA = -4,           /* a CUDA runtime call or launch failed              */
    KDA_ERR_DEVICE_TIMEOUT = -5, /* (device status) a bounded device wait gave up     */
    KDA_ERR_DEVICE_INPUT = -6    /* (device status) bad device-resident index data    */
} kda_status;

typedef enum {
    KDA_GATE_LOWER_BOUND = 0,
    KDA_GATE_SOFTPLUS = 1,
    KDA_GATE_LOG_DECAY = 2
} kda_gate_mode;

typedef enum { KDA_STATE_F32 = 0, KDA_STATE_BF16 = 1 } kda_state_dtype;

/*
 * kda_prefill -- chunk-32 varlen prefill.
 *   q, k, g_raw  BF16 [total_tokens, num_heads, 128]   (q, k as given; no normalisation)
 *   v            BF16 [total_tokens, num_heads, 128]
 *   beta         FP32 [total_tokens, num_heads]
 *   cu_seqlens   int32 [num_seqs + 1], device; cu[0] = 0, non-decreasing,
 *                cu[num_seqs] = total_tokens. Sequence n is tokens
 *                [cu[n], cu[n+1]). Violations cannot fault: every index is
 *                clamped into range and KDA_ERR_DEVICE_INPUT is recorded.
 *   init_state   FP32 [num_seqs, num_heads, 128(dk), 128(dv)], or NULL for zeros
 *   out          BF16 [total_tokens, num_heads, 128], written for every token
 *   final_state  FP32 [num_seqs, num_heads, 128, 128], or NULL to skip. May equal
 *                init_state (in-place carry: each chain reads its initial state
 *                before it writes its final state). A zero-length sequence copies
 *                its initial state (or zeros) to final_state.
 *   scale        multiplies every output (typically 1/sqrt(128))
 *   lower_bound  used by KDA_GATE_LOWER_BOUND only; must be finite and <= 0
 *   gate_mode    a kda_gate_mode
 * q/k/v/g_raw/beta must not overlap out or final_state. num_seqs >= 0,
 * total_tokens >= 0, num_heads >= 1. num_seqs == 0 is a no-op.
 * Work: one thread block per (sequence, head) chain walking its chunks in order;
 * the FP32 state stays on chip for the whole sequence.
 */
KDA_API int kda_prefill(const void *q, const void *k, const void *v, const void *g_raw,
                const float *beta, const int32_t *cu_seqlens, const float *init_state,
                void *out, float *final_state, int32_t num_seqs, int32_t total_tokens,
                int32_t num_heads, float scale, float lower_bound, int32_t gate_mode,
                kda_stream_t stream);

/*
 * kda_prefill_workspace_size -- bytes of device workspace kda_prefill_ex uses for a call
 * of this shape; 0 means it would not use any (the chains fill whole waves of the GPU, or
 * leave a last wave of more than a third of it).
 *   sm_count  multiprocessors of the device the call will run on; 0 = ask the current
 *             device (a CUDA call). With sm_count > 0 this is pure host arithmetic.
 * Returns the byte count, or a negative kda_status (KDA_ERR_INVALID_ARG for bad sizes,
 * KDA_ERR_CUDA if the device query fails).
 */
KDA_API int64_t kda_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                           int32_t sm_count);

/*
 * kda_prefill_ex -- kda_prefill with a caller-owned device workspace (16-byte aligned).
 * When the (sequence, head) chains are too few to fill the GPU, each chain's chunks are
 * cut into windows that run in parallel; with more chains than multiprocessors, the
 * same is done for the chains of a last wave that holds at most a third of the GPU,
 * after the full waves have run one CTA per chain. This follows the windowed "affine
 * composite" of FlashInfer PR #5573 ("1. Composite schedule"): window 0 runs from the
 * initial state; beside it a window pass computes, from a zero start, each later window's
 * end state E and linear map M (S_end = M S_start + E); an FP32 carry pass walks the
 * windows of each chain; the output pass then reruns windows 1 onwards from their true
 * start states. Results match kda_prefill up to rounding.
 *   checkpoints      FP32 [ckpt_rows, num_heads, 128, 128] intermediate states, or NULL with
 *                    ckpt_every = 0 (the FP32 checkpoint rows every 64 tokens of FlashInfer PR
 *                    #5565, "1. Kernel body"): with ckpt_every > 0 (a multiple of 32), the state
 *                    after the first (j + 1) * ckpt_every tokens of sequence n, for
 *                    j = 0 .. T_n / ckpt_every - 1, is written to row ckpt_offsets[n] + j.
 *   ckpt_offsets     int32 [num_seqs], device: first checkpoint row of each sequence. A row
 *                    outside [0, ckpt_rows) is skipped and recorded as KDA_ERR_DEVICE_INPUT.
 *   workspace        NULL: the sequential schedule (same as kda_prefill);
 *                    otherwise at least kda_prefill_workspace_size(..., 0) bytes on the
 *                    current device, or KDA_ERR_INVALID_ARG. Its contents on entry do not
 *                    matter; calls sharing one workspace must not overlap on the GPU.
 * All other arguments as kda_prefill.
 */
KDA_API int kda_prefill_ex(const void *q, const void *k, const void *v, const void *g_raw,
                           const float *beta, const int32_t *cu_seqlens, const float *init_state,
                           void *out, float *final_state, int32_t num_seqs, int32_t total_tokens,
                           int32_t num_heads, float scale, float lower_bound, int32_t gate_mode,
                           float *checkpoints, const int32_t *ckpt_offsets, int64_t ckpt_rows,
                           int32_t ckpt_every, void *workspace, int64_t workspace_bytes,
                           kda_stream_t stream);

/*
 * kda_prefill_noalloc -- kda_prefill_ex for callers that cannot allocate device memory.
 * The pages have no counterpart; this is a library convenience. Some callers cannot hand
 * the library a workspace: code embedded in an application that owns every device
 * allocation through its own pool and forbids raw cudaMalloc, or latency-critical paths
 * where an allocation's synchronisation and cost are not acceptable. This call takes the
 * same arguments as kda_prefill and runs the window schedule with its scratch in a
 * fixed array of KDA_NOALLOC_SCRATCH_BYTES (32 MiB) inside the library image. Every GPU
 * that loads the library holds that array until the process exits. The call allocates
 * nothing.
 *   - The first call on a device looks up the array's device address (a CUDA runtime
 *     query, once per device). Make that first call before any stream capture.
 *   - All calls share the one array. Calls whose GPU work overlaps (other streams, other
 *     host threads on the same device) race and must be serialised by the caller. Each
 *     call writes every scratch byte it reads before reading it, so stale contents from
 *     an earlier call never matter.
 *   - A shape whose window plan needs more than KDA_NOALLOC_SCRATCH_BYTES returns
 *     KDA_ERR_UNSUPPORTED. A plan needs at most (3 * SMs - 2) * 64 KiB plus under 1 KiB
 *     of per-window flags, so every plan fits on GPUs with up to 171 SMs (GB300, 152 SMs:
 *     at most 28.4 MiB).
 *   - Shapes that need no windows run the sequential schedule, as kda_prefill.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)
KDA_API int kda_prefill_noalloc(const void *q, const void *k, const void *v, const void *g_raw,
                                const float *beta, const int32_t *cu_seqlens, const float *init_state,
                                void *out, float *final_state, int32_t num_seqs, int32_t total_tokens,
                                int32_t num_heads, float scale, float lower_bound, int32_t gate_mode,
                                kda_stream_t stream);

/*
 * kda_decode -- one token per row (T = 1) against a slot-indexed state pool.
 *   q, k, g_raw  BF16 [rows, num_heads, 128]
 *   v            BF16 [rows, num_heads, 128]
 *   beta         FP32 [rows, num_heads]
 *   slot_idx     int32 [rows], device. Row r updates pool slot slot_idx[r] for every
 *                head. Slots must be unique: rows that share a slot race on it. A build
 *                compiled with KDA_DEBUG_CHECKS first compares every row with the earlier
 *                ones and records the later row of a repeated slot as KDA_ERR_DEVICE_INPUT
 *                (quadratic in rows; the product build does not check). A
 *                negative slot marks a padding row: its outputs are written as
 *                zeros and no state is touched. A slot >= num_slots is treated as
 *                padding and recorded as KDA_ERR_DEVICE_INPUT.
 *   state_pool   [num_slots, num_heads, 128(dk), 128(dv)] of FP32 or BF16
 *                (state_dtype), updated in place. Offsets are 64-bit, so pools of
 *                2^31 elements and more are fine. Slots not named in slot_idx are
 *                never read or written. BF16 states are computed in FP32 and
 *                stored rounded to nearest even.
 *   out          BF16 [rows, num_heads, 128]
 *   scale, lower_bound, gate_mode as for kda_prefill.
 * rows >= 0 (0 is a no-op), num_heads >= 1, num_slots >= 1.
 */
KDA_API int kda_decode(const void *q, const void *k, const void *v, const void *g_raw,
               const float *beta, const int32_t *slot_idx, void *state_pool, int64_t num_slots,
               int32_t state_dtype, void *out, int32_t rows, int32_t num_heads, float scale,
               float lower_bound, int32_t gate_mode, kda_stream_t stream);

/*
 * kda_decode_ex -- kda_decode with several tokens per row and the decode ABI's input
 * options (FlashInfer PR #5551: the persistent_rows ABI passes norm_eps, and the packed
 * decode routes T > 1 to a multi-token kernel; PR #5573 section 3: the kernel applies the
 * logistic function to beta itself).
 *   tokens_per_row  T in [1, KDA_DECODE_MAX_TOKENS]. Row r applies its T tokens in order to
 *                   pool slot slot_idx[r] (read once, written once). q, k, g_raw, v and out
 *                   are [rows, T, num_heads, 128]; beta is [rows, T, num_heads]. T = 1 is
 *                   kda_decode's layout. Larger T gives KDA_ERR_UNSUPPORTED. A BF16 state
 *                   is kept in FP32 between the row's tokens and rounded once when T >= 4;
 *                   for T = 2, 3 it is rounded after every token, as T calls of kda_decode
 *                   would round it.
 *   flags           bitwise OR of
 *                     KDA_DECODE_L2NORM_QK    q and k are first replaced, in FP32, by
 *                                             x * (sum x^2 + norm_eps)^-1/2
 *                     KDA_DECODE_BETA_LOGITS  beta holds logits b; the step uses 1 / (1 + e^-b)
 *                   other bits give KDA_ERR_INVALID_ARG.
 *   norm_eps        used with KDA_DECODE_L2NORM_QK; must be finite and >= 0.
 * All other arguments as kda_decode (which is kda_decode_ex with T = 1 and flags = 0).
 */
#define KDA_DECODE_L2NORM_QK 1
#define KDA_DECODE_BETA_LOGITS 2
#define KDA_DECODE_MAX_TOKENS 16
KDA_API int kda_decode_ex(const void *q, const void *k, const void *v, const void *g_raw,
                          const float *beta, const int32_t *slot_idx, void *state_pool,
                          int64_t num_slots, int32_t state_dtype, void *out, int32_t rows,
                          int32_t tokens_per_row, int32_t num_heads, float scale,
                          float lower_bound, int32_t gate_mode, int32_t flags, float norm_eps,
                          kda_stream_t stream);

/* A static, human-readable name for a kda_status value. Never NULL. */
KDA_API const char *kda_status_string(int status);

/*
 * kda_device_status -- reads and clears the device status word of the current
 * device. Synchronises `stream` (the only entry point that does). Returns KDA_OK,
 * KDA_ERR_DEVICE_INPUT or KDA_ERR_DEVICE_TIMEOUT (the first error recorded since
 * the last read), or KDA_ERR_CUDA if the read itself failed. If `detail` is not
 * NULL it receives a code-specific detail (for KDA_ERR_DEVICE_INPUT: the
 * offending sequence or row index).
 */
KDA_API int kda_device_status(kda_stream_t stream, int32_t *detail);

/* ABI version of this header: (major << 16) | minor. */
KDA_API int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
