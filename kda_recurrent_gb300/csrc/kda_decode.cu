// T = 1 KDA decode over a slot-indexed state pool (sm_103a).
//
// Per (row r, head h) the kernel applies one token of
//     S <- Diag(exp g) S ;  w = S^T k ;  u = beta (v - w) ;  S <- S + k u^T ;
//     o = scale S^T q = scale ((Diag(exp g) S)^T q + (q . k) u)
// to pool[slot_idx[r], h] in place (FlashInfer PR #5551, "Kimi K3 TP12 H=8 fused KDA
// decode": slot-indexed FP32/BF16 state pool, lower-bound or softplus gate).
//
// The state is the whole cost: 64 KiB (FP32) or 32 KiB (BF16) read and written per
// item against ~1.3 KB of token I/O, so the kernel is an HBM stream. Each CTA owns a
// 128 x JW column block of one item's state: dv columns are independent (w_j, u_j,
// o_j and the update of column j need only column j and the shared vectors k, q, g),
// so an item splits across CTAs by columns with no communication, which keeps the
// GPU full at small row counts. Every thread issues all of its 16-byte streaming
// loads before any arithmetic, holds its slice in registers, and streams the updated
// slice back; one pass over HBM in each direction.
//
// Slot offsets: one 64-bit base pointer per CTA, then 32-bit offsets inside the
// slot (the PR #5551 lesson on 64-bit per-access arithmetic).
//
// Two schedules, chosen by the item count: few items take the register kernel above,
// split by column blocks so the GPU still fills up; many items take the streaming
// kernel, one persistent CTA per SM that keeps a ring of whole states in shared memory,
// each moved in and out by bulk (TMA) copies, so the copy engines always have the next
// items' states in flight while the current one is updated.
#include "kda_internal.cuh"
#include "kda_mma.cuh"
#include "kda_tc.cuh"

#include <algorithm>
#include <type_traits>

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

__device__ __forceinline__ float gate_log_decay(float a, int mode, float lower_bound) {
    if (mode == KDA_GATE_LOWER_BOUND) return lower_bound / (1.0f + expf(-a));
    if (mode == KDA_GATE_SOFTPLUS) return -(fmaxf(a, 0.0f) + log1pf(expf(-fabsf(a))));
    return a;
}

template <typename T>
struct StateVec;

template <>
struct StateVec<float> {
    static constexpr int kElems = 4;
    using Raw = float4;
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[kElems]) {
        x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
    }
    static __device__ __forceinline__ Raw pack(const float (&x)[kElems]) {
        return make_float4(x[0], x[1], x[2], x[3]);
    }
};

template <>
struct StateVec<__nv_bfloat16> {
    static constexpr int kElems = 8;
    using Raw = uint4;
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[kElems]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ Raw pack(const float (&x)[kElems]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&p);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Four BF16 state elements (8 bytes): the vector of the streaming kernel's register layout
// for BF16 states, which then has the FP32 layout's thread mapping (16 rows x 4 columns per
// thread, 8 row partials per column sum).
struct StateVecBF16x4 {
    static constexpr int kElems = 4;
    using Raw = uint2;
    static __device__ __forceinline__ void unpack(const Raw &r, float (&x)[kElems]) {
        x[0] = __uint_as_float(r.x << 16);
        x[1] = __uint_as_float(r.x & 0xffff0000u);
        x[2] = __uint_as_float(r.y << 16);
        x[3] = __uint_as_float(r.y & 0xffff0000u);
    }
    static __device__ __forceinline__ Raw pack(const float (&x)[kElems]) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(x[0], x[1]), p1 = __floats2bfloat162_rn(x[2], x[3]);
        return make_uint2(*reinterpret_cast<uint32_t *>(&p0), *reinterpret_cast<uint32_t *>(&p1));
    }
};

// The state vector type of the streaming kernel: FP32 states and the BF16 group layout use
// 16 bytes, the BF16 register layout 8.
template <typename T, bool kGroupLayout>
using StreamVec = typename std::conditional<sizeof(T) == 2 && !kGroupLayout, StateVecBF16x4, StateVec<T>>::type;

// The two BF16 halves of a word as FP32 (low half first).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

struct TokenScalars {
    float qk;  // q_n . k_n
    float rq;  // q_n = rq q
    float rk;  // k_n = rk k
};

// Every calling warp computes q.k and, when the call asks for it, the L2 normalisation
// factors (sum x^2 + eps)^-1/2 of q and k from the token vectors in shared memory; each
// warp reads the same 2 x 128 values, so no barrier is needed.
template <typename E>
__device__ __forceinline__ TokenScalars token_scalars(const E *s_q, const E *s_k, const DecodeArgs &a) {
    const int lane = threadIdx.x & 31;
    float qk = 0.0f, qq = 0.0f, kk = 0.0f;
#pragma unroll
    for (int i = lane; i < kHeadDim; i += 32) {
        const float q = static_cast<float>(s_q[i]), k = static_cast<float>(s_k[i]);
        qk = fmaf(q, k, qk);
        qq = fmaf(q, q, qq);
        kk = fmaf(k, k, kk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        qk += __shfl_xor_sync(0xffffffffu, qk, o);
        qq += __shfl_xor_sync(0xffffffffu, qq, o);
        kk += __shfl_xor_sync(0xffffffffu, kk, o);
    }
    TokenScalars t;
    const bool norm = (a.flags & KDA_DECODE_L2NORM_QK) != 0;
    t.rq = norm ? rsqrtf(qq + a.norm_eps) : 1.0f;
    t.rk = norm ? rsqrtf(kk + a.norm_eps) : 1.0f;
    t.qk = qk * t.rq * t.rk;
    return t;
}

// beta as given, or the logistic function of a logit.
__device__ __forceinline__ float beta_of(float b, const DecodeArgs &a) {
    return (a.flags & KDA_DECODE_BETA_LOGITS) ? 1.0f / (1.0f + expf(-b)) : b;
}

template <typename T, int JW>
__global__ void __launch_bounds__(kDecodeThreads) kda_decode_kernel(DecodeArgs a) {
    using V = StateVec<T>;
    constexpr int VEC = V::kElems;            // state elements per 16-byte vector
    constexpr int VPR = JW / VEC;             // vectors per row of the column block
    constexpr int RPP = kDecodeThreads / VPR; // rows covered by one pass of the CTA
    constexpr int NPASS = kHeadDim / RPP;     // passes (vectors held per thread)
    constexpr int NSPLIT = kHeadDim / JW;     // column blocks per item
    // column sums: G threads per (vector, column), each adding PER rows of the partial sums
    constexpr int G = kDecodeThreads / (2 * JW);
    constexpr int PER = RPP / G;
    static_assert(kDecodeThreads % VPR == 0 && kHeadDim % RPP == 0, "tile shape");
    static_assert(2 * JW <= kDecodeThreads && kDecodeThreads % (2 * JW) == 0 && RPP % G == 0, "column sums");

    __shared__ float s_k[kHeadDim], s_q[kHeadDim], s_decay[kHeadDim];
    __shared__ float s_red[2][RPP][JW];
    __shared__ float s_part[2][G][JW];
    __shared__ float s_u[JW];

    const int tid = threadIdx.x;
    const int item = blockIdx.x / NSPLIT;
    const int j0 = (blockIdx.x % NSPLIT) * JW;
    const int r = item / a.num_heads;
    const int h = item - r * a.num_heads;
    const int32_t slot = __ldg(a.slot_idx + r);
    __nv_bfloat16 *out = a.out + (size_t)item * kHeadDim + j0;

    if (slot < 0 || (int64_t)slot >= a.num_slots) {
        // Padding row (negative slot) or a slot past the pool: outputs are zero and no
        // state is touched; the latter is recorded for kda_device_status.
        if ((int64_t)slot >= a.num_slots && tid == 0 && j0 == 0 && h == 0)
            report_error(a.status, KDA_ERR_DEVICE_INPUT, r);
        for (int c = tid; c < JW; c += kDecodeThreads) out[c] = __float2bfloat16_rn(0.0f);
        return;
    }

    T *S = reinterpret_cast<T *>(a.state_pool) +
           ((size_t)slot * (size_t)a.num_heads + (size_t)h) * (size_t)(kHeadDim * kHeadDim) + j0;
    const int cg = tid % VPR;  // this thread's column group inside the block
    const int rg = tid / VPR;  // this thread's first row

    // 1. Issue every state load first; they are the long pole.
    typename V::Raw raw[NPASS];
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        const uint32_t off = (uint32_t)(rg + p * RPP) * kHeadDim + (uint32_t)cg * VEC;
        raw[p] = __ldcs(reinterpret_cast<const typename V::Raw *>(S + off));
    }

    // 2. Token vectors and the per-channel decay while the state is in flight; the column
    //    threads also fetch v and beta now, off the path that follows the column sums.
    const size_t tok = (size_t)item * kHeadDim;
    float v_col = 0.0f, beta_item = 0.0f;
    if (tid < JW) {
        v_col = __bfloat162float(a.v[tok + j0 + tid]);
        beta_item = beta_of(a.beta[item], a);
    }
    if (tid < kHeadDim) {
        const float av = __bfloat162float(a.g_raw[tok + tid]);
        s_decay[tid] = expf(gate_log_decay(av, a.gate_mode, a.lower_bound));
        s_k[tid] = __bfloat162float(a.k[tok + tid]);
        s_q[tid] = __bfloat162float(a.q[tok + tid]);
    }
    __syncthreads();
    const TokenScalars ts = token_scalars(s_q, s_k, a);

    // 3. Decay in registers and this thread's partial (D S)^T k and (D S)^T q.
    float st[NPASS][VEC];
    float wk[VEC], wq[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) wk[e] = wq[e] = 0.0f;
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        V::unpack(raw[p], st[p]);
        const int row = rg + p * RPP;
        const float d = s_decay[row], kk = s_k[row], qq = s_q[row];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            st[p][e] *= d;
            wk[e] = fmaf(st[p][e], kk, wk[e]);
            wq[e] = fmaf(st[p][e], qq, wq[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        s_red[0][rg][cg * VEC + e] = wk[e] * ts.rk;
        s_red[1][rg][cg * VEC + e] = wq[e] * ts.rq;
    }
    __syncthreads();

    // 4. Column sums in two levels over all threads (a warp reads one row of 32 columns per
    //    step, so without bank conflicts), then the delta-rule residual u and the output, one
    //    thread per column.
    {
        const int col = tid % JW, rest = tid / JW;
        const int vec = rest & 1, part = rest >> 1;
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc += s_red[vec][part * PER + i][col];
        s_part[vec][part][col] = acc;
    }
    __syncthreads();
    if (tid < JW) {
        float w_k = 0.0f, w_q = 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            w_k += s_part[0][g][tid];
            w_q += s_part[1][g][tid];
        }
        const float u = beta_item * (v_col - w_k);
        s_u[tid] = u;
        out[tid] = __float2bfloat16_rn(a.scale * fmaf(ts.qk, u, w_q));
    }
    __syncthreads();

    // 5. Rank-one update and streaming store of the slice.
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        const int row = rg + p * RPP;
        const float kk = s_k[row] * ts.rk;
#pragma unroll
        for (int e = 0; e < VEC; ++e) st[p][e] = fmaf(kk, s_u[cg * VEC + e], st[p][e]);
        const uint32_t off = (uint32_t)row * kHeadDim + (uint32_t)cg * VEC;
        __stcs(reinterpret_cast<typename V::Raw *>(S + off), V::pack(st[p]));
    }
}

// ------------------------------------------------------------------ streaming schedule

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_but_newest() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Shared-memory shape of the streaming schedule. A stage holds one item's state and the
// q, k, g_raw, v rows of its `tokens` tokens; the stage count is whatever fits in
// kStreamSmem (at most kMaxStages), so that 2-5 items are in flight per SM.
template <typename T, bool kGroupLayout = sizeof(T) == 2>
struct StreamShape {
    static constexpr int kMaxStages = 6;
    static constexpr uint32_t kItemBytes = kHeadDim * kHeadDim * sizeof(T);
    static constexpr uint32_t kPiece = 16384;               // bytes per bulk copy of the state
    static constexpr uint32_t kTokBytes = 4 * kHeadDim * 2;  // q, k, g_raw, v rows of one token
    static constexpr int VEC = StreamVec<T, kGroupLayout>::kElems;
    static constexpr int RPP = kDecodeThreads / (kHeadDim / VEC);
    // BF16 states with one token per row are updated by two groups of four warps, one item
    // each (see below); FP32 states, and BF16 states with several tokens per row, by all eight
    // compute warps, the state in FP32 registers for the whole row
    static constexpr bool kGroups = kGroupLayout;
    static constexpr int kGroupBytes = 2 * 8 * kHeadDim * 4 + 4 * kHeadDim * 4 + kMaxTokensPerRow * 4;
    static constexpr int kRed = 2 * RPP * kHeadDim * 4;
    // FP32 states: the partial sums, u and beta, then the decay, k and q vectors of every
    // token of the item ([tokens][3][128], filled once per item); the mbarriers last
    static constexpr int kScalars = kRed + kHeadDim * 4 + kMaxTokensPerRow * 4 + kMaxTokensPerRow * 16;
    static constexpr int kBarBytes = 2 * kMaxStages * 8 + 16;  // full[], done[], two abort flags
    static __host__ __device__ int fixed(int tokens) {
        return (kGroups ? 2 * kGroupBytes : kScalars + 3 * tokens * kHeadDim * 4) + kBarBytes;
    }
    static constexpr int kStreamSmem = 227 * 1024;
    static __host__ __device__ uint32_t stage_bytes(int tokens) { return kItemBytes + kTokBytes * tokens; }
    static __host__ __device__ int stages(int tokens) {
        const int n = (int)((kStreamSmem - fixed(tokens)) / stage_bytes(tokens));
        // consecutive fills of a stage are NS items apart; with two compute groups taking
        // alternate items, an even NS gives both fills to the same group, which waits for the
        // earlier fill's phase before it can wait for the later one
        return kGroups ? (n < kMaxStages ? n : kMaxStages) & ~1 : (n < kMaxStages ? n : kMaxStages);
    }
    static __host__ __device__ int smem(int tokens) { return stages(tokens) * stage_bytes(tokens) + fixed(tokens); }
};

__device__ __forceinline__ void compute_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kDecodeThreads) : "memory"); }

// BF16 states, streaming schedule: the eight compute warps form two groups of four, and
// group g updates the items with an even (g = 0) or odd (g = 1) local index, so one group's
// barriers and latencies overlap the other's arithmetic. The state stays in its ring stage:
// thread (row group rg, 8-column block cb) reads its 16 x 8 slice once to form the decayed
// projections S^T k and S^T q, and once more to write Diag(exp g) S + k u^T back in place.
__device__ __forceinline__ void stream_groups_bf16(const DecodeArgs &a, uint8_t *stages, uint8_t *scratch, int NS,
                                                 uint32_t stage_bytes, uint64_t *full, uint64_t *done, int64_t first,
                                                 int64_t stride, int mine, volatile int *s_abort) {
    using SS = StreamShape<__nv_bfloat16>;
    const int tid = threadIdx.x;
    const int grp = tid >> 7, gt = tid & 127;
    const int cb = gt & 15, rg = gt >> 4;  // columns 8 cb .. 8 cb + 7, rows 16 rg .. 16 rg + 15
    float *const s_red = reinterpret_cast<float *>(scratch + grp * SS::kGroupBytes);  // [2][8][128]
    float *const s_k = s_red + 2 * 8 * kHeadDim;
    float *const s_q = s_k + kHeadDim;
    float *const s_decay = s_q + kHeadDim;
    float *const s_u = s_decay + kHeadDim;
    float *const s_beta = s_u + kHeadDim;  // [kMaxTokensPerRow]
    const int TT = a.tokens;
    const int H = a.num_heads;
    auto gbar = [&]() {
        if (grp == 0)
            asm volatile("bar.sync 2, 128;" ::: "memory");
        else
            asm volatile("bar.sync 3, 128;" ::: "memory");
    };
    auto slot_of = [&](int64_t item) -> int64_t {
        const int32_t slot = __ldg(a.slot_idx + (int)(item / H));
        return (slot >= 0 && (int64_t)slot < a.num_slots) ? (int64_t)slot : -1;
    };
    auto tok_index = [&](int64_t item, int t) -> size_t {
        const int64_t r = item / H, h = item % H;
        return ((size_t)r * TT + t) * (size_t)H + (size_t)h;
    };
    int64_t slot_next = grp < mine ? slot_of(first + grp * stride) : -1;
    float beta_next = (grp < mine && gt < TT) ? a.beta[tok_index(first + grp * stride, gt)] : 0.0f;
    for (int kk = grp; kk < mine; kk += 2) {
        const int st = kk % NS;
        const int64_t item = first + (int64_t)kk * stride;
        const int r = (int)(item / H);
        const int64_t slot = slot_next;
        const float beta_mine = beta_next;
        if (kk + 2 < mine) {
            slot_next = slot_of(item + 2 * stride);
            if (gt < TT) beta_next = a.beta[tok_index(item + 2 * stride, gt)];
        }
        // a wait that gave up is recorded in the group's flag; the group reads the flag after
        // its next barrier, so all of it takes the same decision (a wait that gave up in some
        // threads only must not split the group at a barrier)
        const bool got = mbar_wait(&full[st], (uint32_t)(kk / NS) & 1u);
        if (!got) {
            report_error(a.status, KDA_ERR_DEVICE_TIMEOUT, (int)blockIdx.x);
            s_abort[grp] = 1;
        }
        if (slot < 0) {
            for (int t = 0; t < TT; ++t) a.out[tok_index(item, t) * kHeadDim + gt] = __float2bfloat16_rn(0.0f);
            const int32_t raw_slot = __ldg(a.slot_idx + r);
            if (gt == 0 && (int64_t)raw_slot >= a.num_slots && item % H == 0)
                report_error(a.status, KDA_ERR_DEVICE_INPUT, r);
            mbar_arrive(&done[st]);
            continue;
        }
        uint8_t *const S = stages + (size_t)st * stage_bytes;  // bf16 [128 dk][128 dv]
        gbar();  // the previous item's use of the group's vectors (and state slice) is over
        if (s_abort[grp] != 0) break;  // read after the group barrier: one decision for the group
        for (int t = 0; t < TT; ++t) {
            const __nv_bfloat16 *trow =
                reinterpret_cast<const __nv_bfloat16 *>(S + SS::kItemBytes + t * SS::kTokBytes);
            if (t > 0) gbar();  // the previous token's use of the group's vectors is over
            {
                const float av = __bfloat162float(trow[2 * kHeadDim + gt]);
                s_decay[gt] = expf(gate_log_decay(av, a.gate_mode, a.lower_bound));
                s_k[gt] = __bfloat162float(trow[kHeadDim + gt]);
                s_q[gt] = __bfloat162float(trow[gt]);
            }
            if (t == 0 && gt < TT) s_beta[gt] = beta_mine;
            gbar();
            const TokenScalars ts = token_scalars(s_q, s_k, a);
            // packed FP32 pairs of columns; the per-row vectors are read four rows at a time
            float2 wk[4], wq[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) wk[e] = wq[e] = make_float2(0.0f, 0.0f);
#pragma unroll 2
            for (int i4 = 0; i4 < 4; ++i4) {
                const int row0 = 16 * rg + 4 * i4;
                const float4 d4 = *reinterpret_cast<const float4 *>(s_decay + row0);
                const float4 k4 = *reinterpret_cast<const float4 *>(s_k + row0);
                const float4 q4 = *reinterpret_cast<const float4 *>(s_q + row0);
                const float dr[4] = {d4.x, d4.y, d4.z, d4.w}, kr[4] = {k4.x, k4.y, k4.z, k4.w};
                const float qr[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(S + ((row0 + r) * kHeadDim + 8 * cb) * 2);
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 y = __fmul2_rn(bf16x2_to_float2(w[e]), make_float2(dr[r], dr[r]));
                        wk[e] = __ffma2_rn(y, make_float2(kr[r], kr[r]), wk[e]);
                        wq[e] = __ffma2_rn(y, make_float2(qr[r], qr[r]), wq[e]);
                    }
                }
            }
            float *const rk = s_red + rg * kHeadDim + 8 * cb;
            float *const rq = s_red + (8 + rg) * kHeadDim + 8 * cb;
            const float2 rk2 = make_float2(ts.rk, ts.rk), rq2 = make_float2(ts.rq, ts.rq);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                reinterpret_cast<float2 *>(rk)[e] = __fmul2_rn(wk[e], rk2);
                reinterpret_cast<float2 *>(rq)[e] = __fmul2_rn(wq[e], rq2);
            }
            gbar();
            {  // column j = gt
                float w_k = 0.0f, w_q = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    w_k += s_red[i * kHeadDim + gt];
                    w_q += s_red[(8 + i) * kHeadDim + gt];
                }
                const float u = beta_of(s_beta[t], a) * (__bfloat162float(trow[3 * kHeadDim + gt]) - w_k);
                s_u[gt] = u;
                a.out[tok_index(item, t) * kHeadDim + gt] = __float2bfloat16_rn(a.scale * fmaf(ts.qk, u, w_q));
            }
            gbar();
            float2 uv[4];
            {
                const float4 u0 = *reinterpret_cast<const float4 *>(s_u + 8 * cb);
                const float4 u1 = *reinterpret_cast<const float4 *>(s_u + 8 * cb + 4);
                uv[0] = make_float2(u0.x, u0.y), uv[1] = make_float2(u0.z, u0.w);
                uv[2] = make_float2(u1.x, u1.y), uv[3] = make_float2(u1.z, u1.w);
            }
#pragma unroll 2
            for (int i4 = 0; i4 < 4; ++i4) {
                const int row0 = 16 * rg + 4 * i4;
                const float4 d4 = *reinterpret_cast<const float4 *>(s_decay + row0);
                const float4 k4 = *reinterpret_cast<const float4 *>(s_k + row0);
                const float dr[4] = {d4.x, d4.y, d4.z, d4.w};
                const float kr[4] = {k4.x * ts.rk, k4.y * ts.rk, k4.z * ts.rk, k4.w * ts.rk};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    uint4 *const p = reinterpret_cast<uint4 *>(S + ((row0 + r) * kHeadDim + 8 * cb) * 2);
                    const uint4 raw = *p;
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = __ffma2_rn(make_float2(kr[r], kr[r]), uv[e],
                                                    __fmul2_rn(bf16x2_to_float2(w[e]), make_float2(dr[r], dr[r])));
                        o[e] = pack_bf16(x.x, x.y);
                    }
                    *p = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        fence_async_smem();
        mbar_arrive(&done[st]);
    }
}

// One CTA per SM: warps 0-7 update states; warp 8 (lane 0) moves them. Stage s is filled by
// bulk copies that complete `full[s]`; the compute warps arrive on `done[s]` once the
// updated state is back in the stage; the producer then stores it with a bulk copy. It
// refills a stage with the state NS items ahead one item later, once the store has read
// the stage: waiting for that read right after issuing the store kept the producer from
// issuing anything else for the length of the read. A ring of only two stages (FP32 states
// with 6 or more tokens per row) is the exception (kRefillAtOnce): there the deferred refill
// would start the next item's load only once the compute warps want it, so each stage is
// refilled as soon as its store has read it. With several tokens per row the state stays in
// registers while its tokens are applied in order, and is stored once.
template <typename T, bool kRefillAtOnce, bool kGroupLayout>
__global__ void __launch_bounds__(kDecodeThreads + 32, 1) kda_decode_stream_kernel(DecodeArgs a) {
    using V = StreamVec<T, kGroupLayout>;
    using SS = StreamShape<T, kGroupLayout>;
    constexpr int VEC = V::kElems;
    constexpr int VPR = kHeadDim / VEC;
    constexpr int RPP = SS::RPP;
    constexpr int NPASS = kHeadDim / RPP;
    const int TT = a.tokens;
    const int NS = SS::stages(TT);
    const uint32_t stage_bytes = SS::stage_bytes(TT);
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *const stages = smem;
    float *const s_red = reinterpret_cast<float *>(smem + NS * stage_bytes);  // [2][RPP][128]
    float *const s_u = s_red + 2 * RPP * kHeadDim;
    float *const s_beta = s_u + kHeadDim;        // [kMaxTokensPerRow]
    float4 *const s_ts = reinterpret_cast<float4 *>(s_beta + kMaxTokensPerRow);  // [kMaxTokensPerRow] (qk, rq, rk)
    float *const s_vec = reinterpret_cast<float *>(s_ts + kMaxTokensPerRow);     // [TT][decay, k, q][128]
    uint64_t *const full = reinterpret_cast<uint64_t *>(smem + NS * stage_bytes + SS::fixed(TT) - SS::kBarBytes);
    uint64_t *const done = full + SS::kMaxStages;

    const int tid = threadIdx.x;
    const int H = a.num_heads;
    const int64_t items = (int64_t)a.rows * H;
    const int64_t first = blockIdx.x, stride = gridDim.x;
    const int mine = items > first ? (int)((items - first + stride - 1) / stride) : 0;
    // per compute group: a stage wait gave up (set by the threads whose wait failed, read by
    // all after the group's next barrier)
    volatile int *const s_abort = reinterpret_cast<volatile int *>(done + SS::kMaxStages);
    if (tid == 0) {
        for (int st = 0; st < NS; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&done[st], SS::kGroups ? kDecodeThreads / 2 : kDecodeThreads);
        }
        fence_mbar_init();
        s_abort[0] = s_abort[1] = 0;
    }
    __syncthreads();

    auto slot_of = [&](int64_t item) -> int64_t {  // slot of an item, or -1 (padding / past the pool)
        const int32_t slot = __ldg(a.slot_idx + (int)(item / H));
        return (slot >= 0 && (int64_t)slot < a.num_slots) ? (int64_t)slot : -1;
    };
    auto state_ptr = [&](int64_t item, int64_t slot) -> uint8_t * {
        const int h = (int)(item % H);
        return reinterpret_cast<uint8_t *>(reinterpret_cast<T *>(a.state_pool) +
                                           ((size_t)slot * (size_t)H + (size_t)h) * (kHeadDim * kHeadDim));
    };
    // element offset of the token rows / flat index of (item, token t): layout [rows][tokens][H]
    auto tok_index = [&](int64_t item, int t) -> size_t {
        const int64_t r = item / H, h = item % H;
        return ((size_t)r * TT + t) * (size_t)H + (size_t)h;
    };

    if (tid >= kDecodeThreads) {
        // ---- producer warp
        if (tid != kDecodeThreads) return;
        auto issue = [&](int kk) {
            const int st = kk % NS;
            const int64_t item = first + (int64_t)kk * stride;
#ifdef KDA_TEST_WITHHOLD_HANDOFF
            // failure-detection test build only: the fill of this item is lost, so the compute
            // warps' bounded wait for it runs out and the CTA takes its abort path
            if (kk == KDA_TEST_WITHHOLD_HANDOFF) return;
#endif
            const int64_t slot = slot_of(item);
            if (slot < 0) {
                mbar_arrive(&full[st]);
                return;
            }
            const uint8_t *src = state_ptr(item, slot);
            uint8_t *dst = stages + (size_t)st * stage_bytes;
            mbar_expect_tx(&full[st], stage_bytes);
#pragma unroll
            for (uint32_t p = 0; p < SS::kItemBytes; p += SS::kPiece)
                bulk_load(smem_addr(dst + p), src + p, SS::kPiece, &full[st]);
            for (int t = 0; t < TT; ++t) {
                const size_t tok = tok_index(item, t) * kHeadDim;
                const __nv_bfloat16 *rows[4] = {a.q + tok, a.k + tok, a.g_raw + tok, a.v + tok};
                uint8_t *tdst = dst + SS::kItemBytes + t * SS::kTokBytes;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    bulk_load(smem_addr(tdst + m * kHeadDim * 2), rows[m], kHeadDim * 2, &full[st]);
            }
        };
        int issued = 0;
        for (int kk = 0; kk < NS && kk < mine; ++kk) issue(kk), issued = kk + 1;
        for (int j = 0; j < mine; ++j) {
            const int st = j % NS;
            if (!mbar_wait(&done[st], (uint32_t)(j / NS) & 1u)) {
                report_error(a.status, KDA_ERR_DEVICE_TIMEOUT, (int)blockIdx.x);
                // the fills of items j .. issued - 1 may still be writing their stages (one per
                // stage): wait for them, bounded, before the CTA's shared memory is released
                for (int kk = j; kk < issued; ++kk) mbar_wait(&full[kk % NS], (uint32_t)(kk / NS) & 1u);
                break;
            }
            const int64_t item = first + (int64_t)j * stride;
            const int64_t slot = slot_of(item);
            if (slot >= 0) {
                uint8_t *dst = state_ptr(item, slot);
#pragma unroll
                for (uint32_t p = 0; p < SS::kItemBytes; p += SS::kPiece)
                    bulk_store(dst + p, smem_addr(stages + (size_t)st * stage_bytes + p), SS::kPiece);
            }
            bulk_commit();  // one group per item, empty for a skipped one
            if constexpr (kRefillAtOnce) {
                // this item's stage takes the item NS ahead as soon as the store has read it
                if (j + NS < mine) {
                    bulk_wait_read_all();
                    issue(j + NS);
                    issued = j + NS + 1;
                }
            } else if (j >= 1 && j - 1 + NS < mine) {
                // the stage of the previous item is refilled once its store has read it, which
                // has had this item's wait to happen in
                bulk_wait_read_but_newest();
                issue(j - 1 + NS);
                issued = j + NS;
            }
        }
        bulk_wait_all();
        return;
    }

    // ---- compute warps
    if constexpr (SS::kGroups) {
        static_assert(sizeof(T) == 2, "the group layout is for BF16 states");
        stream_groups_bf16(a, stages, smem + NS * stage_bytes, NS, stage_bytes, full, done, first, stride, mine,
                           s_abort);
        return;
    }
    const int cg = tid % VPR, rg = tid / VPR;
    int64_t slot_next = mine > 0 ? slot_of(first) : -1;
    float beta_next = (mine > 0 && tid < TT) ? a.beta[tok_index(first, tid)] : 0.0f;
    for (int kk = 0; kk < mine; ++kk) {
        const int st = kk % NS;
        const int64_t item = first + (int64_t)kk * stride;
        const int r = (int)(item / H);
        const int64_t slot = slot_next;
        const float beta_mine = beta_next;  // beta of token `tid` of this item (tid < TT)
        if (kk + 1 < mine) {
            slot_next = slot_of(item + stride);
            if (tid < TT) beta_next = a.beta[tok_index(item + stride, tid)];
        }
        // a wait that gave up is recorded in the flag, which every compute thread reads after
        // the next barrier (a wait that gave up in some threads only must not split them there)
        if (!mbar_wait(&full[st], (uint32_t)(kk / NS) & 1u)) {
            report_error(a.status, KDA_ERR_DEVICE_TIMEOUT, (int)blockIdx.x);
            s_abort[0] = 1;
        }
        if (slot < 0) {
            if (tid < kHeadDim)
                for (int t = 0; t < TT; ++t) a.out[tok_index(item, t) * kHeadDim + tid] = __float2bfloat16_rn(0.0f);
            const int32_t raw_slot = __ldg(a.slot_idx + r);
            if (tid == 0 && (int64_t)raw_slot >= a.num_slots && item % H == 0)
                report_error(a.status, KDA_ERR_DEVICE_INPUT, r);
            mbar_arrive(&done[st]);
            continue;
        }
        T *S = reinterpret_cast<T *>(stages + (size_t)st * stage_bytes);
        float stv[NPASS][VEC];
#pragma unroll
        for (int p = 0; p < NPASS; ++p) {
            const typename V::Raw raw =
                *reinterpret_cast<const typename V::Raw *>(S + (rg + p * RPP) * kHeadDim + cg * VEC);
            V::unpack(raw, stv[p]);
        }
        // the decay, k and q vectors of all the item's tokens at once, so that each token
        // step needs only the two barriers around its column sums. Channel c is stored at
        // (c mod RPP) NPASS + c / RPP, so that the NPASS rows a thread owns are contiguous.
        const __nv_bfloat16 *const rows0 =
            reinterpret_cast<const __nv_bfloat16 *>(stages + (size_t)st * stage_bytes + SS::kItemBytes);
        compute_bar();  // the previous item's use of the shared vectors is over
        // read after the barrier, the flag gives all compute threads one decision
        if (s_abort[0] != 0) break;
        for (int x = tid; x < TT * kHeadDim; x += kDecodeThreads) {
            const int t = x >> 7, c = x & (kHeadDim - 1);
            const int pc = (c % RPP) * NPASS + c / RPP;
            const __nv_bfloat16 *trow = rows0 + t * (SS::kTokBytes / 2);
            float *const v3 = s_vec + t * 3 * kHeadDim;
            v3[pc] = expf(gate_log_decay(__bfloat162float(trow[2 * kHeadDim + c]), a.gate_mode, a.lower_bound));
            v3[kHeadDim + pc] = __bfloat162float(trow[kHeadDim + c]);
            v3[2 * kHeadDim + pc] = __bfloat162float(trow[c]);
        }
        if (tid < TT) s_beta[tid] = beta_mine;
        // q.k and the normalisation factors of token t by warp t mod 8, from the token rows
        for (int t = tid >> 5; t < TT; t += kDecodeThreads / 32) {
            const __nv_bfloat16 *trow = rows0 + t * (SS::kTokBytes / 2);
            const TokenScalars x = token_scalars(trow, trow + kHeadDim, a);
            if ((tid & 31) == 0) s_ts[t] = make_float4(x.qk, x.rq, x.rk, 0.0f);
        }
        compute_bar();
        __nv_bfloat16 *const out_row = a.out + tok_index(item, 0) * kHeadDim;  // token t at t * out_tok_stride
        const size_t out_tok_stride = (size_t)H * kHeadDim;
        for (int t = 0; t < TT; ++t) {
            const __nv_bfloat16 *trow = rows0 + t * (SS::kTokBytes / 2);
            const float *const s_decay = s_vec + t * 3 * kHeadDim;
            const float *const s_k = s_decay + kHeadDim;
            const float *const s_q = s_k + kHeadDim;
            TokenScalars ts;
            {
                const float4 x = s_ts[t];
                ts.qk = x.x, ts.rq = x.y, ts.rk = x.z;
            }
            // this thread's rows rg + p RPP of the decay, k and q vectors, 16 bytes at a time
            float dv[NPASS], kv[NPASS], qv[NPASS];
#pragma unroll
            for (int p4 = 0; p4 < NPASS / 4; ++p4) {
                const float4 d4 = reinterpret_cast<const float4 *>(s_decay + rg * NPASS)[p4];
                const float4 k4 = reinterpret_cast<const float4 *>(s_k + rg * NPASS)[p4];
                const float4 q4 = reinterpret_cast<const float4 *>(s_q + rg * NPASS)[p4];
                dv[4 * p4] = d4.x, dv[4 * p4 + 1] = d4.y, dv[4 * p4 + 2] = d4.z, dv[4 * p4 + 3] = d4.w;
                kv[4 * p4] = k4.x, kv[4 * p4 + 1] = k4.y, kv[4 * p4 + 2] = k4.z, kv[4 * p4 + 3] = k4.w;
                qv[4 * p4] = q4.x, qv[4 * p4 + 1] = q4.y, qv[4 * p4 + 2] = q4.z, qv[4 * p4 + 3] = q4.w;
            }
            // packed FP32 pairs of columns (one instruction for two lanes of the pair)
            float2 wk[VEC / 2], wq[VEC / 2];
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e) wk[e] = wq[e] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int p = 0; p < NPASS; ++p) {
                const float2 d = make_float2(dv[p], dv[p]);
                const float2 kr = make_float2(kv[p], kv[p]), qr = make_float2(qv[p], qv[p]);
#pragma unroll
                for (int e = 0; e < VEC / 2; ++e) {
                    const float2 y = __fmul2_rn(make_float2(stv[p][2 * e], stv[p][2 * e + 1]), d);
                    stv[p][2 * e] = y.x;
                    stv[p][2 * e + 1] = y.y;
                    wk[e] = __ffma2_rn(y, kr, wk[e]);
                    wq[e] = __ffma2_rn(y, qr, wq[e]);
                }
            }
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e) {
                *reinterpret_cast<float2 *>(&s_red[(0 * RPP + rg) * kHeadDim + cg * VEC + 2 * e]) =
                    __fmul2_rn(wk[e], make_float2(ts.rk, ts.rk));
                *reinterpret_cast<float2 *>(&s_red[(1 * RPP + rg) * kHeadDim + cg * VEC + 2 * e]) =
                    __fmul2_rn(wq[e], make_float2(ts.rq, ts.rq));
            }
            compute_bar();
            // the column sums by all compute threads: thread c < 128 sums (S^T k)_c and forms u_c,
            // thread 128 + c sums (S^T q)_c and forms the output once u is published
            float w;
            {
                const float *const src = s_red + (tid >> 7) * RPP * kHeadDim + (tid & (kHeadDim - 1));
                float x[RPP];
#pragma unroll
                for (int i = 0; i < RPP; ++i) x[i] = src[i * kHeadDim];
                w = x[0];
#pragma unroll
                for (int i = 1; i < RPP; ++i) w += x[i];
            }
            if (tid < kHeadDim) s_u[tid] = beta_of(s_beta[t], a) * (__bfloat162float(trow[3 * kHeadDim + tid]) - w);
            compute_bar();
            if (tid >= kHeadDim) {
                const int c = tid - kHeadDim;
                out_row[t * out_tok_stride + c] = __float2bfloat16_rn(a.scale * fmaf(ts.qk, s_u[c], w));
            }
            float2 uv[VEC / 2];
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e) uv[e] = *reinterpret_cast<const float2 *>(&s_u[cg * VEC + 2 * e]);
#pragma unroll
            for (int p = 0; p < NPASS; ++p) {
                const float kr = kv[p] * ts.rk;
#pragma unroll
                for (int e = 0; e < VEC / 2; ++e) {
                    const float2 x = __ffma2_rn(make_float2(kr, kr), uv[e], make_float2(stv[p][2 * e], stv[p][2 * e + 1]));
                    stv[p][2 * e] = x.x;
                    stv[p][2 * e + 1] = x.y;
                }
            }
            // the next token's partial sums overwrite s_red only after this token's column
            // sums were read (the barrier above), and s_u only after the next barrier
        }
#pragma unroll
        for (int p = 0; p < NPASS; ++p)
            *reinterpret_cast<typename V::Raw *>(S + (rg + p * RPP) * kHeadDim + cg * VEC) = V::pack(stv[p]);
        fence_async_smem();
        mbar_arrive(&done[st]);
    }
}

template <typename T, bool kRefillAtOnce, bool kGroupLayout>
cudaError_t launch_decode_stream_t(const DecodeArgs &a, cudaStream_t stream, int sms) {
    using SS = StreamShape<T, kGroupLayout>;
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kda_decode_stream_kernel<T, kRefillAtOnce, kGroupLayout>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SS::kStreamSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const int64_t items = (int64_t)a.rows * a.num_heads;
    const int grid = (int)std::min<int64_t>(items, sms);
    kda_decode_stream_kernel<T, kRefillAtOnce, kGroupLayout>
        <<<grid, kDecodeThreads + 32, SS::smem(a.tokens), stream>>>(a);
    return cudaGetLastError();
}

// Tokens per row from which BF16 states stay in registers for the whole row (measured on
// 4096 rows x H8: the register layout is 17% slower at 2 tokens and 5% at 3, 6% faster at 4,
// 18% at 6, 21% at 8, 24% at 16).
constexpr int kBf16RowRegisterTokens = 4;

template <typename T>
cudaError_t launch_decode_stream(const DecodeArgs &a, cudaStream_t stream, int sms) {
    if constexpr (sizeof(T) == 2) {
        // up to 3 tokens per row: two compute groups on alternate items, the state in its stage
        // (their rings keep an even stage count of at least four); from 4 on, where it is
        // faster, the state in FP32 registers for the whole row, rounded once
        if (a.tokens >= kBf16RowRegisterTokens) {
            if (StreamShape<T, false>::stages(a.tokens) <= 2) return launch_decode_stream_t<T, true, false>(a, stream, sms);
            return launch_decode_stream_t<T, false, false>(a, stream, sms);
        }
        return launch_decode_stream_t<T, false, true>(a, stream, sms);
    } else {
        if (StreamShape<T>::stages(a.tokens) <= 2) return launch_decode_stream_t<T, true, false>(a, stream, sms);
        return launch_decode_stream_t<T, false, false>(a, stream, sms);
    }
}

template <typename T, int JW>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t stream) {
    const int64_t ctas = (int64_t)a.rows * a.num_heads * (kHeadDim / JW);
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    kda_decode_kernel<T, JW><<<(unsigned)ctas, kDecodeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

// Column-block width of the register schedule: whole rows when there are enough items to
// fill the GPU several times over, narrower blocks (more CTAs per item) when there are not.
int pick_decode_width(int64_t items) {
    if (items >= 1024) return 128;
    if (items >= 256) return 64;
    if (items >= 64) return 32;
    return 16;
}

// Items per SM from which the streaming schedule takes over (several per SM, so that its
// ring fills): measured crossovers of the two schedules, BF16 states between 1.7 and 3.4
// items per SM, FP32 states near 3.4.
constexpr int kStreamItemsPerSmF32 = 4;
constexpr int kStreamItemsPerSmBF16 = 3;

}  // namespace

#ifdef KDA_DEBUG_CHECKS
// Debug builds only: a slot named by two rows is recorded as KDA_ERR_DEVICE_INPUT with the
// later row as its detail (the decode of such a batch races on that slot). Padding rows
// (negative slots) may repeat. Every row is compared with every earlier one: quadratic, for
// debugging only.
__global__ void kda_check_slots_kernel(const int32_t *slot_idx, int32_t rows, DeviceStatus *status) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const int32_t s = __ldg(slot_idx + r);
    if (s < 0) return;
    for (int q = 0; q < r; ++q)
        if (__ldg(slot_idx + q) == s) {
            report_error(status, KDA_ERR_DEVICE_INPUT, r);
            return;
        }
}
#endif

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    const int64_t items = (int64_t)a.rows * a.num_heads;
#ifdef KDA_DEBUG_CHECKS
    kda_check_slots_kernel<<<(a.rows + 255) / 256, 256, 0, stream>>>(a.slot_idx, a.rows, a.status);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
#endif
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int per_sm = a.state_dtype == KDA_STATE_F32 ? kStreamItemsPerSmF32 : kStreamItemsPerSmBF16;
    if (a.tokens > 1 || items >= (int64_t)per_sm * sms) {
        if (a.state_dtype == KDA_STATE_F32) return launch_decode_stream<float>(a, stream, sms);
        return launch_decode_stream<__nv_bfloat16>(a, stream, sms);
    }
    const int jw = pick_decode_width(items);
    if (a.state_dtype == KDA_STATE_F32) {
        if (jw == 128) return launch_decode_t<float, 128>(a, stream);
        if (jw == 64) return launch_decode_t<float, 64>(a, stream);
        if (jw == 32) return launch_decode_t<float, 32>(a, stream);
        return launch_decode_t<float, 16>(a, stream);
    }
    if (jw == 128) return launch_decode_t<__nv_bfloat16, 128>(a, stream);
    if (jw == 64) return launch_decode_t<__nv_bfloat16, 64>(a, stream);
    if (jw == 32) return launch_decode_t<__nv_bfloat16, 32>(a, stream);
    return launch_decode_t<__nv_bfloat16, 16>(a, stream);
}

}  // namespace kda
