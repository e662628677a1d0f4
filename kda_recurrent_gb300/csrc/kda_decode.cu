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
#include "kda_internal.cuh"

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

template <typename T, int JW>
__global__ void __launch_bounds__(kDecodeThreads) kda_decode_kernel(DecodeArgs a) {
    using V = StateVec<T>;
    constexpr int VEC = V::kElems;            // state elements per 16-byte vector
    constexpr int VPR = JW / VEC;             // vectors per row of the column block
    constexpr int RPP = kDecodeThreads / VPR; // rows covered by one pass of the CTA
    constexpr int NPASS = kHeadDim / RPP;     // passes (vectors held per thread)
    constexpr int NSPLIT = kHeadDim / JW;     // column blocks per item
    static_assert(kDecodeThreads % VPR == 0 && kHeadDim % RPP == 0, "tile shape");
    static_assert(2 * JW <= kDecodeThreads, "one reducer thread per column sum");

    __shared__ float s_k[kHeadDim], s_q[kHeadDim], s_decay[kHeadDim];
    __shared__ float s_red[2][RPP][JW];
    __shared__ float s_u[JW];
    __shared__ float s_qk;

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

    // 2. Token vectors and the per-channel decay while the state is in flight.
    const size_t tok = (size_t)item * kHeadDim;
    if (tid < kHeadDim) {
        const float av = __bfloat162float(a.g_raw[tok + tid]);
        s_decay[tid] = expf(gate_log_decay(av, a.gate_mode, a.lower_bound));
        s_k[tid] = __bfloat162float(a.k[tok + tid]);
        s_q[tid] = __bfloat162float(a.q[tok + tid]);
    }
    __syncthreads();
    if (tid < 32) {
        float acc = 0.0f;
#pragma unroll
        for (int i = tid; i < kHeadDim; i += 32) acc = fmaf(s_q[i], s_k[i], acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (tid == 0) s_qk = acc;
    }

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
        s_red[0][rg][cg * VEC + e] = wk[e];
        s_red[1][rg][cg * VEC + e] = wq[e];
    }
    __syncthreads();

    // 4. Column sums, the delta-rule residual u and the output, one thread per column.
    if (tid < JW) {
        float w_k = 0.0f, w_q = 0.0f;
#pragma unroll 8
        for (int i = 0; i < RPP; ++i) {
            w_k += s_red[0][i][tid];
            w_q += s_red[1][i][tid];
        }
        const float u = a.beta[item] * (__bfloat162float(a.v[tok + j0 + tid]) - w_k);
        s_u[tid] = u;
        out[tid] = __float2bfloat16_rn(a.scale * fmaf(s_qk, u, w_q));
    }
    __syncthreads();

    // 5. Rank-one update and streaming store of the slice.
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
        const int row = rg + p * RPP;
        const float kk = s_k[row];
#pragma unroll
        for (int e = 0; e < VEC; ++e) st[p][e] = fmaf(kk, s_u[cg * VEC + e], st[p][e]);
        const uint32_t off = (uint32_t)row * kHeadDim + (uint32_t)cg * VEC;
        __stcs(reinterpret_cast<typename V::Raw *>(S + off), V::pack(st[p]));
    }
}

template <typename T, int JW>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t stream) {
    const int64_t ctas = (int64_t)a.rows * a.num_heads * (kHeadDim / JW);
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    kda_decode_kernel<T, JW><<<(unsigned)ctas, kDecodeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

// Column-block width: whole rows when there are enough items to fill the GPU
// several times over, narrower blocks (more CTAs per item) when there are not.
int pick_decode_width(int64_t items) {
    if (items >= 1024) return 128;
    if (items >= 256) return 64;
    return 32;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    const int jw = pick_decode_width((int64_t)a.rows * a.num_heads);
    if (a.state_dtype == KDA_STATE_F32) {
        if (jw == 128) return launch_decode_t<float, 128>(a, stream);
        if (jw == 64) return launch_decode_t<float, 64>(a, stream);
        return launch_decode_t<float, 32>(a, stream);
    }
    if (jw == 128) return launch_decode_t<__nv_bfloat16, 128>(a, stream);
    if (jw == 64) return launch_decode_t<__nv_bfloat16, 64>(a, stream);
    return launch_decode_t<__nv_bfloat16, 32>(a, stream);
}

}  // namespace kda
