// Chunk-32 varlen KDA prefill (sm_103a).
//
// Chunked form ("FlashInfer PR #4262: CAKE KDA Prefill Highlights", section 2). With
// G_i the inclusive per-channel prefix of g (base 2) over a chunk of L <= 32 tokens:
//   Qbar = scale q (x) 2^G,   Kbar = k (x) 2^G,   Kr = k (x) 2^(G_last - G)
//   Mqk[i,j] = scale sum_c q_i k_j 2^(G_i - G_j) (j <= i),  A[i,j] = sum_c k_i k_j 2^(G_i - G_j) (j < i)
//   T' = (I + Diag(beta) A)^-1 Diag(beta)
//   U = T'(V - Kbar S),  O = Qbar S + Mqk U,  S_new = Diag(2^G_last) S + Kr^T U
// The state-independent part is folded into the chunk operands before the state is
// touched:  Wk = T' Kbar,  Wv = T' V,  Q' = Qbar - Mqk Wk,  Ov = Mqk Wv, so that
//   U = Wv - Wk S,   O = Ov + Q' S,   S_new = Diag(2^G_last) S + Kr^T U.
// The serial chain of a chunk is then two GEMMs: [Wk; Q'] S (64 x 128 x 128) and
// Kr^T U (128 x 32 x 128), with the residual in between.
//
// Exponent range. The page factors 2^(G_i - G_j) through a fixed anchor C = 16 lb log2(e)
// (section 1), which leaves the float range at lb = -8 and has no bound for the softplus
// gate. Here each 16-token half uses a per-channel anchor at its own midpoint for its
// diagonal block, and the off-diagonal block factors through the half boundary:
// 2^(G_i - G_15) 2^(G_15 - G_j), both <= 1. Operand exponents stay within half a
// half-chunk span (86.6 bits at lb = -8).
//
// Precision. BF16 operands with FP32 accumulation for the chunk products and the state
// projection; the state update Kr^T U runs in TF32, and Wv = T' V uses T' split into
// BF16 hi + lo (V is exact in BF16), because U's rounding dominates the final-state
// error otherwise. The state itself stays FP32.
//
// Work split. One CTA (8 warps) per (sequence, head) chain walks its chunks in order.
// The state S^T [dv x dk] lives in registers as mma accumulators: warp w owns dv rows
// 16w..16w+15, so the whole serial chain of a chunk (projection, residual, decay, update)
// is warp-local. Chunk operands are prepared by all 8 warps between barriers; raw q/k/v/g
// of the next chunk stream in by cp.async while the current one is processed.
#include "kda_internal.cuh"
#include "kda_mma.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kRowB = 136;  // bf16 row stride of 128-wide tiles: 272-byte rows keep ldmatrix conflict-free
constexpr int kRowF = 132;  // fp32 row stride of 128-wide tiles
constexpr int kSq = 36;     // fp32 row stride of 32 x 32 tiles
constexpr int kSmall = 20;  // fp32 row stride of 16 x 16 tiles
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory map (byte offsets).
constexpr int kTileB = 32 * kRowB * 2;            // one 32 x 128 bf16 tile
constexpr int kTileF = 32 * kRowF * 4;            // one 32 x 128 fp32 tile
constexpr int kSqBytes = 32 * kSq * 4;            // one 32 x 32 fp32 tile
constexpr int kStageBytes = 4 * kTileB + 128;     // raw q, k, v, a tiles + 32 beta
constexpr int kOffRaw0 = 0;
constexpr int kOffRaw1 = kOffRaw0 + kStageBytes;
constexpr int kOffPair = kOffRaw1 + kStageBytes;  // pair operands: 3 x 48 bf16 rows
constexpr int kPairRows = 48;
constexpr int kOffPairQ = kOffPair;
constexpr int kOffPairKL = kOffPairQ + kPairRows * kRowB * 2;
constexpr int kOffPairKR = kOffPairKL + kPairRows * kRowB * 2;
constexpr int kOffPairEnd = kOffPairKR + kPairRows * kRowB * 2;
constexpr int kOffWv = kOffPair;                  // aliases the pair operands (dead by then)
constexpr int kOffOv = kOffWv + kTileF;
static_assert(kOffOv + kTileF <= kOffPairEnd, "Wv/Ov alias fits in the pair region");
constexpr int kOffKbar = kOffPairEnd;             // bf16 [32][136]
constexpr int kOffQbar = kOffKbar + kTileB;       // fp32 [32][132]
constexpr int kOffKr = kOffQbar + kTileF;         // fp32 (tf32-rounded) [32][132]
constexpr int kOffW = kOffKr + kTileF;            // bf16 [64][136]: rows 0-31 Wk, 32-63 Q'
constexpr int kOffA = kOffW + 2 * kTileB;         // fp32 [32][36]: Diag(beta) A
constexpr int kOffM = kOffA + kSqBytes;           // fp32 [32][36]: Mqk
constexpr int kOffTp = kOffM + kSqBytes;          // fp32 [32][36]: T'
constexpr int kOffT22 = kOffTp + kSqBytes;        // fp32 [16][20]
constexpr int kOffX = kOffT22 + 16 * kSmall * 4;  // fp32 [16][20]
constexpr int kOffO = kOffX + 16 * kSmall * 4;    // bf16 [32][136] output staging
constexpr int kOffDec = kOffO + kTileB;           // fp32 [128]
constexpr int kOffHalf = kOffDec + 128 * 4;       // fp32 [2][128]
constexpr int kSmemBytes = kOffHalf + 2 * 128 * 4;
static_assert(kSmemBytes <= 227 * 1024, "fits one CTA per SM");

__device__ __forceinline__ float gate_log_decay(float av, int mode, float lower_bound) {
    if (mode == KDA_GATE_LOWER_BOUND) return lower_bound / (1.0f + expf(-av));
    if (mode == KDA_GATE_SOFTPLUS) return -(fmaxf(av, 0.0f) + log1pf(expf(-fabsf(av))));
    return av;
}

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ void st_bf16(uint8_t *base, int off_bytes, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(base + off_bytes) = __float2bfloat16_rn(x);
}

// Issue the cp.async copies of one chunk's raw q, k, v, a rows and beta into a stage.
__device__ __forceinline__ void load_chunk(const PrefillArgs &a, uint8_t *stage, int t0, int L, int h,
                                           int tid) {
    const __nv_bfloat16 *src[4] = {a.q, a.k, a.v, a.g_raw};
    const uint32_t dst0 = smem_addr(stage);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int idx = tid + kThreads * m;  // 0 .. 2047
        const int tensor = idx >> 9;
        const int row = (idx >> 4) & 31;
        const int vec = idx & 15;
        const bool valid = row < L;
        const size_t tok = (size_t)(t0 + (valid ? row : 0));
        const __nv_bfloat16 *s = src[tensor] + (tok * a.num_heads + h) * kHeadDim + vec * 8;
        cp_async_16(dst0 + tensor * kTileB + (row * kRowB + vec * 8) * 2, s, valid ? 16u : 0u);
    }
    if (tid < 32) {
        const bool valid = tid < L;
        const size_t tok = (size_t)(t0 + (valid ? tid : 0));
        cp_async_4(dst0 + 4 * kTileB + tid * 4, a.beta + tok * a.num_heads + h, valid ? 4u : 0u);
    }
}

__global__ void __launch_bounds__(kThreads, 1) kda_prefill_kernel(const PrefillArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int H = a.num_heads;
    const int chain = blockIdx.x;
    const int n = chain / H;
    const int h = chain - n * H;

    int bos = a.cu_seqlens[n], eos = a.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > a.total_tokens) {
        if (tid == 0 && h == 0) report_error(a.status, KDA_ERR_DEVICE_INPUT, n);
        bos = min(max(bos, 0), a.total_tokens);
        eos = min(max(eos, bos), a.total_tokens);
    }
    const int nchunks = (eos - bos + kChunk - 1) / kChunk;

    // ---- state S^T in registers: st[nt][e] = S[dk = 8nt + 2t4 + (e&1)][dv = 16 warp + g + 8(e>>1)]
    float st[16][4];
    const size_t sbase = (size_t)chain * kHeadDim * kHeadDim;
    const int dv0 = 16 * warp + g;
    if (a.init_state != nullptr) {
        const float *S0 = a.init_state + sbase;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int dk = 8 * nt + 2 * t4;
            st[nt][0] = S0[dk * kHeadDim + dv0];
            st[nt][1] = S0[(dk + 1) * kHeadDim + dv0];
            st[nt][2] = S0[dk * kHeadDim + dv0 + 8];
            st[nt][3] = S0[(dk + 1) * kHeadDim + dv0 + 8];
        }
    } else {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.0f;
    }

    if (nchunks > 0) load_chunk(a, smem + kOffRaw0, bos, min(kChunk, eos - bos), h, tid);
    cp_async_commit();

    uint8_t *const pairQ = smem + kOffPairQ;
    uint8_t *const pairKL = smem + kOffPairKL;
    uint8_t *const pairKR = smem + kOffPairKR;
    float *const wv_s = reinterpret_cast<float *>(smem + kOffWv);
    float *const ov_s = reinterpret_cast<float *>(smem + kOffOv);
    uint8_t *const kbar_s = smem + kOffKbar;
    float *const qbar_s = reinterpret_cast<float *>(smem + kOffQbar);
    float *const kr_s = reinterpret_cast<float *>(smem + kOffKr);
    uint8_t *const w_s = smem + kOffW;
    float *const am_s = reinterpret_cast<float *>(smem + kOffA);
    float *const mq_s = reinterpret_cast<float *>(smem + kOffM);
    float *const tp_s = reinterpret_cast<float *>(smem + kOffTp);
    float *const t22_s = reinterpret_cast<float *>(smem + kOffT22);
    float *const x_s = reinterpret_cast<float *>(smem + kOffX);
    uint8_t *const o_s = smem + kOffO;
    float *const dec_s = reinterpret_cast<float *>(smem + kOffDec);
    float *const half_s = reinterpret_cast<float *>(smem + kOffHalf);

    for (int c = 0; c < nchunks; ++c) {
        const int t0 = bos + kChunk * c;
        const int L = min(kChunk, eos - t0);
        uint8_t *const raw = smem + ((c & 1) ? kOffRaw1 : kOffRaw0);
        if (c + 1 < nchunks) {
            const int t1 = t0 + kChunk;
            load_chunk(a, smem + ((c & 1) ? kOffRaw0 : kOffRaw1), t1, min(kChunk, eos - t1), h, tid);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const __nv_bfloat16 *rq = reinterpret_cast<const __nv_bfloat16 *>(raw);
        const __nv_bfloat16 *rk = reinterpret_cast<const __nv_bfloat16 *>(raw + kTileB);
        const __nv_bfloat16 *ra = reinterpret_cast<const __nv_bfloat16 *>(raw + 3 * kTileB);
        const float *rb = reinterpret_cast<const float *>(raw + 4 * kTileB);

        // ---- 1. gate and inclusive prefix (base 2); thread = (channel, half)
        const int ch = tid & 127, hf = tid >> 7;
        float G[16];
        {
            float run = 0.0f;
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                const int i = 16 * hf + ii;
                float gv = 0.0f;
                if (i < L) gv = gate_log_decay(bf(ra + i * kRowB + ch), a.gate_mode, a.lower_bound);
                run = fmaf(gv, kLog2e, run);
                G[ii] = run;
            }
            half_s[hf * 128 + ch] = run;
        }
        __syncthreads();
        {
            const float tot0 = half_s[ch], tot1 = half_s[128 + ch];
            if (hf) {
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) G[ii] += tot0;
            }
            const float G15 = tot0;
            const float GL = tot0 + tot1;  // gates past L are zero, so this is G_{L-1}
            const float anchor = 0.5f * (G[0] + G[15]);
            // per-channel constants of the factorisations (all <= 1 where used as products)
            const float c_bar = hf ? exp2f(G15) : 0.0f;            // 2^G15
            const float c_kr = hf ? 0.0f : exp2f(GL - G15);        // 2^(G_L - G15)
            bool range_ok = true;
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                const int i = 16 * hf + ii;
                const float x = G[ii];
                const float kk = bf(rk + i * kRowB + ch);
                const float qq = a.scale * bf(rq + i * kRowB + ch);
                const float fl = exp2f(x - anchor);
                const float fr = exp2f(anchor - x);
                range_ok &= (fl < 1e37f) && (fr < 1e37f);
                st_bf16(pairQ, (i * kRowB + ch) * 2, qq * fl);
                st_bf16(pairKL, (i * kRowB + ch) * 2, kk * fl);
                st_bf16(pairKR, (i * kRowB + ch) * 2, kk * fr);
                float fbar, fkr;
                if (hf) {
                    const float fo = exp2f(x - G15);  // <= 1
                    st_bf16(pairQ, ((32 + ii) * kRowB + ch) * 2, qq * fo);
                    st_bf16(pairKL, ((32 + ii) * kRowB + ch) * 2, kk * fo);
                    fbar = fo * c_bar;                // 2^G_i
                    fkr = exp2f(GL - x);              // 2^(G_L - G_i)
                } else {
                    const float fo = exp2f(G15 - x);  // <= 1
                    st_bf16(pairKR, ((32 + ii) * kRowB + ch) * 2, kk * fo);
                    fbar = exp2f(x);
                    fkr = fo * c_kr;
                }
                st_bf16(kbar_s, (i * kRowB + ch) * 2, kk * fbar);
                qbar_s[i * kRowF + ch] = qq * fbar;
                kr_s[i * kRowF + ch] = __uint_as_float(to_tf32(kk * fkr));
            }
            if (!range_ok) report_error(a.status, KDA_ERR_DEVICE_INPUT, n);
            if (hf == 0) dec_s[ch] = exp2f(GL);
        }
        __syncthreads();

        // ---- 2. causal Mqk and Diag(beta) A: three 16x16 blocks each (warps 0-5)
        if (warp < 6) {
            const int which = warp / 3;  // 0: Mqk (left = q operands), 1: A (left = k operands)
            const int blk = warp % 3;    // 0: tokens 0-15 diagonal, 1: 16-31 diagonal, 2: off-diagonal
            const uint8_t *Lb = which ? pairKL : pairQ;
            const int row0 = 16 * blk;   // 0, 16, 32 in both operand arrays
            float acc[2][4] = {};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t af[4], bfr[4];
                ldsm_x4(af, smem_addr(Lb + ((row0 + (lane & 15)) * kRowB + 16 * ks + (lane >> 4) * 8) * 2));
                ldsm_x4(bfr, smem_addr(pairKR + ((row0 + (lane & 7) + ((lane >> 4) << 3)) * kRowB + 16 * ks +
                                                  ((lane >> 3) & 1) * 8) * 2));
                mma_bf16_16816(acc[0], af, bfr[0], bfr[1]);
                mma_bf16_16816(acc[1], af, bfr[2], bfr[3]);
            }
            const int oi = (blk == 0) ? 0 : 16;
            const int oj = (blk == 1) ? 16 : 0;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = oi + g + 8 * (e >> 1);
                    const int j = oj + 8 * nt + 2 * t4 + (e & 1);
                    const float val = acc[nt][e];
                    if (which == 0) {
                        mq_s[i * kSq + j] = (j <= i) ? val : 0.0f;
                    } else {
                        am_s[i * kSq + j] = (j < i) ? val * rb[i] : 0.0f;
                    }
                }
            }
        } else {
            // upper-right blocks are zero
            for (int idx = tid - 192; idx < 256; idx += 64) {
                const int i = idx >> 4, j = 16 + (idx & 15);
                mq_s[i * kSq + j] = 0.0f;
                am_s[i * kSq + j] = 0.0f;
            }
        }
        __syncthreads();

        // ---- 3. T' = (I + Diag(beta) A)^-1 Diag(beta): 16x16 diagonal blocks by forward substitution
        if (warp < 2) {
            const int o = 16 * warp;
            const int j = lane & 15;
            float x[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) x[ii] = (ii == j) ? 1.0f : 0.0f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
#pragma unroll
                for (int ii = kk + 1; ii < 16; ++ii) x[ii] = fmaf(-am_s[(o + ii) * kSq + o + kk], x[kk], x[ii]);
            }
            if (lane < 16) {
                const float bj = rb[o + j];
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) {
                    tp_s[(o + ii) * kSq + o + j] = x[ii] * bj;
                    tp_s[(o + ii) * kSq + (16 - o) + j] = 0.0f;  // clears the block beside it
                }
                if (warp == 1) {
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii) t22_s[ii * kSmall + j] = x[ii];
                }
            }
        }
        __syncthreads();
        {   // X = N21 T'11
            const int i = tid >> 4, j = tid & 15;
            float s = 0.0f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) s = fmaf(am_s[(16 + i) * kSq + kk], tp_s[kk * kSq + j], s);
            x_s[i * kSmall + j] = s;
        }
        __syncthreads();
        {   // T'21 = -T22 X ; the upper-right block stays zero
            const int i = tid >> 4, j = tid & 15;
            float s = 0.0f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) s = fmaf(t22_s[i * kSmall + kk], x_s[kk * kSmall + j], s);
            tp_s[(16 + i) * kSq + j] = -s;
            tp_s[i * kSq + 16 + j] = 0.0f;
        }
        __syncthreads();

        // ---- 4. Wk = T' Kbar, Wv = T' V (T' as bf16 hi + lo); warp w owns columns 16w..16w+15
        {
            uint32_t ah[2][2][4], al[2][2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int row = 16 * mt + g + 8 * (r & 1);
                        const int col = 16 * ks + 2 * t4 + 8 * (r >> 1);
                        const float2 v2 = *reinterpret_cast<const float2 *>(tp_s + row * kSq + col);
                        ah[mt][ks][r] = pack_bf16(v2.x, v2.y);
                        al[mt][ks][r] = pack_bf16(v2.x - bf16_round(v2.x), v2.y - bf16_round(v2.y));
                    }
                }
            }
            float wk[2][2][4] = {}, wvv[2][2][4] = {};
            const uint8_t *rv = raw + 2 * kTileB;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t bk[4], bv[4];
                const int krow = 16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ncol = 16 * warp + (lane >> 4) * 8;
                ldsm_x4_trans(bk, smem_addr(kbar_s + (krow * kRowB + ncol) * 2));
                ldsm_x4_trans(bv, smem_addr(rv + (krow * kRowB + ncol) * 2));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                    for (int nl = 0; nl < 2; ++nl) {
                        mma_bf16_16816(wk[mt][nl], ah[mt][ks], bk[2 * nl], bk[2 * nl + 1]);
                        mma_bf16_16816(wvv[mt][nl], ah[mt][ks], bv[2 * nl], bv[2 * nl + 1]);
                        mma_bf16_16816(wvv[mt][nl], al[mt][ks], bv[2 * nl], bv[2 * nl + 1]);
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int nl = 0; nl < 2; ++nl) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int row = 16 * mt + g + 8 * hr;
                        const int col = 16 * warp + 8 * nl + 2 * t4;
                        *reinterpret_cast<uint32_t *>(w_s + (row * kRowB + col) * 2) =
                            pack_bf16(wk[mt][nl][2 * hr], wk[mt][nl][2 * hr + 1]);
                        *reinterpret_cast<float2 *>(wv_s + row * kRowF + col) =
                            make_float2(wvv[mt][nl][2 * hr], wvv[mt][nl][2 * hr + 1]);
                    }
                }
            }
        }
        __syncthreads();

        // ---- 5. Q' = Qbar - Mqk Wk (into W rows 32-63), Ov = Mqk Wv
        {
            uint32_t am[2][2][4], amn[2][2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int row = 16 * mt + g + 8 * (r & 1);
                        const int col = 16 * ks + 2 * t4 + 8 * (r >> 1);
                        const float2 v2 = *reinterpret_cast<const float2 *>(mq_s + row * kSq + col);
                        am[mt][ks][r] = pack_bf16(v2.x, v2.y);
                        amn[mt][ks][r] = pack_bf16(-v2.x, -v2.y);
                    }
                }
            }
            float qa[2][2][4], oa[2][2][4] = {};
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int nl = 0; nl < 2; ++nl) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int row = 16 * mt + g + 8 * hr;
                        const int col = 16 * warp + 8 * nl + 2 * t4;
                        const float2 q2 = *reinterpret_cast<const float2 *>(qbar_s + row * kRowF + col);
                        qa[mt][nl][2 * hr] = q2.x;
                        qa[mt][nl][2 * hr + 1] = q2.y;
                    }
                }
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t bw[4];
                const int krow = 16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8;
                ldsm_x4_trans(bw, smem_addr(w_s + (krow * kRowB + 16 * warp + (lane >> 4) * 8) * 2));
                uint32_t bv[2][2];
#pragma unroll
                for (int nl = 0; nl < 2; ++nl) {
                    const int col = 16 * warp + 8 * nl + g;
                    const int k0 = 16 * ks + 2 * t4;
                    bv[nl][0] = pack_bf16(wv_s[k0 * kRowF + col], wv_s[(k0 + 1) * kRowF + col]);
                    bv[nl][1] = pack_bf16(wv_s[(k0 + 8) * kRowF + col], wv_s[(k0 + 9) * kRowF + col]);
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                    for (int nl = 0; nl < 2; ++nl) {
                        mma_bf16_16816(qa[mt][nl], amn[mt][ks], bw[2 * nl], bw[2 * nl + 1]);
                        mma_bf16_16816(oa[mt][nl], am[mt][ks], bv[nl][0], bv[nl][1]);
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int nl = 0; nl < 2; ++nl) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int row = 16 * mt + g + 8 * hr;
                        const int col = 16 * warp + 8 * nl + 2 * t4;
                        *reinterpret_cast<uint32_t *>(w_s + ((32 + row) * kRowB + col) * 2) =
                            pack_bf16(qa[mt][nl][2 * hr], qa[mt][nl][2 * hr + 1]);
                        *reinterpret_cast<float2 *>(ov_s + row * kRowF + col) =
                            make_float2(oa[mt][nl][2 * hr], oa[mt][nl][2 * hr + 1]);
                    }
                }
            }
        }
        __syncthreads();

        // ---- 6. serial chain (warp-local): P^T = S^T [Wk; Q']^T, residual, decay, update
        {
            float p[8][4];
#pragma unroll
            for (int pn = 0; pn < 8; ++pn) p[pn][0] = p[pn][1] = p[pn][2] = p[pn][3] = 0.0f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t as[4];
                as[0] = pack_bf16(st[2 * ks][0], st[2 * ks][1]);
                as[1] = pack_bf16(st[2 * ks][2], st[2 * ks][3]);
                as[2] = pack_bf16(st[2 * ks + 1][0], st[2 * ks + 1][1]);
                as[3] = pack_bf16(st[2 * ks + 1][2], st[2 * ks + 1][3]);
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    uint32_t bw[4];
                    ldsm_x4(bw, smem_addr(w_s + ((16 * pp + (lane & 7) + ((lane >> 4) << 3)) * kRowB + 16 * ks +
                                                 ((lane >> 3) & 1) * 8) * 2));
                    mma_bf16_16816(p[2 * pp], as, bw[0], bw[1]);
                    mma_bf16_16816(p[2 * pp + 1], as, bw[2], bw[3]);
                }
            }
            // residual U^T = Wv^T - (Wk S)^T as tf32 A fragments; token order inside an
            // 8-token block is permuted (k = t4 <-> token 2t4, k = t4+4 <-> token 2t4+1),
            // and Kr rows are read with the same permutation below.
            uint32_t ua[4][4];
            const int dv1 = dv0 + 8;
#pragma unroll
            for (int pn = 0; pn < 4; ++pn) {
                const int tk = 8 * pn + 2 * t4;
                const float u00 = wv_s[tk * kRowF + dv0] - p[pn][0];
                const float u01 = wv_s[(tk + 1) * kRowF + dv0] - p[pn][1];
                const float u10 = wv_s[tk * kRowF + dv1] - p[pn][2];
                const float u11 = wv_s[(tk + 1) * kRowF + dv1] - p[pn][3];
                ua[pn][0] = to_tf32(u00);
                ua[pn][1] = to_tf32(u10);
                ua[pn][2] = to_tf32(u01);
                ua[pn][3] = to_tf32(u11);
            }
#pragma unroll
            for (int pn = 4; pn < 8; ++pn) {
                const int tk = 8 * (pn - 4) + 2 * t4;
                st_bf16(o_s, (tk * kRowB + dv0) * 2, ov_s[tk * kRowF + dv0] + p[pn][0]);
                st_bf16(o_s, ((tk + 1) * kRowB + dv0) * 2, ov_s[(tk + 1) * kRowF + dv0] + p[pn][1]);
                st_bf16(o_s, (tk * kRowB + dv1) * 2, ov_s[tk * kRowF + dv1] + p[pn][2]);
                st_bf16(o_s, ((tk + 1) * kRowB + dv1) * 2, ov_s[(tk + 1) * kRowF + dv1] + p[pn][3]);
            }
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const float d0 = dec_s[8 * nt + 2 * t4], d1 = dec_s[8 * nt + 2 * t4 + 1];
                st[nt][0] *= d0;
                st[nt][1] *= d1;
                st[nt][2] *= d0;
                st[nt][3] *= d1;
            }
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                const int tk = 8 * kt + 2 * t4;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const uint32_t b0 = __float_as_uint(kr_s[tk * kRowF + 8 * nt + g]);
                    const uint32_t b1 = __float_as_uint(kr_s[(tk + 1) * kRowF + 8 * nt + g]);
                    mma_tf32_1688(st[nt], ua[kt], b0, b1);
                }
            }
        }
        __syncthreads();

        // ---- 7. output store (rows < L)
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int idx = tid + kThreads * m;
            const int row = idx >> 4, vec = idx & 15;
            if (row < L) {
                const uint4 v4 = *reinterpret_cast<const uint4 *>(o_s + (row * kRowB + vec * 8) * 2);
                *reinterpret_cast<uint4 *>(a.out + ((size_t)(t0 + row) * H + h) * kHeadDim + vec * 8) = v4;
            }
        }
    }
    cp_async_wait<0>();

    if (a.final_state != nullptr) {
        float *Sf = a.final_state + sbase;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int dk = 8 * nt + 2 * t4;
            Sf[dk * kHeadDim + dv0] = st[nt][0];
            Sf[(dk + 1) * kHeadDim + dv0] = st[nt][1];
            Sf[dk * kHeadDim + dv0 + 8] = st[nt][2];
            Sf[(dk + 1) * kHeadDim + dv0 + 8] = st[nt][3];
        }
    }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    // The shared-memory opt-in is set once per device; repeating it is harmless.
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kda_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const int64_t chains = (int64_t)a.num_seqs * a.num_heads;
    kda_prefill_kernel<<<(unsigned)chains, kThreads, kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
