// Chunk-32 varlen KDA prefill, tcgen05 / TMEM version (sm_103a).
//
// Chunk algebra of "FlashInfer PR #4262: CAKE KDA Prefill Highlights", section 2. With
// T' = (I + Diag(beta) A)^-1 Diag(beta) the chunk's WY factor and Kbar, Qbar, Kr the decayed
// keys and queries, the page's U = T'(V - Kbar S) and O = Mqk U + Qbar S are reassociated
// around the residual R = V - Kbar S:
//     S_new = Diag(2^G_last) S + Kt^T R,   Kt = T'^T Kr   (32 x 128)
//     O     = Qbar S + Bo R,               Bo = Mqk T'    (32 x 32)
// so U, Wk = T' Kbar and Wv = T' V are never formed. As on the page, the FP32 recurrent
// state stays in tensor memory for the whole sequence and the state-sized products run on
// tcgen05; the accumulator is preloaded so that the projection itself produces R:
//     D1^T[dv, 0:32]  = V^T,  D1^T[dv, 32:64] = 0                  (producer tcgen05.st)
//     D1^T += S^T [-Kbar; Qbar]^T   M128 N64 K128, kind::tf32, A = S^T read from TMEM
//                                   -> D1^T = [R^T | (Qbar S)^T]
//     D1^T[:, 32:64] += R^T Bo^T    M128 N32 K32,  A = R^T read from TMEM      -> O^T
//     S = S Diag(2^G_last)                       (state warps, in TMEM, after the projection)
//     S^T += R^T Kt                 M128 N128 K32, A = R^T read from TMEM
// Kt^T = Kr^T T' is one more small tcgen05 product (M128 N32 K32, both operands in shared
// memory, TF32), issued by the producers off the serial chain. The decay runs in place, each
// 32-column block of S^T once the projection's MMAs that read it are done: run beside the whole
// projection into a second buffer, the two shared the tensor memory's bandwidth and the
// projection took several times its tensor-core time.
//
// Warp roles (one CTA per (sequence, head) chain, 16 warps), a chunk per group in flight:
//   warps 0-7   group A: raw loads (cp.async), gate and decay products, the pair operands
//               (bf16) and the stage operands ([-Kbar; Qbar], Kr, 2^G_last), in packed FP32
//               arithmetic on the two channels a thread owns;
//   warps 8-11  group B: pair products Mqk and Diag(beta) A (mma.sync), V^T into TMEM,
//               (I + Diag(beta) A)^-1 in FP32 by 16 x 16 blocks, T', the Kt MMA (tcgen05),
//               Bo (mma.sync, TF32) and the hand-off of the stage;
//   warps 12-15 state warps (one per TMEM lane quadrant): initial/final state, the decay,
//               the output read-out and store; lane 0 of warp 12 issues the projection,
//               lane 0 of warp 13 the update and then the output (in the window pass each
//               issues one of the two chains).
// Two stages of operands are in flight; the pair operands, the raw v and beta buffers and
// TMEM's D1 buffers are each released as soon as their reader is done with them. Group B
// hands a chunk to the state warps in two steps: once V^T is in D1 and its Kt MMA is queued,
// the state warps start the projection and the decay; once Kt and Bo are in the stage, the
// output and update MMAs (queued behind the Kt MMA, the projection does not delay it).
// Exponent range: per 16-token half, factors are anchored at the half's 8th token, built
// as running products of the per-token decays and their inverses (no per-element exp of a
// prefix); the off-diagonal block factors through the half boundary (both factors <= 1).
// All mbarrier waits are bounded; on expiry the kernel records KDA_ERR_DEVICE_TIMEOUT,
// drains, frees its tensor memory and returns.
#include <algorithm>
#include <type_traits>

#include "kda_internal.cuh"
#include "kda_mma.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kProducerWarps = 8;  // group A: chunk operands and pair products
constexpr int kSolveWarps = 4;     // group B: the WY inverse, Kt, Bo and the hand-off
constexpr int kStateWarps = 4;
constexpr int kFirstSolveWarp = kProducerWarps;
constexpr int kFirstStateWarp = kProducerWarps + kSolveWarps;
constexpr int kThreadsTc = (kProducerWarps + kSolveWarps + kStateWarps) * 32;
constexpr int kProdThreads = kProducerWarps * 32;
constexpr int kSolveThreads = kSolveWarps * 32;
constexpr int kStateThreads = kStateWarps * 32;
constexpr int kBarProd = 1;   // named barrier of group A
constexpr int kBarState = 2;  // named barrier of the state warps
constexpr int kBarSolve = 3;  // named barrier of group B
constexpr int kKtThread = (kFirstSolveWarp + 1) * 32;  // group B thread that issues and observes the Kt MMA

constexpr int kRowB = 136;  // padded bf16 row stride (ldmatrix operands)
constexpr int kSq = 36;     // fp32 32 x 32 tiles
constexpr float kLog2e = 1.4426950408889634f;
// Operands the tcgen05 MMAs read from shared memory are stored as plain FP32: kind::tf32
// reads only the TF32 bits and drops the 13 low mantissa bits, i.e. truncates toward zero.
// For mantissas spread log-uniformly the mean relative loss of that truncation is
// 2^-11 / ln 2 ~ 0.72 * 2^-11, so values pre-scaled by this factor (folded into a factor
// that is multiplied in anyway) reach the tensor core without bias, and with the same error
// spread as rounding to nearest. It replaces an explicit rounding per element.
constexpr float kTruncBias = 1.0f + 0.75f / 2048.0f;

// ---- shared-memory map (bytes)
constexpr int kRawQ = 0;                          // bf16 [32][128]
constexpr int kRawK = kRawQ + 8192;
constexpr int kRawA = kRawK + 8192;               // bf16 [2][32][128]: the gate tile, two chunks ahead
constexpr int kRawV = kRawA + 2 * 8192;           // bf16 [2][32][136]: v, one buffer per chunk parity
constexpr int kRawVBytes = 32 * kRowB * 2;
constexpr int kRawBeta = kRawV + 2 * kRawVBytes;  // fp32 [2][32]: beta, one buffer per chunk parity
constexpr int kStage0 = (kRawBeta + 256 + 1023) / 1024 * 1024;  // 1024-aligned (swizzle atoms)
// One stage per chunk in flight: the operands the state MMAs read.
constexpr int kStW = 0;                           // tf32 [4 K-atoms][64 tok][32 dk], 128-byte swizzle
// Kr / Kt: 8-row groups 1040 bytes apart instead of 1024, so that rows r and r + 8 fall in
// different 16-byte bank groups: the operand warps store rows 2p and 2p + 1 for channel pairs p,
// and a quarter warp's 8 float4 stores (rows 0, 2, ..., 14) then hit all 8 bank groups
constexpr int kKtSbo = 1040;
constexpr int kStKt = kStW + 4 * 8192;            // tf32 [128 dk][32 tok]: Kr, then Kt in place
constexpr int kStBo = kStKt + 16 * kKtSbo;        // tf32 [32 tok][32 tok]: Bo = Mqk T'
constexpr int kStDec = kStBo + 4096;              // fp32 [128]: 2^G_last
constexpr int kStageBytes = (kStDec + 512 + 1023) / 1024 * 1024;
constexpr int kOst = kStage0 + 2 * kStageBytes;   // bf16x2 [16][128]: output staging (tokens t, 16 + t)
constexpr int kPair = kOst + 16 * 128 * 4;        // 3 x [48][136] bf16
constexpr int kPairQ = kPair;
constexpr int kPairKL = kPairQ + 48 * kRowB * 2;
constexpr int kPairKR = kPairKL + 48 * kRowB * 2;
constexpr int kPairEnd = kPairKR + 48 * kRowB * 2;
// Group B's work space.
constexpr int kAtHi = kPairEnd;                   // tf32 [32][32] core matrices: T'^T
constexpr int kTinv = kAtHi + 4096;               // fp32 [32][36]: (I + Diag(beta) A)^-1
constexpr int kPscr = kTinv + 32 * kSq * 4;       // fp32 [16][16]: N21 T11 (and 2 x [8][8] before)
constexpr int kNt = kPscr + 1024;                 // fp32 [32][36]: (Diag(beta) A)^T
constexpr int kMq = kNt + 32 * kSq * 4;           // fp32 [32][36]: Mqk
constexpr int kBetaS = kMq + 32 * kSq * 4;        // fp32 [32]: beta of the chunk
constexpr int kQuart = kBetaS + 128;              // fp32 [4][128]: per-quarter decay products
constexpr int kBars = kQuart + 4 * 128 * 4;
constexpr int kSmemTc = kBars + 256;
static_assert(kStage0 % 128 == 0 && kStageBytes % 128 == 0 && kAtHi % 128 == 0, "operand alignment");
constexpr int kSmemLaunch = kSmemTc + 1024;  // plus the alignment slack
static_assert(kSmemLaunch <= 227 * 1024, "one CTA per SM");

// ---- tensor-memory map (columns; 512 allocated)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T [0,128) (the window pass keeps M^T at [128,256))
constexpr uint32_t kColD1 = 256;  // D1 double buffer: [256,320) and [320,384)
constexpr uint32_t kColKt = 384;  // Kt^T (lane = dk, column = token), producer-owned

constexpr uint32_t kIdescG1 = instr_desc(2, 128, 64);   // tf32, M128 N64
constexpr uint32_t kIdescG2 = instr_desc(2, 128, 128);  // tf32, M128 N128
constexpr uint32_t kIdescN32 = instr_desc(2, 128, 32);  // tf32, M128 N32

struct Bars {
    uint64_t prep[2];    // group B -> state warps: stage s filled (count kSolveThreads)
    uint64_t vready[2];  // group B -> state warps: V^T of the chunk of parity s in D1 (count
                         //   kSolveThreads); the projection needs only that
    uint64_t g1q[4];     // the projection's MMAs that read S^T columns [32 q, 32 q + 32) complete
    uint64_t go;         // output MMA complete (tcgen05.commit)
    uint64_t g2;         // state update MMA complete (tcgen05.commit)
    uint64_t g2s[2];     // state update of a chunk on stage s complete (tcgen05.commit)
    uint64_t oread[2];   // D1 buffer b read out by the state warps (count kStateThreads); in the
                         //   window pass also the stage of that parity consumed
    uint64_t kt;         // group B's Kt MMA complete (tcgen05.commit)
    uint64_t ab_full[2]; // group A -> B: chunk operands of parity p ready (count kProdThreads)
    uint64_t ab_empty;   // group B -> A: the pair operands of a chunk consumed
                         //   (count kSolveThreads, one phase per chunk)
    uint64_t vfree;      // group B -> A: the raw v, beta of a chunk consumed (same counting)
    uint64_t drain;      // after an abort: the three MMA-issuing threads' work complete (count 3)
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Programmatic dependent launch: let the next kernel of the stream start its launch now, and
// wait until the previous kernel of the stream has completed and its writes are visible
// (a no-op when the kernel was launched without the programmatic attribute).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void bar_named(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Bounded wait; on expiry records a timeout and raises the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, Bars *B, DeviceStatus *st) {
    if (mbar_wait(bar, parity)) return true;
    B->abort = 1;
    report_error(st, KDA_ERR_DEVICE_TIMEOUT, (int)blockIdx.x);
    return false;
}

__device__ __forceinline__ float bfv(const uint8_t *base, int elem) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[elem]);
}

// Byte offset of element (row, col) of a K-major tf32 operand tile made of 8-row x
// 16-byte core matrices; `sbo` = bytes per 8-row group (rows are N, cols are K).
__device__ __forceinline__ int core_off_tf32(int row, int col, int sbo) {
    return (row >> 3) * sbo + (col >> 2) * 128 + (row & 7) * 16 + (col & 3) * 4;
}

// Byte offset of element (token, dk) of the [-Kbar; Qbar] operand: K-major with the 128-byte
// swizzle, one 8 KiB atom per 32 dk (64 rows of 128 bytes); the 16-byte chunk of a row is
// XORed with the row's index within its 8-row group, so a warp's row stores hit all banks.
__device__ __forceinline__ int w_off(int row, int col) {
    return (col >> 5) * 8192 + (row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 2) & 7) ^ (row & 7)) << 4) +
           (col & 3) * 4;
}


__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Per-token decay d = exp(g) of one channel from the raw gate a, for a gate mode fixed at
// compile time (lb2 = lower_bound * log2 e).
template <int kMode>
__device__ __forceinline__ float gate_decay_m(float av, float lb2) {
    if (kMode == KDA_GATE_LOWER_BOUND) return ex2(lb2 * rcp(1.0f + ex2(-av * kLog2e)));  // exp(lb sigmoid(a))
    if (kMode == KDA_GATE_SOFTPLUS) return rcp(1.0f + ex2(av * kLog2e));               // exp(-softplus(a))
    return ex2(av * kLog2e);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Packed FP32 arithmetic on the two channels a producer thread owns (one instruction for both
// lanes of the pair, each rounded to nearest as the scalar operation is).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }

// gate_decay_m for both channels of a pair
template <int kMode>
__device__ __forceinline__ float2 gate_decay2(float2 av, float lb2) {
    if (kMode == KDA_GATE_LOWER_BOUND) {
        const float2 e = mul2(av, splat2(-kLog2e));
        const float2 den = add2(make_float2(ex2(e.x), ex2(e.y)), splat2(1.0f));
        const float2 x = mul2(make_float2(rcp(den.x), rcp(den.y)), splat2(lb2));
        return make_float2(ex2(x.x), ex2(x.y));
    }
    const float2 e = mul2(av, splat2(kLog2e));
    if (kMode == KDA_GATE_SOFTPLUS) {
        const float2 den = add2(make_float2(ex2(e.x), ex2(e.y)), splat2(1.0f));
        return make_float2(rcp(den.x), rcp(den.y));
    }
    return make_float2(ex2(e.x), ex2(e.y));
}

__device__ __forceinline__ void st_pair(uint8_t *base, int elem, float2 v) {
    *reinterpret_cast<uint32_t *>(base + 2 * elem) = pack_bf16(v.x, v.y);
}

// Raw loads of one chunk (cp.async, zero-filled past the sequence end): the gate tile into
// buffer `buf`, the q and k tiles, and the (padded) v tile with beta into buffer `buf`.
__device__ __forceinline__ void load_a(const PrefillArgs &a, uint8_t *smem, int t0, int L, int h, int ptid, int buf) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int idx = ptid + kProdThreads * m;  // 0 .. 511
        const int row = idx >> 4, vec = idx & 15;
        const bool valid = row < L;
        const size_t tok = (size_t)(t0 + (valid ? row : 0));
        cp_async_16(smem_addr(smem + kRawA + buf * 8192 + row * 256 + vec * 16),
                    a.g_raw + (tok * a.num_heads + h) * kHeadDim + vec * 8, valid ? 16u : 0u);
    }
}

__device__ __forceinline__ void load_qk(const PrefillArgs &a, uint8_t *smem, int t0, int L, int h, int ptid) {
    const __nv_bfloat16 *src[2] = {a.q, a.k};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int idx = ptid + kProdThreads * m;  // 0 .. 1023
        const int tensor = idx >> 9;
        const int row = (idx >> 4) & 31;
        const int vec = idx & 15;
        const bool valid = row < L;
        const size_t tok = (size_t)(t0 + (valid ? row : 0));
        cp_async_16(smem_addr(smem + kRawQ + tensor * 8192 + row * 256 + vec * 16),
                    src[tensor] + (tok * a.num_heads + h) * kHeadDim + vec * 8, valid ? 16u : 0u);
    }
}

__device__ __forceinline__ void load_vb(const PrefillArgs &a, uint8_t *smem, int t0, int L, int h, int ptid, int buf) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int idx = ptid + kProdThreads * m;  // 0 .. 511
        const int row = idx >> 4, vec = idx & 15;
        const bool valid = row < L;
        const size_t tok = (size_t)(t0 + (valid ? row : 0));
        cp_async_16(smem_addr(smem + kRawV + buf * kRawVBytes + (row * kRowB + vec * 8) * 2),
                    a.v + (tok * a.num_heads + h) * kHeadDim + vec * 8, valid ? 16u : 0u);
    }
    if (ptid < 32) {
        const bool valid = ptid < L;
        const size_t tok = (size_t)(t0 + (valid ? ptid : 0));
        cp_async_4(smem_addr(smem + kRawBeta + buf * 128 + ptid * 4), a.beta + tok * a.num_heads + h, valid ? 4u : 0u);
    }
}

// ------------------------------------------------------------------ producers

// Kt^T (TMEM lane = dk, column = token) -> the stage's Kt operand ([dk][token], read as TF32
// by the state update, which truncates it; T' carries the factor that offsets that), by
// group B: its warp b owns lane quadrant b.
__device__ __forceinline__ void kt_to_stage(uint32_t tmem, uint8_t *stage, int bwarp, int lane) {
    const int dk = 32 * bwarp + lane;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * bwarp) << 16) + kColKt + 16 * half, v);
        tmem_wait_ld();
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4)
            *reinterpret_cast<float4 *>(stage + kStKt + core_off_tf32(dk, 16 * half + 4 * e4, kKtSbo)) =
                make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
    }
}

// V^T of the chunk into its D1 buffer (lane = dv, column = token), by group B: its warp b
// owns lane quadrant b. The output pass also zeroes the 32 columns the projection
// accumulates Qbar S into.
template <bool kPass1>
__device__ __forceinline__ void v_to_tmem(uint32_t tmem, const uint8_t *rv, int db, int bwarp, int lane) {
    const int dv = 32 * bwarp + lane;
    float v0[16], v1[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        v0[t] = bfv(rv, t * kRowB + dv);
        v1[t] = bfv(rv, (16 + t) * kRowB + dv);
    }
    // output pass: D1 = [V | 0] (64 columns per buffer); window pass: D1 = V (32)
    const uint32_t taddr = tmem + ((uint32_t)(32 * bwarp) << 16) + (kPass1 ? kColD1 + 32 * db : kColD1 + 64 * db);
    tmem_st16(taddr, v0);
    tmem_st16(taddr + 16, v1);
    if (!kPass1) {
#pragma unroll
        for (int t = 0; t < 16; ++t) v0[t] = 0.0f;
        tmem_st16(taddr + 32, v0);
        tmem_st16(taddr + 48, v0);
    }
    tmem_wait_st();
}

// One 16 x 16 block of both pair products by one warp (mma.sync m16n8k16, BF16, FP32
// accumulate), in a single pass over k: N = Diag(beta) A (key rows) and, unless kKeysOnly, Mqk
// (query rows). Block 0 and 1 are the diagonal blocks of the two halves, 2 the off-diagonal
// one. The two products share their right operand (the key columns), so each k step loads it
// once, and the four accumulators give the warp four independent mma.sync chains. Mqk is
// stored row-major with the causal mask, N transposed and strictly lower.
template <bool kKeysOnly>
__device__ __forceinline__ void pair_blocks_nq(const uint8_t *smem, int blk, int lane, const float *rb, float *mq_s,
                                               float *nt_s) {
    const int g = lane >> 2, t4 = lane & 3;
    const uint8_t *const Kl = smem + kPairKL;
    const uint8_t *const Ql = smem + kPairQ;
    const uint8_t *const Rb = smem + kPairKR;
    const int row0 = 16 * blk;
    float an[2][4] = {}, aq[2][4] = {};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t fk[4], fq[4], bfr[4];
        const int aoff = ((row0 + (lane & 15)) * kRowB + 16 * ks + (lane >> 4) * 8) * 2;
        ldsm_x4(fk, smem_addr(Kl + aoff));
        if (!kKeysOnly) ldsm_x4(fq, smem_addr(Ql + aoff));
        ldsm_x4(bfr, smem_addr(Rb + ((row0 + (lane & 7) + ((lane >> 4) << 3)) * kRowB + 16 * ks +
                                     ((lane >> 3) & 1) * 8) * 2));
        mma_bf16_16816(an[0], fk, bfr[0], bfr[1]);
        mma_bf16_16816(an[1], fk, bfr[2], bfr[3]);
        if (!kKeysOnly) {
            mma_bf16_16816(aq[0], fq, bfr[0], bfr[1]);
            mma_bf16_16816(aq[1], fq, bfr[2], bfr[3]);
        }
    }
    const int oi = (blk == 0) ? 0 : 16;
    const int oj = (blk == 1) ? 16 : 0;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = oi + g + 8 * (e >> 1);
            const int j = oj + 8 * nt + 2 * t4 + (e & 1);
            nt_s[j * kSq + i] = (j < i) ? an[nt][e] * rb[i] : 0.0f;
            if (!kKeysOnly) mq_s[i * kSq + j] = (j <= i) ? aq[nt][e] : 0.0f;
        }
    }
}

// (I + N_d)^-1 of the 16 x 16 diagonal block at (o, o) of a strictly lower triangular N
// (given transposed: nt[j * kSq + i] = N[i][j]) into inv[(o + i) * kSq + o + j], by one warp:
// the two 8 x 8 diagonal blocks by forward substitution (lanes 0-15, one column each; lanes
// 16-31 zero the upper 8 x 8 block), then the lower block -T22 N21 T11. `scr`: 64 floats.
__device__ __forceinline__ void invert_diag16(const float *nt, float *inv, float *scr, int o, int lane) {
    if (lane < 16) {
        const int b = o + 8 * (lane >> 3), cc = lane & 7;
        float nv[7][8];  // nv[j][m] = N[b + m][b + j]
#pragma unroll
        for (int j = 0; j < 7; ++j) {
            const float4 n0 = *reinterpret_cast<const float4 *>(nt + (b + j) * kSq + b);
            const float4 n1 = *reinterpret_cast<const float4 *>(nt + (b + j) * kSq + b + 4);
            nv[j][0] = n0.x, nv[j][1] = n0.y, nv[j][2] = n0.z, nv[j][3] = n0.w;
            nv[j][4] = n1.x, nv[j][5] = n1.y, nv[j][6] = n1.z, nv[j][7] = n1.w;
        }
        float t[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) t[m] = (m == cc) ? 1.0f : 0.0f;
#pragma unroll
        for (int j = 0; j < 7; ++j) {
            const float tj = t[j];
#pragma unroll
            for (int m = j + 1; m < 8; ++m) t[m] = fmaf(-nv[j][m], tj, t[m]);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) inv[(b + m) * kSq + b + cc] = t[m];
    } else {
        const int r = (lane - 16) >> 1, c4 = 4 * (lane & 1);
        *reinterpret_cast<float4 *>(inv + (o + r) * kSq + o + 8 + c4) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    __syncwarp();
    const int i = lane >> 2, j2 = 2 * (lane & 3);
    const int r0 = o + 8;
    float nl[8];
    float2 tl[8];
#pragma unroll
    for (int l = 0; l < 8; ++l) {
        nl[l] = nt[(o + l) * kSq + r0 + i];
        tl[l] = *reinterpret_cast<const float2 *>(inv + (o + l) * kSq + o + j2);
    }
    float2 p = splat2(0.0f);
#pragma unroll
    for (int l = 0; l < 8; ++l) p = fma2(splat2(nl[l]), tl[l], p);
    *reinterpret_cast<float2 *>(scr + i * 8 + j2) = p;
    __syncwarp();
    float tr[8];
    float2 pl[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        tr[k] = inv[(r0 + i) * kSq + r0 + k];
        pl[k] = *reinterpret_cast<const float2 *>(scr + k * 8 + j2);
    }
    float2 q = splat2(0.0f);
#pragma unroll
    for (int k = 0; k < 8; ++k) q = fma2(splat2(-tr[k]), pl[k], q);
    *reinterpret_cast<float2 *>(inv + (r0 + i) * kSq + o + j2) = q;
}

// Group A, per chunk: the gate and decay factors, the chunk operands of the state MMAs
// (stage) and of the pair products, and the raw loads of the next chunk.
template <bool kPass1>
__device__ void producer_loop(const PrefillArgs &a, uint8_t *smem, Bars *B, uint32_t tmem, int n, int h, int bos,
                              int eos, int nchunks) {
    (void)tmem;
    const int ptid = threadIdx.x;  // 0 .. 255
    uint8_t *const pairQ = smem + kPairQ;
    uint8_t *const pairKL = smem + kPairKL;
    uint8_t *const pairKR = smem + kPairKR;
    float *const quart_s = reinterpret_cast<float *>(smem + kQuart);
    const uint8_t *const rq = smem + kRawQ;
    const uint8_t *const rk = smem + kRawK;
    // cp.async groups, in commit order: a(0), a(1), [q, k, v, beta](0); then per chunk c: a(c + 2)
    // once the gate of c has read its buffer, [q, k, v, beta](c + 1) once the operands of c are
    // written (groups past the end are empty)
    auto rows_of = [&](int cc) { return min(kChunk, eos - (bos + kChunk * cc)); };
    if (nchunks > 0) load_a(a, smem, bos, rows_of(0), h, ptid, 0);
    cp_async_commit();
    if (nchunks > 1) load_a(a, smem, bos + kChunk, rows_of(1), h, ptid, 1);
    cp_async_commit();
    if (nchunks > 0) {
        load_qk(a, smem, bos, rows_of(0), h, ptid);
        load_vb(a, smem, bos, rows_of(0), h, ptid, 0);
    }
    cp_async_commit();

    bool vlost = false;
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = bos + kChunk * c;
        const int L = min(kChunk, eos - t0);
        const int ps = c & 1;
        uint8_t *const stage = smem + kStage0 + ps * kStageBytes;
        const uint8_t *const ra = smem + kRawA + ps * 8192;
        if (c == 0) {  // later gate tiles were waited for a chunk earlier
            cp_async_wait<2>();
            bar_named(kBarProd, kProdThreads);
        }

        // ---- 1. decays, anchored factors, chunk operands. Thread = (channel pair, 8-token
        //      quarter). With d the per-token decay, every factor is a running product of d or
        //      1/d inside a quarter times whole-quarter products: 2^G_i (prefix), 2^(G_L - G_i)
        //      (suffix), the half-chunk anchors at tokens 7 and 23 and the half boundary 15.
        {
            const int cp = ptid & 63, qt = ptid >> 6;
            const int ch = 2 * cp;
            float2 d[8];  // per-token decays of channels ch, ch + 1
            // the gate mode is uniform, so each mode gets its own loop
            auto decays = [&](auto mode) {
                constexpr int kMode = decltype(mode)::value;
                const float lb2 = a.lower_bound * kLog2e;
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) {
                    const int i = 8 * qt + ii;
                    d[ii] = splat2(1.0f);
                    if (i < L)
                        d[ii] = gate_decay2<kMode>(
                            unpack_bf16x2(*reinterpret_cast<const uint32_t *>(ra + 2 * (i * 128 + ch))), lb2);
                }
            };
            if (a.gate_mode == KDA_GATE_LOWER_BOUND)
                decays(std::integral_constant<int, KDA_GATE_LOWER_BOUND>{});
            else if (a.gate_mode == KDA_GATE_SOFTPLUS)
                decays(std::integral_constant<int, KDA_GATE_SOFTPLUS>{});
            else
                decays(std::integral_constant<int, KDA_GATE_LOG_DECAY>{});
            // P: inclusive prefix of d; S: exclusive suffix of d. The anchored factor F is made
            // of 1/d: the exclusive suffix of 1/d before the anchor (quarters 0 and 2), which
            // is P / P_7, and the inclusive prefix of 1/d from the anchor on (quarters 1 and
            // 3), which is S / P_7, so one reciprocal per channel serves the quarter.
            const bool before_anchor = (qt & 1) == 0;
            float2 P[8], S[8];
            {
                float2 r = splat2(1.0f);
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) {
                    r = mul2(r, d[ii]);
                    P[ii] = r;
                }
                r = splat2(1.0f);
#pragma unroll
                for (int ii = 7; ii >= 0; --ii) {
                    S[ii] = r;
                    r = mul2(r, d[ii]);
                }
            }
            const float2 R = make_float2(rcp(P[7].x), rcp(P[7].y));
            *reinterpret_cast<float2 *>(quart_s + qt * 128 + ch) = P[7];
            {  // the gate needs no shared state; before the stores: stage ps is free once the
               // state update of chunk c - 2 is done with it, the pair operands once group B has
               // read those of chunk c - 1
                bool lost = vlost || (c >= 2 && !wait_or_abort(&B->g2s[ps], ((c >> 1) + 1) & 1, B, a.status));
                lost = lost || (c >= 1 && !wait_or_abort(&B->ab_empty, (c - 1) & 1, B, a.status));
                cp_async_wait<0>();  // q, k, v, beta of chunk c and the gate tile of chunk c + 1
                if (bar_any(kBarProd, kProdThreads, lost)) break;
            }
            // this chunk's gate tile is consumed: its buffer takes chunk c + 2
            if (c + 2 < nchunks) load_a(a, smem, t0 + 2 * kChunk, rows_of(c + 2), h, ptid, ps);
            cp_async_commit();
            float2 T[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) T[q4] = *reinterpret_cast<const float2 *>(quart_s + q4 * 128 + ch);
            const float2 one = splat2(1.0f);
            // whole-quarter products before (pre) and after (post) this quarter
            const float2 pre = mul2(mul2(qt > 0 ? T[0] : one, qt > 1 ? T[1] : one), qt > 2 ? T[2] : one);
            const float2 post = mul2(mul2(qt < 1 ? T[1] : one, qt < 2 ? T[2] : one), qt < 3 ? T[3] : one);
            // the stage operands are truncated to TF32 by the MMAs that read them
            const float2 preT = mul2(pre, splat2(kTruncBias)), npreT = mul2(pre, splat2(-kTruncBias));
            const float2 postT = mul2(post, splat2(kTruncBias));
            // off-diagonal factors 2^(G_i - G_15) (i >= 16) and 2^(G_15 - G_j) (j < 16)
            const float2 od = (qt == 0) ? T[1] : ((qt == 3) ? T[2] : one);
            // the largest factors of the quarter: P_7 and 1/P_7 bound P, S and F when d <= 1,
            // and F at its far end is checked directly for other gates
            const float fmax0 = before_anchor ? P[0].x * R.x : R.x, fmax1 = before_anchor ? P[0].y * R.y : R.y;
            if (!(fmax0 < 3.0e38f && fmax1 < 3.0e38f && R.x < 3.0e38f && R.y < 3.0e38f && P[7].x < 3.0e38f &&
                  P[7].y < 3.0e38f))
                report_error(a.status, KDA_ERR_DEVICE_INPUT, n);
            // left factor fl = P Rl (query / key rows of the diagonal blocks) and right factor
            // fr = S Rr (key columns): F and S before the anchor, P and F from it on
            const float2 Rl = before_anchor ? R : one, Rr = before_anchor ? one : R;
            const float2 sc = splat2(a.scale);
            float2 kr[8];
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const int i = 8 * qt + ii;
                const float2 k2 = unpack_bf16x2(*reinterpret_cast<const uint32_t *>(rk + 2 * (i * 128 + ch)));
                const float2 q2 = mul2(unpack_bf16x2(*reinterpret_cast<const uint32_t *>(rq + 2 * (i * 128 + ch))), sc);
                const float2 fl = mul2(P[ii], Rl), fr = mul2(S[ii], Rr);
                if (!kPass1) st_pair(pairQ, i * kRowB + ch, mul2(q2, fl));
                st_pair(pairKL, i * kRowB + ch, mul2(k2, fl));
                st_pair(pairKR, i * kRowB + ch, mul2(k2, fr));
                if (qt >= 2) {
                    const float2 fo = mul2(od, P[ii]);
                    if (!kPass1) st_pair(pairQ, (16 + i) * kRowB + ch, mul2(q2, fo));
                    st_pair(pairKL, (16 + i) * kRowB + ch, mul2(k2, fo));
                } else {
                    st_pair(pairKR, (32 + i) * kRowB + ch, mul2(k2, mul2(S[ii], od)));
                }
                // 2^G_i and 2^(G_L - G_i); row 32 + i lies 4096 bytes after row i (the same
                // swizzle phase), so both stores share one offset
                uint8_t *const wrow = stage + kStW + w_off(i, ch);
                *reinterpret_cast<float2 *>(wrow) = mul2(k2, mul2(npreT, P[ii]));
                if (!kPass1) *reinterpret_cast<float2 *>(wrow + 4096) = mul2(q2, mul2(preT, P[ii]));
                kr[ii] = mul2(k2, mul2(S[ii], postT));
            }
#pragma unroll
            for (int h4 = 0; h4 < 2; ++h4) {
                const int i0 = 8 * qt + 4 * h4;
                *reinterpret_cast<float4 *>(stage + kStKt + core_off_tf32(ch, i0, kKtSbo)) =
                    make_float4(kr[4 * h4].x, kr[4 * h4 + 1].x, kr[4 * h4 + 2].x, kr[4 * h4 + 3].x);
                *reinterpret_cast<float4 *>(stage + kStKt + core_off_tf32(ch + 1, i0, kKtSbo)) =
                    make_float4(kr[4 * h4].y, kr[4 * h4 + 1].y, kr[4 * h4 + 2].y, kr[4 * h4 + 3].y);
            }
            if (qt == 0)
                *reinterpret_cast<float2 *>(stage + kStDec + 4 * ch) = mul2(mul2(T[0], T[1]), mul2(T[2], T[3]));
        }
        // the operands of chunk c go to group B; the raw q, k tiles refill with chunk c + 1, and
        // v, beta with chunk c + 1 in the other buffer
        // the raw v, beta buffer of chunk c - 1 is free once group B has moved them out; the
        // wait comes before this chunk's hand-off so that group B cannot complete the phase of
        // chunk c before it is observed
        vlost = c >= 1 && !wait_or_abort(&B->vfree, (c - 1) & 1, B, a.status);
        fence_async_smem();
        mbar_arrive(&B->ab_full[ps]);
        bar_named(kBarProd, kProdThreads);
        if (c + 1 < nchunks && !vlost) {
            load_qk(a, smem, t0 + kChunk, rows_of(c + 1), h, ptid);
            load_vb(a, smem, t0 + kChunk, rows_of(c + 1), h, ptid, ps ^ 1);
        }
        cp_async_commit();
    }
    cp_async_wait<0>();
}

// Group B, per chunk: the pair products Mqk and Diag(beta) A (mma.sync), V^T into the chunk's
// D1 buffer, (I + Diag(beta) A)^-1 by 16 x 16 blocks, T' in TF32, the Kt MMA and Bo = Mqk T'
// (mma.sync TF32) while it runs, then the hand-off: Kt read back into the stage in place of
// Kr, and the stage released to the state warps.
template <bool kPass1>
__device__ void solve_loop(const PrefillArgs &a, uint8_t *smem, Bars *B, uint32_t tmem, int nchunks) {
    const int btid = threadIdx.x - kFirstSolveWarp * 32;  // 0 .. 127
    const int bwarp = btid >> 5, lane = btid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const bool kt_thread = threadIdx.x == kKtThread;
    float *const tinv = reinterpret_cast<float *>(smem + kTinv);
    float *const pscr = reinterpret_cast<float *>(smem + kPscr);
    uint8_t *const at_hi = smem + kAtHi;

    float *const nt_s = reinterpret_cast<float *>(smem + kNt);
    float *const mq_s = reinterpret_cast<float *>(smem + kMq);
    float *const beta_s = reinterpret_cast<float *>(smem + kBetaS);

    for (int c = 0; c < nchunks; ++c) {
        const int ps = c & 1, db = c & 1;
        uint8_t *const stage = smem + kStage0 + ps * kStageBytes;
        const uint8_t *const rv = smem + kRawV + ps * kRawVBytes;
        const float *const rb = reinterpret_cast<const float *>(smem + kRawBeta) + ps * 32;
        {  // chunk c's operands are ready; its D1 buffer is free once chunk c - 2 is read out
            bool lost = !wait_or_abort(&B->ab_full[ps], (c >> 1) & 1, B, a.status);
            lost = lost || (c >= 2 && !wait_or_abort(&B->oread[db], ((c >> 1) + 1) & 1, B, a.status));
            if (bar_any(kBarSolve, kSolveThreads, lost)) break;
        }
        tc_fence_after();
        // ---- pair products: warp w takes N block w (the diagonal ones are inverted at once by
        //      the same warp) together with Mqk block w; warp 3 zeroes the blocks above the diagonal.
        //      Then V^T into D1 and beta aside, after which group A may refill what was read.
        if (bwarp < 3) pair_blocks_nq<kPass1>(smem, bwarp, lane, rb, mq_s, nt_s);
        mbar_arrive(&B->ab_empty);  // this thread's reads of the pair operands are done
        if (bwarp < 2) {
            __syncwarp();
            invert_diag16(nt_s, tinv, pscr + 64 * bwarp, 16 * bwarp, lane);
        } else if (bwarp == 3) {
            for (int idx = lane; idx < 256; idx += 32) {
                const int i = idx >> 4, j = 16 + (idx & 15);
                if (!kPass1) mq_s[i * kSq + j] = 0.0f;
                tinv[i * kSq + j] = 0.0f;
            }
        }
        v_to_tmem<kPass1>(tmem, rv, db, bwarp, lane);
        if (btid < kChunk) beta_s[btid] = rb[btid];
        tc_fence_before();
        bar_named(kBarSolve, kSolveThreads);
        mbar_arrive(&B->vfree);

        // ---- T = (I + N)^-1, N = Diag(beta) A strictly lower triangular, in FP32 by 16 x 16
        //      blocks: the diagonal blocks are inverted above, then T21 = -T22 N21 T11.
        {
            const int i = btid >> 3, j2 = 2 * (btid & 7);
            float2 p = splat2(0.0f);
#pragma unroll
            for (int l = 0; l < 16; ++l)
                p = fma2(splat2(nt_s[l * kSq + 16 + i]), *reinterpret_cast<const float2 *>(tinv + l * kSq + j2), p);
            *reinterpret_cast<float2 *>(pscr + i * 16 + j2) = p;
        }
        bar_named(kBarSolve, kSolveThreads);
        {
            const int i = btid >> 3, j2 = 2 * (btid & 7);
            float2 p = splat2(0.0f);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                p = fma2(splat2(-tinv[(16 + i) * kSq + 16 + k]), *reinterpret_cast<const float2 *>(pscr + k * 16 + j2), p);
            *reinterpret_cast<float2 *>(tinv + (16 + i) * kSq + j2) = p;
        }
        bar_named(kBarSolve, kSolveThreads);

        // ---- T' = T Diag(beta), stored as T'^T (row j, K index i) for the TF32 Kt MMA
        {
            const int j = btid & 31;
            // T' is truncated by the Kt MMA and Kt = Kr^T T' again by the state update: the
            // factor twice leaves both without bias
            const float bj = beta_s[j] * (kTruncBias * kTruncBias);
#pragma unroll
            for (int qh = 0; qh < 2; ++qh) {
                const int q = (btid >> 5) + 4 * qh;  // T'[4q .. 4q + 3][j]
                float hi[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) hi[r] = tinv[(4 * q + r) * kSq + j] * bj;
                const int off = core_off_tf32(j, 4 * q, 1024);
                *reinterpret_cast<float4 *>(at_hi + off) = make_float4(hi[0], hi[1], hi[2], hi[3]);
            }
        }
        fence_async_smem();
        bar_named(kBarSolve, kSolveThreads);

        // ---- Kt^T = Kr^T T' on tcgen05 (M128 N32 K32, both operands in shared memory; read
        //      back at the hand-off below), and Bo = Mqk T' (output pass) by mma.sync TF32.
        if (kt_thread) {  // warp 1: its Bo tiles are all zero
            tc_fence_after();
            const uint32_t kra = smem_addr(stage + kStKt), ah = smem_addr(at_hi);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_tf32_ss(tmem + kColKt, smem_desc_kmajor(kra + 256 * s, 128, kKtSbo),
                            smem_desc_kmajor(ah + 256 * s, 128, 1024), kIdescN32, s > 0);

            mma_commit(&B->kt);
        }
        __syncwarp();
        // V^T is in D1 and the Kt MMA is queued ahead of the projection's: the state warps may
        // start the chunk's projection
        mbar_arrive(&B->vready[ps]);
        if (!kPass1) {
            // warp b: the 16 x 8 tiles (b / 2, 2 (b % 2)) and (b / 2, 2 (b % 2) + 1) of Bo; Bo is
            // lower triangular, so K steps outside [column tile, row tile] contribute nothing
            const int mt = bwarp >> 1;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int nt = 2 * (bwarp & 1) + u;
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    if (ks < nt || ks > 2 * mt + 1) continue;
                    const int r0 = 16 * mt + g, k0 = 8 * ks + t4;
                    const uint32_t af[4] = {to_tf32(mq_s[r0 * kSq + k0]), to_tf32(mq_s[(r0 + 8) * kSq + k0]),
                                            to_tf32(mq_s[r0 * kSq + k0 + 4]), to_tf32(mq_s[(r0 + 8) * kSq + k0 + 4])};
                    const int jn = 8 * nt + g;
                    const float bj = beta_s[jn] * kTruncBias;  // Bo is truncated by the output MMA
                    mma_tf32_1688(acc, af, to_tf32(tinv[k0 * kSq + jn] * bj),
                                  to_tf32(tinv[(k0 + 4) * kSq + jn] * bj));
                }
                const int i0 = 16 * mt + g, j0 = 8 * nt + 2 * t4;
                *reinterpret_cast<float2 *>(stage + kStBo + core_off_tf32(i0, j0, 1024)) =
                    make_float2(acc[0], acc[1]);
                *reinterpret_cast<float2 *>(stage + kStBo + core_off_tf32(i0 + 8, j0, 1024)) =
                    make_float2(acc[2], acc[3]);
            }
        }
        // ---- hand-off: Kt in place of Kr, then the stage goes to the state warps
        {
            const bool lost = kt_thread && !wait_or_abort(&B->kt, c & 1, B, a.status);
            if (bar_any(kBarSolve, kSolveThreads, lost)) break;
        }
        tc_fence_after();
        kt_to_stage(tmem, stage, bwarp, lane);
        fence_async_smem();
        tc_fence_before();
#ifdef KDA_TEST_WITHHOLD_HANDOFF
        // failure-detection test build only: the hand-off of this chunk is lost, so the state
        // warps' bounded wait for it runs out and the CTA takes its abort path
        if (c == KDA_TEST_WITHHOLD_HANDOFF) continue;
#endif
        mbar_arrive(&B->prep[ps]);
    }
}

// ------------------------------------------------------------------ state warps

// Checkpoint row of the state after chunk `cg` (0-based within the sequence), or -1 when
// that chunk does not end a checkpoint interval or the row lies past the buffer.
__device__ __forceinline__ int64_t checkpoint_row(const PrefillArgs &a, int n, int cg, bool full_chunk) {
    if (a.ckpt_every <= 0 || !full_chunk) return -1;
    const int64_t end = (int64_t)(cg + 1) * kChunk;
    if (end % a.ckpt_every != 0) return -1;
    const int64_t row = (int64_t)a.ckpt_offsets[n] + end / a.ckpt_every - 1;
    if (row < 0 || row >= a.ckpt_rows) {
        if ((threadIdx.x & 127) == 0) report_error(a.status, KDA_ERR_DEVICE_INPUT, n);
        return -1;
    }
    return row;
}

// S (TMEM columns [col, col + 128), lane = dv) -> FP32 [dk][dv] at dst.
__device__ __forceinline__ void store_state(uint32_t tmem_state, uint32_t lane_base, int dv, float *dst) {
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        float v[16];
        tmem_ld16(tmem_state + lane_base + 16 * j, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[(16 * j + e) * kHeadDim + dv] = v[e];
    }
}

// dst[col] = src[col] * dec[col % 128] over `blocks` blocks of 32 columns of this thread's TMEM
// lane; the load of the next block is in flight while the current one is scaled and stored.
__device__ __forceinline__ void decay_columns(uint32_t src, uint32_t dst, const float *dec, int blocks) {
    float v[2][32];
    tmem_ld32(src, v[0]);
#pragma unroll 1
    for (int j = 0; j < blocks; j += 2) {
        tmem_wait_ld();
        if (j + 1 < blocks) tmem_ld32(src + 32 * (j + 1), v[1]);
        const float *d0 = dec + ((32 * j) & 127);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const float2 x = mul2(make_float2(v[0][e], v[0][e + 1]), *reinterpret_cast<const float2 *>(d0 + e));
            v[0][e] = x.x, v[0][e + 1] = x.y;
        }
        tmem_st32(dst + 32 * j, v[0]);
        if (j + 1 >= blocks) break;
        tmem_wait_ld();
        if (j + 2 < blocks) tmem_ld32(src + 32 * (j + 2), v[0]);
        const float *d1 = dec + ((32 * (j + 1)) & 127);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const float2 x = mul2(make_float2(v[1][e], v[1][e + 1]), *reinterpret_cast<const float2 *>(d1 + e));
            v[1][e] = x.x, v[1][e + 1] = x.y;
        }
        tmem_st32(dst + 32 * (j + 1), v[1]);
    }
    tmem_wait_st();
}

__device__ void state_loop(const PrefillArgs &a, uint8_t *smem, Bars *B, uint32_t tmem, int n, int h, int bos,
                           int eos, int nchunks, int chunk_base, const float *init, float *fin_out) {
    const int stid = threadIdx.x - kFirstStateWarp * 32;  // 0 .. 127
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;
    const int dv = 32 * quad + lane;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const bool mma_thread = (warp == kFirstStateWarp) && (lane == 0);
    const bool mma_thread2 = (warp == kFirstStateWarp + 1) && (lane == 0);  // a second MMA stream

    // initial state -> S^T buffer 0 (lane = dv, column = dk)
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            v[e] = init ? init[(16 * j + e) * kHeadDim + dv] : 0.0f;
        tmem_st16(tmem + lane_base + kColS + 16 * j, v);
    }
    tmem_wait_st();
    tc_fence_before();
    bar_named(kBarState, kStateThreads);
    tc_fence_after();

    bool alive = true;
    for (int c = 0; c < nchunks && alive; ++c) {
        const int ps = c & 1, db = c & 1;
        const uint32_t cur = kColS;  // the state stays in one buffer, decayed in place
        const uint8_t *stage = smem + kStage0 + ps * kStageBytes;
        // the projection needs the chunk's operands (W, the decay), V^T in D1 and the previous
        // update; Kt and Bo, which group B hands over later, only the output and update MMAs
        if (!wait_or_abort(&B->vready[ps], (c >> 1) & 1, B, a.status)) break;
        if (c >= 1 && !wait_or_abort(&B->g2, (c - 1) & 1, B, a.status)) break;
        tc_fence_after();
        if (mma_thread) {
            const uint32_t wbase = smem_addr(stage + kStW);
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                mma_tf32_ts(tmem + kColD1 + 64 * db, tmem + cur + 8 * s,
                            smem_desc_sw128(wbase + (s >> 2) * 8192 + (s & 3) * 32), kIdescG1, true);
                if ((s & 3) == 3) mma_commit(&B->g1q[s >> 2]);  // S^T columns [8 s - 24, 8 s + 8) read
            }
        }
        __syncwarp();
        if (c >= 1) {  // checkpoint of the state after chunk c-1 (read alongside the projection)
            const int64_t row = checkpoint_row(a, n, chunk_base + c - 1, true);
            if (row >= 0)
                store_state(tmem + cur, lane_base, dv,
                            a.ckpt + ((size_t)row * a.num_heads + h) * (kHeadDim * kHeadDim));
        }
        // the decay in place, each 32-column block of S^T as soon as the projection's MMAs
        // that read it are done, the rest of the projection still running (run beside the
        // whole projection, into a second buffer, the two shared the tensor memory's bandwidth)
        bool lost = false;
#pragma unroll 1
        for (int q = 0; q < 4 && !lost; ++q) {
            lost = !wait_or_abort(&B->g1q[q], c & 1, B, a.status);
            tc_fence_after();
            if (!lost)
                decay_columns(tmem + lane_base + cur + 32 * q, tmem + lane_base + cur + 32 * q,
                              reinterpret_cast<const float *>(stage + kStDec) + 32 * q, 1);
        }
        lost = lost || !wait_or_abort(&B->prep[ps], (c >> 1) & 1, B, a.status);  // Kt and Bo
        tc_fence_before();
        if (bar_any(kBarState, kStateThreads, lost)) break;
        tc_fence_after();
        // S^T += R^T Kt on the decayed state, then O^T = (Qbar S)^T + R^T Bo^T (A = R^T =
        // D1^T[:, 0:32]), both from one thread: the update goes first, since the next chunk's
        // projection waits for it; the output, which only its read-out waits for, queues behind
        // it. (Issued from two threads at once, the two interleaved on the tensor pipe.) The
        // stage is released with the update although the output MMAs still read Bo from it:
        // nothing writes Bo there again before group B's wait for this chunk's read-out.
        if (mma_thread2) {
            const uint32_t kbase = smem_addr(stage + kStKt);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_tf32_ts(tmem + cur, tmem + kColD1 + 64 * db + 8 * s,
                            smem_desc_kmajor(kbase + 256 * s, 128, kKtSbo), kIdescG2, true);
            mma_commit(&B->g2);
            mma_commit(&B->g2s[ps]);
            const uint32_t obase = smem_addr(stage + kStBo);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_tf32_ts(tmem + kColD1 + 64 * db + 32, tmem + kColD1 + 64 * db + 8 * s,
                            smem_desc_kmajor(obase + 256 * s, 128, 1024), kIdescN32, true);
            mma_commit(&B->go);
        }
        __syncwarp();
        // output read-out: O^T = D1^T[:, 32:64]
        if (!wait_or_abort(&B->go, c & 1, B, a.status)) break;
        tc_fence_after();
        float o0[16], o1[16];
        tmem_ld16(tmem + lane_base + kColD1 + 64 * db + 32, o0);
        tmem_ld16(tmem + lane_base + kColD1 + 64 * db + 48, o1);
        tmem_wait_ld();
        // D1 buffer db is free again
        tc_fence_before();
        mbar_arrive(&B->oread[db]);
        // staged through shared memory for 16-byte row stores; the buffer is reused by the
        // next chunk only after the barrier that closes this iteration
        // tokens t and 16 + t share a 32-bit word: ost[t][dv] = bf16x2(O[t][dv], O[16 + t][dv]),
        // with the two 16-byte halves of each 32-byte group swapped where dv bit 5 is set, so
        // that a quarter warp's 16-byte reads below (32 bytes apart) hit all 8 bank groups
        uint32_t *const ost = reinterpret_cast<uint32_t *>(smem + kOst);
        const int dvs = dv ^ (((dv >> 5) & 1) << 2);
#pragma unroll
        for (int t = 0; t < 16; ++t) ost[t * kHeadDim + dvs] = pack_bf16(o0[t], o1[t]);
        bar_named(kBarState, kStateThreads);
        const int t0 = bos + kChunk * c;
        const int L = min(kChunk, eos - t0);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int idx = stid + kStateThreads * m;
            const int t = idx >> 4, vec = idx & 15;
            const int sw = 4 * ((vec >> 2) & 1);  // where dv = 8 vec .. 8 vec + 3 was stored
            const uint4 w0 = *reinterpret_cast<const uint4 *>(ost + t * kHeadDim + vec * 8 + sw);
            const uint4 w1 = *reinterpret_cast<const uint4 *>(ost + t * kHeadDim + vec * 8 + (4 - sw));
            __nv_bfloat16 *const orow = a.out + ((size_t)(t0 + t) * a.num_heads + h) * kHeadDim + vec * 8;
            if (t < L)
                *reinterpret_cast<uint4 *>(orow) =
                    make_uint4(__byte_perm(w0.x, w0.y, 0x5410), __byte_perm(w0.z, w0.w, 0x5410),
                               __byte_perm(w1.x, w1.y, 0x5410), __byte_perm(w1.z, w1.w, 0x5410));
            if (16 + t < L)
                *reinterpret_cast<uint4 *>(orow + (size_t)16 * a.num_heads * kHeadDim) =
                    make_uint4(__byte_perm(w0.x, w0.y, 0x7632), __byte_perm(w0.z, w0.w, 0x7632),
                               __byte_perm(w1.x, w1.y, 0x7632), __byte_perm(w1.z, w1.w, 0x7632));
        }
        alive = !bar_any(kBarState, kStateThreads, B->abort != 0);
    }

    // final state (after the last update has completed); the abort decision is uniform
    if (!bar_any(kBarState, kStateThreads, B->abort != 0)) {
        if (nchunks > 0 && !wait_or_abort(&B->g2, (nchunks - 1) & 1, B, a.status)) return;
        tc_fence_after();
        if (nchunks > 0) {
            const bool full = bos + kChunk * nchunks <= eos;
            const int64_t row = checkpoint_row(a, n, chunk_base + nchunks - 1, full);
            if (row >= 0)
                store_state(tmem + kColS, lane_base, dv,
                            a.ckpt + ((size_t)row * a.num_heads + h) * (kHeadDim * kHeadDim));
        }
        if (fin_out != nullptr) {
            const uint32_t fin = kColS;
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                float v[16];
                tmem_ld16(tmem + lane_base + fin + 16 * j, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) fin_out[(16 * j + e) * kHeadDim + dv] = v[e];
            }
        }
    }
}

// ------------------------------------------------------------------ window pass: state warps
//
// From a zero start the window's end state E is the S chain with V; the window's linear map M
// (S_end = M S_start + E) is the same recurrence with V = 0 started from I, so both chains
// share the producers' operands. TMEM: S^T [0,128), M^T [128,256) (lanes = dv resp. dk'),
// D1 for S (= Wv^T + U^T) at [256 + 32b), D1 for M at [320 + 32b). The decay runs in place
// after the projection has read the state.
constexpr uint32_t kColM = 128;
constexpr uint32_t kColD1M = 320;
__device__ void state_loop_pass1(const PrefillArgs &a, uint8_t *smem, Bars *B, uint32_t tmem, int nchunks,
                                 float *E_out, float *Mt_out, int *map_nonzero) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;
    const int row = 32 * quad + lane;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const bool mma_thread = (warp == kFirstStateWarp) && (lane == 0);
    const bool mma_thread2 = (warp == kFirstStateWarp + 1) && (lane == 0);  // a second MMA stream

#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        float z[16], id[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            z[e] = 0.0f;
            id[e] = (16 * j + e == row) ? 1.0f : 0.0f;
        }
        tmem_st16(tmem + lane_base + kColS + 16 * j, z);
        tmem_st16(tmem + lane_base + kColM + 16 * j, id);
    }
    tmem_wait_st();
    tc_fence_before();
    bar_named(kBarState, kStateThreads);
    tc_fence_after();

    for (int c = 0; c < nchunks; ++c) {
        const int ps = c & 1, db = c & 1;
        const uint8_t *stage = smem + kStage0 + ps * kStageBytes;
        // the projections need V^T in D1 (and the chunk's operands); Kt only the updates
        if (!wait_or_abort(&B->vready[ps], (c >> 1) & 1, B, a.status)) break;
        if (c >= 1 && !wait_or_abort(&B->g2, (c - 1) & 1, B, a.status)) break;
        tc_fence_after();
        // the S chain and the M chain from two warps, in parallel (both commit each g1q[q])
        if (mma_thread || mma_thread2) {
            const uint32_t wbase = smem_addr(stage + kStW);
            const uint32_t d = mma_thread ? kColD1 + 32 * db : kColD1M + 32 * db;
            const uint32_t src = mma_thread ? kColS : kColM;
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const uint64_t bd = smem_desc_sw128(wbase + (s >> 2) * 8192 + (s & 3) * 32);
                // D1 for S starts from V; D1 for M from zero
                mma_tf32_ts(tmem + d, tmem + src + 8 * s, bd, kIdescN32, mma_thread || s > 0);
                if ((s & 3) == 3) mma_commit(&B->g1q[s >> 2]);
            }
        }
        __syncwarp();
        // decay S and M in place (columns [0, 128) and [128, 256)), each 32-column block as soon
        // as both projections have read it
        bool dlost = false;
#pragma unroll 1
        for (int q = 0; q < 4 && !dlost; ++q) {
            dlost = !wait_or_abort(&B->g1q[q], c & 1, B, a.status);
            tc_fence_after();
            if (!dlost) {
                const float *const dq = reinterpret_cast<const float *>(stage + kStDec) + 32 * q;
                decay_columns(tmem + lane_base + kColS + 32 * q, tmem + lane_base + kColS + 32 * q, dq, 1);
                decay_columns(tmem + lane_base + kColM + 32 * q, tmem + lane_base + kColM + 32 * q, dq, 1);
            }
        }
        {
            const bool lost = dlost || !wait_or_abort(&B->prep[ps], (c >> 1) & 1, B, a.status);  // Kt
            tc_fence_before();
            if (bar_any(kBarState, kStateThreads, lost)) break;
        }
        mbar_arrive(&B->oread[db]);
        bar_named(kBarState, kStateThreads);
        tc_fence_after();
        if (mma_thread || mma_thread2) {  // both commit g2 and g2s
            const uint32_t kbase = smem_addr(stage + kStKt);
            const uint32_t d = mma_thread ? kColS : kColM;
            const uint32_t r = mma_thread ? kColD1 + 32 * db : kColD1M + 32 * db;
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_tf32_ts(tmem + d, tmem + r + 8 * s, smem_desc_kmajor(kbase + 256 * s, 128, kKtSbo), kIdescG2, true);
            mma_commit(&B->g2);
            mma_commit(&B->g2s[ps]);
        }
        __syncwarp();
        if (bar_any(kBarState, kStateThreads, B->abort != 0)) break;
    }
    if (bar_any(kBarState, kStateThreads, B->abort != 0)) return;
    {  // one decision for all: the map flag below is reduced over a barrier of these threads
        const bool lost = nchunks > 0 && !wait_or_abort(&B->g2, (nchunks - 1) & 1, B, a.status);
        if (bar_any(kBarState, kStateThreads, lost)) return;
    }
    tc_fence_after();
    // E[dk][dv] from S^T (lane dv, column dk); the map is stored transposed, M^T[dk'][dk],
    // straight from its TMEM rows (lane dk', column dk), which is the order the carry reads.
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        float v[16];
        tmem_ld16(tmem + lane_base + kColS + 16 * j, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) E_out[(16 * j + e) * kHeadDim + row] = v[e];
    }
    bool nz = false;
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        float v[16];
        tmem_ld16(tmem + lane_base + kColM + 16 * j, v);
        tmem_wait_ld();
        float4 *dst = reinterpret_cast<float4 *>(Mt_out + (size_t)row * kHeadDim + 16 * j);
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) dst[e4] = make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
#pragma unroll
        for (int e = 0; e < 16; ++e) nz = nz || v[e] != 0.0f;
    }
    // (NaN counts as nonzero)
    const bool any_nz = bar_any(kBarState, kStateThreads, nz);
    if (threadIdx.x == kFirstStateWarp * 32) *map_nonzero = any_nz ? 1 : 0;
}

// ------------------------------------------------------------------ kernel

// Shortest window of the window schedule, in chunks: each window adds a map to the carry.
constexpr int kMinWindowChunks = 4;

struct WindowSpan {
    int bos, eos, w, wins_seq, lw;  // lw: chunks per window of this sequence
    bool live;
};

// Bounds of sequence n (validated and clamped; one caller per sequence, `report`, records
// bad bounds) and the span of window `w` of it.
__device__ __forceinline__ WindowSpan window_span(const PrefillArgs &a, int n, int w, int W, bool report) {
    int sb = a.cu_seqlens[n], se = a.cu_seqlens[n + 1];
    if (sb < 0 || se < sb || se > a.total_tokens) {
        if (threadIdx.x == 0 && w == 0 && report)
            report_error(a.status, KDA_ERR_DEVICE_INPUT, n);
        sb = min(max(sb, 0), a.total_tokens);
        se = min(max(se, sb), a.total_tokens);
    }
    // a sequence's chunks are split into at most W windows of equal length, each at least
    // kMinWindowChunks long (W = 1: one window)
    const int chunks = (se - sb + kChunk - 1) / kChunk;
    const int lw = W > 1 ? max((chunks + W - 1) / W, kMinWindowChunks) : max(chunks, 1);
    WindowSpan sp;
    sp.lw = lw;
    sp.wins_seq = max(1, (chunks + lw - 1) / lw);
    sp.w = w;
    sp.bos = sb + kChunk * lw * w;
    sp.eos = min(se, sp.bos + kChunk * lw);
    sp.live = w < sp.wins_seq;
    if (!sp.live) sp.bos = sp.eos = sb;
    return sp;
}

// Launch order of the chains. CTAs start roughly in index order, one per SM, so a batch of
// unequal sequences finishes soonest when the longest start first (the longest-processing-
// time-first rule of list scheduling). Position p of the order is head p % H of the
// sequence ranked p / H by length, longest first, ties by index; the ranks are a permutation
// for any cu_seqlens, so every chain runs exactly once. Batches of more than kRankedSeqs
// sequences keep index order (ranking them would cost each CTA more than it saves).
constexpr int kRankedSeqs = 256;

// Sequence of rank j; every thread of the CTA calls it (it holds three CTA barriers) with
// `scratch` pointing to kRankedSeqs + 1 ints of shared memory that nothing else uses until
// it returns.
__device__ __forceinline__ int seq_of_rank(const PrefillArgs &a, int j, int *scratch) {
    const int N = a.num_seqs;
    if (N <= 1 || N > kRankedSeqs) return j;
    int *len = scratch;
    int *pick = scratch + kRankedSeqs;
    for (int i = threadIdx.x; i < N; i += blockDim.x)  // wrapping difference: any input orders
        len[i] = (int)((unsigned)__ldg(a.cu_seqlens + i + 1) - (unsigned)__ldg(a.cu_seqlens + i));
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const int li = len[i];
        int r = 0;
        for (int m = 0; m < N; ++m) {
            const int lm = len[m];
            r += (lm > li) | ((lm == li) & (m < i));
        }
        if (r == j) *pick = i;
    }
    __syncthreads();
    const int n = *pick;
    __syncthreads();
    return n;
}

// Slot of windowed chain `lc` (counted from position a.seq_chains): k = 0, the start state of
// window w (w = 1 .. wins - 1); k = 1 and 2, the end state E and the map M of window w
// (w = 1 .. wins - 2).
__device__ __forceinline__ float *window_slot(const PrefillArgs &a, int lc, int w, int k) {
    const int W = a.wins;
    const int idx = (k == 0) ? w - 1 : (k == 1 ? (W - 1) + (w - 1) : (W - 1) + (W - 2) + (w - 1));
    return a.ws + ((size_t)lc * (size_t)window_slots(W) + (size_t)idx) * (kHeadDim * kHeadDim);
}

// Whether window w of windowed chain lc has a map with a nonzero entry (written by the window
// pass; a map whose every entry underflowed to zero makes the carry's step S = E).
__device__ __forceinline__ int *window_flag(const PrefillArgs &a, int lc, int w) {
    const int64_t chains = (int64_t)a.num_seqs * a.num_heads - a.seq_chains;
    int *const flags = reinterpret_cast<int *>(a.ws + (size_t)chains * (size_t)window_slots(a.wins) * (kHeadDim * kHeadDim));
    return flags + (size_t)lc * a.wins + w;
}

template <bool kPass1>
__global__ void __launch_bounds__(kThreadsTc, 1) kda_prefill_tc_kernel(const PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the swizzled operands need 1024-byte alignment; the launch reserves the slack
    uint8_t *const smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    Bars *B = reinterpret_cast<Bars *>(smem + kBars);
    const int warp = threadIdx.x >> 5;
    const int H = a.num_heads;
    // a whole chain, or window w of windowed chain lc
    const bool windowed = (int)blockIdx.x >= a.seq_ctas;
    int pos = blockIdx.x, w = 0, lc = 0;  // pos: position in the launch order
    if (windowed) {
        const int b = (int)blockIdx.x - a.seq_ctas;
        lc = b / a.win_count;
        w = a.win_first + (b - lc * a.win_count);
        pos = a.seq_chains + lc;
    }
    const int h = pos % H;
    // the stage area is free until the pipeline starts
    const int n = seq_of_rank(a, pos / H, reinterpret_cast<int *>(smem + kStage0));
    const int chain = n * H + h;
    const WindowSpan sp = window_span(a, n, w, windowed ? a.wins : 1, h == 0);
    // A window pass that follows a chunk loop over other chains may start while that loop's
    // last chains still run; it ends only after them, so every later launch is ordered after
    // both (griddepcontrol.wait returns at once when nothing precedes the grid).
    if (!kPass1) pdl_launch_dependents();
    // The window pass covers every window but the first (which starts from the initial state)
    // and the last (whose map is never needed); the output pass, every window that exists.
    if (kPass1 ? (w >= sp.wins_seq - 1) : !sp.live) {
        if (kPass1) pdl_wait();
        return;
    }
    const int bos = sp.bos, eos = sp.eos;
    const int nchunks = (eos - bos + kChunk - 1) / kChunk;

    if (threadIdx.x == 0) {
        mbar_init(&B->prep[0], kSolveThreads);
        mbar_init(&B->prep[1], kSolveThreads);
        mbar_init(&B->vready[0], kSolveThreads);
        mbar_init(&B->vready[1], kSolveThreads);
        mbar_init(&B->ab_full[0], kProdThreads);
        mbar_init(&B->ab_full[1], kProdThreads);
        mbar_init(&B->ab_empty, kSolveThreads);
        mbar_init(&B->vfree, kSolveThreads);
        mbar_init(&B->go, 1);
        mbar_init(&B->kt, 1);
        mbar_init(&B->g2, kPass1 ? 2 : 1);
        mbar_init(&B->g2s[0], kPass1 ? 2 : 1);
        mbar_init(&B->g2s[1], kPass1 ? 2 : 1);
        mbar_init(&B->oread[0], kStateThreads);
        mbar_init(&B->oread[1], kStateThreads);
        mbar_init(&B->drain, 3);
        for (int q = 0; q < 4; ++q) mbar_init(&B->g1q[q], kPass1 ? 2 : 1);
        B->abort = 0;
        fence_mbar_init();
    }
    if (warp == kFirstStateWarp) {
        tmem_alloc(&B->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;

    if (warp < kProducerWarps) {
        producer_loop<kPass1>(a, smem, B, tmem, n, h, bos, eos, nchunks);
    } else if (warp < kFirstStateWarp) {
        solve_loop<kPass1>(a, smem, B, tmem, nchunks);
    } else {
        if (kPass1) {
            state_loop_pass1(a, smem, B, tmem, nchunks, window_slot(a, lc, w, 1), window_slot(a, lc, w, 2),
                             window_flag(a, lc, w));
        } else {
            // the start state of a window is the carry's output; the operand and solve warps
            // read only the inputs and start before the carry has finished
            pdl_wait();
            const size_t sbase = (size_t)chain * kHeadDim * kHeadDim;
            const float *init = (w == 0) ? (a.init_state ? a.init_state + sbase : nullptr) : window_slot(a, lc, w, 0);
            // the last window ends the chain; window 0 of a windowed chain starts window 1
            float *fin = (w == sp.wins_seq - 1) ? (a.final_state ? a.final_state + sbase : nullptr)
                                                : (w == 0 ? window_slot(a, lc, 1, 0) : nullptr);
            const int chunk_base = sp.lw * w;
            state_loop(a, smem, B, tmem, n, h, bos, eos, nchunks, chunk_base, init, fin);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // After an abort (every group has left its loop, so all threads read the same flag), the
    // three threads that issue MMAs (group B's Kt thread and the state warps' two) drain
    // whatever they still have in flight before the tensor memory is released; the wait is
    // bounded like every other.
    if (B->abort != 0 && (threadIdx.x == kKtThread || threadIdx.x == kFirstStateWarp * 32 ||
                          threadIdx.x == (kFirstStateWarp + 1) * 32)) {
        mma_commit(&B->drain);
        mbar_wait(&B->drain, 0);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    if (warp == kFirstStateWarp) tmem_dealloc(tmem, kTmemCols);
    if (kPass1) pdl_wait();
}

// ------------------------------------------------------------------ window carry
//
// S_start[w+1] = M_w S_start[w] + E_w for every window of a chain, in FP32 on CUDA cores.
// The dv columns of S are independent: each CTA carries 8 of them through all windows.
// Warp p owns the 16 values of k in [16p, 16p + 16) and, per lane, 4 rows x 8 columns of
// the product. The map arrives transposed (row k of M^T is column k of M), so a warp reads
// 512 contiguous bytes per k. The loads run two window steps ahead, in two register sets
// that alternate between steps: each register is refilled with the map of window w + 2 as
// soon as window w's value has been read (one step ahead, the steps waited on the loads).
// The 8 partial products are summed through shared memory, in the order of the slices, and
// warp p also sums and rewrites rows [16p, 16p + 16) of S, the rows its next window step
// reads, so one CTA barrier per window step suffices. The products run as packed FP32
// pairs of columns. A window whose map underflowed to zero everywhere (the window pass
// records a flag per window) contributes S_start[w+1] = E_w: its map is neither loaded nor
// multiplied, and a chain with only such windows copies its start states in one pass.
constexpr int kCarryCols = 8;
constexpr int kCarryWarps = kHeadDim / 16;
constexpr int kCarryThreads = 32 * kCarryWarps;
// Partial products, double-buffered by window step: [buffer][slice][column][row], rows padded
// to 144 floats, so that columns c and c + 1 start 64 bytes apart in the banks and a warp's
// 16-byte reads of 8 columns x 4 rows take the minimum 4 wavefronts.
constexpr int kCarryRowPad = kHeadDim + 16;
constexpr int kCarryDynSmem = 2 * kCarryWarps * kCarryCols * kCarryRowPad * 4;

constexpr int kCarryFlagWins = 256;  // windows whose map flag the carry keeps; later ones count as nonzero

__global__ void __launch_bounds__(kCarryThreads) kda_window_carry_kernel(const PrefillArgs a) {
    __shared__ __align__(16) float S[kHeadDim][kCarryCols];
    __shared__ int s_nz[kCarryFlagWins];
    extern __shared__ __align__(16) float carry_dyn[];
    auto part = reinterpret_cast<float (*)[kCarryWarps][kCarryCols][kCarryRowPad]>(carry_dyn);
    const int blocks = kHeadDim / kCarryCols;
    const int lc = blockIdx.x / blocks;  // chain of this launch
    const int pos = a.seq_chains + lc;  // position in the launch order
    const int c0 = (blockIdx.x - lc * blocks) * kCarryCols;
    pdl_launch_dependents();  // the output pass may start now; it waits for this grid on the device
    const int n = seq_of_rank(a, pos / a.num_heads, reinterpret_cast<int *>(carry_dyn));
    const WindowSpan sp = window_span(a, n, 0, a.wins, false);
    if (sp.wins_seq <= 2) return;  // window 1's start state comes from window 0 itself
    const int last = sp.wins_seq - 2;  // the steps run over the windows with a map
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // which maps have a nonzero entry: a step whose map underflowed to zero everywhere is
    // S_start[w+1] = E_w, and neither its map nor the product is needed
    for (int t = 1 + tid; t <= last && t < kCarryFlagWins; t += kCarryThreads) s_nz[t] = __ldcg(window_flag(a, lc, t));
    __syncthreads();
    auto nonzero = [&](int w) { return w >= kCarryFlagWins || s_nz[w] != 0; };
    {
        bool any = false;
        for (int w = 1; w <= last; ++w) any = any || nonzero(w);
        if (!any) {
            // every map is zero (fast decay over a window): each start state is the previous
            // window's end state, S_start[w+1] = E_w, independent of the others, so the copies
            // go out 8 windows at a time; thread t moves row t / 2, columns 4 (t % 2) .. + 3
            const size_t off = (size_t)(tid >> 1) * kHeadDim + c0 + 4 * (tid & 1);
            for (int w0 = 1; w0 <= last; w0 += 8) {
                float4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (w0 + j <= last) v[j] = __ldcg(reinterpret_cast<const float4 *>(window_slot(a, lc, w0 + j, 1) + off));
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (w0 + j <= last) *reinterpret_cast<float4 *>(window_slot(a, lc, w0 + j + 1, 0) + off) = v[j];
            }
            return;
        }
    }
    const int k0 = 16 * warp;
    const int rq = lane & 3, cc = lane >> 2;
    // warp p multiplies rows [k0, k0 + 16) of S and also reduces and rewrites exactly those
    // rows, so between window steps it waits only for its own lanes
    const int r4 = k0 + 4 * rq;  // reduction: rows r4 .. r4 + 3, column cc
    {
        const float *const src = window_slot(a, lc, 1, 0) + (size_t)r4 * kHeadDim + c0 + cc;
#pragma unroll
        for (int i = 0; i < 4; ++i) S[r4 + i][cc] = __ldcg(src + i * kHeadDim);
    }
    auto map_row = [&](int w, int kk) {
        return reinterpret_cast<const float4 *>(window_slot(a, lc, w, 2) + (size_t)(k0 + kk) * kHeadDim + 4 * lane);
    };
    float e[4];
    auto load_e = [&](int w) {
        const float *const src = window_slot(a, lc, w, 1) + (size_t)r4 * kHeadDim + c0 + cc;
#pragma unroll
        for (int i = 0; i < 4; ++i) e[i] = __ldcg(src + i * kHeadDim);
    };
    // ma, mb: M^T[k0 + kk][4 lane .. 4 lane + 3] of windows w (set (w - 1) % 2) and w + 1
    float4 ma[16], mb[16];
    if (nonzero(1)) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) ma[kk] = __ldcg(map_row(1, kk));
    }
    if (last >= 2 && nonzero(2)) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) mb[kk] = __ldcg(map_row(2, kk));
    }
    load_e(1);
    __syncwarp();
    auto step = [&](int w, float4 (&mv)[16]) {
        const int b = w & 1;
        const bool ahead = w + 2 <= last && nonzero(w + 2);  // window w + 2's map is needed
        if (!nonzero(w)) {  // S_start[w+1] = E_w
            if (ahead) {
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) mv[kk] = __ldcg(map_row(w + 2, kk));
            }
            // one CTA barrier per step, as in a product step, so that the two partial-sum
            // buffers keep alternating safely
            __syncthreads();
            const float sum[4] = {e[0], e[1], e[2], e[3]};
            if (w + 1 <= last) load_e(w + 1);
            float *const out = window_slot(a, lc, w + 1, 0) + (size_t)r4 * kHeadDim + c0 + cc;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                S[r4 + i][cc] = sum[i];
                out[i * kHeadDim] = sum[i];
            }
            __syncwarp();  // this warp's rows of S are rewritten
            return;
        }
        float acc[4][kCarryCols];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < kCarryCols; ++c) acc[r][c] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4 s0 = *reinterpret_cast<const float4 *>(&S[k0 + kk][0]);
            const float4 s1 = *reinterpret_cast<const float4 *>(&S[k0 + kk][4]);
            const float2 sv[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w), make_float2(s1.x, s1.y),
                                  make_float2(s1.z, s1.w)};
            const float m[4] = {mv[kk].x, mv[kk].y, mv[kk].z, mv[kk].w};
            if (ahead) mv[kk] = __ldcg(map_row(w + 2, kk));
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < kCarryCols / 2; ++c) {
                    const float2 x = __ffma2_rn(make_float2(m[r], m[r]), sv[c],
                                                make_float2(acc[r][2 * c], acc[r][2 * c + 1]));
                    acc[r][2 * c] = x.x;
                    acc[r][2 * c + 1] = x.y;
                }
        }
#pragma unroll
        for (int c = 0; c < kCarryCols; ++c)
            *reinterpret_cast<float4 *>(&part[b][warp][c][4 * lane]) =
                make_float4(acc[0][c], acc[1][c], acc[2][c], acc[3][c]);
        __syncthreads();  // every slice's partial products of step w are written
        float sum[4] = {e[0], e[1], e[2], e[3]};
        if (w + 1 <= last) load_e(w + 1);
#pragma unroll
        for (int p = 0; p < kCarryWarps; ++p) {
            const float4 x = *reinterpret_cast<const float4 *>(&part[b][p][cc][r4]);
            sum[0] += x.x, sum[1] += x.y, sum[2] += x.z, sum[3] += x.w;
        }
        float *const out = window_slot(a, lc, w + 1, 0) + (size_t)r4 * kHeadDim + c0 + cc;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            S[r4 + i][cc] = sum[i];
            out[i * kHeadDim] = sum[i];
        }
        __syncwarp();  // this warp's rows of S are rewritten
    };
    for (int w = 1;;) {  // two steps per turn, so that each names its register set statically
        if (w > last) break;
        step(w, ma);
        ++w;
        if (w > last) break;
        step(w, mb);
        ++w;
    }
}

template <bool kPass1>
cudaError_t configure_once() {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kda_prefill_tc_kernel<kPass1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLaunch);
        // the window pass is configured once per device, and with it the carry it feeds
        if (e == cudaSuccess && kPass1)
            e = cudaFuncSetAttribute(kda_window_carry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCarryDynSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    return cudaSuccess;
}

}  // namespace

// Windows pay off only when the chains alone leave most of the GPU idle: each window
// costs a window pass (about the price of the sequential chunk loop over its chunks) and
// the FP32 carry; at least 3 windows of at least 4 chunks each are required.
WindowPlan plan_windows(int32_t num_seqs, int32_t total_tokens, int32_t num_heads, int32_t sms) {
    WindowPlan p = {1, 0, 0};
    const int64_t chains = (int64_t)num_seqs * num_heads;
    const int64_t max_chunks = ((int64_t)total_tokens + kChunk - 1) / kChunk;  // bound on any one sequence
    if (chains <= 0 || sms <= 0) return p;
    // Chains run one CTA each, a wave of `sms` at a time. When the last wave would hold at
    // most a third of the GPU (or all chains fit in such a wave), those chains are cut into
    // windows instead, at least three per chain, to fill the GPU; the full waves before them
    // are unchanged. Each sequence's window length follows from its own length on the device.
    const int64_t tail = chains % sms;
    if (tail == 0 || tail * 3 > sms) return p;
    // window 0 of each chain runs beside the window pass of windows 1 .. wins - 2, and the
    // output pass covers windows 1 .. wins - 1: wins - 1 CTAs per chain in each phase
    const int64_t wins = std::min<int64_t>(sms / tail + 1, max_chunks / kMinWindowChunks);
    if (wins < 3) return p;
    p.wins = (int32_t)wins;
    p.ws_bytes = tail * window_slots(wins) * kStateBytes + window_flag_bytes(tail, wins);
    p.seq_chains = (int32_t)(chains - tail);
    return p;
}

// Launch on `stream` that may start while the previous kernel of the stream is finishing;
// the kernel orders its dependent reads with griddepcontrol.wait.
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       const PrefillArgs &a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

cudaError_t launch_prefill_tc(const PrefillArgs &args, cudaStream_t stream) {
    cudaError_t e = configure_once<false>();
    if (e != cudaSuccess) return e;
    const int64_t all_chains = (int64_t)args.num_seqs * args.num_heads;
    const int W = args.wins >= 3 ? args.wins : 1;
    // positions [0, seq) run as whole chains, [seq, all) on the window schedule
    const int64_t seq = W == 1 ? all_chains : args.seq_chains;
    const int64_t chains = all_chains - seq;
    PrefillArgs a = args;
    a.wins = W;
    a.seq_chains = (int32_t)seq;
    // 1. The chunk loop: whole chains, then window 0 of each windowed chain, which leaves its
    //    end state as window 1's start.
    a.seq_ctas = (int32_t)seq;
    a.win_first = 0;
    a.win_count = 1;
    kda_prefill_tc_kernel<false><<<(unsigned)(seq + chains), kThreadsTc, kSmemLaunch, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess || W == 1) return e;
    // 2. The window pass over windows 1 .. W - 2, a programmatic dependent of the chunk loop:
    //    it fills the SMs as the loop's last CTAs start or leave, and waits for the loop before
    //    it exits, so every later launch is ordered after both.
    e = configure_once<true>();
    if (e != cudaSuccess) return e;
    a.seq_ctas = 0;
    a.win_first = 1;
    a.win_count = W - 2;
    e = launch_pdl(kda_prefill_tc_kernel<true>, (unsigned)(chains * (W - 2)), kThreadsTc, kSmemLaunch, stream, a);
    if (e != cudaSuccess) return e;
    // 3. The carry: start states of windows 2 .. W - 1.
    kda_window_carry_kernel<<<(unsigned)(chains * (kHeadDim / kCarryCols)), kCarryThreads, kCarryDynSmem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 4. The output pass over windows 1 .. W - 1, a programmatic dependent of the carry: its
    //    operand and solve warps work ahead while its state warps wait on the device for the
    //    carried start states.
    a.win_count = W - 1;
    return launch_pdl(kda_prefill_tc_kernel<false>, (unsigned)(chains * (W - 1)), kThreadsTc, kSmemLaunch, stream, a);
}

}  // namespace kda
