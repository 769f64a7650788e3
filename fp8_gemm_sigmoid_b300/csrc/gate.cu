// gate.cu -- a1: the sigmoid MoEGate with group-limited top-k and the fused per-expert
// histogram.
//
// DeepSeek-V3 co-design teardown (wsisp.com) §2.2, MoEGate listing: logits in FP32,
// sigmoid scores, selection-only bias, group score = sum of the two best selection scores
// of the group, keep topk_group groups, top_k experts among them, weights from the
// un-biased scores, normalised (top_k > 1) and scaled; §2.3: per-expert token counts.
//
// Two kernels:
//  - gate_tc_kernel (BF16 x and Wg, E <= 256): the [128 tokens x E] logit tile is one
//    tcgen05 MMA accumulation in TMEM (BF16 x BF16 products are exact in FP32, FP32
//    accumulation), fed by TMA; then all 8 warps run the selection, two threads per token
//    (each reads half of the token's groups from TMEM, the pair exchanges group scores and
//    merges two local top-k lists through shared memory).  The kernel streams x once.
//    With xq / xs given it also quantises x into 1x128 FP8 tiles (précis §3.2) while the
//    tiles pass through shared memory for the MMA: eight otherwise idle warps, two threads
//    per token row, read each 128-column block from the operand ring, so x is read from HBM
//    once for the gate and the quantisation together.
//  - gate_fused_kernel (FP32 inputs, or shapes outside the tensor-core kernel's range): the
//    [kTok, E] logit tile is formed in shared memory on the CUDA cores, then each warp runs
//    the selection for its tokens with warp shuffles (lane l holds experts l, l+32, ...).
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "gemm_sched.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace moe {
namespace {

constexpr int kTok = 32;     // tokens per CTA
constexpr int kThreads = 256;
constexpr int kKStep = 32;   // H columns staged per step

template <typename T>
__device__ __forceinline__ float load_as_f32(const T* p, int64_t i);
template <>
__device__ __forceinline__ float load_as_f32<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_as_f32<uint16_t>(const uint16_t* p, int64_t i) {
    return bf16_bits_to_f32(p[i]);
}

// (value, index) arg-max with ties to the lower index.
__device__ __forceinline__ bool better(float v, int i, float ov, int oi) {
    return v > ov || (v == ov && i < oi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, o);
        int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(ov, oi, v, i)) { v = ov; i = oi; }
    }
}

// Merge the two largest values of (a1 >= a2) and (b1 >= b2).
__device__ __forceinline__ void top2_merge(float& a1, float& a2, float b1, float b2) {
    if (b1 > a1) {
        a2 = fmaxf(a1, b2);
        a1 = b1;
    } else {
        a2 = fmaxf(a2, b1);
    }
}

// Selection for one token from its E logits in shared memory; runs on one full warp.
// kMaxEpl >= ceil(E / 32) experts per lane.
template <int kMaxEpl>
__device__ void select_token(const float* logit, int E, int G, int TG, int K, float rsf,
                             const float* __restrict__ bias, int64_t t,
                             int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                             int32_t* __restrict__ counts) {
    const int lane = threadIdx.x & 31;
    const int epl = (E + 31) / 32;
    const int gsz = E / G;
    float s[kMaxEpl], c[kMaxEpl];
#pragma unroll
    for (int j = 0; j < kMaxEpl; ++j) {
        int e = lane + 32 * j;
        s[j] = 0.f;
        c[j] = -INFINITY;
        if (j < epl && e < E) {
            float l = logit[e];
            s[j] = 1.0f / (1.0f + expf(-l));
            c[j] = s[j] + bias[e];
        }
    }
    // group scores: the two largest c of each group (lane g keeps group g's score)
    float my_gs = -INFINITY;
    for (int g = 0; g < G; ++g) {
        float a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
        for (int j = 0; j < kMaxEpl; ++j) {
            int e = lane + 32 * j;
            if (j < epl && e < E && e / gsz == g) top2_merge(a1, a2, c[j], -INFINITY);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float b1 = __shfl_xor_sync(0xffffffffu, a1, o);
            float b2 = __shfl_xor_sync(0xffffffffu, a2, o);
            top2_merge(a1, a2, b1, b2);
        }
        if (lane == g) my_gs = a1 + a2;
    }
    // keep topk_group groups: repeated warp arg-max over lanes < G, ties to lower index
    uint32_t kept = 0;
    for (int r = 0; r < TG; ++r) {
        float v = (lane < G && !((kept >> lane) & 1u)) ? my_gs : -INFINITY;
        int i = (lane < G && !((kept >> lane) & 1u)) ? lane : 0x7fffffff;
        warp_argmax(v, i);
        kept |= 1u << (i < G ? i : 0);  // a NaN score leaves no candidate: keep group 0
    }
    // top_k experts among the kept groups; experts of dropped groups are excluded
    uint32_t taken = 0;  // bit j: this lane's j-th expert already chosen
    float den = 0.f;
    float my_w = 0.f;
    int my_e = 0;
    for (int k = 0; k < K; ++k) {
        float v = -INFINITY;
        int i = 0x7fffffff;
        float sv = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxEpl; ++j) {
            int e = lane + 32 * j;
            if (j < epl && e < E && !((taken >> j) & 1u) && ((kept >> (e / gsz)) & 1u)) {
                if (better(c[j], e, v, i)) { v = c[j]; i = e; sv = s[j]; }
            }
        }
        float bv = v;
        int bi = i;
        warp_argmax(bv, bi);
        if (bi >= E) bi = 0;  // no candidate (NaN scores): fall back to expert 0, never out of range
        // the owner lane marks the expert and shares its un-biased score
        int owner = bi & 31;
        if (lane == owner) taken |= 1u << (bi >> 5);
        float sw = __shfl_sync(0xffffffffu, sv, owner);
        den = den + sw;
        if (lane == k) { my_w = sw; my_e = bi; }
    }
    if (K > 1) den = den + 1e-20f;
    if (lane < K) {
        float w = (K > 1) ? my_w / den : my_w;
        topk_idx[t * K + lane] = my_e;
        topk_w[t * K + lane] = w * rsf;
        atomicAdd(&counts[my_e], 1);
    }
}

template <typename T, int kMaxEpl>
__global__ void __launch_bounds__(kThreads)
gate_fused_kernel(int64_t Tn, int H, int E, int G, int TG, int K, float rsf,
                  const T* __restrict__ x, const T* __restrict__ Wg,
                  const float* __restrict__ bias, int32_t* __restrict__ topk_idx,
                  float* __restrict__ topk_w, int32_t* __restrict__ counts) {
    constexpr int kNj = kMaxEpl >= 2 ? kMaxEpl / 2 : 1;  // >= ceil(E / 64)
    extern __shared__ float smem[];
    const int xstride = kTok + 1, wstride = E + 1;  // padded against bank conflicts
    float* xs = smem;                        // [kKStep][kTok + 1]
    float* ws = xs + kKStep * xstride;       // [kKStep][E + 1]
    float* logits = ws + kKStep * wstride;   // [kTok][E]
    const int tid = threadIdx.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
    const int tx = tid % 64, ty = tid / 64;  // experts tx + 64j, tokens ty*8 .. ty*8+7
    float acc[8][kNj];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int j = 0; j < kNj; ++j) acc[a][j] = 0.f;

    for (int h0 = 0; h0 < H; h0 += kKStep) {
        for (int i = tid; i < kTok * kKStep; i += kThreads) {
            int tt = i / kKStep, kk = i % kKStep;
            int64_t t = t0 + tt;
            xs[kk * xstride + tt] = (t < Tn) ? load_as_f32(x, t * H + h0 + kk) : 0.f;
        }
        for (int i = tid; i < E * kKStep; i += kThreads) {
            int e = i / kKStep, kk = i % kKStep;
            ws[kk * wstride + e] = load_as_f32(Wg, static_cast<int64_t>(e) * H + h0 + kk);
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kKStep; ++kk) {
            float xv[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) xv[a] = xs[kk * xstride + ty * 8 + a];
#pragma unroll
            for (int j = 0; j < kNj; ++j) {
                int e = tx + 64 * j;
                if (e < E) {
                    float wv = ws[kk * wstride + e];
#pragma unroll
                    for (int a = 0; a < 8; ++a) acc[a][j] = fmaf(xv[a], wv, acc[a][j]);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < kNj; ++j) {
        int e = tx + 64 * j;
        if (e < E)
#pragma unroll
            for (int a = 0; a < 8; ++a) logits[(ty * 8 + a) * E + e] = acc[a][j];
    }
    __syncthreads();
    const int warp = tid / 32;
    for (int tt = warp; tt < kTok; tt += kThreads / 32) {
        int64_t t = t0 + tt;
        if (t < Tn) select_token<kMaxEpl>(logits + tt * E, E, G, TG, K, rsf, bias, t, topk_idx, topk_w, counts);
    }
}


// ------------------------------------------------------------------------------------------
// tensor-core gate
// ------------------------------------------------------------------------------------------
constexpr int kGtM = 128;           // tokens per CTA (MMA M)
constexpr int kGtK = 64;            // BF16 columns per stage (128 bytes: one swizzle row)
constexpr int kGtStages = 4;
constexpr int kGtThreads = 512;     // warp 0 TMA, warp 1 MMA + TMEM; all 16 warps select
constexpr int kGtParts = kGtThreads / 128;  // threads per token in pass 1
constexpr int kGtMaxE = 256;
constexpr int kGtMaxK = 8;
constexpr int kGtMaxG = 8;
constexpr int kGtABytes = kGtM * kGtK * 2;       // 16 KB
constexpr int kGtBBytes = kGtMaxE * kGtK * 2;    // 32 KB (E rows)
constexpr int kGtStageBytes = kGtABytes + kGtBBytes;
constexpr int kGqStageBytes = 32 * 128;    // one quantising warp's 32 rows x 128 codes
constexpr int kGqOff = kGtStages * kGtStageBytes + 4096;  // 1024-aligned: the TMA store swizzle
constexpr int kGqRedOff = kGqOff + 4 * kGqStageBytes;    // [2][128] partial amax of the two halves
constexpr int kGtSmem = kGqRedOff + 2 * 128 * 4 + 1024;
constexpr long long kGtWaitBudget = 4000000000LL;
constexpr int kGqWarp0 = 4;         // warps 4..11 quantise x: two threads per token row, one per
constexpr int kGqWarps = 8;         // 64-column half of each 128-column block
constexpr int kGqBar = 1;           // their named barrier

__device__ int g_gate_error = 0;

struct GateTcParams {
    int64_t T;
    int H, E, G, TG, K;
    float rsf;
    const float* bias;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    uint8_t* xq;      // [T, H] E4M3 codes, or nullptr (no quantisation)
    float* xs;        // [T, H / 128] scales
    int pow2;         // scales amax / 448 (0) or the power-of-two rule (1)
};

// Eight BF16 values (one 16-byte chunk) -> eight E4M3 codes, as quant_1x128_kernel codes them.
template <bool kPow2>
__device__ __forceinline__ uint2 code8(uint4 c, float mul, int e) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t p[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float f0 = __uint_as_float(w[k] << 16), f1 = __uint_as_float(w[k] & 0xffff0000u);
        p[k] = kPow2 ? f32x2_to_e4m3x2(scale_pow2(f0, e), scale_pow2(f1, e))
                     : f32x2_to_e4m3x2(__fmul_rn(f0, mul), __fmul_rn(f1, mul));
    }
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// Lane-wise maximum of two pairs of BF16 values (a NaN lane yields the other operand's lane,
// as fmaxf does).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// max |v| over one thread's 64 BF16 values (8 chunks of 8), four independent chains.  The
// maximum is taken on the packed values with their sign bits cleared (a maximum of BF16 values
// is one of them, so it equals the FP32 maximum of the widened values), two values per
// instruction, and only the last pair is widened.
__device__ __forceinline__ float amax64(const uint4 (&c)[8]) {
    constexpr uint32_t kAbs = 0x7fff7fffu;
    uint32_t m[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        m[0] = bf16x2_max(m[0], c[j].x & kAbs);
        m[1] = bf16x2_max(m[1], c[j].y & kAbs);
        m[2] = bf16x2_max(m[2], c[j].z & kAbs);
        m[3] = bf16x2_max(m[3], c[j].w & kAbs);
    }
    const uint32_t v = bf16x2_max(bf16x2_max(m[0], m[1]), bf16x2_max(m[2], m[3]));
    return fmaxf(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// sigmoid with the fast exponential and division intrinsics (a few ulp in FP32; the selection
// is compared with the exact scores only where its margin exceeds 1e-5, and the weights within
// 2e-5 of the routing scale).  x -> -inf gives 0, x -> +inf gives 1.
// An unsigned key whose order is the order of the floats (negative values bit-inverted,
// positive ones with the sign bit set); 0 is below every float's key except -NaN patterns.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__global__ void __launch_bounds__(kGtThreads, 1)
gate_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               const __grid_constant__ CUtensorMap tmQ, const GateTcParams p) {
    using namespace sm100;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGtStages * kGtStageBytes);
    uint64_t* empty = full + kGtStages;
    uint64_t* acc_full = empty + kGtStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;
    float* sbias = reinterpret_cast<float*>(tmem_slot + 4);        // [E]
    int* shist = reinterpret_cast<int*>(sbias + kGtMaxE);           // [E]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int nk = p.H / kGtK;
    const uint32_t tmem_cols = 256;
    const bool quant = p.xq != nullptr;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGtStages; ++s) {
            mbar_init(&full[s], 1);
            // the MMA commit, and the four quantising warps of the half the stage holds
            mbar_init(&empty[s], 1 + (quant ? kGqWarps / 2 : 0));
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
    }
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        sbias[e] = p.bias[e];
        shist[e] = 0;
    }
    if (warp == 1) tmem_alloc(tmem_slot, tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kGtM;
    // CTAs start their K sweep at different 64-column chunks so that concurrent loads of x
    // (128 B from each of 128 rows) spread over the memory channels instead of all CTAs
    // hitting the same column offsets at once.  The start is even, so that the two halves of
    // each 128-column block arrive in consecutive stages (H % 128 == 0 when quantising).
    // The sum order is fixed per CTA.
    const int kc0 = 2 * static_cast<int>((static_cast<int64_t>(blockIdx.x) * 37) % (nk / 2 > 0 ? nk / 2 : 1)) % nk;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmW);
            const uint32_t bytes = kGtABytes + p.E * kGtK * 2;
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            for (int it = 0; it < nk; ++it) {
                const int kc = (it + kc0) % nk;
                if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, kGtWaitBudget)) {
                    *abort_flag = 1;
                    atomicCAS(&g_gate_error, 0, 0x201);
                    break;
                }
                uint8_t* sa = smem + s * kGtStageBytes;
                mbar_arrive_expect_tx(&full[s], bytes);
                tma_load_2d(sa, &tmX, &full[s], kc * kGtK, static_cast<int32_t>(t0));
                tma_load_2d(sa + kGtABytes, &tmW, &full[s], kc * kGtK, 0);
                ++issued;
                if (++s == kGtStages) { s = 0; ph ^= 1u; }
            }
            for (int i = 0; i < kGtStages && i < issued; ++i) {
                if (--s < 0) { s = kGtStages - 1; ph ^= 1u; }
                mbar_wait(&full[s], ph, never, kGtWaitBudget);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kGtM, p.E);
            int s = 0;
            uint32_t ph = 0;
            for (int it = 0; it < nk; ++it) {
                if (!mbar_wait(&full[s], ph, abort_flag, kGtWaitBudget)) {
                    *abort_flag = 1;
                    atomicCAS(&g_gate_error, 0, 0x202);
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + s * kGtStageBytes);
                const uint32_t b_addr = a_addr + kGtABytes;
#pragma unroll
                for (int k = 0; k < kGtK / 16; ++k)
                    mma_bf16(tmem_base, umma_desc_sw128(a_addr + k * 32), umma_desc_sw128(b_addr + k * 32),
                             idesc, (it > 0 || k > 0) ? 1u : 0u);
                mma_commit(&empty[s]);
                if (++s == kGtStages) { s = 0; ph ^= 1u; }
            }
            mma_commit(acc_full);  // fires when every MMA above has completed
        }
    } else if (quant && warp >= kGqWarp0 && warp < kGqWarp0 + kGqWarps) {
        // 1x128 quantisation of x from the operand ring.  Even stages hold the first 64 columns
        // of a 128-column block and odd stages the rest; thread (half, r) owns half `half` of
        // token row r of the tile.  Per block: each thread loads its 64 values from its stage
        // (128-byte swizzle: 16-byte chunk j of row r at chunk position j ^ (r % 8)) and
        // releases the stage, the two halves exchange their amax, and each codes its half
        // exactly as quant_1x128_kernel does into a per-row-quarter staging box [32 rows][128 B]
        // (the same swizzle) that one lane sends out by a TMA store, which clips the rows past
        // T; the scales are stored directly.
        const int half = (warp - kGqWarp0) / 4, quarter = warp & 3;
        const int r = quarter * 32 + lane, r7 = r & 7;
        const int64_t t = t0 + r;
        const int nb = p.H / 128;
        uint8_t* stg = smem + kGqOff + quarter * kGqStageBytes + lane * 128;
        float* red = reinterpret_cast<float*>(smem + kGqRedOff);  // [2][128]
        const bool issuer = half == 0 && lane == 0;
        bool ok = true;
        int kb = kc0 / 2;                        // the 128-column block of this iteration (kc0 is even)
        for (int it = half; it < nk; it += 2) {  // this thread's stage: it % kGtStages, parity (it / kGtStages) & 1
            const int s = it % kGtStages;
            const uint32_t ph = (it / kGtStages) & 1u;
            ok = ok && mbar_wait(&full[s], ph, abort_flag, kGtWaitBudget);
            uint4 c[8];
            const uint8_t* row = smem + s * kGtStageBytes + r * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = *reinterpret_cast<const uint4*>(row + ((j ^ r7) << 4));
            red[half * 128 + r] = amax64(c);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
            if (issuer) sched::tma_store_wait_read();  // the previous box has left the staging
            named_bar_sync(kGqBar, kGqWarps * 32);     // both halves' amax; the staging is free
            const float amax = fmaxf(red[r], red[128 + r]);
            if (amax == 0.f) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(stg + (((half * 4 + j) ^ r7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            } else if (p.pow2) {
                const int e = pow2_exponent(amax);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint2 a = code8<true>(c[2 * j], 0.f, e), b = code8<true>(c[2 * j + 1], 0.f, e);
                    *reinterpret_cast<uint4*>(stg + (((half * 4 + j) ^ r7) << 4)) = make_uint4(a.x, a.y, b.x, b.y);
                }
            } else {
                const float mul = __fdiv_rn(448.f, amax);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint2 a = code8<false>(c[2 * j], mul, 0), b = code8<false>(c[2 * j + 1], mul, 0);
                    *reinterpret_cast<uint4*>(stg + (((half * 4 + j) ^ r7) << 4)) = make_uint4(a.x, a.y, b.x, b.y);
                }
            }
            sched::fence_proxy_async_smem();
            named_bar_sync(kGqBar, kGqWarps * 32);     // the box's rows are complete
            if (half == 0) {
                if (lane == 0)
                    sched::tma_store_2d(&tmQ, smem + kGqOff + quarter * kGqStageBytes, kb * 128,
                                        static_cast<int32_t>(t0 + quarter * 32));
                if (t < p.T) {
                    const int e = pow2_exponent(amax);
                    p.xs[t * nb + kb] = amax == 0.f ? 1.f : (p.pow2 ? exp2_int(e) : __fdiv_rn(amax, 448.f));
                }
            }
            if (++kb == nb) kb = 0;
        }
        if (issuer) sched::tma_store_wait_all();  // every code has reached global memory
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicCAS(&g_gate_error, 0, 0x204);
        }
    }
    __syncwarp();  // the producer and MMA lanes rejoin their warps
    // ------------------------------------------------------------------ selection, all warps
    // Pass 1, one thread per (token, part of its groups): warp w reads TMEM lanes 32*(w % 4)..
    // (its tokens) and computes the group scores of part w / 4 of the groups, storing them and
    // the logits in the operand ring, idle once every MMA has completed.
    {
        const int quarter = warp & 3, h = warp >> 2;  // h: which part of the token's groups
        const int tl = quarter * 32 + lane;
        bool ok = mbar_wait(acc_full, 0, abort_flag, kGtWaitBudget);
        ok = __all_sync(0xffffffffu, ok);  // TMEM loads below are warp-collective
        tc_fence_after();
        __syncthreads();  // the quantising warps have read the last stages: the ring is free
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicCAS(&g_gate_error, 0, 0x203);
        }
        float* gsc = reinterpret_cast<float*>(smem);          // [kGtM][kGtMaxG] group scores
        float* lg = gsc + kGtM * kGtMaxG;                      // [kGtM][E + 1] logits (padded row)
        const int lgs = p.E + 1;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const int gsz = p.E / p.G;   // a multiple of 32: each 32-column chunk lies in one group
        const int cpg = gsz / 32;
        const int gper = (p.G + kGtParts - 1) / kGtParts;
        const int g_lo = min(h * gper, p.G), g_hi = min(g_lo + gper, p.G);
        // pass 1: group score = sum of the two largest selection scores of the group
        for (int g = g_lo; g < g_hi && ok; ++g) {
            float a1 = -INFINITY, a2 = -INFINITY;
            for (int cc = 0; cc < cpg; ++cc) {
                float l[32];
                tmem_ld32(taddr + (g * cpg + cc) * 32, l);
                tmem_ld_wait_regs(l);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float c = sigmoid_fast(l[j]) + sbias[(g * cpg + cc) * 32 + j];
                    if (c > a1) { a2 = a1; a1 = c; } else if (c > a2) { a2 = c; }
                    lg[tl * lgs + (g * cpg + cc) * 32 + j] = l[j];  // (tl + e) % 32 banks: no conflicts
                }
            }
            gsc[tl * kGtMaxG + g] = a1 + a2;
        }
        __syncthreads();
        // kept groups (topk_group by group score, ties to the lower index) and the slots they
        // cover, once per token: slot j of a lane holds expert lane + 32 j, in group j / cpg
        uint32_t* kmask = reinterpret_cast<uint32_t*>(lg + kGtM * lgs);  // [kGtM]
        const int epl = p.E / 32;
        if (threadIdx.x < kGtM) {
            const int tok = threadIdx.x;
            uint32_t kept = 0;
            for (int r = 0; r < p.TG; ++r) {
                int best = -1;
                float bv = -INFINITY;
                for (int g = 0; g < p.G; ++g) {
                    const float v = gsc[tok * kGtMaxG + g];
                    if (!((kept >> g) & 1u) && (best < 0 || v > bv)) { best = g; bv = v; }
                }
                kept |= 1u << (best < 0 ? 0 : best);
            }
            uint32_t skept = 0;
            for (int j = 0; j < epl; ++j)
                if ((kept >> (j / cpg)) & 1u) skept |= 1u << j;
            kmask[tok] = skept;
        }
        __syncthreads();
        // pass 2, one warp per token (warp w takes tokens w, w + 16, ...): top_k rounds of a warp
        // arg-max over the kept experts' selection scores, ties to the lower expert index, slots
        // in descending score.  Each round: the lane-local best (slots in ascending index, so a
        // strict '>' keeps the lowest index among equals), the warp maximum of an
        // order-preserving integer key of the score, then the warp minimum of the index among
        // the lanes holding that maximum.  The un-biased scores are recomputed from the stored
        // logits with the same instructions as in pass 1.
        for (int tok = warp; tok < kGtM && ok; tok += kGtThreads / 32) {
            const int64_t tt = t0 + tok;
            if (tt >= p.T) break;
            const uint32_t skept = kmask[tok];
            float sv[kGtMaxE / 32], cv[kGtMaxE / 32];
#pragma unroll
            for (int j = 0; j < kGtMaxE / 32; ++j) {
                const int e = lane + 32 * j;
                cv[j] = -INFINITY;
                sv[j] = 0.f;
                if ((skept >> j) & 1u) {
                    sv[j] = sigmoid_fast(lg[tok * lgs + e]);
                    cv[j] = sv[j] + sbias[e];
                }
            }
            uint32_t avail = skept;  // kept slots not yet chosen
            float den = 0.f, my_w = 0.f;
            int my_e = 0;
            for (int k = 0; k < p.K; ++k) {
                float v = -INFINITY, s_best = 0.f;
                int jb = -1;
#pragma unroll
                for (int j = 0; j < kGtMaxE / 32; ++j)
                    if (((avail >> j) & 1u) && (jb < 0 || cv[j] > v)) { v = cv[j]; jb = j; s_best = sv[j]; }
                const uint32_t key = jb < 0 ? 0u : order_key(v + 0.0f);  // (-0 + 0 = +0: equal zeros, equal keys)
                const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
                int i = __reduce_min_sync(0xffffffffu, (jb >= 0 && key == kmax) ? lane + 32 * jb : 0x7fffffff);
                if (i >= p.E) i = 0;  // no candidate (NaN scores): expert 0, never out of range
                const int owner = i & 31;
                if (lane == owner) avail &= ~(1u << (i >> 5));
                const float sw = __shfl_sync(0xffffffffu, s_best, owner);
                den = den + sw;
                if (lane == k) { my_w = sw; my_e = i; }
            }
            if (p.K > 1) den = den + 1e-20f;
            if (lane < p.K) {
                const float w = (p.K > 1) ? my_w / den : my_w;
                p.topk_idx[tt * p.K + lane] = my_e;
                p.topk_w[tt * p.K + lane] = w * p.rsf;
                atomicAdd(&shist[my_e], 1);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x)
        if (shist[e]) atomicAdd(&p.counts[e], shist[e]);
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

bool gate_tc_supported(const moe_config& c) {
    const int E = c.n_experts, G = c.n_group;
    return c.mode != MOE_FP32 && E % 32 == 0 && E <= kGtMaxE && G <= kGtMaxG &&
           (E / G) % 32 == 0 && c.top_k <= kGtMaxK && c.hidden % kGtK == 0;
}

moe_status launch_gate_tc(const moe_config& c, int64_t T, const uint16_t* x, const uint16_t* Wg,
                          const float* bias, int32_t* idx, float* w, int32_t* counts, cudaStream_t s,
                          uint8_t* xq = nullptr, float* xs = nullptr) {
    CUtensorMap tmX, tmW, tmQ;
    if (!make_tma_map_2d(&tmX, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, c.hidden, kGtM, kGtK))
        return MOE_ERR_CUDA;
    if (xq && !make_tma_map_2d(&tmQ, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, T, c.hidden, 32, 128))
        return MOE_ERR_CUDA;
    if (!xq) tmQ = tmX;  // unused
    if (!make_tma_map_2d(&tmW, Wg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.n_experts, c.hidden, c.n_experts, kGtK))
        return MOE_ERR_CUDA;
    static PerDeviceOnce attr_once;
    MOE_CUDA_CHECK(once_per_device(attr_once, [] {
        return cudaFuncSetAttribute(gate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGtSmem);
    }));
    GateTcParams p{T, c.hidden, c.n_experts, c.n_group, c.topk_group, c.top_k, c.routed_scaling_factor,
                   bias, idx, w, counts, xq, xs, c.mode == MOE_MXFP8 ? 1 : 0};
    gate_tc_kernel<<<static_cast<unsigned>(ceil_div(T, kGtM)), kGtThreads, kGtSmem, s>>>(tmX, tmW, tmQ, p);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace

size_t gate_scratch_bytes(const moe_config&, int64_t) { return 0; }

moe_status gate_read_and_clear_error(int32_t* code) {
    int v = 0;
    MOE_CUDA_CHECK(cudaMemcpyFromSymbol(&v, g_gate_error, sizeof(int)));
    const int zero = 0;
    MOE_CUDA_CHECK(cudaMemcpyToSymbol(g_gate_error, &zero, sizeof(int)));
    *code = v;
    return MOE_OK;
}

template <typename T>
static moe_status launch_typed(const moe_config& c, int64_t T_, const T* x, const T* Wg,
                               const float* bias, int32_t* idx, float* w, int32_t* counts,
                               cudaStream_t s) {
    const int E = c.n_experts;
    size_t smem = sizeof(float) * (kKStep * (kTok + 1) + kKStep * (E + 1) + kTok * E);
    if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    void (*k)(int64_t, int, int, int, int, int, float, const T*, const T*, const float*,
              int32_t*, float*, int32_t*);
    if (E <= 32) k = gate_fused_kernel<T, 1>;
    else if (E <= 64) k = gate_fused_kernel<T, 2>;
    else if (E <= 128) k = gate_fused_kernel<T, 4>;
    else if (E <= 256) k = gate_fused_kernel<T, 8>;
    else if (E <= 512) k = gate_fused_kernel<T, 16>;
    else k = gate_fused_kernel<T, 32>;
    MOE_CUDA_CHECK(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    dim3 grid(static_cast<unsigned>(ceil_div(T_, kTok)));
    k<<<grid, kThreads, smem, s>>>(T_, c.hidden, E, c.n_group, c.topk_group, c.top_k,
                                   c.routed_scaling_factor, x, Wg, bias, idx, w, counts);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

moe_status launch_gate(const moe_config& c, int64_t T, const void* x, const void* Wg,
                       const float* bias, int32_t* idx, float* w, int32_t* counts,
                       float* /*logits_scratch*/, cudaStream_t s) {
    MOE_CUDA_CHECK(cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.n_experts, s));
    if (T == 0) return MOE_OK;
    if (c.mode == MOE_FP32)
        return launch_typed(c, T, static_cast<const float*>(x), static_cast<const float*>(Wg),
                            bias, idx, w, counts, s);
    if (gate_tc_supported(c) && aligned16(x) && aligned16(Wg))
        return launch_gate_tc(c, T, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(Wg),
                              bias, idx, w, counts, s);
    return launch_typed(c, T, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(Wg),
                        bias, idx, w, counts, s);
}

bool gate_quant_supported(const moe_config& c) {
    return gate_tc_supported(c) && c.hidden % 128 == 0;
}

moe_status launch_gate_quant(const moe_config& c, int64_t T, const void* x, const void* Wg,
                             const float* bias, int32_t* idx, float* w, int32_t* counts,
                             uint8_t* xq, float* xs, cudaStream_t s) {
    if (!gate_quant_supported(c) || !aligned16(x) || !aligned16(Wg) || !aligned16(xq))
        return MOE_ERR_UNSUPPORTED;
    MOE_CUDA_CHECK(cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.n_experts, s));
    if (T == 0) return MOE_OK;
    return launch_gate_tc(c, T, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(Wg),
                          bias, idx, w, counts, s, xq, xs);
}

}  // namespace moe
