// gate.cu -- a1: the sigmoid MoEGate with group-limited top-k and the fused per-expert
// histogram.
//
// DeepSeek-V3 co-design teardown (wsisp.com) §2.2, MoEGate listing: logits in FP32,
// sigmoid scores, selection-only bias, group score = sum of the two best selection scores
// of the group, keep topk_group groups, top_k experts among them, weights from the
// un-biased scores, normalised (top_k > 1) and scaled; §2.3: per-expert token counts.
//
// One CTA handles kTok tokens against all E experts: the [kTok, E] logit tile is formed in
// shared memory (FP32 accumulation over H), then each warp runs the selection for its
// tokens with warp shuffles (lane l holds experts l, l+32, ...).
#include "common.cuh"
#include "internal.h"

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

}  // namespace

size_t gate_scratch_bytes(const moe_config&, int64_t) { return 0; }

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
    return launch_typed(c, T, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(Wg),
                        bias, idx, w, counts, s);
}

}  // namespace moe
