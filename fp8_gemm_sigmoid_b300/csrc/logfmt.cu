// logfmt.cu -- LogFMT-nBit, the logarithmic code for 1x128 tiles of the combine payload
// (Insights into DeepSeek-V3 précis §3.2, LogFMT communication compression): per tile the
// natural logs of the non-zero magnitudes give min and max (min held above max - ln 2^32),
// Step = (max - min) / (2^(n-1) - 2); a value is coded with the K >= 1 whose
// exp(min + Step (K - 1)) is nearest to it in linear space (K = 0: nearer to zero than to
// exp(min)); the sign is the code's top bit.  Tile metadata: min and Step as FP32.
//
// Encoding decides K with one base-2 logarithm per value, relative to the tile's first grid
// point g1 = e^min: with r = log2(a / g1) / Step2 (Step2 = Step / ln 2) the value lies between
// the grid points floor(r) + 1 and floor(r) + 2, and the linear midpoint of two neighbours is
// at the fraction theta = log2((1 + 2^Step2) / 2) / Step2 of the way between them in log
// space (the same for every pair of the tile), so K = floor(r) + 1 + (frac(r) >= theta);
// below g1 the midpoint with zero is at r = -1 / Step2.  Logarithms are the hardware base-2
// approximation (absolute error near 2^-22; per tile, for the min and max, as the exponent
// plus the log2 of the significand so that subnormal magnitudes are covered), so r is within
// about 1e-4 of a step for n <= 12 (the step shrinks as 2^-(n-1)).  Decoding forms
// 2^(Step2 (K - 1)) from the hardware exponential of the rounded product and the FMA residual
// of the product, times g1 = e^min computed once per tile, a few 1e-7 off the exact value
// before its rounding to BF16.
// Eight lanes per tile, 16 values per lane (two 16-byte BF16 loads), so the tile's reductions
// take three shuffle steps and its per-tile arithmetic is shared by 16 values; each lane takes
// kTilesPerLane tiles per step with every load issued first.  2 bytes read and 1 (n <= 8) or
// 2 bytes written per value.
#include "common.cuh"

namespace moe {
namespace {

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;
constexpr float kLog2eLo = 1.925963033500011e-08f;  // log2(e) - kLog2e
constexpr int kLanesPerTile = 8;
constexpr int kTilesPerLane = 2;   // tiles per lane and step, loaded together
constexpr int kTilesPerWarpStep = (32 / kLanesPerTile) * kTilesPerLane;

// max / min over the eight lanes of a tile group (lanes 8g .. 8g + 7)
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = kLanesPerTile / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float group_min(float v) {
#pragma unroll
    for (int o = kLanesPerTile / 2; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) for finite x > 0 (subnormals included): exponent + log2(significand in [1, 2)).
__device__ __forceinline__ float log2_split(float x) {
    int bias = 127;
    if (x < 1.17549435e-38f) {  // subnormal: scale into the normal range first
        x *= 18446744073709551616.f;  // 2^64
        bias += 64;
    }
    const uint32_t u = __float_as_uint(x);
    const int e = static_cast<int>((u >> 23) & 0xffu) - bias;
    const float m = __uint_as_float((u & 0x007fffffu) | 0x3f800000u);
    return static_cast<float>(e) + __log2f(m);
}

template <typename CodeT>
__global__ void __launch_bounds__(256)
logfmt_encode_kernel(int64_t n_tiles, int64_t tiles_per_row, int64_t cols, int n_bits,
                     const uint4* __restrict__ x, CodeT* __restrict__ codes,
                     float* __restrict__ lmin_out, float* __restrict__ step_out) {
    const int lane = threadIdx.x & 31, grp = lane / kLanesPerTile, sub = lane % kLanesPerTile;
    const int kmax = (1 << (n_bits - 1)) - 1;
    const uint32_t sign_bit = 1u << (n_bits - 1);
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t t0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) * kTilesPerWarpStep;
         t0 < n_tiles; t0 += nwarps * kTilesPerWarpStep) {
      uint4 raws[kTilesPerLane][2];
#pragma unroll
      for (int j = 0; j < kTilesPerLane; ++j) {  // every load of the step first
        int64_t t = t0 + j * (32 / kLanesPerTile) + grp;
        t = t < n_tiles ? t : t0;
        const int64_t e0 = (t / tiles_per_row) * cols + (t % tiles_per_row) * 128 + sub * 16;  // element
        raws[j][0] = x[e0 / 8];
        raws[j][1] = x[e0 / 8 + 1];
      }
#pragma unroll
      for (int j = 0; j < kTilesPerLane; ++j) {
        const int64_t t = t0 + j * (32 / kLanesPerTile) + grp;
        const int64_t e0 = (t / tiles_per_row) * cols + (t % tiles_per_row) * 128 + sub * 16;
        const uint32_t w[8] = {raws[j][0].x, raws[j][0].y, raws[j][0].z, raws[j][0].w,
                               raws[j][1].x, raws[j][1].y, raws[j][1].z, raws[j][1].w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
        float amax = 0.f, amin = INFINITY;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float a = fabsf(v[i]);
            amax = fmaxf(amax, a);
            if (a > 0.f) amin = fminf(amin, a);
        }
        amax = group_max(amax);
        amin = group_min(amin);
        float step2 = 0.f, l2min = 0.f;
        bool held = false;  // min raised to max - ln 2^32: values below g1 exist
        if (amax > 0.f) {
            const float l2max = log2_split(amax);
            const float full_span = l2max - log2_split(amin);
            held = full_span > 32.f;
            const float span2 = fminf(full_span, 32.f);  // max - min held <= log2 2^32
            l2min = l2max - span2;
            step2 = __fdividef(span2, static_cast<float>(kmax - 1));
        }
        uint32_t c[16];
        if (step2 > 0.f) {
            const float inv = __fdividef(1.f, step2);
            const float theta = log2_split(0.5f + 0.5f * ex2_approx(step2)) * inv;  // linear midpoint, in steps
            const float zero_cut = -inv;
            const bool tiny = l2min < -100.f;
            if (!tiny) {
                // u = r - theta with r = log2(a / g1) / Step2, 0 at g1: a * anchor is a normal
                // number (the hardware logarithm, absolute error near 2^-22, far below the
                // decision margins); a = 0 gives u = -inf and K = 0.  For r >= 0 the code is
                // floor(r) + 1, plus 1 from the fraction theta on: floor(u) + 2.
                // Unless the min was held, every non-zero value lies at or above g1 (u at least
                // -theta, up to the logarithm's error, so floor(u) + 2 >= 1), and zeros give
                // u = -inf: K = floor(u) + 2 clamped to [0, kmax] covers every value.
                const float anchor = ex2_approx(-l2min);
                if (!held) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float u = fmaf(lg2_approx(fabsf(v[i]) * anchor), inv, -theta);
                        const int K = min(max(__float2int_rd(u) + 2, 0), kmax);
                        c[i] = static_cast<uint32_t>(K) | ((__float_as_uint(v[i]) >> (32 - n_bits)) & sign_bit);
                    }
                } else {  // values below g1: K = 1 down to the linear midpoint with zero, else 0
                    const float cut1 = zero_cut - theta;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float u = fmaf(lg2_approx(fabsf(v[i]) * anchor), inv, -theta);
                        const int K = u >= -theta ? min(__float2int_rd(u) + 2, kmax) : (u >= cut1 ? 1 : 0);
                        c[i] = static_cast<uint32_t>(K) | ((__float_as_uint(v[i]) >> (32 - n_bits)) & sign_bit);
                    }
                }
            } else {
                // g1 so low (tiles of subnormal BF16 values) that 1 / g1 would overflow: the
                // logarithm is taken first and g1's subtracted (a rare, slower and slightly less
                // precise path)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a = fabsf(v[i]);
                    int K = 0;
                    if (a > 0.f) {
                        const float r = (log2_split(a) - l2min) * inv;
                        K = r < 0.f ? (r >= zero_cut ? 1 : 0) : min(__float2int_rd(r - theta) + 2, kmax);
                    }
                    c[i] = static_cast<uint32_t>(K) | (signbit(v[i]) ? sign_bit : 0u);
                }
            }
        } else {  // all zero (K = 0), or one magnitude (K = 1)
#pragma unroll
            for (int i = 0; i < 16; ++i)
                c[i] = (fabsf(v[i]) > 0.f ? 1u : 0u) | (signbit(v[i]) ? sign_bit : 0u);
        }
        if (t < n_tiles) {
            if (sizeof(CodeT) == 1) {
                uint32_t q[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)  // bytes c0 c1 c2 c3
                    q[k] = __byte_perm(__byte_perm(c[4 * k], c[4 * k + 1], 0x0040),
                                       __byte_perm(c[4 * k + 2], c[4 * k + 3], 0x0040), 0x5410);
                *reinterpret_cast<uint4*>(codes + e0) = make_uint4(q[0], q[1], q[2], q[3]);
            } else {
                uint32_t q[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) q[k] = __byte_perm(c[2 * k], c[2 * k + 1], 0x5410);
                *reinterpret_cast<uint4*>(codes + e0) = make_uint4(q[0], q[1], q[2], q[3]);
                *reinterpret_cast<uint4*>(codes + e0 + 8) = make_uint4(q[4], q[5], q[6], q[7]);
            }
            if (sub == 0) {
                lmin_out[t] = l2min * kLn2;
                step_out[t] = step2 * kLn2;
            }
        }
      }
    }
}

template <typename CodeT>
__global__ void __launch_bounds__(256)
logfmt_decode_kernel(int64_t n_tiles, int64_t tiles_per_row, int64_t cols, int n_bits,
                     const CodeT* __restrict__ codes, const float* __restrict__ lmin,
                     const float* __restrict__ step, uint4* __restrict__ y) {
    const int lane = threadIdx.x & 31, grp = lane / kLanesPerTile, sub = lane % kLanesPerTile;
    const uint32_t kmask = (1u << (n_bits - 1)) - 1u;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t t0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) * kTilesPerWarpStep;
         t0 < n_tiles; t0 += nwarps * kTilesPerWarpStep) {
      uint4 raws[kTilesPerLane][2];
      float lms[kTilesPerLane], sts[kTilesPerLane];
#pragma unroll
      for (int j = 0; j < kTilesPerLane; ++j) {  // every load of the step in flight together
        int64_t t = t0 + j * (32 / kLanesPerTile) + grp;
        t = t < n_tiles ? t : t0;
        const int64_t e0 = (t / tiles_per_row) * cols + (t % tiles_per_row) * 128 + sub * 16;
        raws[j][0] = *reinterpret_cast<const uint4*>(codes + e0);
        raws[j][1] = sizeof(CodeT) == 1 ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(codes + e0 + 8);
        lms[j] = lmin[t];
        sts[j] = step[t];
      }
#pragma unroll
      for (int j = 0; j < kTilesPerLane; ++j) {
        const int64_t t = t0 + j * (32 / kLanesPerTile) + grp;
        if (t >= n_tiles) continue;
        const int64_t e0 = (t / tiles_per_row) * cols + (t % tiles_per_row) * 128 + sub * 16;
        uint32_t c[16];
        if (sizeof(CodeT) == 1) {
            const uint32_t w[4] = {raws[j][0].x, raws[j][0].y, raws[j][0].z, raws[j][0].w};
#pragma unroll
            for (int i = 0; i < 16; ++i) c[i] = (w[i / 4] >> (8 * (i % 4))) & 0xffu;
        } else {
            const uint32_t w[8] = {raws[j][0].x, raws[j][0].y, raws[j][0].z, raws[j][0].w,
                                   raws[j][1].x, raws[j][1].y, raws[j][1].z, raws[j][1].w};
#pragma unroll
            for (int i = 0; i < 16; ++i) c[i] = (w[i / 2] >> (16 * (i % 2))) & 0xffffu;
        }
        // g1 = e^min once per tile; Step2 = Step * log2(e) as an exact pair (hi + lo)
        const float st = sts[j];
        const float g1 = expf(lms[j]);
        const float s_hi = st * kLog2e;
        const float s_lo = fmaf(st, kLog2e, -s_hi) + st * kLog2eLo;
        float m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float fK = static_cast<float>(c[i] & kmask);
            const float k = fK - 1.f;
            const float e_hi = s_hi * k;                        // 2^(Step2 k) = 2^e_hi * 2^e_lo
            const float e_lo = fmaf(s_lo, k, fmaf(s_hi, k, -e_hi));
            // 2^e_hi by the hardware exponential (exact range reduction, relative error near
            // 2^-22), e_hi in 0 .. 32 for metadata the encoder wrote; K = 0 gives 0 through the
            // factor min(K, 1), the sign bit is moved into place
            const float mag = g1 * (ex2_approx(e_hi) * fmaf(e_lo, kLn2, 1.f)) * fminf(fK, 1.f);
            m[i] = __uint_as_float(__float_as_uint(mag) | ((c[i] << (32 - n_bits)) & 0x80000000u));
        }
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // paired round-to-nearest-even BF16 conversion
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(m[2 * i], m[2 * i + 1]);
            o[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        y[e0 / 8] = make_uint4(o[0], o[1], o[2], o[3]);
        y[e0 / 8 + 1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
}

unsigned warp_grid(int64_t n_tiles) {
    const int64_t blocks = ceil_div(n_tiles, 8 * kTilesPerWarpStep);
    return static_cast<unsigned>(blocks < 148 * 16 ? blocks : 148 * 16);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_logfmt_encode(int32_t n_bits, int64_t rows, int64_t cols, const uint16_t* x,
                                        void* codes, float* lmin, float* step, moe_stream_t stream) {
    if (n_bits < 3 || n_bits > 12 || rows < 0 || cols <= 0 || cols % 128) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!x || !codes || !lmin || !step || !aligned16(x) || !aligned16(codes)) return MOE_ERR_INVALID_ARG;
    const int64_t tpr = cols / 128, n_tiles = rows * tpr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_bits <= 8)
        logfmt_encode_kernel<uint8_t><<<warp_grid(n_tiles), 256, 0, s>>>(
            n_tiles, tpr, cols, n_bits, reinterpret_cast<const uint4*>(x), static_cast<uint8_t*>(codes), lmin, step);
    else
        logfmt_encode_kernel<uint16_t><<<warp_grid(n_tiles), 256, 0, s>>>(
            n_tiles, tpr, cols, n_bits, reinterpret_cast<const uint4*>(x), static_cast<uint16_t*>(codes), lmin, step);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

extern "C" moe_status moe_logfmt_decode(int32_t n_bits, int64_t rows, int64_t cols, const void* codes,
                                        const float* lmin, const float* step, uint16_t* y,
                                        moe_stream_t stream) {
    if (n_bits < 3 || n_bits > 12 || rows < 0 || cols <= 0 || cols % 128) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!codes || !lmin || !step || !y || !aligned16(codes) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    const int64_t tpr = cols / 128, n_tiles = rows * tpr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_bits <= 8)
        logfmt_decode_kernel<uint8_t><<<warp_grid(n_tiles), 256, 0, s>>>(
            n_tiles, tpr, cols, n_bits, static_cast<const uint8_t*>(codes), lmin, step, reinterpret_cast<uint4*>(y));
    else
        logfmt_decode_kernel<uint16_t><<<warp_grid(n_tiles), 256, 0, s>>>(
            n_tiles, tpr, cols, n_bits, static_cast<const uint16_t*>(codes), lmin, step, reinterpret_cast<uint4*>(y));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}
