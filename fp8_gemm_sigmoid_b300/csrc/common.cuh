// common.cuh -- device helpers shared by the libmoe kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "../../include/moe.h"

#define MOE_CUDA_CHECK(expr)                                                    \
    do {                                                                        \
        cudaError_t _e = (expr);                                                \
        if (_e != cudaSuccess) return MOE_ERR_CUDA;                             \
    } while (0)

#define MOE_LAUNCH_CHECK()                                                      \
    do {                                                                        \
        if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;             \
    } while (0)

#define MOE_TRY(expr)                                                           \
    do {                                                                        \
        moe_status _s = (expr);                                                 \
        if (_s != MOE_OK) return _s;                                            \
    } while (0)

// Device-side checks of the MOE_CHECKS build (a stand-in for a memory checker): a failed check
// records its code in the translation unit's check word (the first failure wins) and the
// caller skips the access instead of making it.  The default build compiles them away.
#ifdef MOE_CHECKS
#define MOE_DCHECK(word, cond, code) ((cond) ? true : (atomicCAS(&(word), 0, (code)), false))
#else
#define MOE_DCHECK(word, cond, code) (true)
#endif

namespace moe {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Reads a device word of this translation unit (an error or check word) and clears it.
template <typename T>
inline cudaError_t read_and_clear_word(const T& symbol, int32_t* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, symbol, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(symbol, &zero, sizeof(int));
    *code = v;
    return e;
}

// Host-side set-up that must run once on each device a process uses (kernel attributes such
// as the dynamic shared-memory limit are per device).  Each call site owns one instance.
struct PerDeviceOnce {
    static constexpr int kMaxDevices = 64;
    std::mutex mu;
    bool done[kMaxDevices] = {};
    cudaError_t err[kMaxDevices] = {};
};

// Runs f() on the current device the first time this call site sees that device, and returns
// its result then and on every later call there.
template <typename F>
cudaError_t once_per_device(PerDeviceOnce& o, F&& f) {
    int dev = -1;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= PerDeviceOnce::kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(o.mu);
    if (!o.done[dev]) {
        o.err[dev] = f();
        o.done[dev] = true;
    }
    return o.err[dev];
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// BF16 <-> FP32 (the BF16 bits are the upper half of the FP32 bits).
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Two FP32 -> two OCP E4M3 codes, round-to-nearest-even with saturation to +-448
// (PTX cvt.rn.satfinite.e4m3x2.f32: the first source lands in the upper byte).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// OCP E4M3 code -> FP32 from the format's fields: bias 7, exponent field 0 = subnormal
// m * 2^-9.  (Codes S.1111.111 are NaN; the quantiser never produces them.)
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    uint32_t s = (c & 0x80u) << 24, e = (c >> 3) & 15u, m = c & 7u;
    float mag = (e == 0) ? static_cast<float>(m) * 0x1p-9f
                         : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return __uint_as_float(__float_as_uint(mag) | s);
}

// Power-of-two block scales (the 8-bit exponent scales of microscaling): for a tile with
// amax > 0 the exponent is the smallest e with 448 * 2^e >= amax.  With amax = m * 2^E,
// m in [1, 2), and 448 = 1.75 * 2^8 that is E - 8 when m <= 1.75 and E - 7 otherwise; a
// subnormal amax (below 2^-126) gives the floor -127.  Clamped to [-127, 127].
__device__ __forceinline__ int pow2_exponent(float amax) {
    if (amax < 1.17549435e-38f) return -127;
    const uint32_t u = __float_as_uint(amax);
    const int E = static_cast<int>((u >> 23) & 0xffu) - 127;
    const int e = E - 8 + ((u & 0x7fffffu) > 0x600000u ? 1 : 0);  // significand above 1.75
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^e as an FP32 value for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2_int(int e) {
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// v * 2^-e for e in [-127, 127]: two exact power-of-two factors, so the product is exact
// whenever it is a normal FP32 value.
__device__ __forceinline__ float scale_pow2(float v, int e) {
    const int h = -e / 2;
    return (v * exp2_int(h)) * exp2_int(-e - h);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace moe
