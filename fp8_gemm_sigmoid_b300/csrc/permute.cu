// permute.cu -- a3: token permutation by expert (DeepSeek-V3 co-design teardown, §2.3:
// per-expert counts, then the rows ordered by the argsort of the flat expert ids).
//
// The order is made deterministic and equal to a stable sort: rows are expert-major and,
// within an expert, in ascending token order.  No atomics decide a position:
//   1. chunk histogram: counts of each expert inside each chunk of kChunk tokens;
//   2. scan: offs = exclusive prefix of the counts; base[c][e] = offs[e] + rows of expert e
//      in chunks before c;
//   3. positions: inside a chunk, one thread per expert walks the chunk's tokens in order;
//   4. gather: each destination row copies its token's quantised row; the scales go to a
//      K-block-major [H/128, R] array, the layout the grouped GEMM reads.
// With a shared expert, group E follows with every token once, in order.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kChunk = 64;  // tokens per chunk

__global__ void __launch_bounds__(256)
chunk_hist_kernel(int64_t T, int K, int E, const int32_t* __restrict__ idx,
                  int32_t* __restrict__ chunk_cnt) {
    extern __shared__ int32_t hist[];  // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int64_t n = (T - t0 < kChunk ? T - t0 : kChunk) * K;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const int32_t e = idx[t0 * K + i];
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);  // ids outside [0, E) are dropped
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_cnt[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// One CTA.  Thread e totals expert e's column of chunk counts, an exclusive prefix over the
// totals gives offs, and a second pass over the column gives each chunk's base.  The rows
// are derived from topk_idx alone, so every position stays inside [0, T*K).
__global__ void __launch_bounds__(1024)
scan_kernel(int64_t T, int K, int E, int has_shared, int64_t n_chunks,
            const int32_t* __restrict__ chunk_cnt, int32_t* __restrict__ chunk_base,
            int32_t* __restrict__ offs) {
    __shared__ int32_t part[1024];
    const int e = threadIdx.x;
    int32_t v = 0;
    if (e < E) {
#pragma unroll 8
        for (int64_t c = 0; c < n_chunks; ++c) v += chunk_cnt[c * E + e];
    }
    part[e] = v;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {  // inclusive Hillis-Steele scan (E <= 1024)
        int32_t add = (e >= o) ? part[e - o] : 0;
        __syncthreads();
        part[e] += add;
        __syncthreads();
    }
    if (e < E) {
        const int32_t start = part[e] - v;
        offs[e] = start;
        int32_t run = start;
#pragma unroll 8
        for (int64_t c = 0; c < n_chunks; ++c) {
            chunk_base[c * E + e] = run;
            run += chunk_cnt[c * E + e];
        }
    }
    if (e == 0) {
        const int64_t routed = T * K;
        offs[E] = static_cast<int32_t>(routed);
        if (has_shared) offs[E + 1] = static_cast<int32_t>(routed + T);
    }
}

// One CTA per chunk; thread e walks the chunk's tokens in order.
__global__ void __launch_bounds__(256)
positions_kernel(int64_t T, int K, int E, int has_shared, const int32_t* __restrict__ idx,
                 const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm_tok,
                 int32_t* __restrict__ row_of) {
    extern __shared__ int32_t sidx[];  // [kChunk * K]
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int nt = static_cast<int>(T - t0 < kChunk ? T - t0 : kChunk);
    for (int i = threadIdx.x; i < nt * K; i += blockDim.x) sidx[i] = idx[t0 * K + i];
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t pos = chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
        for (int tt = 0; tt < nt; ++tt)
            for (int k = 0; k < K; ++k)
                if (sidx[tt * K + k] == e) {
                    perm_tok[pos] = static_cast<int32_t>(t0 + tt);
                    row_of[(t0 + tt) * K + k] = pos;
                    ++pos;
                }
    }
    if (has_shared)
        for (int tt = threadIdx.x; tt < nt; tt += blockDim.x)
            perm_tok[T * K + t0 + tt] = static_cast<int32_t>(t0 + tt);
}

// Copy destination rows [r0, r0 + 32) from their tokens: the row payloads (row_bytes, a
// multiple of 16, as 16-byte chunks spread over the block) and, if src_s, the n_scales FP32
// scales of each row, written K-block-major (dst_s[j * R + r]) so that each warp stores 32
// consecutive rows of one scale column.
__global__ void __launch_bounds__(256)
gather_rows_kernel(int64_t R, int64_t T, int64_t row_bytes, int n_scales,
                   const int32_t* __restrict__ perm_tok, const uint8_t* __restrict__ src,
                   const float* __restrict__ src_s, uint8_t* __restrict__ dst,
                   float* __restrict__ dst_s) {
    __shared__ int32_t stok[32];
    const int chunks = static_cast<int>(row_bytes / 16);
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const int64_t n_grp = (R + 31) / 32;
    for (int64_t gi = blockIdx.x; gi < n_grp; gi += gridDim.x) {
        const int64_t r0 = gi * 32;
        const int nr = static_cast<int>(R - r0 < 32 ? R - r0 : 32);
        __syncthreads();  // the previous group is done with stok
        if (threadIdx.x < 32) {
            const int32_t t = threadIdx.x < nr ? perm_tok[r0 + threadIdx.x] : -1;
            stok[threadIdx.x] = (t >= 0 && t < T) ? t : -1;  // -1: a row no valid (token, slot) claimed
        }
        __syncthreads();
#pragma unroll 4
        for (int i = threadIdx.x; i < nr * chunks; i += blockDim.x) {
            const int rr = i / chunks, ch = i - rr * chunks;
            const int64_t t = stok[rr];
            if (t >= 0) d4[(r0 + rr) * chunks + ch] = s4[t * chunks + ch];
        }
        if (src_s) {
            const int lane = threadIdx.x & 31;
            const int64_t t = lane < nr ? stok[lane] : -1;
            for (int j = threadIdx.x >> 5; j < n_scales; j += blockDim.x >> 5)
                if (t >= 0) dst_s[static_cast<int64_t>(j) * R + r0 + lane] = src_s[t * n_scales + j];
        }
    }
}

}  // namespace

size_t permute_scratch_bytes(int64_t T, int E) {
    const int64_t n_chunks = ceil_div(T > 0 ? T : 1, kChunk);
    return static_cast<size_t>(2 * n_chunks * E) * sizeof(int32_t);
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute(const moe_config* cfg, int64_t T, const int32_t* topk_idx,
                                  const int32_t* counts, const void* xq, const float* xs,
                                  int32_t* offs, int32_t* perm_tok, int32_t* row_of, void* aq,
                                  float* as, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!config_ok(cfg) || T < 0) return MOE_ERR_INVALID_ARG;
    const moe_config& c = *cfg;
    const int E = c.n_experts, K = c.top_k, S = c.has_shared;
    const bool fp8 = (c.mode == MOE_FP8_BLOCK);
    if (!offs || !ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe::ws_layout(c, T).total) return MOE_ERR_WORKSPACE;
    if (T > 0 && (!topk_idx || !xq || !perm_tok || !row_of || !aq)) return MOE_ERR_INVALID_ARG;
    (void)counts;  // the rows are derived from topk_idx itself
    if (T > 0 && (!aligned16(xq) || !aligned16(aq))) return MOE_ERR_INVALID_ARG;
    if (fp8 && T > 0 && (!xs || !as || !aligned16(xs) || !aligned16(as))) return MOE_ERR_INVALID_ARG;
    if ((T * K + T) >= 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t n_chunks = ceil_div(T, kChunk);
    const moe::WsLayout L = moe::ws_layout(c, T);
    int32_t* chunk_cnt = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.perm_scratch);
    int32_t* chunk_base = chunk_cnt + n_chunks * E;
    if (T == 0) {  // every group is empty
        MOE_CUDA_CHECK(cudaMemsetAsync(offs, 0, sizeof(int32_t) * (E + 1 + S), s));
        return MOE_OK;
    }
    chunk_hist_kernel<<<static_cast<unsigned>(n_chunks), 256, sizeof(int32_t) * E, s>>>(
        T, K, E, topk_idx, chunk_cnt);
    MOE_LAUNCH_CHECK();
    scan_kernel<<<1, 1024, 0, s>>>(T, K, E, S, n_chunks, chunk_cnt, chunk_base, offs);
    MOE_LAUNCH_CHECK();
    positions_kernel<<<static_cast<unsigned>(n_chunks), 256, sizeof(int32_t) * kChunk * K, s>>>(
        T, K, E, S, topk_idx, chunk_base, perm_tok, row_of);
    MOE_LAUNCH_CHECK();
    const int64_t R = T * K + T * S;
    const int64_t row_bytes = fp8 ? c.hidden : static_cast<int64_t>(c.hidden) * 4;
    const int64_t n_grp = ceil_div(R, 32);
    const int64_t grid = n_grp < 148 * 8 ? n_grp : 148 * 8;
    gather_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
        R, T, row_bytes, fp8 ? c.hidden / 128 : 0, perm_tok, static_cast<const uint8_t*>(xq),
        fp8 ? xs : nullptr, static_cast<uint8_t*>(aq), fp8 ? as : nullptr);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// ---------------------------------------------------------------------------------------
// moe_permute_noalloc: the same permutation for callers that cannot hand over a workspace.
// Its counters live in a fixed array in device memory that every GPU loading the library
// holds until the process exits.  Every entry a call reads is written earlier in that same
// call (chunk histogram, then bases), so nothing has to start at zero; two calls that run
// on the GPU at the same time share the array and race.
// ---------------------------------------------------------------------------------------
namespace {

constexpr int64_t kNoAllocScratchInts = int64_t(1) << 20;  // 4 MiB: 2 * ceil(T/64) * E int32
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device, looked up once per device.
// (In host code the symbol names a host-side shadow, not device memory.)
moe_status noalloc_scratch(int32_t** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_permute_noalloc(const moe_config* cfg, int64_t T,
                                          const int32_t* topk_idx, const void* xq,
                                          const float* xs, int32_t* offs, int32_t* perm_tok,
                                          int32_t* row_of, void* aq, float* as,
                                          moe_stream_t stream) {
    if (!config_ok(cfg) || T < 0) return MOE_ERR_INVALID_ARG;
    const moe_config& c = *cfg;
    const int E = c.n_experts, K = c.top_k, S = c.has_shared;
    const bool fp8 = (c.mode == MOE_FP8_BLOCK);
    if (!offs) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !xq || !perm_tok || !row_of || !aq)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!aligned16(xq) || !aligned16(aq))) return MOE_ERR_INVALID_ARG;
    if (fp8 && T > 0 && (!xs || !as || !aligned16(xs) || !aligned16(as))) return MOE_ERR_INVALID_ARG;
    if ((T * K + T) >= 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
    const int64_t n_chunks = ceil_div(T, kChunk);
    if (2 * n_chunks * E > kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t* scratch = nullptr;
    MOE_TRY(noalloc_scratch(&scratch));
    if (T == 0) {
        MOE_CUDA_CHECK(cudaMemsetAsync(offs, 0, sizeof(int32_t) * (E + 1 + S), s));
        return MOE_OK;
    }
    int32_t* chunk_cnt = scratch;
    int32_t* chunk_base = scratch + n_chunks * E;
    chunk_hist_kernel<<<static_cast<unsigned>(n_chunks), 256, sizeof(int32_t) * E, s>>>(
        T, K, E, topk_idx, chunk_cnt);
    MOE_LAUNCH_CHECK();
    scan_kernel<<<1, 1024, 0, s>>>(T, K, E, S, n_chunks, chunk_cnt, chunk_base, offs);
    MOE_LAUNCH_CHECK();
    positions_kernel<<<static_cast<unsigned>(n_chunks), 256, sizeof(int32_t) * kChunk * K, s>>>(
        T, K, E, S, topk_idx, chunk_base, perm_tok, row_of);
    MOE_LAUNCH_CHECK();
    const int64_t R = T * K + T * S;
    const int64_t row_bytes = fp8 ? c.hidden : static_cast<int64_t>(c.hidden) * 4;
    const int64_t n_grp = ceil_div(R, 32);
    const int64_t grid = n_grp < 148 * 8 ? n_grp : 148 * 8;
    gather_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
        R, T, row_bytes, fp8 ? c.hidden / 128 : 0, perm_tok, static_cast<const uint8_t*>(xq),
        fp8 ? xs : nullptr, static_cast<uint8_t*>(aq), fp8 ? as : nullptr);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}
