// permute.cu -- a3: token permutation by expert (DeepSeek-V3 co-design teardown, §2.3:
// per-expert counts, then the rows ordered by the argsort of the flat expert ids).
//
// The order is made deterministic and equal to a stable sort: rows are expert-major and,
// within an expert, in ascending token order.  No atomics decide a position:
//   1. chunk histogram: counts of each expert inside each chunk of kChunk tokens;
//   2. scan: offs = exclusive prefix of the counts; base[c][e] = offs[e] + rows of expert e
//      in chunks before c;
//   3. positions: inside a chunk, the rank of each (token, slot) among the earlier entries of
//      its expert, from warp match masks and per-warp counts (one thread per expert walking
//      the chunk for large top_k * experts);
//   4. gather: each token's quantised row is read once and written to all of its destination
//      rows (token-major); the scales go, destination-major, to a K-block-major [H/128, R]
//      array, the layout the grouped GEMM reads.
// With a shared expert, group E follows with every token once, in order, from row T*K.
// An expert id outside [0, E) is dropped: its slot gets row_of = -1 and no row.  The V routed
// rows then fill [0, V) and the rows [V, T*K) belong to no (token, slot): they get
// perm_tok = -1, all-zero codes and zero scales, so the GEMMs compute zeros there.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

// Check word of the MOE_CHECKS build (0 = none): 0x301, a position outside the rows.
__device__ int g_permute_check = 0;

moe_status permute_read_and_clear_check(int32_t* code) {
    MOE_CUDA_CHECK(read_and_clear_word(g_permute_check, code));
    return MOE_OK;
}

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

// One CTA per 32 experts (E <= 1024), 1024 threads.  Every CTA totals every expert over all
// chunks (coalesced, independent loads of the [n_chunks, E] counts) and takes the exclusive
// prefix of the totals, the start of each expert's rows; CTA 0 writes it to offs.  Each CTA
// then writes the chunk bases of its own 32 experts: warp w sums part w of the chunks of
// expert (32 * blockIdx.x + lane), and the parts before it give the part's start.  The rows
// are derived from topk_idx alone, so every position stays inside [0, T*K).
constexpr int kScanThreads = 1024;
constexpr int kScanSlice = 32;  // experts per CTA in the base pass (one per lane)
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(int64_t T, int K, int E, int has_shared, int64_t n_chunks,
            const int32_t* __restrict__ chunk_cnt, int32_t* __restrict__ chunk_base,
            int32_t* __restrict__ offs, int32_t* __restrict__ perm_tok) {
    __shared__ int32_t tot[kScanThreads];                  // expert totals, then their starts
    __shared__ int32_t wsum[kScanThreads / 32];
    __shared__ int32_t n_valid;                            // routed rows claimed by valid ids
    __shared__ int32_t psum[kScanThreads / 32][kScanSlice + 1];  // [part][expert of the slice]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    tot[tid] = 0;
    __syncthreads();
    const int64_t n = n_chunks * E;
    if (kScanThreads % E == 0) {  // every count a thread reads belongs to expert tid % E
        int32_t v = 0;
#pragma unroll 8
        for (int64_t i = tid; i < n; i += kScanThreads) v += chunk_cnt[i];
        atomicAdd(&tot[tid % E], v);
    } else {
        for (int64_t i = tid; i < n; i += kScanThreads) atomicAdd(&tot[i % E], chunk_cnt[i]);
    }
    __syncthreads();
    // exclusive prefix over the experts (entries past E are 0): warp scans, then warp totals
    const int32_t x = tot[tid];
    int32_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int32_t own = wsum[lane];
        int32_t w = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        wsum[lane] = w - own;
    }
    __syncthreads();
    tot[tid] = wsum[warp] + incl - x;
    if (tid == E - 1) n_valid = wsum[warp] + incl;
    __syncthreads();
    // rows no valid (token, slot) claims: perm_tok = -1 (the scale gather zeroes them)
    for (int64_t r = n_valid + static_cast<int64_t>(blockIdx.x) * kScanThreads + tid; r < T * K;
         r += static_cast<int64_t>(gridDim.x) * kScanThreads)
        perm_tok[r] = -1;
    if (blockIdx.x == 0) {
        if (tid < E) offs[tid] = tot[tid];
        if (tid == 0) {
            const int64_t routed = T * K;
            offs[E] = static_cast<int32_t>(routed);
            if (has_shared) offs[E + 1] = static_cast<int32_t>(routed + T);
        }
    }
    const int e = blockIdx.x * kScanSlice + lane;
    const int64_t per = (n_chunks + kScanThreads / 32 - 1) / (kScanThreads / 32);
    const int64_t c0 = min(static_cast<int64_t>(warp) * per, n_chunks), c1 = min(c0 + per, n_chunks);
    int32_t v = 0;
    if (e < E) {
#pragma unroll 8
        for (int64_t c = c0; c < c1; ++c) v += chunk_cnt[c * E + e];
    }
    psum[warp][lane] = v;
    __syncthreads();
    if (e < E) {
        int32_t run = tot[e];
        for (int q = 0; q < warp; ++q) run += psum[q][lane];
        for (int64_t c = c0; c < c1; ++c) {
            chunk_base[c * E + e] = run;
            run += chunk_cnt[c * E + e];
        }
    }
}

// One CTA per chunk, entries (token, slot) in flat order, 32 per "entry warp".  The rank of an
// entry among the earlier entries of its expert is its rank inside its entry warp
// (__match_any_sync) plus the counts of that expert in the earlier entry warps: the stable
// order, with no atomics.  Shared memory: [n_ewarps][E] counts.
__global__ void __launch_bounds__(256)
positions_match_kernel(int64_t T, int K, int E, int has_shared, const int32_t* __restrict__ idx,
                       const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm_tok,
                       int32_t* __restrict__ row_of) {
    extern __shared__ int32_t wcnt[];  // [n_ew][E]
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int nt = static_cast<int>(T - t0 < kChunk ? T - t0 : kChunk);
    const int n = nt * K;
    const int n_ew = (n + 31) / 32;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
    const uint32_t lt = (1u << lane) - 1u;
    for (int i = threadIdx.x; i < n_ew * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    for (int ew = warp; ew < n_ew; ew += nwarps) {
        const int i = ew * 32 + lane;
        int32_t e = i < n ? idx[t0 * K + i] : -1;
        if (e < 0 || e >= E) e = -1;  // dropped
        const uint32_t m = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (m & lt) == 0) wcnt[ew * E + e] = __popc(m);  // one leader per expert
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {  // exclusive prefix over entry warps
        int32_t run = chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
        for (int ew = 0; ew < n_ew; ++ew) {
            const int32_t x = wcnt[ew * E + e];
            wcnt[ew * E + e] = run;
            run += x;
        }
    }
    __syncthreads();
    for (int ew = warp; ew < n_ew; ew += nwarps) {
        const int i = ew * 32 + lane;
        int32_t e = i < n ? idx[t0 * K + i] : -1;
        if (e < 0 || e >= E) e = -1;
        const uint32_t m = __match_any_sync(0xffffffffu, e);
        if (e >= 0) {
            const int32_t pos = wcnt[ew * E + e] + __popc(m & lt);
            const int64_t tt = t0 + i / K;
            if (MOE_DCHECK(g_permute_check, pos >= 0 && pos < T * K, 0x301)) {
                perm_tok[pos] = static_cast<int32_t>(tt);
                row_of[t0 * K + i] = pos;
            }
        } else if (i < n) {
            row_of[t0 * K + i] = -1;  // dropped slot: no row
        }
    }
    if (has_shared)
        for (int tt = threadIdx.x; tt < nt; tt += blockDim.x)
            perm_tok[T * K + t0 + tt] = static_cast<int32_t>(t0 + tt);
}

// Fallback for large K * E (the counts of positions_match_kernel would not fit in shared
// memory): one CTA per chunk, thread e walks the chunk's entries in order.
__global__ void __launch_bounds__(256)
positions_kernel(int64_t T, int K, int E, int has_shared, const int32_t* __restrict__ idx,
                 const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm_tok,
                 int32_t* __restrict__ row_of) {
    extern __shared__ int32_t sidx[];  // [kChunk * K]
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int nt = static_cast<int>(T - t0 < kChunk ? T - t0 : kChunk);
    for (int i = threadIdx.x; i < nt * K; i += blockDim.x) {
        const int32_t e = idx[t0 * K + i];
        sidx[i] = e;
        if (e < 0 || e >= E) row_of[t0 * K + i] = -1;  // dropped slot: no row
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t pos = chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
        for (int tt = 0; tt < nt; ++tt)
            for (int k = 0; k < K; ++k)
                if (sidx[tt * K + k] == e) {
                    if (MOE_DCHECK(g_permute_check, pos >= 0 && pos < T * K, 0x301)) {
                        perm_tok[pos] = static_cast<int32_t>(t0 + tt);
                        row_of[(t0 + tt) * K + k] = pos;
                    }
                    ++pos;
                }
    }
    if (has_shared)
        for (int tt = threadIdx.x; tt < nt; tt += blockDim.x)
            perm_tok[T * K + t0 + tt] = static_cast<int32_t>(t0 + tt);
}

// Row payloads, token-major: one warp per token reads the token's row (row_bytes, a
// multiple of 16) once, 8 x 16 bytes per lane at a time, and writes it to each of the token's
// destination rows: row_of[t, k] for the slots whose expert is in [0, E), and T*K + t for
// the shared expert.  Reading each token once keeps the source out of DRAM re-reads.
constexpr int kGatherPiece = 8;  // 16-byte chunks per lane per piece
__global__ void __launch_bounds__(256)
gather_tokens_kernel(int64_t T, int K, int E, int has_shared, int64_t row_bytes,
                     const int32_t* __restrict__ idx, const int32_t* __restrict__ row_of,
                     const uint8_t* __restrict__ src, uint8_t* __restrict__ dst) {
    const int lane = threadIdx.x % 32;
    const int64_t chunks = row_bytes / 16;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; t < T;
         t += nwarps) {
        // destination rows of this token (lane k < K holds slot k's row, -1 if dropped)
        int32_t my_row = -1;
        if (lane < K) {
            const int32_t e = idx[t * K + lane];
            if (e >= 0 && e < E) my_row = row_of[t * K + lane];
        }
        const uint4* s4 = reinterpret_cast<const uint4*>(src + t * row_bytes);
        for (int64_t c0 = 0; c0 < chunks; c0 += 32 * kGatherPiece) {
            uint4 v[kGatherPiece];
#pragma unroll
            for (int j = 0; j < kGatherPiece; ++j) {
                const int64_t c = c0 + j * 32 + lane;
                if (c < chunks) v[j] = s4[c];
            }
            for (int k = 0; k < K + has_shared; ++k) {
                const int64_t r = k < K ? __shfl_sync(0xffffffffu, my_row, k) : T * K + t;
                if (r < 0) continue;
                if (!MOE_DCHECK(g_permute_check, r < T * K + (has_shared ? T : 0), 0x301)) continue;
                uint4* d4 = reinterpret_cast<uint4*>(dst + r * row_bytes);
#pragma unroll
                for (int j = 0; j < kGatherPiece; ++j) {
                    const int64_t c = c0 + j * 32 + lane;
                    if (c < chunks) d4[c] = v[j];
                }
            }
        }
    }
}

// Scales, destination-major: one warp per 32 consecutive destination rows.  For each tile of
// 32 scale columns the warp reads, row by row, the row's run of scales from its token (one
// coalesced load of up to 128 bytes per row), transposes the 32 x 32 tile through shared
// memory, and writes each column's 32 rows as one coalesced store to the K-block-major
// dst_s[j * R + r].  A row with perm_tok = -1 (claimed by no (token, slot)) gets zero scales
// and an all-zero payload row (row_bytes, a multiple of 16); with n_scales = 0 (FP32 rows)
// only that zeroing runs.
constexpr int kScaleWarps = 8;
__global__ void __launch_bounds__(kScaleWarps * 32)
gather_scales_kernel(int64_t R, int64_t T, int n_scales, int64_t row_bytes,
                     const int32_t* __restrict__ perm_tok, const float* __restrict__ src_s,
                     float* __restrict__ dst_s, uint8_t* __restrict__ dst_rows) {
    __shared__ float tile[kScaleWarps][32][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float (*sm)[33] = tile[w];
    const int64_t n_grp = (R + 31) / 32;
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * kScaleWarps + w; gi < n_grp;
         gi += static_cast<int64_t>(gridDim.x) * kScaleWarps) {
        const int64_t r = gi * 32 + lane;
        int64_t t = r < R ? perm_tok[r] : T;
        uint32_t unclaimed = __ballot_sync(0xffffffffu, t < 0);
        while (unclaimed) {  // rare: only when the routing held ids outside [0, E)
            const int i = __ffs(unclaimed) - 1;
            unclaimed &= unclaimed - 1;
            uint4* d4 = reinterpret_cast<uint4*>(dst_rows + (gi * 32 + i) * row_bytes);
            for (int64_t c = lane; c < row_bytes / 16; c += 32) d4[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (t >= T) t = -1;
        for (int j0 = 0; j0 < n_scales; j0 += 32) {
            const int j = j0 + lane;
            for (int i = 0; i < 32; ++i) {  // row i of the group: its token's scales j0 .. j0 + 31
                const int64_t ti = __shfl_sync(0xffffffffu, t, i);
                sm[lane][i] = (ti >= 0 && j < n_scales) ? src_s[ti * n_scales + j] : 0.f;
            }
            __syncwarp();
            const int nj = min(32, n_scales - j0);
            if (r < R)
                for (int jj = 0; jj < nj; ++jj) dst_s[static_cast<int64_t>(j0 + jj) * R + r] = sm[jj][lane];
            __syncwarp();
        }
    }
}

// The whole permutation on `s`: histogram, scan, positions, row and scale gathers.
// chunk_cnt / chunk_base: [ceil(T / kChunk), E] int32 scratch each.
moe_status launch_permute(const moe_config& c, int64_t T, const int32_t* topk_idx, const void* xq,
                          const float* xs, int32_t* offs, int32_t* perm_tok, int32_t* row_of, void* aq,
                          float* as, int32_t* chunk_cnt, int32_t* chunk_base, cudaStream_t s) {
    const int E = c.n_experts, K = c.top_k, S = c.has_shared;
    const bool fp8 = (c.mode != MOE_FP32);
    const int64_t n_chunks = ceil_div(T, kChunk);
    chunk_hist_kernel<<<static_cast<unsigned>(n_chunks), 256, sizeof(int32_t) * E, s>>>(T, K, E, topk_idx,
                                                                                       chunk_cnt);
    MOE_LAUNCH_CHECK();
    scan_kernel<<<static_cast<unsigned>(ceil_div(E, kScanSlice)), kScanThreads, 0, s>>>(T, K, E, S, n_chunks,
                                                                                      chunk_cnt, chunk_base, offs,
                                                                                      perm_tok);
    MOE_LAUNCH_CHECK();
    const size_t match_smem = sizeof(int32_t) * ceil_div(kChunk * K, 32) * E;
    if (match_smem <= 48 * 1024)
        positions_match_kernel<<<static_cast<unsigned>(n_chunks), 256, match_smem, s>>>(
            T, K, E, S, topk_idx, chunk_base, perm_tok, row_of);
    else
        positions_kernel<<<static_cast<unsigned>(n_chunks), 256, sizeof(int32_t) * kChunk * K, s>>>(
            T, K, E, S, topk_idx, chunk_base, perm_tok, row_of);
    MOE_LAUNCH_CHECK();
    if (aq == nullptr) return MOE_OK;  // indices only
    const int64_t R = T * K + T * S;
    const int64_t row_bytes = fp8 ? c.hidden : static_cast<int64_t>(c.hidden) * 4;
    const int64_t tok_blocks = ceil_div(T, 8);
    gather_tokens_kernel<<<static_cast<unsigned>(tok_blocks < 148 * 8 ? tok_blocks : 148 * 8), 256, 0, s>>>(
        T, K, E, S, row_bytes, topk_idx, row_of, static_cast<const uint8_t*>(xq), static_cast<uint8_t*>(aq));
    MOE_LAUNCH_CHECK();
    // scales (FP8 mode) and the zeroing of unclaimed rows (both modes)
    const int64_t blocks = ceil_div(ceil_div(R, 32), kScaleWarps);
    gather_scales_kernel<<<static_cast<unsigned>(blocks < 148 * 8 ? blocks : 148 * 8), kScaleWarps * 32, 0, s>>>(
        R, T, fp8 ? c.hidden / 128 : 0, row_bytes, perm_tok, xs, as, static_cast<uint8_t*>(aq));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
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
    const bool fp8 = (c.mode != MOE_FP32);
    if (!offs || !ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe::ws_layout(c, T).total) return MOE_ERR_WORKSPACE;
    (void)counts;  // the rows are derived from topk_idx itself
    // FP8 modes: aq and as both NULL ask for the indices only (offs, perm_tok, row_of)
    const bool rows_too = !(fp8 && aq == nullptr && as == nullptr);
    if (T > 0 && (!topk_idx || !perm_tok || !row_of)) return MOE_ERR_INVALID_ARG;
    if (rows_too && T > 0 && (!xq || !aq || !aligned16(xq) || !aligned16(aq))) return MOE_ERR_INVALID_ARG;
    if (rows_too && fp8 && T > 0 && (!xs || !as || !aligned16(xs) || !aligned16(as))) return MOE_ERR_INVALID_ARG;
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
    return launch_permute(c, T, topk_idx, xq, xs, offs, perm_tok, row_of, rows_too ? aq : nullptr, as, chunk_cnt,
                          chunk_base, s);
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
    const bool fp8 = (c.mode != MOE_FP32);
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
    return launch_permute(c, T, topk_idx, xq, xs, offs, perm_tok, row_of, aq, as, chunk_cnt, chunk_base, s);
}
