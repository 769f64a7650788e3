// gemm_tc.cu -- a4/a5/a6: the grouped expert GEMM with blockwise FP8 operands on the
// 5th-generation tensor cores (tcgen05 MMA, TMEM accumulators, TMA operand loads).
//
// DeepSeek-V3 co-design teardown (wsisp.com) §5.1: FP8 operands whose block scales are applied
// during accumulation, FP32 accumulation, output quantised as needed.  Insights into
// DeepSeek-V3 précis §3.2: 1x128 activation tiles and 128x128 weight blocks; FP32 (not FP22)
// accumulation.  For group g with rows [offs[g], offs[g+1]):
//   out[r, n] = sum_kb (as[r, kb] * Ws[g, n/128, kb]) * P_kb[r, n],
//   P_kb[r, n] = sum_{k in block kb} A[r, k] * W[g, n, k]                (exact FP32 MMA sums)
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles, warp-specialised:
//   warp 0      TMA producer: A box [128 rows x 128 B] and two B boxes [128 rows x 128 B]
//               per 128-wide K block into a 4-stage shared-memory ring (128-byte swizzle);
//   warp 1      allocates 512 TMEM columns; one lane issues 4 MMAs (K = 32 each) per K block
//               into one of two 256-column FP32 partial buffers, then commits;
//   warps 4-11  promotion + epilogue: read the partial buffer (tcgen05.ld), scale it by
//               as[r,kb] * Ws[g,nb,kb] into FP32 registers, release the buffer; after the last
//               K block, either SwiGLU + 1x128 FP8 re-quantisation (gate/up GEMM) or BF16
//               stores (down GEMM).
// Because each K block lands in its own partial buffer, the per-block scaling is exact
// (no FP22 accumulation, no scale folding) and overlaps the next block's MMAs.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "internal.h"
#include "sm100.cuh"

namespace moe {

// Device error word of the tensor-core kernels (0 = none); see moe_device_error.
__device__ int g_tc_error = 0;

namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 256, kBK = 128;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK;          // 16 KB
constexpr int kBBytes = kBN * kBK;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 384;   // warp 0 TMA, warp 1 MMA + TMEM, 2-3 idle, warps 4..11 epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s)
constexpr int kSmemBytes = kStages * kStageBytes + 4096;  // + alignment slack, barriers, amax exchange

enum : int { kErrTimeoutProducer = 0x101, kErrTimeoutMma = 0x102, kErrTimeoutEpilogue = 0x103 };

struct TcParams {
    int n_groups;
    const int32_t* offs;        // [n_groups + 1]
    const int32_t* tile_start;  // [n_groups + 1] tiles before group g
    int N;                      // rows of W per group
    int nkb;                    // K / 128
    int n_tiles_n;              // 256-column tiles per group
    int swiglu;                 // 1: gate/up pairing + FP8 re-quantisation; 0: BF16 store
    const float* As;            // [rows, nkb]
    const float* Ws;            // [n_groups, N/128, nkb]
    void* out;                  // SwiGLU: [rows, N/2] E4M3; store: [rows, N] BF16
    float* out_s;               // SwiGLU: [rows, N/256]
};

struct TileCoord {
    int g, m_local, n_tile;
    int row0, row_end;
};

__device__ __forceinline__ TileCoord decode_tile(const TcParams& p, int t) {
    TileCoord c;
    c.g = find_group(p.tile_start, p.n_groups, t);
    const int local = t - p.tile_start[c.g];
    c.row0 = p.offs[c.g];
    c.row_end = p.offs[c.g + 1];
    const int mt = (c.row_end - c.row0 + kBM - 1) / kBM;
    c.n_tile = local / mt;
    c.m_local = local - c.n_tile * mt;
    c.row0 += c.m_local * kBM;
    return c;
}

// Row of W (flattened [n_groups * N, K]) and scale block of the two 128-row halves of the
// tile's B operand.  SwiGLU pairs gate block n_tile with the up block I/128 + n_tile, so
// column j of the first half and column 128 + j of the second half belong to the same h.
__device__ __forceinline__ int b_block(const TcParams& p, const TileCoord& c, int half) {
    if (p.swiglu) return half == 0 ? c.n_tile : (p.N / 2) / 128 + c.n_tile;
    return 2 * c.n_tile + half;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_fp8_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* full = bars;                  // [kStages]  TMA -> MMA
    uint64_t* empty = bars + kStages;       // [kStages]  MMA -> TMA
    uint64_t* pfull = bars + 2 * kStages;   // [2]        MMA -> epilogue
    uint64_t* pempty = pfull + 2;           // [2]        epilogue -> MMA
    uint64_t* mma_done = pempty + 2;        // [1]        final MMA drain
    uint64_t* ebar = mma_done + 1;          // [1]        epilogue amax exchange (one phase per tile)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ebar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;   // stays 0: drains wait for in-flight work, not for aborts
    float* red = reinterpret_cast<float*>(tmem_slot + 4);  // [2 tiles][2 sets][128 rows] amax exchange

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&pfull[b], 1);
            mbar_init(&pempty[b], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        mbar_init(ebar, kEpiThreads);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = p.tile_start[p.n_groups];

    if (warp < kEpiWarp0) {
        // register split: 4 x 40 (TMA, MMA, 2 idle) + 8 x 232 (epilogue) = 12 x 168 per CTA
        asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------------------- producer
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileCoord c = decode_tile(p, t);
                const int brow0 = c.g * p.N + b_block(p, c, 0) * 128;
                const int brow1 = c.g * p.N + b_block(p, c, 1) * 128;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, kWaitBudget)) { ok = false; break; }
                    uint8_t* sa = smem + s * kStageBytes;
                    uint8_t* sb = sa + kABytes;
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    tma_load_2d(sa, &tmA, &full[s], kb * kBK, c.row0);
                    tma_load_2d(sb, &tmB, &full[s], kb * kBK, brow0);
                    tma_load_2d(sb + kBBytes / 2, &tmB, &full[s], kb * kBK, brow1);
                    ++issued;
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(&g_tc_error, 0, kErrTimeoutProducer);
            }
            // let every issued copy land before the CTA can exit
            for (int i = 0; i < kStages && i < issued; ++i) {
                if (--s < 0) { s = kStages - 1; ph ^= 1u; }
                mbar_wait(&full[s], ph, never, kWaitBudget);
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);
            int s = 0;
            uint32_t ph = 0;
            int b = 0;
            uint32_t pbits = 0;  // bit b: parity of the next use of partial buffer b
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, kWaitBudget)) { ok = false; break; }
                    if (!mbar_wait(&pempty[b], ((pbits >> b) & 1u) ^ 1u, abort_flag, kWaitBudget)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * kStageBytes);
                    const uint32_t b_addr = a_addr + kABytes;
                    const uint32_t d = tmem_base + static_cast<uint32_t>(b * kBN);
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_f8f6f4(d, umma_desc_sw128(a_addr + k * 32), umma_desc_sw128(b_addr + k * 32),
                                   idesc, k > 0 ? 1u : 0u);
                    mma_commit(&empty[s]);
                    mma_commit(&pfull[b]);
                    pbits ^= 1u << b;
                    b ^= 1;
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(&g_tc_error, 0, kErrTimeoutMma);
            }
            // drain: every MMA this thread issued has completed once mma_done flips
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, never, kWaitBudget);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
        // -------------------------------------------------------------------- promotion + epilogue
        // 128 FP32 accumulators per thread plus one 16-column TMEM load in flight.
        const int ew = warp - kEpiWarp0;       // 0..7
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31 (warp % 4 rule)
        const int set = ew / 4;                // column half within each 128-column half-tile
        const int trow = quarter * 32 + lane;  // row of the tile this thread owns
        const int col0 = set * 64, col1 = 128 + set * 64;
        int b = 0;
        uint32_t pbits = 0;  // bit b: parity of the next phase of pfull[b]
        uint32_t eph = 0;    // phase of ebar
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileCoord c = decode_tile(p, t);
            const int row = c.row0 + trow;
            const bool valid = row < c.row_end;
            const float* as_row = p.As + static_cast<int64_t>(valid ? row : c.row0) * p.nkb;
            const float* ws0 = p.Ws + (static_cast<int64_t>(c.g) * (p.N / 128) + b_block(p, c, 0)) * p.nkb;
            // in the down GEMM the last tile's second half lies past N when N % 256 == 128: it is
            // computed from whatever rows follow (zeros past the tensor) and never stored
            const bool half1 = b_block(p, c, 1) < p.N / 128;
            const float* ws1 = p.Ws + (static_cast<int64_t>(c.g) * (p.N / 128) + (half1 ? b_block(p, c, 1) : 0)) * p.nkb;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.f;
            float sa_next = valid ? __ldg(as_row) : 0.f;
            float w0_next = __ldg(ws0), w1_next = half1 ? __ldg(ws1) : 0.f;
            for (int kb = 0; kb < p.nkb; ++kb) {
                const uint64_t s0 = splat2(sa_next * w0_next), s1 = splat2(sa_next * w1_next);
                if (kb + 1 < p.nkb) {  // scales of the next block, loaded while this one runs
                    sa_next = valid ? __ldg(as_row + kb + 1) : 0.f;
                    w0_next = __ldg(ws0 + kb + 1);
                    w1_next = half1 ? __ldg(ws1 + kb + 1) : 0.f;
                }
                if (!mbar_wait(&pfull[b], (pbits >> b) & 1u, abort_flag, kWaitBudget)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(b * kBN);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float r[16];
                    tmem_ld16(taddr + (q < 4 ? col0 + 16 * q : col1 + 16 * (q - 4)), r);
                    tmem_ld_wait_regs16(r);
                    const uint64_t sc = q < 4 ? s0 : s1;
#pragma unroll
                    for (int i = 0; i < 16; i += 2)
                        ffma2(acc[16 * q + i], acc[16 * q + i + 1], r[i], r[i + 1], sc);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pempty[b]);
                pbits ^= 1u << b;
                b ^= 1;
            }
            if (!ok) break;
            if (p.swiglu) {
                // h = silu(gate) * up for this thread's 64 columns, then the 1x128 tile's amax
                // across the two threads (set 0 and set 1) that share the row
                const int I = p.N / 2;
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    acc[j] = silu_f32(acc[j]) * acc[64 + j];
                    amax = fmaxf(amax, fabsf(acc[j]));
                }
                float* rb = red + eph * 256;  // double-buffered by tile
                rb[set * 128 + trow] = amax;
                mbar_arrive(ebar);
                if (!mbar_wait(ebar, eph, abort_flag, kWaitBudget)) { ok = false; break; }
                amax = fmaxf(rb[trow], rb[128 + trow]);
                eph ^= 1u;
                if (valid) {
                    uint32_t pk[16];
                    if (amax == 0.f) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = 0u;
                    } else {
                        const float mul = __fdiv_rn(448.f, amax);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(acc[4 * i], mul), __fmul_rn(acc[4 * i + 1], mul));
                            const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(acc[4 * i + 2], mul), __fmul_rn(acc[4 * i + 3], mul));
                            pk[i] = lo | (hi << 16);
                        }
                    }
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                                          static_cast<int64_t>(row) * I + c.n_tile * 128 + set * 64);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    if (set == 0) p.out_s[static_cast<int64_t>(row) * (I / 128) + c.n_tile] = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
                }
            } else if (valid) {
                uint16_t* orow = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(row) * p.N + c.n_tile * kBN;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && !half1) break;
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        pk[i] = static_cast<uint32_t>(f32_to_bf16_bits(acc[h * 64 + 2 * i])) |
                                (static_cast<uint32_t>(f32_to_bf16_bits(acc[h * 64 + 2 * i + 1])) << 16);
                    uint4* dst = reinterpret_cast<uint4*>(orow + h * 128 + set * 64);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            atomicCAS(&g_tc_error, 0, kErrTimeoutEpilogue);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// tile_start[g] = sum over groups before g of ceil(count / 128) * n_tiles_n.
__global__ void tc_tile_prefix_kernel(int n_groups, int n_tiles_n, const int32_t* __restrict__ offs,
                                      int32_t* __restrict__ tile_start) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int32_t run = 0;
    for (int g = 0; g < n_groups; ++g) {
        tile_start[g] = run;
        const int32_t cnt = offs[g + 1] - offs[g];
        run += ((cnt + kBM - 1) / kBM) * n_tiles_n;
    }
    tile_start[n_groups] = run;
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

bool make_tma_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                     int64_t rows, int64_t cols, int box_rows, int box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    });
    return n > 0 ? n : 148;
}

namespace {
bool make_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
    return make_tma_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, 128, 128);
}
}  // namespace

size_t tc_scratch_bytes(int32_t n_groups) {
    return (static_cast<size_t>(n_groups) + 1 + 255) / 256 * 1024;
}

moe_status launch_grouped_gemm_fp8_tc(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N,
                                      int32_t Kd, const uint8_t* A, const float* As, const uint8_t* W,
                                      const float* Ws, int32_t epilogue, void* out, float* out_s, void* ws,
                                      cudaStream_t s) {
    const bool swiglu = (epilogue == MOE_EPI_SWIGLU_QUANT);
    if (N % 128 != 0 || (swiglu && N % 256 != 0)) return MOE_ERR_INVALID_ARG;
    if (rows > 0x7fffffffLL || static_cast<int64_t>(n_groups) * N > 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
    CUtensorMap tmA, tmB;
    if (!make_map_u8(&tmA, A, rows, Kd)) return MOE_ERR_CUDA;
    if (!make_map_u8(&tmB, W, static_cast<int64_t>(n_groups) * N, Kd)) return MOE_ERR_CUDA;
    int32_t* tile_start = static_cast<int32_t*>(ws);
    TcParams p;
    p.n_groups = n_groups;
    p.offs = offs;
    p.tile_start = tile_start;
    p.N = N;
    p.nkb = Kd / kBK;
    p.n_tiles_n = swiglu ? (N / 2) / 128 : (N + kBN - 1) / kBN;
    p.swiglu = swiglu ? 1 : 0;
    p.As = As;
    p.Ws = Ws;
    p.out = out;
    p.out_s = out_s;
    tc_tile_prefix_kernel<<<1, 32, 0, s>>>(n_groups, p.n_tiles_n, offs, tile_start);
    MOE_LAUNCH_CHECK();
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(grouped_gemm_fp8_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmemBytes);
    });
    if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
    const int64_t max_tiles = (ceil_div(rows, kBM) + n_groups) * p.n_tiles_n;
    const int grid = static_cast<int>(max_tiles < device_sm_count() ? max_tiles : device_sm_count());
    grouped_gemm_fp8_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tmA, tmB, p);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

moe_status tc_read_and_clear_error(int32_t* code) {
    int v = 0;
    MOE_CUDA_CHECK(cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int)));
    const int zero = 0;
    MOE_CUDA_CHECK(cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int)));
    *code = v;
    return MOE_OK;
}

}  // namespace moe
