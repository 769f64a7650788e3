// gemm_mx.cu -- the grouped expert GEMM in power-of-two (microscaling) mode: FP8 E4M3 operands
// whose 1x128 activation and 128x128 weight scales are powers of two, applied by the tensor
// core itself (tcgen05.mma kind::mxf8f6f4 with 8-bit exponent scale factors, one per 32 K
// elements).  Insights into DeepSeek-V3 précis §3.2 asks for exactly this: tensor cores that
// take the fine-grained scaling factors natively (Blackwell's microscaling) instead of moving
// partial sums to the CUDA cores to scale them.  For group g with rows [offs[g], offs[g+1]):
//   out[r, n] = sum_kb 2^(ea[r,kb] + eb[g,n/128,kb]) * sum_{k in block kb} A[r, k] W[g, n, k],
// accumulated in TMEM over the whole K; the scales are exact, so this is the same sum as the
// FP32-scale path with power-of-two scales, without the per-block promotion.
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles, 12 warps:
//   warp 0      TMA producer: A box [128 rows x 128 B] and two B boxes per 128-deep K block
//               into a 4-stage (gate/up GEMM) or 3-stage (down GEMM) shared-memory ring;
//   warp 1      allocates the 512 TMEM columns; one lane issues the four block-scaled MMAs
//               (K = 32 each) of a K block into the tile's FP32 accumulator (columns 0..255);
//   warps 4-7   scale writers, one per TMEM lane quarter: for each K block they turn the 128
//               activation scales and the tile's two weight scales into 8-bit exponents and
//               store them with tcgen05.st into a 16-slot scale ring (columns 256..511);
//   warps 8-11  epilogue, one thread per tile row: drain the accumulator (tcgen05.ld), release
//               it to the next tile's MMAs, then SwiGLU + 1x128 power-of-two requantisation
//               (gate/up GEMM) or BF16 staged in shared memory and written by TMA (down GEMM).
// Scale-factor layout in TMEM (block-scaled MMA, M = 128, N = 256, one scale per 32 K):
// row r of A reads lane r, column (sfa + r / 32); column n of B reads lane n % 32 of the lane
// quarter of the output row, column (sfb + n / 32); the instruction descriptor's scale-factor
// ids select the byte of the 32-bit cell.  The scale writers store each row's exponent in all
// four bytes of its lane's four SFA cells and the weight exponents (one per 128 columns) in
// every lane of every quarter, so any K chunk of the block reads the block's scale.
#include <cuda.h>

#include "common.cuh"
#include "gemm.h"
#include "gemm_sched.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace moe {

// Device error word of the power-of-two GEMM (0 = none); see moe_device_error.
__device__ int g_mx_error = 0;

namespace {

using namespace sm100;
using namespace sched;

constexpr int kBK = 128;
constexpr int kABytes = kBM * kBK;          // 16 KB
constexpr int kBBytes = kBN * kBK;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kMaxStages = 4;
constexpr int kThreads = 384;
constexpr int kSfWarp0 = 4, kEpiWarp0 = 8;
constexpr uint32_t kTmemCols = 512;
constexpr int kSfSlots = 16;                // K blocks of scale factors in TMEM
constexpr int kSfCols = 16;                 // columns per slot: SFA at +0 (4), SFB at +8 (8)
static_assert(kSfSlots % 4 == 0, "the scale writers fill four contiguous slots with one store");
constexpr uint32_t kSfBase = 256;           // first scale-factor column
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s)
constexpr int kOutBox = 32 * 128;           // 32 rows x 128 B of BF16 output
constexpr int kOutBytes = 4 * 4 * kOutBox;  // 4 epilogue warps x 4 boxes (64 columns each)
constexpr int kRingBytes = (kMaxStages * kStageBytes > 3 * kStageBytes + kOutBytes)
                               ? kMaxStages * kStageBytes : 3 * kStageBytes + kOutBytes;
constexpr int kNumBars = 2 * kMaxStages + 2 * kSfSlots + 3;  // full/empty, sf_full/sf_empty,
                                                             // acc_full, acc_empty, mma_done
constexpr int kCtlSlot = (kNumBars * 8 + 15) / 16 * 16, kCtlWarpSums = kCtlSlot + 16,
              kCtlTiles = kCtlWarpSums + 64;
constexpr int kSmemFixed = 1024 + kRingBytes + kCtlTiles;
constexpr int kSmemMax = kSmemFixed + 4 * (kMaxGemmGroups + 1);

enum : int { kErrTimeoutProducer = 0x111, kErrTimeoutMma = 0x112, kErrTimeoutEpilogue = 0x113,
             kErrTimeoutScales = 0x114 };

struct MxParams : sched::Groups {
    int nkb;                    // K / 128
    int rows;                   // row capacity of A, As and out
    int stages;                 // operand ring depth
    const int32_t* gather;      // non-null: row r of A is token gather[r] of X [n_tok, K], its
    int n_tok;                  //   scales the row-major Xs [n_tok, nkb] (read through As)
    const float* As;            // [nkb, rows] power-of-two scales (K-block-major), or Xs
    const float* Ws;            // [n_groups, N/128, nkb] power-of-two scales
    void* out;                  // SwiGLU: [rows, N/2] E4M3; store: [rows, N] BF16
    float* out_s;               // SwiGLU: [N/256, rows] power-of-two scales (K-block-major)
};

// Instruction descriptor, kind::mxf8f6f4 block-scaled: A and B E4M3 (format 0), both K-major,
// scale-factor ids 0, N >> 3 at bits 17..22, 8-bit exponent scales (bit 23), M >> 4 at 24..28.
constexpr uint32_t idesc_mxf8(int M, int N) {
    return (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
// Four consecutive 16-column groups in one store (columns taddr .. taddr + 63).
__device__ __forceinline__ void tmem_st16x4(uint32_t taddr, const uint32_t (&v)[4][16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::"r"(taddr),
                 "r"(v[0][0]), "r"(v[0][1]), "r"(v[0][2]), "r"(v[0][3]), "r"(v[0][4]), "r"(v[0][5]), "r"(v[0][6]), "r"(v[0][7]), "r"(v[0][8]), "r"(v[0][9]), "r"(v[0][10]), "r"(v[0][11]), "r"(v[0][12]), "r"(v[0][13]), "r"(v[0][14]), "r"(v[0][15]), "r"(v[1][0]), "r"(v[1][1]), "r"(v[1][2]), "r"(v[1][3]), "r"(v[1][4]), "r"(v[1][5]), "r"(v[1][6]), "r"(v[1][7]), "r"(v[1][8]), "r"(v[1][9]), "r"(v[1][10]), "r"(v[1][11]), "r"(v[1][12]), "r"(v[1][13]), "r"(v[1][14]), "r"(v[1][15]), "r"(v[2][0]), "r"(v[2][1]), "r"(v[2][2]), "r"(v[2][3]), "r"(v[2][4]), "r"(v[2][5]), "r"(v[2][6]), "r"(v[2][7]), "r"(v[2][8]), "r"(v[2][9]), "r"(v[2][10]), "r"(v[2][11]), "r"(v[2][12]), "r"(v[2][13]), "r"(v[2][14]), "r"(v[2][15]), "r"(v[3][0]), "r"(v[3][1]), "r"(v[3][2]), "r"(v[3][3]), "r"(v[3][4]), "r"(v[3][5]), "r"(v[3][6]), "r"(v[3][7]), "r"(v[3][8]), "r"(v[3][9]), "r"(v[3][10]), "r"(v[3][11]), "r"(v[3][12]), "r"(v[3][13]), "r"(v[3][14]), "r"(v[3][15])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 8-bit exponent of a power-of-two FP32 scale 2^e (e in [-127, 127]): its biased exponent
// field, which for 2^-127 (the subnormal 0x00400000) is 0, the encoding of 2^-127.
__device__ __forceinline__ uint32_t ue8m0_of(float s) { return (__float_as_uint(s) >> 23) & 0xffu; }

__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_mxf8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmO, const MxParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* out_stage = smem + 3 * kStageBytes;  // down GEMM only (3 stages): [4 warps][4 boxes]
    uint8_t* ctl = smem + kRingBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ctl);
    uint64_t* full = bars;                          // [kMaxStages] TMA -> MMA
    uint64_t* empty = full + kMaxStages;            // [kMaxStages] MMA -> TMA
    uint64_t* sf_full = empty + kMaxStages;         // [kSfSlots]  scale writers -> MMA
    uint64_t* sf_empty = sf_full + kSfSlots;        // [kSfSlots]  MMA -> scale writers
    uint64_t* acc_full = sf_empty + kSfSlots;       // MMA -> epilogue
    uint64_t* acc_empty = acc_full + 1;             // epilogue -> MMA
    uint64_t* mma_done = acc_empty + 1;             // final MMA drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl + kCtlSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;
    int32_t* warp_sums = reinterpret_cast<int32_t*>(ctl + kCtlWarpSums);
    int32_t* tile_start = reinterpret_cast<int32_t*>(ctl + kCtlTiles);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int S = p.stages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < kSfSlots; ++i) {
            mbar_init(&sf_full[i], 4);
            mbar_init(&sf_empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (!p.swiglu) tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    tile_prefix<kThreads>(p, warp_sums, tile_start);
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = offsets_usable<kThreads>(p, p.rows, &g_mx_error, 0x122) ? tile_start[p.n_groups] : 0;

    if (warp < kEpiWarp0) {
        // register split: 8 x 128 (producer, MMA, idle, scale writers) + 4 x 232 (epilogue)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 128;");
        if (warp == 0 && (lane == 0 || p.gather)) {
            // ---------------------------------------------------------------- producer
            // One lane issues the A box and the two B boxes of a K block; with a gathered A
            // every lane gathers four of the tile's 128 rows (tile::gather4) by token index.
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileCoord c = decode_tile(p, tile_start, t);
                const int brow0 = c.g * p.N + b_block(p, c, 0) * 128;
                const int brow1 = c.g * p.N + b_block(p, c, 1) * 128;
                int32_t tok[4] = {0, 0, 0, 0};
                if (p.gather)
                    for (int j = 0; j < 4; ++j) tok[j] = gather_row(p.gather, c.row0 + 4 * lane + j, c.row_end, p.n_tok, p.n_tok, &g_mx_error, 0x132);
                for (int kb = 0; kb < p.nkb; ++kb) {
                    bool w = true;
                    if (lane == 0) w = mbar_wait(&empty[s], ph ^ 1u, abort_flag, kWaitBudget);
                    if (p.gather) w = __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
                    if (!w) { ok = false; break; }
                    uint8_t* sa = smem + s * kStageBytes;
                    uint8_t* sb = sa + kABytes;
                    if (lane == 0) mbar_arrive_expect_tx(&full[s], kStageBytes);
                    if (p.gather) {
                        __syncwarp();
                        tma_gather4(sa + 512 * lane, &tmA, &full[s], kb * kBK, tok[0], tok[1], tok[2], tok[3]);
                    } else {
                        tma_load_2d(sa, &tmA, &full[s], kb * kBK, c.row0);
                    }
                    if (lane == 0) {
                        tma_load_2d(sb, &tmB, &full[s], kb * kBK, brow0);
                        tma_load_2d(sb + kBBytes / 2, &tmB, &full[s], kb * kBK, brow1);
                    }
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok && lane == 0) {
                *abort_flag = 1;
                atomicCAS(&g_mx_error, 0, kErrTimeoutProducer);
            }
            if (lane == 0) {
                for (int i = 0; i < S && i < issued; ++i) {  // let every issued copy land
                    if (--s < 0) { s = S - 1; ph ^= 1u; }
                    mbar_wait(&full[s], ph, never, kWaitBudget);
                }
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_mxf8(kBM, kBN);
            int s = 0, si = 0;
            uint32_t ph = 0, sph = 0;
            uint32_t aph = 0;  // parity of the next acc_empty phase
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(acc_empty, aph ^ 1u, abort_flag, kWaitBudget)) { ok = false; break; }
                aph ^= 1u;
                tc_fence_after();
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, kWaitBudget)) { ok = false; break; }
                    if (!mbar_wait(&sf_full[si], sph, abort_flag, kWaitBudget)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * kStageBytes);
                    const uint32_t b_addr = a_addr + kABytes;
                    const uint32_t sfa = tmem_base + kSfBase + static_cast<uint32_t>(si * kSfCols);
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_mxf8(tmem_base, umma_desc_sw128(a_addr + k * 32), umma_desc_sw128(b_addr + k * 32),
                                 idesc, sfa, sfa + 8, (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                    mma_commit(&sf_empty[si]);
                    if (++s == S) { s = 0; ph ^= 1u; }
                    if (++si == kSfSlots) { si = 0; sph ^= 1u; }
                }
                if (ok) mma_commit(acc_full);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(&g_mx_error, 0, kErrTimeoutMma);
            }
            mma_commit(mma_done);  // every MMA issued has completed once this flips
            mbar_wait(mma_done, 0, never, kWaitBudget);
        } else if (warp >= kSfWarp0) {
            // ---------------------------------------------------------------- scale writers
            // Warp kSfWarp0 + q writes TMEM lane quarter q of each K block's slot: its 32 rows'
            // activation exponents in columns 0..3 (all four bytes) and the two weight
            // exponents in columns 8..11 (first 128 output columns) and 12..15 (second).
            // Rows past the group's end take a valid neighbour's scale (never stored).
            const int q = warp - kSfWarp0;
            const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kSfBase;
            int si = 0;
            uint32_t sph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileCoord c = decode_tile(p, tile_start, t);
                const int64_t nbk = p.N / 128;
                const int b1 = b_block(p, c, 1);
                const float* ws0 = p.Ws + (static_cast<int64_t>(c.g) * nbk + b_block(p, c, 0)) * p.nkb;
                const float* ws1 = b1 < nbk ? p.Ws + (static_cast<int64_t>(c.g) * nbk + b1) * p.nkb : ws0;
                const int r = c.row0 + q * 32 + lane;
                // this row's scale column (K-block-major As) or, gathered, its token's Xs row
                const float* as_col = p.gather ? p.As + static_cast<int64_t>(gather_row(p.gather, r, c.row_end, p.n_tok, 0, &g_mx_error, 0x132)) * p.nkb
                                               : p.As + (r < c.row_end ? r : c.row0);
                const int64_t kstep = p.gather ? 1 : p.rows;
                for (int kb0 = 0; kb0 < p.nkb && ok; kb0 += 4) {
                    // four K blocks of scales in flight at a time
                    float a4[4], w0[4], w1[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int kb = kb0 + j < p.nkb ? kb0 + j : kb0;
                        a4[j] = __ldg(as_col + kb * kstep);
                        w0[j] = __ldg(ws0 + kb);
                        w1[j] = __ldg(ws1 + kb);
                    }
                    if (kb0 + 4 <= p.nkb && si % 4 == 0) {
                        // the four slots si .. si+3 are contiguous: one 64-column store and one
                        // wait for all four K blocks.  The MMA commits each slot's release in
                        // K order, so the release of slot si+3 implies the other three.
                        if (!__all_sync(0xffffffffu, mbar_wait(&sf_empty[si + 3], sph ^ 1u, abort_flag, kWaitBudget))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        uint32_t v[4][16];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t ea = ue8m0_of(a4[j]) * 0x01010101u;
                            const uint32_t e0 = ue8m0_of(w0[j]) * 0x01010101u, e1 = ue8m0_of(w1[j]) * 0x01010101u;
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                v[j][i] = ea;
                                v[j][4 + i] = 0u;
                                v[j][8 + i] = e0;
                                v[j][12 + i] = e1;
                            }
                        }
                        tmem_st16x4(lane_base + static_cast<uint32_t>(si * kSfCols), v);
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            for (int j = 0; j < 4; ++j) mbar_arrive(&sf_full[si + j]);
                        si += 4;
                        if (si == kSfSlots) { si = 0; sph ^= 1u; }
                        continue;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (kb0 + j >= p.nkb) break;
                        // a warp-uniform decision: the TMEM store below is warp-collective
                        if (!__all_sync(0xffffffffu, mbar_wait(&sf_empty[si], sph ^ 1u, abort_flag, kWaitBudget))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t ea = ue8m0_of(a4[j]) * 0x01010101u;
                        const uint32_t e0 = ue8m0_of(w0[j]) * 0x01010101u, e1 = ue8m0_of(w1[j]) * 0x01010101u;
                        const uint32_t v[16] = {ea, ea, ea, ea, 0u, 0u, 0u, 0u, e0, e0, e0, e0, e1, e1, e1, e1};
                        tmem_st16(lane_base + static_cast<uint32_t>(si * kSfCols), v);
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sf_full[si]);
                        if (++si == kSfSlots) { si = 0; sph ^= 1u; }
                    }
                }
            }
            if (!ok && lane == 0) {
                *abort_flag = 1;
                atomicCAS(&g_mx_error, 0, kErrTimeoutScales);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
        // -------------------------------------------------------------------- epilogue
        // One thread per row of the tile (warp kEpiWarp0 + q holds TMEM lanes 32q..32q+31).
        const int q = warp - kEpiWarp0;
        const int trow = q * 32 + lane;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        uint8_t* my_stage = out_stage + q * 4 * kOutBox;
        uint32_t aph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileCoord c = decode_tile(p, tile_start, t);
            const int row = c.row0 + trow;
            const bool valid = row < c.row_end;
            ok = mbar_wait(acc_full, aph, abort_flag, kWaitBudget);
            ok = __all_sync(0xffffffffu, ok);  // TMEM loads below are warp-collective
            if (!ok) break;
            aph ^= 1u;
            tc_fence_after();
            if (p.swiglu) {
                // h = silu(gate) * up over the row's 128 columns, in two halves of 64; the
                // accumulator is released once its last columns are in registers
                float h[128];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float g[64], u[64];
                    tmem_ld32(taddr + half * 64, *reinterpret_cast<float(*)[32]>(&g[0]));
                    tmem_ld32(taddr + half * 64 + 32, *reinterpret_cast<float(*)[32]>(&g[32]));
                    tmem_ld_wait_regs(*reinterpret_cast<float(*)[32]>(&g[0]), *reinterpret_cast<float(*)[32]>(&g[32]));
                    tmem_ld32(taddr + 128 + half * 64, *reinterpret_cast<float(*)[32]>(&u[0]));
                    tmem_ld32(taddr + 128 + half * 64 + 32, *reinterpret_cast<float(*)[32]>(&u[32]));
                    tmem_ld_wait_regs(*reinterpret_cast<float(*)[32]>(&u[0]), *reinterpret_cast<float(*)[32]>(&u[32]));
                    if (half == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_empty);
                    }
#pragma unroll
                    for (int j = 0; j < 64; ++j) h[half * 64 + j] = silu_f32(g[j]) * u[j];
                }
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 128; ++j) amax = fmaxf(amax, fabsf(h[j]));
                if (valid) {
                    const int I = p.N / 2;
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                                          static_cast<int64_t>(row) * I + c.n_tile * 128);
                    const int e = amax == 0.f ? 0 : pow2_exponent(amax);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float* hv = &h[16 * i + 4 * k];
                            const uint32_t lo = f32x2_to_e4m3x2(scale_pow2(hv[0], e), scale_pow2(hv[1], e));
                            const uint32_t hi = f32x2_to_e4m3x2(scale_pow2(hv[2], e), scale_pow2(hv[3], e));
                            w4[k] = amax == 0.f ? 0u : (lo | (hi << 16));
                        }
                        dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    p.out_s[static_cast<int64_t>(c.n_tile) * p.rows + row] = amax == 0.f ? 1.f : exp2_int(e);
                }
            } else {
                // BF16 output: four 64-column boxes per warp in 128B-swizzled shared memory,
                // each written by a TMA store; a warp holding the group's ragged end stores its
                // valid rows directly, so that no write reaches the next group's rows
                const bool half1 = b_block(p, c, 1) < p.N / 128;
                const bool full_warp = c.row0 + q * 32 + 32 <= c.row_end;
                // All four 64-column boxes are read from TMEM and converted to BF16 pairs first,
                // so that the accumulator goes back to the MMA before any store is made.
                uint32_t pk[4][32];
#pragma unroll
                for (int bx = 0; bx < 4; ++bx) {
                    float v[64];
                    tmem_ld32(taddr + bx * 64, *reinterpret_cast<float(*)[32]>(&v[0]));
                    tmem_ld32(taddr + bx * 64 + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
                    tmem_ld_wait_regs(*reinterpret_cast<float(*)[32]>(&v[0]), *reinterpret_cast<float(*)[32]>(&v[32]));
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                        pk[bx][i] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
                if (lane == 0) tma_store_wait_read();  // the staging boxes are free again
                __syncwarp();
#pragma unroll
                for (int bx = 0; bx < 4; ++bx) {
                    if (bx >= 2 && !half1) continue;
                    if (full_warp) {
                        uint8_t* box = my_stage + bx * kOutBox;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4*>(box + lane * 128 + ((j ^ (lane & 7)) * 16)) =
                                make_uint4(pk[bx][4 * j], pk[bx][4 * j + 1], pk[bx][4 * j + 2], pk[bx][4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tma_store_2d(&tmO, box, c.n_tile * kBN + bx * 64, c.row0 + q * 32);
                    } else if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                              static_cast<int64_t>(row) * p.N + c.n_tile * kBN + bx * 64);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_uint4(pk[bx][4 * j], pk[bx][4 * j + 1], pk[bx][4 * j + 2], pk[bx][4 * j + 3]);
                    }
                }
            }
        }
        if (!p.swiglu && lane == 0) tma_store_wait_all();
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicCAS(&g_mx_error, 0, kErrTimeoutEpilogue);
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

bool make_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
    return make_tma_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, 128, 128);
}

}  // namespace

moe_status launch_grouped_gemm_mxf8(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N, int32_t Kd,
                                    const uint8_t* A, const float* As, const uint8_t* W, const float* Ws,
                                    int32_t epilogue, void* out, float* out_s, cudaStream_t s,
                                    const int32_t* gather, int64_t n_tok) {
    const bool swiglu = (epilogue == MOE_EPI_SWIGLU_QUANT);
    if (N % 128 != 0 || (swiglu && N % 256 != 0)) return MOE_ERR_INVALID_ARG;
    if (rows > 0x7fffffffLL || static_cast<int64_t>(n_groups) * N > 0x7fffffffLL || n_tok > 0x7ffffffeLL)
        return MOE_ERR_INVALID_ARG;
    CUtensorMap tmA, tmB, tmO;
    if (gather) {  // A = X [n_tok, K], one-row boxes for tile::gather4
        if (!make_tma_map_2d(&tmA, A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, n_tok, Kd, 1, 128)) return MOE_ERR_CUDA;
    } else if (!make_map_u8(&tmA, A, rows, Kd)) {
        return MOE_ERR_CUDA;
    }
    if (!make_map_u8(&tmB, W, static_cast<int64_t>(n_groups) * N, Kd)) return MOE_ERR_CUDA;
    if (swiglu) tmO = tmA;  // unused
    else if (!make_tma_map_2d(&tmO, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, N, 32, 64)) return MOE_ERR_CUDA;
    MxParams p;
    p.n_groups = n_groups;
    p.offs = offs;
    p.N = N;
    p.n_tiles_n = swiglu ? (N / 2) / 128 : (N + kBN - 1) / kBN;
    p.swiglu = swiglu ? 1 : 0;
    p.nkb = Kd / kBK;
    p.rows = static_cast<int>(rows);
    p.stages = swiglu ? kMaxStages : 3;  // the down GEMM's output staging takes the 4th stage
    p.gather = gather;
    p.n_tok = static_cast<int>(n_tok);
    p.As = As;
    p.Ws = Ws;
    p.out = out;
    p.out_s = out_s;
    static PerDeviceOnce attr_once;
    MOE_CUDA_CHECK(once_per_device(attr_once, [] {
        return cudaFuncSetAttribute(grouped_gemm_mxf8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    }));
    const int64_t max_tiles = (ceil_div(rows, kBM) + n_groups) * p.n_tiles_n;
    const int grid = static_cast<int>(max_tiles < device_sm_count() ? max_tiles : device_sm_count());
    const int smem = kSmemFixed + 4 * (n_groups + 1);
    grouped_gemm_mxf8_kernel<<<grid, kThreads, smem, s>>>(tmA, tmB, tmO, p);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

moe_status mx_read_and_clear_error(int32_t* code) {
    int v = 0;
    MOE_CUDA_CHECK(cudaMemcpyFromSymbol(&v, g_mx_error, sizeof(int)));
    const int zero = 0;
    MOE_CUDA_CHECK(cudaMemcpyToSymbol(g_mx_error, &zero, sizeof(int)));
    *code = v;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_grouped_gemm_mxfp8(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N,
                                             int32_t Kdim, const uint8_t* A, const float* As, const uint8_t* W,
                                             const float* Ws, int32_t epilogue, void* out, float* out_s,
                                             moe_stream_t stream) {
    if (n_groups < 1 || rows < 0 || N <= 0 || Kdim <= 0 || N % 128 || Kdim % 128) return MOE_ERR_INVALID_ARG;
    if (n_groups > kMaxGemmGroups) return MOE_ERR_UNSUPPORTED;
    if (epilogue == MOE_EPI_SWIGLU_QUANT) {
        if (N % 256 != 0 || !out_s || !aligned16(out_s)) return MOE_ERR_INVALID_ARG;
    } else if (epilogue != MOE_EPI_STORE) {
        return MOE_ERR_INVALID_ARG;
    }
    if (!offs || !A || !As || !W || !Ws || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(As) || !aligned16(W) || !aligned16(Ws) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    return launch_grouped_gemm_mxf8(n_groups, offs, rows, N, Kdim, A, As, W, Ws, epilogue, out, out_s,
                                    reinterpret_cast<cudaStream_t>(stream));
}
