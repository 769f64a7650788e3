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
//               per 128-wide K block into a 3-stage shared-memory ring (128-byte swizzle);
//   warp 1      allocates 512 TMEM columns; one lane issues 4 MMAs (K = 32 each) per K block
//               into one of two 256-column FP32 partial buffers, then commits;
//   warp 2      scale loader: for each K block, the tile's 128 activation scales and its two
//               weight scales go into a 16-slot shared-memory ring by asynchronous copies, so
//               that the promotion warps issue no global loads (a pending global load stalls
//               their tcgen05 fences); warp 3 idles;
//   warps 4-11  promotion + epilogue: read the partial buffer (tcgen05.ld, 16 columns at a
//               time with the next load in flight), scale it by as[kb,r] * Ws[g,nb,kb] into
//               FP32 register pairs (packed FP32x2 FMA), release the buffer; after the last
//               K block, either SwiGLU + 1x128 FP8 re-quantisation (gate/up GEMM) or BF16
//               output staged in shared memory and written by TMA stores (down GEMM).
// Activation scales are K-block-major ([K/128, rows]) so that the 32 rows of a warp read one
// contiguous 128-byte line per K block.
// Because each K block lands in its own partial buffer, the per-block scaling is exact
// (no FP22 accumulation, no scale folding) and overlaps the next block's MMAs.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "internal.h"
#include "gemm_sched.cuh"
#include "sm100.cuh"

namespace moe {

// Device error word of the tensor-core kernels (0 = none); see moe_device_error.
__device__ int g_tc_error = 0;

namespace {

using namespace sm100;
using namespace sched;

constexpr int kBK = 128;
constexpr int kStages = 3;     // operand ring; over sparse groups a 4th stage takes the place of
constexpr int kMaxStages = 4;  // the down GEMM's output staging (every row is then stored directly)
constexpr int kABytes = kBM * kBK;          // 16 KB
constexpr int kBBytes = kBN * kBK;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 384;   // warp 0 TMA, warp 1 MMA + TMEM, 2 scales, 3 idle, 4..11 epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s)
constexpr int kMaxGroups = kMaxGemmGroups;
constexpr int kOutBox = 32 * 128;                       // one warp's 32 rows x 128 B of output
constexpr int kOutBytes = kEpiWarps * 2 * kOutBox;      // two staging boxes per epilogue warp
constexpr int kScaleSlots = 16;  // K blocks of scale copies in flight (covers L2 latency under load)
constexpr int kSlotFloats = 132;  // 128 activation scales, 2 weight scales, padding to 16 bytes
// Control block after the operand ring and the output staging (byte offsets): barriers,
// TMEM address and flags, amax exchange, warp sums, scale ring, then the tile prefix.
constexpr int kNumBars = 2 * kMaxStages + 2 + 2 + 1 + 1 + 2 * kScaleSlots;  // full/empty, pfull/pempty,
                                                                      // mma_done, ebar, sfull/sempty
constexpr int kCtlBars = 0, kCtlSlot = (kNumBars * 8 + 15) / 16 * 16, kCtlRed = kCtlSlot + 16,
              kCtlWarpSums = kCtlRed + 2048,
              kCtlScales = kCtlWarpSums + 64, kCtlTiles = kCtlScales + kScaleSlots * kSlotFloats * 4;
constexpr int kSmemFixed = 1024 + kStages * kStageBytes + kOutBytes + kCtlTiles;
constexpr int kSmemMax = kSmemFixed + 4 * (kMaxGroups + 1);
static_assert((kMaxStages - kStages) * kStageBytes <= kOutBytes, "the 4th stage lives in the output staging");

enum : int { kErrTimeoutProducer = 0x101, kErrTimeoutMma = 0x102, kErrTimeoutEpilogue = 0x103,
             kErrTimeoutScales = 0x104 };

struct TcParams : sched::Groups {  // n_groups, offs, N, n_tiles_n, swiglu
    int nkb;                    // K / 128
    int rows;                   // row capacity of A, As and out
    const int32_t* gather;      // non-null: row r of A is token gather[r] of X [n_tok, K], its
    int n_tok;                  //   scales the row-major Xs [n_tok, nkb] (read through As)
    const float* As;            // [nkb, rows] (K-block-major), or Xs when gathering
    const float* Ws;            // [n_groups, N/128, nkb]
    void* out;                  // SwiGLU: [rows, N/2] E4M3; store: [rows, N] BF16
    float* out_s;               // SwiGLU: [N/256, rows] (K-block-major, as the next GEMM reads it)
};

// acc[base + i] += (r[2i], r[2i+1]) * (s, s) for i < 8: one packed FP32x2 FMA per column pair,
// each lane rounded as a separate fmaf.
__device__ __forceinline__ void scale_add16(float2 (&acc)[64], int base, const float (&r)[16], float2 s) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[base + i] = __ffma2_rn(make_float2(r[2 * i], r[2 * i + 1]), s, acc[base + i]);
}

// 4-byte asynchronous global -> shared copy (L1-allocating; the data is read once per CTA).
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed (the arrival is
// one of the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// silu(g) = g * sigmoid(g) with the fast exponential and division intrinsics: h is quantised
// to E4M3 (3 mantissa bits) right after, so their few-ulp FP32 error only matters on a code
// boundary, where the FP32 accumulation order already decides.  g -> -inf gives -0.
__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// kRing: operand ring stages, kStages or kMaxStages.  With kMaxStages the last stage occupies
// the output staging, so the down GEMM's epilogue stores every row directly.
template <int kRing>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_fp8_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmO, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* out_stage = smem + kStages * kStageBytes;   // [8 warps][2 halves][32 x 128 B]
    uint8_t* ctl = out_stage + kOutBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ctl + kCtlBars);
    static_assert(kRing == kStages || kRing == kMaxStages, "ring depth");
    uint64_t* full = bars;                  // [kRing]    TMA -> MMA
    uint64_t* empty = bars + kMaxStages;    // [kRing]    MMA -> TMA
    uint64_t* pfull = bars + 2 * kMaxStages;  // [2]      MMA -> epilogue
    uint64_t* pempty = pfull + 2;           // [2]        epilogue -> MMA
    uint64_t* mma_done = pempty + 2;        // [1]        final MMA drain
    uint64_t* ebar = mma_done + 1;          // [1]        epilogue amax exchange (one phase per tile)
    uint64_t* sfull = ebar + 1;             // [kScaleSlots] scale loaders -> epilogue
    uint64_t* sempty = sfull + kScaleSlots; // [kScaleSlots] epilogue -> scale loaders
    static_assert(2 * kMaxStages + 6 + 2 * kScaleSlots <= kNumBars, "barrier block");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl + kCtlSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;   // stays 0: drains wait for in-flight work, not for aborts
    float* red = reinterpret_cast<float*>(ctl + kCtlRed);  // [2 tiles][2 sets][128 rows] amax exchange
    int32_t* warp_sums = reinterpret_cast<int32_t*>(ctl + kCtlWarpSums);  // [kThreads / 32]
    float* sring = reinterpret_cast<float*>(ctl + kCtlScales);         // [kScaleSlots][kSlotFloats]
    int32_t* tile_start = reinterpret_cast<int32_t*>(ctl + kCtlTiles);  // [n_groups + 1]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&pfull[b], 1);
            mbar_init(&pempty[b], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        mbar_init(ebar, kEpiThreads);
        for (int i = 0; i < kScaleSlots; ++i) {
            mbar_init(&sfull[i], 32);
            mbar_init(&sempty[i], kEpiWarps);
        }
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
    tile_prefix<kThreads>(p, warp_sums, tile_start);  // contains the CTA barriers that publish the set-up
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = offsets_usable<kThreads>(p, p.rows, &g_tc_error, 0x121) ? tile_start[p.n_groups] : 0;

    if (warp < kEpiWarp0) {
        // register split: 4 x 48 (TMA, MMA, scale loader, idle) + 8 x 224 (epilogue) <= 12 x 168
        asm volatile("setmaxnreg.dec.sync.aligned.u32 48;");
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
                    for (int j = 0; j < 4; ++j) tok[j] = gather_row(p.gather, c.row0 + 4 * lane + j, c.row_end, p.n_tok, p.n_tok, &g_tc_error, 0x131);
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
                    if (++s == kRing) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok && lane == 0) {
                *abort_flag = 1;
                atomicCAS(&g_tc_error, 0, kErrTimeoutProducer);
            }
            // let every issued copy land before the CTA can exit
            if (lane == 0) {
                for (int i = 0; i < kRing && i < issued; ++i) {
                    if (--s < 0) { s = kRing - 1; ph ^= 1u; }
                    mbar_wait(&full[s], ph, never, kWaitBudget);
                }
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
                    if (++s == kRing) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(&g_tc_error, 0, kErrTimeoutMma);
            }
            // drain: every MMA this thread issued has completed once mma_done flips
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, never, kWaitBudget);
        } else if (warp == 2) {
            // ---------------------------------------------------------------- scale loader
            // For each K block, once the ring slot is free: every lane copies four activation
            // scales and lane 0 the two weight scales with asynchronous 4-byte global->shared
            // copies, then each lane's copies arrive on the slot's barrier when they land
            // (cp.async.mbarrier.arrive.noinc; 32 arrivals complete the phase).  Up to
            // kScaleSlots blocks of copies are in flight.  Rows past the group's end and the
            // absent second weight block copy a valid neighbour: those values are never stored.
            uint32_t sph = 0;  // bit i: parity of the next use of slot i
            bool ok = true;
            int kc = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileCoord c = decode_tile(p, tile_start, t);
                const int64_t nbk = p.N / 128;
                const int b1 = b_block(p, c, 1);
                const float* ws0 = p.Ws + (static_cast<int64_t>(c.g) * nbk + b_block(p, c, 0)) * p.nkb;
                const float* ws1 = b1 < nbk ? p.Ws + (static_cast<int64_t>(c.g) * nbk + b1) * p.nkb : ws0;
                // each lane's four rows: their scale columns (K-block-major As: stride rows per
                // K block) or, gathered, their tokens' rows of Xs (stride 1 per K block)
                const float* src[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = c.row0 + lane + 32 * j;
                    src[j] = p.gather ? p.As + static_cast<int64_t>(gather_row(p.gather, r, c.row_end, p.n_tok, 0, &g_tc_error, 0x131)) * p.nkb
                                      : p.As + (r < c.row_end ? r : c.row0);
                }
                const int64_t kstep = p.gather ? 1 : p.rows;
                for (int kb = 0; kb < p.nkb; ++kb, ++kc) {
                    const int i = kc % kScaleSlots;
                    if (!mbar_wait(&sempty[i], ((sph >> i) & 1u) ^ 1u, abort_flag, kWaitBudget)) { ok = false; break; }
                    sph ^= 1u << i;
                    float* slot = sring + i * kSlotFloats;
#pragma unroll
                    for (int j = 0; j < 4; ++j) cp_async4(slot + lane + 32 * j, src[j] + kb * kstep);
                    if (lane == 0) {
                        cp_async4(slot + 128, ws0 + kb);
                        cp_async4(slot + 129, ws1 + kb);
                    }
                    cp_async_mbar_arrive(&sfull[i]);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(&g_tc_error, 0, kErrTimeoutScales);
            }
            cp_async_wait_all();  // nothing in flight when the CTA exits
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 224;");
        // -------------------------------------------------------------------- promotion + epilogue
        // 128 FP32 accumulators per thread (64 pairs) plus two 16-column TMEM staging chunks.
        const int ew = warp - kEpiWarp0;       // 0..7
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31 (warp % 4 rule)
        const int set = ew / 4;                // column half within each 128-column half-tile
        const int trow = quarter * 32 + lane;  // row of the tile this thread owns
        const int col0 = set * 64, col1 = 128 + set * 64;
        uint8_t* my_stage = out_stage + ew * 2 * kOutBox;
        int b = 0;
        uint32_t pbits = 0;  // bit b: parity of the next phase of pfull[b]
        uint32_t eph = 0;    // phase of ebar
        uint32_t sfp = 0;    // bit i: parity of the next phase of sfull[i]
        int kc = 0;          // K blocks promoted so far (scale ring position)
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileCoord c = decode_tile(p, tile_start, t);
            const int row = c.row0 + trow;
            const bool valid = row < c.row_end;
            // in the down GEMM the last tile's second half lies past N when N % 256 == 128: it is
            // computed from whatever rows follow (zeros past the tensor) and never stored
            const bool half1 = b_block(p, c, 1) < p.N / 128;
            float2 acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.f, 0.f);
            for (int kb = 0; kb < p.nkb; ++kb, ++kc) {
                // this block's scales from the ring: as[kb, row] * Ws[g, half, kb]
                const int si = kc % kScaleSlots;
                if (!mbar_wait(&sfull[si], (sfp >> si) & 1u, abort_flag, kWaitBudget)) { ok = false; break; }
                sfp ^= 1u << si;
                const float* slot = sring + si * kSlotFloats;
                const float sa = slot[trow];
                const float sc0 = sa * slot[128], sc1 = sa * slot[129];
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[si]);
                const float2 s0 = make_float2(sc0, sc0), s1 = make_float2(sc1, sc1);
                if (!mbar_wait(&pfull[b], (pbits >> b) & 1u, abort_flag, kWaitBudget)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(b * kBN);
                // eight 16-column chunks (gate half at col0, up half at col1); the next chunk's
                // TMEM load is in flight while the current chunk is scaled, and the buffer is
                // released as soon as the last load has landed
                float ra[16], rb[16];
                tmem_ld16(taddr + col0, ra);
                tmem_ld_wait_regs16(ra);
#pragma unroll
                for (int q = 0; q < 7; ++q) {
                    const int cn = (q + 1 < 4) ? col0 + 16 * (q + 1) : col1 + 16 * (q - 3);
                    if (q % 2 == 0) {
                        tmem_ld16(taddr + cn, rb);
                        scale_add16(acc, 8 * q, ra, q < 4 ? s0 : s1);
                        tmem_ld_wait_regs16(rb);
                    } else {
                        tmem_ld16(taddr + cn, ra);
                        scale_add16(acc, 8 * q, rb, q < 4 ? s0 : s1);
                        tmem_ld_wait_regs16(ra);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pempty[b]);
                scale_add16(acc, 56, rb, s1);
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
                for (int j = 0; j < 32; ++j) {
                    acc[j].x = silu_f32(acc[j].x) * acc[32 + j].x;
                    acc[j].y = silu_f32(acc[j].y) * acc[32 + j].y;
                    amax = fmaxf(amax, fmaxf(fabsf(acc[j].x), fabsf(acc[j].y)));
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
                            const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(acc[2 * i].x, mul), __fmul_rn(acc[2 * i].y, mul));
                            const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(acc[2 * i + 1].x, mul), __fmul_rn(acc[2 * i + 1].y, mul));
                            pk[i] = lo | (hi << 16);
                        }
                    }
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                                          static_cast<int64_t>(row) * I + c.n_tile * 128 + set * 64);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    if (set == 0)
                        p.out_s[static_cast<int64_t>(c.n_tile) * p.rows + row] = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
                }
            } else {
                // BF16 output.  A warp whose 32 rows all belong to this group stages them in
                // shared memory (128-byte swizzle: 16-byte chunk j of row r at chunk j ^ (r % 8))
                // and one lane writes each 32 x 64 box with a TMA store; a warp holding the
                // group's ragged end stores its valid rows directly, so that no write reaches
                // the next group's rows.
                const bool full_warp = kRing == kStages && c.row0 + quarter * 32 + 32 <= c.row_end;
                if (lane == 0 && kRing == kStages) tma_store_wait_read();  // the staging boxes are free again
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && !half1) break;
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {  // one paired round-to-nearest-even conversion
                        const __nv_bfloat162 v = __floats2bfloat162_rn(acc[h * 32 + i].x, acc[h * 32 + i].y);
                        pk[i] = *reinterpret_cast<const uint32_t*>(&v);
                    }
                    if (full_warp) {
                        uint8_t* box = my_stage + h * kOutBox;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4*>(box + lane * 128 + ((j ^ (lane & 7)) * 16)) =
                                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0)
                            tma_store_2d(&tmO, box, c.n_tile * kBN + h * 128 + set * 64, c.row0 + quarter * 32);
                    } else if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + static_cast<int64_t>(row) * p.N +
                                                              c.n_tile * kBN + h * 128 + set * 64);
#pragma unroll
                        for (int j = 0; j < 8; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
            }
        }
        if (!p.swiglu && lane == 0) tma_store_wait_all();  // every TMA store has completed
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
    static PerDeviceOnce once;
    static int n[PerDeviceOnce::kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= PerDeviceOnce::kMaxDevices) return 148;
    (void)once_per_device(once, [dev] { return cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev); });
    return n[dev] > 0 ? n[dev] : 148;
}

namespace {
bool make_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
    return make_tma_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, 128, 128);
}
}  // namespace

size_t tc_scratch_bytes(int32_t) { return 0; }

moe_status launch_grouped_gemm_fp8_tc(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N,
                                      int32_t Kd, const uint8_t* A, const float* As, const uint8_t* W,
                                      const float* Ws, int32_t epilogue, void* out, float* out_s, void* ws,
                                      cudaStream_t s, const int32_t* gather, int64_t n_tok) {
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
    (void)ws;  // the tile schedule is built in shared memory
    TcParams p;
    p.n_groups = n_groups;
    p.offs = offs;
    p.N = N;
    p.nkb = Kd / kBK;
    p.rows = static_cast<int>(rows);
    p.n_tiles_n = swiglu ? (N / 2) / 128 : (N + kBN - 1) / kBN;
    p.swiglu = swiglu ? 1 : 0;
    p.gather = gather;
    p.n_tok = static_cast<int>(n_tok);
    p.As = As;
    p.Ws = Ws;
    p.out = out;
    p.out_s = out_s;
    static PerDeviceOnce attr_once;
    MOE_CUDA_CHECK(once_per_device(attr_once, [] {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_fp8_tc_kernel<kStages>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(grouped_gemm_fp8_tc_kernel<kMaxStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemMax);
        return e;
    }));
    const int64_t max_tiles = (ceil_div(rows, kBM) + n_groups) * p.n_tiles_n;
    const int grid = static_cast<int>(max_tiles < device_sm_count() ? max_tiles : device_sm_count());
    const int smem = kSmemFixed + 4 * (n_groups + 1);
    // Sparse groups (fewer than 64 rows each on average, as in decoding) leave the tensor cores
    // idle and make the weight stream from HBM the bound: the kernel then takes a 4th operand
    // stage to keep more of it in flight (few of its warps would fill a 32-row staging box
    // anyway).  Over full groups the 3-stage ring is faster.
    const bool deep = rows < 64LL * n_groups;
    if (deep) grouped_gemm_fp8_tc_kernel<kMaxStages><<<grid, kThreads, smem, s>>>(tmA, tmB, tmO, p);
    else grouped_gemm_fp8_tc_kernel<kStages><<<grid, kThreads, smem, s>>>(tmA, tmB, tmO, p);
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
