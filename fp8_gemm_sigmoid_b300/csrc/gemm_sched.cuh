// gemm_sched.cuh -- the tile schedule shared by the grouped expert GEMM kernels: which group,
// m-tile and n-tile each output tile of a persistent CTA is, built on the device from the
// groups' row offsets (no host synchronisation, no extra launch).
#pragma once

#include <stdint.h>

#include "gemm.h"

namespace moe {
namespace sched {

constexpr int kBM = 128, kBN = 256;
constexpr int kNFastMTiles = 32;  // m-tiles (4096 rows) above which a group runs n-fastest

// The groups of one grouped-GEMM call.
struct Groups {
    int n_groups;
    const int32_t* offs;  // [n_groups + 1] row offsets
    int N;                // rows of W per group
    int n_tiles_n;        // 256-column tiles per group (SwiGLU: 128 h columns each)
    int swiglu;           // 1: tile n pairs gate block n with up block N/256 + n
};

struct TileCoord {
    int g, m_local, n_tile;
    int row0, row_end;
};

// Tile t of the schedule.  In a group of up to kNFastMTiles m-tiles the m-tiles run fastest:
// the concurrent tiles share each weight tile in L2.  A larger group (the shared expert's T
// rows) runs its n-tiles fastest instead, so that its A rows, which would not stay in L2
// between n-tiles, are read once while its weight tiles stay in L2.
__device__ __forceinline__ TileCoord decode_tile(const Groups& p, const int32_t* tile_start, int t) {
    TileCoord c;
    c.g = find_group(tile_start, p.n_groups, t);
    const int local = t - tile_start[c.g];
    c.row0 = p.offs[c.g];
    c.row_end = p.offs[c.g + 1];
    const int mt = (c.row_end - c.row0 + kBM - 1) / kBM;
    if (mt > kNFastMTiles) {
        c.m_local = local / p.n_tiles_n;
        c.n_tile = local - c.m_local * p.n_tiles_n;
    } else {
        c.n_tile = local / mt;
        c.m_local = local - c.n_tile * mt;
    }
    c.row0 += c.m_local * kBM;
    return c;
}

// 128-row block of W (within the group) for the two halves of the tile's B operand.  SwiGLU
// pairs gate block n_tile with the up block I/128 + n_tile, so column j of the first half and
// column 128 + j of the second half belong to the same h.
__device__ __forceinline__ int b_block(const Groups& p, const TileCoord& c, int half) {
    if (p.swiglu) return half == 0 ? c.n_tile : (p.N / 2) / 128 + c.n_tile;
    return 2 * c.n_tile + half;
}

// Tiles of group g: ceil(rows_g / 128) m-tiles times the n-tiles of one group.
__device__ __forceinline__ int group_tiles(const Groups& p, int g) {
    return ((p.offs[g + 1] - p.offs[g] + kBM - 1) / kBM) * p.n_tiles_n;
}

// tile_start[g] = tiles of the groups before g (g = 0..n_groups), computed by the whole CTA
// (kThreads threads) from the device-side row offsets: each thread sums a run of consecutive
// groups, a block scan of the run totals gives each run's start, and the thread writes its
// run's prefixes.  warp_sums: kThreads / 32 ints of shared memory.
template <int kThreads>
__device__ void tile_prefix(const Groups& p, int32_t* warp_sums, int32_t* tile_start) {
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int per = (p.n_groups + kThreads - 1) / kThreads;
    const int g0 = min(tid * per, p.n_groups), g1 = min(g0 + per, p.n_groups);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += group_tiles(p, g);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kThreads / 32 ? warp_sums[lane] : 0;
        const int own = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        if (lane < kThreads / 32) warp_sums[lane] = w - own;  // exclusive warp offsets
    }
    __syncthreads();
    int run = warp_sums[warp] + incl - sum;
    for (int g = g0; g < g1; ++g) {
        tile_start[g] = run;
        run += group_tiles(p, g);
    }
    if (g0 < g1 && g1 == p.n_groups) tile_start[p.n_groups] = run;
    __syncthreads();
}

// TMA gather of four rows (y0..y3, each one box row of 128 bytes at column x) of a 2D tensor
// whose box is one row high, into 4 consecutive 128-byte rows of shared memory at dst (128-byte
// swizzle by destination address, so dst at a 512-byte boundary lands them as rows of an A
// tile); the bytes are reported to `bar`.  A row index outside the tensor reads zeros.
__device__ __forceinline__ void tma_gather4(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y0, int32_t y1, int32_t y2, int32_t y3) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(x),
        "r"(y0), "r"(y1), "r"(y2), "r"(y3)
        : "memory");
}

// Token of row r of a gathered A operand (rows [row0, row_end) of the tile's group): gather[r],
// with rows past the group's end, unclaimed rows (index -1) and indices past the n_tok tokens
// mapped to `none`.  The MOE_CHECKS build records `code` in *word for an index that is
// neither -1 nor a token.
__device__ __forceinline__ int32_t gather_row(const int32_t* gather, int r, int row_end, int32_t n_tok,
                                              int32_t none, int* word, int code) {
    if (r >= row_end) return none;
    const int32_t t = gather[r];
    if (t >= 0 && t < n_tok) return t;
    (void)MOE_DCHECK(*word, t == -1, code);
    (void)word; (void)code;
    return none;
}

// MOE_CHECKS build: whether the groups' offsets are usable (offs[0] >= 0, non-decreasing,
// offs[n_groups] <= rows), agreed by the whole CTA (kThreads threads, every one calls this).
// A CTA that finds them unusable records `code` and runs no tile.
template <int kThreads>
__device__ bool offsets_usable(const Groups& p, int rows, int* word, int code) {
    bool ok = true;
#ifdef MOE_CHECKS
    for (int g = threadIdx.x; g < p.n_groups; g += kThreads)
        ok = ok && p.offs[g] >= 0 && p.offs[g] <= p.offs[g + 1] && p.offs[g + 1] <= rows;
    ok = __syncthreads_and(ok) != 0;
    if (!ok && threadIdx.x == 0) atomicCAS(word, 0, code);
#else
    (void)p; (void)rows; (void)word; (void)code;
#endif
    return ok;
}

// 2D TMA store of a [32 rows x 128 B] box from shared memory (128-byte swizzle) at (x, y).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_src))), "r"(x), "r"(y)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

}  // namespace sched
}  // namespace moe
