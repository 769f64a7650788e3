// gemm.h -- grouped-GEMM launchers shared between translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Largest g with tile_start[g] <= tile (tile < tile_start[n_groups]).
__device__ __forceinline__ int find_group(const int32_t* tile_start, int n_groups, int tile) {
    int lo = 0, hi = n_groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

moe_status launch_tile_prefix(int n_groups, int bm, const int32_t* offs, int32_t* tile_start,
                              cudaStream_t s);
// gather non-null: row r of A is row gather[r] of A [n_tok, Kd] and As is the row-major
// [n_tok, Kd/128] scale matrix of those rows (index < 0: a zero row).
moe_status launch_grouped_gemm_fp8_tc(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N,
                                      int32_t Kd, const uint8_t* A, const float* As, const uint8_t* W,
                                      const float* Ws, int32_t epilogue, void* out, float* out_s, void* ws,
                                      cudaStream_t s, const int32_t* gather = nullptr, int64_t n_tok = 0);
moe_status launch_grouped_gemm_mxf8(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N, int32_t Kd,
                                    const uint8_t* A, const float* As, const uint8_t* W, const float* Ws,
                                    int32_t epilogue, void* out, float* out_s, cudaStream_t s,
                                    const int32_t* gather = nullptr, int64_t n_tok = 0);
moe_status mx_read_and_clear_error(int32_t* code);
size_t tc_scratch_bytes(int32_t n_groups);
constexpr int32_t kMaxGemmGroups = 1040;  // groups of one grouped-GEMM call (tile schedule in shared memory)
moe_status tc_read_and_clear_error(int32_t* code);
// 2D TMA map over a row-major [rows, cols] matrix of `elem_bytes`-byte elements, box
// [box_rows x box_cols elements] (box_cols * elem_bytes == 128), 128-byte swizzle.
bool make_tma_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                     int64_t rows, int64_t cols, int box_rows, int box_cols);
int device_sm_count();

}  // namespace moe
