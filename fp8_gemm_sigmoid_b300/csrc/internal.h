// internal.h -- launchers shared between the libmoe translation units (not part of the ABI).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Workspace layout of moe_forward for T tokens (byte offsets into ws; every region is
// 1024-byte aligned).  R = T*K + T*S rows go through the expert GEMMs.
struct WsLayout {
    int64_t R;         // expert rows
    size_t xq, xs;     // FP8: [T,H] codes, [T,H/128] scales (FP32 mode: unused)
    size_t offs;       // [E+2] int32
    size_t perm_tok;   // [R] int32
    size_t row_of;     // [T*K] int32
    size_t aq, as;     // [R,H] codes (FP32 mode: [R,H] f32), [H/128,R]
    size_t hq, hs;     // [R,I] codes (FP32 mode: h [R,I] f32), [R,I/128]
    size_t yexp;       // [R,H] BF16 (FP32 mode: f32)
    size_t perm_scratch;  // permutation counters
    size_t gemm_scratch;  // grouped-GEMM scheduler / temporaries
    size_t total;
};

WsLayout ws_layout(const moe_config& c, int64_t T);
size_t permute_scratch_bytes(int64_t T, int E);
size_t gemm_scratch_bytes(int32_t n_groups, int64_t rows, int32_t N, int32_t epilogue);
bool config_ok(const moe_config* c);

// gate.cu
bool gate_quant_supported(const moe_config& c);
moe_status launch_gate_quant(const moe_config& c, int64_t T, const void* x, const void* Wg,
                             const float* bias, int32_t* idx, float* w, int32_t* counts,
                             uint8_t* xq, float* xs, cudaStream_t s);
moe_status launch_gate(const moe_config& c, int64_t T, const void* x, const void* Wg,
                       const float* bias, int32_t* idx, float* w, int32_t* counts,
                       float* logits_scratch, cudaStream_t s);
size_t gate_scratch_bytes(const moe_config& c, int64_t T);
moe_status gate_read_and_clear_error(int32_t* code);
moe_status permute_read_and_clear_check(int32_t* code);   // MOE_CHECKS build: 0x301
moe_status combine_read_and_clear_check(int32_t* code);   // MOE_CHECKS build: 0x302

}  // namespace moe
