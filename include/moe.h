/*
 * moe.h -- C ABI of libmoe: the forward pass of a DeepSeek-V3-style fine-grained MoE layer
 * on one B300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *  [P1] "从 1024 块 GPU 到 558 万美元：拆解 DeepSeek-V3 的算法-系统协同设计" (wsisp.com):
 *       §2.2 MoEGate listing; §2.3 dispatch skeleton; §5.1 blockwise FP8 GEMM sketch.
 *  [P2] "深入理解 DeepSeek-V3" (Chinese précis of "Insights into DeepSeek-V3: Scaling
 *       Challenges and Reflections on Hardware for AI Architectures", arXiv 2505.09343):
 *       §3.1 (8 routed + 1 shared expert, FP8 dispatch / BF16 combine);
 *       §3.2 (1x128 activation tiles, 128x128 weight blocks, FP32 accumulation).
 *
 * Conventions for every entry point:
 *  - All data pointers are DEVICE pointers unless a parameter says "host".  The caller
 *    allocates and owns every buffer (inputs, outputs, workspace); the library allocates
 *    nothing, frees nothing and never synchronises the stream it is given.  Work is
 *    enqueued on `stream` (NULL = the legacy default stream) and completes asynchronously.
 *  - Row-major, densely packed tensors; shapes are given as [dim0, dim1, ...].
 *    BF16 tensors are IEEE bfloat16 bit patterns (uint16); FP8 tensors are OCP E4M3 codes
 *    (uint8); scales are FP32.
 *  - A call returns MOE_OK after enqueueing its kernels, or an error code without
 *    enqueueing anything when an argument is invalid.  MOE_ERR_CUDA reports a launch error
 *    (cudaGetLastError).  No exception or longjmp crosses the ABI; no kernel traps.
 *  - Calls on the same stream are ordered; calls that share a workspace must not overlap.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every entry point is exported from libmoe.so (the library is built with hidden default
 * visibility). */
#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* a pointer is NULL or misaligned, or a size is out of range */
    MOE_ERR_UNSUPPORTED = 2,  /* the configuration is valid but this build does not run it */
    MOE_ERR_WORKSPACE = 3,    /* the workspace is smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
    MOE_ERR_TIMEOUT = 5       /* a bounded device-side wait expired (see moe_device_error) */
} moe_status;

/* Numerics of the layer. */
typedef enum moe_mode {
    MOE_FP32 = 0,      /* x, gate weight, expert weights and y in FP32, no quantisation */
    MOE_FP8_BLOCK = 1, /* x, gate weight and y in BF16; expert GEMMs on E4M3 operands with
                          1x128 activation and 128x128 weight FP32 scales amax/448 ([P2] §3.2) */
    MOE_MXFP8 = 2      /* as MOE_FP8_BLOCK, but every scale is a power of two (the smallest
                          2^e with 448 * 2^e >= amax) and the tensor cores apply the scales
                          themselves ([P2] §3.2: scaling factors taken natively, microscaling);
                          weights from moe_quant_128x128_pow2 */
} moe_mode;

/* Layer configuration ([P1] §2.2: hidden_size, n_routed_experts, num_experts_per_tok,
 * n_group, topk_group, routed_scaling_factor; [P1] §2.2 / [P2] §3.1: one shared expert).
 * Valid when: hidden, inter, n_experts, n_group, topk_group, top_k > 0;
 * n_experts % n_group == 0 and n_experts / n_group >= 2 (the group score sums two experts);
 * topk_group <= n_group; top_k <= topk_group * n_experts / n_group; n_experts <= 1024;
 * top_k <= 32; has_shared in {0, 1}; hidden % 128 == 0 and inter % 128 == 0 in both modes. */
typedef struct moe_config {
    int32_t hidden;      /* H: model width */
    int32_t inter;       /* I: FFN width of each routed expert and of the shared expert */
    int32_t n_experts;   /* E: routed experts */
    int32_t n_group;     /* G: expert groups for group-limited routing */
    int32_t topk_group;  /* TG: groups kept per token */
    int32_t top_k;       /* K: routed experts per token */
    float routed_scaling_factor; /* multiplies the (normalised) routing weights */
    int32_t has_shared;  /* 1: add the always-on shared expert */
    int32_t mode;        /* moe_mode */
} moe_config;

/* Epilogues of the grouped expert GEMM. */
typedef enum moe_epilogue {
    MOE_EPI_SWIGLU_QUANT = 0, /* W = stacked [gate; up] (N = 2I rows per group); output
                                 h = silu(gate) * up quantised in 1x128 tiles (FP8 mode) or
                                 h in FP32 (FP32 mode), [rows, I] */
    MOE_EPI_STORE = 1         /* W = down projection (N = H rows per group); output [rows, N]
                                 in BF16 (FP8 mode) or FP32 (FP32 mode) */
} moe_epilogue;

/* Expert weights of the layer.  Routed experts are slots 0..E-1 and the shared expert, if
 * any, is slot E.
 *  FP8 mode: W13 [E+S, 2I, H] E4M3 codes and W13_s [E+S, 2I/128, H/128] scales from
 *            moe_quant_128x128 (rows 0..I-1 of each slot are the gate projection, rows
 *            I..2I-1 the up projection); W2 [E+S, H, I] codes, W2_s [E+S, H/128, I/128].
 *  FP32 mode: W13 [E+S, 2I, H] and W2 [E+S, H, I] FP32; the scale pointers are ignored.
 *  Wg: gate weight [E, H], BF16 (FP8 mode) or FP32 (FP32 mode). */
typedef struct moe_weights {
    const void* Wg;
    const void* W13;
    const float* W13_s;
    const void* W2;
    const float* W2_s;
} moe_weights;

/* Human-readable name of a status code (static storage; never NULL). */
MOE_API const char* moe_status_string(moe_status s);

/* MOE_OK when *cfg satisfies the rules above, else MOE_ERR_INVALID_ARG. */
MOE_API moe_status moe_config_validate(const moe_config* cfg);

/* Bytes of device workspace that moe_forward needs for T tokens (host out-param).  The
 * same workspace also serves moe_permute and moe_grouped_gemm_* for that T. */
MOE_API moe_status moe_workspace_size(const moe_config* cfg, int64_t T, size_t* bytes);

/* a1. [P1] §2.2 MoEGate, with the per-expert histogram of [P1] §2.3 fused in.
 * logits = x . Wg^T accumulated in FP32; scores = sigmoid(logits); selection scores
 * c = scores + bias (the bias steers selection only); group score = sum of the two largest
 * c of each of the n_group groups; the topk_group best groups are kept and the other
 * groups' experts are excluded; the top_k experts by c among the kept ones are chosen
 * (ties to the lower index; slots in descending c); weights = scores (un-biased) at the
 * chosen experts, divided by (their sum + 1e-20) if top_k > 1, times
 * routed_scaling_factor.
 *  x [T, H]: BF16 (FP8 mode) or FP32 (FP32 mode); Wg [E, H] same type; bias [E] FP32.
 *  Outputs: topk_idx [T, K] int32, topk_w [T, K] FP32, counts [E] int32 (overwritten:
 *  counts[e] = number of (token, slot) pairs routed to e).  T == 0 only zeroes counts. */
MOE_API moe_status moe_gate(const moe_config* cfg, int64_t T, const void* x, const void* Wg,
                    const float* bias, int32_t* topk_idx, float* topk_w, int32_t* counts,
                    moe_stream_t stream);

/* a1 + a2 fused ([P1] §2.2 MoEGate; [P2] §3.2 1x128 activation tiles; no counterpart on the
 * pages as one call): moe_gate, plus the 1x128 FP8 quantisation of the same x as moe_quant_1x128
 * (MOE_FP8_BLOCK) or moe_quant_1x128_pow2 (MOE_MXFP8) writes it, bit for bit, while x
 * streams through the gate once.
 *  xq [T, H] E4M3 codes, 16-byte aligned; xs [T, H/128] FP32 scales.
 *  Returns MOE_ERR_UNSUPPORTED (and launches nothing) for configurations outside the fused
 *  kernel: FP32 mode, E not a multiple of 32 or above 256, E / n_group not a multiple of 32,
 *  n_group > 8, top_k > 8, H % 128 != 0, or x / Wg / xq not 16-byte aligned; callers then
 *  use moe_gate and moe_quant_1x128. */
MOE_API moe_status moe_gate_quant(const moe_config* cfg, int64_t T, const void* x, const void* Wg,
                                  const float* bias, int32_t* topk_idx, float* topk_w,
                                  int32_t* counts, uint8_t* xq, float* xs, moe_stream_t stream);

/* moe_forward takes moe_gate_quant from this many tokens up.  The fused kernel's pace is set
 * by its quantising warps, about 100 us per 128-token CTA on a B300 whatever T, so for fewer
 * tokens moe_gate and moe_quant_1x128 launched apart finish first (69 against 103 us at
 * T = 256; 113 against 98 us at T = 8192). */
#define MOE_GATE_QUANT_MIN_TOKENS 6144

/* a2. [P2] §3.2 activation quantisation in 1x128 tiles.  For every row and every 128
 * consecutive columns: amax = max |x|; scale = amax / 448 and q = E4M3(x * (448 / amax))
 * (round to nearest even, saturating to +-448); amax == 0 gives scale 1 and q = 0.
 *  x [rows, cols] BF16, cols % 128 == 0; q [rows, cols] E4M3; s [rows, cols/128] FP32.
 *  Pointers 16-byte aligned. */
MOE_API moe_status moe_quant_1x128(int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q,
                           float* s, moe_stream_t stream);

/* a2'. [P2] §3.2 weight quantisation in 128x128 blocks (same rule, one scale per block).
 *  w [n_mats, rows, cols] BF16, rows % 128 == 0, cols % 128 == 0;
 *  q [n_mats, rows, cols] E4M3; s [n_mats, rows/128, cols/128] FP32.  16-byte aligned. */
MOE_API moe_status moe_quant_128x128(int64_t n_mats, int64_t rows, int64_t cols, const uint16_t* w,
                             uint8_t* q, float* s, moe_stream_t stream);

/* a2 in power-of-two mode ([P2] §3.2, scales the tensor cores take natively): the same tiles
 * and blocks, scale = 2^e with e the smallest integer such that 448 * 2^e >= amax (clamped to
 * [-127, 127]; amax == 0 gives scale 1 and q = 0), q = E4M3(x * 2^-e), an exact scaling, so no
 * value saturates.  Same arguments as moe_quant_1x128 / moe_quant_128x128. */
MOE_API moe_status moe_quant_1x128_pow2(int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q,
                                        float* s, moe_stream_t stream);
MOE_API moe_status moe_quant_128x128_pow2(int64_t n_mats, int64_t rows, int64_t cols, const uint16_t* w,
                                          uint8_t* q, float* s, moe_stream_t stream);

/* a3. [P1] §2.3 token permutation by expert, deterministic: rows are expert-major and,
 * within an expert, in ascending token order (the stable argsort of the flat expert ids).
 * With has_shared, group E follows with every token once, in order, in rows
 * [T*K, T*K + T).  R = T*K + T*S rows.
 *  topk_idx [T, K] int32 with entries in [0, E) (as moe_gate writes them).  An entry outside
 *  that range is dropped: its row_of entry is -1 and it claims no row.  With V valid entries
 *  the routed rows fill [0, V); the rows [V, T*K), which the last routed group's range
 *  [offs[E-1], offs[E]) then also covers, get perm_tok = -1, all-zero codes and zero scales,
 *  so the grouped GEMMs compute zeros there and moe_combine never reads them.
 *  counts [E]: the gate's histogram, accepted for symmetry and not read (may be NULL) -- the
 *  rows are derived from topk_idx;
 *  FP8 mode: xq [T, H] E4M3 and xs [T, H/128] FP32 (from moe_quant_1x128), gathered into
 *            aq [R, H] and as [H/128, R] (K-block-major: as[j * R + r] is the scale of
 *            columns 128j..128j+127 of row r, the layout moe_grouped_gemm_fp8 reads);
 *  FP32 mode: xq is x [T, H] FP32 gathered into aq [R, H] FP32; xs and as are ignored.
 *  FP8 modes: aq and as both NULL ask for the indices only (offs, perm_tok, row_of; xq and xs
 *  are then not read), for moe_grouped_gemm_fp8_gather.
 *  Outputs: offs [E + 1 + S] int32: offs[e] = rows of the experts before e (e <= E-1),
 *  offs[E] = T*K, offs[E+1] = T*K + T with the shared expert; perm_tok [R] int32 (token of
 *  each row, -1 for an unclaimed row), row_of [T, K] int32 (row of each (t, k), -1 if dropped).
 *  ws/ws_bytes: workspace of at least moe_workspace_size(cfg, T) bytes. */
MOE_API moe_status moe_permute(const moe_config* cfg, int64_t T, const int32_t* topk_idx,
                       const int32_t* counts, const void* xq, const float* xs, int32_t* offs,
                       int32_t* perm_tok, int32_t* row_of, void* aq, float* as, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* moe_permute without a workspace (the pages have no counterpart; this is a library
 * convenience).  For callers that cannot allocate device memory or hand over a workspace:
 * code running inside a host framework that owns the whole device-memory budget and forbids
 * extra allocations, latency-critical loops that cannot afford cudaMalloc's implicit device
 * synchronisation, and plugin interfaces whose signature carries only inputs and outputs.
 * Same arguments, results and rules as moe_permute, minus counts, ws and ws_bytes.
 *  - Scratch: a fixed 4 MiB array in device memory (file-scope, 256-byte aligned) that every
 *    GPU which loads libmoe holds until the process exits.  Limit: 2 * ceil(T/64) * E <=
 *    1,048,576 int32 (e.g. T <= 131072 at E = 256); larger calls return MOE_ERR_UNSUPPORTED
 *    and enqueue nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call before any
 *    stream capture.  MOE_ERR_CUDA if the lookup fails.  The address is kept for the life of
 *    the process: after cudaDeviceReset (or any teardown of the device's primary context)
 *    the kept address is stale, so do not call this entry point on that device again.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *  - Every call shares the array and overwrites it; nothing in it needs to start at zero.
 *    Calls that overlap on the GPU (other streams, other threads) race and must be
 *    serialised by the caller. */
MOE_API moe_status moe_permute_noalloc(const moe_config* cfg, int64_t T, const int32_t* topk_idx,
                               const void* xq, const float* xs, int32_t* offs,
                               int32_t* perm_tok, int32_t* row_of, void* aq, float* as,
                               moe_stream_t stream);

/* a4/a5/a6. [P1] §5.1 / [P2] §3.2 grouped expert GEMM with blockwise FP8 operands and
 * FP32 accumulation: for group g with rows [offs[g], offs[g+1]) and every output column n,
 *   out[r, n] = sum_kb (as[r, kb] * Ws[g, n/128, kb]) * sum_{k in kb} A[r, k] * W[g, n, k]
 * followed by the epilogue (moe_epilogue).  The shared expert is simply one more group.
 *  n_groups >= 1; offs [n_groups + 1] device int32, non-decreasing, offs[0] == 0,
 *  offs[n_groups] <= rows; rows = capacity (host) of A and out; N % 128 == 0 (for
 *  SWIGLU_QUANT, N = 2I with I % 128 == 0); Kdim % 128 == 0.
 *  A [rows, Kdim] E4M3, As [Kdim/128, rows] (K-block-major: As[kb * rows + r]);
 *  W [n_groups, N, Kdim] E4M3, Ws [n_groups, N/128, Kdim/128];
 *  SWIGLU_QUANT: out [rows, N/2] E4M3 and out_s [N/256, rows] FP32, K-block-major like As
 *  (the 1x128 quantisation of h in FP32 -> FP8, no intermediate rounding);
 *  STORE: out [rows, N] BF16, out_s unused.
 *  Rows beyond offs[n_groups] are left untouched.  16-byte aligned pointers.
 *  n_groups <= 1040 (MOE_ERR_UNSUPPORTED beyond).  ws/ws_bytes are not used (the tile
 *  schedule is built in shared memory from offs); they may be NULL/0. */
MOE_API moe_status moe_grouped_gemm_fp8(int32_t n_groups, const int32_t* offs, int64_t rows,
                                int32_t N, int32_t Kdim, const uint8_t* A, const float* As,
                                const uint8_t* W, const float* Ws, int32_t epilogue,
                                void* out, float* out_s, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/* [P1] §2.3 with the permuted copy fused away: the same grouped GEMM, with row r of A read
 * straight from the quantised tokens, A[r] = X[perm_tok[r]] and its scales Xs[perm_tok[r], :],
 * by TMA gathers of four token rows at a time (on B300 the gate/up GEMM then runs at half the
 * rate of the box-loaded copy, so moe_forward keeps the copy).  perm_tok [rows] as moe_permute writes it
 * (entries -1, rows no (token, slot) claims, read as zero rows); X [T, Kdim] E4M3 and Xs
 * [T, Kdim/128] FP32 row-major (moe_quant_1x128's outputs); the other arguments and the
 * results as for moe_grouped_gemm_fp8, bit for bit (the same bytes reach the same MMAs). */
MOE_API moe_status moe_grouped_gemm_fp8_gather(int32_t n_groups, const int32_t* offs, int64_t rows,
                                               int32_t N, int32_t Kdim, const int32_t* perm_tok,
                                               int64_t T, const uint8_t* X, const float* Xs,
                                               const uint8_t* W, const float* Ws, int32_t epilogue,
                                               void* out, float* out_s, moe_stream_t stream);

/* The grouped expert GEMM of MOE_MXFP8 mode ([P2] §3.2: tensor cores that take the
 * fine-grained scaling factors natively): as moe_grouped_gemm_fp8, but every scale in As and
 * Ws must be a power of two 2^e, e in [-127, 127] (as moe_quant_*_pow2 write them), and the
 * tensor cores apply them as 8-bit exponents, accumulating the whole K in FP32 with no
 * per-block promotion.  SWIGLU_QUANT re-quantises h with power-of-two scales (out_s holds
 * 2^e).  A scale that is not a power of two is read as its exponent alone.  No workspace. */
MOE_API moe_status moe_grouped_gemm_mxfp8(int32_t n_groups, const int32_t* offs, int64_t rows,
                                          int32_t N, int32_t Kdim, const uint8_t* A, const float* As,
                                          const uint8_t* W, const float* Ws, int32_t epilogue,
                                          void* out, float* out_s, moe_stream_t stream);

/* moe_grouped_gemm_mxfp8 with the gathered A operand of moe_grouped_gemm_fp8_gather
 * (X, Xs from moe_quant_1x128_pow2). */
MOE_API moe_status moe_grouped_gemm_mxfp8_gather(int32_t n_groups, const int32_t* offs, int64_t rows,
                                                 int32_t N, int32_t Kdim, const int32_t* perm_tok,
                                                 int64_t T, const uint8_t* X, const float* Xs,
                                                 const uint8_t* W, const float* Ws, int32_t epilogue,
                                                 void* out, float* out_s, moe_stream_t stream);

/* The same grouped GEMM with FP32 operands and no scales (FP32 mode):
 *  A [rows, Kdim] FP32; W [n_groups, N, Kdim] FP32; SWIGLU_QUANT writes h [rows, N/2] FP32
 *  (no quantisation); STORE writes out [rows, N] FP32. */
MOE_API moe_status moe_grouped_gemm_f32(int32_t n_groups, const int32_t* offs, int64_t rows,
                                int32_t N, int32_t Kdim, const float* A, const float* W,
                                int32_t epilogue, float* out, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/* a7. [P1] §2.2 (MoEGate weights) and §2.3 (reverse exchange), [P2] §3.1 (BF16 combine):
 * for every token t,
 *   y[t] = sum_{k=0..K-1} topk_w[t,k] * yexp[row_of[t,k]] + yshared[t]   (shared, if S)
 * accumulated in FP32 in slot order, shared expert last, rounded once to the output type.
 * A slot whose row_of lies outside [0, T*K) (-1: dropped by moe_permute) adds nothing.
 *  yexp [T*K, H] routed expert rows, BF16 (FP8 mode) or FP32 (FP32 mode); row_of [T, K];
 *  topk_w [T, K]; yshared [T, H] the shared expert's rows, same type (required when
 *  has_shared, NULL otherwise; moe_forward passes the rows T*K.. of its expert output);
 *  y [T, H] same type as yexp.  16-byte aligned. */
MOE_API moe_status moe_combine(const moe_config* cfg, int64_t T, const void* yexp,
                       const int32_t* row_of, const float* topk_w, const void* yshared,
                       void* y, moe_stream_t stream);

/* Row gather for the expert-parallel dispatch ([P1] §2.3: the rows of the tokens routed to
 * the experts of each destination, in the permutation's order): dst[r] = src[idx[r]] for
 * r < n_rows, a zero row where idx[r] < 0.  row_bytes a multiple of 16; src, dst 16-byte
 * aligned; idx [n_rows] int32 with entries < the row count of src. */
MOE_API moe_status moe_gather_rows(int64_t n_rows, int64_t row_bytes, const int32_t* idx, const void* src,
                                   void* dst, moe_stream_t stream);

/* a8. Load-driven selection-bias update (the bias "adjusted from real-time load" of
 * [P1] §2.2): bias[i] += 1e-3 * sign(T*K/E - counts[i]), with the sign taken in integers
 * (sign(T*K - E*counts[i])).  counts [E] int32, bias [E] FP32 updated in place. */
MOE_API moe_status moe_bias_update(const moe_config* cfg, int64_t T, const int32_t* counts,
                           float* bias, moe_stream_t stream);

/* The whole layer forward ([P1] §2.2 MoEGate and the layer's routed + shared experts;
 * [P1] §2.3 dispatch and combine, done on one GPU as a permutation and a gather; [P2] §3.1
 * 8 routed + 1 shared expert per token; [P2] §3.2 the fine-grained FP8 expert GEMMs) on one
 * stream: gate (a1), quantisation (a2, FP8 mode; in the gate's pass from
 * MOE_GATE_QUANT_MIN_TOKENS tokens up where moe_gate_quant takes the shape),
 * permutation (a3), grouped GEMM with SwiGLU (a4), grouped GEMM down-projection (a5), with
 * the shared expert as the last group (a6), combine (a7) and, if update_bias != 0, the bias
 * update (a8) after routing.
 *  x [T, H] BF16 (FP8) / FP32 (FP32); w: the weights; bias [E] FP32 (updated in place
 *  when update_bias); outputs y [T, H] (type of x), topk_idx [T, K], topk_w [T, K],
 *  counts [E] (the load histogram); ws/ws_bytes from moe_workspace_size(cfg, T). */
MOE_API moe_status moe_forward(const moe_config* cfg, int64_t T, const void* x, const moe_weights* w,
                       float* bias, int32_t update_bias, void* y, int32_t* topk_idx,
                       float* topk_w, int32_t* counts, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* The layer forward from and to HOST memory, pipelined across batches (a serving loop's
 * shape; the pages' layer has no host interface, this is a library convenience).  Each
 * batch's tokens are uploaded on a copy stream, run through moe_forward on the caller's
 * stream and its outputs downloaded on a second copy stream, so that batch n+1's upload and
 * batch n-1's download overlap batch n's compute.  Two device slots alternate between
 * consecutive batches; batches compute in submission order (a bias update by batch n is seen
 * by batch n+1).
 *  Ownership: the caller allocates the device workspace (moe_pipeline_workspace_size bytes
 *  for batches of up to max_T tokens, 16-byte aligned) and keeps it, the weights and the
 *  bias alive until moe_pipeline_destroy; the pipeline object owns two CUDA streams and a few
 *  events (host-side handles) and no device memory.  Work enqueued on `stream` before
 *  moe_pipeline_create completes before the pipeline touches the workspace.
 *  Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to
 *  be asynchronous; a submit returns once its work is enqueued, and the host buffers of a
 *  batch may be reused after moe_pipeline_wait (or once later batches' waits show it done).
 *  Errors: MOE_ERR_INVALID_ARG (bad pointer or T > max_T), MOE_ERR_WORKSPACE, MOE_ERR_CUDA. */
typedef struct moe_pipeline moe_pipeline;
MOE_API moe_status moe_pipeline_workspace_size(const moe_config* cfg, int64_t max_T, size_t* bytes);
MOE_API moe_status moe_pipeline_create(const moe_config* cfg, int64_t max_T, void* ws, size_t ws_bytes,
                                       moe_stream_t stream, moe_pipeline** out);
/* x_host [T, H] (BF16 / FP32 by mode); outputs y_host [T, H], topk_idx_host [T, K],
 * topk_w_host [T, K], counts_host [E] (the batch's histogram), all host memory; w and bias
 * as for moe_forward (device). */
MOE_API moe_status moe_pipeline_submit(moe_pipeline* pl, int64_t T, const void* x_host, const moe_weights* w,
                                       float* bias, int32_t update_bias, void* y_host, int32_t* topk_idx_host,
                                       float* topk_w_host, int32_t* counts_host);
/* Blocks the host until every submitted batch's outputs are in host memory. */
MOE_API moe_status moe_pipeline_wait(moe_pipeline* pl);
/* Waits for the pipeline's work, then releases its streams and events (NULL: no-op). */
MOE_API moe_status moe_pipeline_destroy(moe_pipeline* pl);

/* LogFMT-nBit, the logarithmic code for the combine payload ([P2] §3.2, LogFMT communication
 * compression), for 1x128 tiles of a BF16 matrix.  Per tile: min and max of the natural logs
 * of the non-zero magnitudes (min held above max - ln 2^32) and Step = (max - min) /
 * (2^(n-1) - 2); each value gets the n-bit code S|K, S its sign bit and K the index of the
 * value of the grid {0} u {exp(min + Step (K - 1)) : K = 1 .. 2^(n-1) - 1} nearest to its
 * magnitude in linear space (ties to the larger K); a tile of zeros has min = Step = 0, a tile
 * of one magnitude Step = 0 and K = 1.
 *  n_bits: 3 .. 12 (the précis evaluates 8 and 10; above 12 the FP32 tile metadata cannot
 *  place the grid to a fraction of its step).  x [rows, cols] BF16, cols % 128 == 0;
 *  codes [rows, cols]: uint8 for n_bits <= 8, uint16 otherwise; lmin, step [rows, cols/128]
 *  FP32 (the tile metadata).
 *  x and codes 16-byte aligned.  rows == 0 enqueues nothing. */
MOE_API moe_status moe_logfmt_encode(int32_t n_bits, int64_t rows, int64_t cols, const uint16_t* x,
                                     void* codes, float* lmin, float* step, moe_stream_t stream);

/* The inverse: y = (S ? -1 : 1) * (K ? exp(min + Step (K - 1)) : 0), rounded to BF16.
 *  Same shapes and rules as moe_logfmt_encode; y [rows, cols] BF16, 16-byte aligned. */
MOE_API moe_status moe_logfmt_decode(int32_t n_bits, int64_t rows, int64_t cols, const void* codes,
                                     const float* lmin, const float* step, uint16_t* y,
                                     moe_stream_t stream);

/* Device-side error word written by bounded waits inside the kernels (0 = none).  Reading
 * it synchronises the device.  *code receives the word; the call then clears it.
 *  Bounded waits: 0x101-0x104 (FP32-scale GEMM), 0x111-0x114 (power-of-two GEMM), gate
 *  codes, 0x1ff (moe_selftest_wait_timeout).
 *  libmoe_checks.so, the same sources built with -DMOE_CHECKS (no counterpart on the pages:
 *  a debug build in place of a memory checker), also checks the indices that callers pass in
 *  and the permutation's own positions; a failed check records its code and skips the access
 *  (the first failure of a kind wins):
 *   0x121 / 0x122  a grouped GEMM's offs not 0 <= offs[g] <= offs[g+1] <= rows (the CTA runs
 *                  no tile); FP32-scale / power-of-two GEMM
 *   0x131 / 0x132  a gathered GEMM's perm_tok entry neither -1 nor in [0, T) (read as a zero row)
 *   0x301          a permutation position outside [0, T*K) (not reachable through the ABI)
 *   0x302          a combine row_of entry neither -1 nor in [0, T*K) (the slot is skipped)
 *  The default libmoe.so compiles these checks away.  It clamps the gathered GEMM's token
 *  indices the same way, and the combine skips out-of-range rows, but a GEMM given unusable
 *  offs reads and writes out of bounds. */
MOE_API moe_status moe_device_error(int32_t* code);

/* Self-test of the bounded-wait error path (no counterpart on the pages): one thread of a
 * one-block kernel waits on an mbarrier that nothing arrives at, gives up after
 * budget_cycles SM clock cycles (1 .. 4e9) and records error word 0x1ff, which the next
 * moe_device_error returns.  Nothing traps or hangs; the context stays usable. */
MOE_API moe_status moe_selftest_wait_timeout(int64_t budget_cycles, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
