// pipeline.cu -- the layer forward from and to host memory, with the copies of one batch
// overlapping the compute of its neighbours.
//
// The layer is per-token independent, but splitting one batch into small chunks would starve
// the grouped GEMMs (fewer rows per expert, more padded tiles), so the overlap is across
// batches instead: batch n's upload runs on a copy stream while batch n-1 computes, and
// batch n-1's results go back on a second copy stream while batch n computes.  Two device
// slots (x, y, routing, histogram) alternate between consecutive batches; the layer
// workspace is shared because the batches compute one after another on the caller's stream.
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

struct moe_pipeline {
    moe_config cfg;
    int64_t max_T;
    cudaStream_t compute;   // the caller's stream
    cudaStream_t h2d, d2h;  // owned
    cudaEvent_t ev_h2d[2], ev_comp[2], ev_d2h[2];
    cudaEvent_t ev_ready;   // the caller's work enqueued before create
    char* ws;               // caller's workspace
    size_t layer_ws_bytes;
    size_t slot_off[2];
    size_t off_x, off_y, off_idx, off_w, off_cnt;  // within a slot
    int64_t n_submitted;
};

namespace {

size_t align_kb(size_t v) { return (v + 1023) & ~static_cast<size_t>(1023); }

// Layout: [layer workspace for max_T tokens][slot 0][slot 1]; a slot holds x [T, H],
// y [T, H], topk_idx [T, K], topk_w [T, K] and counts [E] for max_T tokens.
void pipeline_layout(const moe_config& c, int64_t max_T, size_t* layer, size_t* slot, size_t* off) {
    const size_t esz = c.mode == MOE_FP32 ? 4 : 2;
    const size_t xb = static_cast<size_t>(max_T) * c.hidden * esz;
    const size_t ib = static_cast<size_t>(max_T) * c.top_k * 4;
    *layer = align_kb(moe::ws_layout(c, max_T).total);
    size_t o = 0;
    off[0] = o; o = align_kb(o + xb);   // x
    off[1] = o; o = align_kb(o + xb);   // y
    off[2] = o; o = align_kb(o + ib);   // topk_idx
    off[3] = o; o = align_kb(o + ib);   // topk_w
    off[4] = o; o = align_kb(o + static_cast<size_t>(c.n_experts) * 4);  // counts
    *slot = o;
}

}  // namespace

extern "C" moe_status moe_pipeline_workspace_size(const moe_config* cfg, int64_t max_T, size_t* bytes) {
    if (!moe::config_ok(cfg) || max_T < 1 || !bytes) return MOE_ERR_INVALID_ARG;
    size_t layer, slot, off[5];
    pipeline_layout(*cfg, max_T, &layer, &slot, off);
    *bytes = layer + 2 * slot;
    return MOE_OK;
}

extern "C" moe_status moe_pipeline_create(const moe_config* cfg, int64_t max_T, void* ws, size_t ws_bytes,
                                          moe_stream_t stream, moe_pipeline** out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    size_t need = 0;
    MOE_TRY(moe_pipeline_workspace_size(cfg, max_T, &need));
    if (!ws || !moe::aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < need) return MOE_ERR_WORKSPACE;
    moe_pipeline* pl = static_cast<moe_pipeline*>(calloc(1, sizeof(moe_pipeline)));
    if (!pl) return MOE_ERR_INVALID_ARG;
    pl->cfg = *cfg;
    pl->max_T = max_T;
    pl->compute = reinterpret_cast<cudaStream_t>(stream);
    pl->ws = static_cast<char*>(ws);
    size_t slot, off[5];
    pipeline_layout(*cfg, max_T, &pl->layer_ws_bytes, &slot, off);
    pl->slot_off[0] = pl->layer_ws_bytes;
    pl->slot_off[1] = pl->layer_ws_bytes + slot;
    pl->off_x = off[0];
    pl->off_y = off[1];
    pl->off_idx = off[2];
    pl->off_w = off[3];
    pl->off_cnt = off[4];
    bool ok = cudaStreamCreateWithFlags(&pl->h2d, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaStreamCreateWithFlags(&pl->d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (int k = 0; k < 2 && ok; ++k) {
        ok = cudaEventCreateWithFlags(&pl->ev_h2d[k], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&pl->ev_comp[k], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&pl->ev_d2h[k], cudaEventDisableTiming) == cudaSuccess;
    }
    ok = ok && cudaEventCreateWithFlags(&pl->ev_ready, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventRecord(pl->ev_ready, pl->compute) == cudaSuccess;
    if (!ok) {
        moe_pipeline_destroy(pl);
        return MOE_ERR_CUDA;
    }
    *out = pl;
    return MOE_OK;
}

extern "C" moe_status moe_pipeline_submit(moe_pipeline* pl, int64_t T, const void* x_host, const moe_weights* w,
                                          float* bias, int32_t update_bias, void* y_host, int32_t* topk_idx_host,
                                          float* topk_w_host, int32_t* counts_host) {
    if (!pl || T < 0 || T > pl->max_T || !w || !bias || !counts_host) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x_host || !y_host || !topk_idx_host || !topk_w_host)) return MOE_ERR_INVALID_ARG;
    const moe_config& c = pl->cfg;
    const int k = static_cast<int>(pl->n_submitted & 1);
    char* slot = pl->ws + pl->slot_off[k];
    void* x = slot + pl->off_x;
    void* y = slot + pl->off_y;
    int32_t* idx = reinterpret_cast<int32_t*>(slot + pl->off_idx);
    float* tw = reinterpret_cast<float*>(slot + pl->off_w);
    int32_t* cnt = reinterpret_cast<int32_t*>(slot + pl->off_cnt);
    const size_t esz = c.mode == MOE_FP32 ? 4 : 2;
    const size_t xb = static_cast<size_t>(T) * c.hidden * esz;
    const size_t ib = static_cast<size_t>(T) * c.top_k * 4;
    // upload: x slot k is free once batch n-2 finished computing (the first two batches wait
    // for the caller's earlier work on the stream instead)
    MOE_CUDA_CHECK(cudaStreamWaitEvent(pl->h2d, pl->n_submitted < 2 ? pl->ev_ready : pl->ev_comp[k], 0));
    if (xb) MOE_CUDA_CHECK(cudaMemcpyAsync(x, x_host, xb, cudaMemcpyHostToDevice, pl->h2d));
    MOE_CUDA_CHECK(cudaEventRecord(pl->ev_h2d[k], pl->h2d));
    // compute: after the upload, and once batch n-2's outputs have left slot k
    MOE_CUDA_CHECK(cudaStreamWaitEvent(pl->compute, pl->ev_h2d[k], 0));
    MOE_CUDA_CHECK(cudaStreamWaitEvent(pl->compute, pl->ev_d2h[k], 0));
    MOE_TRY(moe_forward(&c, T, x, w, bias, update_bias, y, idx, tw, cnt, pl->ws, pl->layer_ws_bytes,
                        reinterpret_cast<moe_stream_t>(pl->compute)));
    MOE_CUDA_CHECK(cudaEventRecord(pl->ev_comp[k], pl->compute));
    // download
    MOE_CUDA_CHECK(cudaStreamWaitEvent(pl->d2h, pl->ev_comp[k], 0));
    if (xb) MOE_CUDA_CHECK(cudaMemcpyAsync(y_host, y, xb, cudaMemcpyDeviceToHost, pl->d2h));
    if (ib) {
        MOE_CUDA_CHECK(cudaMemcpyAsync(topk_idx_host, idx, ib, cudaMemcpyDeviceToHost, pl->d2h));
        MOE_CUDA_CHECK(cudaMemcpyAsync(topk_w_host, tw, ib, cudaMemcpyDeviceToHost, pl->d2h));
    }
    MOE_CUDA_CHECK(cudaMemcpyAsync(counts_host, cnt, static_cast<size_t>(c.n_experts) * 4, cudaMemcpyDeviceToHost,
                                   pl->d2h));
    MOE_CUDA_CHECK(cudaEventRecord(pl->ev_d2h[k], pl->d2h));
    ++pl->n_submitted;
    return MOE_OK;
}

extern "C" moe_status moe_pipeline_wait(moe_pipeline* pl) {
    if (!pl) return MOE_ERR_INVALID_ARG;
    MOE_CUDA_CHECK(cudaStreamSynchronize(pl->d2h));
    return MOE_OK;
}

extern "C" moe_status moe_pipeline_destroy(moe_pipeline* pl) {
    if (!pl) return MOE_OK;
    moe_status st = MOE_OK;
    if (pl->d2h && cudaStreamSynchronize(pl->d2h) != cudaSuccess) st = MOE_ERR_CUDA;
    if (pl->h2d && cudaStreamSynchronize(pl->h2d) != cudaSuccess) st = MOE_ERR_CUDA;
    for (int k = 0; k < 2; ++k) {
        if (pl->ev_h2d[k]) cudaEventDestroy(pl->ev_h2d[k]);
        if (pl->ev_comp[k]) cudaEventDestroy(pl->ev_comp[k]);
        if (pl->ev_d2h[k]) cudaEventDestroy(pl->ev_d2h[k]);
    }
    if (pl->ev_ready) cudaEventDestroy(pl->ev_ready);
    if (pl->h2d) cudaStreamDestroy(pl->h2d);
    if (pl->d2h) cudaStreamDestroy(pl->d2h);
    free(pl);
    return st;
}
