// smoe_internal.h -- host-side launchers behind the C ABI (one per step); each returns the CUDA error of its launches.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "smoe.h"

namespace smoe {

// a failed CUDA runtime call: remembered for smoe_last_error_string and cleared; returns SMOE_ERR_CUDA
smoe_status note_cuda_error(cudaError_t err);

size_t group_work_bytes(int64_t n, int E);

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int K, int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_group(const int32_t* ids, int64_t n, int K, int E, int32_t* counts, int32_t* offsets,
                         int32_t* src, int32_t* slot, int32_t* tiles, int32_t* hist, cudaStream_t s);
cudaError_t launch_quantize_q8(const float* x, int64_t rows, int cols, int8_t* codes, uint16_t* scales,
                               cudaStream_t s);
cudaError_t launch_swiglu_requant(const float* gu, int64_t n, int F, int8_t* hc, uint16_t* hs, uint16_t* hop,
                                  cudaStream_t s);
cudaError_t launch_pack_q2(const uint8_t* codes, const uint16_t* scales, const smoe_q2w* desc, int E, int rows,
                           int cols, int half, uint8_t* packed, int32_t* status, cudaStream_t s);
cudaError_t launch_gather_q8(const int8_t* codes, const uint16_t* scales, int64_t in_rows, int cols,
                             const int32_t* src, int64_t n, uint16_t* out, cudaStream_t s);
cudaError_t launch_combine(const float* dm, const int32_t* slot, const float* w, int64_t T, int K, int H,
                           const float* ds, const float* sg, float* y, cudaStream_t s);
cudaError_t launch_combine_h(const uint16_t* dm, const int32_t* slot, const float* w, int64_t T, int K, int H,
                             float* y, cudaStream_t s);
cudaError_t launch_router_topk(const float* x, const uint16_t* wr, int64_t T, int H, int E, int K, uint16_t* work,
                               int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_shared_gate(const float* x, const float* wsg, int64_t T, int H, float* sg, cudaStream_t s);

// Grouped expert product (both the gate/up and the down step): for every tile of the tile list and every 128-row
// slice of the expert's weight matrix, OUT[row][j] = sum over K of W[e][j][i] * B[row][i], W the decoded 2-bit
// weights and B = d q the q8 rows, given as the exact fp16 split hi + lo.
struct ExpertsGemmArgs {
    const uint16_t* bop;  // B rows in operand form: fp16 planes [2][b_rows][K] (hi, then lo), routed-row order
    int32_t* tiles;       // tile list; header[3] receives SMOE_ERR_TIMEOUT
    const uint8_t* wp;    // packed weights: per (expert, 128-row tile, 64-value slice) 2560 bytes
    int a_rows;           // weight rows per expert (2F or H)
    int K;                // contraction length (H or F)
    float* out;           // [b_rows][a_rows] (null in SwiGLU mode)
    int64_t b_rows;       // n
    int n_experts;        // E
    bool two_level;       // add every 64-wide K slice into fp32 registers (gate/up); else one accumulator over K
    int cluster;          // CTAs per cluster: 2 (a CTA pair) or 1 (set by the launcher)
    // SwiGLU mode (gate/up with weights packed interleaved): h = silu(gate) * up requantised in the epilogue
    int8_t* hc;           // [b_rows][a_rows / 2] q8 codes of h, or null: fp32 rows to `out`
    uint16_t* hs;         // [b_rows][a_rows / 64] fp16 scales
    uint16_t* hop;        // [2][b_rows][a_rows / 2] h in operand form
    int max_tiles = 0;    // entries the tile list holds (set by the launcher): a larger header count is an error
    uint16_t* out_h = nullptr;  // fp16 rows [b_rows][a_rows] in place of `out` (the down product's narrow form)
};
cudaError_t launch_experts_gemm(const ExpertsGemmArgs& a, int64_t max_tiles, cudaStream_t s);

}  // namespace smoe
