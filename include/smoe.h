/* smoe.h -- C ABI of libsmoe: the prompt-chunk (prefill) routed-expert block of a mixture-of-experts layer on one
 * GB300 (sm_103a).
 *
 * The block, for a chunk of T tokens of hidden size H, E experts, top-K routing and expert FFN width F, runs as these
 * eight calls in this order (each the step of the same name in the Strata engine's prompt path -- page
 * "src/prefill/prefill.cpp", Prefill::run, MoE half -- and its fused int8 expert contract -- page "Strata compare
 * v0.1.35...v0.1.37", include/strata/prefill/moe_fused.hpp):
 *
 *   smoe_route_topk      router softmax, top-K of the E logits, weights renormalised over the K
 *   smoe_group           stable counting sort of the T*K (token, k) pairs by expert: counts, offsets, src, slot, tiles
 *   smoe_quantize_q8     activations to int8 once per token, one fp16 scale per 32 values
 *   smoe_gather_q8       the q8 rows of the routed pairs in routed-row order, in operand form
 *   smoe_experts_gateup  grouped gate/up product of each routed row against its expert's 2-bit weights
 *   smoe_swiglu_requant  h = silu(gate) * up, requantised to int8 per 32 values
 *                        (smoe_experts_gateup_swiglu runs these two steps as one pass)
 *   smoe_experts_down    grouped down product into one fp32 row per routed pair
 *   smoe_combine         Y[t] = sum_k w[t][k] * Dm[slot[t*K+k]] (gather form, no atomics)
 *
 * With the shared expert (the same page's "shared expert and its scalar gate"): one more expert in the routed
 * experts' form that every token takes -- grouped by smoe_group with E = 1, K = 1 and all ids 0, gathered by
 * smoe_gather_q8, multiplied by smoe_experts_gateup / smoe_swiglu_requant / smoe_experts_down with E = 1 --, its
 * scalar gate from smoe_shared_gate, and smoe_combine_shared in place of smoe_combine.
 *
 * FORMATS (all row-major, little-endian):
 *   q8 activations   codes int8 [rows][cols] and scales fp16 (as uint16 bits) [rows][cols/32].  A block of 32 values
 *                    x has amax = max|x|, d = fp16_rne(amax / 127.0f) (IEEE fp32 division) and codes
 *                    q = clamp(roundf(x / float(d)), -127, 127) (IEEE fp32 division, roundf = half away from zero);
 *                    d == 0 gives all-zero codes.  The value of a code is d * q.
 *   Q2 weights       per matrix, all E experts contiguous: codes uint8 [E][rows][cols/4], weight 4j+i of a row in
 *                    bits 2i..2i+1 of byte j; scales fp16 [E][rows][cols/32].  The value of a weight is d * (q - 2),
 *                    q in {0,1,2,3}.  Gate/up matrix: rows [0, F) gate, [F, 2F) up, cols H.  Down matrix: rows H,
 *                    cols F.
 *   q8 operand form  the q8 values as the expert products read them: two fp16 planes [2][rows][cols], plane 0
 *                    hi = fp16_rn(d * q) and plane 1 lo = d * q - hi (exact: d * q has at most 18 significant
 *                    bits), and within every group of 16 values position 2j holds value j and position 2j+1 value
 *                    j+8 (j = 0..7).  hi + lo = d * q exactly.  Written by smoe_gather_q8 (routed activations) and
 *                    smoe_swiglu_requant (H).
 *   packed Q2        what the expert products read as weights (smoe_pack_q2 writes it once from the row-major form):
 *                    per (expert, 128-row tile, 64-value slice) a 2560-byte block = the tile's 128 rows x 16 code
 *                    bytes, then its 128 rows x 2 fp16 scales; blocks ordered by expert, tile, slice.
 *   tiles            int32 [4 + 4 * smoe_max_tiles(n, E)]: header {n_tiles, group_status, n, kernel_status}, then
 *                    per tile {expert, first row, rows, 0}; each expert's c rows split into ceil(c/192) near-equal
 *                    tiles [floor(i*c/nt), floor((i+1)*c/nt)), experts in id order.
 *
 * CONVENTIONS
 *   - Every pointer argument is a DEVICE pointer owned by the caller; the library allocates nothing and keeps no
 *     state between calls.  Every buffer must be 16-byte aligned.  The one exception is the block object
 *     (smoe_block_*, at the end of this header): it owns the device buffers, streams, events and CUDA graphs of a
 *     whole block and takes HOST pointers for its inputs and output.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream) and never
 *     synchronises with the host.
 *   - A call returns SMOE_OK or an error found on the host before anything is launched (a bad argument, an
 *     unsupported shape, a device that is not sm_103) or a launch error (SMOE_ERR_LAUNCH, with the CUDA error
 *     cleared).  Errors found on the device (a routed id outside [0, E), a kernel's internal wait that ran out) are
 *     written to the tiles header, which the caller reads after the stream has run:
 *     header[1] = SMOE_ERR_RANGE, header[3] = SMOE_ERR_TIMEOUT.  No call traps, asserts or exits.
 *   - Calls on different streams that share an output buffer race; the library does no locking.
 */
#ifndef SMOE_H
#define SMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int smoe_status;
#define SMOE_OK 0
#define SMOE_ERR_ARG 1          /* null or misaligned pointer, or a size out of range */
#define SMOE_ERR_LAUNCH 2       /* a kernel launch failed (cudaGetLastError was not cudaSuccess) */
#define SMOE_ERR_UNSUPPORTED 3  /* a shape the kernels do not cover, or a device other than sm_103 */
#define SMOE_ERR_RANGE 4        /* (device, tiles header[1]) a routed id outside [0, E) */
#define SMOE_ERR_TIMEOUT 5      /* (device, tiles header[3]) a kernel's internal wait gave up; outputs undefined */
#define SMOE_ERR_CUDA 6         /* (smoe_block_*) a CUDA runtime call failed: an allocation, a copy, a stream, event
                                   or graph operation; smoe_last_error_string() names the CUDA error */

/* Largest supported sizes. */
#define SMOE_MAX_EXPERTS 1024
#define SMOE_MAX_TOPK 32
#define SMOE_TILE_ROWS 192

/* Human-readable name of a status code (static storage). */
const char* smoe_status_string(smoe_status s);

/* Name of the CUDA error behind this thread's most recent SMOE_ERR_LAUNCH (static storage; "no error" before any). */
const char* smoe_last_error_string(void);

/* SMOE_OK when the current CUDA device is an sm_103 part the kernels were built for. */
smoe_status smoe_device_check(void);

/* Most tiles smoe_group can emit for n pairs over E experts: ceil(n / 192) + min(E, n). */
int64_t smoe_max_tiles(int64_t n, int E);
/* Bytes of the tiles buffer: 16 * (1 + smoe_max_tiles(n, E)). */
size_t smoe_tiles_bytes(int64_t n, int E);
/* Bytes of smoe_group's scratch space for n pairs over E experts. */
size_t smoe_group_work_bytes(int64_t n, int E);

/* Step 1 -- route.  Page "src/prefill/prefill.cpp", Prefill::run, MoE half: route(logits, ids, w, T, n_expert) after
 * the router projection; the engine's "fused 512-expert top-10 router".
 *   logits  fp32 [T][E] router logits (finite).
 *   ids     int32 [T][K] out: the K largest logits of each token, largest first; ties go to the lower expert id
 *           (the engine's top-k tie rule, page "Strata compare v0.1.35...v0.1.37", qsa_select.hpp).
 *   w       fp32 [T][K] out: softmax restricted to the K and renormalised,
 *           w_k = exp(l_k - l_1) / sum_j exp(l_j - l_1) (the full softmax denominator cancels).
 *   1 <= K <= min(E, 32), 1 <= E <= 1024, T >= 0 (T == 0 launches nothing). */
smoe_status smoe_route_topk(const float* logits, int64_t T, int E, int K, int32_t* ids, float* w, void* stream);

/* Step 2 -- group.  Page "src/prefill/prefill.cpp", Prefill::run: the host loop that groups the (token, k) pairs by
 * expert (counts, exclusive offsets, then in pair order slot[i] = the next row of expert ids[i] and
 * src[row] = i / K); page "Strata compare v0.1.35...v0.1.37", moe_fused.hpp group(): the same tables built on the
 * GPU, plus a tile list, so that the host never waits for the routing.  The order is stable (by pair index).
 *   ids      int32 [T][K] (n = T*K pairs, pair i = t*K + k).
 *   counts   int32 [E] out;  offsets int32 [E+1] out (offsets[E] = n);  src int32 [n] out;  slot int32 [n] out.
 *   tiles    int32 out, tiles_bytes >= smoe_tiles_bytes(n, E).
 *   work     scratch, work_bytes >= smoe_group_work_bytes(n, E); its contents are undefined afterwards.
 * An id outside [0, E) sets tiles header[1] = SMOE_ERR_RANGE; the pair is then left out of every table and the
 * expert calls do no work for that chunk. */
smoe_status smoe_group(const int32_t* ids, int64_t T, int K, int E, int32_t* counts, int32_t* offsets, int32_t* src,
                       int32_t* slot, int32_t* tiles, size_t tiles_bytes, void* work, size_t work_bytes,
                       void* stream);

/* smoe_group without a caller-provided scratch buffer (the paper has no counterpart: this is a library service).
 * For callers that cannot allocate device memory themselves -- e.g. a runtime whose device memory is planned once up
 * front, or a serving loop that must not call cudaMalloc between requests because it can synchronise the device.
 * Same arguments, outputs and errors as smoe_group, minus `work`: the scratch (at most 48 x 1024 int32 counts,
 * 192 KiB) lives in a __device__ array inside the library that every GPU loading it keeps until the process exits.
 * No cudaMalloc, cudaFree or allocating routine is called.  The first call on a device looks the array's device
 * address up (cudaGetSymbolAddress, with that device current); make that first call before any stream capture.
 * The address is kept with the identity of the device's context: the first call after that context was destroyed
 * (cudaDeviceReset) looks it up again, so it too belongs before any capture.
 * Every call on a device shares the one array: calls whose kernels overlap on the GPU race and give wrong tables.
 * A size whose scratch would not fit is refused with SMOE_ERR_UNSUPPORTED (no valid T, K, E reaches it). */
smoe_status smoe_group_noalloc(const int32_t* ids, int64_t T, int K, int E, int32_t* counts, int32_t* offsets,
                               int32_t* src, int32_t* slot, int32_t* tiles, size_t tiles_bytes, void* stream);

/* Step 3 -- q8 activations.  Page "Strata compare v0.1.35...v0.1.37", moe_fused.hpp quantize_act: the layer input is
 * rounded to int8 once per TOKEN (not per routed slot) with one scale per 32 values.
 *   x fp32 [rows][cols] (|x| < 65504) -> codes int8 [rows][cols], scales fp16 [rows][cols/32].  cols % 32 == 0. */
smoe_status smoe_quantize_q8(const float* x, int64_t rows, int cols, int8_t* codes, uint16_t* scales, void* stream);

/* Weight preparation (once per weight set): the row-major Q2 matrices of E experts (codes [E][rows][cols/4], scales
 * [E][rows][cols/32]) into the packed form the expert products read.  rows % 128 == 0, cols % 64 == 0.
 * packed: smoe_pack_q2_bytes(E, rows, cols) bytes (the same size as codes + scales). */
smoe_status smoe_pack_q2(const uint8_t* codes, const uint16_t* scales, int E, int rows, int cols, uint8_t* packed,
                         void* stream);
size_t smoe_pack_q2_bytes(int E, int rows, int cols);

/* Weight preparation for the fused gate/up + SwiGLU product (smoe_experts_gateup_swiglu): the row-major Q2 gate/up
 * matrix of E experts (codes [E][2F][H/4], scales [E][2F][H/32]; rows [0, F) gate, [F, 2F) up) packed with gate and
 * up rows interleaved: packed 128-row tile m holds outputs j in [64m, 64m + 64), its row 32a + l being gate row
 * 64m + 16a + l (l < 16) or up row F + 64m + 16a + l - 16 (l >= 16).  F % 64 == 0, H % 64 == 0.
 * packed: smoe_pack_q2_bytes(E, 2F, H) bytes. */
smoe_status smoe_pack_q2_swiglu(const uint8_t* codes, const uint16_t* scales, int E, int F, int H, uint8_t* packed,
                                void* stream);

/* Step 4a -- routed rows of the q8 activations.  moe_fused.hpp experts() reads each routed row's activations
 * "through the rows of group": this call lays them out once in routed-row order and operand form, so that every
 * tile of the expert products reads its rows as one contiguous block.
 *   codes, scales  int8 [in_rows][cols] and fp16 [in_rows][cols/32] (from smoe_quantize_q8).
 *   src      int32 [n], from smoe_group; every entry in [0, in_rows) (an entry outside it is not read: its output rows
 *            are zero-filled and the call still returns SMOE_OK, which a bad grouping has already reported).
 *   out      fp16 [2][n][cols] out, operand form: row r = row src[r].   cols % 32 == 0. */
smoe_status smoe_gather_q8(const int8_t* codes, const uint16_t* scales, int64_t in_rows, int cols, const int32_t* src,
                           int64_t n, uint16_t* out, void* stream);

/* Step 4b -- grouped gate/up.  moe_fused.hpp experts(): gate/up of the routed rows; per routed row r of expert e and
 * output j in [0, 2F):
 *   GU[r][j] = sum_b dX[src r][b] * dW[e][j][b] * sum_{i in block b} (qW - 2) * qX[src r][i]     (fp32 result)
 *   xop      the routed rows in operand form, fp16 [2][n][H] (from smoe_gather_q8).
 *   tiles    from smoe_group (header[3] receives SMOE_ERR_TIMEOUT, or SMOE_ERR_ARG when its tile count exceeds
 *            smoe_max_tiles(n, E): then no tile is read and nothing is written).   n = T*K (sizes the launch).
 *   wgu      gate/up weights [E][2F][H] packed by smoe_pack_q2.
 *   gu       fp32 [n][2F] out, row r = routed row r.
 *   H % 128 == 0, F % 64 == 0. */
smoe_status smoe_experts_gateup(const uint16_t* xop, int32_t* tiles, int64_t n, int E, const uint8_t* wgu, int H, int F,
                                float* gu, void* stream);

/* Steps 4b + 5 fused -- gate/up, SwiGLU and requantisation in one pass (the SwiGLU runs in the product's epilogue on
 * the fp32 gate and up values; GU is never written).  Same arguments as smoe_experts_gateup with the weights packed
 * by smoe_pack_q2_swiglu, and the outputs of smoe_swiglu_requant:
 *   hc int8 [n][F], hs fp16 [n][F/32], hop fp16 [2][n][F] (operand form).
 * h_j = silu(GU_j) * GU_{F+j} in fp32 and the q8 rule with the scale computed exactly as in smoe_swiglu_requant
 * (IEEE amax / 127); h and the codes use a reciprocal where that step divides, so a code can differ from
 * smoe_swiglu_requant's only next to a .5 tie.  GU is the same fp32 sum as smoe_experts_gateup computes. */
smoe_status smoe_experts_gateup_swiglu(const uint16_t* xop, int32_t* tiles, int64_t n, int E, const uint8_t* wgs, int H,
                                       int F, int8_t* hc, uint16_t* hs, uint16_t* hop, void* stream);

/* One expert's 2-bit weight matrix in the row-major Q2 form (page "Strata compare v0.1.35...v0.1.37", moe_fused.hpp
 * experts(): the batch carries one weight blob pointer per expert): codes uint8 [rows][cols/4] and scales fp16 bits
 * [rows][cols/32], each pointer 16-byte aligned. */
typedef struct {
    const uint8_t* codes;
    const uint16_t* scales;
} smoe_q2w;

/* Bytes of the scratch of smoe_experts_gateup_q8 / smoe_experts_down_q8 for n routed rows (one size serves both). */
size_t smoe_experts_q8_work_bytes(int64_t n, int E, int H, int F);

/* Step 4 in the form of moe_fused.hpp experts(batch, ..., Xq, src, ...): the grouped gate/up product straight from the
 * per-token q8 activations and the routed rows' token indices, with the weights given per expert.
 *   xc, xs   int8 [in_rows][H] and fp16 [in_rows][H/32], from smoe_quantize_q8.
 *   src      int32 [n], from smoe_group: routed row r reads token src[r] (entries outside [0, in_rows) read zeros).
 *   tiles    from smoe_group (header[3] receives SMOE_ERR_TIMEOUT, or SMOE_ERR_ARG when a descriptor is null or
 *            misaligned: that expert's weights are then taken as zero).
 *   w_gu     DEVICE array of E descriptors, expert e's gate/up matrix [2F][H] (rows [0, F) gate, [F, 2F) up).
 *   work     caller scratch of smoe_experts_q8_work_bytes(n, E, H, F) bytes: the call lays the routed rows out in the
 *            operand form and packs the weights there, then runs smoe_experts_gateup's product.  A caller that calls
 *            repeatedly with the same weights saves the packing by calling smoe_pack_q2 once and smoe_experts_gateup.
 *   gu       fp32 [n][2F] out, exactly as smoe_experts_gateup computes it.   H % 128 == 0, F % 64 == 0. */
smoe_status smoe_experts_gateup_q8(const int8_t* xc, const uint16_t* xs, int64_t in_rows, const int32_t* src,
                                   int32_t* tiles, int64_t n, int E, const smoe_q2w* w_gu, int H, int F, void* work,
                                   size_t work_bytes, float* gu, void* stream);

/* Step 6 in the same form: the grouped down product from planar q8 H (routed-row order) and per-expert weights.
 *   hc, hs   int8 [n][F] and fp16 [n][F/32], from smoe_swiglu_requant.
 *   w_d      DEVICE array of E descriptors, expert e's down matrix [H][F].
 *   tiles, work as smoe_experts_gateup_q8;  dm fp32 [n][H] out, exactly as smoe_experts_down computes it. */
smoe_status smoe_experts_down_q8(const int8_t* hc, const uint16_t* hs, int32_t* tiles, int64_t n, int E,
                                 const smoe_q2w* w_d, int H, int F, void* work, size_t work_bytes, float* dm,
                                 void* stream);

/* Step 5 -- SwiGLU and requantisation.  Page "src/prefill/prefill.cpp": mmq::swiglu(GU, H, rows, ...) then the
 * int8 rounding of H; moe_fused.hpp: "SwiGLU, H as int8".
 *   gu fp32 [n][2F] -> h_j = silu(gu[r][j]) * gu[r][F + j] (fp32; silu(g) = g / (1 + exp(-g))), then the q8 rule:
 *   hc int8 [n][F], hs fp16 [n][F/32].  F % 32 == 0.
 *   hop      optional (NULL: not written): H in operand form, fp16 [2][n][F]; needs F % 64 == 0. */
smoe_status smoe_swiglu_requant(const float* gu, int64_t n, int F, int8_t* hc, uint16_t* hs, uint16_t* hop,
                                void* stream);

/* Step 6 -- grouped down.  moe_fused.hpp experts(): "down into dm [n][2560] FP32 at the rows of group":
 *   Dm[r][o] = sum_b dH[r][b] * dW[e][o][b] * sum_{i in block b} (qW - 2) * qH[r][i],   o in [0, H)
 *   hop      H in operand form, fp16 [2][n][F] (from smoe_swiglu_requant).   tiles from smoe_group.
 *   wd       down weights [E][H][F] packed by smoe_pack_q2.
 *   dm       fp32 [n][H] out.   H % 128 == 0, F % 64 == 0. */
smoe_status smoe_experts_down(const uint16_t* hop, int32_t* tiles, int64_t n, int E, const uint8_t* wd, int H, int F,
                              float* dm, void* stream);

/* Step 7 -- combine.  The combine that reads the per-slot rows (page "src/prefill/prefill.cpp", the engine's
 * "fused CUDA weighted reduction"): Y[t][o] = sum_{k=0}^{K-1} w[t][k] * dm[slot[t*K+k]][o], summed in k order in
 * fp32; each token gathers its own K rows, so no output is written twice and no atomics are used.
 *   dm fp32 [n][H], slot int32 [T*K], w fp32 [T][K] -> y fp32 [T][H].   H % 4 == 0. */
smoe_status smoe_combine(const float* dm, const int32_t* slot, const float* w, int64_t T, int K, int H, float* y,
                         void* stream);

/* Steps 6 and 7 with a narrow Dm (not the pages' form, which keeps the down rows in fp32; an option for layers whose
 * down outputs fit fp16): the down product stores each row as fp16, rounded to nearest from the same fp32 value that
 * smoe_experts_down writes (a value beyond the fp16 range becomes +-inf), and the combine reads fp16 rows.  This
 * halves the bytes of Dm that the down product writes and the combine reads again (839 MB each way at T=8192,
 * H=2560, K=10); each term of a token's sum then carries one more fp16 rounding (relative 2^-11 at most).
 *   smoe_experts_down_h: arguments as smoe_experts_down; dm_h fp16 bits [n][H] out.
 *   smoe_combine_h: arguments as smoe_combine, with dm_h fp16 bits [n][H]; the sum is fp32 in k order of the values
 *   widened from fp16.  H % 8 == 0. */
smoe_status smoe_experts_down_h(const uint16_t* hop, int32_t* tiles, int64_t n, int E, const uint8_t* wd, int H,
                                int F, uint16_t* dm_h, void* stream);
smoe_status smoe_combine_h(const uint16_t* dm_h, const int32_t* slot, const float* w, int64_t T, int K, int H,
                           float* y, void* stream);

/* Step 1 with the router projection fused in (the logits are never written).  Page "src/prefill/prefill.cpp",
 * Prefill::run, MoE half: the router is a BF16 projection of the hidden state, with the low part of its BF16 copy,
 * followed by route().  Here
 *   xh = bf16_rne(x), xl = bf16_rne(x - xh);  logit[t][e] = sum_h wr[e][h] * (xh[t][h] + xl[t][h])
 * accumulated in fp32 on the tensor cores, then the top-K and weights exactly as smoe_route_topk (ties to the lower
 * id; weights exp(l_k - l_1) / sum_j exp(l_j - l_1) over the K).
 *   x fp32 [T][H], wr bf16 (uint16 bits) [E][H] -> ids int32 [T][K], w fp32 [T][K].
 *   work: caller scratch of smoe_router_work_bytes(T, H) bytes (the split activations, bf16 [2][T][H], then the
 *   top-K candidates of the two halves of E when E > 256).
 *   H % 64 == 0; 16 <= E <= 512, E % 16 == 0 (E % 32 == 0 above 256); 1 <= K <= min(E, 16); all pointers
 *   16-byte aligned.
 *   If an internal wait gives up, the affected tokens get id -1, which smoe_group reports as SMOE_ERR_RANGE. */
smoe_status smoe_router_topk(const float* x, const uint16_t* wr, int64_t T, int H, int E, int K, uint16_t* work,
                             int32_t* ids, float* w, void* stream);
size_t smoe_router_work_bytes(int64_t T, int H);

/* Shared expert, scalar gate.  Page "src/prefill/prefill.cpp", Prefill::run, MoE half ("the shared expert and its
 * scalar gate": a projection of each token onto one row); the gate's nonlinearity is not given there and is read as
 * the logistic sigmoid:  sg[t] = 1 / (1 + exp(-(x[t] . w_sg))), the dot product in fp32.
 *   x fp32 [T][H], w_sg fp32 [H] -> sg fp32 [T].   H % 4 == 0; x, w_sg, sg 16-byte aligned. */
smoe_status smoe_shared_gate(const float* x, const float* wsg, int64_t T, int H, float* sg, void* stream);

/* Step 7 with the shared expert: smoe_combine's sum, then + sg[t] * ds[t][o] (fp32):
 *   Y[t][o] = sum_{k=0}^{K-1} w[t][k] * dm[slot[t*K+k]][o]  +  sg[t] * ds[t][o].
 *   ds fp32 [T][H] (the shared expert's down rows, row t = token t), sg fp32 [T] (smoe_shared_gate); the other
 *   arguments and rules as smoe_combine. */
smoe_status smoe_combine_shared(const float* dm, const int32_t* slot, const float* w, int64_t T, int K, int H,
                                const float* ds, const float* sg, float* y, void* stream);

/* THE BLOCK AS ONE OBJECT (a library service over the calls above; the pages' Prefill::run owns the equivalent
 * buffers).  A smoe_block holds every device buffer of the eight steps for chunks of T tokens, two device sets of
 * the chunk's inputs and output, three streams of its own (a copy-in, a copy-out and a compute stream) and a CUDA
 * graph of the eight calls for each input set.  It is created and used with the same device current; calls on one
 * block must not run concurrently from several host threads.
 *
 * smoe_block_create: T >= 1 tokens a chunk; H, E, K, F as for the calls above (H % 128 == 0, F % 64 == 0,
 *   1 <= K <= min(E, 32), E <= 1024).  wgu and wd are the routed experts' weights packed by smoe_pack_q2 (DEVICE
 *   pointers, owned by the caller, read by every chunk: they must outlive the block).  *out receives the block, or
 *   NULL on an error (SMOE_ERR_ARG for a bad size or pointer, SMOE_ERR_UNSUPPORTED off sm_103, SMOE_ERR_CUDA when an
 *   allocation fails; nothing is left allocated then).
 * smoe_block_destroy: waits for the block's queued work, then frees everything it owns (NULL is ignored).
 * smoe_block_run: one chunk device to device on `stream`: logits fp32 [T][E], x fp32 [T][H] -> y fp32 [T][H] (DEVICE
 *   pointers, 16-byte aligned), exactly the eight calls in order (the q8 quantisation on a side stream beside the
 *   routing and grouping); asynchronous like the calls above.
 * smoe_block_submit_host: one chunk from and into HOST memory, queued behind the chunks submitted before it:
 *   logits fp32 [T][E] and x fp32 [T][H] are copied to one of the two device input sets while the previous chunk
 *   computes, the chunk runs as a replay of that set's graph, and y fp32 [T][H] is copied back while the next chunk
 *   computes.  The call returns at once; the host buffers must stay valid and unchanged (y: unread) until
 *   smoe_block_sync returns.  Page-locked host memory (cudaHostAlloc, cudaHostRegister) lets the copies run beside
 *   the compute; pageable memory is correct but serialises them.  The first submit of a block runs the chunk
 *   eagerly once on zero inputs and captures the two graphs (about a millisecond); do that before timing.  The
 *   block's work starts after the work queued on `stream` before the call.
 * smoe_block_sync: `stream` waits for every chunk submitted so far (their outputs are then in host memory) and the
 *   host waits for them too.  Errors found on the device are in the tiles header (smoe_block_status).
 * smoe_block_run and the submitted chunks share the block's intermediate buffers: call smoe_block_sync before a
 *   smoe_block_run, and let a smoe_block_run finish (its stream) before the next submit.  After an error status from
 *   any of these calls, destroy the block. */
typedef struct smoe_block smoe_block;
smoe_status smoe_block_create(int64_t T, int H, int E, int K, int F, const uint8_t* wgu, const uint8_t* wd,
                              smoe_block** out);
void smoe_block_destroy(smoe_block* b);
smoe_status smoe_block_run(smoe_block* b, const float* logits, const float* x, float* y, void* stream);
smoe_status smoe_block_submit_host(smoe_block* b, const float* logits, const float* x, float* y, void* stream);
smoe_status smoe_block_sync(smoe_block* b, void* stream);
/* The last chunk's device-side status (synchronises): header[1] (grouping: SMOE_OK or SMOE_ERR_RANGE) into *group,
 * header[3] (the expert products: SMOE_OK or SMOE_ERR_TIMEOUT) into *kernel. */
smoe_status smoe_block_status(smoe_block* b, int* group, int* kernel);

#ifdef __cplusplus
}
#endif

#endif /* SMOE_H */
