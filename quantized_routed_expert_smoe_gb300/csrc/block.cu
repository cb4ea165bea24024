// block.cu -- the routed-expert block as one object (smoe_block_*, declared and documented in include/smoe.h): the
// device buffers of the eight steps allocated once, chunks run device to device or fed from and into host memory
// with the copies overlapped with the compute (two device input/output sets, a copy-in, a copy-out and a compute
// stream, a CUDA graph of the eight calls per set).
//
// Page "src/prefill/prefill.cpp", Prefill::run, MoE half: the engine's prompt path owns its activation, routing and
// expert buffers for a chunk and runs the steps in this order; the steps themselves are the C-ABI calls of
// smoe_api.cu, issued here unchanged.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "smoe.h"
#include "smoe_internal.h"

struct smoe_block {
    int64_t T = 0, n = 0;
    int H = 0, E = 0, K = 0, F = 0;
    const uint8_t* wgu = nullptr;
    const uint8_t* wd = nullptr;
    // the steps' buffers (shared by consecutive chunks: the chunks run one after another on the compute stream)
    int32_t* ids = nullptr;
    float* w = nullptr;
    int32_t* counts = nullptr;
    int32_t* offsets = nullptr;
    int32_t* src = nullptr;
    int32_t* slot = nullptr;
    int32_t* tiles = nullptr;
    size_t tiles_bytes = 0;
    void* work = nullptr;
    size_t work_bytes = 0;
    int8_t* xc = nullptr;
    uint16_t* xs = nullptr;
    uint16_t* xop = nullptr;
    float* gu = nullptr;
    int8_t* hc = nullptr;
    uint16_t* hs = nullptr;
    uint16_t* hop = nullptr;
    float* dm = nullptr;
    // two device sets of a chunk's inputs and output (set b serves the chunks b, b + 2, ...)
    float* d_logits[2] = {nullptr, nullptr};
    float* d_x[2] = {nullptr, nullptr};
    float* d_y[2] = {nullptr, nullptr};
    cudaStream_t side = nullptr, copy_in = nullptr, copy_out = nullptr, compute = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, start = nullptr, finish = nullptr;
    cudaEvent_t ev_in[2] = {nullptr, nullptr};    // set b's inputs are on the device
    cudaEvent_t ev_done[2] = {nullptr, nullptr};  // set b's chunk has computed
    cudaEvent_t ev_out[2] = {nullptr, nullptr};   // set b's output is back in host memory
    cudaGraphExec_t graph[2] = {nullptr, nullptr};
    int64_t submitted = 0;  // chunks submitted since the last sync
};

namespace {

bool aligned16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

template <typename Ptr>
cudaError_t alloc(Ptr*& p, size_t bytes) {
    void* q = nullptr;
    const cudaError_t e = cudaMalloc(&q, bytes < 16 ? 16 : bytes);
    p = static_cast<Ptr*>(q);
    return e;
}

void release(smoe_block* b) {
    if (b == nullptr) return;
    for (int k = 0; k < 2; ++k) {
        if (b->graph[k]) cudaGraphExecDestroy(b->graph[k]);
        cudaFree(b->d_logits[k]);
        cudaFree(b->d_x[k]);
        cudaFree(b->d_y[k]);
        if (b->ev_in[k]) cudaEventDestroy(b->ev_in[k]);
        if (b->ev_done[k]) cudaEventDestroy(b->ev_done[k]);
        if (b->ev_out[k]) cudaEventDestroy(b->ev_out[k]);
    }
    for (cudaEvent_t e : {b->fork, b->join, b->start, b->finish})
        if (e) cudaEventDestroy(e);
    for (cudaStream_t s : {b->side, b->copy_in, b->copy_out, b->compute})
        if (s) cudaStreamDestroy(s);
    void* bufs[] = {b->ids, b->w, b->counts, b->offsets, b->src, b->slot, b->tiles, b->work, b->xc,
                    b->xs,  b->xop, b->gu,   b->hc,      b->hs,  b->hop,  b->dm};
    for (void* q : bufs) cudaFree(q);
    delete b;
}

// the eight calls of one chunk on `main`, the quantisation forked onto the side stream
smoe_status run_chunk(smoe_block* b, const float* logits, const float* x, float* y, cudaStream_t main) {
    smoe_status st = smoe::note_cuda_error(cudaEventRecord(b->fork, main));
    if (st == SMOE_OK) st = smoe::note_cuda_error(cudaStreamWaitEvent(b->side, b->fork, 0));
    if (st == SMOE_OK) st = smoe_quantize_q8(x, b->T, b->H, b->xc, b->xs, b->side);
    if (st == SMOE_OK) st = smoe::note_cuda_error(cudaEventRecord(b->join, b->side));
    if (st == SMOE_OK) st = smoe_route_topk(logits, b->T, b->E, b->K, b->ids, b->w, main);
    if (st == SMOE_OK)
        st = smoe_group(b->ids, b->T, b->K, b->E, b->counts, b->offsets, b->src, b->slot, b->tiles, b->tiles_bytes,
                        b->work, b->work_bytes, main);
    if (st == SMOE_OK) st = smoe::note_cuda_error(cudaStreamWaitEvent(main, b->join, 0));
    if (st == SMOE_OK) st = smoe_gather_q8(b->xc, b->xs, b->T, b->H, b->src, b->n, b->xop, main);
    if (st == SMOE_OK) st = smoe_experts_gateup(b->xop, b->tiles, b->n, b->E, b->wgu, b->H, b->F, b->gu, main);
    if (st == SMOE_OK) st = smoe_swiglu_requant(b->gu, b->n, b->F, b->hc, b->hs, b->hop, main);
    if (st == SMOE_OK) st = smoe_experts_down(b->hop, b->tiles, b->n, b->E, b->wd, b->H, b->F, b->dm, main);
    if (st == SMOE_OK) st = smoe_combine(b->dm, b->slot, b->w, b->T, b->K, b->H, y, main);
    return st;
}

// the graphs of the two input sets: one eager chunk first (the calls' one-time per-device set-up is not captured),
// then one capture per set on the compute stream
smoe_status make_graphs(smoe_block* b) {
    smoe_status st = run_chunk(b, b->d_logits[0], b->d_x[0], b->d_y[0], b->compute);
    if (st == SMOE_OK) st = smoe::note_cuda_error(cudaStreamSynchronize(b->compute));
    for (int k = 0; k < 2 && st == SMOE_OK; ++k) {
        cudaGraph_t g = nullptr;
        st = smoe::note_cuda_error(cudaStreamBeginCapture(b->compute, cudaStreamCaptureModeThreadLocal));
        if (st != SMOE_OK) break;
        const smoe_status run = run_chunk(b, b->d_logits[k], b->d_x[k], b->d_y[k], b->compute);
        const cudaError_t end = cudaStreamEndCapture(b->compute, &g);  // ends the capture on every path
        st = run != SMOE_OK ? run : smoe::note_cuda_error(end);
        if (st == SMOE_OK) st = smoe::note_cuda_error(cudaGraphInstantiate(&b->graph[k], g, 0));
        if (g) cudaGraphDestroy(g);
    }
    return st;
}

}  // namespace

extern "C" {

smoe_status smoe_block_create(int64_t T, int H, int E, int K, int F, const uint8_t* wgu, const uint8_t* wd,
                              smoe_block** out) {
    if (out == nullptr) return SMOE_ERR_ARG;
    *out = nullptr;
    if (T < 1 || H < 128 || H % 128 != 0 || F < 64 || F % 64 != 0 || E < 1 || E > SMOE_MAX_EXPERTS || K < 1 ||
        K > E || K > SMOE_MAX_TOPK || !aligned16(wgu) || !aligned16(wd))
        return SMOE_ERR_ARG;
    if (T > (int64_t)1 << 31 || T * K > (int64_t)1 << 31) return SMOE_ERR_ARG;
    if (smoe_device_check() != SMOE_OK) return SMOE_ERR_UNSUPPORTED;
    smoe_block* b = new (std::nothrow) smoe_block;
    if (b == nullptr) return SMOE_ERR_CUDA;
    b->T = T;
    b->n = T * K;
    b->H = H;
    b->E = E;
    b->K = K;
    b->F = F;
    b->wgu = wgu;
    b->wd = wd;
    const size_t n = (size_t)b->n, t = (size_t)T;
    b->tiles_bytes = smoe_tiles_bytes(b->n, E);
    b->work_bytes = smoe_group_work_bytes(b->n, E);
    cudaError_t e = cudaSuccess;
    auto A = [&](auto*& p, size_t bytes) {
        if (e == cudaSuccess) e = alloc(p, bytes);
    };
    A(b->ids, t * K * 4);
    A(b->w, t * K * 4);
    A(b->counts, (size_t)E * 4);
    A(b->offsets, ((size_t)E + 4) * 4);
    A(b->src, n * 4);
    A(b->slot, n * 4);
    A(b->tiles, b->tiles_bytes);
    A(b->work, b->work_bytes);
    A(b->xc, t * H);
    A(b->xs, t * (H / 32) * 2);
    A(b->xop, 2 * n * H * 2);
    A(b->gu, n * 2 * F * 4);
    A(b->hc, n * F);
    A(b->hs, n * (F / 32) * 2);
    A(b->hop, 2 * n * F * 2);
    A(b->dm, n * H * 4);
    for (int k = 0; k < 2; ++k) {
        A(b->d_logits[k], t * E * 4);
        A(b->d_x[k], t * H * 4);
        A(b->d_y[k], t * H * 4);
    }
    // zero inputs: the eager chunk before the graph capture runs on them
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
        e = cudaMemset(b->d_logits[k], 0, t * E * 4);
        if (e == cudaSuccess) e = cudaMemset(b->d_x[k], 0, t * H * 4);
    }
    for (cudaStream_t* s : {&b->side, &b->copy_in, &b->copy_out, &b->compute})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&b->fork, &b->join, &b->start, &b->finish, &b->ev_in[0], &b->ev_in[1], &b->ev_done[0],
                            &b->ev_done[1], &b->ev_out[0], &b->ev_out[1]})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        const smoe_status st = smoe::note_cuda_error(e);
        release(b);
        return st;
    }
    *out = b;
    return SMOE_OK;
}

void smoe_block_destroy(smoe_block* b) {
    if (b == nullptr) return;
    for (cudaStream_t s : {b->side, b->copy_in, b->copy_out, b->compute})
        if (s) cudaStreamSynchronize(s);
    release(b);
}

smoe_status smoe_block_run(smoe_block* b, const float* logits, const float* x, float* y, void* stream) {
    if (b == nullptr || !aligned16(logits) || !aligned16(x) || !aligned16(y)) return SMOE_ERR_ARG;
    return run_chunk(b, logits, x, y, static_cast<cudaStream_t>(stream));
}

smoe_status smoe_block_submit_host(smoe_block* b, const float* logits, const float* x, float* y, void* stream) {
    if (b == nullptr || logits == nullptr || x == nullptr || y == nullptr) return SMOE_ERR_ARG;
    const cudaStream_t caller = static_cast<cudaStream_t>(stream);
    smoe_status st = SMOE_OK;
    if (b->graph[0] == nullptr || b->graph[1] == nullptr) {
        for (int k = 0; k < 2; ++k)
            if (b->graph[k]) {
                cudaGraphExecDestroy(b->graph[k]);
                b->graph[k] = nullptr;
            }
        st = make_graphs(b);
        if (st != SMOE_OK) return st;
    }
    auto ok = [&](cudaError_t e) {
        if (st == SMOE_OK) st = smoe::note_cuda_error(e);
        return st == SMOE_OK;
    };
    const int64_t i = b->submitted;
    const int k = (int)(i & 1);
    const size_t in_logits = (size_t)b->T * b->E * 4, in_x = (size_t)b->T * b->H * 4, out_y = in_x;
    if (i == 0) {
        // the block's first chunk since the last sync starts after the work queued on the caller's stream
        ok(cudaEventRecord(b->start, caller));
        ok(cudaStreamWaitEvent(b->copy_in, b->start, 0));
        ok(cudaStreamWaitEvent(b->compute, b->start, 0));
        ok(cudaStreamWaitEvent(b->copy_out, b->start, 0));
    }
    // inputs: set k must be free (its chunk i - 2 has computed)
    if (i >= 2) ok(cudaStreamWaitEvent(b->copy_in, b->ev_done[k], 0));
    ok(cudaMemcpyAsync(b->d_logits[k], logits, in_logits, cudaMemcpyHostToDevice, b->copy_in));
    ok(cudaMemcpyAsync(b->d_x[k], x, in_x, cudaMemcpyHostToDevice, b->copy_in));
    ok(cudaEventRecord(b->ev_in[k], b->copy_in));
    // the chunk: after its inputs, and after set k's previous output has been copied back
    ok(cudaStreamWaitEvent(b->compute, b->ev_in[k], 0));
    if (i >= 2) ok(cudaStreamWaitEvent(b->compute, b->ev_out[k], 0));
    ok(cudaGraphLaunch(b->graph[k], b->compute));
    ok(cudaEventRecord(b->ev_done[k], b->compute));
    // the output
    ok(cudaStreamWaitEvent(b->copy_out, b->ev_done[k], 0));
    ok(cudaMemcpyAsync(y, b->d_y[k], out_y, cudaMemcpyDeviceToHost, b->copy_out));
    ok(cudaEventRecord(b->ev_out[k], b->copy_out));
    if (st == SMOE_OK) ++b->submitted;
    return st;
}

smoe_status smoe_block_sync(smoe_block* b, void* stream) {
    if (b == nullptr) return SMOE_ERR_ARG;
    const cudaStream_t caller = static_cast<cudaStream_t>(stream);
    smoe_status st = SMOE_OK;
    if (b->submitted > 0) {
        st = smoe::note_cuda_error(cudaEventRecord(b->finish, b->copy_out));
        if (st == SMOE_OK) st = smoe::note_cuda_error(cudaStreamWaitEvent(caller, b->finish, 0));
        if (st == SMOE_OK) st = smoe::note_cuda_error(cudaEventSynchronize(b->finish));
    }
    b->submitted = 0;
    return st;
}

smoe_status smoe_block_status(smoe_block* b, int* group, int* kernel) {
    if (b == nullptr || group == nullptr || kernel == nullptr) return SMOE_ERR_ARG;
    int32_t h[4] = {0, 0, 0, 0};
    for (cudaStream_t s : {b->compute, b->copy_out}) {
        const cudaError_t e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return smoe::note_cuda_error(e);
    }
    const smoe_status st = smoe::note_cuda_error(cudaMemcpy(h, b->tiles, sizeof(h), cudaMemcpyDeviceToHost));
    *group = h[1];
    *kernel = h[3];
    return st;
}

}  // extern "C"
