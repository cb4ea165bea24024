// smoe_api.cu -- the extern "C" entry points of libsmoe (declared and documented in include/smoe.h): host-side
// argument checks, then the launches of each step on the caller's stream.  Nothing here allocates memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "smoe.h"
#include "smoe_internal.h"

namespace {

bool aligned16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

thread_local const char* g_last_cuda_error = "no error";

smoe_status launch_status(cudaError_t err) {
    if (err == cudaSuccess) return SMOE_OK;
    g_last_cuda_error = cudaGetErrorName(err);
    cudaGetLastError();  // clear a sticky launch error so that the caller's next call starts clean
    return SMOE_ERR_LAUNCH;
}

// 1: sm_103 device, 0: not, cached per device
int device_is_sm103() {
    static int cache[64] = {0};  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < 64 && cache[dev] != 0) return cache[dev] == 1;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    const bool ok = major == 10 && minor == 3;
    if (dev >= 0 && dev < 64) cache[dev] = ok ? 1 : 2;
    return ok;
}

constexpr int64_t kMaxGridY = 65535;

}  // namespace

namespace smoe {
smoe_status note_cuda_error(cudaError_t err) {
    if (err == cudaSuccess) return SMOE_OK;
    g_last_cuda_error = cudaGetErrorName(err);
    cudaGetLastError();
    return SMOE_ERR_CUDA;
}
}  // namespace smoe

extern "C" {

const char* smoe_status_string(smoe_status s) {
    switch (s) {
        case SMOE_OK: return "ok";
        case SMOE_ERR_ARG: return "bad argument (null or misaligned pointer, or a size out of range)";
        case SMOE_ERR_LAUNCH: return "kernel launch failed";
        case SMOE_ERR_UNSUPPORTED: return "unsupported shape or device (libsmoe runs on sm_103 only)";
        case SMOE_ERR_RANGE: return "a routed expert id is outside [0, E)";
        case SMOE_ERR_TIMEOUT: return "a kernel's internal wait ran out";
        case SMOE_ERR_CUDA: return "a CUDA runtime call failed (allocation, copy, stream, event or graph)";
        default: return "unknown status";
    }
}

const char* smoe_last_error_string(void) { return g_last_cuda_error; }

smoe_status smoe_device_check(void) { return device_is_sm103() ? SMOE_OK : SMOE_ERR_UNSUPPORTED; }

int64_t smoe_max_tiles(int64_t n, int E) {
    if (n <= 0 || E <= 0) return 0;
    return (n + SMOE_TILE_ROWS - 1) / SMOE_TILE_ROWS + (n < E ? n : E);
}

size_t smoe_tiles_bytes(int64_t n, int E) { return (size_t)16 * (size_t)(1 + smoe_max_tiles(n, E)); }

size_t smoe_group_work_bytes(int64_t n, int E) { return smoe::group_work_bytes(n, E); }

smoe_status smoe_route_topk(const float* logits, int64_t T, int E, int K, int32_t* ids, float* w, void* stream) {
    if (T < 0 || E < 1 || E > SMOE_MAX_EXPERTS || K < 1 || K > SMOE_MAX_TOPK || K > E) return SMOE_ERR_ARG;
    if (T == 0) return SMOE_OK;
    if (!aligned16(logits) || !aligned16(ids) || !aligned16(w)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_route_topk(logits, T, E, K, ids, w, (cudaStream_t)stream));
}

smoe_status smoe_group(const int32_t* ids, int64_t T, int K, int E, int32_t* counts, int32_t* offsets, int32_t* src,
                       int32_t* slot, int32_t* tiles, size_t tiles_bytes, void* work, size_t work_bytes,
                       void* stream) {
    if (T < 0 || E < 1 || E > SMOE_MAX_EXPERTS || K < 1 || K > SMOE_MAX_TOPK) return SMOE_ERR_ARG;
    if (T > (int64_t)(INT32_MAX / 2) / K) return SMOE_ERR_ARG;  // checked before T * K can overflow
    const int64_t n = T * K;
    if (!aligned16(counts) || !aligned16(offsets) || !aligned16(tiles)) return SMOE_ERR_ARG;
    if (n > 0 && (!aligned16(ids) || !aligned16(src) || !aligned16(slot))) return SMOE_ERR_ARG;
    if (tiles_bytes < smoe_tiles_bytes(n, E)) return SMOE_ERR_ARG;
    const size_t need = smoe_group_work_bytes(n, E);
    if (n > 0 && (work_bytes < need || !aligned16(work))) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_group(ids, n, K, E, counts, offsets, src, slot, tiles,
                                            reinterpret_cast<int32_t*>(work), (cudaStream_t)stream));
}

smoe_status smoe_quantize_q8(const float* x, int64_t rows, int cols, int8_t* codes, uint16_t* scales, void* stream) {
    if (rows < 0 || cols < 32 || cols % 32 != 0) return SMOE_ERR_ARG;
    if (rows == 0) return SMOE_OK;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_quantize_q8(x, rows, cols, codes, scales, (cudaStream_t)stream));
}

size_t smoe_pack_q2_bytes(int E, int rows, int cols) {
    return E <= 0 || rows <= 0 || cols <= 0 ? 0 : (size_t)E * rows * (cols / 4 + cols / 16);
}

smoe_status smoe_pack_q2(const uint8_t* codes, const uint16_t* scales, int E, int rows, int cols, uint8_t* packed,
                         void* stream) {
    if (E < 1 || rows < 128 || cols < 64 || rows % 128 != 0 || cols % 64 != 0) return SMOE_ERR_ARG;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(packed)) return SMOE_ERR_ARG;
    if ((int64_t)E * (rows / 128) * (cols / 64) > INT32_MAX) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(
        smoe::launch_pack_q2(codes, scales, nullptr, E, rows, cols, 0, packed, nullptr, (cudaStream_t)stream));
}

smoe_status smoe_pack_q2_swiglu(const uint8_t* codes, const uint16_t* scales, int E, int F, int H, uint8_t* packed,
                                void* stream) {
    if (E < 1 || F < 64 || H < 64 || F % 64 != 0 || H % 64 != 0) return SMOE_ERR_ARG;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(packed)) return SMOE_ERR_ARG;
    if ((int64_t)E * (2 * F / 128) * (H / 64) > INT32_MAX) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(
        smoe::launch_pack_q2(codes, scales, nullptr, E, 2 * F, H, F, packed, nullptr, (cudaStream_t)stream));
}

static smoe_status check_gemm_shape(int64_t n, int E, int H, int F) {
    if (n < 0 || E < 1 || E > SMOE_MAX_EXPERTS) return SMOE_ERR_ARG;
    if (H < 128 || F < 64) return SMOE_ERR_UNSUPPORTED;
    if (H % 128 != 0 || F % 64 != 0) return SMOE_ERR_UNSUPPORTED;
    if (smoe_max_tiles(n, E) > kMaxGridY) return SMOE_ERR_UNSUPPORTED;
    return SMOE_OK;
}

smoe_status smoe_gather_q8(const int8_t* codes, const uint16_t* scales, int64_t in_rows, int cols, const int32_t* src,
                           int64_t n, uint16_t* out, void* stream) {
    if (in_rows < 0 || n < 0 || cols < 32 || cols % 32 != 0) return SMOE_ERR_ARG;
    if (n == 0) return SMOE_OK;
    if (in_rows < 1 || n > INT32_MAX) return SMOE_ERR_ARG;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(src) || !aligned16(out)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_gather_q8(codes, scales, in_rows, cols, src, n, out, (cudaStream_t)stream));
}

smoe_status smoe_experts_gateup(const uint16_t* xop, int32_t* tiles, int64_t n, int E, const uint8_t* wgu, int H, int F,
                                float* gu, void* stream) {
    const smoe_status st = check_gemm_shape(n, E, H, F);
    if (st != SMOE_OK) return st;
    if (n == 0) return SMOE_OK;
    if (!aligned16(xop) || !aligned16(tiles) || !aligned16(wgu) || !aligned16(gu)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    smoe::ExpertsGemmArgs a{xop, tiles, wgu, 2 * F, H, gu, n, E, true, 1, nullptr, nullptr, nullptr};
    return launch_status(smoe::launch_experts_gemm(a, smoe_max_tiles(n, E), (cudaStream_t)stream));
}

smoe_status smoe_experts_gateup_swiglu(const uint16_t* xop, int32_t* tiles, int64_t n, int E, const uint8_t* wgs, int H,
                                       int F, int8_t* hc, uint16_t* hs, uint16_t* hop, void* stream) {
    const smoe_status st = check_gemm_shape(n, E, H, F);
    if (st != SMOE_OK) return st;
    if (n == 0) return SMOE_OK;
    if (!aligned16(xop) || !aligned16(tiles) || !aligned16(wgs) || !aligned16(hc) || !aligned16(hs) ||
        !aligned16(hop))
        return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    smoe::ExpertsGemmArgs a{xop, tiles, wgs, 2 * F, H, nullptr, n, E, true, 1, hc, hs, hop};
    return launch_status(smoe::launch_experts_gemm(a, smoe_max_tiles(n, E), (cudaStream_t)stream));
}

smoe_status smoe_swiglu_requant(const float* gu, int64_t n, int F, int8_t* hc, uint16_t* hs, uint16_t* hop,
                                void* stream) {
    if (n < 0 || F < 32 || F % 32 != 0) return SMOE_ERR_ARG;
    if (hop != nullptr && F % 64 != 0) return SMOE_ERR_ARG;
    if (n == 0) return SMOE_OK;
    if (!aligned16(gu) || !aligned16(hc) || !aligned16(hs)) return SMOE_ERR_ARG;
    if (hop != nullptr && !aligned16(hop)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_swiglu_requant(gu, n, F, hc, hs, hop, (cudaStream_t)stream));
}

smoe_status smoe_experts_down(const uint16_t* hop, int32_t* tiles, int64_t n, int E, const uint8_t* wd, int H, int F,
                              float* dm, void* stream) {
    const smoe_status st = check_gemm_shape(n, E, H, F);
    if (st != SMOE_OK) return st;
    if (n == 0) return SMOE_OK;
    if (!aligned16(hop) || !aligned16(tiles) || !aligned16(wd) || !aligned16(dm)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    smoe::ExpertsGemmArgs a{hop, tiles, wd, H, F, dm, n, E, false, 1, nullptr, nullptr, nullptr};
    return launch_status(smoe::launch_experts_gemm(a, smoe_max_tiles(n, E), (cudaStream_t)stream));
}

smoe_status smoe_experts_down_h(const uint16_t* hop, int32_t* tiles, int64_t n, int E, const uint8_t* wd, int H,
                                int F, uint16_t* dm_h, void* stream) {
    const smoe_status st = check_gemm_shape(n, E, H, F);
    if (st != SMOE_OK) return st;
    if (n == 0) return SMOE_OK;
    if (!aligned16(hop) || !aligned16(tiles) || !aligned16(wd) || !aligned16(dm_h)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    smoe::ExpertsGemmArgs a{hop, tiles, wd, H, F, nullptr, n, E, false, 1, nullptr, nullptr, nullptr};
    a.out_h = dm_h;
    return launch_status(smoe::launch_experts_gemm(a, smoe_max_tiles(n, E), (cudaStream_t)stream));
}

size_t smoe_experts_q8_work_bytes(int64_t n, int E, int H, int F) {
    if (n < 0 || E < 1 || H < 1 || F < 1) return 0;
    // the routed rows in operand form (fp16 [2][n][K]), then the packed weights; the larger of the two products
    const size_t gu = (size_t)4 * (size_t)n * (size_t)H + smoe_pack_q2_bytes(E, 2 * F, H);
    const size_t dn = (size_t)4 * (size_t)n * (size_t)F + smoe_pack_q2_bytes(E, H, F);
    return gu > dn ? gu : dn;
}

smoe_status smoe_experts_gateup_q8(const int8_t* xc, const uint16_t* xs, int64_t in_rows, const int32_t* src,
                                   int32_t* tiles, int64_t n, int E, const smoe_q2w* w_gu, int H, int F, void* work,
                                   size_t work_bytes, float* gu, void* stream) {
    const smoe_status st = check_gemm_shape(n, E, H, F);
    if (st != SMOE_OK) return st;
    if (n == 0) return SMOE_OK;
    if (in_rows < 1 || n > INT32_MAX) return SMOE_ERR_ARG;
    if (!aligned16(xc) || !aligned16(xs) || !aligned16(src) || !aligned16(tiles) || !aligned16(w_gu) ||
        !aligned16(work) || !aligned16(gu))
        return SMOE_ERR_ARG;
    if (work_bytes < smoe_experts_q8_work_bytes(n, E, H, F)) return SMOE_ERR_ARG;
    if ((int64_t)E * (2 * F / 128) * (H / 64) > INT32_MAX) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    uint16_t* xop = static_cast<uint16_t*>(work);
    uint8_t* wp = static_cast<uint8_t*>(work) + (size_t)4 * (size_t)n * (size_t)H;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t err = smoe::launch_gather_q8(xc, xs, in_rows, H, src, n, xop, s);
    if (err == cudaSuccess) err = smoe::launch_pack_q2(nullptr, nullptr, w_gu, E, 2 * F, H, 0, wp, tiles + 3, s);
    if (err != cudaSuccess) return launch_status(err);
    smoe::ExpertsGemmArgs a{xop, tiles, wp, 2 * F, H, gu, n, E, true, 1, nullptr, nullptr, nullptr};
    return launch_status(smoe::launch_experts_gemm(a, smoe_max_tiles(n, E), s));
}

smoe_status smoe_experts_down_q8(const int8_t* hc, const uint16_t* hs, int32_t* tiles, int64_t n, int E,
                                 const smoe_q2w* w_d, int H, int F, void* work, size_t work_bytes, float* dm,
                                 void* stream) {
    const smoe_status st = check_gemm_shape(n, E, H, F);
    if (st != SMOE_OK) return st;
    if (n == 0) return SMOE_OK;
    if (n > INT32_MAX) return SMOE_ERR_ARG;
    if (!aligned16(hc) || !aligned16(hs) || !aligned16(tiles) || !aligned16(w_d) || !aligned16(work) ||
        !aligned16(dm))
        return SMOE_ERR_ARG;
    if (work_bytes < smoe_experts_q8_work_bytes(n, E, H, F)) return SMOE_ERR_ARG;
    if ((int64_t)E * (H / 128) * (F / 64) > INT32_MAX) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    uint16_t* hop = static_cast<uint16_t*>(work);
    uint8_t* wp = static_cast<uint8_t*>(work) + (size_t)4 * (size_t)n * (size_t)F;
    const cudaStream_t s = (cudaStream_t)stream;
    // H is already in routed-row order: the operand form of row r is row r itself (no src)
    cudaError_t err = smoe::launch_gather_q8(hc, hs, n, F, nullptr, n, hop, s);
    if (err == cudaSuccess) err = smoe::launch_pack_q2(nullptr, nullptr, w_d, E, H, F, 0, wp, tiles + 3, s);
    if (err != cudaSuccess) return launch_status(err);
    smoe::ExpertsGemmArgs a{hop, tiles, wp, H, F, dm, n, E, false, 1, nullptr, nullptr, nullptr};
    return launch_status(smoe::launch_experts_gemm(a, smoe_max_tiles(n, E), s));
}

smoe_status smoe_combine(const float* dm, const int32_t* slot, const float* w, int64_t T, int K, int H, float* y,
                         void* stream) {
    if (T < 0 || K < 1 || K > SMOE_MAX_TOPK || H < 4 || H % 4 != 0) return SMOE_ERR_ARG;
    if (T == 0) return SMOE_OK;
    if (!aligned16(dm) || !aligned16(slot) || !aligned16(w) || !aligned16(y)) return SMOE_ERR_ARG;
    if ((H / 4 + 127) / 128 > kMaxGridY) return SMOE_ERR_UNSUPPORTED;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_combine(dm, slot, w, T, K, H, nullptr, nullptr, y, (cudaStream_t)stream));
}

smoe_status smoe_combine_h(const uint16_t* dm_h, const int32_t* slot, const float* w, int64_t T, int K, int H,
                           float* y, void* stream) {
    if (T < 0 || T > INT32_MAX || K < 1 || K > SMOE_MAX_TOPK || H < 8 || H % 8 != 0) return SMOE_ERR_ARG;
    if (T == 0) return SMOE_OK;
    if (!aligned16(dm_h) || !aligned16(slot) || !aligned16(w) || !aligned16(y)) return SMOE_ERR_ARG;
    if ((H / 8 + 63) / 64 > kMaxGridY) return SMOE_ERR_UNSUPPORTED;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_combine_h(dm_h, slot, w, T, K, H, y, (cudaStream_t)stream));
}

smoe_status smoe_router_topk(const float* x, const uint16_t* wr, int64_t T, int H, int E, int K, uint16_t* work,
                             int32_t* ids, float* w, void* stream) {
    if (T < 0 || T > INT32_MAX || H < 64 || H % 64 != 0 || E < 16 || E > 512 || E % 16 != 0 ||
        (E > 256 && E % 32 != 0) || K < 1 || K > 16 || K > E)
        return SMOE_ERR_ARG;
    if (T == 0) return SMOE_OK;
    if (!aligned16(x) || !aligned16(wr) || !aligned16(work) || !aligned16(ids) || !aligned16(w)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_router_topk(x, wr, T, H, E, K, work, ids, w, (cudaStream_t)stream));
}

size_t smoe_router_work_bytes(int64_t T, int H) {
    // the bf16 hi and lo planes [2][T][H], then two parts' candidates (fp32 logit, int32 id) [T][2][16] each
    return T <= 0 || H <= 0 ? 0 : (size_t)T * (size_t)H * 4 + (size_t)T * 256;
}

smoe_status smoe_shared_gate(const float* x, const float* wsg, int64_t T, int H, float* sg, void* stream) {
    if (T < 0 || H < 4 || H % 4 != 0) return SMOE_ERR_ARG;
    if (T == 0) return SMOE_OK;
    if (!aligned16(x) || !aligned16(wsg) || !aligned16(sg)) return SMOE_ERR_ARG;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_shared_gate(x, wsg, T, H, sg, (cudaStream_t)stream));
}

smoe_status smoe_combine_shared(const float* dm, const int32_t* slot, const float* w, int64_t T, int K, int H,
                                const float* ds, const float* sg, float* y, void* stream) {
    if (T < 0 || K < 1 || K > SMOE_MAX_TOPK || H < 4 || H % 4 != 0) return SMOE_ERR_ARG;
    if (T == 0) return SMOE_OK;
    if (!aligned16(dm) || !aligned16(slot) || !aligned16(w) || !aligned16(y) || !aligned16(ds) || !aligned16(sg))
        return SMOE_ERR_ARG;
    if ((H / 4 + 127) / 128 > kMaxGridY) return SMOE_ERR_UNSUPPORTED;
    if (!device_is_sm103()) return SMOE_ERR_UNSUPPORTED;
    return launch_status(smoe::launch_combine(dm, slot, w, T, K, H, ds, sg, y, (cudaStream_t)stream));
}

}  // extern "C"
