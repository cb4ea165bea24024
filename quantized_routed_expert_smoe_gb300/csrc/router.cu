// router.cu -- the router projection fused into the routing step (step 1): the logits are computed on the tensor
// cores and selected from tensor memory, never written to HBM.
//
// Page "src/prefill/prefill.cpp", Prefill::run, MoE half: the router is a BF16 projection of the hidden state
// (bf16_proj of the router weight "ffn_gate_inp" on the hidden state's BF16 copy, with its low part), then
// route(logits, ids, w, T, n_expert).  Here:
//   xh = bf16_rne(x), xl = bf16_rne(x - xh)                (x - xh is exact in fp32)
//   logit[t][e] = sum_h Wr[e][h] * (xh[t][h] + xl[t][h])    (bf16 x bf16 products exact, fp32 accumulation)
// then the top-K by logit (ties to the lower id) and the weights renormalised over the K, as smoe_route_topk.
//
// Kernels:
//   router_split_kernel   x fp32 [T][H] -> the bf16 planes [2][T][H] (hi, lo) the tensor cores read;
//   router_topk_kernel    one CTA per 128 tokens and part of E (one part for E <= 256, two halves above, so that a
//                         part is one MMA's N <= 256 and twice as many SMs work): per 64-wide K slice, TMA loads of
//                         the two activation tiles (128-byte swizzle) and of the part's router rows; eight
//                         tcgen05.mma (M = 128, N = the part, K = 16: four K16 steps of each activation part)
//                         accumulate the part's logits in tensor memory; then the logits of 64 tokens at a time
//                         pass through shared memory so that one warp holds one token, and K rounds of a warp
//                         arg-max pick the K best -- the final ids and weights for one part, else each half's K
//                         candidates (logit, id) into scratch;
//   router_merge_kernel   (two parts) one warp a token: the same K rounds over its 2K candidates, then the weights.
//                         The top-K of the union of the halves' top-K lists is the top-K of all E.
// Roles (192 threads): warp 0 lane 0 the producer, warp 1 the tensor-memory allocation and lane 0 the MMAs; warps
// 2-5 read the logits out of tensor memory (warp w reads lanes 32 (w mod 4) ..), all six warps select.  A wait that
// gives up writes id -1 for the CTA's tokens, which the grouping reports as an out-of-range id.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "smoe_device.cuh"
#include "smoe_internal.h"

namespace smoe {
namespace {

constexpr int kRM = 128;         // tokens a CTA (MMA M)
constexpr int kRK = 64;          // K values a slice: one 128-byte swizzle row of bf16
constexpr int kRThreads = 192;
constexpr int kRMaxE = 512;      // tensor-memory columns allocated
constexpr int kRMaxN = 256;      // experts a CTA (one MMA's N)
constexpr int kRMaxCand = 16;    // candidates a part keeps per token at most (K <= 16)
constexpr int kRSmem = 232448;   // the per-CTA maximum: [align slack][ring][barriers]
constexpr int kRBarBytes = 256;
constexpr int kRRing = kRSmem - 1024 - kRBarBytes;
constexpr int kRMaxDepth = 4;

struct RouterMaps {
    CUtensorMap xh, xl;  // bf16 [T][H] planes, box 64 x 128 rows
    CUtensorMap wr;      // bf16 [E][H], box 64 x (E or E/2) rows
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__global__ void __launch_bounds__(256) router_split_kernel(const float4* __restrict__ x, int64_t n8,
                                                           uint4* __restrict__ xh, uint4* __restrict__ xl) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = __ldcs(x + 2 * i), b = __ldcs(x + 2 * i + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * k]), h1 = __float2bfloat16_rn(v[2 * k + 1]);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * k] - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * k + 1] - __bfloat162float(h1));
            hw[k] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lw[k] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        }
        xh[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        xl[i] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

// K rounds of a warp arg-max over the values lane l holds (v[i], id[i]; -inf / INT_MAX where empty), ties to the
// lower id; lane k < K ends with the k-th best in (my_v, my_i).
template <int VPL>
__device__ __forceinline__ void warp_topk(float (&v)[VPL], const int (&id)[VPL], int K, float& my_v, int& my_i) {
    const int lane = threadIdx.x & 31;
    my_v = -INFINITY;
    my_i = 0x7fffffff;
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (v[i] > bv || (v[i] == bv && id[i] < bi)) {
                bv = v[i];
                bi = id[i];
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == k) {
            my_v = bv;
            my_i = bi;
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (id[i] == bi) v[i] = -INFINITY;  // ids are distinct: only the winner's lane retires one
    }
}

// The weights exp(l_k - l_1) / sum_j exp(l_j - l_1) over the K (summed in k order) and the ids of token t.
__device__ __forceinline__ void write_topk(float my_v, int my_i, int K, int64_t t, int32_t* ids, float* w) {
    const int lane = threadIdx.x & 31;
    const float lmax = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < K ? expf(my_v - lmax) : 0.0f;
    float sum = 0.0f;
    for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, ex, k);
    if (lane < K) {
        ids[t * K + lane] = my_i;
        w[t * K + lane] = __fdiv_rn(ex, sum);
    }
}

__global__ void __launch_bounds__(kRThreads, 1) router_topk_kernel(const __grid_constant__ RouterMaps maps, int64_t T,
                                                                   int H, int E, int K, int32_t* __restrict__ ids,
                                                                   float* __restrict__ w, float* __restrict__ cand_v,
                                                                   int32_t* __restrict__ cand_i) {
    const int nk = H / kRK;
    const int nsplit = (int)gridDim.y;  // parts of E
    const int En = E / nsplit;           // this CTA's experts [e0, e0 + En), En <= 256: one MMA's N
    const int e0 = (int)blockIdx.y * En;
    const uint32_t a_bytes = kRM * 128u;                      // one activation part of a slice
    const int sbytes = 2 * (int)a_bytes + En * 128;            // hi tile, lo tile, the part's router rows
    const int depth = min(kRMaxDepth, kRRing / sbytes);
    const uint32_t tx = (uint32_t)sbytes;
    const int64_t row0 = (int64_t)blockIdx.x * kRM;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    const uint32_t ring = smem_u32(smem_raw + pad);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + kRSmem - kRBarBytes);  // [kRMaxDepth]
    uint64_t* empty = full + kRMaxDepth;                                          // [kRMaxDepth]
    uint64_t* accf = empty + kRMaxDepth;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int r = 0; r < kRMaxDepth; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&empty[r], 1);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, (uint32_t)kRMaxE);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ producer
            asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.wr) : "memory");
            int issued = 0;
            for (int kt = 0; kt < nk; ++kt) {
                const int r = kt % depth;
                if (kt >= depth && !mbar_wait(&empty[r], (uint32_t)(kt / depth - 1) & 1u, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
                const uint32_t slot = ring + (uint32_t)(r * sbytes);
                mbar_arrive_expect_tx(&full[r], tx);
                tma_load_2d(slot, &maps.xh, kt * kRK, (int)row0, &full[r]);
                tma_load_2d(slot + a_bytes, &maps.xl, kt * kRK, (int)row0, &full[r]);
                tma_load_2d(slot + 2 * a_bytes, &maps.wr, kt * kRK, e0, &full[r]);
                ++issued;
            }
            // no copy may still be landing when the CTA exits: wait (bounded) for the last slices issued
            for (int kt = max(0, issued - depth); kt < issued; ++kt)
                mbar_wait(&full[kt % depth], (uint32_t)(kt / depth) & 1u, nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issue
            const uint32_t idesc = idesc_bf16_f32(kRM, En);
            for (int kt = 0; kt < nk; ++kt) {
                const int r = kt % depth;
                if (!mbar_wait(&full[r], (uint32_t)(kt / depth) & 1u, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;  // before the final commit: the epilogue must not take partial sums
                    __threadfence_block();
                    break;
                }
                tc_fence_after();
                const uint32_t slot = ring + (uint32_t)(r * sbytes);
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16)
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint64_t a = sdesc_k_sw128(slot + (uint32_t)part * a_bytes + 32u * (uint32_t)k16);
                        const uint64_t b = sdesc_k_sw128(slot + 2 * a_bytes + 32u * (uint32_t)k16);
                        mma_f16(tmem, a, b, idesc, (kt > 0 || k16 > 0 || part > 0) ? 1u : 0u);
                    }
                mma_commit(&empty[r]);
            }
            mma_commit(accf);  // every MMA issued above has completed (abort path included)
        }
        __syncwarp();
    }
    // -------------------------------------------------------------------- epilogue (every warp)
    // The logits of 64 tokens at a time go from tensor memory (lane = token) through the idle ring (rows of E + 1
    // floats: the stores of a warp hit 32 different banks) to a layout where one warp holds one token (lane l the
    // logits l, l + 32, ...); then K rounds of a warp arg-max, ties to the lower id, as in the routing kernel.
    bool done = true;
    if (warp >= 2) done = mbar_wait(accf, 0u, nullptr) && *abort_flag == 0;
    const bool good = __syncthreads_and(done) != 0;
    tc_fence_after();
    if (!good) {
        // id -1, which the grouping reports as out of range (a candidate -1 wins the merge with its +inf)
        if (warp >= 2) {
            const int64_t t = row0 + 32 * (warp & 3) + lane;
            if (t < T)
                for (int j = 0; j < K; ++j) {
                    if (nsplit == 1) {
                        ids[t * K + j] = -1;
                    } else {
                        cand_i[(t * nsplit + blockIdx.y) * K + j] = -1;
                        cand_v[(t * nsplit + blockIdx.y) * K + j] = INFINITY;
                    }
                }
        }
        ok = false;
    } else {
        float* const sl = reinterpret_cast<float*>(smem_raw + pad);
        const int ld = En + 1;
        for (int hh = 0; hh < 2; ++hh) {
            if (warp >= 2 && ((warp & 3) >> 1) == hh) {
                const int q = warp & 3;
                const int rr = 32 * (q & 1) + lane;  // row within the 64 tokens
                const uint32_t base = tmem + ((uint32_t)(32 * q) << 16);
                for (int c = 0; c < En; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(base + (uint32_t)c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c + i < En) sl[rr * ld + c + i] = __uint_as_float(v[i]);
                }
            }
            __syncthreads();
            for (int rr = warp; rr < 64; rr += kRThreads / 32) {
                const int64_t t = row0 + 64 * hh + rr;
                if (t >= T) break;  // the same in every lane; later rows are further past T
                const float* lt = sl + rr * ld;
                float v[kRMaxN / 32];
                int id[kRMaxN / 32];
#pragma unroll
                for (int i = 0; i < kRMaxN / 32; ++i) {
                    const int e = lane + 32 * i;
                    v[i] = e < En ? lt[e] : -INFINITY;
                    id[i] = e < En ? e0 + e : 0x7fffffff;
                }
                float my_v;
                int my_i;
                warp_topk(v, id, K, my_v, my_i);
                if (nsplit == 1) {
                    write_topk(my_v, my_i, K, t, ids, w);
                } else if (lane < K) {
                    cand_v[(t * nsplit + blockIdx.y) * K + lane] = my_v;
                    cand_i[(t * nsplit + blockIdx.y) * K + lane] = my_i;
                }
            }
            __syncthreads();  // the rows are rewritten for the next 64 tokens
        }
    }
    if (!ok) *abort_flag = 1;
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)kRMaxE);
    }
}

// Two parts of E: the top-K of each token's 2K candidates (lane l < 2K holds candidate l), then its weights.
__global__ void __launch_bounds__(256) router_merge_kernel(const float* __restrict__ cand_v,
                                                           const int32_t* __restrict__ cand_i, int64_t T, int K,
                                                           int32_t* __restrict__ ids, float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // the whole warp
    float v[1];
    int id[1];
    v[0] = lane < 2 * K ? cand_v[t * 2 * K + lane] : -INFINITY;
    id[0] = lane < 2 * K ? cand_i[t * 2 * K + lane] : 0x7fffffff;
    float my_v;
    int my_i;
    warp_topk(v, id, K, my_v, my_i);
    write_topk(my_v, my_i, K, t, ids, w);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn router_encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool bf16_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = router_encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kRK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_router_topk(const float* x, const uint16_t* wr, int64_t T, int H, int E, int K, uint16_t* work,
                               int32_t* ids, float* w, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    static uint64_t attr_done = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !(attr_done & (1ull << dev))) {
        const cudaError_t err =
            cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
        if (err != cudaSuccess) return err;
        attr_done |= 1ull << dev;
    }
    uint16_t* xh = work;
    uint16_t* xl = work + T * (int64_t)H;
    const int64_t n8 = T * (int64_t)H / 8;
    const int64_t blocks = (n8 + 255) / 256;
    router_split_kernel<<<(unsigned)(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, s>>>(
        reinterpret_cast<const float4*>(x), n8, reinterpret_cast<uint4*>(xh), reinterpret_cast<uint4*>(xl));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int nsplit = E > kRMaxN ? 2 : 1;
    const int En = E / nsplit;
    // candidates of the two parts (after the split planes): logits fp32 [T][2][K], ids int32 [T][2][K]
    float* cand_v = reinterpret_cast<float*>(work + 2 * T * (int64_t)H);
    int32_t* cand_i = reinterpret_cast<int32_t*>(cand_v + T * 2 * kRMaxCand);
    RouterMaps maps;
    if (!bf16_map(&maps.xh, xh, (uint64_t)H, (uint64_t)T, kRM) || !bf16_map(&maps.xl, xl, (uint64_t)H, (uint64_t)T, kRM) ||
        !bf16_map(&maps.wr, wr, (uint64_t)H, (uint64_t)E, (uint32_t)En))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((T + kRM - 1) / kRM), (unsigned)nsplit);
    router_topk_kernel<<<grid, kRThreads, kRSmem, s>>>(maps, T, H, E, K, ids, w, cand_v, cand_i);
    err = cudaGetLastError();
    if (err != cudaSuccess || nsplit == 1) return err;
    router_merge_kernel<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(cand_v, cand_i, T, K, ids, w);
    return cudaGetLastError();
}

}  // namespace smoe
