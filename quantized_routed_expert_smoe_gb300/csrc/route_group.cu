// route_group.cu -- steps 1 and 2 of the routed-expert block: the warp-level top-K router and the GPU grouping of the
// (token, k) pairs by expert (a stable counting sort).
//
// route:  page "src/prefill/prefill.cpp", Prefill::run, MoE half, route(logits, ids, w, T, n_expert) -- softmax over
//         the experts, top-K, weights renormalised over the K; ties to the lower id as in the engine's top-k
//         kernels (page "Strata compare v0.1.35...v0.1.37", qsa_select.hpp).
// group:  page "src/prefill/prefill.cpp", the host grouping loop (counts, exclusive offsets, slot[i] = row,
//         src[row] = i / K, in pair order), moved onto the GPU as moe_fused.hpp group() does.
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <mutex>

#include "smoe_device.cuh"
#include "smoe_internal.h"

namespace smoe {
namespace {

// ------------------------------------------------------------------------------------------------ route
// One warp per token.  Every logit becomes a 64-bit key that orders like (value descending, expert id ascending):
// the high word maps the fp32 value to an unsigned integer of the same order (-0 taken as +0, so that equal values
// tie and the lower id wins, as in a float comparison), the low word is 0xFFFF - id.  The largest key is the best
// expert.  Lane l holds the logits of experts 4l..4l+3 + 128 i (float4 loads) and keeps its own three largest keys in
// order; each of the K rounds takes the warp's largest head by two warp reductions and the lane that owned it pops
// it.  Winners leave in descending key order, so a lane that has popped all three rescans its keys below the last one
// it popped.  Lane k keeps round k's winner; the K weights are exp(l_k - l_1) / sum_j exp(l_j - l_1), summed in k
// order.
__device__ __forceinline__ uint64_t route_key(float v, int e) {
    if (v == 0.0f) v = 0.0f;  // -0 -> +0
    const uint32_t b = __float_as_uint(v);
    const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((uint64_t)o << 32) | (uint32_t)(0xFFFF - e);
}
__device__ __forceinline__ float key_value(uint64_t k) {
    const uint32_t o = (uint32_t)(k >> 32);
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ int key_id(uint64_t k) { return 0xFFFF - (int)(k & 0xFFFFu); }

// the lane's three largest keys below `bound` among kv (0 = empty), in order
template <int NV>
__device__ __forceinline__ void top3(const uint64_t (&kv)[NV], uint64_t bound, uint64_t& a, uint64_t& b,
                                     uint64_t& c) {
    a = b = c = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const uint64_t k = kv[i] < bound ? kv[i] : 0ull;
        if (k > c) {
            if (k > b) {
                c = b;
                if (k > a) {
                    b = a;
                    a = k;
                } else {
                    b = k;
                }
            } else {
                c = k;
            }
        }
    }
}

template <int VPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int K,
                                                         int32_t* __restrict__ ids, float* __restrict__ w) {
    constexpr int NQ = VPL / 4;  // float4 loads a lane
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* lt = logits + t * E;
    uint64_t kv[VPL];
    const bool vec = (E & 3) == 0;  // rows 16-byte aligned: E % 4 == 0 (the pointer itself is 16-byte aligned)
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        const int e0 = 128 * i + 4 * lane;
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (vec && e0 + 3 < E) f = __ldg(reinterpret_cast<const float4*>(lt + e0));
        else if (e0 < E) {
            f.x = __ldg(lt + e0);
            if (e0 + 1 < E) f.y = __ldg(lt + e0 + 1);
            if (e0 + 2 < E) f.z = __ldg(lt + e0 + 2);
            if (e0 + 3 < E) f.w = __ldg(lt + e0 + 3);
        }
        kv[4 * i + 0] = e0 + 0 < E ? route_key(f.x, e0 + 0) : 0ull;
        kv[4 * i + 1] = e0 + 1 < E ? route_key(f.y, e0 + 1) : 0ull;
        kv[4 * i + 2] = e0 + 2 < E ? route_key(f.z, e0 + 2) : 0ull;
        kv[4 * i + 3] = e0 + 3 < E ? route_key(f.w, e0 + 3) : 0ull;
    }
    uint64_t h0, h1, h2;
    top3(kv, ~0ull, h0, h1, h2);
    int popped = 0;
    uint64_t mine = 0;
    for (int k = 0; k < K; ++k) {
        // the warp's largest head as two 32-bit reductions: the largest high word, then the largest low word among
        // the lanes that hold it (the 64-bit order is lexicographic in the two words)
        const uint32_t hh = (uint32_t)(h0 >> 32);
        const uint32_t bh = __reduce_max_sync(0xffffffffu, hh);
        const uint32_t bl = __reduce_max_sync(0xffffffffu, hh == bh ? (uint32_t)h0 : 0u);
        const uint64_t best = ((uint64_t)bh << 32) | bl;
        if (lane == k) mine = best;
        if (best == h0) {  // this lane owned the winner (keys are unique): pop it
            h0 = h1;
            h1 = h2;
            h2 = 0;
            if (++popped % 3 == 0) top3(kv, best, h0, h1, h2);
        }
    }
    const float lmax = key_value(__shfl_sync(0xffffffffu, mine, 0));
    const float mv = key_value(mine);
    const float ex = lane < K ? expf(mv - lmax) : 0.0f;
    float sum = 0.0f;
    for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, ex, k);
    if (lane < K) {
        ids[t * K + lane] = key_id(mine);
        w[t * K + lane] = __fdiv_rn(ex, sum);
    }
}

// ------------------------------------------------------------------------------------------------ group
constexpr int kGroupThreads = 1024;
constexpr int kMaxChunks = 48;  // chunks * E int32 counts fit the scan's shared memory

// pass 1: per chunk of pairs, the count of each expert (chunk b covers pairs [b*chunk, (b+1)*chunk)).
__global__ void __launch_bounds__(kGroupThreads) group_hist_kernel(const int32_t* __restrict__ ids, int64_t n, int E,
                                                                   int64_t chunk, int32_t* __restrict__ hist,
                                                                   int32_t* __restrict__ tiles) {
    extern __shared__ int32_t cnt[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int64_t p0 = (int64_t)blockIdx.x * chunk, p1 = min(n, p0 + chunk);
    bool bad = false;
    for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const int32_t e = ids[p];
        if (e < 0 || e >= E) bad = true;
        else atomicAdd(&cnt[e], 1);
    }
    if (bad) tiles[1] = SMOE_ERR_RANGE;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = cnt[e];
}

// block-wide exclusive scan of one value per thread (blockDim.x == 1024); returns the exclusive prefix, *total = sum
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        warp_sums[lane] = s;  // inclusive
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[31];
    __syncthreads();
    return before;
}

// pass 2 (one block, thread e = expert e): counts, offsets, each chunk's first row for each expert, and the tile
// list (each expert's c rows in ceil(c / 192) near-equal tiles, experts in id order).  The [chunks][E] counts are
// staged in shared memory by one coalesced sweep.
__global__ void __launch_bounds__(kGroupThreads) group_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E,
                                                                   int64_t n, int32_t* __restrict__ counts,
                                                                   int32_t* __restrict__ offsets,
                                                                   int32_t* __restrict__ tiles) {
    extern __shared__ int32_t hs[];
    __shared__ int warp_sums[32];
    const int total_cells = nchunks * E;
    // eight loads in flight a thread (a load-then-store loop would wait out every load's latency in turn)
    constexpr int kBatch = 8;
    for (int i0 = 0; i0 < total_cells; i0 += kBatch * kGroupThreads) {
        int32_t h[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kGroupThreads + threadIdx.x;
            h[u] = i < total_cells ? hist[i] : 0;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kGroupThreads + threadIdx.x;
            if (i < total_cells) hs[i] = h[u];
        }
    }
    __syncthreads();
    const int e = threadIdx.x;
    int c = 0;
    if (e < E) {
#pragma unroll 8
        for (int b = 0; b < nchunks; ++b) c += hs[b * E + e];
    }
    int total;
    const int off = block_exclusive_scan(e < E ? c : 0, warp_sums, &total);
    if (e < E) {
        counts[e] = c;
        offsets[e] = off;
        int run = off;
        for (int b = 0; b < nchunks; ++b) {
            const int h = hs[b * E + e];
            hs[b * E + e] = run;
            run += h;
        }
    }
    if (e == 0) offsets[E] = total;
    __syncthreads();
    for (int i = threadIdx.x; i < total_cells; i += blockDim.x) hist[i] = hs[i];
    const int nt = (e < E) ? (c + SMOE_TILE_ROWS - 1) / SMOE_TILE_ROWS : 0;
    int nt_total;
    const int tb = block_exclusive_scan(nt, warp_sums, &nt_total);
    int4* tl = reinterpret_cast<int4*>(tiles) + 1;
    for (int i = 0; i < nt; ++i) {
        const int a = (int)((int64_t)i * c / nt), b = (int)((int64_t)(i + 1) * c / nt);
        tl[tb + i] = make_int4(e, off + a, b - a, 0);
    }
    if (e == 0) {
        tiles[0] = nt_total;
        tiles[2] = (int32_t)n;
    }
}

// pass 3: per chunk, in pair order, each pair's row = (its chunk's first row of the expert) + (earlier pairs of the
// expert in the chunk).  Rounds of 1024 pairs: inside a warp __match_any_sync gives the rank among equal experts;
// across the warps of a round a [32][E] table of per-warp counts gives the pairs of earlier warps.
__global__ void __launch_bounds__(kGroupThreads) group_scatter_kernel(const int32_t* __restrict__ ids, int64_t n,
                                                                      int K, int E, int64_t chunk,
                                                                      const int32_t* __restrict__ hist,
                                                                      int32_t* __restrict__ src,
                                                                      int32_t* __restrict__ slot) {
    extern __shared__ int32_t sm[];
    int32_t* run = sm;                                            // [E]
    uint16_t* wcnt = reinterpret_cast<uint16_t*>(sm + E);         // [32][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        run[e] = hist[(int64_t)blockIdx.x * E + e];
        for (int w2 = 0; w2 < 32; ++w2) wcnt[w2 * E + e] = 0;
    }
    __syncthreads();
    const int64_t p0 = (int64_t)blockIdx.x * chunk, p1 = min(n, p0 + chunk);
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int64_t base = p0; base < p1; base += blockDim.x) {
        const int64_t p = base + threadIdx.x;
        int32_t e = p < p1 ? ids[p] : -1;
        if (e >= E) e = -1;
        if (e < -1) e = -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        if (e >= 0 && rank == 0) wcnt[warp * E + e] = (uint16_t)__popc(peers);
        __syncthreads();
        if (e >= 0) {
            int pre = 0;
            for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * E + e];
            const int32_t row = run[e] + pre + rank;
            slot[p] = row;
            src[row] = (int32_t)(p / K);
        } else if (p < p1) {
            slot[p] = -1;
        }
        __syncthreads();
        for (int e2 = threadIdx.x; e2 < E; e2 += blockDim.x) {
            int s = 0;
            for (int w2 = 0; w2 < 32; ++w2) {
                s += wcnt[w2 * E + e2];
                wcnt[w2 * E + e2] = 0;
            }
            run[e2] += s;
        }
        __syncthreads();
    }
}

// The scan and scatter kernels take more than 48 KB of dynamic shared memory at the largest E; the attribute that
// allows it is set per device (it does not carry over to another device), once, and only marked done on success.
cudaError_t group_attributes() {
    static std::mutex mu;
    static uint64_t done = 0;  // one bit per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done & (1ull << dev)) return cudaSuccess;
    err = cudaFuncSetAttribute(group_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMaxChunks * SMOE_MAX_EXPERTS * (int)sizeof(int32_t));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(group_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)((size_t)SMOE_MAX_EXPERTS * 4 + (size_t)32 * SMOE_MAX_EXPERTS * 2));
    if (err != cudaSuccess) return err;
    done |= 1ull << dev;
    return cudaSuccess;
}

int64_t group_chunk(int64_t n) {
    int64_t chunk = (n + kMaxChunks - 1) / kMaxChunks;
    chunk = (chunk + kGroupThreads - 1) / kGroupThreads * kGroupThreads;
    return chunk < kGroupThreads ? kGroupThreads : chunk;
}

}  // namespace

size_t group_work_bytes(int64_t n, int E) {
    const int64_t chunks = n > 0 ? (n + group_chunk(n) - 1) / group_chunk(n) : 1;
    return (size_t)chunks * (size_t)E * sizeof(int32_t);
}

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int K, int32_t* ids, float* w,
                              cudaStream_t s) {
    const int warps = 8;
    const dim3 grid((unsigned)((T + warps - 1) / warps)), block(32 * warps);
    if (E <= 128) route_topk_kernel<4><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E <= 256) route_topk_kernel<8><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E <= 512) route_topk_kernel<16><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else route_topk_kernel<32><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    return cudaGetLastError();
}

cudaError_t launch_group(const int32_t* ids, int64_t n, int K, int E, int32_t* counts, int32_t* offsets,
                         int32_t* src, int32_t* slot, int32_t* tiles, int32_t* hist, cudaStream_t s) {
    cudaError_t err = cudaMemsetAsync(tiles, 0, 4 * sizeof(int32_t), s);
    if (err != cudaSuccess) return err;
    const int64_t chunk = group_chunk(n);
    const int nchunks = n > 0 ? (int)((n + chunk - 1) / chunk) : 0;
    if (nchunks > 0) {
        group_hist_kernel<<<nchunks, kGroupThreads, E * sizeof(int32_t), s>>>(ids, n, E, chunk, hist, tiles);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if ((err = group_attributes()) != cudaSuccess) return err;
    group_scan_kernel<<<1, kGroupThreads, (size_t)nchunks * E * sizeof(int32_t), s>>>(hist, nchunks, E, n, counts,
                                                                                       offsets, tiles);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (nchunks > 0) {
        const size_t smem = (size_t)E * sizeof(int32_t) + (size_t)32 * E * sizeof(uint16_t);
        group_scatter_kernel<<<nchunks, kGroupThreads, smem, s>>>(ids, n, K, E, chunk, hist, src, slot);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace smoe
