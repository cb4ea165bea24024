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
// One warp per token.  Every logit has a key that orders like (value descending, expert id ascending), as two 32-bit
// words: the high word maps the fp32 value to an unsigned integer of the same order (-0 taken as +0, so that equal
// values tie and the lower id wins, as in a float comparison), the low word is 0xFFFF - id.  The largest key is the
// best expert.  Lane l holds the logits of experts 128 i + 4 l + j (float4 loads; position 4 i + j of the lane), so a
// lane meets its experts in increasing id order and needs only the high words to order its own keys: with strict
// comparisons, of two equal values the earlier (lower id, larger key) stays ahead.  It keeps its three largest keys
// in order; each of the K rounds takes the warp's largest head by two warp reductions (the largest high word, then
// the largest low word among the lanes holding it) and the lane that owned it pops it.  Winners leave in descending
// key order, so a lane that has popped all three rescans its keys below the last one it popped.  Lane k keeps round
// k's winner; the K weights are exp(l_k - l_1) / sum_j exp(l_j - l_1), summed in k order.  A high word of 0 marks an
// empty place (an expert id >= E); the only value it also stands for is one NaN bit pattern, and NaN logits have no
// order.
__device__ __forceinline__ uint32_t key_hi(float v) {
    if (v == 0.0f) v = 0.0f;  // -0 -> +0
    const uint32_t b = __float_as_uint(v);
    return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);  // negative: ~b; else b | sign bit
}
__device__ __forceinline__ float key_value(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// The lane's three largest keys (a >= b >= c as high word h and low word l; h = 0: none), among its places after
// (below) the key (bh, bl) when kBounded, else among all.  Place p holds high word kh[p] and low word lo0 - off(p).
template <int VPL, bool kBounded>
__device__ __forceinline__ void lane_top3(const uint32_t (&kh)[VPL], uint32_t lo0, uint32_t bh, uint32_t bl,
                                          uint32_t& ah, uint32_t& al, uint32_t& bh2, uint32_t& bl2, uint32_t& ch,
                                          uint32_t& cl) {
    ah = bh2 = ch = 0u;
    al = bl2 = cl = 0u;
#pragma unroll
    for (int p = 0; p < VPL; ++p) {
        const uint32_t lo = lo0 - (uint32_t)(128 * (p >> 2) + (p & 3));
        uint32_t h = kh[p];
        // below the bound: a smaller high word, or the same one at a later place (a higher id)
        if (kBounded && !(h < bh || (h == bh && lo < bl))) h = 0u;
        const bool ga = h > ah, gb = h > bh2, gc = h > ch;
        ch = gb ? bh2 : (gc ? h : ch);
        cl = gb ? bl2 : (gc ? lo : cl);
        bh2 = ga ? ah : (gb ? h : bh2);
        bl2 = ga ? al : (gb ? lo : bl2);
        ah = ga ? h : ah;
        al = ga ? lo : al;
    }
}

template <int VPL, bool kFull>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int K,
                                                         int32_t* __restrict__ ids, float* __restrict__ w) {
    constexpr int NQ = VPL / 4;  // float4 loads a lane
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* lt = logits + t * E;
    uint32_t kh[VPL];
    const bool vec = kFull || (E & 3) == 0;  // rows 16-byte aligned: E % 4 == 0 (the pointer itself is 16-byte aligned)
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        const int e0 = 128 * i + 4 * lane;
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kFull || (vec && e0 + 3 < E)) f = __ldg(reinterpret_cast<const float4*>(lt + e0));
        else if (e0 < E) {
            f.x = __ldg(lt + e0);
            if (e0 + 1 < E) f.y = __ldg(lt + e0 + 1);
            if (e0 + 2 < E) f.z = __ldg(lt + e0 + 2);
            if (e0 + 3 < E) f.w = __ldg(lt + e0 + 3);
        }
        kh[4 * i + 0] = (kFull || e0 + 0 < E) ? key_hi(f.x) : 0u;
        kh[4 * i + 1] = (kFull || e0 + 1 < E) ? key_hi(f.y) : 0u;
        kh[4 * i + 2] = (kFull || e0 + 2 < E) ? key_hi(f.z) : 0u;
        kh[4 * i + 3] = (kFull || e0 + 3 < E) ? key_hi(f.w) : 0u;
    }
    const uint32_t lo0 = 0xFFFFu - 4u * (uint32_t)lane;
    uint32_t ah, al, bh, bl, ch, cl;
    lane_top3<VPL, false>(kh, lo0, 0u, 0u, ah, al, bh, bl, ch, cl);
    int left = 3;  // heads the lane holds before it must rescan
    uint32_t mine_h = 0u, mine_l = 0u;
    for (int k = 0; k < K; ++k) {
        const uint32_t wh = __reduce_max_sync(0xffffffffu, ah);
        const uint32_t wl = __reduce_max_sync(0xffffffffu, ah == wh ? al : 0u);
        if (lane == k) {
            mine_h = wh;
            mine_l = wl;
        }
        if (ah == wh && al == wl) {  // this lane owned the winner (keys are unique): pop it
            ah = bh;
            al = bl;
            bh = ch;
            bl = cl;
            ch = 0u;
            cl = 0u;
            if (--left == 0) {
                lane_top3<VPL, true>(kh, lo0, wh, wl, ah, al, bh, bl, ch, cl);
                left = 3;
            }
        }
    }
    const float lmax = key_value(__shfl_sync(0xffffffffu, mine_h, 0));
    const float mv = key_value(mine_h);
    const float ex = lane < K ? expf(mv - lmax) : 0.0f;
    float sum = 0.0f;
    for (int k = 0; k < K; ++k) sum += __shfl_sync(0xffffffffu, ex, k);
    if (lane < K) {
        ids[t * K + lane] = 0xFFFF - (int)mine_l;
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
    const int64_t p0 = (int64_t)blockIdx.x * chunk, p1 = min(n, p0 + chunk);
    // the first round's ids are loaded before the tables are set up, each later round's during the round before
    int32_t e_next = p0 + threadIdx.x < p1 ? ids[p0 + threadIdx.x] : -1;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        run[e] = hist[(int64_t)blockIdx.x * E + e];
        for (int w2 = 0; w2 < 32; ++w2) wcnt[w2 * E + e] = 0;
    }
    __syncthreads();
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int64_t base = p0; base < p1; base += blockDim.x) {
        const int64_t p = base + threadIdx.x;
        int32_t e = e_next;
        const int64_t pn = p + blockDim.x;
        e_next = pn < p1 ? ids[pn] : -1;
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
    // E a whole number of 128-expert rows: every place of every lane holds an expert (no range checks)
    if (E == 128) route_topk_kernel<4, true><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E == 256) route_topk_kernel<8, true><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E == 512) route_topk_kernel<16, true><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E == 1024) route_topk_kernel<32, true><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E <= 128) route_topk_kernel<4, false><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E <= 256) route_topk_kernel<8, false><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else if (E <= 512) route_topk_kernel<16, false><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
    else route_topk_kernel<32, false><<<grid, block, 0, s>>>(logits, T, E, K, ids, w);
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
