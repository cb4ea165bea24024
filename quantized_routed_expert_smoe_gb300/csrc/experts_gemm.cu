// experts_gemm.cu -- the grouped expert products of the routed-expert block (steps 4 and 6) on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), sm_103a.
//
// Page "Strata compare v0.1.35...v0.1.37", include/strata/prefill/moe_fused.hpp experts(): for each expert, gate/up
// of its routed rows from the per-token int8 activations (gathered through src) against its 2-bit weights, then
// down into one fp32 row per routed pair.  Per output:  sum_b dW[b] * dA[b] * sum_{i in b} (qW - 2) * qA.
//
// GB300 design.  The int8 tensor rate of this part is far below its fp16 rate, so the contraction runs as
// tcgen05.mma.kind::f16 on EXACT fp16 re-encodings of the two quantised operands:
//   - a weight d * (q - 2), q in {0..3}, is d times {-2, -1, 0, 1}: exactly representable in fp16;
//   - an activation d * q (fp16 d, |q| <= 127) needs up to 18 significant bits; it is split into
//     hi = fp16_rn(d * q) and lo = d * q - hi, which is exact in fp16 (at most 8 significant bits), so
//     hi + lo = d * q exactly.
// Every product of an fp16 weight and an fp16 hi/lo part is exact in the fp32 accumulator, so each output is the
// sum of the exact products d_w (q_w - 2) d_a q_a.  The K loop runs two MMAs per 16-wide K step (A x B_hi,
// A x B_lo).  The tensor core's fp32 accumulation aligns its addends with truncation, which over the 2 * K / 16 steps
// of a whole row costs about 3e-6 of the result -- enough to flip requantised H codes -- so the accumulation is
// two-level: each 64-wide K slice accumulates from zero into one of two tensor-memory buffers (the slice's partial is
// small, so its truncation error is too), and the converter warps add each finished slice into fp32 registers with
// round-to-nearest while the tensor core fills the other buffer.
//
// Tile: one CTA = one tile of the tile list (an expert and up to 256 of its routed rows, the MMA's N, a multiple of
// 16) x one 128-row slice of the expert's weight matrix (the MMA's M; swap-AB: weights are the M operand so that a
// small expert wastes little).  Eight warps read the 2-bit weight codes and the int8 rows from global memory, decode
// them into the fp16 operand tiles in shared memory (K-major, 128-byte swizzle, 64 K values per stage, two stages),
// promote each slice's partial from tensor memory into their registers, and finally write the fp32 rows; lane 0 of
// warp 0 also issues the MMAs of each stage once all eight warps have filled it.  (Eight warps, two per SM
// sub-partition, leave each thread up to 255 registers; the 128 fp32 sums a thread keeps need that room.)
//
// K order inside the operand tiles: within each group of 16 K values, shared-memory position 2m holds value m and
// position 2m+1 holds value m+8 (m = 0..7) -- the order in which 2-bit codes unpack in pairs -- for A and B alike, so
// the contraction is unchanged.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "smoe_device.cuh"
#include "smoe_internal.h"

namespace smoe {
namespace {

constexpr int kBM = 128;                       // weight rows per CTA (MMA M)
constexpr int kBK = 64;                        // K values per stage: one 128-byte swizzle row of fp16
constexpr int kMaxBN = SMOE_TILE_ROWS;         // routed rows per tile (MMA N <= 256)
constexpr int kStages = 2;
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;  // 256
constexpr int kThreads = kConvThreads;         // every warp converts and promotes; lane 0 of warp 0 issues MMAs
constexpr int kATile = kBM * 128;              // 16 KB of fp16 weights
constexpr int kBTile = kMaxBN * 128;           // 32 KB of fp16 activations (one of hi / lo)
constexpr int kStage = kATile + 2 * kBTile;
constexpr int kSmemBytes = 1024 + kStages * kStage + 256;
constexpr uint32_t kTmemCols = 512;            // two fp32 partial buffers, 128 lanes x N <= 256 columns each

struct AReg {
    uint2 codes;      // 32 2-bit codes
    uint16_t scale;   // their fp16 scale
};
struct BReg {
    uint4 c0, c1;     // 32 int8 codes
    uint16_t scale;
};

// 32 weights of one row (codes r) into 4 16-byte chunks of the row's swizzled shared-memory line: d * (q - 2).
__device__ __forceinline__ void decode_weights(const AReg& r, uint32_t row_addr, int row, int half) {
    const __half2 d2 = __half2half2(__ushort_as_half(r.scale));
    const __half2 k1026 = __float2half2_rn(1026.0f);
    uint32_t h[16];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const uint32_t w = g ? r.codes.y : r.codes.x;  // 16 codes: value i at bits 2i..2i+1
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            // values m and m+8 as fp16 1024 + q in the two halves, then (1024 + q - 1026) * d = d * (q - 2)
            const uint32_t v = ((w >> (2 * m)) & 0x00030003u) | 0x64006400u;
            h[8 * g + m] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(v), k1026), d2));
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int lc = half * 4 + c;
        st_shared_v4(row_addr + ((uint32_t)(lc ^ (row & 7)) << 4), h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
    }
}

// 32 int8 activations of one row into the hi and lo tiles: hi = fp16_rn(d q), lo = d q - hi (exact).
__device__ __forceinline__ void split_activations(const BReg& r, uint32_t hi_addr, uint32_t lo_addr, int row,
                                                  int half) {
    const __half2 d2 = __half2half2(__ushort_as_half(r.scale));
    const __half2 k1152 = __float2half2_rn(1152.0f);
    const uint32_t w[8] = {r.c0.x, r.c0.y, r.c0.z, r.c0.w, r.c1.x, r.c1.y, r.c1.z, r.c1.w};
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            // bytes of values m and m+8 of the group into the low bytes of two halves; (b ^ 0x80) = b + 128 for a
            // signed byte b, so the halves read 1024 + 128 + q
            const uint32_t t = __byte_perm(w[4 * g + (m >> 2)], w[4 * g + 2 + (m >> 2)], (m & 3) | ((4 + (m & 3)) << 8));
            const uint32_t v = (t & 0x00FF00FFu) ^ 0x64806480u;
            const __half2 q = __hsub2(u32_as_h2(v), k1152);
            const __half2 ph = __hmul2(q, d2);
            const __half2 pl = __hfma2(q, d2, __hneg2(ph));
            hi[8 * g + m] = h2_as_u32(ph);
            lo[8 * g + m] = h2_as_u32(pl);
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t off = (uint32_t)((half * 4 + c) ^ (row & 7)) << 4;
        st_shared_v4(hi_addr + off, hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
        st_shared_v4(lo_addr + off, lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
    }
}

__device__ __forceinline__ void zero_activations(uint32_t hi_addr, uint32_t lo_addr, int row, int half) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t off = (uint32_t)((half * 4 + c) ^ (row & 7)) << 4;
        st_shared_v4(hi_addr + off, 0u, 0u, 0u, 0u);
        st_shared_v4(lo_addr + off, 0u, 0u, 0u, 0u);
    }
}

// 256 threads, two warps per sub-partition: up to 255 registers a thread; one CTA per SM (shared and tensor memory).
__global__ void __launch_bounds__(kThreads, 1) experts_gemm_kernel(const ExpertsGemmArgs p) {
    int32_t* tiles = p.tiles;
    const int ti = blockIdx.y;
    if (ti >= tiles[0] || tiles[1] != 0) return;  // no such tile, or the grouping failed: nothing to do
    const int4 tile = reinterpret_cast<const int4*>(tiles)[1 + ti];
    const int e = tile.x, row0 = tile.y, rows = tile.z;
    if (rows <= 0 || rows > kMaxBN) return;
    const int N = (rows + 15) & ~15;
    const int m0 = blockIdx.x * kBM;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStage);
    uint64_t* empty = full + kStages;
    uint64_t* pfull = empty + kStages;   // a slice's partial is complete in tensor-memory buffer b
    uint64_t* pempty = pfull + 2;        // the converters have added buffer b into their registers
    uint64_t* accf = pempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kConvThreads);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&pfull[b], 1);
            mbar_init(&pempty[b], kConvThreads);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int nk = p.K / kBK;
    const uint32_t sbase = smem_u32(smem);

    {
        const int ct = threadIdx.x;
        const int ar = ct >> 1, half = ct & 1;  // weight row of this thread, and which 32 of the stage's 64 K
        const int64_t arow = (int64_t)e * p.a_rows + m0 + ar;
        const uint2* acodes = reinterpret_cast<const uint2*>(p.wc + arow * (p.K / 4)) + half;
        const uint16_t* ascales = p.ws + arow * (p.K / 32) + half;
        const int br0 = ar, br1 = ar + 128;     // routed rows of this thread (two passes)
        const int64_t bsrc0 = br0 < rows ? (p.src ? (int64_t)p.src[row0 + br0] : (int64_t)(row0 + br0)) : -1;
        const int64_t bsrc1 = br1 < rows ? (p.src ? (int64_t)p.src[row0 + br1] : (int64_t)(row0 + br1)) : -1;
        const int8_t* b0p = bsrc0 >= 0 ? p.bc + bsrc0 * p.K + half * 32 : nullptr;
        const int8_t* b1p = bsrc1 >= 0 ? p.bc + bsrc1 * p.K + half * 32 : nullptr;
        const uint16_t* b0s = bsrc0 >= 0 ? p.bs + bsrc0 * (p.K / 32) + half : nullptr;
        const uint16_t* b1s = bsrc1 >= 0 ? p.bs + bsrc1 * (p.K / 32) + half : nullptr;

        AReg an;
        BReg bn0, bn1;
        auto load = [&](int kt) {
            an.codes = __ldg(acodes + 2 * kt);
            an.scale = __ldg(ascales + 2 * kt);
            if (b0p) {
                const uint4* q = reinterpret_cast<const uint4*>(b0p + kt * kBK);
                bn0.c0 = __ldg(q);
                bn0.c1 = __ldg(q + 1);
                bn0.scale = __ldg(b0s + 2 * kt);
            }
            if (b1p) {
                const uint4* q = reinterpret_cast<const uint4*>(b1p + kt * kBK);
                bn1.c0 = __ldg(q);
                bn1.c1 = __ldg(q + 1);
                bn1.scale = __ldg(b1s + 2 * kt);
            }
        };
        // promotion: this thread owns TMEM lane 32*q + lane (weight row mrow) and columns [chalf*128, +128)
        const int q = warp & 3;             // the TMEM lane quarter this warp may access
        const int chalf = warp >> 2;        // warps 0-3: columns [0, 128); 4-7: [128, 256)
        const int mrow = 32 * q + lane;
        float acc[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
        auto promote = [&](int k) -> bool {
            const int b = k & 1;
            if (!mbar_wait(&pfull[b], (uint32_t)(k / 2) & 1u, abort_flag)) return false;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int c0 = chalf * 128 + 32 * c;
                if (c0 < N) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + 256u * (uint32_t)b + (uint32_t)c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[32 * c + i] += __uint_as_float(v[i]);
                }
            }
            tc_fence_before();
            mbar_arrive(&pempty[b]);
            return true;
        };
        // the MMAs of slice kt (lane 0 of warp 0): after every warp has filled stage kt and buffer kt & 1 has been
        // promoted (slice kt - 2)
        const uint32_t idesc = idesc_f16_f32(kBM, N);
        auto issue = [&](int kt) -> bool {
            const int s = kt % kStages, b = kt & 1;
            if (!mbar_wait(&full[s], (uint32_t)(kt / kStages) & 1u, abort_flag)) return false;
            if (kt >= 2 && !mbar_wait(&pempty[b], (uint32_t)(kt / 2 - 1) & 1u, abort_flag)) return false;
            tc_fence_after();
            const uint32_t a = sbase + s * kStage, bh = a + kATile, bl = bh + kBTile;
            const uint32_t d = tmem + 256u * (uint32_t)b;
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j) {
                const uint64_t ad = sdesc_k_sw128(a + 32 * j);
                mma_f16(d, ad, sdesc_k_sw128(bh + 32 * j), idesc, j > 0 ? 1u : 0u);
                mma_f16(d, ad, sdesc_k_sw128(bl + 32 * j), idesc, 1u);
            }
            mma_commit(&empty[s]);
            mma_commit(&pfull[b]);
            return true;
        };

        load(0);
        bool ok = true;
        for (int kt = 0; kt < nk && ok; ++kt) {
            const int s = kt % kStages;
            if (kt >= kStages && !mbar_wait(&empty[s], (uint32_t)(kt / kStages - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t sa = sbase + s * kStage, sh = sa + kATile, sl = sh + kBTile;
            decode_weights(an, sa + ar * 128, ar, half);
            if (br0 < N) {
                if (b0p) split_activations(bn0, sh + br0 * 128, sl + br0 * 128, br0, half);
                else zero_activations(sh + br0 * 128, sl + br0 * 128, br0, half);
            }
            if (br1 < N) {
                if (b1p) split_activations(bn1, sh + br1 * 128, sl + br1 * 128, br1, half);
                else zero_activations(sh + br1 * 128, sl + br1 * 128, br1, half);
            }
            fence_async_smem();
            mbar_arrive(&full[s]);
            if (warp == 0) {
                bool issued = true;
                if (lane == 0) issued = issue(kt);
                ok = __shfl_sync(0xffffffffu, issued ? 1 : 0, 0) != 0;
                if (!ok) break;
            }
            if (kt + 1 < nk) load(kt + 1);          // in flight while the previous slice is promoted
            if (kt >= 1 && !promote(kt - 1)) ok = false;
        }
        if (ok && !promote(nk - 1)) ok = false;
        if (warp == 0 && lane == 0) mma_commit(accf);  // completes once every MMA issued above has completed
        if (!ok) {
            *abort_flag = 1;
            tiles[3] = SMOE_ERR_TIMEOUT;
        } else {
            // ------------------------------------------------------------------ epilogue: fp32 rows out
            float* outcol = p.out + (m0 + mrow);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int col = chalf * 128 + 32 * c + i;
                    if (col < rows) outcol[(int64_t)(row0 + col) * p.a_rows] = acc[32 * c + i];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        mbar_wait(accf, 0, nullptr);  // every MMA has completed before the accumulator is released
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_experts_gemm(const ExpertsGemmArgs& a, int64_t max_tiles, cudaStream_t s) {
    int dev = 0;
    cudaGetDevice(&dev);
    static uint64_t attr_done = 0;  // one bit per device
    if (dev < 64 && !(attr_done & (1ull << dev))) {
        cudaError_t err = cudaFuncSetAttribute(experts_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSmemBytes);
        if (err != cudaSuccess) return err;
        attr_done |= 1ull << dev;
    }
    if (max_tiles <= 0) return cudaSuccess;
    const dim3 grid((unsigned)(a.a_rows / kBM), (unsigned)max_tiles);
    experts_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace smoe
