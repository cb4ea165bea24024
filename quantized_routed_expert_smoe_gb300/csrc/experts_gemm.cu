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
// small expert wastes little).  Warp roles (three warpgroups, registers rebalanced with setmaxnreg):
//   warpgroup 0   warp 0: tensor-memory allocation and, on one lane, the MMAs of each slice;
//                 warps 1-3: producers -- cp.async copies of each slice's 2-bit weight codes, int8 rows (gathered
//                 through src) and scales into a ring of up to 16 slices in shared memory;
//   warpgroups 1-2  converters: decode a ring slice into the fp16 operand tiles of one of two stages (K-major,
//                 128-byte swizzle), then add the previous slice's partial from tensor memory into their registers;
//                 at the end they write the fp32 rows.
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
constexpr int kBK = 64;                        // K values per slice: one 128-byte swizzle row of fp16
constexpr int kMaxBN = SMOE_TILE_ROWS;         // routed rows per tile (MMA N <= 256)
constexpr int kStages = 2;                     // fp16 operand stages
constexpr int kThreads = 384;                  // three warpgroups
constexpr int kProducers = 96;                 // warps 1-3
constexpr int kConverters = 256;               // warpgroups 1-2
constexpr int kATile = kBM * 128;              // 16 KB of fp16 weights
constexpr int kBTile = kMaxBN * 128;           // 32 KB of fp16 activations (one of hi / lo)
constexpr int kStage = kATile + 2 * kBTile;
constexpr int kRingBytes = 64 * 1024;          // raw-data ring
constexpr int kMaxRing = 16;                   // slices in flight at most
constexpr uint32_t kTmemCols = 512;            // two fp32 partial buffers, 128 lanes x N <= 256 columns each
// shared memory: [1 KB alignment slack][stages][ring][src rows 1 KB][barriers]
constexpr int kSmemBytes = 1024 + kStages * kStage + kRingBytes + 1024 + 512;
// registers: launched at 168 a thread (384 x 168 = 64,512 of 65,536); warpgroup 0 gives back to 56 and the two
// converter warpgroups take 224: 128 x 56 + 256 x 224 = 64,512.
constexpr int kRegsWg0 = 56;
constexpr int kRegsConv = 224;

// Raw slice layout in the ring (one 64-wide K slice of the tile): weight codes [128][16 B], weight scales [128][4 B],
// activation codes [N][64 B], activation scales [N][4 B].
__host__ __device__ constexpr int raw_slice_bytes(int N) { return (2048 + 512 + N * 68 + 127) & ~127; }

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// arrive on `bar` once every cp.async this thread issued so far has landed (the arrival counts toward the phase)
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// This thread's 32 weights of one row into 4 16-byte chunks of the row's swizzled line: d * (q - 2).
// `codes` holds 32 2-bit codes, value i at bits 2i..2i+1 of the 64-bit word.
__device__ __forceinline__ void decode_weights(uint2 codes, uint16_t scale, uint4* row_line, int row, int half) {
    const __half2 d2 = __half2half2(__ushort_as_half(scale));
    const __half2 k1026 = __float2half2_rn(1026.0f);
    uint32_t h[16];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const uint32_t w = g ? codes.y : codes.x;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            // values m and m+8 as fp16 1024 + q in the two halves, then (1024 + q - 1026) * d = d * (q - 2)
            const uint32_t v = ((w >> (2 * m)) & 0x00030003u) | 0x64006400u;
            h[8 * g + m] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(v), k1026), d2));
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
        row_line[(half * 4 + c) ^ (row & 7)] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
}

// 32 int8 activations of one row into the hi and lo tiles: hi = fp16_rn(d q), lo = d q - hi (exact).
__device__ __forceinline__ void split_activations(uint4 c0, uint4 c1, uint16_t scale, uint4* hi_line,
                                                  uint4* lo_line, int row, int half) {
    const __half2 d2 = __half2half2(__ushort_as_half(scale));
    const __half2 k1152 = __float2half2_rn(1152.0f);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
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
        const int pc = (half * 4 + c) ^ (row & 7);
        hi_line[pc] = make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
        lo_line[pc] = make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
    }
}

__device__ __forceinline__ void zero_activations(uint4* hi_line, uint4* lo_line, int row, int half) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int pc = (half * 4 + c) ^ (row & 7);
        hi_line[pc] = make_uint4(0u, 0u, 0u, 0u);
        lo_line[pc] = make_uint4(0u, 0u, 0u, 0u);
    }
}

__global__ void __launch_bounds__(kThreads, 1) experts_gemm_kernel(const ExpertsGemmArgs p) {
    int32_t* tiles = p.tiles;
    const int ti = blockIdx.y;
    if (ti >= tiles[0] || tiles[1] != 0) return;  // no such tile, or the grouping failed: nothing to do
    const int4 tile = reinterpret_cast<const int4*>(tiles)[1 + ti];
    const int e = tile.x, row0 = tile.y, rows = tile.z;
    if (rows <= 0 || rows > kMaxBN) return;
    const int N = (rows + 15) & ~15;
    const int m0 = blockIdx.x * kBM;
    const int nk = p.K / kBK;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    uint8_t* ring = smem + kStages * kStage;
    int32_t* srcs = reinterpret_cast<int32_t*>(ring + kRingBytes);          // [256] B row of each tile row
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kRingBytes + 1024);  // operand stage s is filled
    uint64_t* empty = full + kStages;                                         // ... and consumed by the MMAs
    uint64_t* pfull = empty + kStages;     // a slice's partial is complete in tensor-memory buffer b
    uint64_t* pempty = pfull + 2;          // the converters have added buffer b into their registers
    uint64_t* rfull = pempty + 2;          // ring slot r holds its slice [kMaxRing]
    uint64_t* rempty = rfull + kMaxRing;   // ring slot r has been read [kMaxRing]
    uint64_t* accf = rempty + kMaxRing;    // every MMA has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int sbytes = raw_slice_bytes(N);
    const int depth = min(kMaxRing, kRingBytes / sbytes);
    const int o_as = 2048, o_bc = 2560, o_bs = 2560 + N * 64;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kConverters);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&pfull[b], 1);
            mbar_init(&pempty[b], kConverters);
        }
        for (int r = 0; r < kMaxRing; ++r) {
            mbar_init(&rfull[r], kProducers);
            mbar_init(&rempty[r], kConverters);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // the B row of every tile row (rows past the tile: -1)
    for (int r = threadIdx.x; r < kMaxBN; r += kThreads)
        srcs[r] = r < rows ? (p.src ? p.src[row0 + r] : row0 + r) : -1;
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(smem);
    bool ok = true;

    if (warp < 4) {
        setmaxnreg_dec<kRegsWg0>();
        if (warp == 0) {
            // ------------------------------------------------------------------ MMA issue (one thread)
            if (lane == 0) {
                const uint32_t idesc = idesc_f16_f32(kBM, N);
                for (int kt = 0; kt < nk; ++kt) {
                    const int s = kt % kStages, b = kt & 1;
                    if (!mbar_wait(&full[s], (uint32_t)(kt / kStages) & 1u, abort_flag) ||
                        (kt >= 2 && !mbar_wait(&pempty[b], (uint32_t)(kt / 2 - 1) & 1u, abort_flag))) {
                        ok = false;
                        break;
                    }
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
                }
                mma_commit(accf);  // completes once every MMA issued above has completed (abort path included)
            }
            __syncwarp();
        } else {
            // ------------------------------------------------------------------ producers (96 threads)
            const int pt = threadIdx.x - 32;
            const int64_t wrow0 = (int64_t)e * p.a_rows + m0;
            const uint8_t* wc = p.wc + wrow0 * (p.K / 4);
            const uint16_t* ws = p.ws + wrow0 * (p.K / 32);
            const int items = 128 + 128 + N * 4 + N;  // weight code rows, weight scale pairs, row chunks, row scales
            for (int kt = 0; kt < nk; ++kt) {
                const int r = kt % depth;
                if (kt >= depth && !mbar_wait(&rempty[r], (uint32_t)(kt / depth - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t slot = smem_u32(ring) + (uint32_t)(r * sbytes);
                for (int i = pt; i < items; i += kProducers) {
                    if (i < 128) {
                        cp_async_16(slot + i * 16, wc + (int64_t)i * (p.K / 4) + kt * 16);
                    } else if (i < 256) {
                        const int row = i - 128;
                        cp_async_4(slot + o_as + row * 4, ws + (int64_t)row * (p.K / 32) + kt * 2);
                    } else if (i < 256 + N * 4) {
                        const int row = (i - 256) >> 2, ch = (i - 256) & 3;
                        const int32_t sr = srcs[row];
                        if (sr >= 0) cp_async_16(slot + o_bc + row * 64 + ch * 16, p.bc + (int64_t)sr * p.K + kt * kBK + ch * 16);
                    } else {
                        const int row = i - 256 - N * 4;
                        const int32_t sr = srcs[row];
                        if (sr >= 0) cp_async_4(slot + o_bs + row * 4, p.bs + (int64_t)sr * (p.K / 32) + kt * 2);
                    }
                }
                cp_async_arrive(&rfull[r]);
            }
            cp_async_wait_all();  // no copy may land after the CTA has moved on
        }
    } else {
        setmaxnreg_inc<kRegsConv>();
        // ------------------------------------------------------------------ converters (256 threads)
        const int ct = threadIdx.x - 128;
        const int ar = ct >> 1, half = ct & 1;  // weight row of this thread, and which 32 of the slice's 64 K
        const int br0 = ar, br1 = ar + 128;     // routed rows of this thread (two passes)
        const bool has0 = srcs[br0] >= 0, has1 = srcs[br1] >= 0;
        // promotion: this thread owns TMEM lane 32*q + lane (weight row mrow) and columns [chalf*128, +128)
        const int q = warp & 3;                 // the TMEM lane quarter this warp may access
        const int chalf = (warp - 4) >> 2;      // warpgroup 1: columns [0, 128); warpgroup 2: [128, 256)
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

        for (int kt = 0; kt < nk && ok; ++kt) {
            const int r = kt % depth;
            if (!mbar_wait(&rfull[r], (uint32_t)(kt / depth) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            const uint8_t* slot = ring + r * sbytes;
            const uint2 acodes = *reinterpret_cast<const uint2*>(slot + ar * 16 + half * 8);
            const uint16_t ascale = *reinterpret_cast<const uint16_t*>(slot + o_as + ar * 4 + half * 2);
            uint4 b0c0 = make_uint4(0, 0, 0, 0), b0c1 = b0c0, b1c0 = b0c0, b1c1 = b0c0;
            uint16_t b0s = 0, b1s = 0;
            if (has0) {
                const uint4* c = reinterpret_cast<const uint4*>(slot + o_bc + br0 * 64 + half * 32);
                b0c0 = c[0];
                b0c1 = c[1];
                b0s = *reinterpret_cast<const uint16_t*>(slot + o_bs + br0 * 4 + half * 2);
            }
            if (has1) {
                const uint4* c = reinterpret_cast<const uint4*>(slot + o_bc + br1 * 64 + half * 32);
                b1c0 = c[0];
                b1c1 = c[1];
                b1s = *reinterpret_cast<const uint16_t*>(slot + o_bs + br1 * 4 + half * 2);
            }
            mbar_arrive(&rempty[r]);
            const int s = kt % kStages;
            if (kt >= kStages && !mbar_wait(&empty[s], (uint32_t)(kt / kStages - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            uint8_t* st = smem + s * kStage;
            uint4* a_tile = reinterpret_cast<uint4*>(st);
            uint4* hi_tile = reinterpret_cast<uint4*>(st + kATile);
            uint4* lo_tile = reinterpret_cast<uint4*>(st + kATile + kBTile);
            decode_weights(acodes, ascale, a_tile + ar * 8, ar, half);
            if (br0 < N) {
                if (has0) split_activations(b0c0, b0c1, b0s, hi_tile + br0 * 8, lo_tile + br0 * 8, br0, half);
                else zero_activations(hi_tile + br0 * 8, lo_tile + br0 * 8, br0, half);
            }
            if (br1 < N) {
                if (has1) split_activations(b1c0, b1c1, b1s, hi_tile + br1 * 8, lo_tile + br1 * 8, br1, half);
                else zero_activations(hi_tile + br1 * 8, lo_tile + br1 * 8, br1, half);
            }
            fence_async_smem();
            mbar_arrive(&full[s]);
            if (kt >= 1 && !promote(kt - 1)) ok = false;
        }
        if (ok && !promote(nk - 1)) ok = false;
        if (ok) {
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
    if (!ok) {
        *abort_flag = 1;
        tiles[3] = SMOE_ERR_TIMEOUT;
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
