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
// two-level for gate/up (whose output is requantised): each 64-wide K slice accumulates from zero into one of two
// tensor-memory buffers (the partial is small, so its truncation error is too), and the converter warps add each
// finished partial into fp32 registers with round-to-nearest while the tensor core fills the other buffer.  One slice per partial keeps the
// requantised H of the smallest test chunk identical to the oracle's; two slices flipped one H scale there.  The down
// product feeds the fp32 combine only, so it accumulates the whole K in one buffer.
//
// Tile: one CTA = one tile of the tile list (an expert and up to 256 of its routed rows, the MMA's N, a multiple of
// 16) x one 128-row slice of the expert's weight matrix (the MMA's M; swap-AB: weights are the M operand so that a
// small expert wastes little).  Warp roles (three warpgroups, registers rebalanced with setmaxnreg):
//   warpgroup 0   warp 0: tensor-memory allocation and, on one lane, the MMAs of each slice;
//                 warps 1-3: producers -- each slice's packed weight block (codes and scales: one 2560-byte bulk
//                 copy) and the tile's q8 rows in slice form (codes and scales, 80 bytes a row: TMA tile::gather4
//                 loads through src, four rows each) into a ring of up to 16 slices in shared memory;
//   warpgroups 1-2  converters: decode a ring slice into the fp16 operand tiles of one of two stages (K-major,
//                 128-byte swizzle), 16 K values of one row per work item, then add the previous partial from tensor
//                 memory into their registers; at the end they write the fp32 rows.
//
// K order inside the operand tiles: within each group of 16 K values, shared-memory position 2m holds value m and
// position 2m+1 holds value m+8 (m = 0..7) -- the order in which 2-bit codes unpack in pairs -- for A and B alike, so
// the contraction is unchanged.
#include <cuda.h>
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

// Raw slice layout in the ring (one 64-wide K slice of the tile): the packed weight block (codes [128][16 B], scales
// [128][4 B]), then the tile's rows in slice form (80 B a row: 64 codes, 2 scales, padding), four rows per gather4
// load placed at a 384-byte stride so that every TMA destination is 128-byte aligned.
constexpr int kWBlock = 2560;
constexpr int kRowPiece = 80;
constexpr int kGroupStride = 384;  // 4 rows x 80 bytes, rounded up to 128
__host__ __device__ constexpr int raw_slice_bytes(int N) { return kWBlock + (N / 4) * kGroupStride; }

// bulk copy (no tensor map) of `bytes` (a multiple of 16) into shared memory, completing on `bar`
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// TMA: four rows (y0..y3) of a one-row-high box, placed one after another in shared memory
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0, int y1, int y2, int y3,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar)) : "memory");
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// 16 weights of one row (codes: value i at bits 2i..2i+1) into chunks 2*quarter and 2*quarter + 1 of the row's
// swizzled 128-byte line: d * (q - 2).
__device__ __forceinline__ void decode_weights16(uint32_t codes, uint16_t scale, uint4* row_line, int row,
                                                 int quarter) {
    const __half2 d2 = __half2half2(__ushort_as_half(scale));
    const __half2 k1026 = __float2half2_rn(1026.0f);
    uint32_t h[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        // values m and m+8 as fp16 1024 + q in the two halves, then (1024 + q - 1026) * d = d * (q - 2)
        const uint32_t v = ((codes >> (2 * m)) & 0x00030003u) | 0x64006400u;
        h[m] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(v), k1026), d2));
    }
    row_line[(2 * quarter) ^ (row & 7)] = make_uint4(h[0], h[1], h[2], h[3]);
    row_line[(2 * quarter + 1) ^ (row & 7)] = make_uint4(h[4], h[5], h[6], h[7]);
}

// 16 int8 activations of one row into the hi and lo tiles: hi = fp16_rn(d q), lo = d q - hi (exact).
__device__ __forceinline__ void split_activations16(uint4 c, uint16_t scale, uint4* hi_line, uint4* lo_line, int row,
                                                    int quarter) {
    const __half2 d2 = __half2half2(__ushort_as_half(scale));
    const __half2 k1152 = __float2half2_rn(1152.0f);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        // bytes of values m and m+8 into the low bytes of two halves; (b ^ 0x80) = b + 128 for a signed byte b, so
        // the halves read 1024 + 128 + q
        const uint32_t t = __byte_perm(w[m >> 2], w[2 + (m >> 2)], (m & 3) | ((4 + (m & 3)) << 8));
        const uint32_t v = (t & 0x00FF00FFu) ^ 0x64806480u;
        const __half2 q = __hsub2(u32_as_h2(v), k1152);
        const __half2 ph = __hmul2(q, d2);
        const __half2 pl = __hfma2(q, d2, __hneg2(ph));
        hi[m] = h2_as_u32(ph);
        lo[m] = h2_as_u32(pl);
    }
    const int c0 = (2 * quarter) ^ (row & 7), c1 = (2 * quarter + 1) ^ (row & 7);
    hi_line[c0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    hi_line[c1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    lo_line[c0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    lo_line[c1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
}

__device__ __forceinline__ void zero_activations16(uint4* hi_line, uint4* lo_line, int row, int quarter) {
    const int c0 = (2 * quarter) ^ (row & 7), c1 = (2 * quarter + 1) ^ (row & 7);
    hi_line[c0] = hi_line[c1] = lo_line[c0] = lo_line[c1] = make_uint4(0u, 0u, 0u, 0u);
}

struct GemmMaps {
    CUtensorMap b;  // q8 rows in slice form: [rows][K/64 * 80 bytes], box 80 bytes x 1 row (gather4)
};

__global__ void __launch_bounds__(kThreads, 1) experts_gemm_kernel(const ExpertsGemmArgs p,
                                                                   const __grid_constant__ GemmMaps maps) {
    int32_t* tiles = p.tiles;
    const int ti = blockIdx.y;
    if (ti >= tiles[0] || tiles[1] != 0) return;  // no such tile, or the grouping failed: nothing to do
    const int4 tile = reinterpret_cast<const int4*>(tiles)[1 + ti];
    const int e = tile.x, row0 = tile.y, rows = tile.z;
    if (rows <= 0 || rows > kMaxBN) return;
    const int N = (rows + 15) & ~15;
    const int m0 = blockIdx.x * kBM;
    const int nk = p.K / kBK;
    const int P = p.two_level ? 1 : nk;  // slices per tensor-memory partial

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
    const int o_as = 2048, o_b = kWBlock;  // weight scales, row pieces

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
            mbar_init(&rfull[r], 1);  // the arrival that posts the slice's byte count
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
                    // slices kt of partial g = kt / P go to buffer g & 1, which partial g - 2 has left
                    const int s = kt % kStages, g = kt / P, b = g & 1;
                    const bool first = kt % P == 0, last = kt % P == P - 1 || kt == nk - 1;
                    if (!mbar_wait(&full[s], (uint32_t)(kt / kStages) & 1u, abort_flag) ||
                        (first && g >= 2 && !mbar_wait(&pempty[b], (uint32_t)(g / 2 - 1) & 1u, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = sbase + s * kStage, bh = a + kATile, bl = bh + kBTile;
                    const uint32_t d = tmem + 256u * (uint32_t)b;
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j) {
                        const uint64_t ad = sdesc_k_sw128(a + 32 * j);
                        mma_f16(d, ad, sdesc_k_sw128(bh + 32 * j), idesc, (j > 0 || !first) ? 1u : 0u);
                        mma_f16(d, ad, sdesc_k_sw128(bl + 32 * j), idesc, 1u);
                    }
                    mma_commit(&empty[s]);
                    if (last) mma_commit(&pfull[b]);
                }
                mma_commit(accf);  // completes once every MMA issued above has completed (abort path included)
            }
            __syncwarp();
        } else {
            // ------------------------------------------------------------------ producers (96 threads)
            const int pt = threadIdx.x - 32;
            const uint8_t* wblocks = p.wp + ((int64_t)e * (p.a_rows / kBM) + blockIdx.x) * nk * (int64_t)kWBlock;
            const int groups = (rows + 3) >> 2;  // gather4 loads of this tile's rows
            const uint32_t tx_bytes = (uint32_t)kWBlock + (uint32_t)groups * 4u * kRowPiece;
            for (int kt = 0; kt < nk; ++kt) {
                const int r = kt % depth;
                if (kt >= depth && !mbar_wait(&rempty[r], (uint32_t)(kt / depth - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t slot = smem_u32(ring) + (uint32_t)(r * sbytes);
                if (pt == 0) {
                    mbar_arrive_expect_tx(&rfull[r], tx_bytes);
                    bulk_load(slot, wblocks + (int64_t)kt * kWBlock, kWBlock, &rfull[r]);
                }
                for (int g = pt; g < groups; g += kProducers) {
                    const int r0 = 4 * g;
                    const int y0 = srcs[r0];
                    const int y1 = r0 + 1 < rows ? srcs[r0 + 1] : y0;
                    const int y2 = r0 + 2 < rows ? srcs[r0 + 2] : y0;
                    const int y3 = r0 + 3 < rows ? srcs[r0 + 3] : y0;
                    tma_gather4(slot + o_b + g * kGroupStride, &maps.b, kt * kRowPiece, y0, y1, y2, y3, &rfull[r]);
                }
            }
        }
    } else {
        setmaxnreg_inc<kRegsConv>();
        // ------------------------------------------------------------------ converters (256 threads)
        const int ct = threadIdx.x - 128;
        // work items of 16 K values: weight items ct and ct + 256 (row = item / 4, quarter = item % 4); row items
        // ct + 256 i of the tile's 4 N (row, quarter) pairs
        const int nb = (4 * N - ct + 255) / 256;     // row items of this thread (0..4)
        // promotion: this thread owns TMEM lane 32*q + lane (weight row mrow) and the 32-column chunks
        // 2 i + chalf, i = 0..3
        const int q = warp & 3;                 // the TMEM lane quarter this warp may access
        const int chalf = (warp - 4) >> 2;      // warpgroup 1: even chunks; warpgroup 2: odd chunks
        const int mrow = 32 * q + lane;
        float acc[4][32];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int k = 0; k < 32; ++k) acc[i][k] = 0.0f;
        auto promote = [&](int g) -> bool {
            const int b = g & 1;
            if (!mbar_wait(&pfull[b], (uint32_t)(g / 2) & 1u, abort_flag)) return false;
            tc_fence_after();
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + 256u * (uint32_t)b;
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
                const int c0 = 32 * (2 * i + chalf), c1 = 32 * (2 * i + 2 + chalf);
                if (c0 < N) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(base + (uint32_t)c0, v0);
                    if (c1 < N) tmem_ld_32x32b_x32(base + (uint32_t)c1, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) acc[i][k] += __uint_as_float(v0[k]);
                    if (c1 < N) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) acc[i + 1][k] += __uint_as_float(v1[k]);
                    }
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
            // read this thread's raw values, then give the ring slot back
            uint32_t wcode[2];
            uint16_t wscale[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int item = ct + 256 * i, row = item >> 2, qu = item & 3;
                wcode[i] = *reinterpret_cast<const uint32_t*>(slot + row * 16 + qu * 4);
                wscale[i] = *reinterpret_cast<const uint16_t*>(slot + o_as + row * 4 + (qu >> 1) * 2);
            }
            uint4 bcode[4];
            uint16_t bscale[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int item = ct + 256 * i, row = item >> 2, qu = item & 3;
                if (i < nb && row < rows) {
                    const uint8_t* piece = slot + o_b + (row >> 2) * kGroupStride + (row & 3) * kRowPiece;
                    bcode[i] = *reinterpret_cast<const uint4*>(piece + qu * 16);
                    bscale[i] = *reinterpret_cast<const uint16_t*>(piece + 64 + (qu >> 1) * 2);
                } else {
                    bcode[i] = make_uint4(0u, 0u, 0u, 0u);
                    bscale[i] = 0;
                }
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
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int item = ct + 256 * i, row = item >> 2, qu = item & 3;
                decode_weights16(wcode[i], wscale[i], a_tile + row * 8, row, qu);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int item = ct + 256 * i, row = item >> 2, qu = item & 3;
                if (i < nb) {
                    if (row < rows) split_activations16(bcode[i], bscale[i], hi_tile + row * 8, lo_tile + row * 8, row, qu);
                    else zero_activations16(hi_tile + row * 8, lo_tile + row * 8, row, qu);
                }
            }
            fence_async_smem();
            mbar_arrive(&full[s]);
            // after the first slice of partial g has been handed over, add partial g - 1
            if (kt % P == 0 && kt >= P && !promote(kt / P - 1)) ok = false;
        }
        if (ok && !promote((nk - 1) / P)) ok = false;
        if (ok) {
            // ------------------------------------------------------------------ epilogue: fp32 rows out
            float* outcol = p.out + (m0 + mrow);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int col = 32 * (2 * i + chalf) + k;
                    if (col < rows) outcol[(int64_t)(row0 + col) * p.a_rows] = acc[i][k];
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
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

// 2D uint8 tensor [rows][row_bytes] (row stride row_bytes), box box_x bytes x box_y rows, no swizzle
bool make_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_x, uint32_t box_y) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_x, box_y};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    GemmMaps maps;
    if (!make_map(&maps.b, a.bsl, (uint64_t)(a.K / kBK) * kRowPiece, (uint64_t)a.b_rows, kRowPiece, 1))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(a.a_rows / kBM), (unsigned)max_tiles);
    experts_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace smoe
