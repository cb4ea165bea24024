// experts_gemm.cu -- the grouped expert products of the routed-expert block (steps 4 and 6) on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), sm_103a.
//
// Page "Strata compare v0.1.35...v0.1.37", include/strata/prefill/moe_fused.hpp experts(): for each expert, gate/up
// of its routed rows from the per-token int8 activations against its 2-bit weights, then down into one fp32 row per
// routed pair.  Per output:  sum_b dW[b] * dA[b] * sum_{i in b} (qW - 2) * qA.
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
// two-level where it matters: for gate/up, whose output is requantised, each 64-wide K slice accumulates from zero
// into one of two tensor-memory buffers (the partial is small, so its truncation error is too) and the promoter
// warps add each finished partial into fp32 registers with round-to-nearest while the tensor core fills the other
// buffer (one slice per partial: two flipped one H scale of the smallest test chunk).  The down product feeds the
// fp32 combine only, where 4e-6 is far inside the output bound, so it accumulates the whole K in one buffer.
//
// Tile: one CTA = one tile of the tile list (an expert and up to 256 of its routed rows, contiguous in routed-row
// order; the MMA's N, a multiple of 16) x one 128-row slice of the expert's weight matrix (the MMA's M; swap-AB:
// weights are the M operand so that a small expert wastes little).  Five warpgroups, registers rebalanced with
// setmaxnreg:
//   warpgroup 0   warp 0: tensor-memory allocation and, on one lane, the MMAs of each slice;
//                 warp 1, one lane: the producer -- per 64-wide K slice one bulk copy of the packed weight block
//                 (codes and scales) and TMA tile loads of the tile's q8 rows in slice form (codes and scales, 80
//                 bytes a row, 16 rows a load), into a ring of up to 16 slices in shared memory;
//   warpgroups 1-2  promoters: add each finished partial from tensor memory into fp32 registers (128 columns of
//                 one TMEM lane a thread), then write the fp32 rows;
//   warpgroups 3-4  converters: decode a ring slice into the fp16 operand tiles of one of two stages (K-major,
//                 128-byte swizzle), 16 K values of one row per work item.
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
constexpr int kThreads = 640;                  // five warpgroups
constexpr int kPromoters = 256;                // warpgroups 1-2
constexpr int kConverters = 256;               // warpgroups 3-4
constexpr int kATile = kBM * 128;              // 16 KB of fp16 weights
constexpr int kBTile = kMaxBN * 128;           // 32 KB of fp16 activations (one of hi / lo)
constexpr int kStage = kATile + 2 * kBTile;
constexpr int kRingBytes = 65 * 1024;          // raw-data ring
constexpr int kMaxRing = 16;                   // slices in flight at most
constexpr uint32_t kTmemCols = 512;            // two fp32 partial buffers, 128 lanes x N <= 256 columns each
// shared memory: [1 KB alignment slack][stages][ring][barriers]
constexpr int kSmemBytes = 1024 + kStages * kStage + kRingBytes + 512;
// registers: launched at 96 a thread (640 x 96 = 61,440 of 65,536); warpgroup 0 gives back to 24, the converters to
// 40 and the promoters take 176: 128 x 24 + 256 x 40 + 256 x 176 = 58,368 <= 61,440.  Per SM sub-partition (one
// warp of each warpgroup): 32 x (24 + 176 + 176 + 40 + 40) = 14,592 <= 16,384.
constexpr int kRegsWg0 = 24;
constexpr int kRegsConv = 40;
constexpr int kRegsProm = 176;
static_assert(128 * kRegsWg0 + 256 * kRegsConv + 256 * kRegsProm <= 640 * 96, "register split exceeds the launch");

// Raw slice layout in the ring (one 64-wide K slice of the tile): the packed weight block (codes [128][16 B], scales
// [128][4 B]), then the tile's N rows in slice form (80 B a row: 64 codes, 2 scales, padding).  Every TMA
// destination (the block, each 16-row box) is 128-byte aligned.
constexpr int kWBlock = 2560;
constexpr int kRowPiece = 80;
constexpr int kRowBox = 16;                    // rows per TMA box
__host__ __device__ constexpr int raw_slice_bytes(int N) { return kWBlock + N * kRowPiece; }

// bulk copy (no tensor map) of `bytes` (a multiple of 16) into shared memory, completing on `bar`
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// TMA: a 2D tile (x bytes along the row, y the first row) into shared memory, completing its bytes on `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
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
    CUtensorMap b;  // q8 rows in slice form: [rows][K/64 * 80 bytes], box 80 bytes x 16 rows
};

__global__ void __launch_bounds__(kThreads, 1) experts_gemm_kernel(const ExpertsGemmArgs p,
                                                                   const __grid_constant__ GemmMaps maps) {
    int32_t* tiles = p.tiles;
    const int ti = blockIdx.y;
    if (ti >= tiles[0] || tiles[1] != 0) return;  // no such tile, or the grouping failed: nothing to do
    const int4 tile = reinterpret_cast<const int4*>(tiles)[1 + ti];
    const int e = tile.x, row0 = tile.y, rows = tile.z;
    // a tile the grouping cannot have written (a bad expert id or row range): nothing is read or written for it
    if (rows <= 0 || rows > kMaxBN || e < 0 || e >= p.n_experts || row0 < 0 || row0 + (int64_t)rows > p.b_rows) return;
    const int N = (rows + 15) & ~15;
    const int m0 = blockIdx.x * kBM;
    const int nk = p.K / kBK;
    const int P = p.two_level ? 1 : nk;  // slices per tensor-memory partial

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    uint8_t* ring = smem + kStages * kStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kRingBytes);  // operand stage s is filled
    uint64_t* empty = full + kStages;      // ... and consumed by the MMAs
    uint64_t* pfull = empty + kStages;     // a partial is complete in tensor-memory buffer b
    uint64_t* pempty = pfull + 2;          // the promoters have added buffer b into their registers
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
            mbar_init(&pempty[b], kPromoters);
        }
        for (int r = 0; r < kMaxRing; ++r) {
            mbar_init(&rfull[r], 1);  // the arrival that posts the slice's byte count
            mbar_init(&rempty[r], kConverters);
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
    const uint32_t sbase = smem_u32(smem);
    bool ok = true;

    if (warp < 4) {
        setmaxnreg_dec<kRegsWg0>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------------ MMA issue (one thread)
            const uint32_t idesc = idesc_f16_f32(kBM, N);
            for (int kt = 0; kt < nk; ++kt) {
                // slice kt of partial g = kt / P goes to buffer g & 1, which partial g - 2 has left
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
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------------ producer (one thread)
            const uint8_t* wblocks = p.wp + ((int64_t)e * (p.a_rows / kBM) + blockIdx.x) * nk * (int64_t)kWBlock;
            const uint32_t tx_bytes = (uint32_t)kWBlock + (uint32_t)N * kRowPiece;
            int issued = 0;
            for (int kt = 0; kt < nk; ++kt, ++issued) {
                const int r = kt % depth;
                if (kt >= depth && !mbar_wait(&rempty[r], (uint32_t)(kt / depth - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t slot = smem_u32(ring) + (uint32_t)(r * sbytes);
                mbar_arrive_expect_tx(&rfull[r], tx_bytes);
                bulk_load(slot, wblocks + (int64_t)kt * kWBlock, kWBlock, &rfull[r]);
                for (int b0 = 0; b0 < N; b0 += kRowBox)
                    tma_load_2d(slot + o_b + b0 * kRowPiece, &maps.b, kt * kRowPiece, row0 + b0, &rfull[r]);
            }
            // no copy may still be writing shared memory when the CTA exits (on the abort path the converters have
            // not waited for the last slices): wait, bounded, for the last `depth` slices issued
            for (int kt = max(0, issued - depth); kt < issued; ++kt)
                mbar_wait(&rfull[kt % depth], (uint32_t)(kt / depth) & 1u, nullptr);
        }
        __syncwarp();
    } else if (warp < 12) {
        setmaxnreg_inc<kRegsProm>();
        // ------------------------------------------------------------------ promoters (256 threads)
        // this thread owns TMEM lane 32*q + lane (weight row mrow) and the 32-column chunks 2 i + chalf, i = 0..3
        const int q = warp & 3;
        const int chalf = (warp - 4) >> 2;  // warpgroup 1: even chunks; warpgroup 2: odd chunks
        const int mrow = 32 * q + lane;
        float acc[4][32];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int k = 0; k < 32; ++k) acc[i][k] = 0.0f;
        const int groups = (nk + P - 1) / P;
        for (int g = 0; g < groups && ok; ++g) {
            const int b = g & 1;
            if (!mbar_wait(&pfull[b], (uint32_t)(g / 2) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + 256u * (uint32_t)b;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c0 = 32 * (2 * i + chalf);
                if (c0 < N) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(base + (uint32_t)c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) acc[i][k] += __uint_as_float(v[k]);
                }
            }
            tc_fence_before();
            mbar_arrive(&pempty[b]);
        }
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
    } else {
        setmaxnreg_dec<kRegsConv>();
        // ------------------------------------------------------------------ converters (256 threads)
        // work items of 16 K values: weight items ct and ct + 256 (row = item / 4, quarter = item % 4); row items
        // ct + 256 i of the tile's 4 N (row, quarter) pairs
        const int ct = threadIdx.x - 384;
        const int nb = (4 * N - ct + 255) / 256;  // row items of this thread (0..4)
        for (int kt = 0; kt < nk && ok; ++kt) {
            const int r = kt % depth, s = kt % kStages;
            if (!mbar_wait(&rfull[r], (uint32_t)(kt / depth) & 1u, abort_flag) ||
                (kt >= kStages && !mbar_wait(&empty[s], (uint32_t)(kt / kStages - 1) & 1u, abort_flag))) {
                ok = false;
                break;
            }
            const uint8_t* slot = ring + r * sbytes;
            uint8_t* st = smem + s * kStage;
            uint4* a_tile = reinterpret_cast<uint4*>(st);
            uint4* hi_tile = reinterpret_cast<uint4*>(st + kATile);
            uint4* lo_tile = reinterpret_cast<uint4*>(st + kATile + kBTile);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int item = ct + 256 * i, row = item >> 2, qu = item & 3;
                const uint32_t code = *reinterpret_cast<const uint32_t*>(slot + row * 16 + qu * 4);
                const uint16_t scale = *reinterpret_cast<const uint16_t*>(slot + o_as + row * 4 + (qu >> 1) * 2);
                decode_weights16(code, scale, a_tile + row * 8, row, qu);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int item = ct + 256 * i, row = item >> 2, qu = item & 3;
                if (i < nb) {
                    if (row < rows) {
                        const uint8_t* piece = slot + o_b + row * kRowPiece;
                        const uint4 code = *reinterpret_cast<const uint4*>(piece + qu * 16);
                        const uint16_t scale = *reinterpret_cast<const uint16_t*>(piece + 64 + (qu >> 1) * 2);
                        split_activations16(code, scale, hi_tile + row * 8, lo_tile + row * 8, row, qu);
                    } else {
                        zero_activations16(hi_tile + row * 8, lo_tile + row * 8, row, qu);
                    }
                }
            }
            mbar_arrive(&rempty[r]);
            fence_async_smem();
            mbar_arrive(&full[s]);
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
    if (!make_map(&maps.b, a.bsl, (uint64_t)(a.K / kBK) * kRowPiece, (uint64_t)a.b_rows, kRowPiece, kRowBox))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(a.a_rows / kBM), (unsigned)max_tiles);
    experts_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace smoe
