// elementwise.cu -- the HBM-bound steps of the routed-expert block: q8 quantisation of the activations (step 3),
// SwiGLU + requantisation of the gate/up rows (step 5) and the weighted combine (step 7).
//
// Page "Strata compare v0.1.35...v0.1.37", include/strata/prefill/moe_fused.hpp: the layer input is rounded to int8
// once per token with one scale per 32 values (quantize_act); gate/up is followed by SwiGLU and the int8 rounding of
// H; down writes one row per routed pair that the combine reads.  Page "src/prefill/prefill.cpp": mmq::swiglu, and
// the engine's fused weighted reduction of the K rows of each token.
//
// The q8 rule (the library's activation format): for 32 fp32 values, amax = max |x|, d = fp16_rne(amax / 127) with
// an IEEE fp32 division, and q = clamp(roundf(x / float(d)), -127, 127), again an IEEE fp32 division, roundf
// rounding half away from zero; d == 0 gives zero codes.  Four threads share a block, eight values each.
//
// The expert products read q8 rows in OPERAND FORM: the value d * q of every code split exactly into two fp16
// planes [2][rows][cols], hi = fp16_rn(d * q) and lo = d * q - hi (d * q has at most 18 significant bits, so the
// remainder is exact in fp16); within every group of 16 values position 2j holds value j and position 2j+1 value
// j+8 (j = 0..7) -- the K order in which the products unpack 2-bit weights in pairs.  SwiGLU writes it for H beside
// the planar codes; the routed-row gather writes it for the activations of every routed pair.
#include <climits>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "smoe_device.cuh"
#include "smoe_internal.h"

namespace smoe {
namespace {

// codes a[k] (bytes of a) and b[k] (bytes of b), k = 0..3, as the four fp16 pairs (a[k], b[k]): for a signed byte
// q, (q ^ 0x80) = q + 128, so the half with low byte (q ^ 0x80) and high byte 0x64 reads 1024 + 128 + q
__device__ __forceinline__ uint4 interleave_codes8(uint32_t a, uint32_t b) {
    const __half2 k1152 = __float2half2_rn(1152.0f);
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t t = __byte_perm(a, b, k | ((4 + k) << 8));
        const uint32_t v = (t & 0x00FF00FFu) ^ 0x64806480u;
        const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&v), k1152);
        h[k] = *reinterpret_cast<const uint32_t*>(&q);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

// fp16 code pairs q (exact integers) scaled by d and split: hi = fp16_rn(q d), lo = q d - hi (exact)
__device__ __forceinline__ void split_pairs(uint4 qp, __half2 d2, uint4& hi, uint4& lo) {
    const uint32_t w[4] = {qp.x, qp.y, qp.z, qp.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __half2 q = *reinterpret_cast<const __half2*>(&w[k]);
        const __half2 ph = __hmul2(q, d2);
        const __half2 pl = __hfma2(q, d2, __hneg2(ph));
        h[k] = *reinterpret_cast<const uint32_t*>(&ph);
        l[k] = *reinterpret_cast<const uint32_t*>(&pl);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// q8 of the NV values v held by this thread (NV = 8 or 16), its 32-value block being spread over 32 / NV consecutive
// lanes; writes the NV codes packed little-endian into `out` and returns the block's fp16 scale bits.
//
// Each code is round-half-away(x / d) of the IEEE (correctly rounded) fp32 quotient, clamped to [-127, 127], taken
// from a multiply by the correctly rounded reciprocal inv = RN(1/d): g = RN(x * inv) is within |x/d| 2^-23 of x/d and
// RN(x/d) within |x/d| 2^-24, so both round to the same integer unless a half-integer lies within |x/d| 2^-22 of g.
// Here |x/d| < 192 (d = fp16_rn(amax/127) is at least amax/127 (1 - 2^-11) when normal, and at least 2/3 of it when
// subnormal), so that margin is below 2^-14: only values whose g lies within 2^-14 of a half-integer (exact .5 ties
// included) take the IEEE division itself.  Elsewhere g rounds to the same integer under any tie rule, so it is
// rounded by adding and subtracting 1.5 * 2^23 (round to nearest even, exact for |g| < 2^22), and the clamped
// integer's low byte is read off the bits of (r + 1.5 * 2^23).  A zero scale gives zero codes.
template <int NV>
__device__ __forceinline__ uint16_t q8_encode(const float (&v)[NV], uint32_t (&out)[NV / 4]) {
    static_assert(NV == 8 || NV == 16, "a block spread over 4 or 2 lanes");
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int off = 1; off < 32 / NV; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const __half dh = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float d = __half2float(dh);
    if (d == 0.0f) {
#pragma unroll
        for (int w = 0; w < NV / 4; ++w) out[w] = 0u;
        return __half_as_ushort(dh);
    }
    const float inv = __frcp_rn(d);
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    uint32_t b[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const float g = v[i] * inv;
        float r = (g + kRound) - kRound;
        if (fabsf(g - r) >= 0.5f - 6.103515625e-05f) r = roundf(__fdiv_rn(v[i], d));  // within 2^-14 of a tie
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        b[i] = __float_as_uint(r + kRound);  // low byte: r mod 256
    }
#pragma unroll
    for (int w = 0; w < NV / 4; ++w)
        out[w] = __byte_perm(__byte_perm(b[4 * w], b[4 * w + 1], 0x0040),
                             __byte_perm(b[4 * w + 2], b[4 * w + 3], 0x0040), 0x5410);
    return __half_as_ushort(dh);
}

// step 3: x [rows][cols] -> codes, scales.  Thread i covers elements [16i, 16i + 16) of the flattened rows (four
// 16-byte loads, all issued before the encode; a 32-value block over two lanes).
__global__ void __launch_bounds__(256) quantize_q8_kernel(const float4* __restrict__ x, int64_t n16,
                                                          uint4* __restrict__ codes, uint16_t* __restrict__ scales) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // n16 is even (cols % 32 == 0), so both lanes of a block are in range or both out; lanes past the end still take
    // part in the shuffle
    const bool in = i < n16;
    float v[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in) a = __ldcs(x + 4 * i + u);
        v[4 * u] = a.x;
        v[4 * u + 1] = a.y;
        v[4 * u + 2] = a.z;
        v[4 * u + 3] = a.w;
    }
    uint32_t q[4];
    const uint16_t sb = q8_encode<16>(v, q);
    if (in) {
        codes[i] = make_uint4(q[0], q[1], q[2], q[3]);
        if ((i & 1) == 0) scales[i >> 1] = sb;
    }
}

// step 5: per routed row, h_j = silu(g_j) * u_j with g = gu[r][j], u = gu[r][F + j], then the q8 rule per 32 of h.
// thread i covers h values [8c, 8c + 8) of row r = i / (F/8), c = i % (F/8); lanes 2l and 2l+1 hold the two halves of
// one group of 16 (one scale), so after one exchange each writes 8 operand-form values of both planes at its own
// planar offset.
__global__ void __launch_bounds__(256) swiglu_requant_kernel(const float* __restrict__ gu, int64_t n, int F,
                                                             uint2* __restrict__ hc, uint16_t* __restrict__ hs,
                                                             uint4* __restrict__ hop, int64_t plane) {
    const int64_t per_row = F / 8;
    const int64_t total = n * per_row;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = base + threadIdx.x;
        const bool in = i < total;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (in) {
            const int64_t r = i / per_row, c = i - r * per_row;
            const float4* g4 = reinterpret_cast<const float4*>(gu + r * 2 * F + 8 * c);
            const float4* u4 = reinterpret_cast<const float4*>(gu + r * 2 * F + F + 8 * c);
            const float4 g0 = __ldcs(g4), g1 = __ldcs(g4 + 1), u0 = __ldcs(u4), u1 = __ldcs(u4 + 1);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __fdiv_rn(g[k], 1.0f + expf(-g[k])) * u[k];
        }
        uint32_t qw[2];
        const uint16_t sb = q8_encode<8>(v, qw);
        const uint2 q = make_uint2(qw[0], qw[1]);
        // the even lane holds values 0..7 of its group of 16, the odd lane 8..15; F % 16 == 0 keeps the pairs aligned
        const bool even = (threadIdx.x & 1) == 0;
        const uint32_t other = __shfl_xor_sync(0xffffffffu, even ? q.y : q.x, 1);
        if (in) {
            hc[i] = q;  // row r's codes start at r * F = 8 * (r * per_row): element offset 8i
            if ((i & 3) == 0) hs[i >> 2] = sb;
            // even lane: positions 0..7 = (v0, v8, v1, v9, ...); odd lane: positions 8..15 = (v4, v12, v5, v13, ...)
            if (hop) {
                const uint4 qp = even ? interleave_codes8(q.x, other) : interleave_codes8(other, q.y);
                uint4 hi, lo;
                split_pairs(qp, __half2half2(__ushort_as_half(sb)), hi, lo);
                hop[i] = hi;
                hop[plane + i] = lo;
            }
        }
    }
}

// step 7: Y[t][o] = sum_k w[t][k] * dm[slot[t*K+k]][o], in k order, fp32, then (with a shared expert) + sg[t] *
// ds[t][o].  Block (t, y): 128 threads, a float4 each.  A slot outside [0, n) (a pair dropped for an out-of-range id)
// contributes nothing.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ dm, const int32_t* __restrict__ slot,
                                                      const float* __restrict__ w, int K, int H, int64_t n,
                                                      const float* __restrict__ ds, const float* __restrict__ sg,
                                                      float* __restrict__ y) {
    const int64_t t = blockIdx.x;
    const int o4 = blockIdx.y * blockDim.x + threadIdx.x;
    if (4 * o4 >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
        const int32_t r = __ldg(slot + t * K + k);
        const float wk = __ldg(w + t * K + k);
        if (r < 0 || r >= n) continue;
        const float4 d = __ldcs(reinterpret_cast<const float4*>(dm + (int64_t)r * H) + o4);
        acc.x = fmaf(wk, d.x, acc.x);
        acc.y = fmaf(wk, d.y, acc.y);
        acc.z = fmaf(wk, d.z, acc.z);
        acc.w = fmaf(wk, d.w, acc.w);
    }
    if (ds != nullptr) {
        const float g = __ldg(sg + t);
        const float4 d = __ldcs(reinterpret_cast<const float4*>(ds + t * H) + o4);
        acc.x = fmaf(g, d.x, acc.x);
        acc.y = fmaf(g, d.y, acc.y);
        acc.z = fmaf(g, d.z, acc.z);
        acc.w = fmaf(g, d.w, acc.w);
    }
    reinterpret_cast<float4*>(y + t * H)[o4] = acc;
}

// Step 7 from fp16 down rows (the narrow form of Dm): Y[t][o] = sum_k w[t][k] * float(dm[slot[t*K+k]][o]), fp32 fmaf
// in k order.  Block (t, y): 64 threads, 8 outputs each (one 16-byte load of 8 fp16 values a row); the rows of four
// k at a time are loaded before they are added, so that each thread keeps four loads in flight.
constexpr int kCombineHThreads = 64;
__global__ void __launch_bounds__(kCombineHThreads) combine_h_kernel(const uint4* __restrict__ dm,
                                                                     const int32_t* __restrict__ slot,
                                                                     const float* __restrict__ w, int K, int H,
                                                                     int64_t n, float* __restrict__ y) {
    const int64_t t = blockIdx.x;
    const int o8 = blockIdx.y * blockDim.x + threadIdx.x;
    if (8 * o8 >= H) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < K; k0 += 4) {
        uint4 d[4];
        float wk[4];
        bool ok[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = k0 + j;
            const int32_t r = k < K ? __ldg(slot + t * K + k) : -1;
            ok[j] = r >= 0 && r < n;  // a pair dropped for an out-of-range id (or past K) contributes nothing
            wk[j] = ok[j] ? __ldg(w + t * K + k) : 0.0f;
            d[j] = ok[j] ? __ldcs(dm + (int64_t)r * (H / 8) + o8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (!ok[j]) continue;
            const uint32_t v[4] = {d[j].x, d[j].y, d[j].z, d[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v[i]));
                acc[2 * i] = fmaf(wk[j], f.x, acc[2 * i]);
                acc[2 * i + 1] = fmaf(wk[j], f.y, acc[2 * i + 1]);
            }
        }
    }
    float4* yo = reinterpret_cast<float4*>(y + t * H) + 2 * o8;
    yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// The shared expert's scalar gate (page "src/prefill/prefill.cpp", Prefill::run, MoE half: "the shared expert and
// its scalar gate", a projection of the token onto one row): sg[t] = 1 / (1 + exp(-(x[t] . w_sg))), the dot product
// in fp32 (lane l sums the float4s l, l + 32, ... of the row, then a butterfly).  One warp per token.
__global__ void __launch_bounds__(256) shared_gate_kernel(const float4* __restrict__ x, const float4* __restrict__ wsg,
                                                          int64_t T, int H4, float* __restrict__ sg) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // the whole warp
    const float4* xt = x + t * H4;
    float acc = 0.0f;
    for (int i = lane; i < H4; i += 32) {
        const float4 a = __ldcs(xt + i), b = __ldg(wsg + i);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
        acc = fmaf(a.z, b.z, acc);
        acc = fmaf(a.w, b.w, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) sg[t] = __fdiv_rn(1.0f, 1.0f + expf(-acc));
}

// Q2 weights, row-major [E][rows][cols/4] codes + [E][rows][cols/32] scales, to the expert products' packed form:
// per (expert, 128-row tile, 64-value slice) one 2560-byte block = the tile's 128 x 16 code bytes, then its 128 x 2
// scales.  One thread per 16-byte piece of a block (128 code pieces, 32 scale pieces).
// `half` > 0 packs a gate/up matrix for the fused SwiGLU product: tile mt holds outputs j in [64 mt, 64 mt + 64),
// and its row 32 q + l is gate row 64 mt + 16 q + l (l < 16) or up row half + 64 mt + 16 q + l - 16 (l >= 16), so
// that each 32-row warp of the product holds the gate and up rows of the same 16 outputs.
// the source row of packed row r of 128-row tile mt, within one expert's matrix
__device__ __forceinline__ int packed_source_row(int mt, int r, int half) {
    if (half <= 0) return mt * 128 + r;
    const int q = r >> 5, l = r & 31;
    const int j = 64 * mt + 16 * q + (l & 15);
    return l < 16 ? j : half + j;
}

// desc == nullptr: the E experts contiguous in codes / scales; else expert e's matrix at desc[e] (a block whose
// descriptor is null or not 16-byte aligned is written as zeros and reported in status[0] as SMOE_ERR_ARG)
__global__ void __launch_bounds__(160) pack_q2_kernel(const uint8_t* __restrict__ codes,
                                                      const uint16_t* __restrict__ scales,
                                                      const smoe_q2w* __restrict__ desc, int rows, int cols,
                                                      int half, uint8_t* __restrict__ packed, int32_t* status) {
    const int64_t blk = blockIdx.x;  // ((e * rows/128 + mt) * cols/64 + kt)
    const int nkt = cols / 64, nmt = rows / 128;
    const int kt = (int)(blk % nkt);
    const int64_t emt = blk / nkt;  // e * nmt + mt
    const int64_t e = emt / nmt;
    const int mt = (int)(emt - e * nmt);
    const uint8_t* ce = codes + e * rows * (int64_t)(cols / 4);
    const uint16_t* se = scales + e * rows * (int64_t)(cols / 32);
    if (desc != nullptr) {
        ce = desc[e].codes;
        se = desc[e].scales;
    }
    uint8_t* out = packed + blk * 2560;
    const int t = threadIdx.x;
    if (ce == nullptr || se == nullptr || (((uintptr_t)ce | (uintptr_t)se) & 15u) != 0) {
        if (t < 160) *reinterpret_cast<uint4*>(out + t * 16) = make_uint4(0u, 0u, 0u, 0u);
        if (t == 0 && status != nullptr) status[0] = SMOE_ERR_ARG;
        return;
    }
    if (t < 128) {
        const int64_t sr = packed_source_row(mt, t, half);
        const uint4 v = *reinterpret_cast<const uint4*>(ce + sr * (cols / 4) + kt * 16);
        *reinterpret_cast<uint4*>(out + t * 16) = v;
    } else {
        const int r = (t - 128) * 4;  // four rows' scale pairs per piece
        uint32_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t sr = packed_source_row(mt, r + j, half);
            v[j] = *reinterpret_cast<const uint32_t*>(se + sr * (cols / 32) + kt * 2);
        }
        *reinterpret_cast<uint4*>(out + 2048 + r * 4) = make_uint4(v[0], v[1], v[2], v[3]);
    }
}

// Routed rows of the q8 activations in operand form: out row r = codes row src[r] (row r itself when src is null)
// scaled by its scales and split into the hi and lo planes, in operand order.  One warp per output row.  Lane l makes the output words (8 fp16
// each) l, l + 32, ... of both planes, so every store instruction writes 512 contiguous bytes: word w is half w % 2
// of group w / 2, i.e. values 4h..4h+3 and 8+4h..8+4h+3 of the group (h = w % 2).  An src entry outside
// [0, in_rows) gives zero rows.
__global__ void __launch_bounds__(256) gather_q8_kernel(const uint32_t* __restrict__ codes,
                                                        const uint16_t* __restrict__ scales, int64_t in_rows,
                                                        int groups, const int32_t* __restrict__ src, int64_t n,
                                                        uint4* __restrict__ out) {
    constexpr int kAhead = 16;  // words a lane loads before it converts and stores them (cols up to 4096 a pass)
    const int lane = threadIdx.x & 31;
    const int words = 2 * groups;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t plane = n * words;  // uint4 words per plane
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n; r += warps) {
        const int64_t t = src != nullptr ? (int64_t)__ldg(src + r) : r;  // no src: row r itself
        uint4* o = out + r * words;
        if (t < 0 || t >= in_rows) {
            for (int w = lane; w < words; w += 32) {
                __stcs(o + w, make_uint4(0u, 0u, 0u, 0u));
                __stcs(o + plane + w, make_uint4(0u, 0u, 0u, 0u));
            }
            continue;
        }
        const uint32_t* i = codes + (int64_t)t * groups * 4;  // 4 code words (16 codes) a group
        const uint16_t* sc = scales + (int64_t)t * (groups / 2);
        for (int w0 = lane; w0 < words; w0 += 32 * kAhead) {
            // every load of this pass first (independent, in flight together), then the conversions and stores
            uint32_t a[kAhead], b[kAhead];
            uint16_t d[kAhead];
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                const int w = w0 + 32 * k;
                if (w < words) {
                    const int g = w >> 1, h = w & 1;
                    a[k] = __ldg(i + 4 * g + h);      // values 4h .. 4h+3 of the group
                    b[k] = __ldg(i + 4 * g + 2 + h);  // values 8+4h .. 8+4h+3
                    d[k] = __ldg(sc + g / 2);
                }
            }
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                const int w = w0 + 32 * k;
                if (w < words) {
                    uint4 hi, lo;
                    split_pairs(interleave_codes8(a[k], b[k]), __half2half2(__ushort_as_half(d[k])), hi, lo);
                    // streaming stores: the rows are read once, by the gate/up product
                    __stcs(o + w, hi);
                    __stcs(o + plane + w, lo);
                }
            }
        }
    }
}

int grid_for(int64_t threads, int block) {
    const int64_t blocks = (threads + block - 1) / block;
    const int64_t cap = 152 * 16;  // a few waves of resident blocks; the kernels stride beyond this
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_quantize_q8(const float* x, int64_t rows, int cols, int8_t* codes, uint16_t* scales,
                               cudaStream_t s) {
    const int64_t n16 = rows * (int64_t)cols / 16;
    if (n16 == 0) return cudaSuccess;
    // one 16-value item a thread and no grid-stride loop: the blocks stream through the SMs as earlier ones retire,
    // which keeps more loads in flight than a resident grid looping over the rows
    const int64_t blocks = (n16 + 255) / 256;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    quantize_q8_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(x), n16,
                                                        reinterpret_cast<uint4*>(codes), scales);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_requant(const float* gu, int64_t n, int F, int8_t* hc, uint16_t* hs, uint16_t* hop,
                                  cudaStream_t s) {
    const int64_t total = n * (int64_t)(F / 8);
    if (total == 0) return cudaSuccess;
    swiglu_requant_kernel<<<grid_for(total, 256), 256, 0, s>>>(gu, n, F, reinterpret_cast<uint2*>(hc), hs,
                                                               reinterpret_cast<uint4*>(hop), total);
    return cudaGetLastError();
}

cudaError_t launch_pack_q2(const uint8_t* codes, const uint16_t* scales, const smoe_q2w* desc, int E, int rows,
                           int cols, int half, uint8_t* packed, int32_t* status, cudaStream_t s) {
    const int64_t blocks = (int64_t)E * (rows / 128) * (cols / 64);
    if (blocks == 0) return cudaSuccess;
    pack_q2_kernel<<<(unsigned)blocks, 160, 0, s>>>(codes, scales, desc, rows, cols, half, packed, status);
    return cudaGetLastError();
}

cudaError_t launch_gather_q8(const int8_t* codes, const uint16_t* scales, int64_t in_rows, int cols,
                             const int32_t* src, int64_t n, uint16_t* out, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    gather_q8_kernel<<<grid_for(n * 32, 256), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(codes), scales, in_rows,
                                                           cols / 16, src, n, reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* dm, const int32_t* slot, const float* w, int64_t T, int K, int H,
                           const float* ds, const float* sg, float* y, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)T, (unsigned)((H / 4 + 127) / 128));
    combine_kernel<<<grid, 128, 0, s>>>(dm, slot, w, K, H, T * (int64_t)K, ds, sg, y);
    return cudaGetLastError();
}

cudaError_t launch_combine_h(const uint16_t* dm, const int32_t* slot, const float* w, int64_t T, int K, int H,
                             float* y, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)T, (unsigned)((H / 8 + kCombineHThreads - 1) / kCombineHThreads));
    combine_h_kernel<<<grid, kCombineHThreads, 0, s>>>(reinterpret_cast<const uint4*>(dm), slot, w, K, H,
                                                       T * (int64_t)K, y);
    return cudaGetLastError();
}

cudaError_t launch_shared_gate(const float* x, const float* wsg, int64_t T, int H, float* sg, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int warps = 8;
    shared_gate_kernel<<<(unsigned)((T + warps - 1) / warps), 32 * warps, 0, s>>>(
        reinterpret_cast<const float4*>(x), reinterpret_cast<const float4*>(wsg), T, H / 4, sg);
    return cudaGetLastError();
}

}  // namespace smoe
