// smoe_oracle.cpp -- the CPU oracle of the routed-expert block (TEST INFRASTRUCTURE ONLY).
//
// A plain, slow, obviously correct CPU implementation of what the prompt-chunk routed-expert block computes.  It is
// the checker that the CUDA library is compared against; it is not part of the product.  Only tests/, the package's
// smoke() and bench.py's cpu_baseline / reference legs load it.  It shares no code, header, table or constant
// generator with the CUDA library, and neither includes the other.
//
// Sources (web pages of the "Strata" inference engine; cited by page title and the function / header they belong to):
//   [P1] src/prefill/prefill.cpp, Prefill::run, the MoE half: the router call route(logits, ids, w, T, n_expert),
//        the fused int8 expert path (quantize_act -> group -> experts per batch), and the host grouping of the
//        (token, k) pairs by expert (the counting-sort loop: counts, exclusive offsets, slot[i] = row,
//        src[row] = i / k).
//   [P3] Strata compare v0.1.35...v0.1.37, include/strata/prefill/moe_fused.hpp: activations rounded to int8 once
//        per token with one scale per 32 values; grouping tables (counts, offsets, rows per expert, a tile list);
//        gate/up + SwiGLU + int8 H, then down into per-slot rows that the combine reads.
//   [P3] same page, include/strata/kernels/qsa_select.hpp: the engine's top-k rule "ties to the lowest index".
//
// Readings where the pages are silent or disagree:
//   R1 weight code offset: w = d * (q - 2) for a 2-bit code q in {0..3}, i.e. d * {-2, -1, 0, 1}: the weight format
//      of this library (the moe_fused.hpp header's "q - 1" is not followed).
//   R2 weight blob: planar per matrix, codes uint8 [rows][cols/4] with weight 4j+i in bits 2i..2i+1 of byte j,
//      scales fp16 [rows][cols/32]; all experts of one matrix contiguous, expert-major.  Gate rows [0, F), up rows
//      [F, 2F) of the gate/up matrix.
//   R3 q8 rule (format-defining, in fp32): amax = max |x| over the 32 values; d = fp16_rne(amax / 127.0f);
//      d == 0 -> all codes 0; else q = clamp(roundf(x / float(d)), -127, 127) with IEEE fp32 division and roundf
//      rounding half away from zero.
//   R4 top-k order: by logit descending, ties to the lower expert id; ids are emitted in that order.
//   R5 weights: softmax, top-K, renormalised over the K:  w_k = exp(l_k - l_1) / sum_{j in top-K} exp(l_j - l_1);
//      the full softmax denominator cancels.
//   R6 grouping: stable by pair index i = t*K + k (the host loop's order).  The pages' group() also emits a tile list
//      (64-row tiles) that only schedules their kernels; which rows share a tile changes no value of the block, so
//      the oracle defines no tile list (the library's own is checked by the invariants any valid tiling meets).
//   R7 SwiGLU: h_j = silu(g_j) * u_j, silu(g) = g / (1 + exp(-g)), gate = rows [0, F), up = rows [F, 2F); h is
//      rounded to fp32 before the q8 rule of R3 (the rule is defined on fp32 input).
//   R8 combine: Y[t] = sum over k (in k order) of w[t][k] * Dm[slot[t*K+k]].
//   R14 shared expert (the "shared expert and its scalar gate" of [P1]; its weight format, width and the gate's
//      nonlinearity are not given): one more expert of the routed experts' form (2-bit weights, gate/up [2F][H],
//      down [H][F]) that every token takes, on the same int8 activations; its scalar gate is
//      sg[t] = sigmoid(x[t] . w_sg) with w_sg fp32 [H]; the combine adds sg[t] * S[t] after the routed sum.
//   R15 router projection ([P1]: "bf16_proj" of the router weight on the hidden state's BF16 copy and its low part):
//      router weights bf16 [E][H]; xh = bf16_rne(x), xl = bf16_rne(x - xh) (x - xh exact in fp32);
//      logit[t][e] = sum_h w[e][h] * (xh + xl) in double, rounded to fp32, then step 1 (R4, R5).
//
// Arithmetic: double everywhere except the q8 rule (R3), which is defined in fp32 and emulated here in `float`.
// Build with -ffp-contract=off so that no fused multiply-add changes a fp32 step.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- IEEE binary16 conversions (own, from the format)
float h2f(uint16_t h) {
    const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    const uint32_t e = (h >> 10) & 0x1fu;
    const uint32_t m = h & 0x3ffu;
    float out;
    if (e == 0) {
        // zero or subnormal: m * 2^-24, exact in float
        out = (float)m * 5.9604644775390625e-08f;
        if (sign) out = -out;
        return out;
    }
    uint32_t bits;
    if (e == 31) bits = sign | 0x7f800000u | (m << 13);
    else bits = sign | ((e - 15 + 127) << 23) | (m << 13);
    std::memcpy(&out, &bits, 4);
    return out;
}

uint16_t f2h_rne(float f) {
    uint32_t x;
    std::memcpy(&x, &f, 4);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x200u : 0u));
    if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);  // >= 65520 rounds to infinity
    const int e = (int)(ax >> 23) - 127;
    if (e >= -14) {
        const uint32_t mant = ax & 0x7fffffu;
        uint32_t h = ((uint32_t)(e + 15) << 10) | (mant >> 13);
        const uint32_t rem = mant & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1;
        return (uint16_t)(sign | h);
    }
    if (e < -25) return (uint16_t)sign;
    const uint32_t mant = (ax & 0x7fffffu) | 0x800000u;  // value = mant * 2^(e-23)
    const int shift = -(e + 1);                           // to units of 2^-24
    uint32_t q = mant >> shift;
    const uint32_t rem = mant & ((1u << shift) - 1u);
    const uint32_t halfv = 1u << (shift - 1);
    if (rem > halfv || (rem == halfv && (q & 1u))) q += 1;
    return (uint16_t)(sign | q);
}

// ---------------------------------------------------------------- bfloat16 (own, from the format: the top 16 bits
// of binary32, rounded to nearest, ties to even)
uint16_t f2bf(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);  // NaN
    const uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    uint32_t r = keep;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) ++r;  // carries into the exponent as the format wants
    return (uint16_t)r;
}
float bf2f(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// ---------------------------------------------------------------- threads
template <class Fn>
void parallel_for(int64_t n, int nthreads, Fn fn) {
    if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
    if (n <= 0) return;
    if (nthreads > n) nthreads = (int)n;
    if (nthreads == 1) {
        fn((int64_t)0, n);
        return;
    }
    std::vector<std::thread> th;
    for (int i = 0; i < nthreads; ++i) {
        const int64_t a = n * i / nthreads, b = n * (i + 1) / nthreads;
        th.emplace_back([=] { fn(a, b); });
    }
    for (auto& t : th) t.join();
}

// ---------------------------------------------------------------- R3: the q8 rule on one block of 32 fp32 values
void q8_block(const float* x, int8_t* q, uint16_t* d_out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(x[i]));
    const float d32 = amax / 127.0f;
    const uint16_t d16 = f2h_rne(d32);
    *d_out = d16;
    const float d = h2f(d16);
    for (int i = 0; i < 32; ++i) {
        if (d == 0.0f) {
            q[i] = 0;
            continue;
        }
        float r = std::roundf(x[i] / d);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
}

// the 2-bit code of weight c of a row (R2)
inline int q2_code(const uint8_t* row_codes, int64_t c) { return (row_codes[c >> 2] >> (2 * (c & 3))) & 3; }

// one output of a block-quantised product (moe_fused.hpp: per-32 integer dot scaled by the two fp16 scales)
//   sum_b  d_w[b] * d_a[b] * sum_{i in b} (q_w - 2) * q_a
double q2_q8_dot(const uint8_t* wc, const uint16_t* ws, const int8_t* ac, const uint16_t* as, int64_t cols) {
    double acc = 0.0;
    for (int64_t b = 0; b < cols / 32; ++b) {
        int64_t idot = 0;
        for (int64_t i = b * 32; i < b * 32 + 32; ++i) idot += (int64_t)(q2_code(wc, i) - 2) * (int64_t)ac[i];
        acc += (double)h2f(ws[b]) * (double)h2f(as[b]) * (double)idot;
    }
    return acc;
}

double silu(double g) { return g / (1.0 + std::exp(-g)); }

}  // namespace

extern "C" {

// ------------------------------------------------------------------------------------------------ helpers exposed
uint16_t oracle_f2h(float f) { return f2h_rne(f); }
float oracle_h2f(uint16_t h) { return h2f(h); }


// ------------------------------------------------------------------------------------------------ step 1: route
/// [P1] Prefill::run, MoE half, route(logits, ids, w, T, n_expert): softmax over the E router logits of each token,
/// the top-K experts, and their weights renormalised over the K (R4, R5).
/// logits fp32 [T][E] -> ids int32 [T][K] (best first), w double [T][K].
void oracle_route(const float* logits, int64_t T, int E, int K, int32_t* ids, double* w, int nthreads) {
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        std::vector<int32_t> order((size_t)E);
        for (int64_t t = t0; t < t1; ++t) {
            const float* l = logits + t * E;
            for (int e = 0; e < E; ++e) order[(size_t)e] = e;
            std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
                if (l[a] != l[b]) return l[a] > l[b];
                return a < b;
            });
            const double lmax = (double)l[order[0]];
            double den = 0.0;
            for (int k = 0; k < K; ++k) den += std::exp((double)l[order[(size_t)k]] - lmax);
            for (int k = 0; k < K; ++k) {
                ids[t * K + k] = order[(size_t)k];
                w[t * K + k] = std::exp((double)l[order[(size_t)k]] - lmax) / den;
            }
        }
    });
}

/// [P1] the router's BF16 projection of the hidden state with its low part (R15): x fp32 [T][H] -> the two bf16
/// parts (bits) xh, xl [T][H].
void oracle_bf16_split(const float* x, int64_t n, uint16_t* xh, uint16_t* xl) {
    for (int64_t i = 0; i < n; ++i) {
        xh[i] = f2bf(x[i]);
        const float rest = x[i] - bf2f(xh[i]);  // exact in fp32
        xl[i] = f2bf(rest);
    }
}

/// logit[t][e] = sum_h wr[e][h] * (xh[t][h] + xl[t][h]) in double (R15); wr bf16 bits [E][H]; logits double [T][E].
void oracle_router_logits(const float* x, const uint16_t* wr, int64_t T, int H, int E, double* logits,
                          int nthreads) {
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        std::vector<uint16_t> xh((size_t)H), xl((size_t)H);
        std::vector<double> a((size_t)H);
        for (int64_t t = t0; t < t1; ++t) {
            oracle_bf16_split(x + t * H, H, xh.data(), xl.data());
            for (int h = 0; h < H; ++h) a[(size_t)h] = (double)bf2f(xh[(size_t)h]) + (double)bf2f(xl[(size_t)h]);
            for (int e = 0; e < E; ++e) {
                double s = 0.0;
                for (int h = 0; h < H; ++h) s += (double)bf2f(wr[(int64_t)e * H + h]) * a[(size_t)h];
                logits[t * E + e] = s;
            }
        }
    });
}

/// Step 1 from the hidden state (R15): the logits above rounded to fp32, then oracle_route.  logits_out (double
/// [T][E]) may be null.
void oracle_router_route(const float* x, const uint16_t* wr, int64_t T, int H, int E, int K, int32_t* ids, double* w,
                         double* logits_out, int nthreads) {
    std::vector<double> lg((size_t)(T * E));
    oracle_router_logits(x, wr, T, H, E, lg.data(), nthreads);
    std::vector<float> lf((size_t)(T * E));
    for (size_t i = 0; i < lf.size(); ++i) lf[i] = (float)lg[i];
    oracle_route(lf.data(), T, E, K, ids, w, nthreads);
    if (logits_out) std::memcpy(logits_out, lg.data(), lg.size() * sizeof(double));
}

// ------------------------------------------------------------------------------------------------ step 2: group
/// [P1] the host grouping loop of Prefill::run (count per expert, exclusive offsets, then in pair order
/// slot[i] = next row of expert ids[i], src[row] = i / K), as [P3] moe_fused.hpp group() builds the same tables (R6).
/// Returns 0, or -1 if an id is out of range (nothing else is then defined).
int oracle_group(const int32_t* ids, int64_t T, int K, int E, int32_t* counts, int32_t* offsets, int32_t* src,
                 int32_t* slot) {
    const int64_t n = T * K;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) return -1;
        ++counts[ids[i]];
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    std::vector<int32_t> fill(offsets, offsets + E);
    for (int64_t i = 0; i < n; ++i) {
        const int32_t row = fill[(size_t)ids[i]]++;
        slot[i] = row;
        src[row] = (int32_t)(i / K);
    }
    return 0;
}

// ------------------------------------------------------------------------------------------------ step 3: q8
/// [P3] moe_fused.hpp quantize_act: fp32 rows to int8 once per token with one scale per 32 values, by the rule R3.
/// x fp32 [rows][cols] -> codes int8 [rows][cols], scales fp16 bits [rows][cols/32].  cols % 32 == 0.
void oracle_quantize_q8(const float* x, int64_t rows, int64_t cols, int8_t* codes, uint16_t* scales, int nthreads) {
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t b = 0; b < cols / 32; ++b)
                q8_block(x + r * cols + b * 32, codes + r * cols + b * 32, scales + r * (cols / 32) + b);
    });
}

// ------------------------------------------------------------------------------------------------ step 4: gate/up
/// [P3] moe_fused.hpp experts(): gate/up of each routed row from the token's int8 activations (through src) and
/// the expert's 2-bit rows:  G[r][j] = sum_b d_w[e][j][b] * d_a[src r][b] * sum_{i in b} (q_w - 2) * q_a,
/// j in [0, 2F).  Expert e owns rows [offsets[e], offsets[e+1]).
/// xc int8 [T][H], xs fp16 [T][H/32]; wc uint8 [E][2F][H/4], ws fp16 [E][2F][H/32]; gu double [n][2F].
void oracle_gateup(const int8_t* xc, const uint16_t* xs, const int32_t* src, const int32_t* offsets, int E,
                   const uint8_t* wc, const uint16_t* ws, int H, int F, double* gu, int nthreads) {
    const int64_t n = offsets[E];
    std::vector<int32_t> expert_of((size_t)n);
    for (int e = 0; e < E; ++e)
        for (int32_t r = offsets[e]; r < offsets[e + 1]; ++r) expert_of[(size_t)r] = e;
    parallel_for(n, nthreads, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r) {
            const int64_t e = expert_of[(size_t)r], t = src[r];
            for (int64_t j = 0; j < 2 * (int64_t)F; ++j) {
                const int64_t wrow = e * 2 * F + j;
                gu[r * 2 * F + j] = q2_q8_dot(wc + wrow * (H / 4), ws + wrow * (H / 32), xc + t * H, xs + t * (H / 32), H);
            }
        }
    });
}

// ------------------------------------------------------------------------------------------------ step 5: SwiGLU
/// [P1] mmq::swiglu(GU, H, rows, ...) and [P3] moe_fused.hpp's "SwiGLU, H as int8": h_j = silu(g_j) * u_j in
/// double (R7), rounded to fp32, then the q8 rule (R3) per 32 values of h.
/// gu double [n][2F] -> hc int8 [n][F], hs fp16 [n][F/32].
void oracle_swiglu_requant(const double* gu, int64_t n, int F, int8_t* hc, uint16_t* hs, int nthreads) {
    parallel_for(n, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<float> h((size_t)F);
        for (int64_t r = r0; r < r1; ++r) {
            const double* g = gu + r * 2 * F;
            for (int j = 0; j < F; ++j) h[(size_t)j] = (float)(silu(g[j]) * g[F + j]);
            for (int b = 0; b < F / 32; ++b) q8_block(h.data() + b * 32, hc + r * F + b * 32, hs + r * (F / 32) + b);
        }
    });
}

/// The same step on fp32 gate/up values (a kernel's own GU buffer type): each value widened to double first.
void oracle_swiglu_requant_f32(const float* gu, int64_t n, int F, int8_t* hc, uint16_t* hs, int nthreads) {
    parallel_for(n, nthreads, [&](int64_t r0, int64_t r1) {
        std::vector<double> g((size_t)2 * F);
        for (int64_t r = r0; r < r1; ++r) {
            for (int64_t j = 0; j < 2 * (int64_t)F; ++j) g[(size_t)j] = (double)gu[r * 2 * F + j];
            oracle_swiglu_requant(g.data(), 1, F, hc + r * F, hs + r * (F / 32), 1);
        }
    });
}

// ------------------------------------------------------------------------------------------------ step 6: down
/// [P3] moe_fused.hpp experts(): "down into dm [n][2560] FP32 at the rows of group":
/// D[r][o] = sum_b d_w[e][o][b] * d_h[r][b] * sum_{i in b} (q_w - 2) * q_h, o in [0, H).
/// hc int8 [n][F], hs fp16 [n][F/32]; wc uint8 [E][H][F/4], ws fp16 [E][H][F/32]; dm double [n][H].
void oracle_down(const int8_t* hc, const uint16_t* hs, const int32_t* offsets, int E, const uint8_t* wc,
                 const uint16_t* ws, int H, int F, double* dm, int nthreads) {
    const int64_t n = offsets[E];
    std::vector<int32_t> expert_of((size_t)n);
    for (int e = 0; e < E; ++e)
        for (int32_t r = offsets[e]; r < offsets[e + 1]; ++r) expert_of[(size_t)r] = e;
    parallel_for(n, nthreads, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r) {
            const int64_t e = expert_of[(size_t)r];
            for (int64_t o = 0; o < H; ++o) {
                const int64_t wrow = e * H + o;
                dm[r * H + o] = q2_q8_dot(wc + wrow * (F / 4), ws + wrow * (F / 32), hc + r * F, hs + r * (F / 32), F);
            }
        }
    });
}

// ------------------------------------------------------------------------------------------------ step 7: combine
/// [P1] the combine that reads the per-slot rows (R8): Y[t][o] = sum_{k=0}^{K-1} w[t][k] * Dm[slot[t*K+k]][o].
void oracle_combine(const double* dm, const int32_t* slot, const double* w, int64_t T, int K, int H, double* y,
                    int nthreads) {
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        for (int64_t t = t0; t < t1; ++t)
            for (int64_t o = 0; o < H; ++o) {
                double acc = 0.0;
                for (int k = 0; k < K; ++k) acc += w[t * K + k] * dm[(int64_t)slot[t * K + k] * H + o];
                y[t * H + o] = acc;
            }
    });
}

// ------------------------------------------------------------------------------------------------ shared expert
/// [P1] Prefill::run, MoE half, "the shared expert and its scalar gate": the gate is a projection of the token onto
/// one row, read as sg[t] = sigmoid(sum_h x[t][h] * w_sg[h]) in double (R14).  x fp32 [T][H], wsg fp32 [H].
void oracle_shared_gate(const float* x, const float* wsg, int64_t T, int H, double* sg, int nthreads) {
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        for (int64_t t = t0; t < t1; ++t) {
            double z = 0.0;
            for (int64_t h = 0; h < H; ++h) z += (double)x[t * H + h] * (double)wsg[h];
            sg[t] = 1.0 / (1.0 + std::exp(-z));
        }
    });
}

/// [P1] the shared expert's gate and up projections, SwiGLU, and down projection of every token (R14): the steps
/// 3-6 above with one expert that all T tokens take (row r = token r).  s double [T][H].
void oracle_shared_expert(const float* x, int64_t T, int H, int F, const uint8_t* wgu_c, const uint16_t* wgu_s,
                          const uint8_t* wd_c, const uint16_t* wd_s, double* s, int nthreads) {
    std::vector<int8_t> xc((size_t)(T * H));
    std::vector<uint16_t> xs((size_t)(T * H / 32));
    oracle_quantize_q8(x, T, H, xc.data(), xs.data(), nthreads);
    std::vector<int32_t> src((size_t)T);
    for (int64_t t = 0; t < T; ++t) src[(size_t)t] = (int32_t)t;
    const int32_t offsets[2] = {0, (int32_t)T};
    std::vector<double> gu((size_t)(T * 2 * F));
    oracle_gateup(xc.data(), xs.data(), src.data(), offsets, 1, wgu_c, wgu_s, H, F, gu.data(), nthreads);
    std::vector<int8_t> hc((size_t)(T * F));
    std::vector<uint16_t> hs((size_t)(T * F / 32));
    oracle_swiglu_requant(gu.data(), T, F, hc.data(), hs.data(), nthreads);
    oracle_down(hc.data(), hs.data(), offsets, 1, wd_c, wd_s, H, F, s, nthreads);
}

/// The combine with the shared expert (R8, R14): Y[t][o] = sum_{k=0}^{K-1} w[t][k] * Dm[slot[t*K+k]][o], then
/// + sg[t] * S[t][o].
void oracle_combine_shared(const double* dm, const int32_t* slot, const double* w, const double* s, const double* sg,
                           int64_t T, int K, int H, double* y, int nthreads) {
    oracle_combine(dm, slot, w, T, K, H, y, nthreads);
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        for (int64_t t = t0; t < t1; ++t)
            for (int64_t o = 0; o < H; ++o) y[t * H + o] += sg[t] * s[t * H + o];
    });
}

// ------------------------------------------------------------------------------------------------ whole block
/// The seven steps in the pages' order on one prompt chunk; y double [T][H].  Returns oracle_group's status.
int oracle_layer(const float* logits, const float* x, int64_t T, int H, int E, int K, int F, const uint8_t* wgu_c,
                 const uint16_t* wgu_s, const uint8_t* wd_c, const uint16_t* wd_s, double* y, int nthreads) {
    const int64_t n = T * K;
    std::vector<int32_t> ids((size_t)n), counts((size_t)E), offsets((size_t)E + 1), src((size_t)n), slot((size_t)n);
    std::vector<double> w((size_t)n);
    oracle_route(logits, T, E, K, ids.data(), w.data(), nthreads);
    if (oracle_group(ids.data(), T, K, E, counts.data(), offsets.data(), src.data(), slot.data()) != 0)
        return -1;
    std::vector<int8_t> xc((size_t)(T * H));
    std::vector<uint16_t> xs((size_t)(T * H / 32));
    oracle_quantize_q8(x, T, H, xc.data(), xs.data(), nthreads);
    std::vector<double> gu((size_t)(n * 2 * F));
    oracle_gateup(xc.data(), xs.data(), src.data(), offsets.data(), E, wgu_c, wgu_s, H, F, gu.data(), nthreads);
    std::vector<int8_t> hc((size_t)(n * F));
    std::vector<uint16_t> hs((size_t)(n * F / 32));
    oracle_swiglu_requant(gu.data(), n, F, hc.data(), hs.data(), nthreads);
    std::vector<double>().swap(gu);
    std::vector<double> dm((size_t)(n * H));
    oracle_down(hc.data(), hs.data(), offsets.data(), E, wd_c, wd_s, H, F, dm.data(), nthreads);
    oracle_combine(dm.data(), slot.data(), w.data(), T, K, H, y, nthreads);
    return 0;
}

/// The block with the shared expert (R14): oracle_layer, then + sg[t] * S[t].  y double [T][H].
int oracle_layer_shared(const float* logits, const float* x, int64_t T, int H, int E, int K, int F,
                        const uint8_t* wgu_c, const uint16_t* wgu_s, const uint8_t* wd_c, const uint16_t* wd_s,
                        const uint8_t* sgu_c, const uint16_t* sgu_s, const uint8_t* sd_c, const uint16_t* sd_s,
                        const float* wsg, double* y, int nthreads) {
    if (oracle_layer(logits, x, T, H, E, K, F, wgu_c, wgu_s, wd_c, wd_s, y, nthreads) != 0) return -1;
    std::vector<double> s((size_t)(T * H)), sg((size_t)T);
    oracle_shared_expert(x, T, H, F, sgu_c, sgu_s, sd_c, sd_s, s.data(), nthreads);
    oracle_shared_gate(x, wsg, T, H, sg.data(), nthreads);
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        for (int64_t t = t0; t < t1; ++t)
            for (int64_t o = 0; o < H; ++o) y[t * H + o] += sg[(size_t)t] * s[(size_t)(t * H + o)];
    });
    return 0;
}

/// The block for a chosen set of tokens only, one token at a time (no grouping: a routed row's values do not depend
/// on where the grouping puts it).  Used where the whole chunk is too large for the oracle.  For each listed token
/// t: route its logits, quantise its x row, and for each of its K experts: gate/up, SwiGLU + requant, down; then the
/// weighted combine.  y double [ntok][H]; ids_out int32 [ntok][K] and w_out double [ntok][K] may be null.
void oracle_layer_tokens_h(const float* logits, const float* x, const int64_t* tokens, int64_t ntok, int H, int E,
                           int K, int F, const uint8_t* wgu_c, const uint16_t* wgu_s, const uint8_t* wd_c,
                           const uint16_t* wd_s, double* y, int32_t* ids_out, double* w_out, float* h_out,
                           int8_t* hc_out, uint16_t* hs_out, int nthreads);

void oracle_layer_tokens(const float* logits, const float* x, const int64_t* tokens, int64_t ntok, int H, int E,
                         int K, int F, const uint8_t* wgu_c, const uint16_t* wgu_s, const uint8_t* wd_c,
                         const uint16_t* wd_s, double* y, int32_t* ids_out, double* w_out, int nthreads) {
    oracle_layer_tokens_h(logits, x, tokens, ntok, H, E, K, F, wgu_c, wgu_s, wd_c, wd_s, y, ids_out, w_out, nullptr,
                          nullptr, nullptr, nthreads);
}

/// oracle_layer_tokens that also hands out, per listed token s and slot k, the step-5 intermediates of that pair:
/// h_out fp32 [ntok][K][F] (h rounded to fp32, the q8 rule's input), hc_out int8 [ntok][K][F] and hs_out fp16 bits
/// [ntok][K][F/32] (its q8 codes and scales).  Any of the three may be null.
void oracle_layer_tokens_h(const float* logits, const float* x, const int64_t* tokens, int64_t ntok, int H, int E,
                           int K, int F, const uint8_t* wgu_c, const uint16_t* wgu_s, const uint8_t* wd_c,
                           const uint16_t* wd_s, double* y, int32_t* ids_out, double* w_out, float* h_out,
                           int8_t* hc_out, uint16_t* hs_out, int nthreads) {
    parallel_for(ntok, nthreads, [&](int64_t s0, int64_t s1) {
        std::vector<int32_t> ids((size_t)K);
        std::vector<double> w((size_t)K), gu((size_t)2 * F), dm((size_t)H);
        std::vector<int8_t> xc((size_t)H), hc((size_t)F);
        std::vector<uint16_t> xs((size_t)H / 32), hs((size_t)F / 32);
        for (int64_t s = s0; s < s1; ++s) {
            const int64_t t = tokens[s];
            oracle_route(logits + t * E, 1, E, K, ids.data(), w.data(), 1);
            oracle_quantize_q8(x + t * H, 1, H, xc.data(), xs.data(), 1);
            double* yt = y + s * H;
            for (int64_t o = 0; o < H; ++o) yt[o] = 0.0;
            for (int k = 0; k < K; ++k) {
                const int64_t e = ids[(size_t)k];
                for (int64_t j = 0; j < 2 * (int64_t)F; ++j) {
                    const int64_t wrow = e * 2 * F + j;
                    gu[(size_t)j] = q2_q8_dot(wgu_c + wrow * (H / 4), wgu_s + wrow * (H / 32), xc.data(), xs.data(), H);
                }
                oracle_swiglu_requant(gu.data(), 1, F, hc.data(), hs.data(), 1);
                const int64_t pk = s * K + k;
                if (h_out)
                    for (int j = 0; j < F; ++j) h_out[pk * F + j] = (float)(silu(gu[(size_t)j]) * gu[(size_t)(F + j)]);
                if (hc_out) std::memcpy(hc_out + pk * F, hc.data(), (size_t)F);
                if (hs_out) std::memcpy(hs_out + pk * (F / 32), hs.data(), (size_t)(F / 32) * sizeof(uint16_t));
                for (int64_t o = 0; o < H; ++o) {
                    const int64_t wrow = e * H + o;
                    dm[(size_t)o] = q2_q8_dot(wd_c + wrow * (F / 4), wd_s + wrow * (F / 32), hc.data(), hs.data(), F);
                }
                for (int64_t o = 0; o < H; ++o) yt[o] += w[(size_t)k] * dm[(size_t)o];
            }
            if (ids_out)
                for (int k = 0; k < K; ++k) ids_out[s * K + k] = ids[(size_t)k];
            if (w_out)
                for (int k = 0; k < K; ++k) w_out[s * K + k] = w[(size_t)k];
        }
    });
}

/// A second route to the same numbers, for pinning: every weight and every q8 value dequantised to double first
/// (w = d * (q - 2), a = d_a * q_a, h = d_h * q_h), then plain dot products per token and expert, with no block
/// structure and no grouping.  Equal to oracle_layer up to double rounding.  y double [T][H].
void oracle_layer_bruteforce(const float* logits, const float* x, int64_t T, int H, int E, int K, int F,
                             const uint8_t* wgu_c, const uint16_t* wgu_s, const uint8_t* wd_c, const uint16_t* wd_s,
                             double* y, int nthreads) {
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        std::vector<int32_t> ids((size_t)K);
        std::vector<double> w((size_t)K), a((size_t)H), g((size_t)2 * F), hd((size_t)F);
        std::vector<int8_t> xc((size_t)H), hc((size_t)F);
        std::vector<uint16_t> xs((size_t)H / 32), hs((size_t)F / 32);
        std::vector<float> hf((size_t)F);
        for (int64_t t = t0; t < t1; ++t) {
            oracle_route(logits + t * E, 1, E, K, ids.data(), w.data(), 1);
            oracle_quantize_q8(x + t * H, 1, H, xc.data(), xs.data(), 1);
            for (int i = 0; i < H; ++i) a[(size_t)i] = (double)h2f(xs[(size_t)i / 32]) * (double)xc[(size_t)i];
            for (int o = 0; o < H; ++o) y[t * H + o] = 0.0;
            for (int k = 0; k < K; ++k) {
                const int64_t e = ids[(size_t)k];
                for (int64_t j = 0; j < 2 * (int64_t)F; ++j) {
                    const int64_t wrow = e * 2 * F + j;
                    double s = 0.0;
                    for (int64_t i = 0; i < H; ++i)
                        s += (double)h2f(wgu_s[wrow * (H / 32) + i / 32]) * (double)(q2_code(wgu_c + wrow * (H / 4), i) - 2) * a[(size_t)i];
                    g[(size_t)j] = s;
                }
                for (int j = 0; j < F; ++j) hf[(size_t)j] = (float)(silu(g[(size_t)j]) * g[(size_t)F + j]);
                oracle_quantize_q8(hf.data(), 1, F, hc.data(), hs.data(), 1);
                for (int j = 0; j < F; ++j) hd[(size_t)j] = (double)h2f(hs[(size_t)j / 32]) * (double)hc[(size_t)j];
                for (int64_t o = 0; o < H; ++o) {
                    const int64_t wrow = e * H + o;
                    double s = 0.0;
                    for (int64_t i = 0; i < F; ++i)
                        s += (double)h2f(wd_s[wrow * (F / 32) + i / 32]) * (double)(q2_code(wd_c + wrow * (F / 4), i) - 2) * hd[(size_t)i];
                    y[t * H + o] += w[(size_t)k] * s;
                }
            }
        }
    });
}

}  // extern "C"
