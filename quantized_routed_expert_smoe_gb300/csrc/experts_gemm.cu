// experts_gemm.cu -- the grouped expert products of the routed-expert block (steps 4 and 6) on the 5th-generation
// tensor cores (tcgen05.mma, operands in tensor and shared memory, accumulators in tensor memory), sm_103a.
//
// Page "Strata compare v0.1.35...v0.1.37", include/strata/prefill/moe_fused.hpp experts(): for each expert, gate/up
// of its routed rows from the per-token int8 activations against its 2-bit weights, then down into one fp32 row per
// routed pair.  Per output:  sum_b dB[b] * (dW[b] * sum_{i in b} (qW - 2) * qB)  over the 32-value blocks b of K.
//
// Arithmetic.  The 5th-generation tensor cores of this part have no int8 kind (ptxas rejects kind::i8 for
// sm_103a), so the contraction runs as tcgen05.mma.kind::f16 on fp16 operands that carry the quantised values
// EXACTLY:
//   - the weight operand is d_w * (q_w - 2), q_w in {0..3}: d_w times {-2, -1, 0, 1}, exact in fp16;
//   - the row operand d * q (at most 18 significant bits) comes as two fp16 parts, hi = fp16_rn(d q) and
//     lo = d q - hi (exact), written by the routed-row gather (activations) and by SwiGLU (H).
// Every product of a weight and a part is exact in fp32, and the K loop runs two MMAs per 16-wide K step (A x hi,
// A x lo).  The tensor core's fp32 accumulation aligns its addends with truncation, which over a whole row of K
// costs about 3e-6 of the result -- enough to flip requantised H codes -- so for gate/up (whose output is
// requantised) each 128-wide piece of K (two slices) accumulates from zero into one of two tensor-memory buffers (a
// small partial, so a small truncation error) and the promoter warps add each finished partial into fp32 registers
// with round-to-nearest while the tensor core fills the other buffer.  The down product feeds the fp32 combine only,
// where 4e-6 is far inside the output bound, so it accumulates the whole K in one buffer, read once at the end.
//
// Data movement, chosen to keep the CUDA-core work per slice small (shared-memory traffic and the converters'
// latency bounded the earlier designs):
//   - both parts of the row operand are stored in HBM in operand order, so TMA loads them straight into the
//     canonical K-major 128-byte-swizzled layout the MMA reads (no conversion pass through shared memory);
//   - the weight operand (A) is decoded from the packed 2-bit block by the converter warps directly into TENSOR
//     memory (tcgen05.st; lane = weight row, 32-bit column = a pair of K values) and the MMA reads it from there.
//
// Tile: one CTA = one tile of the tile list (an expert and up to 192 of its routed rows, contiguous in routed-row
// order; the MMA's N, a multiple of 16) x one 128-row slice of the expert's weight matrix (the MMA's M; swap-AB:
// weights are the M operand so that a small expert wastes little).
//
// Two forms.  The CTA-pair form (a weight matrix with an even number of 128-row slices and K a multiple of 128) runs
// the MMAs over a pair of CTAs with tcgen05 cta_group::2: M = 256, each CTA decoding and accumulating its own 128
// weight rows, and the tile's B rows split between the two CTAs' shared memories (a tile of at most 96 rows: its hi
// rows in the even CTA and its lo rows in the odd one, one MMA of 2N; a larger tile: N/2 rows of each part in each).
// The tensor cores of both SMs read both halves, so each SM takes in half the row bytes per MMA of the single-CTA
// form, its ring slots are half as large and twice as many slices are in flight.  A cluster is one pair.  The even
// CTA issues the pair's MMAs: both CTAs' converter warps meet on its `ready` barrier, both CTAs' B copies count
// their bytes on its stage barrier (the cta_group::2 form of the TMA load) and both CTAs' promoter warps arrive on
// its `pempty`; its commits release the slots and signal the partials in both CTAs.  The single-CTA form (any other
// shape) issues its own MMAs.  No TMA load is multicast.
//
// Stages.  Every barrier hand-over costs a few hundred cycles, so the ring's barriers are per STAGE: S consecutive
// 64-wide slices (pair form S = 2, 128 values of K; single form S = 1) share one wait of the producer, one arrival
// of each converter warp, one wait and one commit of the MMA thread.
//
// Five warpgroups, registers rebalanced with setmaxnreg (launched at 96; warpgroup 0 and the converters 48, the
// promoters 128):
//   warpgroup 0   warps 0 and 2, one lane each: the MMAs of alternate stages -- of alternate groups of 128 values
//                 of K for gate/up (one thread's waits overlap the other's MMAs; a stage's MMAs go out from one
//                 asm block with every operand computed before the wait); warp 0 also allocates the tensor memory;
//                 warp 1: the producer -- per 64-wide K slice, one TMA tile load of the tile's rows of each part
//                 (128-byte swizzle; pair form: this CTA's half of them) and one bulk copy of the packed weight
//                 block into a ring slot;
//   warpgroups 1-3  promoters: add each finished partial into fp32 registers (a TMEM lane a thread, every third
//                 32-column chunk a warpgroup), then write the fp32 rows (or, for the down product's narrow form,
//                 the same values rounded to fp16) -- or, for the fused SwiGLU product (gate and up rows interleaved
//                 in the packed weights), h = silu(g) * u requantised to q8, planar and in operand form;
//   warpgroup 4   converters: thread = weight row: decode its 64 weights of the slice into the slice's A buffer in
//                 tensor memory (three register instructions a column of two weights).
// Tensor memory (512 columns): 4 A buffers of 32 columns, then the partial buffers in the other 384 -- as many as
// the launch's widest partial allows (2 for 97..192 columns, 3 up to 128, 4 up to 96; a tile's partial takes N
// columns, or 2N for a tile of at most 96 rows, which stacks its hi and lo rows into one MMA).  Gate/up promotes a
// partial every 128 values of K, down one partial per MMA thread at the item's end.  A tile has at most 192 rows: a
// promoter thread then holds its 64 accumulators and one 32-column load.
//
// Synchronisation: a satisfied mbarrier wait still costs a round trip of a few hundred cycles, and the ring's slots
// circulate through a chain of latencies (slot released -> copies issued -> landed -> A decoded -> MMAs -> released),
// so each role waits as little as it can and nothing waits on what it does not need.  A stage's packed weights land
// on their own barrier, so the converters decode while the B tiles are still in flight; in the single form they
// wait on nothing else -- its ring has as many slots as A buffers, so a slot's new contents also mean that the MMAs
// of the slice that last used its A buffer have completed (the pair form's ring is twice as deep, so there they also
// wait for the release of the stage that last used the A buffers) -- and test the next stage's barriers while a
// stage's stores complete.  The MMA thread waits once per stage, in one round trip, on "A decoded", "B tiles landed"
// and, for a stage that starts a partial in a buffer used before, "the promoters have taken that buffer's previous
// partial".
//
// K order: within each group of 16 K values, operand position 2m holds value m and position 2m+1 value m+8
// (m = 0..7) -- the order in which 2-bit codes unpack in pairs -- for A and B alike, so the contraction is unchanged
// and each 32-value half of a slice is two whole K16 steps.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "smoe_device.cuh"
#include "smoe_internal.h"

namespace smoe {
namespace {

constexpr int kBM = 128;                       // weight rows per CTA (MMA M)
constexpr int kBK = 64;                        // K values per slice: one 128-byte swizzle row of fp16
constexpr int kMaxBN = SMOE_TILE_ROWS;         // routed rows per tile (MMA N <= 224)
constexpr int kThreads = 640;                  // five warpgroups
constexpr int kPromoters = 384;                // warpgroups 1-3
constexpr int kConverters = 128;               // warpgroup 4 (a weight row a thread)
constexpr int kMaxRing = 8;                    // slices in flight at most
constexpr int kMmaThreads = 2;                 // MMA-issuing threads (warps 0, 2): slice groups in turn
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = 32;                // one slice of A: 128 lanes x 64 fp16
constexpr int kMaxA = 8;                       // A buffers at most
constexpr int kMaxBufs = 4;                    // partial buffers at most
constexpr int kMaxStackN = 96;                 // tiles up to this N stack hi and lo rows into one MMA
constexpr int kSmemBytes = 232448;             // the per-CTA maximum (227 KB): [align slack][ring][barriers]
constexpr int kBarBytes = 512;
constexpr int kScratchBytes = SMOE_TILE_ROWS * 4 * 4;  // SwiGLU epilogue: a warp's block amax per column [col][4]
constexpr int kRingBytes = kSmemBytes - 1024 - kBarBytes - kScratchBytes;
// registers: launched at 96 a thread (640 x 96 = 61,440 of 65,536); warpgroup 0 and the converters give back to 48,
// the promoters take 128: 128 x 48 + 128 x 48 + 384 x 128 = 61,440.  Per SM sub-partition (one warp of each
// warpgroup): 32 x (48 + 48 + 3 x 128) = 15,360 <= 16,384.
constexpr int kRegsLaunch = 96;
constexpr int kRegsWg0 = 48;
constexpr int kRegsConv = 48;
constexpr int kRegsProm = 128;
static_assert(128 * kRegsWg0 + kConverters * kRegsConv + kPromoters * kRegsProm <= kThreads * kRegsLaunch,
              "register split exceeds the launch");
static_assert(kMaxBN <= 224 && kMaxBN % 32 == 0, "two partial buffers and two A buffers must fit in tensor memory");
static_assert(kMaxBN % 96 == 0, "the promoter warpgroups take whole 32-column chunks in turn");

// Ring slot (one 64-wide K slice of the tile): the rows of the hi part, then of the lo part (128 bytes a row,
// 128-byte swizzle, 1024-aligned), then the packed weight block (codes [128][16 B], scales [128][4 B]); slots are
// 1024-byte multiples.  A stacked tile's lo rows follow its N hi rows (one MMA reads both); a larger tile's parts
// take fixed regions of kMaxBN rows each.
constexpr int kWBlock = 2560;
// One TMA copy per part and slice, of exactly the tile's N rows: the map whose box is N = 16 (m + 1) rows (the
// SM's TMA unit, which every copy of the CTA shares, is on the ring's critical path; rows that are never read are
// not loaded).
constexpr int kRowBox = 16;                    // box-height step of the maps
constexpr int kNumMaps = kMaxBN / kRowBox;
__host__ __device__ constexpr int slot_bytes(int N) { return (2 * N * 128 + kWBlock + 1023) & ~1023; }
static_assert(kRingBytes / slot_bytes(kMaxBN) >= 3, "the ring must hold three slices of a full tile");
static_assert(kMaxStackN % kRowBox == 0 && kMaxBN % kRowBox == 0 && kMaxBN <= 256, "box heights");

// CTA-pair form (tcgen05 cta_group::2): the two CTAs of a pair hold 128 weight rows each (M = 256) and split the
// tile's B rows between their shared memories, so each SM receives half of the row bytes per MMA of the single form.
// A slot holds at most kPairRows rows of each part (a stacked tile: all N rows of ONE part -- hi in the leader, lo in
// the peer; a larger tile: N/2 rows of both parts), then the packed weights at a fixed offset.
constexpr int kPairRows = kMaxBN / 2;          // 96
constexpr int kPairBox = 8;                    // box-height step of the pair maps (N/2 is a multiple of 8)
constexpr int kPairWOfs = 2 * kPairRows * 128;  // the packed weight block within a pair slot
constexpr int kPairSlot = (kPairWOfs + kWBlock + 1023) & ~1023;
static_assert(kPairRows / kPairBox == kNumMaps && kMaxStackN <= kPairRows, "pair boxes");
static_assert(kRingBytes / kPairSlot >= 4, "the pair ring must hold four slices");

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

// TMA: a 2D tile into this CTA's shared memory whose completion is counted on the barrier at shared::cluster address
// `bar`, which may be the other CTA's of this CTA's pair (the pair's even CTA gathers both CTAs' bytes)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// every thread of every CTA of the cluster
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// --- barriers that receive arrivals from the other CTA of a pair.  What crosses between the two CTAs is tensor
// memory (ordered by tcgen05.wait::st/ld and the tcgen05 thread-sync fences around the barrier) and shared memory
// written by TMA (the async proxy, completed through the barrier's byte count), never generic stores that the other
// CTA loads, so the arrivals and waits keep the default CTA-scope release / acquire: a cluster-scope one is a full
// memory fence on every arrival and every poll, which stalled the pipeline's threads for most of their time.
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) { return mbar_try_wait(bar, parity); }
// wait (bounded, as mbar_wait) for the phases of two barriers
__device__ __forceinline__ bool mbar_wait2_cl(uint64_t* bar0, uint32_t parity0, uint64_t* bar1, uint32_t parity1,
                                              volatile int* abort) {
    const uint32_t a0 = smem_u32(bar0), a1 = smem_u32(bar1);
    bool d0 = mbar_try_wait_cl(a0, parity0), d1 = mbar_try_wait_cl(a1, parity1);
    if (d0 && d1) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (!d0) d0 = mbar_try_wait_cl(a0, parity0);
        if (!d1) d1 = mbar_try_wait_cl(a1, parity1);
        if (d0 && d1) return true;
        if (abort != nullptr && *abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort) {
    return mbar_wait2_cl(bar, parity, bar, parity, abort);
}
// the shared::cluster address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// one arrival on the barrier at shared::cluster address `addr` (of this CTA or another CTA of the cluster)
__device__ __forceinline__ void mbar_arrive_cl(uint32_t addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// arrive once on `bar` in every CTA of `mask` when the pair MMAs issued so far by this thread have completed
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}
// tensor-memory allocation of a CTA pair: one warp of EACH CTA of the pair executes these (collectively)
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// named barrier of `count` threads (whole warps)
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// named barrier that also returns whether `pred` held in every participating thread
__device__ __forceinline__ bool bar_red_and(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// 16 consecutive 32-bit TMEM columns of 32 lanes: thread i of the warp gets / gives lane (base lane + i)
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// One 64-wide K slice of MMAs (four K16 steps), issued back to back from one asm block: A columns a + 8 k and B
// descriptor b + 2 k (its start address 32 bytes further along the 128-byte swizzled rows) for step k; accumulate
// 0 starts the accumulator at step 0.  The issuing thread runs in order and each tensor-core instruction holds it
// for tens of cycles, so the operand arithmetic comes first and the MMAs follow without anything between them.
// kGroup: 2 = the pair form (cta_group::2), 1 = one CTA.
#define SMOE_MMA_SLICE4(GROUP)                                                                                      \
    "{\n\t.reg .pred p, t;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"                                  \
    "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, %3, %3;\n\t"                                                           \
    "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"                                        \
    "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"                                           \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [%1], %2, %3, p;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], b1, %3, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a2], b2, %3, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a3], b3, %3, t;\n\t}"
template <int kGroup>
__device__ __forceinline__ void mma_slice4(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    if constexpr (kGroup == 2)
        asm volatile(SMOE_MMA_SLICE4("2")::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
    else
        asm volatile(SMOE_MMA_SLICE4("1")::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
#undef SMOE_MMA_SLICE4
// The same with both parts of the row operand: per step k, the hi rows (descriptor bh + 2 k) then the lo rows
// (bl + 2 k) into the same accumulator.
#define SMOE_MMA_SLICE8(GROUP)                                                                                      \
    "{\n\t.reg .pred p, t;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 h1, h2, h3, l1, l2, l3;\n\t"                     \
    "setp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"                                                           \
    "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"                                        \
    "add.u64 h1, %2, 2;\n\tadd.u64 h2, %2, 4;\n\tadd.u64 h3, %2, 6;\n\t"                                           \
    "add.u64 l1, %3, 2;\n\tadd.u64 l2, %3, 4;\n\tadd.u64 l3, %3, 6;\n\t"                                           \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [%1], %2, %4, p;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [%1], %3, %4, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], h1, %4, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a1], l1, %4, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a2], h2, %4, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a2], l2, %4, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a3], h3, %4, t;\n\t"                                         \
    "tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], [a3], l3, %4, t;\n\t}"
template <int kGroup>
__device__ __forceinline__ void mma_slice8(uint32_t d, uint32_t a, uint64_t bh, uint64_t bl, uint32_t idesc,
                                           uint32_t accumulate) {
    if constexpr (kGroup == 2)
        asm volatile(SMOE_MMA_SLICE8("2")::"r"(d), "r"(a), "l"(bh), "l"(bl), "r"(idesc), "r"(accumulate) : "memory");
    else
        asm volatile(SMOE_MMA_SLICE8("1")::"r"(d), "r"(a), "l"(bh), "l"(bl), "r"(idesc), "r"(accumulate) : "memory");
}
#undef SMOE_MMA_SLICE8

// (a0, a1) += (p0, p1), each rounded to nearest (packed fp32x2 add)
__device__ __forceinline__ void add2(float& a0, float& a1, uint32_t p0, uint32_t p1) {
    asm("{\n\t.reg .b64 a, p;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 p, {%2, %3};\n\t"
        "add.rn.f32x2 a, a, p;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(p0), "r"(p1));
}

// 16 weights (codes: value i at bits 2i..2i+1) as 8 TMEM columns of fp16 pairs (value m, value m+8): d * (q - 2).
// Pair m's codes sit at bits 2m of each 16-bit half.  OR-ed under the exponent of 2^(10 - 2m) they read as the fp16
// value 2^(10 - 2m) + q exactly (a mantissa bit at position 2m weighs 2^(10 - 2m - 10 + 2m) = 1), so pairs 0-4 need
// no shift; pairs 5-7 take the word shifted by 10 (their codes at bits 0, 2, 4).  Subtracting 2^e + 2 leaves q - 2
// exactly, and the product with d is exact in fp16.  Three instructions a column, all on registers.
template <int kPos>
__device__ __forceinline__ uint32_t decode_pair(uint32_t codes, uint32_t d2) {
    constexpr int e = 10 - 2 * kPos;
    constexpr uint32_t mask = 0x00030003u << (2 * kPos);
    constexpr uint32_t expo = ((uint32_t)(e + 15) << 10) * 0x00010001u;
    constexpr uint32_t base = (((uint32_t)(e + 15) << 10) | (2u << (10 - e))) * 0x00010001u;  // 2^e + 2, both halves
    uint32_t out;
    asm("{\n\t.reg .b32 v;\n\t"
        "lop3.b32 v, %1, %2, %3, 0xEA;\n\t"  // (codes & mask) | expo
        "sub.rn.f16x2 v, v, %4;\n\t"
        "mul.rn.f16x2 %0, v, %5;\n\t}"
        : "=r"(out)
        : "r"(codes), "n"(mask), "n"(expo), "r"(base), "r"(d2));
    return out;
}
// d2: the block's fp16 scale in both halves
__device__ __forceinline__ void decode_weights16(uint32_t codes, uint32_t d2, uint32_t* col) {
    const uint32_t high = codes >> 10;
    col[0] = decode_pair<0>(codes, d2);
    col[1] = decode_pair<1>(codes, d2);
    col[2] = decode_pair<2>(codes, d2);
    col[3] = decode_pair<3>(codes, d2);
    col[4] = decode_pair<4>(codes, d2);
    col[5] = decode_pair<0>(high, d2);
    col[6] = decode_pair<1>(high, d2);
    col[7] = decode_pair<2>(high, d2);
}

struct GemmMaps {
    // the two parts of the B rows: fp16 [b_rows][K] each, 128-byte swizzle, boxes of 64 values x 16 (m + 1) rows
    CUtensorMap hi[kNumMaps], lo[kNumMaps];
};

// One work item: a tile of the tile list x one group of C consecutive 128-row weight slices (one per CTA of the
// cluster).  Every role of every CTA walks the same item sequence and skips the same invalid items.
struct Item {
    int e, row0, rows, N, m0;
    bool stacked;  // N <= kMaxStackN: hi and lo rows in one MMA of 2N columns
    int ncols;     // partial columns
    int lo_rows;   // slot row where the lo part starts (N stacked, kMaxBN otherwise; pair form: kPairRows)
    int map;       // tensor maps of its parts (one box per part)
};
template <bool kPair>
__device__ __forceinline__ bool load_item(const int32_t* tiles, int item, int mgroups, int C, uint32_t crank,
                                          const ExpertsGemmArgs& p, Item& t) {
    const int ti = item / mgroups, mg = item - ti * mgroups;
    const int4 te = reinterpret_cast<const int4*>(tiles)[1 + ti];
    t.e = te.x;
    t.row0 = te.y;
    t.rows = te.z;
    // a tile the grouping cannot have written (a bad expert id or row range): nothing is read or written for it
    if (t.rows <= 0 || t.rows > kMaxBN || t.e < 0 || t.e >= p.n_experts || t.row0 < 0 ||
        t.row0 + (int64_t)t.rows > p.b_rows)
        return false;
    t.N = (t.rows + 15) & ~15;
    t.m0 = (mg * C + (int)crank) * kBM;
    t.stacked = t.N <= kMaxStackN;
    t.ncols = t.stacked ? 2 * t.N : t.N;
    if (kPair) {
        // each CTA's box: all N rows of its one part (stacked) or N/2 rows of each part
        t.lo_rows = kPairRows;
        t.map = (t.stacked ? t.N : t.N / 2) / kPairBox - 1;
    } else {
        t.lo_rows = t.stacked ? t.N : kMaxBN;
        t.map = t.N / kRowBox - 1;
    }
    return true;
}

// kPair: the CTA-pair form (cluster of C = 2 or 4 CTAs = C/2 pairs).  Ranks 2q and 2q + 1 form pair q; the even CTA
// (the leader) issues the pair's MMAs.  Per slice the leader waits on its `ready` barrier, which both CTAs' converter
// warps (A decoded into their tensor memory) and B relays (their B rows landed) arrive on, and -- before a partial
// buffer is reused -- on `pempty`, which both CTAs' promoter warps arrive on.  The leader's commits signal slot
// releases in every CTA of the cluster and partials and the final drain in both CTAs of its pair.
template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1) experts_gemm_kernel(const ExpertsGemmArgs p,
                                                                   const __grid_constant__ GemmMaps maps) {
    int32_t* tiles = p.tiles;
    if (tiles[1] != 0) return;  // the grouping failed: nothing to do (the same answer in every CTA)
    const int n_tiles = tiles[0];
    if (n_tiles < 0 || n_tiles > p.max_tiles) {  // not a tile list of this size: read nothing beyond it
        if (blockIdx.x == 0 && threadIdx.x == 0) tiles[3] = SMOE_ERR_ARG;
        return;
    }
    const int nk = p.K / kBK;  // slices of an item
    // A stage is S consecutive slices (pair form: S = 2, K a multiple of 128; single form: S = 1) with one set of
    // ring barriers: one wait of the MMA thread, one commit, one arrival of each converter warp for S slices' work.
    constexpr int S = kPair ? 2 : 1;
    const int nsi = nk / S;  // stages of an item
    // two MMA threads take alternate groups of Gs stages.  Two-level: a partial per 128 values of K (Gs = 2 / S
    // stages); else one partial per thread of an item (Gs = 1: stages ks, ks + 2, ... of one parity), summed by the
    // promoters
    const int Gs = p.two_level ? 2 / S : 1;
    const int pitem = p.two_level ? nk / 2 : min(kMmaThreads, nsi);  // partials an item

    // persistent: cluster cid of NC takes items cid, cid + NC, ...; its CTAs take the C weight slices of an item
    // (pair form: a cluster is one pair; single form: one CTA)
    constexpr int C = kPair ? 2 : 1;
    const uint32_t crank = kPair ? cluster_rank() : 0u;
    const int mgroups = p.a_rows / kBM / C;
    const int n_items = n_tiles * mgroups;
    const int cid = blockIdx.x / C, NC = gridDim.x / C;
    // pair form: this CTA's position in its pair (0 = the leader, which issues the MMAs)
    const uint32_t ppos = crank, leader = 0u;
    constexpr uint16_t pmask = 3u;  // both CTAs of the pair

    // fixed geometry for every item (tiles of up to kMaxBN rows): a ring of `depth` slots, na A buffers and nbuf
    // partial buffers (nbuf set per launch, below) in tensor memory
    constexpr int sbytes = kPair ? kPairSlot : slot_bytes(kMaxBN);
    constexpr int na = ((int)kTmemCols - 2 * kMaxBN) / (int)kACols;
    // the single form: as many ring slots as A buffers (its slots are large); the pair form: twice as many (its slots
    // hold half the B rows), so that twice the slices are in flight against the ring's chain of latencies
    constexpr int depth = kPair ? 2 * na : na;
    constexpr int nst = depth / S;  // stage slots of the ring (stage slot j: ring slots S j .. S j + S - 1)
    static_assert(depth % S == 0 && na % S == 0, "whole stages");
    constexpr uint32_t part_base = (uint32_t)na * kACols;
    constexpr int kPartCols = (int)kTmemCols - (int)part_base;  // the partial buffers' columns
    static_assert(na >= 2 && na <= kMaxA && kPartCols / kMaxBN >= 2, "tensor-memory split");
    static_assert(depth <= kMaxRing && depth <= kMaxA && depth * sbytes <= kRingBytes, "ring");
    // slice gs uses ring slot gs mod depth and A buffer gs mod na; its stage gs / S uses stage slot (gs / S) mod nst,
    // whose barriers it shares with the other slices of the stage.  Single form (depth == na): its copies can land
    // only after the producer has seen the slot's previous slice (gs - depth) released by the MMA commits, which
    // follow that slice's MMAs, the last readers of the A buffer, so "weights landed" also means "A buffer free".
    // Pair form (depth == 2 na): the converters also wait for the release of stage gs / S - na / S, the previous user
    // of the stage's A buffers, before they overwrite them

    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t* ring = smem_raw + pad;
    // (indexed by stage slot)
    uint64_t* sfull = reinterpret_cast<uint64_t*>(smem_raw + kSmemBytes - kBarBytes);  // the stage's B tiles [nst]
    uint64_t* wfull = sfull + kMaxRing;     // the stage's packed weight blocks landed [nst]
    uint64_t* sempty = wfull + kMaxRing;    // the MMAs and the converters are done with the stage's slots [nst]
    uint64_t* afull = sempty + kMaxRing;    // the stage's A buffers decoded [nst] (pair form: on the leader)
    uint64_t* pfull = afull + kMaxA;        // partial in tensor-memory buffer b is complete [kMaxBufs]
    uint64_t* pempty = pfull + kMaxBufs;    // the promoters have added buffer b into their registers [kMaxBufs]
    uint64_t* accf = pempty + kMaxBufs;     // every MMA has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* total_slot = const_cast<int*>(abort_flag + 1);  // stages this CTA ran (for the teardown)
    int* maxcols_slot = total_slot + 1;                  // the launch's widest partial (columns)
    float* scratch = reinterpret_cast<float*>(smem_raw + kSmemBytes - kBarBytes - kScratchBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        // pair form: arrivals are per warp (converters, promoters) and come from both CTAs of the pair
        for (int r = 0; r < kMaxRing; ++r) {
            // the arrival that posts the B tiles' byte count (pair form: the leader's, with both CTAs' bytes)
            mbar_init(&sfull[r], 1);
            mbar_init(&wfull[r], 1);                 // the arrival that posts the weight block's
            // the MMAs' commit (the leader's, in both CTAs of a pair), then the own converters
            mbar_init(&sempty[r], kPair ? 1 + kConverters / 32 : 1 + kConverters);
        }
        // A decoded: every converter (pair form: the converter warps of both CTAs, on the leader's barrier)
        for (int a = 0; a < kMaxA; ++a) mbar_init(&afull[a], kPair ? 2 * (kConverters / 32) : kConverters);
        for (int b = 0; b < kMaxBufs; ++b) {
            mbar_init(&pfull[b], 1);
            mbar_init(&pempty[b], kPair ? 2 * (kPromoters / 32) : kPromoters);
        }
        mbar_init(accf, kMmaThreads);  // one final commit of each MMA thread
        *abort_flag = 0;
        *total_slot = 0;
        *maxcols_slot = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        if constexpr (kPair) {
            tmem_alloc_pair(tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync();  // both CTAs' barriers are initialised before any remote copy or arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the launch's widest partial (every CTA finds the same in the tile list) sets the partial buffers: as many as
    // tensor memory holds, at most kMaxBufs -- two for tiles of 97 rows and more, four for tiles of at most 48 rows
    // (96 stacked columns), so that small tiles keep more partials in flight against the promoters' round trip
    {
        int m = 0;
        for (int ti = threadIdx.x; ti < n_tiles; ti += kThreads) {
            const int rows = tiles[4 * (1 + ti) + 2];
            if (rows > 0 && rows <= kMaxBN) {
                const int N = (rows + 15) & ~15;
                m = max(m, N <= kMaxStackN ? 2 * N : N);
            }
        }
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0 && m > 0) atomicMax(maxcols_slot, m);
    }
    __syncthreads();
    const int bufw = (max(*maxcols_slot, 32) + 31) & ~31;  // columns of a partial buffer
    const int nbuf = min(kMaxBufs, kPartCols / bufw);      // 2, 3 or 4
    // partial gp's buffer and its use of it (nbuf is a power of two or 3: no division on the MMA thread's path)
    auto buf_of = [nbuf](int gp) { return nbuf == 3 ? gp % 3 : gp & (nbuf - 1); };
    auto use_of = [nbuf](int gp) { return nbuf == 3 ? gp / 3 : gp >> (nbuf >> 1); };
    const uint32_t ring_s = smem_u32(ring);
    const uint64_t desc_ring = sdesc_k_sw128(ring_s);  // slot r's hi rows: + (r * sbytes) >> 4
    bool ok = true;

    if (warp < 4) {
        setmaxnreg_dec<kRegsWg0>();
        if ((warp == 0 || (kMmaThreads == 2 && warp == 2)) && lane == 0 && (!kPair || ppos == 0)) {
            // ------------------------------------------------------------------ MMA issue (two threads)
            // stream st issues the global slices of groups st, st + 2, ... (slice gs: ring slot gs mod depth, A buffer
            // gs mod na -- both powers of two --, the slot's hi and lo tiles, the slice's partial buffer); the other
            // thread's waits overlap this one's MMAs.  The item's first slice and its partial index advance by
            // counting (a division by a runtime value costs tens of cycles on this thread's critical path).
            const int st = warp >> 1;
            int gst = st * Gs, sbase = 0, seq = 0;  // this thread's next global stage; the item's first; items done
            Item t;
            for (int item = cid; item < n_items && ok; item += NC) {
                if (!load_item<kPair>(tiles, item, mgroups, C, crank, p, t)) continue;
                const uint32_t idesc = idesc_f16_f32(kPair ? 2 * kBM : kBM, t.ncols);
                for (; gst < sbase + nsi && ok; gst += (Gs == 1 || (gst & 1)) ? (kMmaThreads - 1) * Gs + 1 : 1) {
                    const int ks = gst - sbase;  // the stage within the item
                    const int j = gst % nst;
                    const uint32_t aph = (uint32_t)(gst / nst) & 1u;  // parity of stage slot j's barriers for it
                    // the stage's partial: one per 128 values of K (two-level), else the item's partial of this thread
                    const int gp = seq * pitem + (p.two_level ? ks / Gs : (pitem == 2 ? (ks & 1) : 0));
                    const int b = buf_of(gp);
                    const bool first = p.two_level ? ks % Gs == 0 : ks < kMmaThreads;
                    const bool last = p.two_level ? ks % Gs == Gs - 1 : ks + kMmaThreads >= nsi;
                    // A decoded and the stage's B tiles landed; a stage that starts a partial in a buffer used before
                    // also needs the promoters to have taken the previous partial there (partial gp - nbuf: phase
                    // gp / nbuf - 1 of its pempty).  The waits overlap.  (Pair form: both CTAs' converters arrive on
                    // the leader's afull and both CTAs' B bytes land on its sfull.)
                    const bool reuse = first && gp >= nbuf;
                    const uint32_t eph = reuse ? (uint32_t)(use_of(gp) - 1) & 1u : aph;
                    // the stage's operands, before the wait (its round trip hides this arithmetic)
                    const uint32_t d = tmem + part_base + (uint32_t)(b * bufw);
                    const int g0 = gst * S;  // the stage's first global slice
                    uint64_t bh[S], bl[S];
                    uint32_t a[S];
#pragma unroll
                    for (int q = 0; q < S; ++q) {
                        bh[q] = desc_ring + (uint64_t)((((g0 + q) % depth) * sbytes) >> 4);
                        bl[q] = bh[q] + (uint64_t)(t.lo_rows * (128 >> 4));
                        a[q] = tmem + (uint32_t)((g0 + q) % na) * kACols;
                    }
                    const uint32_t acc = first ? 0u : 1u;
                    if (!mbar_wait3(&afull[j], aph, &sfull[j], aph, reuse ? &pempty[b] : &afull[j], eph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // a stacked tile: one MMA of 2N columns a step (pair form: the leader's slot holds the N hi rows
                    // and the peer's the N lo rows at the same offset, i.e. columns [0, N) and [N, 2N))
#pragma unroll
                    for (int q = 0; q < S; ++q) {
                        if (t.stacked) mma_slice4<C>(d, a[q], bh[q], idesc, q == 0 ? acc : 1u);
                        else mma_slice8<C>(d, a[q], bh[q], bl[q], idesc, q == 0 ? acc : 1u);
                    }
                    if constexpr (kPair) {
                        mma_commit_pair_mc(&sempty[j], pmask);  // the stage's slots free in both CTAs
                        if (last) mma_commit_pair_mc(&pfull[b], pmask);
                    } else {
                        mma_commit(&sempty[j]);
                        if (last) mma_commit(&pfull[b]);
                    }
                }
                sbase += nsi;
                ++seq;
            }
            // completes once every MMA issued above has completed (abort path included)
            if constexpr (kPair) mma_commit_pair_mc(accf, pmask);
            else mma_commit(accf);
        } else if (warp == 1) {
            // ------------------------------------------------------------------ producer (one warp)
            // lane 0 waits for the slot and posts its byte counts and the weight copy; lanes 1 and 2 issue the B copies
            if (lane < 2 * kNumMaps) {
                const CUtensorMap* m = lane < kNumMaps ? &maps.hi[lane] : &maps.lo[lane - kNumMaps];
                asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
            }
            int gs = 0;
            const uint32_t sfull_leader = kPair ? cluster_addr(&sfull[0], leader) : 0u;
            Item t;
            for (int item = cid; item < n_items && ok; item += NC) {
                if (!load_item<kPair>(tiles, item, mgroups, C, crank, p, t)) continue;
                const uint8_t* wblocks =
                    p.wp + ((int64_t)t.e * (p.a_rows / kBM) + t.m0 / kBM) * nk * (int64_t)kWBlock;
                // the B bytes that land in THIS CTA's slot per slice: both parts of N rows (single form); N rows of
                // one part (pair form, stacked) or N/2 rows of both parts (pair form)
                const uint32_t b_bytes = kPair ? (uint32_t)t.N * 128u : 2u * (uint32_t)t.N * 128u;
                const CUtensorMap* const mhi = &maps.hi[t.map];
                const CUtensorMap* const mlo = &maps.lo[t.map];
                for (int kt = 0; kt < nk; ++kt, ++gs) {
                    const int gst = gs / S, j = gst % nst, r = gs % depth;
                    if (gs % S == 0) {
                        // a new stage: its slots free (the MMA commits of stage gst - nst and its converters), then
                        // its barriers armed for all S slices' bytes
                        bool go = true;
                        if (lane == 0) {
                            bool free_ = true;
                            if (gst >= nst) {
                                const uint32_t eph = (uint32_t)(gst / nst - 1) & 1u;
                                if constexpr (kPair) free_ = mbar_wait_cl(&sempty[j], eph, abort_flag);
                                else free_ = mbar_wait(&sempty[j], eph, abort_flag);
                            }
                            if (!free_) go = false;
                            else {
                                mbar_arrive_expect_tx(&wfull[j], (uint32_t)(S * kWBlock));
                                // pair form: the leader's sfull counts both CTAs' B bytes; the peer arms none
                                if (!kPair) mbar_arrive_expect_tx(&sfull[j], (uint32_t)S * b_bytes);
                                else if (ppos == 0) mbar_arrive_expect_tx(&sfull[j], 2u * (uint32_t)S * b_bytes);
                            }
                        }
                        if (!__shfl_sync(0xffffffffu, go, 0)) {
                            ok = false;
                            break;
                        }
                    }
                    const uint32_t slot = ring_s + (uint32_t)(r * sbytes);
                    // lane 0 the weights (on their own barrier: the converters need nothing else), lanes 1 and 2 the
                    // hi and lo boxes
                    if (lane == 0)
                        bulk_load(slot + (uint32_t)(kPair ? kPairWOfs : 2 * t.lo_rows * 128),
                                  wblocks + (int64_t)kt * kWBlock, kWBlock, &wfull[j]);
                    const int part = lane - 1;
                    if (part == 0 || part == 1) {
                        const CUtensorMap* map = part ? mlo : mhi;
                        if constexpr (kPair) {
                            // this CTA's rows: stacked -- part ppos, all N rows; else rows [ppos N/2, (ppos + 1) N/2)
                            // of both parts; the copy counts its bytes on the leader's sfull
                            const bool mine = t.stacked ? part == (int)ppos : true;
                            const int y = t.row0 + (t.stacked ? 0 : (int)ppos * (t.N / 2));
                            const uint32_t dst = slot + (uint32_t)((t.stacked ? 0 : part) * kPairRows * 128);
                            if (mine) tma_load_2d_pair(dst, map, kt * kBK, y, sfull_leader + (uint32_t)(j * 8));
                        } else {
                            const uint32_t dst = slot + (uint32_t)(part ? t.lo_rows * 128 : 0);
                            tma_load_2d(dst, map, kt * kBK, t.row0, &sfull[j]);
                        }
                    }
                }
            }
            if (lane == 0) *total_slot = gs / S;
            // no copy may still be writing shared memory when the CTA exits (on the abort path nobody has waited
            // for the last stages): wait, bounded, for the last `nst` stages issued
            // (pair form: the peer's B copies are counted on the leader's sfull, which the leader waits for here before
            // the final cluster barrier that the peer cannot pass without it)
            if (lane == 0) {
                const int stages = gs / S;
                for (int k = max(0, stages - nst); k < stages; ++k) {
                    mbar_wait(&wfull[k % nst], (uint32_t)(k / nst) & 1u, nullptr);
                    if (!kPair || ppos == 0) mbar_wait(&sfull[k % nst], (uint32_t)(k / nst) & 1u, nullptr);
                }
            }
        }
        __syncwarp();
    } else if (warp < 16) {
        setmaxnreg_inc<kRegsProm>();
        // ------------------------------------------------------------------ promoters (384 threads)
        // this thread owns TMEM lane 32*q + lane (weight row mrow of the item's slice) and the 32-column chunks
        // cg + 3 i of the tile (16-column chunks for a stacked tile); three warps a sub-partition hide each other's
        // load latency
        const int q = warp & 3;
        const int cg = (warp - 4) >> 2;  // promoter warpgroup 0..2
        const int mrow = 32 * q + lane;
        constexpr int kChunks = kMaxBN / 96;  // most 32-column chunks of a thread
        // pair form: a promoter warp arrives once on the leader's pempty when all its lanes have loaded the partial
        const uint32_t pempty0 = kPair ? cluster_addr(&pempty[0], leader) : 0u;
        int b = 0;
        uint32_t bph = 0;
        Item t;
        for (int item = cid; item < n_items && ok; item += NC) {
            if (!load_item<kPair>(tiles, item, mgroups, C, crank, p, t)) continue;
            const int N = t.N;
            const bool stacked = t.stacked;
            const int mine = (N / 32 - cg + 2) / 3;                         // whole 32-column chunks of this thread
            const bool half = !stacked && (N & 16) && cg == (N / 32) % 3;  // a last 16-column chunk is this thread's
            float acc[kChunks][32];
#pragma unroll
            for (int i = 0; i < kChunks; ++i)
#pragma unroll
                for (int k = 0; k < 32; ++k) acc[i][k] = 0.0f;
            for (int g = 0; g < pitem && ok; ++g) {
                bool got;
                if constexpr (kPair) got = mbar_wait_cl(&pfull[b], bph, abort_flag);
                else got = mbar_wait(&pfull[b], bph, abort_flag);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + part_base + (uint32_t)(b * bufw);
                uint32_t v[32];
                if (stacked) {
                    // 16-column chunks cg + 3 i: hi columns c.. and lo columns N + c.., added in turn
                    uint32_t(&h)[16] = *reinterpret_cast<uint32_t(*)[16]>(&v[0]);
                    uint32_t(&l)[16] = *reinterpret_cast<uint32_t(*)[16]>(&v[16]);
#pragma unroll
                    for (int i = 0; i < kMaxStackN / 48; ++i) {
                        const int c = 16 * (cg + 3 * i);
                        if (c < N) {
                            tmem_ld_32x32b_x16(base + (uint32_t)c, h);
                            tmem_ld_32x32b_x16(base + (uint32_t)(N + c), l);
                            tmem_ld_wait();
                            float* a = &acc[i >> 1][16 * (i & 1)];
#pragma unroll
                            for (int k = 0; k < 16; k += 2) {
                                add2(a[k], a[k + 1], h[k], h[k + 1]);
                                add2(a[k], a[k + 1], l[k], l[k + 1]);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < kChunks; ++i) {
                        if (i < mine) {
                            tmem_ld_32x32b_x32(base + (uint32_t)(32 * (cg + 3 * i)), v);
                            tmem_ld_wait();
#pragma unroll
                            for (int k = 0; k < 32; k += 2) add2(acc[i][k], acc[i][k + 1], v[k], v[k + 1]);
                        }
                    }
                    if (half) {  // the tile's last 16 columns (N = 32 m + 16) into the first half of chunk `mine`
                        uint32_t(&h)[16] = *reinterpret_cast<uint32_t(*)[16]>(&v[0]);
                        tmem_ld_32x32b_x16(base + (uint32_t)(N - 16), h);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < kChunks; ++i)
                            if (i == mine) {
#pragma unroll
                                for (int k = 0; k < 16; k += 2) add2(acc[i][k], acc[i][k + 1], h[k], h[k + 1]);
                            }
                    }
                }
                tc_fence_before();
                if constexpr (kPair) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cl(pempty0 + (uint32_t)(b * sizeof(uint64_t)));
                } else {
                    mbar_arrive(&pempty[b]);
                }
                if (++b == nbuf) {
                    b = 0;
                    bph ^= 1u;
                }
            }
            // the item's outputs; column col of chunk slot (i, k), as the partials were added
            auto column = [&](int i, int k) {
                // a stacked tile's 16-column chunk j = cg + 3 i' sits at acc[i' / 2][16 (i' % 2) ..]
                return stacked ? 16 * (cg + 3 * (2 * i + (k >> 4))) + (k & 15)
                               : ((i < mine || !half) ? 32 * (cg + 3 * i) + k : (N - 16) + k);
            };
            auto owned = [&](int i, int k) {
                return stacked ? (2 * i + (k >> 4)) < kMaxStackN / 48 : (i < mine || (half && i == mine && k < 16));
            };
            if (p.hc == nullptr && p.out_h != nullptr) {
                if (!ok) break;
                // ------------------------------------------------------------ epilogue: fp16 rows out (round to
                // nearest; a value beyond the fp16 range becomes +-inf)
                uint16_t* outcol = p.out_h + (t.m0 + mrow);
#pragma unroll
                for (int i = 0; i < kChunks; ++i) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int col = column(i, k);
                        if (owned(i, k) && col < t.rows)
                            outcol[(int64_t)(t.row0 + col) * p.a_rows] = __half_as_ushort(__float2half_rn(acc[i][k]));
                    }
                }
            } else if (p.hc == nullptr) {
                if (!ok) break;
                // ------------------------------------------------------------ epilogue: fp32 rows out
                float* outcol = p.out + (t.m0 + mrow);
#pragma unroll
                for (int i = 0; i < kChunks; ++i) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int col = column(i, k);
                        if (owned(i, k) && col < t.rows) outcol[(int64_t)(t.row0 + col) * p.a_rows] = acc[i][k];
                    }
                }
            } else {
                // ------------------------------------------------------------ epilogue: SwiGLU + requantisation
                // the weights are packed interleaved: lane l < 16 holds gate output j, lane l + 16 the up output of
                // the same j, and the 16 outputs of a warp are one operand-form group.  h = silu(g) * u and the q8
                // rule with the scale exactly as in the SwiGLU step (IEEE amax / 127); h and the codes use a
                // reciprocal instead of a division (a code can differ from the SwiGLU step's only next to a .5
                // tie).  The 32-value block of h spans warps q and q ^ 1.
                if (!bar_red_and(1 + cg, 128, ok)) {  // every thread of the warpgroup takes the same way out
                    ok = false;
                    break;
                }
                const int Fh = p.a_rows >> 1;
                const int jl = lane & 15;
                const bool gate = lane < 16;
                const int j = (t.m0 >> 1) + 16 * q + jl;
                const int pos = jl < 8 ? 2 * jl : 2 * (jl - 8) + 1;  // operand-form position within the group
                int8_t* const hc0 = p.hc + (int64_t)t.row0 * Fh + j;
                uint16_t* const hi0 = p.hop + (int64_t)t.row0 * Fh + (j - jl) + pos;
                uint16_t* const lo0 = hi0 + p.b_rows * Fh;
                uint16_t* const hs0 = p.hs + (int64_t)t.row0 * (Fh / 32) + (j >> 5);
#pragma unroll
                for (int i = 0; i < kChunks; ++i) {  // a chunk at a time: fewer values live at once
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int col = column(i, k);
                        if (owned(i, k) && col < N) {  // the same in every lane of the warp
                            const float g = acc[i][k];
                            const float u = __shfl_down_sync(0xffffffffu, g, 16);
                            const float h = gate ? g * u * __frcp_rn(1.0f + __expf(-g)) : 0.0f;
                            acc[i][k] = h;
                            // |h| compares as its bit pattern; the up lanes give 0
                            const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h)));
                            if (lane == 0) scratch[col * 4 + q] = __uint_as_float(m);
                        }
                    }
                    bar_sync(1 + cg, 128);
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int col = column(i, k);
                        if (owned(i, k) && col < t.rows) {
                            const float amax = fmaxf(scratch[col * 4 + q], scratch[col * 4 + (q ^ 1)]);
                            const __half dh = __float2half_rn(__fdiv_rn(amax, 127.0f));
                            const float d = __half2float(dh);
                            const int off = col * Fh;
                            if (gate) {
                                float qf = 0.0f;
                                if (d != 0.0f) qf = fminf(fmaxf(roundf(acc[i][k] * __frcp_rn(d)), -127.0f), 127.0f);
                                hc0[off] = (int8_t)(int)qf;
                                const __half qh = __float2half_rn(qf);
                                const __half hi = __hmul(qh, dh);
                                hi0[off] = __half_as_ushort(hi);
                                lo0[off] = __half_as_ushort(__hfma(qh, dh, __hneg(hi)));
                            }
                            if (lane == 0 && (q & 1) == 0) hs0[col * (Fh / 32)] = __half_as_ushort(dh);
                        }
                    }
                    bar_sync(1 + cg, 128);  // the scratch is reused by the next chunk
                }
            }
        }
    } else {
        setmaxnreg_dec<kRegsConv>();
        // ------------------------------------------------------------------ converters (128 threads)
        // thread = weight row ct = TMEM lane of its warp: 64 weights a slice into the 32 columns of A buffer ab
        const int ct = threadIdx.x - 512;
        const uint32_t lane_base = (uint32_t)(ct & ~31) << 16;
        // pair form: a converter warp arrives once on the leader's `ready` when all its lanes' stores are done
        const uint32_t ready0 = kPair ? cluster_addr(&afull[0], leader) : 0u;
        int gs = 0;          // the slice's global index
        bool ready = false;  // the stage's copies are known to have landed (tested while the last stage was stored)
        bool afree = false;  // pair form: its A buffers are known to be free (tested likewise)
        Item t;
        for (int item = cid; item < n_items && ok; item += NC) {
            if (!load_item<kPair>(tiles, item, mgroups, C, crank, p, t)) continue;
            const int wofs = kPair ? kPairWOfs : 2 * t.lo_rows * 128;  // the packed weight block within a slot
            for (int kt = 0; kt < nk && ok; ++kt, ++gs) {
                const int gst = gs / S, j = gst % nst, r = gs % depth;
                if (gs % S == 0) {
                    // a new stage: all its weight blocks landed
                    if (!ready && !mbar_wait(&wfull[j], (uint32_t)(gst / nst) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if constexpr (kPair) {
                        // the stage's A buffers were last read by stage gst - na / S: released by its MMAs' commit
                        const int pg = gst - na / S;
                        if (!afree && pg >= 0 && !mbar_wait(&sempty[pg % nst], (uint32_t)(pg / nst) & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                }
                const int ab = gs % na;
                const uint8_t* wb = ring + r * sbytes + wofs;
                const uint4 codes = *reinterpret_cast<const uint4*>(wb + ct * 16);
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(wb + 2048 + ct * 4);  // the two blocks' scales
                const uint32_t d_lo = __byte_perm(sc, 0u, 0x1010), d_hi = __byte_perm(sc, 0u, 0x3232);
                uint32_t col[16];  // one 32-value block at a time
                decode_weights16(codes.x, d_lo, col);
                decode_weights16(codes.y, d_lo, col + 8);
                tmem_st_32x32b_x16(tmem + lane_base + (uint32_t)ab * kACols, col);
                decode_weights16(codes.z, d_hi, col);
                decode_weights16(codes.w, d_hi, col + 8);
                tmem_st_32x32b_x16(tmem + lane_base + (uint32_t)ab * kACols + 16u, col);
                if (gs % S == S - 1) {
                    // the stage's last slice: test the next stage's barrier while the stores complete (a stage whose
                    // weights have landed then costs no wait round trip), then signal the stage
                    ready = mbar_test(smem_u32(&wfull[(gst + 1) % nst]), (uint32_t)((gst + 1) / nst) & 1u);
                    if constexpr (kPair) {
                        const int pn = gst + 1 - na / S;  // the next stage's A buffers' previous stage
                        afree = pn < 0 || mbar_test(smem_u32(&sempty[pn % nst]), (uint32_t)(pn / nst) & 1u);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    if constexpr (kPair) {
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive_cl(ready0 + (uint32_t)(j * sizeof(uint64_t)));
                            mbar_arrive(&sempty[j]);
                        }
                    } else {
                        mbar_arrive(&afull[j]);
                        mbar_arrive(&sempty[j]);
                    }
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
        // every MMA has completed before the tensor memory is released (pair form: the leader's final commits arrive
        // in both CTAs of the pair)
        if constexpr (kPair) mbar_wait_cl(accf, 0, nullptr);
        else mbar_wait(accf, 0, nullptr);
        if (kPair && lane == 0) {
            // every MMA commit that targets this CTA's slot barriers has arrived (each slot's last phase completes
            // only after all of them): nothing arrives on this CTA's barriers after it leaves
            const int total = *total_slot;  // stages
            for (int k = max(0, total - nst); k < total; ++k) {
                bool done;
                if constexpr (kPair) done = mbar_wait_cl(&sempty[k % nst], (uint32_t)(k / nst) & 1u, abort_flag);
                else done = mbar_wait(&sempty[k % nst], (uint32_t)(k / nst) & 1u, abort_flag);
                if (!done) break;
            }
        }
        __syncwarp();
        tc_fence_after();
        if constexpr (kPair) tmem_dealloc_pair(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
    // no CTA leaves while another may still copy into its shared memory, arrive on its barriers or (pair form) read
    // its tensor memory
    if (kPair) cluster_sync();
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

// 2D tensor [rows][cols] of `esize`-byte elements (row stride cols * esize), box box_x x box_y elements
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint32_t esize, uint64_t cols,
              uint64_t rows, uint32_t box_x, uint32_t box_y, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};
    const cuuint32_t box[2] = {box_x, box_y};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per-device, once: the dynamic shared-memory attribute of both forms, and the resident clusters of each form and
// cluster size
struct DeviceState {
    bool attr = false;
    int resident[2][5] = {};
};
DeviceState g_dev[64];
std::mutex g_dev_mu;

template <bool kPair>
cudaError_t launch_form(const ExpertsGemmArgs& a, int64_t max_tiles, int dev, cudaStream_t s) {
    GemmMaps maps;
    const uint16_t* lo = a.bop + a.b_rows * (int64_t)a.K;
    const int step = kPair ? kPairBox : kRowBox;
    for (int m = 0; m < kNumMaps; ++m) {
        const uint32_t box = (uint32_t)(step * (m + 1));
        if (!make_map(&maps.hi[m], a.bop, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)a.K, (uint64_t)a.b_rows, kBK,
                      box, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&maps.lo[m], lo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)a.K, (uint64_t)a.b_rows, kBK,
                      box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const int mt = a.a_rows / kBM;
    ExpertsGemmArgs args = a;
    // the pair form is a cluster of one CTA pair; the single form runs without clusters
    args.cluster = kPair ? 2 : 1;
    args.max_tiles = (int)max_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)args.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent: as many clusters as fit on the GPU at once (each CTA takes a whole SM), at most one per item
    const int64_t items = max_tiles * (mt / args.cluster);
    cfg.gridDim = dim3((unsigned)(args.cluster * 512));
    int resident = 0;
    {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        resident = g_dev[dev].resident[kPair][args.cluster];
    }
    if (resident <= 0) {
        cudaError_t err = cudaOccupancyMaxActiveClusters(&resident, experts_gemm_kernel<kPair>, &cfg);
        if (err != cudaSuccess || resident <= 0) {
            cudaGetLastError();
            return err != cudaSuccess ? err : cudaErrorInvalidConfiguration;
        }
        std::lock_guard<std::mutex> lock(g_dev_mu);
        g_dev[dev].resident[kPair][args.cluster] = resident;
    }
    const int64_t nclusters = items < resident ? items : resident;
    cfg.gridDim = dim3((unsigned)(nclusters * args.cluster));
    const cudaError_t err = cudaLaunchKernelEx(&cfg, experts_gemm_kernel<kPair>, args, maps);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_experts_gemm(const ExpertsGemmArgs& a, int64_t max_tiles, cudaStream_t s) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (!g_dev[dev].attr) {
            err = cudaFuncSetAttribute(experts_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
            if (err == cudaSuccess)
                err = cudaFuncSetAttribute(experts_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
            if (err != cudaSuccess) return err;
            g_dev[dev].attr = true;
        }
    }
    if (max_tiles <= 0) return cudaSuccess;
    // the CTA-pair form: an even number of 128-row weight slices (each pair takes 256 rows) and whole stages of two
    // 64-wide K slices
    if ((a.a_rows / kBM) % 2 == 0 && (a.K / kBK) % 2 == 0) return launch_form<true>(a, max_tiles, dev, s);
    return launch_form<false>(a, max_tiles, dev, s);
}

}  // namespace smoe
