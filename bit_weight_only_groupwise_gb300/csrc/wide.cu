// Wide-T route: a persistent, stream-K tcgen05 (5th-generation tensor core)
// dequant-GEMM.
//
// From a few dozen token columns up the operation is a dense contraction and
// belongs on the tensor cores; prefill widths are compute-bound ("ninfer-3080
// docs/performance.md", token tile section: the token tile width sets how
// often the weights are re-streamed, and the per-group rescale and the operand
// assembly are the costs beside the MMAs).  An output tile is 128 weight rows
// by BN = 32, 64, 128 or 256 tokens:
//
//   D[128 rows x BN tokens] = sum over 64-column groups g of s[:, g] * P_g,
//   P_g = A_g (exact integer codes as bf16, 128 x 64) . B_g (X tile, BN x 64)^T
//
// A 256-token tile runs as two 128-token halves over the same decoded A_g, so
// each decoded weight feeds twice the tensor work (the page's lesson: wider
// token tiles remove weight passes, they are not cached away).
//
// Work split (stream-K): the (tile, group) units of all parents of the launch
// are numbered tile-major and cut into one contiguous range per CTA, one CTA
// per SM, so every SM gets the same number of groups whatever the tile count.
// A tile whose groups span several CTAs is finished by the CTA that completes
// it last: the others leave their fp32 partial sums in the workspace and
// count in, and the last one adds them in ascending CTA order (a fixed order,
// so results are bitwise repeatable) and writes Y; the tile's first segment,
// usually the last to finish, keeps its own partial in registers when it
// finds the others counted in.  No CTA waits for another.
//
// Warp roles (16 warps; every single-issuer role is a converged warp whose
// elected lane issues, and every wait is taken by the whole warp):
//   warp 0        weight producer: 1-D bulk copies of pairs of packed units
//                 into a shared-memory ring (the only role that runs before
//                 the programmatic wait on the previous kernel);
//   warps 1, 3    MMA issuers (alternate steps; warp 1 also owns tensor
//                 memory);
//   warp 2        activation producer: 2-D TMA loads of 128B-swizzled X tiles;
//   warps 4..7    dequant: one thread per weight row decodes its 64 codes of
//                 a group (magic-number bf16 decode, exact) into tensor memory
//                 as the A operand (tcgen05.st); the row's scale goes to the
//                 epilogue through a shared-memory ring (the 32- and
//                 64-token tiles: warps 4..11, two groups taking alternate
//                 unit pairs);
//   warps 8..15   epilogue: read P from tensor memory (tcgen05.ld), multiply
//                 by the row's fp16 scale and accumulate in fp32 registers
//                 (packed f32x2 FMA); write Y, or a partial sum and its count
//                 (the 32- and 64-token tiles: warps 12..15, 32 or 64 columns
//                 each).
// A step is one MMA width (BH = 128, 64 or 32 tokens) of one group: step
// j = unit * H + h.
// Tensor memory: NA A stages of 32 columns (4; 8 for the 32- and 64-token
// tiles) and NP P buffers of BH columns in the rest (step j uses j mod NP, so
// the epilogue has NP - 1 steps of MMA time to drain a buffer).  Barriers:
//   xa_full[s]   A_g stored (the 4 dequant warps of a group) and X_g landed
//                (TMA bytes)
//   xa_empty[s]  the MMAs of both halves of group g completed (one commit
//                per step): X stage s and A stage g mod NA are free
//   pfull[b]     the MMAs of the step in P buffer b completed
//   pfree[b]     every epilogue warp has read P buffer b
// Every mbarrier wait is bounded; a wait that runs out sets the device status
// to timeout and the CTA winds down (after a bounded pause that lets copies
// and MMAs already issued land before tensor memory is released).
#include <atomic>

#include <cuda.h>

#include "qgemm_internal.cuh"

namespace qg {

namespace wide {

constexpr int BM = 128;                   // weight rows per tile (tensor-memory lanes)
constexpr int DQ_WARPS = 4;               // dequant warps of a unit: one per tensor-memory lane quarter
constexpr int EPI_WARPS = 8;              // at most: two epilogue warps per lane quarter (column halves)
constexpr int DQ0 = 4;                    // the first dequant warp (warps 0..3: producers, MMA issuers)
constexpr int THREADS = 16 * 32;
constexpr int P_COL = 0;                  // P buffers from column 0, then the A stages
constexpr int TMEM_COLS = 512;

// BH: tokens per MMA (32, 64 or 128); H: MMAs ("halves") per tile, so BN = BH H
// tokens; F8: a parent of the launch holds FP8 or NVFP4 codes (larger units,
// so fewer weight stages fit).  Tensor memory holds the A stages and as many
// P buffers of BH columns as fit beside them (at most 6): 3 of 128 columns
// beside 4 A stages, 4 of 64 or 6 of 32 beside 8.  The dequant limited the
// 32- and 64-token tiles (a unit's MMAs are short), so they get two dequant
// groups, twice the A stages, half the activation stages (their X tiles are
// at most half as large) and twice the weight stages, and run four unit pairs
// ahead of the MMAs instead of two.
template <int BH_, int H, bool F8>
struct Geo {
    static constexpr int BH = BH_;
    // Warps 4 .. 15: DQG groups of four dequant warps (a group decodes every
    // DQG-th unit pair) and EPI_N epilogue warps.  The 32- and 64-token tiles
    // run two groups beside four epilogue warps that read all 32 or 64
    // columns of a step; the others one group beside eight.
    static constexpr int DQG = BH <= 64 ? 2 : 1;
    static constexpr int EPI_N = 12 - 4 * DQG;
    static constexpr int EPI_0 = DQ0 + 4 * DQG;
    static constexpr int NA = BH <= 64 ? 8 : 4;           // A stages (unit u uses u mod NA)
    // P buffers (step j uses j mod NP): as many as fit, at most 6 (8 or 12 on
    // the 32-token tile measured no faster; the scale ring below bounds NP)
    static constexpr int NP = (TMEM_COLS - 32 * NA) / BH < 6 ? (TMEM_COLS - 32 * NA) / BH : 6;
    static constexpr int A_COL = P_COL + NP * BH;         // A stages: 32 columns each
    static constexpr int EW = BH / (EPI_N / 4);           // P columns per epilogue warp
    static constexpr int NJ = EW / 2;                     // column pairs per epilogue thread and MMA
    static constexpr int HALF_BYTES = BH * GROUP * 2;     // one MMA's X tile of one group
    static constexpr int BN = H * BH;
    static constexpr int XST = H * HALF_BYTES;           // X stage: BN tokens x 64 columns
    static constexpr int X_REGION = BH <= 64 ? 64 * 1024 : 128 * 1024;  // activation stages
    static constexpr int NS = X_REGION / XST;             // 8 (64- and 128-token tiles) or 4 stages
    static constexpr int WSLOT = 2 * (F8 ? UNIT8 : UNIT5);
    static constexpr int NWP = BH <= 64 ? (F8 ? 8 : 12) : (F8 ? 4 : 6);  // weight stages (pairs of units)
    static constexpr int X_OFF = 0;                       // 1024-aligned (128B swizzle atoms)
    static constexpr int W_OFF = X_REGION;
    static constexpr int BAR_OFF = W_OFF + NWP * WSLOT;
    static constexpr int NBAR = 2 * NWP + 2 * NS + 2 * NP;
    // Scales in flight: the dequant writes unit u's scale while decoding it,
    // before it waits for the MMAs of unit u - NA; a group's previous pair
    // waited for those of its own units, which came after the epilogue had
    // read NP steps earlier -- so a group writes up to NA + NP + 2 units past
    // the epilogue, and DQG groups (alternate pairs) 2 (DQG - 1) more.
    static constexpr int SC_RING = DQG > 1 ? 32 : 16;
    static constexpr int SC_OFF = BAR_OFF + NBAR * 8;     // float [SC_RING][BM]
    static constexpr int MISC_OFF = SC_OFF + SC_RING * BM * 4;
    static constexpr int BYTES = MISC_OFF + 16 + 1024;    // + slack to align the base
    static_assert(NS >= NA, "A stages are recycled through the X stage barriers");
    static_assert(NA % 2 == 0, "a unit pair starting at an even unit owns two adjacent A stages");
    static_assert(BYTES <= 227 * 1024, "shared memory budget");
    static_assert(A_COL + 32 * NA <= TMEM_COLS, "tensor memory budget");
    static_assert(SC_RING >= NA + NP + 2 * DQG, "scale ring shorter than the dequant lead");
    static_assert(BH == 32 || BH == 64 || BH == 128, "MMA widths of the route");
    static_assert(EPI_N % 4 == 0 && EPI_N <= EPI_WARPS, "whole lane quarters of epilogue warps");
    static_assert(DQG == 1 || NWP % 2 == 0, "each group's weight stages reuse its own slots");
};

}  // namespace wide

struct WideArgs {
    WideParent p[MAX_PARENTS];
    int nparents;
    int T, K, G;
    int ntt;              // token tiles of BN tokens
    int ntiles;           // output tiles of all parents (parent i owns p[i].cta_begin ...)
    long long units;      // ntiles * G
    float *part;          // partial sums of split tiles: [grid][2][BN / 4][BM] float4
    unsigned int *status;
};

// An output tile: its parent, 128-row block and token tile.
struct WideTile {
    const WideParent *P;
    int local, blk, tt;
};

__device__ __forceinline__ WideTile wide_tile(const WideArgs &a, int tile) {
    int pi = 0;
#pragma unroll
    for (int i = 1; i < MAX_PARENTS; ++i)
        if (i < a.nparents && tile >= a.p[i].cta_begin) pi = i;
    const int local = tile - a.p[pi].cta_begin;
    return {&a.p[pi], local, local / a.ntt, local % a.ntt};
}

// Stream-K ranges: CTA c owns units [lo(c), lo(c + 1)), lo(c) = floor(c U / grid);
// every CTA owns at least one unit when grid <= U.
__device__ __forceinline__ long long range_lo(long long U, int grid, int c) { return (long long)c * U / grid; }
// the CTA whose range holds unit u
__device__ __forceinline__ int range_cta(long long U, int grid, long long u) {
    return (int)(((u + 1) * grid - 1) / U);
}

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// One 64-column group of one step: D(tmem) = A(tmem) . B(smem)^T as four
// K = 16 MMAs (bf16 inputs, fp32 accumulate; the first overwrites D), then
// commits of their completion to two mbarriers.  One elected lane of a
// converged warp issues all six instructions under one predicate, with the
// operand addresses precomputed: a warp issuing this way keeps the tensor pipe
// busy (one M128 N128 K16 MMA per 64 cycles measured), where computing each
// descriptor and electing per instruction took about 100 cycles per MMA.
// a: A's tensor-memory address (K advances 8 columns per MMA); bd: B's
// shared-memory descriptor (K advances 32 bytes, 2 in its address field).
__device__ __forceinline__ void tc_mma_group(uint32_t d, uint32_t a, uint64_t bd, uint32_t idesc, uint64_t *bar0,
                                             uint64_t *bar1) {
    asm volatile(
        "{.reg .pred e, z; elect.sync _|e, 0xffffffff; setp.ne.u32 z, %3, %3;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, z;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %5, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %7, %3, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %9, %3, 1;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];}"
        ::"r"(d), "r"(a), "l"(bd), "r"(idesc), "r"(a + 8), "l"(bd + 2), "r"(a + 16), "l"(bd + 4), "r"(a + 24),
          "l"(bd + 6), "r"(smem_u32(bar0)), "r"(smem_u32(bar1)) : "memory");
}

#define QG_R32(a) a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], a[8], a[9], a[10], a[11], a[12], a[13], a[14], \
                  a[15], a[16], a[17], a[18], a[19], a[20], a[21], a[22], a[23], a[24], a[25], a[26], a[27], a[28], \
                  a[29], a[30], a[31]

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 64 consecutive columns in one load (columns 0..31 into r0, 32..63 into r1):
// one tensor-memory instruction where two 32-column loads took two.
__device__ __forceinline__ void tc_ld64(uint32_t taddr, uint32_t (&r0)[32], uint32_t (&r1)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]), "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]), "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r0[16]), "=r"(r0[17]), "=r"(r0[18]), "=r"(r0[19]), "=r"(r0[20]), "=r"(r0[21]), "=r"(r0[22]), "=r"(r0[23]), "=r"(r0[24]), "=r"(r0[25]), "=r"(r0[26]), "=r"(r0[27]), "=r"(r0[28]), "=r"(r0[29]), "=r"(r0[30]), "=r"(r0[31]),
          "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15]), "=r"(r1[16]), "=r"(r1[17]), "=r"(r1[18]), "=r"(r1[19]), "=r"(r1[20]), "=r"(r1[21]), "=r"(r1[22]), "=r"(r1[23]), "=r"(r1[24]), "=r"(r1[25]), "=r"(r1[26]), "=r"(r1[27]), "=r"(r1[28]), "=r"(r1[29]), "=r"(r1[30]), "=r"(r1[31])
        : "r"(taddr));
}

// 64 consecutive columns in one store (r0 to columns 0..31, r1 to 32..63).
__device__ __forceinline__ void tc_st64(uint32_t taddr, const uint32_t (&r0)[32], const uint32_t (&r1)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};"
        :
        : "r"(taddr), "r"(r0[0]), "r"(r0[1]), "r"(r0[2]), "r"(r0[3]), "r"(r0[4]), "r"(r0[5]), "r"(r0[6]), "r"(r0[7]), "r"(r0[8]), "r"(r0[9]), "r"(r0[10]), "r"(r0[11]), "r"(r0[12]), "r"(r0[13]), "r"(r0[14]), "r"(r0[15]), "r"(r0[16]), "r"(r0[17]), "r"(r0[18]), "r"(r0[19]), "r"(r0[20]), "r"(r0[21]), "r"(r0[22]), "r"(r0[23]), "r"(r0[24]), "r"(r0[25]), "r"(r0[26]), "r"(r0[27]), "r"(r0[28]), "r"(r0[29]), "r"(r0[30]), "r"(r0[31]),
          "r"(r1[0]), "r"(r1[1]), "r"(r1[2]), "r"(r1[3]), "r"(r1[4]), "r"(r1[5]), "r"(r1[6]), "r"(r1[7]), "r"(r1[8]), "r"(r1[9]), "r"(r1[10]), "r"(r1[11]), "r"(r1[12]), "r"(r1[13]), "r"(r1[14]), "r"(r1[15]), "r"(r1[16]), "r"(r1[17]), "r"(r1[18]), "r"(r1[19]), "r"(r1[20]), "r"(r1[21]), "r"(r1[22]), "r"(r1[23]), "r"(r1[24]), "r"(r1[25]), "r"(r1[26]), "r"(r1[27]), "r"(r1[28]), "r"(r1[29]), "r"(r1[30]), "r"(r1[31])
        : "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Ties registers filled by tcgen05.ld to a point after tcgen05.wait::ld: code
// that reads them depends on this statement's outputs, so the compiler cannot
// move it above the wait.
__device__ __forceinline__ void tc_regs_ready(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                   "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]),
                   "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2-D tiled TMA load of box {64 columns, 128 rows} at (x, y) into smem.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored as
// 128-byte rows in 8-row, 1024-byte swizzle atoms (128B swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);          // start address
    d |= (uint64_t)1 << 16;                         // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;                         // descriptor version for this architecture
    d |= (uint64_t)2 << 61;                         // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}

// Register budgets per warpgroup: the epilogue keeps up to 128 fp32
// accumulators per thread, with 64 loaded P values beside them, so the
// producer, MMA and dequant warps give registers up for it.  The block
// launches with 512 threads x 128 registers (65,536); the shares below add up
// to at most that for every tile shape: 128 x (40 + 136) + 256 x 160
// (128-token tiles), 128 x (32 + 64) + 256 x 208 (256), 128 x 40 + 256 x 152
// + 128 x 160 (64: two dequant groups, four epilogue warps).
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
constexpr int REGS_AT_LAUNCH = 128;
// A warpgroup's register count from the launch's 128 to N: .dec may only
// lower the count and .inc only raise it.
template <int N>
__device__ __forceinline__ void regs_set() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg range");
    if constexpr (N < REGS_AT_LAUNCH) regs_dec<N>();
    else if constexpr (N > REGS_AT_LAUNCH) regs_inc<N>();
}
// The 128-token tile's dequant decodes a pair of units at once (more
// registers); the 256-token tile's epilogue holds twice the accumulators.
template <int BH, int H> struct Regs {
    static constexpr int WG0 = H == 2 ? 32 : 40;      // (the same for every BH <= 64)
    static constexpr int DQ = BH <= 64 ? 152 : H == 1 ? 136 : 64;
    static constexpr int EPI = BH <= 64 ? 160 : H == 1 ? 160 : 208;
    static constexpr int DQG = wide::Geo<BH, H, false>::DQG, EPI_N = wide::Geo<BH, H, false>::EPI_N;
    static_assert(128 * WG0 + 128 * DQG * DQ + 32 * EPI_N * EPI <= 512 * REGS_AT_LAUNCH, "register split");
};

// ---------------------------------------------------------------- dequant

// Weight row r of a unit in shared memory as 32 bf16x2 words in natural k
// order (word m = columns 2m, 2m + 1), and the scale of its group: the fp16
// scale, or for NVFP4 (codes times their block scales) the tensor scale ts.
template <int CODEC>
__device__ __forceinline__ float decode_row(const uint8_t *u, int r, uint32_t (&av)[32], float ts) {
    const int tile = r >> 4, i = r & 15, gi_ = i & 7, half = i >> 3;
    if constexpr (CODEC == NVFP4) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 v = *reinterpret_cast<const uint2 *>(u + tile * 512 + (4 * gi_ + c) * 16 + 8 * half);
            const uint32_t bsb = u[NIB_BYTES + tile * 64 + (4 * gi_ + c) * 2 + half];   // block c of row r
            const uint32_t bs2 = ue4m3x2_to_bf16x2(bsb | (bsb << 8));
            const uint32_t wv[2] = {v.x, v.y};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t *o = av + 8 * c + 4 * h;
                o[0] = dec16_pair<0>(wv[h], bs2); o[1] = dec16_pair<1>(wv[h], bs2);
                o[2] = dec16_pair<2>(wv[h], bs2); o[3] = dec16_pair<3>(wv[h], bs2);
            }
        }
        return ts;
    } else if constexpr (CODEC == 8) {
        // E4M3: the row's 16 codes of lane chunk c (k 16c .. 16c+15)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(u + tile * 1024 + (4 * gi_ + c) * 32 + 16 * half);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j2 = 0; j2 < 4; ++j2) {
                av[8 * c + 2 * j2] = dec8_pair<0>(wv[j2]);
                av[8 * c + 2 * j2 + 1] = dec8_pair<1>(wv[j2]);
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 v = *reinterpret_cast<const uint2 *>(u + tile * 512 + (4 * gi_ + c) * 16 + 8 * half);
            const uint32_t hw = CODEC == 5 ? *reinterpret_cast<const uint32_t *>(u + NIB_BYTES + tile * 128 + (4 * gi_ + c) * 4)
                                           : 0u;
            const uint32_t wv[2] = {v.x, v.y};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w = wv[h];
                uint32_t *o = av + 8 * c + 4 * h;
                if constexpr (CODEC == 4) {
                    o[0] = dec4_pair<0>(w); o[1] = dec4_pair<4>(w); o[2] = dec4_pair<8>(w); o[3] = dec4_pair<12>(w);
                } else {
                    // this row's words in the lane's high word: m = 2*half + h
                    const uint32_t hh = hw >> (4 * (2 * half + h));
                    o[0] = dec5_pair<0, -4>(w, hh); o[1] = dec5_pair<4, -3>(w, hh);
                    o[2] = dec5_pair<8, -2>(w, hh); o[3] = dec5_pair<12, -1>(w, hh);
                }
            }
        }
    }
    return __half2float(*reinterpret_cast<const __half *>(u + scale_off(CODEC) + tile * 32 + gi_ * 4 + half * 2));
}

// The dequant warps over one segment (units k0 .. k1 - 1 of a tile of codec
// CODEC): pairs of units per weight stage; a unit's codes go into A stage
// gi mod NA once the MMAs of unit gi - NA have freed it.  PAIR: both units of
// a stage are decoded before either is stored, so that one store wait serves
// two units (the integer codecs on the 64- and 128-token tiles, where a unit's
// MMAs are short); otherwise one unit at a time (fewer live registers: the FP8
// decode, the 256-token tile's accumulators).  ST64: a pair starting at an
// even unit is stored with one 64-column instruction (its two A stages are
// adjacent); the kernels that also decode FP8 keep two 32-column stores, which
// need fewer registers.
template <int CODEC, int NS, int NA, int NWP, int WSLOT, int A_COL, bool PAIR, bool ST64, int DQG, int SC_RING>
__device__ __forceinline__ bool dequant_segment(int k0, int k1, int &gi, int &jp, uint8_t *ws, uint64_t *w_full,
                                                uint64_t *w_empty, uint64_t *xa_full, uint64_t *xa_empty,
                                                float *sc_ring, uint32_t tmem, int q, int g, int lane, float ts,
                                                unsigned int *status) {
    using namespace wide;
    constexpr int UB = unit_bytes(CODEC);
    const int r = q * 32 + lane;
    const uint32_t tlane = (uint32_t)(q * 32) << 16;
    for (int k = k0; k < k1; k += 2, ++jp) {
        const int n = k + 1 < k1 ? 2 : 1;
        if (DQG > 1 && jp % DQG != g) {                   // another group's weight stage
            gi += n;
            continue;
        }
        const int wsl = jp % NWP;
        if (!mbar_wait_warp(&w_full[wsl], (jp / NWP) & 1, status)) return false;
        if constexpr (PAIR) {
            uint32_t av[2][32];
            sc_ring[(gi % SC_RING) * BM + r] = decode_row<CODEC>(ws + wsl * WSLOT, r, av[0], ts);
            if (n == 2) sc_ring[((gi + 1) % SC_RING) * BM + r] = decode_row<CODEC>(ws + wsl * WSLOT + UB, r, av[1], ts);
            __syncwarp();
            if (lane == 0) mbar_arrive(&w_empty[wsl]);
            // A stages of both units were last read by the MMAs of units gi - NA
            // and gi + 1 - NA
            const int h0 = gi - NA, h1 = gi + 1 - NA;
            bool ok = true;
            if (n == 2 && h0 >= 0) {
                ok = __all_sync(0xffffffffu, mbar_wait2(&xa_empty[h0 % NS], (h0 / NS) & 1, &xa_empty[h1 % NS],
                                                        (h1 / NS) & 1, status));
            } else if (h0 >= 0) {
                ok = mbar_wait_warp(&xa_empty[h0 % NS], (h0 / NS) & 1, status);
            } else if (n == 2 && h1 >= 0) {
                ok = mbar_wait_warp(&xa_empty[h1 % NS], (h1 / NS) & 1, status);
            }
            if (!ok) return false;
            tc_fence_after();
            if (ST64 && n == 2 && (gi & 1) == 0) {
                // stages gi mod NA and the next one are adjacent (NA is even)
                tc_st64(tmem + tlane + A_COL + (gi % NA) * 32, av[0], av[1]);
            } else {
                tc_st32(tmem + tlane + A_COL + (gi % NA) * 32, av[0]);
                if (n == 2) tc_st32(tmem + tlane + A_COL + ((gi + 1) % NA) * 32, av[1]);
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&xa_full[gi % NS]);
                if (n == 2) mbar_arrive(&xa_full[(gi + 1) % NS]);
            }
            gi += n;
        } else {
            for (int e = 0; e < n; ++e, ++gi) {
                uint32_t av[32];
                sc_ring[(gi % SC_RING) * BM + r] = decode_row<CODEC>(ws + wsl * WSLOT + e * UB, r, av, ts);
                if (e == n - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&w_empty[wsl]);
                }
                // A stage gi mod NA was last read by the MMAs of unit gi - NA
                const int h = gi - NA;
                if (h >= 0 && !mbar_wait_warp(&xa_empty[h % NS], (h / NS) & 1, status)) return false;
                tc_fence_after();
                tc_st32(tmem + tlane + A_COL + (gi % NA) * 32, av);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xa_full[gi % NS]);
            }
        }
    }
    return true;
}

// ---------------------------------------------------------------- outputs

// A tile's fused outputs for one thread's 64 tokens t0 .. t0 + 63 of row n
// (acc[j] = tokens t0 + 2j, t0 + 2j + 1): residual add, bf16, or SwiGLU,
// where lanes l and l + 8 hold the gate and the up row of one output.
template <int NJ>
__device__ __forceinline__ void wide_fused_out(const WideParent &P, int n, int t0, int T, const float2 (&acc)[NJ]) {
    if (P.epi == EPI_SWIGLU) {
        const int f = (n >> 4) * 8 + (n & 7);
        const bool gate = (n & 8) == 0 && f < P.ncols;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const float ux = __shfl_down_sync(0xffffffffu, acc[j].x, 8);
            const float uy = __shfl_down_sync(0xffffffffu, acc[j].y, 8);
            const int t = t0 + 2 * j;
            if (gate && t < T) store_y(P.Y, P.ybf16, (size_t)t * P.ncols + f, silu_mul(acc[j].x, ux));
            if (gate && t + 1 < T) store_y(P.Y, P.ybf16, (size_t)(t + 1) * P.ncols + f, silu_mul(acc[j].y, uy));
        }
    } else if (n < P.N && P.epi == EPI_ADD) {
        // the residual's 64 values in batches of 8 loads before their stores:
        // one at a time, each add waited a full memory round trip (R may be Y,
        // so the compiler cannot move a load above an earlier store; every
        // element is read before it is written either way)
#pragma unroll
        for (int jb = 0; jb < NJ; jb += 4) {
            float rv[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = t0 + 2 * (jb + j);
                rv[2 * j] = t < T ? P.R[(size_t)t * P.ncols + n] : 0.f;
                rv[2 * j + 1] = t + 1 < T ? P.R[(size_t)(t + 1) * P.ncols + n] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = t0 + 2 * (jb + j);
                if (t < T) store_y(P.Y, P.ybf16, (size_t)t * P.ncols + n, rv[2 * j] + acc[jb + j].x);
                if (t + 1 < T) store_y(P.Y, P.ybf16, (size_t)(t + 1) * P.ncols + n, rv[2 * j + 1] + acc[jb + j].y);
            }
        }
    } else if (n < P.N) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int t = t0 + 2 * j;
            if (t < T) epi_out(P, t, n, acc[j].x);
            if (t + 1 < T) epi_out(P, t + 1, n, acc[j].y);
        }
    }
}

// Write one thread's finished accumulators: row n, tokens t0 + BH h + 2j
// (+1) for each half h (t0 includes the thread's column block).
template <int BH, int H, int NJ, bool FUSED>
__device__ __forceinline__ void store_tile(const WideParent &P, int n, int t0, int T, const float2 (&acc)[H][NJ]) {
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const int th = t0 + h * BH;
        if constexpr (FUSED) {
            wide_fused_out(P, n, th, T, acc[h]);
        } else if (n < P.N) {
            float *Y = static_cast<float *>(P.Y);
            const int N = P.ncols;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int t = th + 2 * j;
                if (t < T) Y[(size_t)t * N + n] = acc[h][j].x;
                if (t + 1 < T) Y[(size_t)(t + 1) * N + n] = acc[h][j].y;
            }
        }
    }
}

// Partial-sum slots of split tiles hold float4 groups of 4 consecutive tokens,
// [BN / 4][BM] of them: element (token t, row r) at float4 (t / 4) BM + r,
// component t mod 4, so that the 32 lanes of a warp (32 consecutive rows)
// move 512 contiguous bytes per 16-byte access.
__device__ __forceinline__ size_t part_q(int t, int r) { return (size_t)(t >> 2) * wide::BM + r; }

// The sum of a split tile's partials, for one epilogue thread (row r, its
// column block c of each half), over the segments' CTAs c_first .. c_last in
// ascending order, so the order does not depend on which CTA finishes last.
// own: this CTA is c_first and acc still holds its segment, the first term;
// otherwise every segment's partial, this CTA's own included, is read back
// from the workspace and acc is overwritten.  An fp32 value read back equals
// the one written, so both give the same bits.  (acc holds the running sum,
// 32 column pairs of one segment in flight beside it.)
template <int BH, int H, int NJ, int BN>
__device__ __forceinline__ void fixup_sum(float2 (&acc)[H][NJ], const float *part, long long U, int grid,
                                          int c_first, int c_last, long long u0, int c, int r, bool own) {
    constexpr int BM = wide::BM, EW = 2 * NJ;
    constexpr int CH = H == 1 ? NJ : 16;              // column pairs in flight (registers)
#pragma unroll
    for (int h = 0; h < H; ++h)
#pragma unroll
        for (int jb = 0; jb < NJ; jb += CH) {
            // a CTA's first segment sits in its slot 0, its last in slot 1
            auto seg = [&](int cc) {
                return reinterpret_cast<const float4 *>(part + (size_t)(cc * 2 + (range_lo(U, grid, cc) >= u0 ? 0 : 1)) *
                                                                   BN * BM) +
                       part_q(h * BH + EW * c + 2 * jb, r);
            };
            if (!own) {
                const float4 *p0 = seg(c_first);
#pragma unroll
                for (int j = 0; j < CH; j += 2) {
                    const float4 x = __ldcg(p0 + (size_t)(j / 2) * BM);
                    acc[h][jb + j] = make_float2(x.x, x.y);
                    acc[h][jb + j + 1] = make_float2(x.z, x.w);
                }
            }
            for (int cc = c_first + 1; cc <= c_last; ++cc) {
                const float4 *pc = seg(cc);
                float4 v[CH / 2];
#pragma unroll
                for (int j = 0; j < CH / 2; ++j) v[j] = __ldcg(pc + (size_t)j * BM);
#pragma unroll
                for (int j = 0; j < CH / 2; ++j) {
                    acc[h][jb + 2 * j] = make_float2(acc[h][jb + 2 * j].x + v[j].x, acc[h][jb + 2 * j].y + v[j].y);
                    acc[h][jb + 2 * j + 1] =
                        make_float2(acc[h][jb + 2 * j + 1].x + v[j].z, acc[h][jb + 2 * j + 1].y + v[j].w);
                }
            }
        }
}

// ---------------------------------------------------------------- the kernel

// H: 128-token halves per tile (1 or 2).  FUSED: a parent of the launch has a
// fused output (residual add, SwiGLU or bf16); the plain instantiation keeps
// the store loop, and the code, of the plain GEMM (the fused store code in
// every launch measured 12% slower at T = 4096).  F8: a parent holds FP8
// or NVFP4 codes.  Parents of different codecs share one launch: the codec is
// resolved per tile.
template <int BH, int H, bool FUSED, bool F8>
__global__ void __launch_bounds__(wide::THREADS, 1)
    wide_kernel(const __grid_constant__ WideArgs args, const __grid_constant__ CUtensorMap xmap) {
    using namespace wide;
    using Gm = Geo<BH, H, F8>;
    constexpr int BN = Gm::BN, NS = Gm::NS, NWP = Gm::NWP, WSLOT = Gm::WSLOT, XST = Gm::XST;
    constexpr int NA = Gm::NA, NP = Gm::NP, A_COL = Gm::A_COL, EW = Gm::EW, NJ = Gm::NJ, HALF_BYTES = Gm::HALF_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xs = smem + Gm::X_OFF;
    uint8_t *ws = smem + Gm::W_OFF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Gm::BAR_OFF);
    uint64_t *w_full = bars, *w_empty = w_full + NWP;
    uint64_t *xa_full = w_empty + NWP, *xa_empty = xa_full + NS;
    uint64_t *pfull = xa_empty + NS, *pfree = pfull + NP;
    float *sc_ring = reinterpret_cast<float *>(smem + Gm::SC_OFF);
    volatile uint32_t *taddr_slot = reinterpret_cast<volatile uint32_t *>(smem + Gm::MISC_OFF);
    volatile uint32_t *abort_flag = taddr_slot + 1;

    // ---- this CTA's units: [lo, hi) of the tile-major (tile, group)
    // numbering; every role walks the same units in the same order (unit
    // index gi counts from 0 in this CTA), so rings and barrier phases run on
    // across tile boundaries
    const int G = args.G, T = args.T;
    const long long U = args.units;
    const long long lo = range_lo(U, gridDim.x, blockIdx.x), hi = range_lo(U, gridDim.x, blockIdx.x + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NWP; ++i) { mbar_init(&w_full[i], 1); mbar_init(&w_empty[i], DQ_WARPS); }
        for (int i = 0; i < NS; ++i) { mbar_init(&xa_full[i], DQ_WARPS + 1); mbar_init(&xa_empty[i], H); }
        for (int i = 0; i < NP; ++i) { mbar_init(&pfull[i], 1); mbar_init(&pfree[i], Gm::EPI_N); }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32((const void *)taddr_slot)), "n"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;

    if (warp < DQ0) {
        regs_set<Regs<BH, H>::WG0>();
        if (warp == 0) {
            // ---------------- weight producer: units (k, k + 1) of a segment in
            // one 1-D bulk copy (a row block's units are consecutive)
            bool ok = true;
            int jp = 0;                                   // weight stages used so far
            for (long long u = lo; u < hi && ok;) {
                const int tile = (int)(u / G), k0 = (int)(u % G);
                const int k1 = (int)min((long long)G, k0 + (hi - u));
                const WideTile tr = wide_tile(args, tile);
                const int UB = unit_bytes(tr.P->codec);
                const uint8_t *units = tr.P->packed + (size_t)tr.blk * G * UB;
                for (int k = k0; k < k1; k += 2, ++jp) {
                    const int wsl = jp % NWP;
                    const uint32_t bytes = (k + 1 < k1 ? 2 : 1) * UB;
                    if (jp >= NWP && !(ok = mbar_wait_warp(&w_empty[wsl], ((jp / NWP) - 1) & 1, args.status))) break;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&w_full[wsl], bytes);
                        bulk_g2s(ws + wsl * WSLOT, units + (size_t)k * UB, bytes, &w_full[wsl]);
                    }
                    __syncwarp();
                }
                u += k1 - k0;
            }
            if (!ok && lane == 0) *abort_flag = 1;
        } else if (warp == 2) {
            // ---------------- activation producer: 128B-swizzled X tiles, 2-D TMA
            pdl_wait_prior();                             // X may belong to the previous kernel
            if (lane == 0) pdl_launch_dependents();
            bool ok = true;
            int gi = 0;
            for (long long u = lo; u < hi && ok;) {
                const int tile = (int)(u / G), k0 = (int)(u % G);
                const int k1 = (int)min((long long)G, k0 + (hi - u));
                const WideTile tr = wide_tile(args, tile);
                for (int k = k0; k < k1; ++k, ++gi) {
                    const int s = gi % NS;
                    if (gi >= NS && !(ok = mbar_wait_warp(&xa_empty[s], ((gi / NS) - 1) & 1, args.status))) break;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&xa_full[s], XST);
                        tma_load_2d(xs + s * XST, &xmap, k * GROUP, tr.tt * BN, &xa_full[s]);
                    }
                    __syncwarp();
                }
                u += k1 - k0;
            }
            if (!ok && lane == 0) *abort_flag = 1;
        } else {
            // ---------------- MMA issuers: warp 1 the even steps, warp 3 the odd
            // ones (for H = 2: the first and the second half of every unit).
            // Issuing a tensor-core instruction occupies the issuing warp's
            // scheduler for tens of cycles; two issuers on two schedulers halve
            // what the epilogue and dequant warps sharing them lose.
            bool ok = true;
            const int parity = warp >> 1;
            const uint32_t idesc = idesc_bf16(BM, BH);
            const int steps = (int)(hi - lo) * H;
            int last = -1;
            for (int j = parity; j < steps; j += 2) {
                const int gi = j / H, h = j % H;
                const int s = gi % NS, b = j % NP;
                if (!(ok = mbar_wait_warp(&xa_full[s], (gi / NS) & 1, args.status))) break;
                if (j >= NP && !(ok = mbar_wait_warp(&pfree[b], ((j / NP) - 1) & 1, args.status))) break;
                tc_fence_after();
                const uint32_t d = tmem + P_COL + b * BH;
                const uint32_t a = tmem + A_COL + (gi % NA) * 32;
                tc_mma_group(d, a, smem_desc_sw128(smem_u32(xs + s * XST + h * HALF_BYTES)), idesc, &pfull[b],
                             &xa_empty[s]);
                __syncwarp();
                last = j;
            }
            if (!ok) {
                if (lane == 0) *abort_flag = 1;
                // let the MMAs this warp issued complete before tensor memory goes
                if (last >= 0) mbar_wait_limit(&pfull[last % NP], (last / NP) & 1, args.status, 64);
            }
        }
    } else if (warp < Gm::EPI_0) {
        // ---------------- dequant: thread = weight row of the tile
        regs_set<Regs<BH, H>::DQ>();
        const int q = warp & 3;                           // tensor-memory lane quarter
        const int g = (warp - DQ0) >> 2;                  // dequant group
        bool ok = true;
        int gi = 0, jp = 0;
        for (long long u = lo; u < hi && ok;) {
            const int tile = (int)(u / G), k0 = (int)(u % G);
            const int k1 = (int)min((long long)G, k0 + (hi - u));
            const WideParent &P = *wide_tile(args, tile).P;
            const int codec = P.codec;
            const float ts = P.tscale;
            if (F8 && codec == 8)
                ok = dequant_segment<8, NS, NA, NWP, WSLOT, A_COL, false, false, Gm::DQG, Gm::SC_RING>(k0, k1, gi, jp, ws, w_full, w_empty, xa_full,
                                                                      xa_empty, sc_ring, tmem, q, g, lane, ts, args.status);
            else if (F8 && codec == NVFP4)
                ok = dequant_segment<NVFP4, NS, NA, NWP, WSLOT, A_COL, false, false, Gm::DQG, Gm::SC_RING>(k0, k1, gi, jp, ws, w_full, w_empty, xa_full,
                                                                          xa_empty, sc_ring, tmem, q, g, lane, ts,
                                                                          args.status);
            else if (codec == 5)
                ok = dequant_segment<5, NS, NA, NWP, WSLOT, A_COL, H == 1, !F8, Gm::DQG, Gm::SC_RING>(k0, k1, gi, jp, ws, w_full, w_empty, xa_full,
                                                                       xa_empty, sc_ring, tmem, q, g, lane, ts, args.status);
            else
                ok = dequant_segment<4, NS, NA, NWP, WSLOT, A_COL, H == 1, !F8, Gm::DQG, Gm::SC_RING>(k0, k1, gi, jp, ws, w_full, w_empty, xa_full,
                                                                       xa_empty, sc_ring, tmem, q, g, lane, ts, args.status);
            u += k1 - k0;
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else {
        // ---------------- epilogue: thread = row r of the tile, tokens
        // [64 c, 64 c + 64) of each 128-token half
        regs_set<Regs<BH, H>::EPI>();
        pdl_wait_prior();                                 // Y, R and the workspace follow the previous kernel
        const int q = warp & 3, c = (warp - Gm::EPI_0) >> 2, e = warp - Gm::EPI_0;
        const int r = q * 32 + lane;
        const uint32_t tl = (uint32_t)(q * 32) << 16;
        bool ok = true;
        int gi = 0;
        for (long long u = lo; u < hi && ok;) {
            const int tile = (int)(u / G), k0 = (int)(u % G);
            const int k1 = (int)min((long long)G, k0 + (hi - u));
            float2 acc[H][NJ];
#pragma unroll
            for (int h = 0; h < H; ++h)
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc[h][j] = make_float2(0.f, 0.f);
            for (int k = k0; k < k1 && ok; ++k, ++gi) {
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const int j = gi * H + h;
                    const int b = j % NP;
                    // a suspending wait: with three P buffers the epilogue has
                    // two steps of MMA time to drain one, and polling warps
                    // would take the dequant warps' issue slots
                    if (!(ok = mbar_wait_warp(&pfull[b], (j / NP) & 1, args.status))) break;
                    tc_fence_after();
                    // the unit's scale (stored by the dequant before the MMAs
                    // of this step could start)
                    const float sc = sc_ring[(gi % Gm::SC_RING) * BM + r];
                    const float2 s2 = make_float2(sc, sc);
                    const uint32_t base = tmem + tl + P_COL + b * BH + EW * c;
                    if constexpr (EW == 32) {
                        uint32_t v[32];
                        tc_ld32(base, v);
                        tc_wait_ld();
                        tc_regs_ready(v);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&pfree[b]);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[h][i] = ffma2(s2, make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                              acc[h][i]);
                    } else {
                        static_assert(EW == 64, "one 32- or 64-column load per warp and step");
                        // the buffer is released one load latency after it
                        // filled, before the rescale
                        uint32_t v0[32], v1[32];
                        tc_ld64(base, v0, v1);
                        tc_wait_ld();
                        tc_regs_ready(v0);
                        tc_regs_ready(v1);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&pfree[b]);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[h][i] = ffma2(s2, make_float2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1])),
                                              acc[h][i]);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[h][16 + i] = ffma2(s2, make_float2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1])),
                                                   acc[h][16 + i]);
                    }
                }
            }
            if (!ok) break;
            // ---- the segment is done: write the tile, or leave a partial sum
            // (the MMAs of the next segment run meanwhile)
            const WideTile tr = wide_tile(args, tile);
            const int n = tr.blk * BM + r;
            const int t0 = tr.tt * BN + EW * c;
            if (k0 == 0 && k1 == G) {
                store_tile<BH, H, NJ, FUSED>(*tr.P, n, t0, T, acc);
            } else {
                const long long u0 = (long long)tile * G;
                const int c_first = range_cta(U, gridDim.x, u0), c_last = range_cta(U, gridDim.x, u0 + G - 1);
                const unsigned int others = (unsigned int)(c_last - c_first);
                unsigned int *cnt = tr.P->cnt + (size_t)tr.local * EPI_WARPS + e;
                // The head segment (the tile's first groups) closes its CTA's
                // range while the tile's other segments open theirs, so it
                // usually finishes last.  If every other segment has counted
                // in, it sums from its registers and writes no partial: the
                // counter then never reaches the count that would make
                // another segment the summing one.
                bool own = false;
                if ((int)blockIdx.x == c_first) {
                    unsigned int seen = 0;
                    if (lane == 0) seen = ld_acquire_gpu(cnt);
                    own = __shfl_sync(0xffffffffu, seen, 0) == others;
                }
                bool sum = own;
                if (!own) {
                    // a CTA's first segment goes to its slot 0, its last to slot 1
                    float4 *mine =
                        reinterpret_cast<float4 *>(args.part + (size_t)(blockIdx.x * 2 + (lo >= u0 ? 0 : 1)) * BN * BM);
#pragma unroll
                    for (int h = 0; h < H; ++h)
#pragma unroll
                        for (int j = 0; j < NJ; j += 2)
                            mine[part_q(h * BH + EW * c + 2 * j, r)] =
                                make_float4(acc[h][j].x, acc[h][j].y, acc[h][j + 1].x, acc[h][j + 1].y);
                    __threadfence();
                    __syncwarp();
                    unsigned int old = 0;
                    if (lane == 0) old = atomicAdd(cnt, 1u);
                    sum = __shfl_sync(0xffffffffu, old, 0) == others;
                    if (sum) __threadfence();
                }
                if (sum) {
                    // the last of the tile's segments sums them all
                    fixup_sum<BH, H, NJ, BN>(acc, args.part, U, (int)gridDim.x, c_first, c_last, u0, c, r, own);
                    if (lane == 0) *cnt = 0;              // zero again for the next run
                    store_tile<BH, H, NJ, FUSED>(*tr.P, n, t0, T, acc);
                }
            }
            u += k1 - k0;
        }
        if (!ok && lane == 0) *abort_flag = 1;
    }

    // ---- every role is done with tensor memory: release it
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // a wait gave up: the MMA warps have waited (bounded) for their own
        // MMAs; bulk and TMA copies already issued move at most 32 KB each and
        // land within microseconds even on a loaded GPU, so a 200 us pause
        // bounds them before the memory they write is released
        for (int i = 0; i < 200; ++i) __nanosleep(1000);
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once (a function-local static: thread-safe initialisation).
static EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// Tensor map of X [T][K] bf16 with {64 columns x BN rows} boxes, 128B
// swizzle, zero fill beyond T.
static cudaError_t make_xmap(CUtensorMap *map, const void *X, int T, int K, int BN) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {GROUP, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(X), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Units (tile, group) per CTA below which a launch uses fewer CTAs: a CTA
// with a handful of groups spends more on its pipeline fill and partial sum
// than it saves.
constexpr int MIN_UNITS_PER_CTA = 8;

// Workspace of the wide route for a plan of `rows` packed rows and widths up
// to T_max: the partial-sum slots of one launch (two per CTA, sized for the
// widest token tile the plan's widths can take, wide_max_tokens) and the
// plan's split-tile counters (eight per tile at the largest tile count any of
// the route's widths gives, that of 32-token tiles).
int wide_max_tokens(int T_max) {
    return T_max <= 16 ? 0 : T_max <= 32 ? 32 : T_max <= 64 ? 64 : T_max <= 128 ? 128 : 256;
}

size_t wide_partial_bytes(int T_max, int sms) {
    return (size_t)sms * 2 * wide_max_tokens(T_max) * wide::BM * sizeof(float);
}

size_t wide_workspace_bytes(int rows, int T_max, int sms) {
    if (wide_max_tokens(T_max) == 0) return 0;
    const int NB = (rows + wide::BM - 1) / wide::BM;
    const size_t tiles = (size_t)NB * ((T_max + 31) / 32);
    return wide_partial_bytes(T_max, sms) + tiles * wide::EPI_WARPS * sizeof(unsigned int);
}

template <int BH, int H, bool FUSED, bool F8>
static cudaError_t launch_t(const WideArgs &a, const CUtensorMap &xmap, int grid, bool pdl, cudaStream_t stream) {
    static std::atomic<bool> attr_set[64];
    using Gm = wide::Geo<BH, H, F8>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        // setmaxnreg moves each warpgroup from the launch's register count
        // (REGS_AT_LAUNCH) to its share, raising or lowering it as regs_set
        // decided at compile time; a kernel built with any other count would
        // run a lowering that raises (an illegal instruction), so it is never
        // launched
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, wide_kernel<BH, H, FUSED, F8>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != REGS_AT_LAUNCH) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(wide_kernel<BH, H, FUSED, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gm::BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(wide::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Gm::BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, wide_kernel<BH, H, FUSED, F8>, a, xmap);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BH, int H>
static cudaError_t launch_h(const WideArgs &a, const CUtensorMap &xmap, int grid, bool fused, bool f8, bool pdl,
                            cudaStream_t stream) {
    if (f8) return fused ? launch_t<BH, H, true, true>(a, xmap, grid, pdl, stream)
                         : launch_t<BH, H, false, true>(a, xmap, grid, pdl, stream);
    return fused ? launch_t<BH, H, true, false>(a, xmap, grid, pdl, stream)
                 : launch_t<BH, H, false, false>(a, xmap, grid, pdl, stream);
}

// All parents (any mix of codecs) over one shared X in one launch of tiles of
// BN = bh * halves tokens: bh = 64 (halves 1), or bh = 128 (halves 1 or 2).
// part: the partial-sum slots (wide_partial_bytes covers the launch's width);
// each parent's cnt its zeroed counters.  At most `sms` CTAs.
cudaError_t launch_wide(const WideParent *parents, int np, const void *X, int T, int K, int bh, int halves,
                        float *part, unsigned int *status, bool pdl, int sms, cudaStream_t stream) {
    if (!(((bh == 32 || bh == 64) && halves == 1) || (bh == 128 && (halves == 1 || halves == 2))))
        return cudaErrorInvalidValue;
    const int BN = halves * bh;
    CUtensorMap xmap;
    cudaError_t e = make_xmap(&xmap, X, T, K, BN);
    if (e != cudaSuccess) return e;
    WideArgs a;
    memset(&a, 0, sizeof a);
    const int ntt = (T + BN - 1) / BN;
    int tiles = 0;
    bool fused = false, f8 = false;
    for (int i = 0; i < np; ++i) {
        WideParent &d = a.p[a.nparents++];
        d = parents[i];
        d.cta_begin = tiles;
        d.nblocks = (parents[i].N + wide::BM - 1) / wide::BM;
        tiles += d.nblocks * ntt;
        fused = fused || parents[i].epi != EPI_STORE || parents[i].ybf16;
        f8 = f8 || parents[i].codec == 8 || parents[i].codec == NVFP4;
    }
    a.T = T;
    a.K = K;
    a.G = K / GROUP;
    a.ntt = ntt;
    a.ntiles = tiles;
    a.units = (long long)tiles * a.G;
    a.part = part;
    a.status = status;
    // one CTA per SM (the shared memory allows no more), each with an equal
    // share of the units
    long long grid = a.units / MIN_UNITS_PER_CTA;
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    if (bh == 32) return launch_h<32, 1>(a, xmap, (int)grid, fused, f8, pdl, stream);
    if (bh == 64) return launch_h<64, 1>(a, xmap, (int)grid, fused, f8, pdl, stream);
    return halves == 2 ? launch_h<128, 2>(a, xmap, (int)grid, fused, f8, pdl, stream)
                       : launch_h<128, 1>(a, xmap, (int)grid, fused, f8, pdl, stream);
}

}  // namespace qg
