// Wide-T route: a tcgen05 (5th-generation tensor core) dequant-GEMM.
//
// From a few dozen token columns up the operation is a dense contraction and
// belongs on the tensor cores; prefill widths are compute-bound ("ninfer-3080
// docs/performance.md", token tile section: the token tile width sets how
// often the weights are re-streamed, and the per-group rescale and the operand
// assembly are the costs beside the MMAs).  One CTA computes a 128-row block of
// Y^T for a 128-token tile:
//
//   D[128 rows x 128 tokens] = sum over 64-column groups g of s[:, g] * P_g,
//   P_g = A_g (exact integer codes as bf16, 128 x 64) . B_g (X tile, 128 x 64)^T
//
// Warp roles (16 warps; every single-issuer role is a converged warp whose
// elected lane issues, and every wait is taken by the whole warp):
//   warp 0        weight producer: 1-D bulk copies of the packed units into a
//                 deep smem ring;
//   warp 1        allocates tensor memory and issues the MMAs of even
//                 groups; warp 3 issues those of odd groups;
//   warp 2        activation producer: 2-D TMA loads of 128B-swizzled X tiles;
//   warps 4..7    dequant: one thread per weight row decodes its 64 codes of
//                 the group (magic-number bf16 decode, exact) and stores them
//                 into tensor memory as the A operand (tcgen05.st), so shared
//                 memory bandwidth is left to the B operand; the row's scale
//                 goes to the epilogue through a small shared-memory ring;
//   warps 8..15   epilogue: read P_g from tensor memory (tcgen05.ld), multiply
//                 by the row's fp16 scale and accumulate in fp32 registers
//                 (packed f32x2 FMA), then write Y.
// Tensor memory: NP P buffers of 128 columns (the MMA fills one while the
// epilogue drains another) and NA A stages of 32 columns (64 bf16 per row).
// Synchronisation per group g (stage s = g mod NS):
//   go[s]     completes when A_g is in tensor memory (4 dequant arrivals),
//             X_g has landed (TMA transaction bytes + 1 arrival) and the P
//             buffer of g is drained (8 epilogue arrivals after group g - NP):
//             the MMA warp waits on this one barrier per group;
//   done[s]   the MMA commit of group g: P_g is complete (the epilogue waits
//             on it) and A and X stage s may be overwritten (the dequant and
//             the activation producer wait on it for group g + NS); one
//             commit per group, as every MMA issue costs the issuing thread.
// Every mbarrier wait is bounded; a wait that runs out sets the device status
// to timeout and the CTA winds down (after a bounded pause that lets copies
// and MMAs already issued land before tensor memory is released).
#include <atomic>

#include <cuda.h>

#include "qgemm_internal.cuh"

namespace qg {

namespace wide {

constexpr int BM = 128;                   // weight rows per CTA (TMEM lanes)
constexpr int BN = 128;                   // tokens per CTA (MMA N)
constexpr int NS = 8;                     // activation stages (and the go / done ring)
constexpr int NA = 8;                     // A stages in tensor memory (group g uses g % NA)
constexpr int NWP = 8;                    // weight stages, each a pair of consecutive groups' units
constexpr int NP = 2;                     // P buffers in tensor memory
constexpr int DQ_WARPS = 4;               // one dequant warp per TMEM lane quarter
constexpr int EPI_WARPS = 8;              // two epilogue warps per lane quarter (column halves)
constexpr int DQ0 = 4, EPI0 = DQ0 + DQ_WARPS;
constexpr int THREADS = (EPI0 + EPI_WARPS) * 32;
constexpr int GO_COUNT = DQ_WARPS + 1 + EPI_WARPS;
constexpr int SC_RING = 16;               // groups of scales in flight
// the dequant stores the scale of group g once the epilogue has finished group g - NS - NP - 1
static_assert(SC_RING >= NA + NP + 2, "scale ring shorter than the dequant lead");
static_assert(NA <= NS && NA % 2 == 0, "A stages: even (pairs of groups) and no more than the ring");
static_assert(NS > NP, "go barrier phases need more stages than P buffers");
constexpr int X_STAGE = BN * GROUP * 2;   // 16 KB
constexpr int P_COL = 0;                  // P buffers: columns [0, 128*NP)
constexpr int A_COL = NP * BN;            // A stages: columns [128*NP, 128*NP + 32*NA)
static_assert(A_COL + 32 * NA <= 512, "tensor memory budget");
constexpr int TMEM_COLS = 512;

struct Smem {
    static constexpr int X_OFF = 0;                          // 1024-aligned (128B swizzle atoms)
    static constexpr int W_OFF = X_OFF + NS * X_STAGE;
    static constexpr int BAR_OFF = W_OFF + NWP * 2 * UNIT5;
    static constexpr int NBAR = 2 * NWP + 2 * NS;
    static constexpr int SC_OFF = BAR_OFF + NBAR * 8;                 // float [SC_RING][BM]
    static constexpr int TADDR_OFF = SC_OFF + SC_RING * BM * 4;
    static constexpr int BYTES = TADDR_OFF + 16 + 1024;      // + slack to align the base
};
static_assert(Smem::BYTES <= 227 * 1024, "shared memory budget");

}  // namespace wide

struct WideArgs {
    WideParent p[MAX_PARENTS];
    int nparents;
    int T, K, G;
    int ntt;              // token tiles
    int ntiles;           // output tiles of all parents (parent i owns p[i].cta_begin ...)
    unsigned int *status;
};

// An output tile: its parent, 128-row block and 128-token tile.
struct WideTile {
    const WideParent *P;
    int blk, tt;
};

__device__ __forceinline__ WideTile wide_tile(const WideArgs &a, int tile) {
    int pi = 0;
#pragma unroll
    for (int i = 1; i < MAX_PARENTS; ++i)
        if (i < a.nparents && tile >= a.p[i].cta_begin) pi = i;
    const int local = tile - a.p[pi].cta_begin;
    return {&a.p[pi], local / a.ntt, local % a.ntt};
}

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(tmem) . B(smem desc)^T, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, bool accum) {
    asm volatile(
        "{.reg .pred p; setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;}"
        ::"r"(d), "r"(a), "l"(bdesc), "r"(idesc), "r"(accum ? 1u : 0u) : "memory");
}

// arrive on an mbarrier once all previously issued MMAs of this thread complete
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
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

// ---------------------------------------------------------------- the kernel

// Fused outputs of one tile's accumulators (thread = row n, tokens t0 + 2j,
// t0 + 2j + 1): residual add, bf16, or SwiGLU, where lanes l and l + 8 hold
// the gate and the up row of one output.
__device__ __forceinline__ void wide_fused_out(const WideParent &P, int n, int t0, int T, const float2 (&acc)[32]) {
    if (P.epi == EPI_SWIGLU) {
        const int f = (n >> 4) * 8 + (n & 7);
        const bool gate = (n & 8) == 0 && f < P.ncols;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
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
        for (int jb = 0; jb < 32; jb += 4) {
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
        for (int j = 0; j < 32; ++j) {
            const int t = t0 + 2 * j;
            if (t < T) epi_out(P, t, n, acc[j].x);
            if (t + 1 < T) epi_out(P, t + 1, n, acc[j].y);
        }
    }
}

// CODEC: the codec of every parent of the launch (4 or 5); a launch whose
// parents mix codecs is split into one launch per codec by the host.  FUSED:
// the launch's parent has a fused output (residual add, SwiGLU or bf16); the
// plain instantiation keeps the store loop, and the code, of the plain GEMM
// (the fused store code in every launch measured 12% slower at T = 4096).
template <int CODEC, bool FUSED>
__global__ void __launch_bounds__(wide::THREADS, 1)
    wide_kernel(const __grid_constant__ WideArgs args, const __grid_constant__ CUtensorMap xmap) {
    using namespace wide;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xs = smem + Smem::X_OFF;
    uint8_t *ws = smem + Smem::W_OFF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Smem::BAR_OFF);
    uint64_t *w_full = bars, *w_empty = w_full + NWP;
    uint64_t *go = w_empty + NWP, *done = go + NS;
    float *sc_ring = reinterpret_cast<float *>(smem + Smem::SC_OFF);
    volatile uint32_t *taddr_slot = reinterpret_cast<volatile uint32_t *>(smem + Smem::TADDR_OFF);
    volatile uint32_t *abort_flag = taddr_slot + 1;

    // ---- this CTA's work: output tiles blockIdx.x, blockIdx.x + gridDim.x,
    // ... of all parents (parent i owns tiles [p[i].cta_begin, p[i].cta_begin
    // + nblocks * ntt)); every role walks the same steps gi = it * G + k over
    // the groups k of its it-th tile, so the rings and barrier phases run on
    // across tiles and the next tile's copies and MMAs overlap this tile's
    // epilogue
    const int G = args.G, T = args.T;
    const int my_tiles = (int)blockIdx.x < args.ntiles ? (args.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int steps = my_tiles * G;
    constexpr int codec = CODEC;
    constexpr int UB = unit_bytes(CODEC);
    // weight stages: pairs of units; FP8 units are larger, so the same region
    // holds fewer pairs
    constexpr int WSLOT = 2 * UB;
    constexpr int nwp = (NWP * 2 * UNIT5) / WSLOT < NWP ? (NWP * 2 * UNIT5) / WSLOT : NWP;
    static_assert(nwp >= 2, "weight ring");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NWP; ++i) { mbar_init(&w_full[i], 1); mbar_init(&w_empty[i], DQ_WARPS); }
        for (int i = 0; i < NS; ++i) { mbar_init(&go[i], GO_COUNT); mbar_init(&done[i], 1); }
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

    if (warp == 0) {
        // ---------------- weight producer: the units of groups (2j, 2j+1) of a
        // tile in one 1-D bulk copy (a row block's units are consecutive)
        bool ok = true;
        int jp = 0;                                   // weight stages used so far
        for (int it = 0; it < my_tiles && ok; ++it) {
            const WideTile tr = wide_tile(args, blockIdx.x + it * gridDim.x);
            const uint8_t *units = tr.P->packed + (size_t)tr.blk * G * UB;
            for (int j = 0; j < (G + 1) / 2; ++j, ++jp) {
                const int wsl = jp % nwp;
                const uint32_t bytes = (2 * j + 1 < G ? 2 : 1) * UB;
                if (jp >= nwp && !(ok = mbar_wait_warp(&w_empty[wsl], ((jp / nwp) - 1) & 1, args.status))) break;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&w_full[wsl], bytes);
                    bulk_g2s(ws + wsl * WSLOT, units + (size_t)(2 * j) * UB, bytes, &w_full[wsl]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else if (warp == 2) {
        // ---------------- activation producer: 128B-swizzled X tiles, 2-D TMA
        bool ok = true;
        int gi = 0;
        for (int it = 0; it < my_tiles && ok; ++it) {
            const WideTile tr = wide_tile(args, blockIdx.x + it * gridDim.x);
            for (int k = 0; k < G; ++k, ++gi) {
                const int s = gi % NS;
                if (gi >= NS && !(ok = mbar_wait_warp(&done[s], ((gi / NS) - 1) & 1, args.status))) break;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&go[s], X_STAGE);
                    tma_load_2d(xs + s * X_STAGE, &xmap, k * GROUP, tr.tt * BN, &go[s]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else if (warp == 1 || warp == 3) {
        // ---------------- MMA issuers: warp 1 even steps, warp 3 odd steps.
        // Issuing a tensor-core instruction occupies the issuing warp's
        // scheduler for tens of cycles; two issuers on two schedulers halve
        // what the epilogue and dequant warps sharing them lose, and
        // consecutive groups' MMA chains (different P buffers) interleave.
        bool ok = true;
        const uint32_t idesc = idesc_bf16(BM, BN);
        for (int gi = warp >> 1; gi < steps; gi += 2) {
            const int s = gi % NS, pb = gi % NP;
            if (!(ok = mbar_wait_warp(&go[s], (gi / NS) & 1, args.status))) break;
            tc_fence_after();
            const uint32_t d = tmem + P_COL + pb * BN;
            const uint32_t a = tmem + A_COL + (gi % NA) * 32;
            const uint32_t b0 = smem_u32(xs + s * X_STAGE);
            // one elected lane per instruction: measured cheaper to issue than
            // one elected block of four
#pragma unroll
            for (int kk = 0; kk < GROUP / 16; ++kk)
                if (elect_one()) tc_mma_ts(d, a + kk * 8, smem_desc_sw128(b0 + kk * 32), idesc, kk > 0);
            if (elect_one()) tc_commit(&done[s]);
            __syncwarp();
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else if (warp >= DQ0 && warp < EPI0) {
        // ---------------- dequant: thread = weight row r of the block; groups
        // (2j, 2j+1) of a tile per iteration, so that one weight wait, one
        // stage wait and one tensor-memory store wait serve two groups and the
        // two decodes overlap
        const int q = warp & 3;                   // TMEM lane quarter
        const int r = q * 32 + lane;
        const int tile = r >> 4, i = r & 15, gi_ = i & 7, half = i >> 3;
        const int soff = scale_off(codec) + tile * 32 + gi_ * 4 + half * 2;
        const uint32_t tlane = (uint32_t)(q * 32) << 16;
        bool ok = true;
        int jp = 0;                                   // weight stages used so far
        for (int it = 0; it < my_tiles && ok; ++it) {
            for (int j = 0; j < (G + 1) / 2; ++j, ++jp) {
                const int g0 = it * G + 2 * j;        // step of the pair's first group
                const bool two = 2 * j + 1 < G;
                const int wsl = jp % nwp;
                if (!(ok = mbar_wait_warp(&w_full[wsl], (jp / nwp) & 1, args.status))) break;
                uint32_t av[2][32];
                if constexpr (CODEC == 8) {
                    // E4M3: the row's 16 codes of lane chunk c (k 16c .. 16c+15)
                    // decoded straight from shared memory, in natural k order
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint8_t *u = ws + wsl * WSLOT + e * UB;
                        if (e == 0 || two) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint4 v = *reinterpret_cast<const uint4 *>(u + tile * 1024 + (4 * gi_ + c) * 32 + 16 * half);
                                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                for (int j2 = 0; j2 < 4; ++j2) {
                                    av[e][8 * c + 2 * j2] = dec8_pair<0>(wv[j2]);
                                    av[e][8 * c + 2 * j2 + 1] = dec8_pair<1>(wv[j2]);
                                }
                            }
                            sc_ring[((g0 + e) % SC_RING) * BM + r] = __half2float(*reinterpret_cast<const __half *>(u + soff));
                        } else {
#pragma unroll
                            for (int m = 0; m < 32; ++m) av[e][m] = 0u;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&w_empty[wsl]);
                } else {
                uint32_t wd[2][8], hw[2][4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint8_t *u = ws + wsl * WSLOT + e * UB;
                    if (e == 0 || two) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint2 v = *reinterpret_cast<const uint2 *>(u + tile * 512 + (4 * gi_ + c) * 16 + 8 * half);
                            wd[e][2 * c] = v.x;
                            wd[e][2 * c + 1] = v.y;
                            hw[e][c] = CODEC == 5 ? *reinterpret_cast<const uint32_t *>(u + NIB_BYTES + tile * 128 + (4 * gi_ + c) * 4) : 0u;
                        }
                        // the epilogue of step g0 + e reads this row's scale from the ring
                        sc_ring[((g0 + e) % SC_RING) * BM + r] = __half2float(*reinterpret_cast<const __half *>(u + soff));
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) { wd[e][2 * c] = wd[e][2 * c + 1] = 0u; hw[e][c] = 0u; }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[wsl]);
                // decode to 32 bf16x2 words per group in natural k order: word m = (k 2m, 2m+1)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t w = wd[e][2 * c + h];
                            uint32_t *o = av[e] + 8 * c + 4 * h;
                            if (CODEC == 4) {
                                o[0] = dec4_pair<0>(w); o[1] = dec4_pair<4>(w); o[2] = dec4_pair<8>(w); o[3] = dec4_pair<12>(w);
                            } else {
                                // this row's words in the lane's high word: m = 2*half + h
                                const uint32_t hh = hw[e][c] >> (4 * (2 * half + h));   // bits 4m+p / 16+4m+p -> p / 16+p
                                o[0] = dec5_pair<0, -4>(w, hh); o[1] = dec5_pair<4, -3>(w, hh);
                                o[2] = dec5_pair<8, -2>(w, hh); o[3] = dec5_pair<12, -1>(w, hh);
                            }
                        }
                    }
                }
                }
                // the A stages of both groups are free once the MMAs of steps
                // g0 - NA and g0 + 1 - NA have completed
                const int h0 = g0 - NA, h1 = g0 + 1 - NA;
                if (two && h1 >= 0 && h0 >= 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait2(&done[h0 % NS], (h0 / NS) & 1, &done[h1 % NS], (h1 / NS) & 1,
                                                            args.status));
                } else if (h0 >= 0) {
                    ok = mbar_wait_warp(&done[h0 % NS], (h0 / NS) & 1, args.status);
                } else if (two && h1 >= 0) {
                    ok = mbar_wait_warp(&done[h1 % NS], (h1 / NS) & 1, args.status);
                }
                if (!ok) break;
                tc_fence_after();
                tc_st32(tmem + tlane + A_COL + (g0 % NA) * 32, av[0]);
                if (two) tc_st32(tmem + tlane + A_COL + ((g0 + 1) % NA) * 32, av[1]);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&go[g0 % NS]);
                    if (two) mbar_arrive(&go[(g0 + 1) % NS]);
                }
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    } else if (warp >= EPI0) {
        // ---------------- epilogue: thread = row r, columns [64*hc, 64*hc + 64)
        const int q = warp & 3, hc = (warp - EPI0) >> 2;
        const int r = q * 32 + lane;
        // the first NP steps find their P buffer empty
        if (lane == 0)
            for (int g = 0; g < NP && g < steps; ++g) mbar_arrive(&go[g]);
        bool ok = true;
        int gi = 0;
        for (int it = 0; it < my_tiles && ok; ++it) {
            float2 acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = make_float2(0.f, 0.f);
            for (int k = 0; k < G; ++k, ++gi) {
                const int ps = gi % NP;
                // polled: the epilogue gates the MMAs of step gi + NP
                if (!(ok = mbar_spin_warp(&done[gi % NS], (gi / NS) & 1, args.status))) break;
                tc_fence_after();
                const float s = sc_ring[(gi % SC_RING) * BM + r];
                const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + P_COL + ps * BN + hc * 64;
                // both loads in flight before one wait: the P buffer is released
                // one load latency after it filled
                uint32_t v0[32], v1[32];
                tc_ld32(base, v0);
                tc_ld32(base + 32, v1);
                tc_wait_ld();
                tc_regs_ready(v0);
                tc_regs_ready(v1);
                tc_fence_before();
                __syncwarp();
                // P buffer ps is free for step gi + NP
                if (lane == 0 && gi + NP < steps) mbar_arrive(&go[(gi + NP) % NS]);
                // packed f32x2 FMAs: half the instructions of scalar ones
                const float2 s2 = make_float2(s, s);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    acc[j] = ffma2(s2, make_float2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1])), acc[j]);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    acc[16 + j] = ffma2(s2, make_float2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1])), acc[16 + j]);
            }
            if (!ok) break;
            // ---- write this tile's Y[t][n] (consecutive lanes = consecutive rows
            // n) while the MMAs of the next tile run
            const WideTile tr = wide_tile(args, blockIdx.x + it * gridDim.x);
            const int n = tr.blk * BM + r;
            if constexpr (FUSED) {
                wide_fused_out(*tr.P, n, tr.tt * BN + hc * 64, T, acc);
            } else if (n < tr.P->N) {
                float *Y = static_cast<float *>(tr.P->Y);
                const int N = tr.P->ncols;
                const int t0 = tr.tt * BN + hc * 64;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = t0 + 2 * j;
                    if (t < T) Y[(size_t)t * N + n] = acc[j].x;
                    if (t + 1 < T) Y[(size_t)(t + 1) * N + n] = acc[j].y;
                }
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
    }

    // ---- every role is done with tensor memory: release it
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // a wait gave up: copies and MMAs already issued finish within
        // microseconds; give them a bounded pause before the memory they
        // write is released
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

// Tensor map of X [T][K] bf16 with {64 columns x 128 rows} boxes, 128B swizzle,
// zero fill beyond T.
static cudaError_t make_xmap(CUtensorMap *map, const void *X, int T, int K) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {GROUP, wide::BN};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(X), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int wide_tile_tokens() { return wide::BN; }

template <int CODEC, bool FUSED>
static cudaError_t launch_codec(const WideParent *parents, int np, const CUtensorMap &xmap, int T, int K,
                                unsigned int *status, cudaStream_t stream) {
    static std::atomic<bool> attr_set[64];
    static std::atomic<int> sms[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(wide_kernel<CODEC, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 wide::Smem::BYTES);
        if (e != cudaSuccess) return e;
        int n = 0;
        if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        sms[dev].store(n, std::memory_order_relaxed);
        attr_set[dev].store(true, std::memory_order_release);
    }
    WideArgs a;
    memset(&a, 0, sizeof a);
    const int ntt = (T + wide::BN - 1) / wide::BN;
    int tiles = 0;
    for (int i = 0; i < np; ++i) {
        if (parents[i].codec != CODEC) continue;
        WideParent &d = a.p[a.nparents++];
        d = parents[i];
        d.cta_begin = tiles;
        d.nblocks = (parents[i].N + wide::BM - 1) / wide::BM;
        tiles += d.nblocks * ntt;
    }
    if (tiles == 0) return cudaSuccess;
    a.T = T;
    a.K = K;
    a.G = K / GROUP;
    a.ntt = ntt;
    a.ntiles = tiles;
    a.status = status;
    // persistent: one CTA per SM (its shared memory allows no more), each
    // taking the tiles blockIdx.x, blockIdx.x + grid, ...
    const int nsm = sms[dev].load(std::memory_order_relaxed);
    const int grid = tiles < nsm ? tiles : nsm;
    wide_kernel<CODEC, FUSED><<<grid, wide::THREADS, wide::Smem::BYTES, stream>>>(a, xmap);
    return cudaGetLastError();
}

// Parents of both codecs in one call become one launch per codec.
cudaError_t launch_wide(const WideParent *parents, int np, const void *X, int T, int K, unsigned int *status,
                        cudaStream_t stream, int *launches) {
    CUtensorMap xmap;
    cudaError_t e = make_xmap(&xmap, X, T, K);
    if (e != cudaSuccess) return e;
    int n4 = 0, n5 = 0, n8 = 0;
    bool fused = false;
    for (int i = 0; i < np; ++i) {
        (parents[i].codec == 4 ? n4 : parents[i].codec == 5 ? n5 : n8)++;
        fused = fused || parents[i].epi != EPI_STORE || parents[i].ybf16;
    }
    if (n4 && (e = fused ? launch_codec<4, true>(parents, np, xmap, T, K, status, stream)
                         : launch_codec<4, false>(parents, np, xmap, T, K, status, stream)) != cudaSuccess)
        return e;
    if (n5 && (e = fused ? launch_codec<5, true>(parents, np, xmap, T, K, status, stream)
                         : launch_codec<5, false>(parents, np, xmap, T, K, status, stream)) != cudaSuccess)
        return e;
    if (n8 && (e = fused ? launch_codec<8, true>(parents, np, xmap, T, K, status, stream)
                         : launch_codec<8, false>(parents, np, xmap, T, K, status, stream)) != cudaSuccess)
        return e;
    *launches = (n4 > 0) + (n5 > 0) + (n8 > 0);
    return cudaSuccess;
}

}  // namespace qg
