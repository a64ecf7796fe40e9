// Small-T route: a weight-streaming skinny GEMM.
//
// At decode and verify widths the operation streams the whole weight matrix
// once for a handful of token columns, so HBM bandwidth bounds it ("ninfer-3080
// docs/performance.md": the small-T kernels section measures its Q4/Q5
// kernels against the streaming floor and finds the remainder at one stream
// to be kernel ramp-up and drain; the route boundaries section notes that
// cold weight streaming is the production regime).  The design:
//
// * grid: one CTA per 16-row tile of the weight matrix; its warps split K.
//   Two kernels share this scheme.  Where K / 64 is a multiple of 8 (the
//   shapes of the pages' models), each warp owns 8 consecutive groups and
//   copies all of them into shared memory at once, with 16-byte asynchronous
//   copies of exactly the 16-byte code chunk each lane will decode (512
//   contiguous bytes per warp and group), so the group loop is straight-line
//   code with immediate offsets and the codec is resolved once per CTA.
//   Otherwise warp kw takes groups kw, kw+KW, ... through a private ring of 8
//   stages.  Both keep the bytes in flight out of registers and need no
//   cross-warp synchronisation until the end; a CTA owns whole output rows and
//   leaves as soon as it is done, so no CTA waits on another;
// * the warps decode their lane's 16 codes per row in registers
//   (magic-number bf16 decode) and run bf16 m16n8k16 tensor-core MMAs against
//   the activation fragments, whose k order is permuted the same way as the
//   codes (any permutation inside a group is valid when A and B agree -- the
//   small-T kernels section's permuted k order);
// * each 64-column group's fp32 partial is multiplied by its fp16 scale and
//   added to the fp32 accumulator (the per-group rescale of the token-tile
//   section's ablation): scale * code is never rounded;
// * the K split inside the CTA is combined in shared memory in warp order --
//   deterministic, no workspace, no atomics;
// * programmatic dependent launch: the weights do not depend on the previous
//   kernel in the stream, so each warp issues its weight copies before
//   griddepcontrol.wait, and back-to-back calls overlap their ramp and drain
//   (the pages name ramp and drain at kernel boundaries as what is left at
//   one stream).  Where the next kernel may start is measured per kernel:
//   see the trigger placements below.
#include <atomic>
#include <utility>

#include "qgemm_internal.cuh"

namespace qg {

constexpr int RING = 8;                 // groups in flight per warp
constexpr int STAGE = 672;              // codes 512 B | int5 high words 128 B | scales 32 B
constexpr int STAGE8 = 1056;            // fp8: codes 1024 B | scales 32 B
constexpr int SC8 = 1024;               // fp8: offset of the scale pairs in a stage

// Row r, token t of a tile: the warps' partials summed in warp order.
template <int RS>
__device__ __forceinline__ float red_sum(const float *red, int T8, int KW, int t, int r) {
    float v = red[t * RS + r];
#pragma unroll 4
    for (int q = 1; q < KW; ++q) v += red[(q * T8 + t) * RS + r];
    return v;
}

// Write a tile's outputs through the parent's epilogue: its 16 rows (STORE,
// ADD), or its 8 SwiGLU outputs from the gate rows 0..7 and up rows 8..15.
template <int RS>
__device__ __forceinline__ void write_tile(const SkinnyParent &P, const float *red, int T8, int KW, int tile,
                                           int T) {
    if (P.epi == EPI_SWIGLU) {
        for (int e = threadIdx.x; e < T * 8; e += KW * 32) {
            const int t = e >> 3, r = e & 7;
            const int f = tile * 8 + r;
            if (f < P.ncols)
                store_y(P.Y, P.ybf16, (size_t)t * P.ncols + f,
                        silu_mul(red_sum<RS>(red, T8, KW, t, r), red_sum<RS>(red, T8, KW, t, r + 8)));
        }
    } else if (P.epi == EPI_STORE && !P.ybf16) {
        float *Y = static_cast<float *>(P.Y);
        const int n0 = tile * 16;
        const int rows = min(16, P.N - n0);
        for (int e = threadIdx.x; e < T * 16; e += KW * 32) {
            const int t = e >> 4, r = e & 15;
            const float v = red_sum<RS>(red, T8, KW, t, r);
            if (r < rows) Y[(size_t)t * P.ncols + n0 + r] = v;
        }
    } else {
        const int n0 = tile * 16;
        const int rows = min(16, P.N - n0);
        for (int e = threadIdx.x; e < T * 16; e += KW * 32) {
            const int t = e >> 4, r = e & 15;
            const float v = red_sum<RS>(red, T8, KW, t, r);
            if (r < rows) epi_out(P, t, n0 + r, v);
        }
    }
}

template <int NT, int KW, int ST = STAGE>
struct SkinnySmem {
    static constexpr int RED_STRIDE = 17;                        // floats per token row (bank spread)
    static constexpr int RINGS = KW * RING * ST;
    static constexpr int RED = KW * NT * 8 * RED_STRIDE * 4;     // [KW][8*NT][16] partials
    static constexpr int BYTES = RINGS + RED;
};

// A fragments of one 16-row tile for the four k16 steps of a group.
// word m: 0 = cw.x, 1 = cw.y (row g); 2 = cw.z, 3 = cw.w (row g+8).
__device__ __forceinline__ void decode_tile(int codec, uint4 cw, uint32_t hw, uint32_t (&a)[4][4]) {
    if (codec == 4) {
        a[0][0] = dec4_pair<0>(cw.x);  a[0][1] = dec4_pair<0>(cw.z);  a[0][2] = dec4_pair<4>(cw.x);  a[0][3] = dec4_pair<4>(cw.z);
        a[1][0] = dec4_pair<8>(cw.x);  a[1][1] = dec4_pair<8>(cw.z);  a[1][2] = dec4_pair<12>(cw.x); a[1][3] = dec4_pair<12>(cw.z);
        a[2][0] = dec4_pair<0>(cw.y);  a[2][1] = dec4_pair<0>(cw.w);  a[2][2] = dec4_pair<4>(cw.y);  a[2][3] = dec4_pair<4>(cw.w);
        a[3][0] = dec4_pair<8>(cw.y);  a[3][1] = dec4_pair<8>(cw.w);  a[3][2] = dec4_pair<12>(cw.y); a[3][3] = dec4_pair<12>(cw.w);
    } else {
        // high bit of word m, pair i sits HSH = 4m + i - 4 bits above bit 4
        a[0][0] = dec5_pair<0, -4>(cw.x, hw);  a[0][1] = dec5_pair<0, 4>(cw.z, hw);
        a[0][2] = dec5_pair<4, -3>(cw.x, hw);  a[0][3] = dec5_pair<4, 5>(cw.z, hw);
        a[1][0] = dec5_pair<8, -2>(cw.x, hw);  a[1][1] = dec5_pair<8, 6>(cw.z, hw);
        a[1][2] = dec5_pair<12, -1>(cw.x, hw); a[1][3] = dec5_pair<12, 7>(cw.z, hw);
        a[2][0] = dec5_pair<0, 0>(cw.y, hw);   a[2][1] = dec5_pair<0, 8>(cw.w, hw);
        a[2][2] = dec5_pair<4, 1>(cw.y, hw);   a[2][3] = dec5_pair<4, 9>(cw.w, hw);
        a[3][0] = dec5_pair<8, 2>(cw.y, hw);   a[3][1] = dec5_pair<8, 10>(cw.w, hw);
        a[3][2] = dec5_pair<12, 3>(cw.y, hw);  a[3][3] = dec5_pair<12, 11>(cw.w, hw);
    }
}

// NVFP4 A fragments: the lane's nibble words as for int4 (x, y row g; z, w row
// g+8) times the rows' block scales (bytes 0 and 1 of bsw), exact in bf16.
__device__ __forceinline__ void decode_tile16(uint4 cw, uint32_t bsw, uint32_t (&a)[4][4]) {
    const uint32_t bsp = ue4m3x2_to_bf16x2(bsw);
    const uint32_t b0 = __byte_perm(bsp, 0, 0x1010), b1 = __byte_perm(bsp, 0, 0x3232);
    a[0][0] = dec16_pair<0>(cw.x, b0); a[0][1] = dec16_pair<0>(cw.z, b1); a[0][2] = dec16_pair<1>(cw.x, b0); a[0][3] = dec16_pair<1>(cw.z, b1);
    a[1][0] = dec16_pair<2>(cw.x, b0); a[1][1] = dec16_pair<2>(cw.z, b1); a[1][2] = dec16_pair<3>(cw.x, b0); a[1][3] = dec16_pair<3>(cw.z, b1);
    a[2][0] = dec16_pair<0>(cw.y, b0); a[2][1] = dec16_pair<0>(cw.w, b1); a[2][2] = dec16_pair<1>(cw.y, b0); a[2][3] = dec16_pair<1>(cw.w, b1);
    a[3][0] = dec16_pair<2>(cw.y, b0); a[3][1] = dec16_pair<2>(cw.w, b1); a[3][2] = dec16_pair<3>(cw.y, b0); a[3][3] = dec16_pair<3>(cw.w, b1);
}

// FP8 A fragments from the lane's 32-byte chunk: lo = row g, hi = row g+8,
// word q of a row = k 4q .. 4q+3 (pairs in bytes 0/2 and 1/3).
__device__ __forceinline__ void decode_tile8(uint4 lo, uint4 hi, uint32_t (&a)[4][4]) {
    const uint32_t l[4] = {lo.x, lo.y, lo.z, lo.w}, h[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        a[q][0] = dec8_pair<0>(l[q]);
        a[q][1] = dec8_pair<0>(h[q]);
        a[q][2] = dec8_pair<1>(l[q]);
        a[q][3] = dec8_pair<1>(h[q]);
    }
}

// One CTA per 16-row tile: KW warps split the tile's K groups (warp kw takes
// groups kw, kw + KW, ...), each streaming its groups through a private ring
// of RING stages; then the CTA sums the warps' partials in warp order.
//
// The loop is unrolled by the ring depth so that stage offsets are immediates,
// and every global address advances by a constant stride: the integer pipe,
// which also carries the nibble unpacking, is the tightest resource here.
// ST: the stage size, STAGE8 when a parent of the launch holds FP8 codes.
template <int NT, int KW, int ST>
__global__ void __launch_bounds__(KW * 32) skinny_kernel(const __grid_constant__ SkinnyArgs args) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int RS = SkinnySmem<NT, KW, ST>::RED_STRIDE;
    constexpr int T8 = 8 * NT;

    // ---- which parent and tile this CTA owns
    int pi = 0;
#pragma unroll
    for (int i = 1; i < MAX_PARENTS; ++i)
        if (i < args.nparents && (int)blockIdx.x >= args.p[i].cta_begin) pi = i;
    const SkinnyParent &P = args.p[pi];
    const int tile = blockIdx.x - P.cta_begin;       // 16-row tile of this parent
    const int b = tile / TILES, w = tile % TILES;    // its block and position in the block
    const int G = args.G;
    const int codec = P.codec;
    const int UB = unit_bytes(codec);

    const int kw = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int T = args.T;
    uint8_t *ring = smem + kw * RING * ST;
    float *red = reinterpret_cast<float *>(smem + SkinnySmem<NT, KW, ST>::RINGS);
    const int nj = (G - kw + KW - 1) / KW;           // groups of this warp: kw + KW*j

    // per-lane copy plan: every lane its 16-byte code chunk (FP8: 32 bytes,
    // two copies); lanes 8..15 the int5 high words, or lanes 8..11 the NVFP4
    // block scales; lanes 16..17 the scale pairs (not NVFP4: its tensor scale
    // stands in for them)
    const bool f8 = ST == STAGE8 && codec == 8;
    const bool fp4 = ST == STAGE8 && codec == NVFP4;
    const int ch = f8 ? 32 : 16;                     // code bytes per lane
    const int sco = f8 ? SC8 : 640;                  // scale pairs in the stage
    const uint8_t *src = P.packed + ((size_t)b * G + kw) * UB + w * 32 * ch + lane * ch;
    const size_t step = (size_t)KW * UB;
    const bool cp_hi = (codec == 5 && lane >= 8 && lane < 16) || (fp4 && lane >= 8 && lane < 12);
    const bool cp_sc = !fp4 && lane >= 16 && lane < 18;
    const int ex_dst = cp_hi ? 512 + (lane - 8) * 16 : sco + (lane - 16) * 16;
    const long ex_src = cp_hi ? (long)(NIB_BYTES + w * (fp4 ? 64 : 128) + (lane - 8) * 16) - (w * 512 + lane * 16)
                              : (long)(scale_off(codec) + w * 32 + (lane - 16) * 16) - (w * 32 * ch + lane * ch);
    const bool cp_ex = cp_hi || cp_sc;

    // per-lane activation plan: token 8*nt + g, k = 64*grp + 16c
    const __nv_bfloat16 *xp = args.X + (size_t)g * args.K + (size_t)kw * GROUP + 16 * c;
    const size_t xstep = (size_t)KW * GROUP;
    const size_t xtok8 = (size_t)8 * args.K;
    bool tok_ok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) tok_ok[nt] = nt * 8 + g < T;
    const bool pf = c == 0;

    // The weights do not depend on the previous kernel in the stream: fill the
    // ring, and only then wait for that kernel.
#pragma unroll
    for (int r = 0; r < RING; ++r) {
        if (r < nj) {
            const uint8_t *sr = src + r * step;
            cp_async16(ring + r * ST + lane * ch, sr);
            if (f8) cp_async16(ring + r * ST + lane * ch + 16, sr + 16);
            if (cp_ex) cp_async16(ring + r * ST + ex_dst, sr + ex_src);
        }
        cp_async_commit();
    }
    pdl_wait_prior();   // X and Y may belong to the previous kernel
    if (pf) {
#pragma unroll
        for (int r = 0; r < RING; ++r)
            if (r < nj)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    if (tok_ok[nt]) prefetch_l1(xp + r * xstep + nt * xtok8);
    }

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

    const uint8_t *src_next = src + RING * step;      // group j + RING
    const __nv_bfloat16 *x_cur = xp;                  // group j
    for (int j0 = 0; j0 < nj; j0 += RING) {
#pragma unroll
        for (int r = 0; r < RING; ++r) {
            if (j0 + r < nj) {
                // activation fragments of this group (L1-resident after the prefetch)
                uint32_t xb[NT][8];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (tok_ok[nt]) {
                        const uint4 *q = reinterpret_cast<const uint4 *>(x_cur + nt * xtok8);
                        const uint4 v0 = __ldg(q), v1 = __ldg(q + 1);
                        xb[nt][0] = v0.x; xb[nt][1] = v0.y; xb[nt][2] = v0.z; xb[nt][3] = v0.w;
                        xb[nt][4] = v1.x; xb[nt][5] = v1.y; xb[nt][6] = v1.z; xb[nt][7] = v1.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) xb[nt][e] = 0u;
                    }
                }
                cp_async_wait<RING - 1>();            // this group of every lane has landed
                __syncwarp();
                uint8_t *st = ring + r * ST;
                const uint4 cw = *reinterpret_cast<const uint4 *>(st + lane * ch);
                const uint4 cw8 = f8 ? *reinterpret_cast<const uint4 *>(st + lane * ch + 16) : make_uint4(0, 0, 0, 0);
                const uint32_t hw = codec == 5 ? *reinterpret_cast<const uint32_t *>(st + 512 + lane * 4)
                                    : fp4      ? *reinterpret_cast<const uint16_t *>(st + 512 + lane * 2)
                                               : 0u;
                const uint32_t sp = fp4 ? 0u : *reinterpret_cast<const uint32_t *>(st + sco + g * 4);
                __syncwarp();                         // every lane has read the stage
                if (j0 + r + RING < nj) {
                    cp_async16(st + lane * ch, src_next);
                    if (f8) cp_async16(st + lane * ch + 16, src_next + 16);
                    if (cp_ex) cp_async16(st + ex_dst, src_next + ex_src);
                    if (pf) {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (tok_ok[nt]) prefetch_l1(x_cur + RING * xstep + nt * xtok8);
                    }
                }
                cp_async_commit();
                src_next += step;
                x_cur += xstep;

                uint32_t a[4][4];
                if (f8) decode_tile8(cw, cw8, a);
                else if (fp4) decode_tile16(cw, hw, a);
                else decode_tile(codec, cw, hw, a);
                const float2 sc = fp4 ? make_float2(P.tscale, P.tscale)
                                      : __half22float2(*reinterpret_cast<const __half2 *>(&sp));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t bf[2] = {xb[nt][2 * q], xb[nt][2 * q + 1]};
                        mma_bf16_16816(p, a[q], bf, p);
                    }
                    acc[nt][0] = fmaf(sc.x, p[0], acc[nt][0]);
                    acc[nt][1] = fmaf(sc.x, p[1], acc[nt][1]);
                    acc[nt][2] = fmaf(sc.y, p[2], acc[nt][2]);
                    acc[nt][3] = fmaf(sc.y, p[3], acc[nt][3]);
                }
            }
        }
    }
    cp_async_wait<0>();
    // this CTA's weights are all in: the next kernel in the stream may start
    // its own weight stream while this one finishes
    if (threadIdx.x == 0) pdl_launch_dependents();

    // ---- combine the warps' partials in warp order and write Y
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int t = nt * 8 + 2 * c;
        float *rw = red + (kw * T8) * RS;
        rw[t * RS + g] = acc[nt][0];
        rw[(t + 1) * RS + g] = acc[nt][1];
        rw[t * RS + g + 8] = acc[nt][2];
        rw[(t + 1) * RS + g + 8] = acc[nt][3];
    }
    __syncthreads();
    write_tile<RS>(P, red, T8, KW, tile, T);
}

// ---------------------------------------------------------------- straight-line kernels
//
// When K / 64 is a multiple of NJ, each warp owns NJ consecutive groups of its
// tile.  Its copies go through a private ring of RG stages (RG == NJ: all of
// them in flight at once; RG < NJ: the stage a group was read from is refilled
// with group + RG right after the read), the group loop is fully unrolled
// with immediate offsets, and the codec is resolved once per CTA, which leaves
// per group little beyond the decode, the four MMAs and the rescale.  A CTA
// has K / (64 NJ) warps.  A smaller ring lets more CTAs share an SM, so that
// the next call's CTAs can start their weight stream while this call's CTAs
// still compute.

template <int NJ, int RG, int NT>
struct LineSmem {
    static constexpr int RED_STRIDE = 17;
    // st: the stage size of the CTA's codec (the launch sizes for the largest)
    __host__ __device__ static constexpr int rings(int kw, int st) { return kw * RG * st; }
    __host__ __device__ static constexpr int bytes(int kw, int st) {
        return rings(kw, st) + kw * NT * 8 * RED_STRIDE * 4;
    }
};

// Stage geometry of a codec, by its unit size: code bytes per lane, the
// offset of the scale pairs, the stage size.
template <int UB>
struct LineStage {
    static constexpr bool F8 = UB == UNIT8;
    static constexpr int CH = F8 ? 32 : 16;
    static constexpr int SC = F8 ? SC8 : 640;
    static constexpr int BYTES = F8 ? STAGE8 : STAGE;
};

// Activation fragment of group R for token row pointer xr: the lane's 16 k.
// (volatile, so that the compiler keeps the loads where they are written: the
// up-front loads must not sink to their uses)
template <int R>
__device__ __forceinline__ void load_x(const __nv_bfloat16 *xr, uint32_t (&xb)[8]) {
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(xb[0]), "=r"(xb[1]), "=r"(xb[2]), "=r"(xb[3]) : "l"(xr + R * GROUP));
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(xb[4]), "=r"(xb[5]), "=r"(xb[6]), "=r"(xb[7]) : "l"(xr + R * GROUP + 8));
}

// The copies of one lane for the warp's groups: its 16-byte code chunk, and
// for lanes 8..15 (int5 high words) and 16..17 (scale pairs) one more chunk.
struct LaneCopies {
    const uint8_t *src;      // the lane's code chunk of the warp's first group
    int ex_dst, ex_src;      // the extra chunk: offset in the stage, offset from src
    bool ex;
};

template <int UB, int RG, int R>
__device__ __forceinline__ void issue_group(uint8_t *ring, const LaneCopies &lc, int lane) {
    using S = LineStage<UB>;
    uint8_t *st = ring + (R % RG) * S::BYTES;
    cp_async16(st + lane * S::CH, lc.src + R * UB);
    if (S::F8) cp_async16(st + lane * S::CH + 16, lc.src + R * UB + 16);
    if (lc.ex) cp_async16(st + lc.ex_dst, lc.src + R * UB + lc.ex_src);
    cp_async_commit();
}

template <int UB, int RG, int... R>
__device__ __forceinline__ void issue_groups(std::integer_sequence<int, R...>, uint8_t *ring, const LaneCopies &lc,
                                             int lane) {
    (issue_group<UB, RG, R>(ring, lc, lane), ...);
}

// Group R of the warp: wait for its copy, refill its stage, decode, MMA
// against the activation fragments, rescale into acc.  xpre holds the
// activation fragments of every group when they were loaded up front.
template <int NT, int CODEC, int NJ, int RG, int XP, int R>
__device__ __forceinline__ void line_group(uint8_t *ring, const LaneCopies &lc, int lane, int g,
                                           const __nv_bfloat16 *const (&xr)[NT], const uint32_t (&xpre)[XP][8],
                                           float (&acc)[NT][4], float ts) {
    constexpr int UB = unit_bytes(CODEC);
    using S = LineStage<UB>;
    constexpr int ISSUED = RG + R < NJ ? RG + R : NJ;     // groups whose copies are issued
    uint32_t xb[NT][8];
    if (XP == NJ) {
#pragma unroll
        for (int e = 0; e < 8; ++e) xb[0][e] = xpre[R][e];
    } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) load_x<R>(xr[nt], xb[nt]);
    }
    cp_async_wait<ISSUED - 1 - R>();                   // groups 0..R of this lane have landed
    __syncwarp();                                      // ... and of every lane
    const uint8_t *st = ring + (R % RG) * S::BYTES;
    const uint4 cw = *reinterpret_cast<const uint4 *>(st + lane * S::CH);
    const uint4 cw8 = S::F8 ? *reinterpret_cast<const uint4 *>(st + lane * S::CH + 16) : make_uint4(0, 0, 0, 0);
    const uint32_t hw = CODEC == 5       ? *reinterpret_cast<const uint32_t *>(st + 512 + lane * 4)
                        : CODEC == NVFP4 ? *reinterpret_cast<const uint16_t *>(st + 512 + lane * 2)
                                         : 0u;
    const uint32_t sp = CODEC == NVFP4 ? 0u : *reinterpret_cast<const uint32_t *>(st + S::SC + g * 4);
    if (R + RG < NJ) {
        __syncwarp();                                  // every lane has read the stage
        issue_group<UB, RG, R + RG>(ring, lc, lane);
    }
    uint32_t a[4][4];
    if (S::F8) decode_tile8(cw, cw8, a);
    else if (CODEC == NVFP4) decode_tile16(cw, hw, a);
    else decode_tile(CODEC, cw, hw, a);
    const float2 sc = CODEC == NVFP4 ? make_float2(ts, ts) : __half22float2(*reinterpret_cast<const __half2 *>(&sp));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t bf[2] = {xb[nt][2 * q], xb[nt][2 * q + 1]};
            mma_bf16_16816(p, a[q], bf, p);
        }
        acc[nt][0] = fmaf(sc.x, p[0], acc[nt][0]);
        acc[nt][1] = fmaf(sc.x, p[1], acc[nt][1]);
        acc[nt][2] = fmaf(sc.y, p[2], acc[nt][2]);
        acc[nt][3] = fmaf(sc.y, p[3], acc[nt][3]);
    }
}

template <int NT, int CODEC, int NJ, int RG, int XP, int... R>
__device__ __forceinline__ void line_groups(std::integer_sequence<int, R...>, uint8_t *ring, const LaneCopies &lc,
                                            int lane, int g, const __nv_bfloat16 *const (&xr)[NT],
                                            const uint32_t (&xpre)[XP][8], float (&acc)[NT][4], float ts) {
    (line_group<NT, CODEC, NJ, RG, XP, R>(ring, lc, lane, g, xr, xpre, acc, ts), ...);
}

template <int XP, int... R>
__device__ __forceinline__ void load_x_all(std::integer_sequence<int, R...>, const __nv_bfloat16 *xr,
                                           uint32_t (&xpre)[XP][8]) {
    (load_x<R>(xr, xpre[R]), ...);
}

template <int NT, int CODEC, int NJ, int RG>
__device__ __forceinline__ void line_tile(const SkinnyArgs &args, const SkinnyParent &P, int tile, uint8_t *smem) {
    constexpr int RS = LineSmem<NJ, RG, NT>::RED_STRIDE;
    constexpr int T8 = 8 * NT;
    constexpr int UB = unit_bytes(CODEC);
    using S = LineStage<UB>;
    constexpr int XP = (NT == 1 && NJ <= 8) ? NJ : 1;   // activation fragments loaded up front
    const int KW = blockDim.x >> 5;
    const int b = tile / TILES, w = tile % TILES;
    const int G = args.G;
    const int kw = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int T = args.T;
    const int gb = kw * NJ;                           // this warp's first group
    uint8_t *ring = smem + kw * RG * S::BYTES;
    float *red = reinterpret_cast<float *>(smem + LineSmem<NJ, RG, NT>::rings(KW, S::BYTES));

    // per-lane copy plan (as the ring kernel's): every lane its 16-byte code
    // chunk (FP8: 32 bytes); lanes 8..15 the int5 high words, or 8..11 the
    // NVFP4 block scales; lanes 16..17 the scale pairs (not for NVFP4)
    const bool cp_hi = (CODEC == 5 && lane >= 8 && lane < 16) || (CODEC == NVFP4 && lane >= 8 && lane < 12);
    const int own = w * 32 * S::CH + lane * S::CH;    // the lane's chunk in the unit
    LaneCopies lc;
    lc.src = P.packed + ((size_t)b * G + gb) * UB + own;
    lc.ex = cp_hi || (CODEC != NVFP4 && lane >= 16 && lane < 18);
    lc.ex_dst = cp_hi ? 512 + (lane - 8) * 16 : S::SC + (lane - 16) * 16;
    lc.ex_src = cp_hi ? (NIB_BYTES + w * (CODEC == NVFP4 ? 64 : 128) + (lane - 8) * 16) - own
                      : (scale_off(CODEC) + w * 32 + (lane - 16) * 16) - own;
    issue_groups<UB, RG>(std::make_integer_sequence<int, RG>{}, ring, lc, lane);
    // Programmatic dependent launch: with one token tile the next kernel in the
    // stream may start once this CTA's weight copies are issued and the
    // previous kernel has finished (its own weight stream then overlaps this
    // kernel's compute, and no kernel runs more than one call ahead); with
    // more token tiles the CTA's compute is longer and an early start measured
    // slower, so the trigger waits until this CTA's groups are done.
    pdl_wait_prior();   // X and Y may belong to the previous kernel
    if (NT == 1 && threadIdx.x == 0) pdl_launch_dependents();

    // activation fragments: token 8*nt + g, k = 64*(gb + r) + 16c.  Lanes of
    // tokens >= T read row T - 1 instead: their MMA columns are never written,
    // and every lane then runs the same loads with no branch.  With one token
    // tile and few groups per warp the fragments of all groups are loaded up
    // front, in the shadow of the weight copies; otherwise lanes with c == 0
    // pull the rows' lines into L1 and each group loads its own.
    const __nv_bfloat16 *xr[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        xr[nt] = args.X + (size_t)min(nt * 8 + g, T - 1) * args.K + (size_t)gb * GROUP + 16 * c;
    uint32_t xpre[XP][8];
    if (XP == NJ) {
        load_x_all<XP>(std::make_integer_sequence<int, XP>{}, xr[0], xpre);
    } else if (c == 0) {
#pragma unroll
        for (int r = 0; r < NJ; ++r)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) prefetch_l1(xr[nt] + r * GROUP);
    }

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    line_groups<NT, CODEC, NJ, RG, XP>(std::make_integer_sequence<int, NJ>{}, ring, lc, lane, g, xr, xpre, acc,
                                       P.tscale);
    if (NT > 1 && threadIdx.x == 0) pdl_launch_dependents();

    // ---- combine the warps' partials in warp order and write Y
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int t = nt * 8 + 2 * c;
        float *rw = red + (kw * T8) * RS;
        rw[t * RS + g] = acc[nt][0];
        rw[(t + 1) * RS + g] = acc[nt][1];
        rw[t * RS + g + 8] = acc[nt][2];
        rw[(t + 1) * RS + g + 8] = acc[nt][3];
    }
    __syncthreads();
    write_tile<RS>(P, red, T8, KW, tile, T);
}

// F8: the launch has FP8 or NVFP4 parents (the kernel then also serves the
// integer codecs, for multi-parent launches); the integer-only instantiation
// keeps the code of the integer codecs alone.
template <int NT, int NJ, int RG, bool F8>
__global__ void __launch_bounds__(16 * 32) skinny_line_kernel(const __grid_constant__ SkinnyArgs args) {
    extern __shared__ __align__(128) uint8_t smem[];
    int pi = 0;
#pragma unroll
    for (int i = 1; i < MAX_PARENTS; ++i)
        if (i < args.nparents && (int)blockIdx.x >= args.p[i].cta_begin) pi = i;
    const SkinnyParent &P = args.p[pi];
    const int tile = blockIdx.x - P.cta_begin;
    if (F8 && P.codec == 8) line_tile<NT, 8, NJ, RG>(args, P, tile, smem);
    else if (F8 && P.codec == NVFP4) line_tile<NT, NVFP4, NJ, RG>(args, P, tile, smem);
    else if (P.codec == 4) line_tile<NT, 4, NJ, RG>(args, P, tile, smem);
    else line_tile<NT, 5, NJ, RG>(args, P, tile, smem);
}

template <int NT, int NJ, int RG, bool F8>
static cudaError_t launch_line_t(const SkinnyArgs &a, int grid, bool pdl, cudaStream_t stream) {
    static std::atomic<bool> done[64];
    constexpr int ST = F8 ? STAGE8 : STAGE;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int kw = a.G / NJ;
    if (!done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(skinny_line_kernel<NT, NJ, RG, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 LineSmem<NJ, RG, NT>::bytes(16, ST));
        if (e != cudaSuccess) return e;
        done[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kw * 32, 1, 1);
    cfg.dynamicSmemBytes = LineSmem<NJ, RG, NT>::bytes(kw, ST);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, skinny_line_kernel<NT, NJ, RG, F8>, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Groups per warp of the straight-line kernel that serves K / 64 = G groups
// (at most 16 warps per CTA): 8, all in flight, or 0 if none does.  (16
// groups per warp through an 8-stage ring measured slower and is gone.)
int skinny_line_groups(int G, int nj_pref) {
    if (nj_pref >= 8 && G % 8 == 0 && G / 8 <= 16) return 8;
    return 0;
}

template <bool F8>
static cudaError_t launch_line_f(const SkinnyArgs &a, int nt, int nj, int grid, bool pdl, cudaStream_t stream) {
    if (nj == 8 && a.G % 8 == 0 && a.G / 8 <= 16) {
        switch (nt) {
            case 1: return launch_line_t<1, 8, 8, F8>(a, grid, pdl, stream);
            case 2: return launch_line_t<2, 8, 8, F8>(a, grid, pdl, stream);
            case 4: return launch_line_t<4, 8, 8, F8>(a, grid, pdl, stream);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_skinny_line(const SkinnyArgs &a, int nt, int nj, int grid, bool pdl, bool f8,
                               cudaStream_t stream) {
    return f8 ? launch_line_f<true>(a, nt, nj, grid, pdl, stream) : launch_line_f<false>(a, nt, nj, grid, pdl, stream);
}

template <int NT, int KW, int ST>
static cudaError_t prepare(int dev) {
    static std::atomic<bool> done[64];
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(skinny_kernel<NT, KW, ST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SkinnySmem<NT, KW, ST>::BYTES);
    if (e != cudaSuccess) return e;
    done[dev].store(true, std::memory_order_release);
    return cudaSuccess;
}

template <int NT, int KW, int ST>
static cudaError_t launch_skinny_t(const SkinnyArgs &a, int grid, bool pdl, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if ((e = prepare<NT, KW, ST>(dev)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(KW * 32, 1, 1);
    cfg.dynamicSmemBytes = SkinnySmem<NT, KW, ST>::BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, skinny_kernel<NT, KW, ST>, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int ST>
static cudaError_t launch_skinny_s(const SkinnyArgs &a, int nt, int kw, int grid, bool pdl, cudaStream_t stream) {
    if (kw == 8) {
        switch (nt) {
            case 1: return launch_skinny_t<1, 8, ST>(a, grid, pdl, stream);
            case 2: return launch_skinny_t<2, 8, ST>(a, grid, pdl, stream);
            case 4: return launch_skinny_t<4, 8, ST>(a, grid, pdl, stream);
        }
    }
    return cudaErrorInvalidValue;
}

// Tokens per launch: 8 * nt with nt in {1, 2, 4}; kw = 8 warps per CTA;
// f8: some parent holds FP8 codes (larger stages).
cudaError_t launch_skinny(const SkinnyArgs &a, int nt, int kw, int grid, bool pdl, bool f8, cudaStream_t stream) {
    return f8 ? launch_skinny_s<STAGE8>(a, nt, kw, grid, pdl, stream)
              : launch_skinny_s<STAGE>(a, nt, kw, grid, pdl, stream);
}

}  // namespace qg
