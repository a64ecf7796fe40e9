// Internal definitions shared by the qgemm CUDA translation units: the packed
// device layout, kernel parameter blocks and small PTX wrappers (mbarrier,
// bulk async copies, bf16 tensor-core MMA).
//
// Packed device layout ("units").  Rows are grouped in blocks of 128 (eight
// 16-row tiles); K in groups of 64.  Unit (b, g) holds block b's 128 x 64 codes
// and their 128 scales, and units are stored block-major:
//     offset(b, g) = (b * G + g) * UNIT_BYTES(codec)
// so the units of one block and a run of groups are one contiguous span, which
// a kernel streams with a few bulk copies.  Inside a unit:
//   [nibble plane: 8 tiles x 32 lanes x 16 B][int5 only: high-bit plane:
//    8 tiles x 32 lanes x 4 B][scales: 8 tiles x 8 pairs x 2 x fp16]
// Lane l = 4*g + c of tile w owns rows r0 = 16w + g and r1 = r0 + 8 and the 16
// consecutive k = 16c .. 16c+15 of the group:
//   word 0: r0, k 16c+0..7    word 1: r0, k 16c+8..15
//   word 2: r1, k 16c+0..7    word 3: r1, k 16c+8..15
// Inside a word, k offset j sits in nibble position (j >> 1) + 4 * (j & 1), so
// nibble positions (i, i+4) hold the k pair (2i, 2i+1): masking the word
// shifted right by 4i with 0x000F000F yields that pair in the two 16-bit
// halves.  Nibbles hold the biased code u = q + 8 (int4) or the low 4 bits of
// u = q + 16 (int5).  The int5 high bit of word m, nibble position p sits in
// bit 4m + p (p < 4) or 16 + 4m + (p - 4) (p >= 4) of the lane's high word.
// Scale pair i of tile w is (s[16w + i], s[16w + i + 8]).
// Rows n >= N (padding of the last block) hold u = bias (q = 0) and s = 0.
//
// FP8 (E4M3) units: the lane's chunk is 32 bytes, row r0's 16 codes (k 16c ..
// 16c+15) in words 0..3 and row r1's in words 4..7; word j of a row holds k
// = 4j .. 4j+3 in byte order (4j, 4j+2, 4j+1, 4j+3), so that the k pair
// (4j, 4j+1) sits in bytes 0 and 2 and (4j+2, 4j+3) in bytes 1 and 3.  The
// code plane (8 tiles x 1024 B) is followed by the scales as above.  Padding
// rows hold code 0 (+0.0) and s = 0.
//
// NVFP4 units: the nibble plane as for int4, holding the raw E2M1 codes (no
// bias; padding rows hold code 0, +0.0), then the UE4M3 block scales: 8 tiles
// x 32 lanes x 2 B, lane l = 4g + c of tile w holding the scale bytes of rows
// r0 and r1 for the lane's 16 columns (block c of the group).  The fp32
// tensor scale travels with the launch and takes the place of the per-group
// rescale.
//
// Decode: OR a biased code into the mantissa of bf16 128.0 (0x4300; the
// mantissa of [128, 256) counts in steps of 1) and subtract 128 + bias: the
// result is the exact integer q as bf16, with no integer-to-float conversion.
// This is the magic-number conversion the Q4 small-T MMA of "ninfer-3080
// docs/performance.md" (small-T kernels section) describes.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qg {

constexpr int GROUP = 64;
constexpr int BLOCK_ROWS = 128;
constexpr int TILES = 8;                   // 16-row tiles per block
constexpr int NIB_BYTES = 4096;            // nibble plane of a unit
constexpr int HI_BYTES = 1024;             // int5 high-bit plane of a unit
constexpr int SCALE_BYTES = 256;           // 128 fp16 scales
constexpr int UNIT4 = NIB_BYTES + SCALE_BYTES;
constexpr int UNIT5 = NIB_BYTES + HI_BYTES + SCALE_BYTES;
constexpr int CODE8_BYTES = 8192;          // fp8 code plane of a unit: 8 tiles x 32 lanes x 32 B
constexpr int UNIT8 = CODE8_BYTES + SCALE_BYTES;
constexpr int NVFP4 = 16;                  // codec id of NVFP4 weights
constexpr int BS_BYTES = 512;              // NVFP4 block scales of a unit: 8 tiles x 32 lanes x 2 B
constexpr int UNIT16 = NIB_BYTES + BS_BYTES;

__host__ __device__ constexpr int unit_bytes(int codec) {
    return codec == NVFP4 ? UNIT16 : codec == 8 ? UNIT8 : codec == 5 ? UNIT5 : UNIT4;
}
// offset of the scales in a unit (the block scales for NVFP4)
__host__ __device__ constexpr int scale_off(int codec) {
    return codec == 8 ? CODE8_BYTES : codec == 5 ? NIB_BYTES + HI_BYTES : NIB_BYTES;
}

// nibble position of k offset j (0..7) inside a code word
__host__ __device__ constexpr int nib_pos(int j) { return (j >> 1) + 4 * (j & 1); }
// bit of the lane's high word holding the int5 high bit of word m, nibble position p
__host__ __device__ constexpr int hi_bit(int m, int p) { return p < 4 ? 4 * m + p : 16 + 4 * m + (p - 4); }

// ---------------------------------------------------------------- device status

// Kernels receive the address of the library's device status word and set it
// to QGEMM_ERR_TIMEOUT when a bounded wait gives up.

constexpr long long SPIN_LIMIT = 1ll << 16;   // tries of one mbarrier wait
constexpr uint32_t SUSPEND_HINT_NS = 20000;    // at most ~1.3 s per wait in total

// ---------------------------------------------------------------- kernel parameters

constexpr int MAX_PARENTS = 4;

// Fused outputs (qgemm_epilogue): what the kernels do where they write Y.
enum : int { EPI_STORE = 0, EPI_ADD = 1, EPI_SWIGLU = 2 };

struct SkinnyParent {
    const uint8_t *packed;   // units of this parent
    void *Y;                 // [T][ncols], fp32 or bf16
    const float *R;          // EPI_ADD: residual [T][ncols]
    float tscale;            // NVFP4: the tensor scale (in place of the group scales)
    int N, codec;            // N: packed rows
    int cta_begin;           // first CTA of this parent in the grid
    int ncols;               // columns of Y: N, or F of a SwiGLU pair (N = pair_rows(F))
    int epi, ybf16;
};

// The grid has one CTA per 16-row tile of every parent (ceil(N/16) each).
struct SkinnyArgs {
    SkinnyParent p[MAX_PARENTS];
    int nparents;
    const __nv_bfloat16 *X;  // [T][K]
    int T, K, G;
    unsigned int *status;    // device status word
};

// The wide route covers ceil(N/128) x ceil(T/BN) output tiles per parent
// (BN = 32, 64, 128 or 256 tokens).
struct WideParent {
    const uint8_t *packed;   // units of this parent
    void *Y;                 // [T][ncols], fp32 or bf16
    const float *R;          // EPI_ADD: residual [T][ncols]
    unsigned int *cnt;       // this parent's split-tile counters (zero between runs)
    float tscale;            // NVFP4: the tensor scale (in place of the group scales)
    int N, codec;            // N: packed rows
    int cta_begin;           // first output tile of this parent in its launch
    int nblocks;             // 128-row blocks
    int ncols, epi, ybf16;   // as in SkinnyParent
};

// Where a kernel has the fp32 value v of Y[t][col] (its row `col` of the
// packed matrix for STORE and ADD): apply the residual and store it in the
// output type.  SwiGLU outputs go through swiglu_out with their gate and up
// values.
__device__ __forceinline__ void store_y(void *Y, int ybf16, size_t idx, float v) {
    if (ybf16) reinterpret_cast<__nv_bfloat16 *>(Y)[idx] = __float2bfloat16_rn(v);
    else reinterpret_cast<float *>(Y)[idx] = v;
}

template <class P>
__device__ __forceinline__ void epi_out(const P &p, int t, int col, float v) {
    const size_t idx = (size_t)t * p.ncols + col;
    if (p.epi == EPI_ADD) v = p.R[idx] + v;
    store_y(p.Y, p.ybf16, idx, v);
}

// silu(g) * u = g / (1 + e^-g) * u, in fp32.
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// SwiGLU pair layout: packed row 16 b + i holds gate row 8 b + i (i < 8) and
// packed row 16 b + 8 + i the up row 8 b + i.
__host__ __device__ constexpr int pair_rows(int F) { return 16 * ((F + 7) / 8); }

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Test of the phase with the given parity.  If the phase is not complete the
// thread is suspended in hardware until it completes or the hint (in ns)
// expires, instead of spinning: many waiting warps polling shared memory in a
// loop slowed every barrier access of the kernel's critical thread.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(SUSPEND_HINT_NS) : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false (and the device
// status set to timeout) if it did not complete within SPIN_LIMIT tries.  A
// phase that has already completed is seen by the non-blocking test, which
// is cheaper than the suspending form.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, unsigned int *status,
                                                long long limit) {
    if (mbar_test(bar, parity)) return true;
    for (long long i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicExch(status, 7u /* QGEMM_ERR_TIMEOUT */);
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned int *status) {
    return mbar_wait_limit(bar, parity, status, SPIN_LIMIT);
}

// One lane of a converged warp: true in exactly one lane.
__device__ __forceinline__ bool elect_one() {
    uint32_t p;
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
    return p != 0;
}

// Bounded wait for two phases; the two non-blocking tests are issued together
// so that two completed phases cost one round trip.
__device__ __forceinline__ bool mbar_wait2(uint64_t *bar0, uint32_t parity0, uint64_t *bar1, uint32_t parity1,
                                           unsigned int *status) {
    const bool r0 = mbar_test(bar0, parity0);
    const bool r1 = mbar_test(bar1, parity1);
    if (r0 && r1) return true;
    return (r0 || mbar_wait(bar0, parity0, status)) && (r1 || mbar_wait(bar1, parity1, status));
}

// Bounded wait by every lane of a converged warp; the result is the same in
// all lanes (false if any lane gave up), so the warp stays converged.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, unsigned int *status) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// 16-byte asynchronous global -> shared copy (L2 only), committed in groups.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A load with acquire semantics at GPU scope: the writes other CTAs made
// before their release on this word (a fence, then an atomic) are visible
// after it.
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// 1-D bulk async copy global -> shared, completion counted on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// D = A * B + C, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], const uint32_t b[2],
                                               const float c[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]),
          "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// ---- programmatic dependent launch

// Let the next kernel in the stream start launching its CTAs.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the previous kernel in the stream has completed and its memory
// is visible (a no-op when launched without a programmatic dependency).
__device__ __forceinline__ void pdl_wait_prior() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// bf16x2 subtract (exact here: both halves are small integers)
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (a & b) | c as one three-input logic instruction (truth table 0xEA); the
// compiler otherwise splits the mask and the OR of two constants into two.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Codes (i, i+4) of a nibble word as an exact bf16x2 pair of integers.
template <int SHIFT>
__device__ __forceinline__ uint32_t dec4_pair(uint32_t w) {
    return bf16x2_sub(and_or(w >> SHIFT, 0x000F000Fu, 0x43004300u), 0x43084308u);   // - (128 + 8)
}

// FP8: two E4M3 codes as an exact bf16x2 pair.  An E4M3 code's 7 magnitude
// bits placed at bf16 bits 4..10 (exponent field = the code's exponent,
// mantissa = its 3 bits) read as the code's value times 2^-120, subnormal
// codes included; the sign goes to bit 15, and one bf16x2 multiply by 2^120
// (exact: a power of two, results in the normal range) gives the value.
// Codes in bytes 0 and 2 of w (SHI = 0) or in bytes 1 and 3 (SHI = 1).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

template <int SHI>
__device__ __forceinline__ uint32_t dec8_pair(uint32_t w) {
    const uint32_t mag = (SHI ? (w >> 4) : (w << 4)) & 0x07F007F0u;
    const uint32_t sgn = SHI ? w : (w << 8);
    return bf16x2_mul(and_or(sgn, 0x80008000u, mag), 0x7B807B80u);   // x 2^120
}

// NVFP4: two E2M1 codes (nibble positions I and I + 4 of w, the k pair
// (2I, 2I + 1)) times the block scale pair bs2, as an exact bf16x2 pair.  A
// code's exponent and mantissa bits placed at bf16 bits 6..8 read as the
// code's value times 2^-126 (the subnormal code included: bf16's own
// subnormal), its sign goes to bit 15; one bf16x2 multiply by 2^126 and one
// by the block scale give the value (E2M1 has 2 significant bits, UE4M3 4: the
// product is exact, between 2^-10 and 2688).
template <int I>
__device__ __forceinline__ uint32_t dec16_pair(uint32_t w, uint32_t bs2) {
    constexpr int MS = 6 - 4 * I, SS = 12 - 4 * I;   // shifts of the magnitude and sign bits
    const uint32_t mag = (MS >= 0 ? (w << MS) : (w >> (-MS))) & 0x01C001C0u;
    const uint32_t sgn = w << SS;
    return bf16x2_mul(bf16x2_mul(and_or(sgn, 0x80008000u, mag), 0x7E807E80u), bs2);   // x 2^126, x scale
}

// Two UE4M3 block-scale bytes (bits 0..7 and 8..15 of b) as a bf16x2 pair:
// the code's 7 bits at bf16 bits 4..10 read as its value times 2^-120.
__device__ __forceinline__ uint32_t ue4m3x2_to_bf16x2(uint32_t b) {
    const uint32_t lo = b & 0xFFu, hi = (b >> 8) & 0xFFu;
    return bf16x2_mul(((lo << 4) | (hi << 20)) & 0x07F007F0u, 0x7B807B80u);   // x 2^120
}

// int5: nibble pair plus the two high bits taken from the lane's high word.
template <int SHIFT, int HSH>
__device__ __forceinline__ uint32_t dec5_pair(uint32_t w, uint32_t h) {
    const uint32_t hm = and_or(HSH >= 0 ? (h >> HSH) : (h << (-HSH)), 0x00100010u, 0x43004300u);
    return bf16x2_sub(and_or(w >> SHIFT, 0x000F000Fu, hm), 0x43104310u);   // - (128 + 16)
}

}  // namespace qg
