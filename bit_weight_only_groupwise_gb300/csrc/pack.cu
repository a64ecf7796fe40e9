// Repack canonical int4/int5 codes and fp16 scales into the unit layout
// described in qgemm_internal.cuh.  One CTA per unit (block b, group grp), one
// thread per (tile, lane): each thread builds one lane's 16-byte code chunk,
// its int5 high word, and (lanes with c == 0) one scale pair.
//
// A SwiGLU pair (gate and up, F rows each) is packed as one matrix of
// pair_rows(F) rows whose 16-row tiles hold 8 gate rows and then the same 8
// up rows: packed row 16 b + 8 h + i is row 8 b + i of the gate (h = 0) or of
// the up matrix (h = 1), so that the lane owning rows g and g + 8 of a tile
// holds the gate and the up value of one output.
#include "qgemm_internal.cuh"

namespace qg {

// Source of packed row `row`: the matrix (0: the plain or gate matrix, 1: the
// up matrix) and its row, or row -1 for padding.
struct SrcRow { int which, row; };

__device__ __forceinline__ SrcRow src_row(int row, int N, int F) {
    if (F == 0) return {0, row < N ? row : -1};
    const int f = (row >> 4) * 8 + (row & 7);
    return {(row >> 3) & 1, f < F ? f : -1};
}

__global__ void __launch_bounds__(256) pack_kernel(int codec, int N, int K, const uint8_t *__restrict__ canon,
                                                   const uint16_t *__restrict__ scales,
                                                   const uint8_t *__restrict__ canon_up,
                                                   const uint16_t *__restrict__ scales_up, int F,
                                                   uint8_t *__restrict__ out) {
    const int G = K / GROUP;
    const int unit = blockIdx.x;            // b * G + grp
    const int b = unit / G, grp = unit % G;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int UB = unit_bytes(codec);
    uint8_t *u = out + (size_t)unit * UB;

    if (codec == 8) {
        // E4M3 codes: the lane's 32-byte chunk, row r0 then row r1, each word
        // holding k = 4j .. 4j+3 in byte order (4j, 4j+2, 4j+1, 4j+3)
        uint32_t w8[8];
        for (int half = 0; half < 2; ++half) {
            const SrcRow sr = src_row(b * BLOCK_ROWS + 16 * w + g + 8 * half, N, F);
            const uint8_t *src = (sr.which ? canon_up : canon) + (size_t)(sr.row < 0 ? 0 : sr.row) * K +
                                 grp * GROUP + 16 * c;
            for (int j = 0; j < 4; ++j) {
                uint32_t v = 0;
                if (sr.row >= 0)
                    v = (uint32_t)src[4 * j] | ((uint32_t)src[4 * j + 2] << 8) | ((uint32_t)src[4 * j + 1] << 16) |
                        ((uint32_t)src[4 * j + 3] << 24);
                w8[4 * half + j] = v;
            }
        }
        *reinterpret_cast<uint4 *>(u + w * 1024 + lane * 32) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
        *reinterpret_cast<uint4 *>(u + w * 1024 + lane * 32 + 16) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
    } else {
    uint32_t words[4] = {0, 0, 0, 0};
    uint32_t hi = 0;
    for (int half = 0; half < 2; ++half) {          // rows r0 and r0 + 8
        const SrcRow sr = src_row(b * BLOCK_ROWS + 16 * w + g + 8 * half, N, F);
        const int row = sr.row;
        const uint8_t *src = sr.which ? canon_up : canon;
        const int k0 = grp * GROUP + 16 * c;
        for (int j = 0; j < 16; ++j) {
            int ub;                                   // biased code (NVFP4: the raw E2M1 code)
            if (row < 0) {
                ub = codec == 5 ? 16 : codec == NVFP4 ? 0 : 8;
            } else if (codec == NVFP4) {
                const uint8_t byte = src[(size_t)row * (K / 2) + (k0 + j) / 2];
                ub = ((k0 + j) & 1) ? (byte >> 4) : (byte & 15);
            } else if (codec == 4) {
                const uint8_t byte = src[(size_t)row * (K / 2) + (k0 + j) / 2];
                const int nib = ((k0 + j) & 1) ? (byte >> 4) : (byte & 15);
                ub = nib ^ 8;                         // two's complement nibble -> q + 8
            } else {
                const size_t rowbits = (size_t)row * (size_t)(5 * K);
                int v = 0;
                for (int t = 0; t < 5; ++t) {
                    const size_t p = rowbits + (size_t)5 * (k0 + j) + t;
                    v |= ((src[p >> 3] >> (p & 7)) & 1) << t;
                }
                ub = v ^ 16;                          // two's complement 5-bit field -> q + 16
            }
            const int m = 2 * half + (j >> 3);        // word index
            const int pos = nib_pos(j & 7);
            words[m] |= (uint32_t)(ub & 15) << (4 * pos);
            if (codec == 5) hi |= (uint32_t)((ub >> 4) & 1) << hi_bit(m, pos);
        }
    }
    *reinterpret_cast<uint4 *>(u + w * 512 + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
    if (codec == 5) *reinterpret_cast<uint32_t *>(u + NIB_BYTES + w * 128 + lane * 4) = hi;
    }
    if (codec == NVFP4) {
        // the lane's block (c) of rows r0 and r1: UE4M3 bytes [rows][K/16]
        const uint8_t *bs = reinterpret_cast<const uint8_t *>(scales);
        const uint8_t *bs_up = reinterpret_cast<const uint8_t *>(scales_up);
        const int KB = K / 16;
        const SrcRow a0 = src_row(b * BLOCK_ROWS + 16 * w + g, N, F);
        const SrcRow a1 = src_row(b * BLOCK_ROWS + 16 * w + g + 8, N, F);
        const uint32_t b0 = a0.row >= 0 ? (a0.which ? bs_up : bs)[(size_t)a0.row * KB + grp * 4 + c] : 0;
        const uint32_t b1 = a1.row >= 0 ? (a1.which ? bs_up : bs)[(size_t)a1.row * KB + grp * 4 + c] : 0;
        *reinterpret_cast<uint16_t *>(u + NIB_BYTES + w * 64 + lane * 2) = (uint16_t)(b0 | (b1 << 8));
    } else if (c == 0) {
        const SrcRow a0 = src_row(b * BLOCK_ROWS + 16 * w + g, N, F);
        const SrcRow a1 = src_row(b * BLOCK_ROWS + 16 * w + g + 8, N, F);
        const uint16_t s0 = a0.row >= 0 ? (a0.which ? scales_up : scales)[(size_t)a0.row * G + grp] : 0;
        const uint16_t s1 = a1.row >= 0 ? (a1.which ? scales_up : scales)[(size_t)a1.row * G + grp] : 0;
        *reinterpret_cast<uint32_t *>(u + scale_off(codec) + w * 32 + g * 4) = (uint32_t)s0 | ((uint32_t)s1 << 16);
    }
}

cudaError_t launch_pack(int codec, int N, int K, const void *canon, const uint16_t *scales, void *out,
                        cudaStream_t stream) {
    const int NB = (N + BLOCK_ROWS - 1) / BLOCK_ROWS;
    const int G = K / GROUP;
    pack_kernel<<<NB * G, 256, 0, stream>>>(codec, N, K, static_cast<const uint8_t *>(canon), scales, nullptr,
                                            nullptr, 0, static_cast<uint8_t *>(out));
    return cudaGetLastError();
}

cudaError_t launch_pack_pair(int codec, int F, int K, const void *gate, const uint16_t *gate_scales,
                             const void *up, const uint16_t *up_scales, void *out, cudaStream_t stream) {
    const int N = pair_rows(F);
    const int NB = (N + BLOCK_ROWS - 1) / BLOCK_ROWS;
    const int G = K / GROUP;
    pack_kernel<<<NB * G, 256, 0, stream>>>(codec, N, K, static_cast<const uint8_t *>(gate), gate_scales,
                                            static_cast<const uint8_t *>(up), up_scales, F,
                                            static_cast<uint8_t *>(out));
    return cudaGetLastError();
}

__global__ void fence_kernel() {}

// Diagnostic: one bounded wait on an mbarrier that nothing arrives at, the
// path every kernel takes when a wait runs out (device status set to
// timeout, the thread returns).  `tries` suspending tests of at most ~20 us.
__global__ void wait_timeout_kernel(unsigned int *status, int tries) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait_limit(&bar, 0, status, tries);
    }
}

cudaError_t launch_wait_timeout(unsigned int *status, int tries, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, tries);
    return cudaGetLastError();
}

cudaError_t launch_fence(cudaStream_t stream) {
    fence_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

}  // namespace qg
