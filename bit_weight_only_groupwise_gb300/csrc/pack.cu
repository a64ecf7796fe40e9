// Repack canonical int4/int5 codes and fp16 scales into the unit layout
// described in qgemm_internal.cuh.  One CTA per unit (block b, group grp), one
// thread per (tile, lane): each thread builds one lane's 16-byte code chunk,
// its int5 high word, and (lanes with c == 0) one scale pair.
#include "qgemm_internal.cuh"

namespace qg {

__global__ void __launch_bounds__(256) pack_kernel(int codec, int N, int K, const uint8_t *__restrict__ canon,
                                                   const uint16_t *__restrict__ scales, uint8_t *__restrict__ out) {
    const int G = K / GROUP;
    const int unit = blockIdx.x;            // b * G + grp
    const int b = unit / G, grp = unit % G;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int UB = unit_bytes(codec);
    uint8_t *u = out + (size_t)unit * UB;

    uint32_t words[4] = {0, 0, 0, 0};
    uint32_t hi = 0;
    for (int half = 0; half < 2; ++half) {          // rows r0 and r0 + 8
        const int row = b * BLOCK_ROWS + 16 * w + g + 8 * half;
        const int k0 = grp * GROUP + 16 * c;
        for (int j = 0; j < 16; ++j) {
            int ub;                                   // biased code
            if (row >= N) {
                ub = codec == 5 ? 16 : 8;
            } else if (codec == 4) {
                const uint8_t byte = canon[(size_t)row * (K / 2) + (k0 + j) / 2];
                const int nib = ((k0 + j) & 1) ? (byte >> 4) : (byte & 15);
                ub = nib ^ 8;                         // two's complement nibble -> q + 8
            } else {
                const size_t rowbits = (size_t)row * (size_t)(5 * K);
                int v = 0;
                for (int t = 0; t < 5; ++t) {
                    const size_t p = rowbits + (size_t)5 * (k0 + j) + t;
                    v |= ((canon[p >> 3] >> (p & 7)) & 1) << t;
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
    if (c == 0) {
        const int r0 = b * BLOCK_ROWS + 16 * w + g;
        const uint16_t s0 = r0 < N ? scales[(size_t)r0 * G + grp] : 0;
        const uint16_t s1 = r0 + 8 < N ? scales[(size_t)(r0 + 8) * G + grp] : 0;
        *reinterpret_cast<uint32_t *>(u + scale_off(codec) + w * 32 + g * 4) = (uint32_t)s0 | ((uint32_t)s1 << 16);
    }
}

cudaError_t launch_pack(int codec, int N, int K, const void *canon, const uint16_t *scales, void *out,
                        cudaStream_t stream) {
    const int NB = (N + BLOCK_ROWS - 1) / BLOCK_ROWS;
    const int G = K / GROUP;
    pack_kernel<<<NB * G, 256, 0, stream>>>(codec, N, K, static_cast<const uint8_t *>(canon), scales,
                                            static_cast<uint8_t *>(out));
    return cudaGetLastError();
}

__global__ void fence_kernel() {}

cudaError_t launch_fence(cudaStream_t stream) {
    fence_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

}  // namespace qg
