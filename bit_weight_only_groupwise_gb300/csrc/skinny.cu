// Small-T route: a weight-streaming split-K skinny GEMM.
//
// At decode and verify widths the operation streams the whole weight matrix
// once for a handful of token columns, so HBM bandwidth bounds it ("ninfer-3080
// docs/performance.md": the small-T kernels section measures its Q4/Q5
// kernels against the streaming floor, and the route boundaries section notes
// that cold weight streaming is the production regime).  The design:
//
// * grid: one CTA per (128-row block b, K split s); each CTA's units form one
//   contiguous span of the packed buffer, streamed by a producer warp with
//   1-D bulk async copies (cp.async.bulk) into a ring of unit-sized stages;
// * eight consumer warps, one per 16-row tile, decode their lane's 16 codes
//   per row in registers (magic-number bf16 decode) and run bf16 m16n8k16
//   tensor-core MMAs against the activation fragments, whose k order is
//   permuted the same way as the codes (any permutation inside a group is
//   valid when A and B agree -- the small-T kernels section's permuted k order);
// * each 64-column group's fp32 partial is multiplied by its fp16 scale and
//   added to the fp32 accumulator (the per-group rescale of the token-tile
//   section's ablation): scale * code is never rounded;
// * split-K combine: every split writes its [T][128] partial to the
//   workspace; the last CTA to arrive at the block's counter sums the
//   partials in split order and writes Y -- deterministic, with no spin.
#include "qgemm_internal.cuh"

namespace qg {

constexpr int STAGES = 8;
constexpr int RED_STRIDE = 132;   // floats per token row of the reduction tile (bank spread)

template <int NT>
struct SkinnySmem {
    static constexpr int RING = STAGES * UNIT5;
    static constexpr int RED = NT * 8 * RED_STRIDE * 4;
    static_assert(RED <= RING, "reduction tile reuses the ring");
    static constexpr int BYTES = RING + 2 * STAGES * 8 + 16;
};

template <int NT>
__global__ void __launch_bounds__(288) skinny_kernel(const __grid_constant__ SkinnyArgs args) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + SkinnySmem<NT>::RING);
    uint64_t *empty = full + STAGES;
    volatile int *flag = reinterpret_cast<volatile int *>(empty + STAGES);

    // ---- which parent, block and split this CTA owns
    int pi = 0;
#pragma unroll
    for (int i = 1; i < MAX_PARENTS; ++i)
        if (i < args.nparents && (int)blockIdx.x >= args.p[i].cta_begin) pi = i;
    const SkinnyParent &P = args.p[pi];
    const int local = blockIdx.x - P.cta_begin;
    const int b = local / P.S, s = local % P.S;
    const int G = args.G;
    const int g0 = (int)(((long long)s * G) / P.S), g1 = (int)(((long long)(s + 1) * G) / P.S);
    const int ng = g1 - g0;
    const int codec = P.codec;
    const int UB = unit_bytes(codec);
    const uint8_t *src = P.packed + ((size_t)b * G + g0) * UB;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int T = args.T;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 8);
        }
        *flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    bool ok = true;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

    if (warp == 8) {
        // ---------------- producer: stream the CTA's contiguous span of units
        if (lane == 0) {
            for (int i = 0; i < ng && ok; ++i) {
                const int slot = i % STAGES;
                if (i >= STAGES) ok = mbar_wait(&empty[slot], ((i / STAGES) - 1) & 1, args.status);
                if (!ok) break;
                mbar_arrive_expect_tx(&full[slot], UB);
                bulk_g2s(ring + slot * UNIT5, src + (size_t)i * UB, UB, &full[slot]);
            }
            // every issued copy has landed before the CTA may leave
            for (int i = ng - STAGES > 0 ? ng - STAGES : 0; i < ng && ok; ++i)
                ok = mbar_wait(&full[i % STAGES], (i / STAGES) & 1, args.status);
            if (!ok) *flag = 1;
        }
    } else {
        // ---------------- consumer warp: 16-row tile `warp`
        const int w = warp;
        for (int i = 0; i < ng; ++i) {
            const int slot = i % STAGES;
            // activation fragments do not depend on the stage: issue them first
            const int k0 = (g0 + i) * GROUP + 16 * c;
            uint32_t xb[NT][8];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int tok = nt * 8 + g;
                if (tok < T) {
                    const uint4 *xp = reinterpret_cast<const uint4 *>(args.X + (size_t)tok * args.K + k0);
                    const uint4 v0 = __ldg(xp), v1 = __ldg(xp + 1);
                    xb[nt][0] = v0.x; xb[nt][1] = v0.y; xb[nt][2] = v0.z; xb[nt][3] = v0.w;
                    xb[nt][4] = v1.x; xb[nt][5] = v1.y; xb[nt][6] = v1.z; xb[nt][7] = v1.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xb[nt][e] = 0u;
                }
            }
            if (!mbar_wait(&full[slot], (i / STAGES) & 1, args.status)) { ok = false; break; }
            const uint8_t *u = ring + slot * UNIT5;
            const uint4 cw = *reinterpret_cast<const uint4 *>(u + w * 512 + lane * 16);
            const uint32_t hw = codec == 5 ? *reinterpret_cast<const uint32_t *>(u + NIB_BYTES + w * 128 + lane * 4) : 0u;
            const uint32_t sp = *reinterpret_cast<const uint32_t *>(u + scale_off(codec) + w * 32 + g * 4);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);

            // decode: a[j] = A fragment of k16 step j (rows g / g+8, k 16c + 4j .. 4j+3)
            uint32_t a[4][4];
            if (codec == 4) {
                a[0][0] = dec4_pair<0>(cw.x);  a[0][1] = dec4_pair<0>(cw.z);  a[0][2] = dec4_pair<4>(cw.x);  a[0][3] = dec4_pair<4>(cw.z);
                a[1][0] = dec4_pair<8>(cw.x);  a[1][1] = dec4_pair<8>(cw.z);  a[1][2] = dec4_pair<12>(cw.x); a[1][3] = dec4_pair<12>(cw.z);
                a[2][0] = dec4_pair<0>(cw.y);  a[2][1] = dec4_pair<0>(cw.w);  a[2][2] = dec4_pair<4>(cw.y);  a[2][3] = dec4_pair<4>(cw.w);
                a[3][0] = dec4_pair<8>(cw.y);  a[3][1] = dec4_pair<8>(cw.w);  a[3][2] = dec4_pair<12>(cw.y); a[3][3] = dec4_pair<12>(cw.w);
            } else {
                // word m: 0 = cw.x, 1 = cw.y (row g); 2 = cw.z, 3 = cw.w (row g+8); HSH = 4m + i - 4
                a[0][0] = dec5_pair<0, -4>(cw.x, hw);  a[0][1] = dec5_pair<0, 4>(cw.z, hw);
                a[0][2] = dec5_pair<4, -3>(cw.x, hw);  a[0][3] = dec5_pair<4, 5>(cw.z, hw);
                a[1][0] = dec5_pair<8, -2>(cw.x, hw);  a[1][1] = dec5_pair<8, 6>(cw.z, hw);
                a[1][2] = dec5_pair<12, -1>(cw.x, hw); a[1][3] = dec5_pair<12, 7>(cw.z, hw);
                a[2][0] = dec5_pair<0, 0>(cw.y, hw);   a[2][1] = dec5_pair<0, 8>(cw.w, hw);
                a[2][2] = dec5_pair<4, 1>(cw.y, hw);   a[2][3] = dec5_pair<4, 9>(cw.w, hw);
                a[3][0] = dec5_pair<8, 2>(cw.y, hw);   a[3][1] = dec5_pair<8, 10>(cw.w, hw);
                a[3][2] = dec5_pair<12, 3>(cw.y, hw);  a[3][3] = dec5_pair<12, 11>(cw.w, hw);
            }
            const float2 sc = __half22float2(*reinterpret_cast<const __half2 *>(&sp));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t bf[2] = {xb[nt][2 * j], xb[nt][2 * j + 1]};
                    mma_bf16_16816(p, a[j], bf, p);
                }
                acc[nt][0] = fmaf(sc.x, p[0], acc[nt][0]);
                acc[nt][1] = fmaf(sc.x, p[1], acc[nt][1]);
                acc[nt][2] = fmaf(sc.y, p[2], acc[nt][2]);
                acc[nt][3] = fmaf(sc.y, p[3], acc[nt][3]);
            }
        }
        if (!ok) *flag = 1;
    }
    __syncthreads();
    const bool cta_ok = (*flag == 0);

    // ---------------- stage the CTA's [T][128] result in shared memory
    float *red = reinterpret_cast<float *>(ring);
    if (warp < 8) {
        const int r = 16 * warp + g;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int t = nt * 8 + 2 * c;
            red[t * RED_STRIDE + r] = acc[nt][0];
            red[(t + 1) * RED_STRIDE + r] = acc[nt][1];
            red[t * RED_STRIDE + r + 8] = acc[nt][2];
            red[(t + 1) * RED_STRIDE + r + 8] = acc[nt][3];
        }
    }
    __syncthreads();
    if (!cta_ok) return;

    const int n0 = b * BLOCK_ROWS;
    const int rows = min(BLOCK_ROWS, P.N - n0);
    const int nthreads = blockDim.x;
    if (P.S == 1) {
        for (int e = threadIdx.x; e < T * BLOCK_ROWS; e += nthreads) {
            const int t = e >> 7, r = e & 127;
            if (r < rows) P.Y[(size_t)t * P.N + n0 + r] = red[t * RED_STRIDE + r];
        }
        return;
    }

    // ---------------- split-K: publish the partial, the last arriver sums in split order
    const int tpad = NT * 8;
    float *mine = P.partials + ((size_t)(b * P.S + s) * tpad) * BLOCK_ROWS;
    for (int e = threadIdx.x; e < T * BLOCK_ROWS; e += nthreads) {
        const int t = e >> 7, r = e & 127;
        mine[t * BLOCK_ROWS + r] = red[t * RED_STRIDE + r];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(&P.counters[b], 1u);
        *flag = (prev == (unsigned)(P.S - 1)) ? 2 : 0;
    }
    __syncthreads();
    if (*flag != 2) return;
    __threadfence();
    for (int e = threadIdx.x; e < T * BLOCK_ROWS; e += nthreads) {
        const int t = e >> 7, r = e & 127;
        float v = 0.f;
        for (int ss = 0; ss < P.S; ++ss) {
            const float part = (ss == s) ? red[t * RED_STRIDE + r]
                                         : __ldcg(P.partials + ((size_t)(b * P.S + ss) * tpad + t) * BLOCK_ROWS + r);
            v += part;
        }
        if (r < rows) P.Y[(size_t)t * P.N + n0 + r] = v;
    }
    if (threadIdx.x == 0) P.counters[b] = 0u;   // ready for the next call
}

template <int NT>
static cudaError_t launch_skinny_nt(const SkinnyArgs &a, int grid, cudaStream_t stream) {
    const int bytes = SkinnySmem<NT>::BYTES;
    static bool attr_set[64] = {};   // per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(skinny_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    skinny_kernel<NT><<<grid, 288, bytes, stream>>>(a);
    return cudaGetLastError();
}

// Tokens per launch of the skinny kernel: 8 * NT with NT in {1, 2, 4}.
cudaError_t launch_skinny(const SkinnyArgs &a, int nt, int grid, cudaStream_t stream) {
    switch (nt) {
        case 1: return launch_skinny_nt<1>(a, grid, stream);
        case 2: return launch_skinny_nt<2>(a, grid, stream);
        case 4: return launch_skinny_nt<4>(a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
