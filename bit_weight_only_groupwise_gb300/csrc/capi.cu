// C-ABI of the qgemm library: argument validation, plans, route choice and
// launches.  Declarations and the contract of every entry point are in
// include/qgemm.h.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <new>

#include "qgemm.h"
#include "qgemm_internal.cuh"

namespace qg {
cudaError_t launch_pack(int codec, int N, int K, const void *canon, const uint16_t *scales, void *out,
                        cudaStream_t stream);
cudaError_t launch_fence(cudaStream_t stream);
cudaError_t launch_wait_timeout(unsigned int *status, int tries, cudaStream_t stream);
cudaError_t launch_pack_pair(int codec, int F, int K, const void *gate, const uint16_t *gate_scales,
                             const void *up, const uint16_t *up_scales, void *out, cudaStream_t stream);
cudaError_t launch_skinny(const SkinnyArgs &a, int nt, int kw, int grid, bool pdl, bool f8, cudaStream_t stream);
int skinny_line_groups(int G, int nj_pref);
cudaError_t launch_skinny_line(const SkinnyArgs &a, int nt, int nj, int grid, bool pdl, bool f8,
                               cudaStream_t stream);
cudaError_t launch_wide(const WideParent *parents, int np, const void *X, int T, int K, int bh, int halves,
                        float *part, unsigned int *status, bool pdl, int sms, cudaStream_t stream);
size_t wide_workspace_bytes(int rows, int T_max, int sms);
size_t wide_partial_bytes(int T_max, int sms);
int wide_max_tokens(int T_max);
}  // namespace qg

using namespace qg;

// ---------------------------------------------------------------- routes

enum Route : int {
    ROUTE_SKINNY8 = 0,     // weight-streaming skinny GEMM, 8-token MMA tile
    ROUTE_SKINNY16 = 1,    // 16-token tile
    ROUTE_SKINNY32 = 2,    // 32-token tile
    ROUTE_WIDE128 = 3,     // stream-K tcgen05 tiles of 128 rows x 128 tokens
    ROUTE_WIDE256 = 4,     // stream-K tcgen05 tiles of 128 rows x 256 tokens (two 128-token halves)
    ROUTE_WIDE64 = 5,      // stream-K tcgen05 tiles of 128 rows x 64 tokens
    ROUTE_WIDE32 = 6,      // stream-K tcgen05 tiles of 128 rows x 32 tokens
    ROUTE_COUNT
};

static const char *kRouteNames[ROUTE_COUNT] = {"skinny8", "skinny16", "skinny32", "tcgen05_128x128",
                                               "tcgen05_128x256", "tcgen05_128x64", "tcgen05_128x32"};

static int route_tokens(int route) {
    switch (route) {
        case ROUTE_SKINNY8: return 8;
        case ROUTE_SKINNY16: return 16;
        case ROUTE_SKINNY32: return 32;
        case ROUTE_WIDE32: return 32;
        case ROUTE_WIDE64: return 64;
        case ROUTE_WIDE128: return 128;
        default: return 256;
    }
}

static bool wide_route(int route) {
    return route == ROUTE_WIDE32 || route == ROUTE_WIDE64 || route == ROUTE_WIDE128 || route == ROUTE_WIDE256;
}

// The route table, from per-T sweeps with every route forced on the pages'
// projection shapes (5120 x 6144, 7168 x 5120, 12288 x 5120; cold weights):
// the narrowest tile that covers T (the padded width sets the cost, not the
// live column count), except that the tcgen05 tiles beat the 32-token
// small-T tile from T = 17 on (the 32-token one to T = 32, 12-16% ahead of
// the 64-token one there), and that above 128 tokens the 256-token tile pays
// only from 512 tokens, or from 129 when the launch has at least 96 row
// blocks of 128 (enough tiles to fill the GPU either way).
// nb: the launch's 128-row blocks, summed over its parents.  A route forced
// on the plan (qgemm_plan_force_route) takes every T its token tile covers.
static int table_route(int T, int nb) {
    if (T <= 8) return ROUTE_SKINNY8;
    if (T <= 16) return ROUTE_SKINNY16;
    if (T <= 32) return ROUTE_WIDE32;
    if (T <= 64) return ROUTE_WIDE64;
    if (T <= 128) return ROUTE_WIDE128;
    return (T >= 512 || nb >= 96) ? ROUTE_WIDE256 : ROUTE_WIDE128;
}

// the tcgen05 routes walk any number of token tiles
static bool route_covers(int route, int T) { return wide_route(route) || T <= route_tokens(route); }

struct qgemm_plan_s {
    int N, K, codec, T_max;
    int rows;              // packed rows: N, or pair_rows(N) for a SwiGLU pair
    int epi, out;          // qgemm_epilogue, qgemm_out
    int G, NB, UB;
    int sms;
    bool pdl;              // launch with programmatic dependent launch
    int forced_route;      // -1: the route table; else qgemm_plan_force_route's route
    float tscale;          // NVFP4: the tensor scale (qgemm_plan_set_tensor_scale)
    size_t ws_bytes;       // workspace the plan's routes need (the tcgen05 routes' split tiles)
    size_t ws_part;        // of it, the partial-sum slots (the counters follow)
    const uint8_t *packed;
    uint8_t *ws;
    bool bound;
};

static int choose_route(const qgemm_plan_s *p, int T, int nb) {
    return (p->forced_route >= 0 && route_covers(p->forced_route, T)) ? p->forced_route : table_route(T, nb);
}

static std::atomic<uint64_t> g_launches{0};

// Device status word (QGEMM_OK or QGEMM_ERR_TIMEOUT); kernels get its address.
__device__ unsigned int g_device_status = 0;

// Address of the status word on the current device, looked up once per device
// (the lookup is not a stream operation, so later calls may be captured).
static unsigned int *status_ptr() {
    constexpr int MAX_DEVICES = 64;
    static std::atomic<unsigned int *> cache[MAX_DEVICES];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return nullptr;
    }
    unsigned int *p = cache[dev].load();
    if (p) return p;
    void *raw = nullptr;
    if (cudaGetSymbolAddress(&raw, g_device_status) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    cache[dev].store(static_cast<unsigned int *>(raw));
    return static_cast<unsigned int *>(raw);
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool valid_codec(int c) { return c == QGEMM_INT4 || c == QGEMM_INT5 || c == QGEMM_FP8 || c == QGEMM_NVFP4; }

extern "C" {

const char *qgemm_status_string(qgemm_status st) {
    switch (st) {
        case QGEMM_OK: return "ok";
        case QGEMM_ERR_INVALID_ARG: return "invalid argument";
        case QGEMM_ERR_SHAPE: return "invalid shape";
        case QGEMM_ERR_ALIGNMENT: return "buffer not 16-byte aligned";
        case QGEMM_ERR_T_OUT_OF_DOMAIN: return "T outside the plan's domain";
        case QGEMM_ERR_WORKSPACE: return "workspace missing or too small";
        case QGEMM_ERR_CUDA: return "CUDA error";
        case QGEMM_ERR_TIMEOUT: return "device-side wait timed out";
        case QGEMM_ERR_UNSUPPORTED: return "no supported GPU";
    }
    return "unknown status";
}

size_t qgemm_packed_bytes(int N, int K, qgemm_codec codec) {
    if (!valid_codec(codec) || N < 1 || K < GROUP || K % GROUP) return 0;
    const size_t NB = (size_t)(N + BLOCK_ROWS - 1) / BLOCK_ROWS;
    return NB * (size_t)(K / GROUP) * (size_t)unit_bytes(codec);
}

qgemm_status qgemm_pack_weights(qgemm_codec codec, int N, int K, const void *codes_canonical_dev,
                                const uint16_t *scales_fp16_dev, void *packed_dev, qgemm_stream_t stream) {
    if (!valid_codec(codec)) return QGEMM_ERR_INVALID_ARG;
    if (N < 1 || K < GROUP || K % GROUP) return QGEMM_ERR_SHAPE;
    if (!codes_canonical_dev || !scales_fp16_dev || !packed_dev) return QGEMM_ERR_INVALID_ARG;
    if (!aligned16(packed_dev)) return QGEMM_ERR_ALIGNMENT;
    if (launch_pack(codec, N, K, codes_canonical_dev, scales_fp16_dev, packed_dev, (cudaStream_t)stream) !=
        cudaSuccess)
        return QGEMM_ERR_CUDA;
    // Runs prefetch weights before their programmatic wait on the preceding
    // kernel; an empty kernel after the pack keeps the pack's writes complete
    // before any run on this stream can start.
    if (launch_fence((cudaStream_t)stream) != cudaSuccess) return QGEMM_ERR_CUDA;
    g_launches.fetch_add(2);
    return QGEMM_OK;
}

qgemm_status qgemm_plan(int N, int K, qgemm_codec codec, int T_max, qgemm_plan_t *out) {
    if (!out) return QGEMM_ERR_INVALID_ARG;
    *out = nullptr;
    if (!valid_codec(codec) || T_max < 1) return QGEMM_ERR_INVALID_ARG;
    if (N < 1 || K < GROUP || K % GROUP) return QGEMM_ERR_SHAPE;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
        cudaGetLastError();
        return QGEMM_ERR_UNSUPPORTED;
    }
    qgemm_plan_s *p = new (std::nothrow) qgemm_plan_s();
    if (!p) return QGEMM_ERR_INVALID_ARG;
    p->N = N;
    p->K = K;
    p->codec = codec;
    p->T_max = T_max;
    p->rows = N;
    p->epi = QGEMM_EPILOGUE_STORE;
    p->out = QGEMM_OUT_F32;
    p->G = K / GROUP;
    p->NB = (N + BLOCK_ROWS - 1) / BLOCK_ROWS;
    p->UB = unit_bytes(codec);
    p->sms = sms;
    p->pdl = true;
    p->forced_route = -1;
    p->tscale = 1.0f;
    p->ws_bytes = wide_workspace_bytes(N, T_max, sms);
    p->ws_part = p->ws_bytes ? wide_partial_bytes(T_max, sms) : 0;
    *out = p;
    return QGEMM_OK;
}

size_t qgemm_plan_workspace_bytes(qgemm_plan_t plan) { return plan ? plan->ws_bytes : 0; }

qgemm_status qgemm_plan_bind(qgemm_plan_t plan, const void *packed_dev, void *workspace_dev, size_t ws_bytes) {
    if (!plan || !packed_dev) return QGEMM_ERR_INVALID_ARG;
    if (!aligned16(packed_dev)) return QGEMM_ERR_ALIGNMENT;
    if (plan->ws_bytes) {
        if (!workspace_dev || ws_bytes < plan->ws_bytes) return QGEMM_ERR_WORKSPACE;
        if (!aligned16(workspace_dev)) return QGEMM_ERR_ALIGNMENT;
    }
    plan->packed = static_cast<const uint8_t *>(packed_dev);
    plan->ws = static_cast<uint8_t *>(workspace_dev);
    plan->bound = true;
    return QGEMM_OK;
}

qgemm_status qgemm_plan_destroy(qgemm_plan_t plan) {
    delete plan;
    return QGEMM_OK;
}

size_t qgemm_pair_packed_bytes(int F, int K, qgemm_codec codec) {
    if (F < 1 || F > (1 << 29)) return 0;
    return qgemm_packed_bytes(pair_rows(F), K, codec);
}

qgemm_status qgemm_pack_pair(qgemm_codec codec, int F, int K, const void *gate_codes_dev,
                             const uint16_t *gate_scales_dev, const void *up_codes_dev,
                             const uint16_t *up_scales_dev, void *packed_dev, qgemm_stream_t stream) {
    if (!valid_codec(codec)) return QGEMM_ERR_INVALID_ARG;
    if (F < 1 || F > (1 << 29) || K < GROUP || K % GROUP) return QGEMM_ERR_SHAPE;
    if (!gate_codes_dev || !gate_scales_dev || !up_codes_dev || !up_scales_dev || !packed_dev)
        return QGEMM_ERR_INVALID_ARG;
    if (!aligned16(packed_dev)) return QGEMM_ERR_ALIGNMENT;
    if (launch_pack_pair(codec, F, K, gate_codes_dev, gate_scales_dev, up_codes_dev, up_scales_dev, packed_dev,
                         (cudaStream_t)stream) != cudaSuccess)
        return QGEMM_ERR_CUDA;
    if (launch_fence((cudaStream_t)stream) != cudaSuccess) return QGEMM_ERR_CUDA;
    g_launches.fetch_add(2);
    return QGEMM_OK;
}

qgemm_status qgemm_plan_set_epilogue(qgemm_plan_t plan, qgemm_epilogue epilogue, qgemm_out out) {
    if (!plan || plan->bound) return QGEMM_ERR_INVALID_ARG;
    if (epilogue != QGEMM_EPILOGUE_STORE && epilogue != QGEMM_EPILOGUE_ADD && epilogue != QGEMM_EPILOGUE_SWIGLU)
        return QGEMM_ERR_INVALID_ARG;
    if (out != QGEMM_OUT_F32 && out != QGEMM_OUT_BF16) return QGEMM_ERR_INVALID_ARG;
    if (epilogue == QGEMM_EPILOGUE_SWIGLU && plan->N > (1 << 29)) return QGEMM_ERR_SHAPE;   // pair rows fit an int
    plan->epi = epilogue;
    plan->out = out;
    plan->rows = epilogue == QGEMM_EPILOGUE_SWIGLU ? pair_rows(plan->N) : plan->N;
    plan->NB = (plan->rows + BLOCK_ROWS - 1) / BLOCK_ROWS;
    plan->ws_bytes = wide_workspace_bytes(plan->rows, plan->T_max, plan->sms);
    plan->ws_part = plan->ws_bytes ? wide_partial_bytes(plan->T_max, plan->sms) : 0;
    return QGEMM_OK;
}

qgemm_status qgemm_plan_set_tensor_scale(qgemm_plan_t plan, float scale) {
    if (!plan || plan->codec != QGEMM_NVFP4) return QGEMM_ERR_INVALID_ARG;
    plan->tscale = scale;
    return QGEMM_OK;
}

qgemm_status qgemm_plan_set_pdl(qgemm_plan_t plan, int enable) {
    if (!plan) return QGEMM_ERR_INVALID_ARG;
    plan->pdl = enable != 0;
    return QGEMM_OK;
}

int qgemm_plan_route(qgemm_plan_t plan, int T) {
    if (!plan || T < 1 || T > plan->T_max) return -1;
    return choose_route(plan, T, plan->NB);
}

// Whether the plan's workspace holds what `route` needs: the tcgen05 routes
// keep partial sums of their token tile, and a plan's workspace is sized for
// the widest tile its T_max can take (64 tokens above T_max = 16, 128 above
// 64, 256 above 128).
static bool workspace_fits(const qgemm_plan_s *p, int route) {
    return !wide_route(route) || route_tokens(route) <= wide_max_tokens(p->T_max);
}

qgemm_status qgemm_plan_force_route(qgemm_plan_t plan, int route) {
    if (!plan || route < -1 || route >= ROUTE_COUNT) return QGEMM_ERR_INVALID_ARG;
    if (route >= 0 && !workspace_fits(plan, route)) return QGEMM_ERR_INVALID_ARG;
    plan->forced_route = route;
    return QGEMM_OK;
}

const char *qgemm_route_name(int route) {
    return (route >= 0 && route < ROUTE_COUNT) ? kRouteNames[route] : "none";
}

uint64_t qgemm_launch_count(void) { return g_launches.load(); }

qgemm_status qgemm_selftest_timeout(qgemm_stream_t stream) {
    unsigned int *status = status_ptr();
    if (!status) return QGEMM_ERR_CUDA;
    if (launch_wait_timeout(status, 16, (cudaStream_t)stream) != cudaSuccess) return QGEMM_ERR_CUDA;
    g_launches.fetch_add(1);
    return QGEMM_OK;
}

qgemm_status qgemm_device_status(qgemm_stream_t stream, int clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_device_status, sizeof v, 0, cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return QGEMM_ERR_CUDA;
    if (clear && v) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                    (cudaStream_t)stream) != cudaSuccess ||
            cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
            return QGEMM_ERR_CUDA;
    }
    return v ? (qgemm_status)v : QGEMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- runs

static void fill_parent(SkinnyParent &sp, const qgemm_plan_s *p, void *Y, const float *R, int cta_begin) {
    sp.packed = p->packed;
    sp.Y = Y;
    sp.R = R;
    sp.N = p->rows;
    sp.codec = p->codec;
    sp.tscale = p->tscale;
    sp.cta_begin = cta_begin;
    sp.ncols = p->N;
    sp.epi = p->epi;
    sp.ybf16 = p->out == QGEMM_OUT_BF16;
}

// One or more parents over the same X in one launch of the route T selects.
static qgemm_status run_parents(const qgemm_plan_s *const *plans, int np, const void *X, int T,
                                void *const *Ys, const float *R, cudaStream_t stream) {
    // parents of one launch share its route: the first plan's choice for the
    // launch's row blocks
    int nb = 0;
    for (int i = 0; i < np; ++i) nb += plans[i]->NB;
    const int route = choose_route(plans[0], T, nb);
    const int K = plans[0]->K;
    const int G = K / GROUP;
    unsigned int *status = status_ptr();
    if (!status) return QGEMM_ERR_CUDA;
    bool pdl = true;
    for (int i = 0; i < np; ++i) pdl = pdl && plans[i]->pdl;
    if (wide_route(route)) {
        for (int i = 0; i < np; ++i)
            if (!workspace_fits(plans[i], route)) return QGEMM_ERR_INVALID_ARG;
        WideParent wp[MAX_PARENTS];
        memset(wp, 0, sizeof wp);
        for (int i = 0; i < np; ++i) {
            wp[i].packed = plans[i]->packed;
            wp[i].Y = Ys[i];
            wp[i].R = R;
            wp[i].cnt = reinterpret_cast<unsigned int *>(plans[i]->ws + plans[i]->ws_part);
            wp[i].N = plans[i]->rows;
            wp[i].codec = plans[i]->codec;
            wp[i].tscale = plans[i]->tscale;
            wp[i].ncols = plans[i]->N;
            wp[i].epi = plans[i]->epi;
            wp[i].ybf16 = plans[i]->out == QGEMM_OUT_BF16;
        }
        // the partial-sum slots of the first parent's workspace serve the launch
        if (launch_wide(wp, np, X, T, K, route == ROUTE_WIDE32 ? 32 : route == ROUTE_WIDE64 ? 64 : 128,
                        route == ROUTE_WIDE256 ? 2 : 1,
                        reinterpret_cast<float *>(plans[0]->ws), status, pdl, plans[0]->sms, stream) != cudaSuccess)
            return QGEMM_ERR_CUDA;
        g_launches.fetch_add(1);
        return QGEMM_OK;
    }
    SkinnyArgs a;
    memset(&a, 0, sizeof a);
    int grid = 0;
    for (int i = 0; i < np; ++i) {
        fill_parent(a.p[i], plans[i], Ys[i], R, grid);
        grid += (plans[i]->rows + 15) / 16;
    }
    a.nparents = np;
    a.status = status;
    a.X = reinterpret_cast<const __nv_bfloat16 *>(X);
    a.T = T;
    a.K = K;
    a.G = G;
    bool f8 = false;
    for (int i = 0; i < np; ++i) f8 = f8 || plans[i]->codec == QGEMM_FP8 || plans[i]->codec == QGEMM_NVFP4;
    // the straight-line kernel (8 groups per warp, all in flight) where K / 64
    // is a multiple of 8, else the ring kernel with 8 warps per CTA
    const int nj = skinny_line_groups(G, 8);
    const cudaError_t e = nj ? launch_skinny_line(a, route_tokens(route) / 8, nj, grid, pdl, f8, stream)
                             : launch_skinny(a, route_tokens(route) / 8, 8, grid, pdl, f8, stream);
    if (e != cudaSuccess) return QGEMM_ERR_CUDA;
    g_launches.fetch_add(1);
    return QGEMM_OK;
}

static qgemm_status check_run(const qgemm_plan_s *p, const void *X, int T, const void *Y) {
    if (!p || !p->bound) return QGEMM_ERR_INVALID_ARG;
    if (T < 0) return QGEMM_ERR_INVALID_ARG;
    if (T > p->T_max) return QGEMM_ERR_T_OUT_OF_DOMAIN;
    if (T == 0) return QGEMM_OK;
    if (!X || !Y) return QGEMM_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y)) return QGEMM_ERR_ALIGNMENT;
    if (p->ws_bytes && !p->ws) return QGEMM_ERR_WORKSPACE;
    return QGEMM_OK;
}

static bool plain_output(const qgemm_plan_s *p) {
    return p->epi == QGEMM_EPILOGUE_STORE && p->out == QGEMM_OUT_F32;
}

extern "C" qgemm_status qgemm_run(qgemm_plan_t plan, const void *X, int T, float *Y, qgemm_stream_t stream) {
    if (plan && !plain_output(plan)) return QGEMM_ERR_INVALID_ARG;
    const qgemm_status st = check_run(plan, X, T, Y);
    if (st != QGEMM_OK || T == 0) return st;
    const qgemm_plan_s *plans[1] = {plan};
    void *Ys[1] = {Y};
    return run_parents(plans, 1, X, T, Ys, nullptr, (cudaStream_t)stream);
}

extern "C" qgemm_status qgemm_run_ex(qgemm_plan_t plan, const void *X, int T, const void *R, void *Y,
                                     qgemm_stream_t stream) {
    if (!plan) return QGEMM_ERR_INVALID_ARG;
    if ((plan->epi == QGEMM_EPILOGUE_ADD) != (R != nullptr)) return QGEMM_ERR_INVALID_ARG;
    const qgemm_status st = check_run(plan, X, T, Y);
    if (st != QGEMM_OK || T == 0) return st;
    if (R && !aligned16(R)) return QGEMM_ERR_ALIGNMENT;
    const qgemm_plan_s *plans[1] = {plan};
    void *Ys[1] = {Y};
    return run_parents(plans, 1, X, T, Ys, static_cast<const float *>(R), (cudaStream_t)stream);
}

extern "C" qgemm_status qgemm_run_multi(const qgemm_plan_t *plans, int n_parents, const void *X, int T,
                                        float *const *Ys, qgemm_stream_t stream) {
    if (!plans || !Ys || n_parents < 1 || n_parents > MAX_PARENTS) return QGEMM_ERR_INVALID_ARG;
    for (int i = 0; i < n_parents; ++i) {
        if (!plans[i] || !plain_output(plans[i])) return QGEMM_ERR_INVALID_ARG;
        if (plans[i]->K != plans[0]->K) return QGEMM_ERR_SHAPE;
        for (int j = 0; j < i; ++j)
            if (plans[j] == plans[i]) return QGEMM_ERR_INVALID_ARG;   // one workspace per parent
        const qgemm_status st = check_run(plans[i], X, T, Ys[i]);
        if (st != QGEMM_OK) return st;
    }
    if (T == 0) return QGEMM_OK;
    const qgemm_plan_s *ps[MAX_PARENTS];
    void *ys[MAX_PARENTS];
    for (int i = 0; i < n_parents; ++i) {
        ps[i] = plans[i];
        ys[i] = Ys[i];
    }
    return run_parents(ps, n_parents, X, T, ys, nullptr, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- allocation-free runs
//
// Some callers cannot allocate device memory when they run a projection: an
// engine that has reserved the GPU's memory up front under its own allocator,
// a plugin loaded into a host whose memory budget is fixed, or code that must
// not call cudaMalloc while other streams are being captured into CUDA graphs
// (an allocation there synchronises the device or is refused).  Such callers
// cannot provide the workspace that the tcgen05 route keeps its split tiles'
// partial sums in.  qgemm_run_noalloc runs that route with a scratch array
// the library owns instead: a file-scope device array of fixed size, which
// every GPU that loads the library holds until the process exits.

constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)32 << 20;   // the whole array
constexpr size_t NOALLOC_COUNTER_BYTES = (size_t)256 << 10;  // of it, the split-tile counters
constexpr size_t NOALLOC_MAX_TILES = NOALLOC_COUNTER_BYTES / (8 * sizeof(unsigned int));

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up on the
// first call on each device (the host-side name of a __device__ array is not a
// device address).
static uint8_t *noalloc_scratch_ptr() {
    constexpr int MAX_DEVICES = 64;
    static std::atomic<uint8_t *> cache[MAX_DEVICES];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return nullptr;
    }
    uint8_t *p = cache[dev].load();
    if (p) return p;
    uint8_t *ptr = nullptr;
    if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return nullptr;
    }
    cache[dev].store(ptr);
    return ptr;
}

extern "C" qgemm_status qgemm_run_noalloc(qgemm_plan_t plan, const void *packed_dev, const void *X, int T, float *Y,
                                          qgemm_stream_t stream) {
    if (!plan || !plain_output(plan) || !packed_dev || T < 0) return QGEMM_ERR_INVALID_ARG;
    if (T > plan->T_max) return QGEMM_ERR_T_OUT_OF_DOMAIN;
    if (T == 0) return QGEMM_OK;
    if (!X || !Y) return QGEMM_ERR_INVALID_ARG;
    if (!aligned16(packed_dev) || !aligned16(X) || !aligned16(Y)) return QGEMM_ERR_ALIGNMENT;
    const int halves = T > 128 ? 2 : 1;
    const int BN = 128 * halves;
    const size_t tiles = (size_t)plan->NB * (size_t)((T + BN - 1) / BN);
    if (tiles > NOALLOC_MAX_TILES) return QGEMM_ERR_WORKSPACE;   // more tiles than the counters cover
    uint8_t *scratch = noalloc_scratch_ptr();
    unsigned int *status = status_ptr();
    if (!scratch || !status) return QGEMM_ERR_CUDA;
    // the counters start at zero on every call (a run that gave up leaves
    // some behind); the partial sums need no clearing
    if (cudaMemsetAsync(scratch, 0, tiles * 8 * sizeof(unsigned int), (cudaStream_t)stream) != cudaSuccess)
        return QGEMM_ERR_CUDA;
    // as many CTAs as the partial-sum slots (two per CTA) fit
    const size_t slot_pair = (size_t)2 * BN * 128 * sizeof(float);
    const int fit = (int)((NOALLOC_SCRATCH_BYTES - NOALLOC_COUNTER_BYTES) / slot_pair);
    WideParent wp;
    memset(&wp, 0, sizeof wp);
    wp.packed = static_cast<const uint8_t *>(packed_dev);
    wp.Y = Y;
    wp.cnt = reinterpret_cast<unsigned int *>(scratch);
    wp.N = plan->rows;
    wp.codec = plan->codec;
    wp.tscale = plan->tscale;
    wp.ncols = plan->N;
    wp.epi = plan->epi;
    if (launch_wide(&wp, 1, X, T, plan->K, 128, halves, reinterpret_cast<float *>(scratch + NOALLOC_COUNTER_BYTES),
                    status, false, plan->sms < fit ? plan->sms : fit, (cudaStream_t)stream) != cudaSuccess)
        return QGEMM_ERR_CUDA;
    g_launches.fetch_add(1);
    return QGEMM_OK;
}
