/*
 * qgemm -- groupwise int4/int5/FP8 weight-only dequant-GEMM for GB300 (sm_103a).
 *
 *     Y[t][n] = sum_k X[t][k] * deq(W)[n][k],   deq(W)[n][k] = s[n][k/64] * q[n][k]
 *
 * for t < T token columns, n < N weight rows and k < K input channels.
 *
 * The operation is the fused "unpack the weights and multiply them in one pass
 * shaped for a batch" of "Fused kernels" (ark-labs.cloud research note, section
 * "Why standard kernels stall"), on the groupwise-int weight format of
 * "ninfer-3080 docs/performance.md": integer codes with one scale per 64
 * K-columns per row (cuBLAS prefill route section) in the Q4 and Q5 codecs
 * (small-T kernels section), evaluated at the decode, speculative-verify,
 * batched-decode and prefill token widths the same page routes separately
 * (route boundaries section).
 *
 * Number formats
 *   q  symmetric two's-complement code, no zero point: int4 in [-8, 7],
 *      int5 in [-16, 15]; or an FP8 E4M3 value (below), exact in bf16;
 *   s  IEEE fp16, one per (row, 64-column group); any finite value, negative
 *      and subnormal included (non-finite scales propagate but the result is
 *      then unspecified beyond being non-finite);
 *   X  bf16, row-major [T][K] (K contiguous);
 *   Y  fp32, row-major [T][N] (N contiguous), overwritten (no accumulate).
 *   s * q is never rounded: products run on the exact integer codes and each
 *   group's fp32 partial sum is multiplied by its scale.  Accumulation is fp32.
 *
 * Canonical packed codes (the input of qgemm_pack_weights)
 *   int4: K/2 bytes per row, row-major; byte j holds code 2j in bits 0-3 and
 *         code 2j+1 in bits 4-7.
 *   int5: 5K/8 bytes per row, row-major; LSB-first bitstream, code k in bits
 *         5k .. 5k+4.
 *   fp8:  K bytes per row, row-major; byte k is the OCP FP8 E4M3 code of
 *         column k (bias 7, subnormals, no infinities; the NaN codes S.1111.111
 *         are outside the codec and give unspecified results), weighted by the
 *         same fp16 scale per 64 columns.  FP8 is the weight-only FP8 format
 *         of the FP8-weight kernel the "Speculative decoding" page checks at
 *         verify widths; every route serves it.
 *   nvfp4: K/2 bytes per row like int4 (column 2j in bits 0-3, 2j+1 in bits
 *         4-7), each nibble an FP4 E2M1 code (sign, 2 exponent bits with bias
 *         1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), weighted
 *         by an unsigned E4M3 scale per 16 columns per row (bias 7, subnormals;
 *         0x7F and codes with bit 7 set are outside the codec) and by one fp32
 *         scale for the whole matrix (qgemm_plan_set_tensor_scale):
 *         deq(W)[n][k] = e2m1(c[n][k]) * ue4m3(b[n][k/16]) * s_t.  This is the
 *         "nvfp4" weight profile of "ninfer-3080 docs/performance.md" (RTX
 *         5090 publication index), read as the common NVFP4 definition.
 *         E2M1 times UE4M3 is exact in bf16, so the kernels multiply each code
 *         by its block scale in the decode and apply s_t where the other codecs
 *         apply their group scales.
 *   scales: fp16 bit patterns, row-major [N][K/64]; for NVFP4 the same
 *         argument points to the UE4M3 block-scale bytes, row-major [N][K/16].
 *
 * Conventions for every call
 *   - All pointers named *_dev and X, Y are device pointers (or managed /
 *     mapped memory the GPU can reach).  The caller allocates and owns every
 *     buffer; the library owns only the host-side plan object.
 *   - Everything is asynchronous on the given stream (0 = legacy default
 *     stream); no call synchronises the device.
 *   - Argument errors return a status before anything is launched; a launch
 *     failure returns QGEMM_ERR_CUDA.  Nothing aborts, no C++ exception crosses
 *     this interface.
 *   - Results are bitwise repeatable for a given (plan, T); different T may
 *     take different routes and summation orders and then agree only within
 *     the fp32 rounding tolerance.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qgemm_stream_t;   /* a cudaStream_t */

typedef enum {
    QGEMM_OK = 0,
    QGEMM_ERR_INVALID_ARG = 1,     /* null pointer, unknown codec, negative size, plan not bound */
    QGEMM_ERR_SHAPE = 2,           /* K not a positive multiple of 64, N < 1, shapes of parents differ */
    QGEMM_ERR_ALIGNMENT = 3,       /* a buffer is not 16-byte aligned */
    QGEMM_ERR_T_OUT_OF_DOMAIN = 4, /* T larger than the plan's T_max */
    QGEMM_ERR_WORKSPACE = 5,       /* workspace missing or smaller than qgemm_plan_workspace_bytes */
    QGEMM_ERR_CUDA = 6,            /* a CUDA call or launch failed */
    QGEMM_ERR_TIMEOUT = 7,         /* a bounded device-side wait ran out (see qgemm_device_status) */
    QGEMM_ERR_UNSUPPORTED = 8      /* no usable GPU of the architecture this library was built for */
} qgemm_status;

typedef enum { QGEMM_INT4 = 4, QGEMM_INT5 = 5, QGEMM_FP8 = 8, QGEMM_NVFP4 = 16 } qgemm_codec;

typedef struct qgemm_plan_s *qgemm_plan_t;

/* Human-readable name of a status (static string, never NULL).
 * Passage: none; a library convention. */
const char *qgemm_status_string(qgemm_status st);

/*
 * Bytes of the device-side packed weight buffer for an N x K matrix of the
 * given codec, or 0 for an invalid shape (K not a positive multiple of 64,
 * N < 1, unknown codec).  Rows are padded to a multiple of 128.
 * Passage: the count of scales follows the one scale per 64 K-columns per row
 * of "ninfer-3080 docs/performance.md" (cuBLAS prefill route section); the
 * device layout itself is the library's own (see qgemm_pack_weights).
 */
size_t qgemm_packed_bytes(int N, int K, qgemm_codec codec);

/*
 * Repack canonical codes and fp16 scales into the library's device layout
 * (one launch on `stream`).  Weight-only quantised serving packs each matrix
 * once at load time; the layout is private to the library and shared by all
 * of its routes.
 *   codes_canonical_dev  canonical packed codes, N rows (see above)
 *   scales_fp16_dev      fp16 patterns [N][K/64]
 *   packed_dev           qgemm_packed_bytes(N, K, codec) bytes, 16-byte aligned
 * The inputs may be freed once the stream has passed the launch.
 * Passage: "ninfer-3080 docs/performance.md", small-T kernels section: the
 * k slots of an MMA may be any permutation of a group as long as both
 * operands agree, and the Q5 codec keeps a separate high-bit plane; the token
 * tile section notes that the operand layout lever needs a repack, which this
 * call performs once at load time.
 * Errors: QGEMM_ERR_INVALID_ARG (unknown codec, NULL pointer), QGEMM_ERR_SHAPE,
 * QGEMM_ERR_ALIGNMENT (packed_dev), QGEMM_ERR_CUDA (launch failure).
 */
qgemm_status qgemm_pack_weights(qgemm_codec codec, int N, int K,
                                const void *codes_canonical_dev,
                                const uint16_t *scales_fp16_dev,
                                void *packed_dev, qgemm_stream_t stream);

/*
 * Host-only: choose the routes for an N x K matrix and token widths
 * 1 .. T_max from the built-in route table (measured per token width; the
 * "ninfer-3080 docs/performance.md" route boundaries section explains why
 * boundaries must come from measurement).  Queries the current device's SM
 * count; launches nothing.  *out must be released with qgemm_plan_destroy.
 * Passage: "ninfer-3080 docs/performance.md", route boundaries section: each
 * schedule has an explicit domain of column counts, boundaries are measured
 * rather than inherited, and the narrowest tile covering the extent wins;
 * T_max is this plan's domain (qgemm_run rejects T > T_max).
 * Errors: QGEMM_ERR_INVALID_ARG (NULL out, unknown codec, T_max < 1),
 * QGEMM_ERR_SHAPE (N < 1 or K not a positive multiple of 64),
 * QGEMM_ERR_UNSUPPORTED (no CUDA device).
 */
qgemm_status qgemm_plan(int N, int K, qgemm_codec codec, int T_max, qgemm_plan_t *out);

/* Workspace bytes the plan needs at its T_max; NULL plan: 0.  Plans with
 * T_max <= 16 run on the small-T routes only and need none.  Above that the
 * tcgen05 routes split output tiles across CTAs (stream-K) and need, per
 * launch, two fp32 partial-sum slots per SM of the widest token tile the
 * plan's widths can take (32 tokens up to T_max = 32, 64 up to 64, 128 up to
 * 128, else 256) times 128 rows, plus eight 32-bit counters per 128-row block
 * and 32-token tile.  Passage: "ninfer-3080 docs/performance.md", token tile section (the
 * token tile sets the weight passes); the split and its workspace are this
 * library's, not the pages'. */
size_t qgemm_plan_workspace_bytes(qgemm_plan_t plan);

/*
 * Attach the packed weights and the workspace to a plan.  The workspace must
 * be zero-filled before its first use (the library leaves it zeroed after
 * every completed run).  Runs that share one plan, and hence one workspace,
 * must not overlap on the GPU.  ws_bytes may exceed the requirement.
 * The plan keeps both pointers; the caller keeps them alive and unchanged for
 * as long as runs of the plan may execute.
 * Passage: none; a library convention (weights are packed once and bound to
 * the plan, so a run takes only X, T and Y).
 * Errors: QGEMM_ERR_INVALID_ARG (NULL plan or packed_dev),
 * QGEMM_ERR_ALIGNMENT, QGEMM_ERR_WORKSPACE.
 */
qgemm_status qgemm_plan_bind(qgemm_plan_t plan, const void *packed_dev,
                             void *workspace_dev, size_t ws_bytes);

/*
 * Y[T][N] = X[T][K] . deq(W)^T on `stream`.  X (bf16 bit patterns) and Y
 * must be 16-byte aligned.  T == 0 is a no-op; T > T_max returns
 * QGEMM_ERR_T_OUT_OF_DOMAIN.  The plan must have the default output (STORE,
 * F32; see qgemm_plan_set_epilogue), else QGEMM_ERR_INVALID_ARG.
 * X holds at least T*K bf16 values and Y at least T*N floats: the library
 * sees only pointers and cannot check their extents.
 * Passage: the one-pass unpack-and-multiply of "Fused kernels" (section "Why
 * standard kernels stall"), over the token widths of "ninfer-3080
 * docs/performance.md" (route boundaries section: a decode round covers
 * concurrency x (draft window + 1) columns; prefill chunks are wider).
 * Errors: QGEMM_ERR_INVALID_ARG (NULL or unbound plan, NULL X/Y with T > 0,
 * T < 0), QGEMM_ERR_T_OUT_OF_DOMAIN, QGEMM_ERR_ALIGNMENT, QGEMM_ERR_CUDA.
 */
qgemm_status qgemm_run(qgemm_plan_t plan, const void *X, int T, float *Y, qgemm_stream_t stream);

/*
 * Several weight matrices ("parents") over one shared activation X in a
 * single launch, as the two-parent projections of "ninfer-3080
 * docs/performance.md" (A8 prefill routes section: two parents over one
 * activation share its preparation).  All plans must have the same K and
 * T <= each plan's T_max; codecs may differ (on the tensor-core route, used
 * from T = 33 up, parents of different codecs take one launch per codec).
 * Ys[i] receives parent i's [T][N_i] result.  1 <= n_parents <= 4.  Every
 * plan must have the default output (STORE, F32).
 */
qgemm_status qgemm_run_multi(const qgemm_plan_t *plans, int n_parents, const void *X, int T,
                             float *const *Ys, qgemm_stream_t stream);

/* Release a plan (NULL is accepted).  Runs already enqueued keep working:
 * they hold copies of what they need.
 * Passage: none; a library convention. */
qgemm_status qgemm_plan_destroy(qgemm_plan_t plan);

/*
 * ---------------------------------------------------------------- fused outputs
 *
 * The pages' projections end in two fused outputs ("ninfer-3080
 * docs/performance.md"): a residual add on the attention o_proj and the GDN
 * out_proj (LinearAdd, A8 prefill routes section) and the SwiGLU of the MLP's
 * gate/up pair (route boundaries section).  A plan may carry one of them and
 * an output type; the epilogue runs where the kernel writes Y, on the fp32
 * result, so the GEMM's accuracy contract is unchanged:
 *   ADD     Y[t][n] = R[t][n] + (X . deq(W)^T)[t][n]   (one fp32 add)
 *   SWIGLU  Y[t][f] = silu(g) * u,  silu(z) = z / (1 + exp(-z)) in fp32, with
 *           g and u row f of the gate and of the up matrix applied to X[t]
 *   bf16    the fp32 value rounded to nearest even
 */
typedef enum {
    QGEMM_EPILOGUE_STORE = 0,   /* Y = X . deq(W)^T (the default) */
    QGEMM_EPILOGUE_ADD = 1,     /* Y = R + X . deq(W)^T, R fp32 [T][N] */
    QGEMM_EPILOGUE_SWIGLU = 2   /* weights from qgemm_pack_pair; Y [T][F] */
} qgemm_epilogue;

typedef enum { QGEMM_OUT_F32 = 0, QGEMM_OUT_BF16 = 1 } qgemm_out;

/*
 * Bytes of the packed buffer of a SwiGLU pair of F x K matrices, or 0 for an
 * invalid shape (as qgemm_packed_bytes; F >= 1).
 */
size_t qgemm_pair_packed_bytes(int F, int K, qgemm_codec codec);

/*
 * Pack the gate and the up matrix of a SwiGLU pair (each F x K, canonical codes
 * and fp16 scales as for qgemm_pack_weights, same codec) into one buffer of
 * qgemm_pair_packed_bytes(F, K, codec) bytes whose 16-row tiles hold 8 gate
 * rows followed by the same 8 up rows, so that one kernel lane owns each pair.
 * One launch plus the ordering kernel, like qgemm_pack_weights.
 */
qgemm_status qgemm_pack_pair(qgemm_codec codec, int F, int K,
                             const void *gate_codes_dev, const uint16_t *gate_scales_dev,
                             const void *up_codes_dev, const uint16_t *up_scales_dev,
                             void *packed_dev, qgemm_stream_t stream);

/*
 * Give a plan a fused output, before qgemm_plan_bind.  For SWIGLU the plan's N
 * is F (the output width) and the weights must come from qgemm_pack_pair.
 * The fused outputs run through qgemm_run_ex on one matrix (qgemm_run and
 * qgemm_run_multi take plain STORE / F32 plans only).  Returns
 * QGEMM_ERR_INVALID_ARG for an unknown epilogue or output type, or a bound plan,
 * and QGEMM_ERR_SHAPE for a SwiGLU plan with F > 2^29.
 */
qgemm_status qgemm_plan_set_epilogue(qgemm_plan_t plan, qgemm_epilogue epilogue, qgemm_out out);

/*
 * Y = epilogue(X . deq(W)^T) on `stream`, for any plan.
 *   R  ADD: fp32 [T][N], 16-byte aligned; it may be Y itself (an in-place
 *      residual add) but must not otherwise overlap Y.  Other epilogues: NULL.
 *   Y  [T][N] (STORE, ADD) or [T][F] (SWIGLU), fp32 or bf16 bit patterns as
 *      the plan's output type says, 16-byte aligned.
 * Errors as qgemm_run; a missing or superfluous R is QGEMM_ERR_INVALID_ARG.
 */
qgemm_status qgemm_run_ex(qgemm_plan_t plan, const void *X, int T, const void *R, void *Y,
                          qgemm_stream_t stream);

/*
 * Programmatic dependent launch (enabled by default): a run's kernel may be
 * scheduled while the preceding kernel on the stream is still draining and
 * prefetches its packed weights before waiting for that kernel to finish; it
 * reads X and writes Y only after the wait.  So the packed buffer must not
 * be written by the kernel immediately preceding a run on the same stream
 * (qgemm_pack_weights itself ends with an empty kernel for this reason).
 * enable = 0 turns it off for runs of this plan.
 * Passage: "ninfer-3080 docs/performance.md", small-T kernels section: what
 * is left at one stream is ramp-up and drain at kernel boundaries, and
 * programmatic dependent launch is the lever named for hiding the ramp.
 * Errors: QGEMM_ERR_INVALID_ARG (NULL plan).
 */
qgemm_status qgemm_plan_set_pdl(qgemm_plan_t plan, int enable);

/*
 * The fp32 tensor scale s_t of an NVFP4 plan (1.0 until set).  It applies to
 * the runs that follow; set it before capturing runs into a CUDA graph.
 * Passage: the "nvfp4" weight profile of "ninfer-3080 docs/performance.md"
 * (RTX 5090 publication index); the per-tensor scale is part of the NVFP4
 * format read there.
 * Errors: QGEMM_ERR_INVALID_ARG (NULL plan, or a plan of another codec).
 */
qgemm_status qgemm_plan_set_tensor_scale(qgemm_plan_t plan, float scale);

/*
 * Route the plan takes at width T (a small integer naming the kernel family
 * and its tile width, see qgemm_route_name), or -1 if T is outside 1..T_max.
 * Passage: "ninfer-3080 docs/performance.md", route boundaries section (the
 * cost of a route is set by its padded tile width).
 */
int qgemm_plan_route(qgemm_plan_t plan, int T);
const char *qgemm_route_name(int route);

/*
 * Route sweeps and tests: make the plan take `route` at every T its token
 * tile covers (the other T keep the built-in table); -1 restores the table.
 * Results stay within the accuracy contract on every route, and a forced
 * plan is bitwise repeatable for a given T like any other.
 * Passage: "ninfer-3080 docs/performance.md", route boundaries section (every
 * schedule of an Op is timed at the same column count to place a boundary).
 * Errors: QGEMM_ERR_INVALID_ARG (NULL plan, route outside -1 .. routes - 1).
 */
qgemm_status qgemm_plan_force_route(qgemm_plan_t plan, int route);

/*
 * Number of kernels this library has launched since it was loaded (host
 * counter), so that callers and tests can check that one call runs exactly
 * the kernels its route names.
 * Passage: "ninfer-3080 docs/performance.md", route boundaries section (a
 * dispatch fallthrough once ran a second kernel after the first).
 */
uint64_t qgemm_launch_count(void);

/*
 * Device-side status word: QGEMM_OK, or QGEMM_ERR_TIMEOUT after a bounded
 * wait inside a kernel ran out (the kernel then skipped its remaining work
 * and returned).  Synchronises `stream` to read it; `clear` resets it.
 * Passage: none; a library convention (bounded waits instead of hangs).
 */
qgemm_status qgemm_device_status(qgemm_stream_t stream, int clear);

/*
 * Diagnostic of the timeout path: launches one kernel whose single bounded
 * wait is on a barrier nothing completes, so that it runs out after a few
 * hundred microseconds and sets the device status word to QGEMM_ERR_TIMEOUT,
 * as any kernel does when one of its waits runs out.  The kernel faults
 * nothing and leaves the context usable; read and clear the word with
 * qgemm_device_status.  Returns QGEMM_ERR_CUDA if the launch fails.
 * Passage: none; a library diagnostic.
 */
qgemm_status qgemm_selftest_timeout(qgemm_stream_t stream);

/*
 * ---------------------------------------------------------- allocation-free run
 *
 * Y[T][N] = X[T][K] . deq(W)^T like qgemm_run, on the tcgen05 route at every
 * T, for callers that cannot allocate device memory when they run: an engine
 * that has reserved the GPU's memory up front for its own allocator, a plugin
 * in a host with a fixed memory budget, code that must not call cudaMalloc
 * while streams are being captured.  They cannot supply the workspace that
 * route keeps its split tiles' partial sums in (qgemm_plan_bind), so this call
 * uses a scratch array inside the library: 32 MiB of device memory that every
 * GPU which loads the library holds until the process exits (256 KiB of it
 * counts the tiles whose groups several CTAs share, the rest holds their
 * partial sums).  The call allocates nothing itself.
 *   plan        from qgemm_plan (default output, STORE / F32); it need not be
 *               bound -- the weights come from packed_dev
 *   packed_dev  the matrix packed by qgemm_pack_weights for this plan's N, K
 *               and codec, 16-byte aligned
 *   X, Y        as qgemm_run
 * The scratch array is looked up on the first call on each device (make that
 * first call before any stream capture on the device).  Every call clears the
 * array's counters at its start on `stream` (one memset) and uses as many
 * CTAs as its partial-sum slots fit (up to the SM count for 128-token tiles,
 * T <= 128; 127 for 256-token tiles).  All calls on a device share the array,
 * so calls that overlap on the GPU (other streams, other host threads)
 * corrupt each other's results: order them on one stream.
 * No passage of the pages corresponds to this call; it is a deployment
 * convenience of the library.
 * Errors: as qgemm_run (a NULL packed_dev is QGEMM_ERR_INVALID_ARG), and
 * QGEMM_ERR_WORKSPACE when ceil(N / 128) * ceil(T / BN) tiles (BN = 128 for
 * T <= 128, else 256) exceed the 8,192 the counters cover.
 */
qgemm_status qgemm_run_noalloc(qgemm_plan_t plan, const void *packed_dev, const void *X, int T, float *Y,
                               qgemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
