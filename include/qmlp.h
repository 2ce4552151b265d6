/*
 * qmlp.h -- C ABI of libqmlp.so, the weight-quantized SwiGLU MLP for GB300
 * (sm_103a). Plain pointers and sizes only.
 *
 * The operation (vllm.cpp issue "tp>1 fp8w tail-MLP shard host-dequantizes
 * every layer", "Proposed fix"):
 *   act[m, i] = bf16( SiLU(sigma_g[i] * sum_k x[m,k] Wg[i,k]) *
 *                          (sigma_u[i] * sum_k x[m,k] Wu[i,k]) )
 *   out[m, o] = bf16( sigma_d[o] * sum_i act[m,i] Wd[o,i] )
 * with the weights dequantized on the fly from resident packed bytes:
 *   NVFP4 (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented"):
 *     W[n,k] = E2M1(nibble) * E4M3(scale[n, k/16]); byte k/2 of row n holds k
 *     in its low nibble when k is even; sigma = fp32(1 / global_scale).
 *   FP8 per-channel W8A16 (vllm.cpp issue, "Mechanism on the tp>1 path"):
 *     W[n,k] = e4m3fn(w[n,k]); sigma[n] = scale[n] (fp32).
 * SiLU(t) = t / (1 + exp(-t)). Accumulation is fp32 on the GPU; act is
 * rounded to bf16 before the down projection; out is bf16.
 *
 * Conventions for every entry point:
 *  - A status is returned; no entry point falls back to a CPU computation and
 *    none aborts the process. QMLP_OK is 0.
 *  - "device" pointers are CUDA device addresses on the current device;
 *    "host" pointers are host addresses (pinned or pageable).
 *  - All device pointers passed to forward calls must be 16-byte aligned.
 *  - Streams: a CUstream/cudaStream_t value; NULL means the legacy default
 *    stream. Forward calls only enqueue work (except *_host, which waits).
 *  - One handle serves one stream at a time: its workspace is shared by all
 *    calls on it.
 *  - One GPU per process: the kernels' shared-memory attributes are set on
 *    the first launch of each kernel in the process, for the device current
 *    then; handles on a second device of the same process get QMLP_ERR_CUDA
 *    from the launches that need a large shared-memory window. Run one
 *    process per GPU.
 *  - Validation happens before any launch; a rejected call launches nothing.
 *  - Launch failures return QMLP_ERR_CUDA. Errors raised asynchronously by a
 *    kernel surface on a later call or on the caller's synchronization; a
 *    kernel that gives up a bounded wait records it in the handle, and
 *    qmlp_check / qmlp_moe_check return QMLP_ERR_DEVICE_TIMEOUT.
 */
#ifndef QMLP_H
#define QMLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qmlp_stream_t; /* identical to cudaStream_t */

typedef enum {
    QMLP_OK = 0,
    QMLP_ERR_INVALID_ARG = 1,     /* null pointer, bad enum, bad count     */
    QMLP_ERR_ALIGNMENT = 2,       /* a device pointer not 16-byte aligned  */
    QMLP_ERR_ALIAS = 3,           /* output overlaps an input or workspace */
    QMLP_ERR_SHAPE = 4,           /* K, I, M, E or topk outside the limits */
    QMLP_ERR_UNSUPPORTED_ARCH = 5,/* device is not compute capability 10.3 */
    QMLP_ERR_OOM = 6,             /* device allocation failed at create    */
    QMLP_ERR_CUDA = 7,            /* a CUDA runtime call or launch failed  */
    QMLP_ERR_DEVICE_TIMEOUT = 8,  /* a kernel gave up a bounded wait       */
    QMLP_ERR_DEVICE_BOUNDS = 9    /* an index check failed (checking build) */
} qmlp_status;

typedef enum { QMLP_FMT_NVFP4 = 1, QMLP_FMT_FP8_PC = 2 } qmlp_format;
typedef enum { QMLP_DT_BF16 = 1, QMLP_DT_FP16 = 2 } qmlp_dtype;
typedef enum { QMLP_META_3B = 3, QMLP_META_4B = 4 } qmlp_meta;
/* Kernel family used by a forward call: AUTO picks the decode (GEMV) family
 * for small token counts and the tensor-core GEMM above. GEMM_PAIR is the
 * tensor-core GEMM on CTA pairs (tcgen05.mma.cta_group::2: two SMs share a
 * 256-token x 256-row tile, each decoding half of its weight rows) for
 * M >= 256; AUTO does not choose it (the single-CTA GEMM measured faster on
 * the 27B-class prefill shape). GEMM_DQ is the dequantise-once GEMM: each
 * projection is first decoded, once per call, into bf16 tiles in buffers
 * the handle holds (6 I K bytes, allocated by qmlp_create when max_M >=
 * 768, with a CUDA stream and two events of the handle's own: in a whole
 * forward the down projection is decoded on that stream while the gate/up
 * GEMM runs, forked from and joined back to the caller's stream with
 * events, so the call stays stream-ordered and can be captured in a CUDA
 * graph), and the tensor-core GEMM then multiplies those tiles with the bf16
 * activations as given (no per-token prescale), with no decoding in its main
 * loop (on CTA pairs from M = 256, as GEMM_PAIR, each CTA loading
 * half of every decoded tile); AUTO takes it from M = 768 on. The products
 * are of the same exact weight values either way. */
typedef enum {
    QMLP_PATH_AUTO = 0,
    QMLP_PATH_GEMV = 1,
    QMLP_PATH_GEMM = 2,
    QMLP_PATH_GEMM_PAIR = 3,
    QMLP_PATH_GEMM_DQ = 4
} qmlp_path;

/* One projection [N, K] as the checkpoint stores it. Pointers may be host or
 * device memory; they are only read during qmlp_create.
 *  NVFP4: w     = u8 [N, K/2], two E2M1 codes per byte, low nibble = even k
 *         scale = u8 [N, K/16], E4M3 group scales
 *         global_scale = fp32; the dequantization factor is 1/global_scale
 *  FP8:   w     = u8 [N, K], e4m3fn codes
 *         scale = fp32 [N], per output channel; global_scale is ignored */
typedef struct {
    const uint8_t* w;
    const void* scale;
    float global_scale;
} qmlp_proj;

/* Dense MLP description: hidden size K, intermediate size I, largest token
 * count max_M any forward call will use. gate/up are [I, K], down is [K, I].
 * Limits: K % 16 == 0, I % 16 == 0, 16 <= K, I <= 65536, 1 <= max_M <= 65536. */
typedef struct {
    qmlp_format fmt;
    int K;
    int I;
    int max_M;
    qmlp_proj gate;
    qmlp_proj up;
    qmlp_proj down;
} qmlp_desc;

typedef struct qmlp_s qmlp_t;

/* Create a dense MLP handle. Copies the weights into memory the handle owns,
 * reordered for the kernels (create-time repack; the weight bytes are kept
 * packed, never expanded), computes sigma = fp32(1/global) for NVFP4, and
 * allocates the forward workspace for max_M tokens. Synchronizes `stream`
 * before returning, so the caller may free its buffers afterwards.
 * Errors: INVALID_ARG (null/unknown fmt), SHAPE, UNSUPPORTED_ARCH, OOM, CUDA.
 * On error *out is NULL and nothing is leaked. */
qmlp_status qmlp_create(qmlp_t** out, const qmlp_desc* desc, qmlp_stream_t stream);

/* Free every buffer owned by the handle (waits for its pending work). NULL is
 * a no-op. */
void qmlp_destroy(qmlp_t* h);

/* The MLP block (see the top of this file) on M tokens.
 *  x   = device bf16 [M, K] (row-major), read only
 *  out = device bf16 [M, K] (row-major), written
 * Allocates nothing; enqueues its kernels on `stream`.
 * Errors: INVALID_ARG (null), ALIGNMENT (x/out not 16-B aligned), ALIAS (out
 * overlaps x), SHAPE (M < 1 or M > max_M), CUDA. */
qmlp_status qmlp_forward(qmlp_t* h, const void* x, int M, void* out, qmlp_stream_t stream);

/* As qmlp_forward, forcing a kernel family. GEMM, GEMM_PAIR and GEMM_DQ
 * require a handle whose max_M reaches the GEMM threshold (and K % 256,
 * I % 128 == 0); GEMM_PAIR also M >= 256; GEMM_DQ a handle created with
 * max_M >= 768 (any M up to max_M; the handle's buffers and side stream,
 * see qmlp_path). Otherwise SHAPE. */
qmlp_status qmlp_forward_path(qmlp_t* h, qmlp_path path, const void* x, int M, void* out,
                              qmlp_stream_t stream);

/* One half of the forward, for callers that overlap or time the two
 * projections separately (stage 0 followed by stage 1 equals qmlp_forward):
 *  stage 0: act = SwiGLU(x) into the handle's workspace; x = device bf16
 *           [M, K]; out must be NULL.
 *  stage 1: out = the down projection of the workspace act written by the
 *           previous stage-0 call with the same M; x must be NULL; out =
 *           device bf16 [M, K].
 * Errors: as qmlp_forward_path (INVALID_ARG for a wrong NULL pattern). */
qmlp_status qmlp_forward_stage(qmlp_t* h, int stage, qmlp_path path, const void* x, int M, void* out,
                               qmlp_stream_t stream);

/* End-to-end call from host buffers (x: host bf16 [M, K], out: host bf16
 * [M, K]); returns after `stream` has finished. Pinned (device-mapped) host
 * buffers, 16-byte aligned and not overlapping: one small kernel copies x
 * over the coherent CPU-GPU link into the handle's device stage, and the
 * kernels write the output in place into the host buffer. Otherwise x is
 * copied to the staging buffer and the result copied back by the copy engine
 * (pageable memory works but serializes the copies).
 * Errors: as qmlp_forward. */
qmlp_status qmlp_forward_host(qmlp_t* h, const void* x_host, int M, void* out_host,
                              qmlp_stream_t stream);

/* Forward that also returns the intermediate: act = device bf16 [M, I]
 * (the values the down projection consumed). Errors: as qmlp_forward_path,
 * plus ALIAS if act overlaps x or out. */
qmlp_status qmlp_forward_debug(qmlp_t* h, qmlp_path path, const void* x, int M, void* act,
                               void* out, qmlp_stream_t stream);

/* One projection in isolation, through the same kernels, with no scale
 * factor applied (no 1/global, no per-channel scale) and fp32 output:
 *   y[m, n] = sum_k x[m,k] * W[n,k],  W = E2M1*E4M3 (NVFP4) or e4m3fn (FP8)
 *  which = 0 gate, 1 up (x is [M, K]); 2 down (x is [M, I]).
 *  x = device bf16 [M, Kp], y = device fp32 [M, N].
 * With a one-hot x this returns single decoded weights exactly.
 * Errors: as qmlp_forward_path. */
qmlp_status qmlp_debug_project(qmlp_t* h, int which, qmlp_path path, const void* x, int M,
                               float* y, qmlp_stream_t stream);

/* CTAs of the decode kernel that partitions the intermediate dimension (each
 * CTA computes gate/up for its slice of I and the down projection over that
 * slice; the partial outputs are added in a fixed order -- after a grid
 * barrier inside the kernel for one NVFP4 token, else by a small reduce
 * kernel launched after it). 0 when the shape has no such partition on this
 * device (the stream-K kernel is used instead). Used for M <= 8; the tensor-
 * core GEMM takes M >= 9 when this partition exists.
 * The one-token NVFP4 schedule waits (bounded, 2 s) at that grid barrier for
 * all its CTAs, one per SM: if kernels of other streams hold SMs for longer,
 * the call gives up, its output is not valid and qmlp_check returns
 * QMLP_ERR_DEVICE_TIMEOUT. */
int qmlp_decode_ctas(qmlp_t* h);

/* The I-partitioned decode kernel (see qmlp_decode_ctas) with its raw
 * epilogues, for tests that check its own weight layouts bit for bit:
 *  x      = device bf16 [M, K]; act_in = device bf16 [M, I] (the down
 *           projection consumes act_in instead of the SwiGLU of x)
 *  g, u   = device fp32 [M, I]: sum_k x[m,k] W[i,k] of gate / up, no factor
 *  out_f32= device fp32 [M, K]: sum_i act_in[m,i] Wd[o,i], no factor
 * With one-hot x (act_in) every value is a single decoded weight exactly.
 * 1 <= M <= 8. Errors: INVALID_ARG, ALIGNMENT, ALIAS, SHAPE (no partition for
 * this shape, or M out of range), CUDA. */
qmlp_status qmlp_debug_split(qmlp_t* h, const void* x, const void* act_in, int M, float* g, float* u,
                             float* out_f32, qmlp_stream_t stream);

/* Error-path tests only: every later launch of this handle's decode
 * (I-partitioned) and tensor-core GEMM kernels gives up a wait on another
 * role or CTA after limit_ns (0: the default of 2 s), and, when
 * withhold_last_step is non-zero, their producers never issue their last
 * weight step, so those waits run out: the kernels record it, leave without
 * a fault, and qmlp_check returns QMLP_ERR_DEVICE_TIMEOUT. Errors: INVALID_ARG. */
qmlp_status qmlp_debug_set_wait(qmlp_t* h, uint64_t limit_ns, int withhold_last_step);

/*
 * Index checks. A library built with -DQMLP_DEBUG_BOUNDS (libqmlp_bounds.so;
 * the default build compiles the checks away) checks, in every kernel, the
 * index of each global access whose address comes from layout arithmetic or
 * runtime data (weight-bank blocks and records, partial buffers, outputs,
 * route lists) against the size of its buffer. A failed check never traps:
 * the kernel records the first one and skips the access (a load reads zero,
 * a store is dropped, a bulk copy is taken from the start of its buffer), so
 * the call's outputs are then invalid but the device stays usable. This
 * build stands in for a memory checker where none can run.
 */
/* 1 for a checking build, else 0. */
int qmlp_debug_bounds_enabled(void);

/* Synchronize the device, then report and clear the first failed index
 * check of any kernel since the last call: *site = the check's number
 * (per source file: 1-9 decode kernel, 11-19 tensor-core GEMM, 21-29 stream-K
 * and split-K decode kernels, 31-39 one-token routed experts, 41-49 grouped
 * routed experts, 51-59 tensor-parallel combine) and *index = the checked
 * index (low 48 bits), or 0 and 0. Returns OK, DEVICE_BOUNDS (a check
 * failed), INVALID_ARG (a NULL pointer) or CUDA. A default build always
 * reports OK. */
qmlp_status qmlp_debug_bounds(int* site, unsigned long long* index);

/* Checking builds, tests only: from now on the decode kernel's checks allow
 * only the first gate_up_bank_bytes bytes of each of its gate and up record
 * banks (0: the whole bank), so its later weight steps fail their check --
 * the copies are then taken from the bank's start, which exists -- and
 * qmlp_debug_bounds reports site 1. Errors: INVALID_ARG (NULL handle, or a
 * default build). */
qmlp_status qmlp_debug_bounds_limit(qmlp_t* h, size_t gate_up_bank_bytes);

/*
 * Tensor-parallel shard over the intermediate dimension (vllm.cpp issue "tp>1
 * fp8w tail-MLP shard host-dequantizes every layer", "Proposed fix"): rank r
 * of n keeps gate/up rows [r I/n, (r+1) I/n) and the same columns of down, and
 * one sum over the ranks' [M, K] partials gives the layer's output.
 */
/* Create rank `rank`'s shard from the description of the WHOLE layer (the
 * same pointers and sizes qmlp_create takes; only the shard's rows and columns
 * are read). The handle's intermediate size is I / nranks; forward on it
 * returns bf16(sigma_d x its own partial). Limits: as qmlp_create, plus
 * 0 <= rank < nranks, I % nranks == 0, (I / nranks) % 16 == 0.
 * Errors: as qmlp_create (INVALID_ARG for a bad rank). */
qmlp_status qmlp_create_shard(qmlp_t** out, const qmlp_desc* desc, int rank, int nranks, qmlp_stream_t stream);

/* This shard's partial: partial[m, o] = sum over the shard's i of act[m,i]
 * Wd[o,i] in fp32 with no down factor (act = bf16 SwiGLU, as qmlp_forward).
 *  x = device bf16 [M, K]; partial = device fp32 [M, K].
 * Errors: as qmlp_forward. */
qmlp_status qmlp_forward_partial(qmlp_t* h, const void* x, int M, float* partial, qmlp_stream_t stream);

/* The exchange step after the partials are gathered (an all-gather of the
 * [M, K] fp32 partials, rank-major): out[m, o] = bf16( sigma_d[o] * sum over
 * r = 0..nranks-1 in rank order of partials[r][m][o] ). The order is fixed,
 * so every rank computes the same bytes.
 *  partials = device fp32 [nranks][M][K]; out = device bf16 [M, K]
 * nranks must equal the handle's. Errors: INVALID_ARG, SHAPE, ALIGNMENT,
 * ALIAS, CUDA. */
qmlp_status qmlp_shard_combine(qmlp_t* h, const float* partials, int nranks, int M, void* out,
                               qmlp_stream_t stream);

/* Rank, rank count and intermediate size of a handle (0, 1 and I for a
 * whole-layer handle). Returns 0 for a NULL handle, else 1. */
int qmlp_shard_info(qmlp_t* h, int* rank, int* nranks, int* I_shard);

/* Synchronize `stream` and report (then clear) a bounded-wait give-up
 * recorded by this handle's kernels: OK or DEVICE_TIMEOUT (CUDA on a sticky
 * device error). */
qmlp_status qmlp_check(qmlp_t* h, qmlp_stream_t stream);

/*
 * Routed-expert AWQ int4 group-32 MLP, one token (1Cat-vLLM PR "[Kernel][SM70]
 * Add native-g32 AWQ QPN M1 operator", "What it does"):
 *   for each route r in router order with 0 <= ids[r] < E:
 *     h      = x . W13[ids[r]]^T             (fp32 accumulation, N = 2I)
 *     g, u   = fp16(h[:I]), fp16(h[I:])
 *     act[r] = fp16(SiLU(g) * u)
 *     y[r]   = fp16(act[r] . W2[ids[r]]^T)   (fp32 accumulation, N = K)
 *   out = fp16( sum over valid r, in router order, of router_w[r] * y[r] )
 *         (fp32 accumulation, no atomics)
 * Weights: W[e, n, k] = half_fma(q, scale, bias): q is the u4 code (low nibble
 * = even k), one metadata record per (e, n, k/32): 4-byte {fp16 scale, fp16
 * bias} or 3-byte {fp16 scale, u8 zero} with bias = half(-zero*scale); records
 * are little-endian, scale first. Invalid ids (< 0 or >= E) contribute zero;
 * duplicate valid ids are separate routes with their own router weights.
 */
typedef struct {
    int E;            /* experts                     */
    int K;            /* hidden size (W13 in, W2 out) */
    int I;            /* intermediate per expert     */
    qmlp_meta meta;   /* 3- or 4-byte records        */
    const uint8_t* w13;       /* [E, 2I, K/2]              host or device */
    const uint8_t* w13_meta;  /* [E, 2I, K/32] x meta bytes              */
    const uint8_t* w2;        /* [E, K, I/2]                             */
    const uint8_t* w2_meta;   /* [E, K, I/32] x meta bytes               */
} qmlp_moe_desc;

typedef struct qmlp_moe_s qmlp_moe_t;

/* Create a routed-expert handle: copies the banks into handle-owned device
 * memory (reordered for the kernels, same bytes). Limits: K % 64 == 0,
 * I % 32 == 0, 32 <= I <= 1024, 64 <= K <= 16384, 1 <= E. Synchronizes.
 * Errors: INVALID_ARG, SHAPE, UNSUPPORTED_ARCH, OOM, CUDA. */
qmlp_status qmlp_moe_create(qmlp_moe_t** out, const qmlp_moe_desc* desc, qmlp_stream_t stream);
void qmlp_moe_destroy(qmlp_moe_t* h);

/* The routed-expert step above for one token.
 *  x          = device [K], bf16 or fp16 per xdt
 *  expert_ids = device int32 [topk]  (read on the device: may change between
 *               CUDA-graph replays)
 *  router_w   = device fp32 [topk]
 *  out        = device fp16 [K]
 * 1 <= topk <= 16. Allocates nothing; graph-capturable.
 * Errors: INVALID_ARG, ALIGNMENT, ALIAS (out overlaps x, ids or router_w),
 * SHAPE, CUDA. */
qmlp_status qmlp_moe_m1_forward(qmlp_moe_t* h, const void* x, qmlp_dtype xdt,
                                const int32_t* expert_ids, const float* router_w, int topk,
                                void* out, qmlp_stream_t stream);

/* As qmlp_moe_m1_forward, also writing the per-stage fp16 tensors (device):
 *  gu [topk, 2I], act [topk, I], y [topk, K]; rows of invalid routes are not
 *  written. Any of gu/act/y may be NULL. */
qmlp_status qmlp_moe_debug_stages(qmlp_moe_t* h, const void* x, qmlp_dtype xdt,
                                  const int32_t* expert_ids, const float* router_w, int topk,
                                  void* out, void* gu, void* act, void* y, qmlp_stream_t stream);

/* Reserve the workspace of multi-token calls: after this, qmlp_moe_forward
 * accepts 1 <= M <= max_tokens (routes = M * topk <= max_tokens * 16). Sizes
 * the handle-owned fp16 intermediates for max_tokens * 16 routes (act [.., I],
 * y [.., K]) plus the route and group lists; a larger later reservation adds
 * a larger workspace (the old one is freed by destroy). Allocates and
 * synchronizes the stream: call it before capturing graphs. A handle starts
 * with max_tokens = 1. Limits: K <= 8192 and E <= 8192 for M > 1.
 * Errors: INVALID_ARG, SHAPE, OOM, CUDA. */
qmlp_status qmlp_moe_reserve(qmlp_moe_t* h, int max_tokens, qmlp_stream_t stream);

/* The routed-expert step for M tokens, every token independently exactly as
 * qmlp_moe_m1_forward computes it (the source PR defines the one-token
 * operator; tokens do not interact):
 *  x          = device [M, K], bf16 or fp16 per xdt (row-major)
 *  expert_ids = device int32 [M, topk] (token t's routes in router order)
 *  router_w   = device fp32 [M, topk]
 *  out        = device fp16 [M, K]
 * M == 1 runs the one-token kernels. For M > 1 the valid routes of all tokens
 * are sorted by expert on the device and tokens that share an expert share
 * its weight reads (groups of up to 16 routes); results do not depend on the
 * grouping and are the same bytes every call. 1 <= topk <= 16,
 * 1 <= M <= the reserved max_tokens. Allocates nothing; graph-capturable.
 * Errors: INVALID_ARG, ALIGNMENT, ALIAS (out overlaps x, ids or router_w),
 * SHAPE, CUDA. */
qmlp_status qmlp_moe_forward(qmlp_moe_t* h, const void* x, qmlp_dtype xdt, const int32_t* expert_ids,
                             const float* router_w, int topk, int M, void* out, qmlp_stream_t stream);

qmlp_status qmlp_moe_check(qmlp_moe_t* h, qmlp_stream_t stream);

/* The routed-expert step of qmlp_moe_m1_forward without a handle, for callers
 * that cannot allocate device memory when they run it (an allocator-owning
 * runtime that forbids foreign allocations, or code whose device memory is
 * fixed after warm-up). It allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library call. The source pages have no counterpart; this is a
 * library convenience over the same kernels.
 *  banks = the expert banks as DEVICE pointers in the checkpoint layout of
 *          qmlp_moe_desc (read directly, never copied), w13/w2 16-byte aligned
 *  x, expert_ids, router_w, out: as qmlp_moe_m1_forward.
 * Scratch: the fp16 SwiGLU intermediate lives in one file-scope device array
 * of 16 x 1024 fp16 (32 KiB) that every GPU loading the library keeps until
 * exit; hence topk <= 16 and I <= 1024, larger sizes return QMLP_ERR_SHAPE.
 * The first call on a device looks up the array's device address (once per
 * device, on the current device); make that first call before any stream
 * capture. All calls share the array, which keeps the last call's contents
 * (no call needs it cleared: each route's row is written before it is read);
 * calls whose kernels overlap on the GPU (other streams, or other threads)
 * race on it and must be serialized by the caller. The looked-up address is
 * kept for the life of the process: resetting the device (cudaDeviceReset,
 * or tearing down and recreating its primary context) while the library
 * stays loaded is not supported for this entry point.
 * Errors: INVALID_ARG, ALIGNMENT, ALIAS (out overlaps x, ids, router_w or any
 * of the four banks), SHAPE, UNSUPPORTED_ARCH, CUDA. */
qmlp_status qmlp_moe_m1_forward_noalloc(const qmlp_moe_desc* banks, const void* x, qmlp_dtype xdt,
                                        const int32_t* expert_ids, const float* router_w, int topk,
                                        void* out, qmlp_stream_t stream);

/* Human-readable name of a status ("QMLP_OK", ...). Never NULL. */
const char* qmlp_status_str(qmlp_status s);

/* ABI version of this header (major * 100 + minor): 104 (dequantise-once GEMM path). */
int qmlp_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* QMLP_H */
