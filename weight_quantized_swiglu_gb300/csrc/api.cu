// api.cu -- the C ABI of libqmlp.so (declared in include/qmlp.h).
//
// Host side only: argument validation (before any launch), handle ownership,
// create-time residency and repack, workspace, and dispatch to the kernel
// families. There is no CPU compute path anywhere in this library: a failed
// launch returns QMLP_ERR_CUDA.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "internal.h"
#include "qmlp.h"

using namespace qmlp;

namespace {

constexpr int kMaxGemvM = 16;

// x of a host-buffer call, from pinned host memory (over the CPU-GPU link)
// into device memory, once: the decode kernel's CTAs would otherwise each read
// all of it over the link. The decode kernel, launched next with programmatic
// dependent launch, streams its first weights meanwhile.
__global__ void __launch_bounds__(256) fetch_x_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                      int n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

qmlp_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return QMLP_OK;
    if (e == cudaErrorMemoryAllocation) return QMLP_ERR_OOM;
    return QMLP_ERR_CUDA;
}

// Fault injection for host-side tests of the error paths: QMLP_FAULT_INJECT=
// "alloc" makes every device allocation fail, "alloc:N" the N-th one a handle
// makes (N >= 1; the earlier ones succeed and must be released), "launch"
// makes forward calls return QMLP_ERR_CUDA before launching anything.
bool fault(const char* what) {
    const char* v = getenv("QMLP_FAULT_INJECT");
    return v && strcmp(v, what) == 0;
}
long fault_alloc_index() {
    const char* v = getenv("QMLP_FAULT_INJECT");
    if (!v || strncmp(v, "alloc:", 6) != 0) return 0;
    return strtol(v + 6, nullptr, 10);
}

struct Owner {
    std::vector<void*> ptrs;
    long count = 0;  // allocations attempted by this owner
    cudaError_t alloc(void** p, size_t bytes) {
        *p = nullptr;
        ++count;
        if (fault("alloc") || fault_alloc_index() == count) return cudaErrorMemoryAllocation;
        if (bytes == 0) bytes = 16;
        cudaError_t e = cudaMalloc(p, bytes);
        if (e == cudaSuccess) ptrs.push_back(*p);
        return e;
    }
    void release() {
        for (void* p : ptrs) cudaFree(p);
        ptrs.clear();
    }
};

qmlp_status check_device(int* dev, int* num_sms) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return QMLP_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
        return QMLP_ERR_CUDA;
    if (major != 10 || minor != 3) return QMLP_ERR_UNSUPPORTED_ARCH;
    return QMLP_OK;
}

}  // namespace

struct qmlp_s {
    int fmt = 0, K = 0, I = 0, max_M = 0, device = 0, num_sms = 0;
    GemvProj gv[3];  // gate, up, down
    int layout_warps = 0;       // streaming warps of the GEMV record layout
    SplitPlan sp;               // I-partitioned decode plan (sp.G == 0: none)
    uint8_t* wsplit = nullptr;  // down records in the CTA-sliced layout
    float* spart = nullptr;     // [G][16][K] fp32 partial outputs
    unsigned long long* ticket = nullptr;  // grid-barrier ticket counter
    size_t lim_a = 0;  // index-check tests: bytes of the decode kernel's gate/up banks the checks allow (0: all)
    bool has_gemm = false;
    GemmProj gm_gu, gm_d;
    void* a16 = nullptr;       // fp16 [max_M, max(K, I)] (GEMM prescaled activations)
    uint8_t* wdec = nullptr;   // dequantise-once GEMM: one projection's decoded bf16 stage images
    size_t wdec_bytes = 0;
    uint8_t* wdec2 = nullptr;  // the down projection's images, decoded on `side` beside the gate/up GEMM
    size_t wdec2_bytes = 0;
    cudaStream_t side = nullptr;  // the handle's own stream for that predecode
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    float* gemm_ws = nullptr;  // split-K partials of the GEMM (small M)
    int* sig = nullptr;        // [max_M] per-token prescale exponents
    void* act = nullptr;       // bf16 [max_M, I]
    float* part = nullptr;     // split-K partials
    size_t part_cap = 0;
    int* counters = nullptr;   // [Nt(gate/up) + Nt(down)]
    int* err = nullptr;        // device error word
    unsigned* bar = nullptr;   // grid barrier {count, generation}
    void* x_stage = nullptr;   // bf16 [max_M, K] (forward_host)
    void* out_stage = nullptr; // bf16 [max_M, K]
    int rank = 0, nranks = 1;  // tensor-parallel shard of the intermediate dimension
    uint64_t wait_ns = 0;      // error-path tests: bounded-wait limit of the kernels (0: default)
    bool withhold = false;     // error-path tests: the kernels' producers skip their last step
    Owner mem;
};

// Frees everything a (possibly half-built) dense handle owns.
static void release_handle(qmlp_s* h) {
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->side) cudaStreamDestroy(h->side);
    h->mem.release();
    delete h;
}

// Largest token block one launch of the I-partitioned decode kernel takes: 16
// for FP8 (two 8-token column tiles, x staged in two halves) where the
// partition allows it, else 8. Measured on the 27B-class shape at 16 tokens:
// FP8 85 us against 96 us on the split-K GEMM; NVFP4 144 us against 87 us
// (its group scales cost two fp32 FMAs per accumulator element, and every CTA
// writes and the reduce kernel reads a [16, K] fp32 partial: 2 x 44.6 MB).
static int split_max_m(const qmlp_s* h) {
    if (!h->sp.G) return 0;
    return h->fmt == kFP8 && split_fits(h->fmt, kMaxGemvM, h->K, h->sp) ? kMaxGemvM : 8;
}

// Fewest tokens the automatic path sends to the tensor-core GEMM: past what
// one launch of the I-partitioned decode kernel takes (a second launch, which
// streams the weights again, loses to the split-K GEMM: measured on the
// 27B-class shape, 106-142 us for 9..16 tokens as two 8-token launches
// against 87-117 us). Shapes without the I partition decode 16 tokens per
// stream-K pass.
static int gemm_min_m(const qmlp_s* h) { return h->sp.G ? split_max_m(h) + 1 : kMaxGemvM + 1; }

// Fewest tokens the automatic path sends to the dequantise-once GEMM (each
// projection decoded once per call into fp16 stage images, then a GEMM
// without decoder warps), and the handle's max_M from which it holds the
// decode buffer (4 I K bytes: the larger projection). Measured on the
// 27B-class shape (NVFP4 / FP8, ms, decoder warps against decoded once):
// M = 512 0.322 / 0.345 against 0.357 / 0.386; M = 1024 0.607 / 0.644
// against 0.552 / 0.578; M = 8192 3.49 / 3.70 against 2.79 / 2.80. With the
// CTA-pair form: M = 640 0.360 / 0.386 against 0.378 / 0.409, M = 768
// 0.402 / 0.428 against 0.383 / 0.414 (below, the down projection's few
// 256-token tiles leave most pairs idle).
constexpr int kDqMinM = 768;
// The dequantise-once GEMM runs on CTA pairs from kPairMinM tokens (measured
// at M = 8192, NVFP4 / FP8: 2.67 / 2.72 ms against 2.79 / 2.81 on single
// CTAs; at M = 1024 0.520 / 0.550 against 0.553 / 0.578).
constexpr bool kDqPair = true;

struct qmlp_moe_s {
    int E = 0, K = 0, I = 0, meta = 0, device = 0, num_sms = 0;
    uint8_t *w13 = nullptr, *w13_meta = nullptr, *w2 = nullptr, *w2_meta = nullptr;
    __half* act_ws = nullptr;
    int* err = nullptr;
    // multi-token workspace (qmlp_moe_reserve): routes = max_tokens * 16
    int max_tokens = 1;
    __half* g_act = nullptr;   // [routes, I]
    __half* g_y = nullptr;     // [routes, K]
    int* g_route = nullptr;    // [routes]
    int4* g_groups = nullptr;  // [moe_grouped_max_groups(routes, E)]
    int* g_ngroups = nullptr;
    Owner mem;
};

extern "C" {

const char* qmlp_status_str(qmlp_status s) {
    switch (s) {
        case QMLP_OK: return "QMLP_OK";
        case QMLP_ERR_INVALID_ARG: return "QMLP_ERR_INVALID_ARG";
        case QMLP_ERR_ALIGNMENT: return "QMLP_ERR_ALIGNMENT";
        case QMLP_ERR_ALIAS: return "QMLP_ERR_ALIAS";
        case QMLP_ERR_SHAPE: return "QMLP_ERR_SHAPE";
        case QMLP_ERR_UNSUPPORTED_ARCH: return "QMLP_ERR_UNSUPPORTED_ARCH";
        case QMLP_ERR_OOM: return "QMLP_ERR_OOM";
        case QMLP_ERR_CUDA: return "QMLP_ERR_CUDA";
        case QMLP_ERR_DEVICE_TIMEOUT: return "QMLP_ERR_DEVICE_TIMEOUT";
        case QMLP_ERR_DEVICE_BOUNDS: return "QMLP_ERR_DEVICE_BOUNDS";
    }
    return "QMLP_ERR_UNKNOWN";
}

int qmlp_abi_version(void) { return 104; }

// ---------------------------------------------------------------------------
// dense MLP
// ---------------------------------------------------------------------------
static qmlp_status load_proj(qmlp_t* h, const qmlp_proj& src, int N, int K, int Rr, GemvProj& dst,
                             uint8_t** w_tmp, uint8_t** s_tmp, cudaStream_t s) {
    const bool nv = h->fmt == kNVFP4;
    const size_t wbytes = (size_t)N * (nv ? K / 2 : K);
    const size_t sbytes = nv ? (size_t)N * (K / 16) : (size_t)N * sizeof(float);
    void *wt = nullptr, *st = nullptr, *wc = nullptr;
    cudaError_t e;
    if ((e = h->mem.alloc(&wt, wbytes)) != cudaSuccess) return from_cuda(e);
    if ((e = h->mem.alloc(&st, sbytes)) != cudaSuccess) return from_cuda(e);
    if ((e = cudaMemcpyAsync(wt, src.w, wbytes, cudaMemcpyDefault, s)) != cudaSuccess) return QMLP_ERR_CUDA;
    if ((e = cudaMemcpyAsync(st, src.scale, sbytes, cudaMemcpyDefault, s)) != cudaSuccess) return QMLP_ERR_CUDA;
    dst.N = N;
    dst.K = K;
    dst.Nt = N / kTileRows;
    dst.Kc = (K + kChunkK - 1) / kChunkK;
    dst.TWr = h->layout_warps;
    dst.Rr = Rr;
    dst.Lr = (int)(((long)dst.Nt * dst.Kc + dst.TWr - 1) / dst.TWr);
    dst.Lr = (dst.Lr + dst.Rr - 1) / dst.Rr * dst.Rr;
    const size_t cbytes = gemv_codes_bytes(h->fmt, N, K, dst.Lr, dst.TWr);
    if ((e = h->mem.alloc(&wc, cbytes)) != cudaSuccess) return from_cuda(e);
    if (cudaMemsetAsync(wc, 0, cbytes, s) != cudaSuccess) return QMLP_ERR_CUDA;
    dst.wc = static_cast<const uint8_t*>(wc);
    if (nv) {
        dst.inv_g = 1.0f / src.global_scale;
        e = repack_nvfp4_gemv(static_cast<uint8_t*>(wt), static_cast<uint8_t*>(st), N, K, dst.Lr, dst.TWr,
                              dst.Rr, static_cast<uint8_t*>(wc), s);
    } else {
        dst.chs = static_cast<const float*>(st);  // kept: per-channel scales
        e = repack_fp8_gemv(static_cast<uint8_t*>(wt), N, K, dst.Lr, dst.TWr, dst.Rr, static_cast<uint8_t*>(wc), s);
    }
    if (e != cudaSuccess) return QMLP_ERR_CUDA;
    *w_tmp = static_cast<uint8_t*>(wt);
    *s_tmp = static_cast<uint8_t*>(st);
    return QMLP_OK;
}

static void free_tmp(qmlp_t* h, void* p) {
    if (!p) return;
    auto it = std::find(h->mem.ptrs.begin(), h->mem.ptrs.end(), p);
    if (it != h->mem.ptrs.end()) {
        cudaFree(p);
        h->mem.ptrs.erase(it);
    }
}

static qmlp_status validate_desc(const qmlp_desc* d) {
    if (!d) return QMLP_ERR_INVALID_ARG;
    if (d->fmt != QMLP_FMT_NVFP4 && d->fmt != QMLP_FMT_FP8_PC) return QMLP_ERR_INVALID_ARG;
    if (!d->gate.w || !d->gate.scale || !d->up.w || !d->up.scale || !d->down.w || !d->down.scale)
        return QMLP_ERR_INVALID_ARG;
    if (d->K < 16 || d->I < 16 || d->K > 65536 || d->I > 65536 || d->K % 16 || d->I % 16 || d->max_M < 1 ||
        d->max_M > 65536)
        return QMLP_ERR_SHAPE;
    if (d->fmt == QMLP_FMT_NVFP4 &&
        (!(d->gate.global_scale != 0.0f) || !(d->up.global_scale != 0.0f) || !(d->down.global_scale != 0.0f)))
        return QMLP_ERR_INVALID_ARG;
    return QMLP_OK;
}

// Build a handle from a validated description (the whole layer, or one
// shard's slice of it). `h` is a fresh handle whose Owner may already hold
// allocations; on error everything it owns is released and h is deleted.
static qmlp_status create_impl(qmlp_t* h, qmlp_t** out, const qmlp_desc* d, int dev, int sms, cudaStream_t s);

qmlp_status qmlp_create(qmlp_t** out, const qmlp_desc* d, qmlp_stream_t stream) {
    if (!out) return QMLP_ERR_INVALID_ARG;
    *out = nullptr;
    qmlp_status st = validate_desc(d);
    if (st != QMLP_OK) return st;
    int dev = 0, sms = 0;
    st = check_device(&dev, &sms);
    if (st != QMLP_OK) return st;
    return create_impl(new qmlp_t(), out, d, dev, sms, reinterpret_cast<cudaStream_t>(stream));
}

// Tensor-parallel shard over the intermediate dimension (vllm.cpp issue "tp>1
// fp8w tail-MLP shard ...", "Proposed fix": gate/up row-sliced, down
// column-sliced, one sum over the hidden output): rank r of n keeps gate/up
// rows [r I/n, (r+1) I/n) -- contiguous rows of the checkpoint -- and the same
// columns of down, copied out of each down row into a temporary buffer (a
// strided copy, host or device source) before the normal create.
qmlp_status qmlp_create_shard(qmlp_t** out, const qmlp_desc* d, int rank, int nranks, qmlp_stream_t stream) {
    if (!out) return QMLP_ERR_INVALID_ARG;
    *out = nullptr;
    qmlp_status st = validate_desc(d);
    if (st != QMLP_OK) return st;
    if (nranks < 1 || rank < 0 || rank >= nranks) return QMLP_ERR_INVALID_ARG;
    if (d->I % nranks || (d->I / nranks) % 16) return QMLP_ERR_SHAPE;
    int dev = 0, sms = 0;
    st = check_device(&dev, &sms);
    if (st != QMLP_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool nv = d->fmt == QMLP_FMT_NVFP4;
    const size_t K = (size_t)d->K, I = (size_t)d->I, Is = I / nranks, i0 = Is * rank;
    qmlp_desc sd = *d;
    sd.I = (int)Is;
    const qmlp_proj* src[2] = {&d->gate, &d->up};
    qmlp_proj* dst[2] = {&sd.gate, &sd.up};
    for (int p = 0; p < 2; ++p) {
        dst[p]->w = src[p]->w + i0 * (nv ? K / 2 : K);
        dst[p]->scale = static_cast<const uint8_t*>(src[p]->scale) + i0 * (nv ? K / 16 : sizeof(float));
    }
    qmlp_t* h = new qmlp_t();
    h->rank = rank;
    h->nranks = nranks;
    // the down columns [i0, i0 + Is) of every one of its K rows
    void *dw = nullptr, *ds = nullptr;
    cudaError_t e;
    const size_t wrow = nv ? I / 2 : I, wsh = nv ? Is / 2 : Is, woff = nv ? i0 / 2 : i0;
    if ((e = h->mem.alloc(&dw, K * wsh)) != cudaSuccess) st = from_cuda(e);
    else if (cudaMemcpy2DAsync(dw, wsh, d->down.w + woff, wrow, wsh, K, cudaMemcpyDefault, s) != cudaSuccess)
        st = QMLP_ERR_CUDA;
    if (st == QMLP_OK && nv) {
        if ((e = h->mem.alloc(&ds, K * (Is / 16))) != cudaSuccess) st = from_cuda(e);
        else if (cudaMemcpy2DAsync(ds, Is / 16, static_cast<const uint8_t*>(d->down.scale) + i0 / 16, I / 16,
                                   Is / 16, K, cudaMemcpyDefault, s) != cudaSuccess)
            st = QMLP_ERR_CUDA;
    }
    if (st != QMLP_OK) {
        cudaStreamSynchronize(s);
        release_handle(h);
        return st;
    }
    sd.down.w = static_cast<const uint8_t*>(dw);
    if (nv) sd.down.scale = ds;  // FP8 keeps the K per-channel scales of down as they are
    return create_impl(h, out, &sd, dev, sms, s);
}


static qmlp_status create_impl(qmlp_t* h, qmlp_t** out, const qmlp_desc* d, int dev, int sms, cudaStream_t s) {
    qmlp_status st = QMLP_OK;
    // allocations made for the shard's down columns before this point are
    // temporaries: freed once the repack has consumed them
    std::vector<void*> pre_tmp(h->mem.ptrs);
    h->fmt = d->fmt;
    h->K = d->K;
    h->I = d->I;
    h->max_M = d->max_M;
    h->device = dev;
    h->num_sms = sms;
    h->sp = plan_split(d->fmt, d->K, d->I, sms);
    h->layout_warps = h->sp.G ? h->sp.G * 16 : gemv_layout_warps(sms);
    uint8_t* tmp[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    const qmlp_proj* srcs[3] = {&d->gate, &d->up, &d->down};
    const int Ns[3] = {d->I, d->I, d->K}, Ks[3] = {d->K, d->K, d->I};
    cudaError_t e = cudaSuccess;
    for (int p = 0; p < 3 && st == QMLP_OK; ++p)
        st = load_proj(h, *srcs[p], Ns[p], Ks[p], p < 2 ? gemv_recs_pair(d->fmt) : gemv_recs_single(d->fmt), h->gv[p],
                       &tmp[2 * p], &tmp[2 * p + 1], s);

    // the CTA-sliced copy of the down projection for the I-partitioned kernel
    if (st == QMLP_OK && h->sp.G) {
        void *wsp = nullptr, *part = nullptr, *tk = nullptr;
        const size_t wb = split_codes_bytes(h->fmt, h->sp);
        if ((e = h->mem.alloc(&wsp, wb)) != cudaSuccess) st = from_cuda(e);
        else if ((e = h->mem.alloc(&part, split_part_elems(d->K, h->sp) * sizeof(float))) != cudaSuccess)
            st = from_cuda(e);
        else if ((e = h->mem.alloc(&tk, 64)) != cudaSuccess) st = from_cuda(e);
        else if (cudaMemsetAsync(wsp, 0, wb, s) != cudaSuccess || cudaMemsetAsync(tk, 0, 64, s) != cudaSuccess)
            st = QMLP_ERR_CUDA;
        else if ((h->fmt == kNVFP4 ? repack_nvfp4_split(tmp[4], tmp[5], d->K, d->I, h->sp, static_cast<uint8_t*>(wsp), s)
                                   : repack_fp8_split(tmp[4], d->K, d->I, h->sp, static_cast<uint8_t*>(wsp), s)) !=
                 cudaSuccess)
            st = QMLP_ERR_CUDA;
        if (st == QMLP_OK) {
            h->wsplit = static_cast<uint8_t*>(wsp);
            h->spart = static_cast<float*>(part);
            h->ticket = static_cast<unsigned long long*>(tk);
        }
    }

    if (st == QMLP_OK && d->max_M >= gemm_min_m(h) && gemm_supported(d->K, 2 * d->I) && gemm_supported(d->I, d->K)) {
        void *gu = nullptr, *dn = nullptr;
        const bool nv = h->fmt == kNVFP4;
        if ((e = h->mem.alloc(&gu, gemm_tiles_bytes(h->fmt, 2 * d->I, d->K))) != cudaSuccess) st = from_cuda(e);
        else if ((e = h->mem.alloc(&dn, gemm_tiles_bytes(h->fmt, d->K, d->I))) != cudaSuccess) st = from_cuda(e);
        else if (nv ? (repack_nvfp4_gemm(tmp[0], tmp[1], tmp[2], tmp[3], 2 * d->I, d->K, true,
                                         static_cast<uint8_t*>(gu), s) != cudaSuccess ||
                       repack_nvfp4_gemm(tmp[4], tmp[5], nullptr, nullptr, d->K, d->I, false,
                                         static_cast<uint8_t*>(dn), s) != cudaSuccess)
                    : (repack_fp8_gemm(tmp[0], tmp[2], 2 * d->I, d->K, true, static_cast<uint8_t*>(gu), s) !=
                           cudaSuccess ||
                       repack_fp8_gemm(tmp[4], nullptr, d->K, d->I, false, static_cast<uint8_t*>(dn), s) !=
                           cudaSuccess))
            st = QMLP_ERR_CUDA;
        if (st == QMLP_OK) {
            h->has_gemm = true;
            h->gm_gu.fmt = h->gm_d.fmt = h->fmt;
            h->gm_gu.tiles = static_cast<uint8_t*>(gu);
            h->gm_gu.N = 2 * d->I;
            h->gm_gu.K = d->K;
            h->gm_gu.inv_g0 = h->gv[0].inv_g;
            h->gm_gu.inv_g1 = h->gv[1].inv_g;
            h->gm_gu.cs0 = h->gv[0].chs;  // FP8: the per-channel scales (NVFP4: null)
            h->gm_gu.cs1 = h->gv[1].chs;
            h->gm_gu.interleaved = true;
            h->gm_d.tiles = static_cast<uint8_t*>(dn);
            h->gm_d.N = d->K;
            h->gm_d.K = d->I;
            h->gm_d.inv_g0 = h->gm_d.inv_g1 = h->gv[2].inv_g;
            h->gm_d.cs0 = h->gm_d.cs1 = h->gv[2].chs;
            // GEMM workspace: prescaled fp16 activations (x, then act) and
            // the per-token exponents
            const size_t cols = (size_t)std::max(d->K, d->I);
            if ((e = h->mem.alloc(&h->a16, (size_t)d->max_M * cols * 2)) != cudaSuccess) st = from_cuda(e);
            else if ((e = h->mem.alloc(reinterpret_cast<void**>(&h->gemm_ws),
                                       gemm_splitk_ws_elems(sms) * sizeof(float))) != cudaSuccess)
                st = from_cuda(e);
            else if ((e = h->mem.alloc(reinterpret_cast<void**>(&h->sig), (size_t)d->max_M * sizeof(int))) !=
                     cudaSuccess)
                st = from_cuda(e);
        }
        if (st == QMLP_OK && d->max_M >= kDqMinM) {
            // one buffer for a projection's images (gate/up, or down alone in
            // a stage call), one for the down images of a whole forward, and
            // the side stream that decodes those while the gate/up GEMM runs
            const size_t b2 = gemm_decoded_bytes(d->K, d->I);
            const size_t b = std::max(gemm_decoded_bytes(2 * d->I, d->K), b2);
            void *p = nullptr, *p2 = nullptr;
            if ((e = h->mem.alloc(&p, b)) != cudaSuccess) st = from_cuda(e);
            else if ((e = h->mem.alloc(&p2, b2)) != cudaSuccess) st = from_cuda(e);
            else if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
                     cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
                     cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess)
                st = QMLP_ERR_CUDA;
            h->wdec = static_cast<uint8_t*>(p);
            h->wdec_bytes = b;
            h->wdec2 = static_cast<uint8_t*>(p2);
            h->wdec2_bytes = b2;
        }
    }
    // workspace
    if (st == QMLP_OK) {
        void* p = nullptr;
        const size_t Ntot = (size_t)(d->I / kTileRows) + (size_t)(d->K / kTileRows);
        h->part_cap = std::max(gemv_part_elems(d->K, d->I, sms), gemv_stream_part_elems(d->K, d->I, sms));
        if ((e = h->mem.alloc(&h->act, (size_t)d->max_M * d->I * 2)) != cudaSuccess) st = from_cuda(e);
        else if ((e = h->mem.alloc(&p, h->part_cap * sizeof(float))) != cudaSuccess) st = from_cuda(e);
        else {
            h->part = static_cast<float*>(p);
            if ((e = h->mem.alloc(&p, Ntot * sizeof(int) + 16)) != cudaSuccess) st = from_cuda(e);
            else {
                h->counters = static_cast<int*>(p);
                if (cudaMemsetAsync(p, 0, Ntot * sizeof(int) + 16, s) != cudaSuccess) st = QMLP_ERR_CUDA;
            }
        }
        if (st == QMLP_OK) {
            if ((e = h->mem.alloc(&p, 64)) != cudaSuccess) st = from_cuda(e);
            else {
                h->err = static_cast<int*>(p);
                h->bar = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(p) + 32);
                if (cudaMemsetAsync(p, 0, 64, s) != cudaSuccess) st = QMLP_ERR_CUDA;
            }
        }
        if (st == QMLP_OK && (e = h->mem.alloc(&h->x_stage, (size_t)d->max_M * d->K * 2)) != cudaSuccess)
            st = from_cuda(e);
        if (st == QMLP_OK && (e = h->mem.alloc(&h->out_stage, (size_t)d->max_M * d->K * 2)) != cudaSuccess)
            st = from_cuda(e);
    }
    if (st == QMLP_OK && cudaStreamSynchronize(s) != cudaSuccess) st = QMLP_ERR_CUDA;
    // the checkpoint-layout copies are no longer needed (FP8 keeps its scales)
    if (st == QMLP_OK) {
        for (int p = 0; p < 3; ++p) {
            free_tmp(h, tmp[2 * p]);
            if (h->fmt == kNVFP4) free_tmp(h, tmp[2 * p + 1]);
        }
        for (void* p : pre_tmp) free_tmp(h, p);
    }
    if (st != QMLP_OK) {
        cudaStreamSynchronize(s);
        release_handle(h);
        return st;
    }
    *out = h;
    return QMLP_OK;
}

void qmlp_destroy(qmlp_t* h) {
    if (!h) return;
    cudaDeviceSynchronize();
    release_handle(h);
}

static qmlp_status validate_fwd(qmlp_t* h, const void* x, int M, const void* out, size_t out_elem_bytes,
                                int out_cols) {
    if (!h || !x || !out) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_M) return QMLP_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(out)) return QMLP_ERR_ALIGNMENT;
    (void)out_elem_bytes;
    (void)out_cols;
    return QMLP_OK;
}

static bool valid_path(qmlp_path p) {
    return p == QMLP_PATH_AUTO || p == QMLP_PATH_GEMV || p == QMLP_PATH_GEMM || p == QMLP_PATH_GEMM_PAIR ||
           p == QMLP_PATH_GEMM_DQ;
}

static bool use_gemm(qmlp_t* h, qmlp_path path, int M) {
    if (path == QMLP_PATH_GEMV) return false;
    if (path == QMLP_PATH_GEMM || path == QMLP_PATH_GEMM_PAIR || path == QMLP_PATH_GEMM_DQ) return true;
    return h->has_gemm && M >= gemm_min_m(h);
}

// The decode buffer for a GEMM call (null: the decoder warps decode).
static uint8_t* dq_buffer(const qmlp_t* h, qmlp_path path, int M) {
    if (path == QMLP_PATH_GEMM_DQ) return h->wdec;
    return path == QMLP_PATH_AUTO && M >= kDqMinM ? h->wdec : nullptr;
}

// stage bit 0: gate/up + SwiGLU (x -> workspace act); bit 1: down (act ->
// out). With out_f32 the down stage writes its fp32 sums without the down
// factor there (a tensor-parallel shard's partial) instead of bf16 to out.
static qmlp_status run_stages(qmlp_t* h, qmlp_path path, int stages, const void* x, int M, void* out,
                              cudaStream_t s, bool host_io = false, float* out_f32 = nullptr) {
    if (fault("launch")) return QMLP_ERR_CUDA;
    const bool gemm = use_gemm(h, path, M);
    if (gemm && !h->has_gemm) return QMLP_ERR_SHAPE;
    if (path == QMLP_PATH_GEMM_PAIR && M < kPairMinM) return QMLP_ERR_SHAPE;
    if (path == QMLP_PATH_GEMM_DQ && !h->wdec) return QMLP_ERR_SHAPE;
    if (gemm) {
        GemmLaunch g;
        g.wdec = dq_buffer(h, path, M);
        g.wdec_bytes = h->wdec_bytes;
        g.pair = path == QMLP_PATH_GEMM_PAIR || (g.wdec && kDqPair && M >= kPairMinM);
        g.M = M;
        g.err = h->err;
        g.a16 = h->a16;
        g.sig = h->sig;
        g.ws = h->gemm_ws;
        g.wait_ns = h->wait_ns;
        g.withhold = h->withhold;
        // dequantise-once, whole block: the gate/up images here, then the
        // down images on the side stream while the gate/up GEMM runs (the
        // fork follows everything already on s, so the previous call's down
        // GEMM has finished reading wdec2)
        const bool fork = g.wdec && stages == 3 && h->wdec2 && h->side;
        if (fork && (launch_gemm_predecode(h->gm_gu, h->wdec, h->wdec_bytes, h->num_sms, s) != cudaSuccess ||
                     cudaEventRecord(h->ev_fork, s) != cudaSuccess ||
                     cudaStreamWaitEvent(h->side, h->ev_fork, 0) != cudaSuccess ||
                     launch_gemm_predecode(h->gm_d, h->wdec2, h->wdec2_bytes, h->num_sms, h->side) != cudaSuccess ||
                     cudaEventRecord(h->ev_join, h->side) != cudaSuccess))
            return QMLP_ERR_CUDA;
        g.images_ready = fork;
        if (stages & 1) {
            g.epi = kEpiSwiGLU;
            g.w = h->gm_gu;
            g.a = x;
            g.out = h->act;
            if (launch_gemm(g, h->num_sms, s) != cudaSuccess) return QMLP_ERR_CUDA;
        }
        if (stages & 2) {
            if (fork) {
                if (cudaStreamWaitEvent(s, h->ev_join, 0) != cudaSuccess) return QMLP_ERR_CUDA;
                g.wdec = h->wdec2;
                g.wdec_bytes = h->wdec2_bytes;
            }
            g.epi = out_f32 ? kEpiRaw : kEpiPlain;
            g.raw_sel = 0;
            g.w = h->gm_d;
            g.a = h->act;
            g.out = out_f32 ? static_cast<void*>(out_f32) : out;
            if (launch_gemm(g, h->num_sms, s) != cudaSuccess) return QMLP_ERR_CUDA;
        }
        return QMLP_OK;
    }
    const size_t Ntg = (size_t)(h->I / kTileRows);
    // the whole MLP in token blocks: up to 8 tokens per launch of the
    // I-partitioned kernel when the shape has a partition (its shared-memory
    // staging of x grows with M), else 16 per stream-K / split-K pass
    const bool split = stages == 3 && h->sp.G && split_fits(h->fmt, 1, h->K, h->sp);
    const int block = split ? split_max_m(h) : kMaxGemvM;
    for (int m0 = 0; m0 < M; m0 += block) {
        const int mb = std::min(block, M - m0);
        const void* xb = static_cast<const uint8_t*>(x) + (size_t)m0 * h->K * 2;
        void* ab = static_cast<uint8_t*>(h->act) + (size_t)m0 * h->I * 2;
        void* ob = out_f32 ? static_cast<void*>(out_f32 + (size_t)m0 * h->K)
                           : static_cast<void*>(static_cast<uint8_t*>(out) + (size_t)m0 * h->K * 2);
        GemvStreamPhase A, B;
        A.epi = kEpiSwiGLU;
        A.p0 = h->gv[0];
        A.p1 = h->gv[1];
        A.x = xb;
        A.out = ab;
        A.counters = h->counters;
        B.epi = out_f32 ? kEpiRaw : kEpiPlain;
        B.p0 = h->gv[2];
        B.x = ab;
        B.out = ob;
        B.counters = h->counters + Ntg;
        const bool fitA = gemv_stream_fits(h->fmt, mb, h->K, 2, h->gv[0].Rr),
                   fitB = gemv_stream_fits(h->fmt, mb, h->I, 1, h->gv[2].Rr);
        const bool fitAB = gemv_stream_fits(h->fmt, mb, std::max(h->K, h->I), 2, h->gv[0].Rr) &&
                           gemv_stream_fits(h->fmt, mb, std::max(h->K, h->I), 1, h->gv[2].Rr);
        if (split && split_fits(h->fmt, mb, h->K, h->sp)) {
            SplitLaunch S;
            S.fmt = h->fmt;
            S.M = mb;
            S.K = h->K;
            S.I = h->I;
            S.gate = h->gv[0];
            S.up = h->gv[1];
            S.wdown = h->wsplit;
            S.chsd = h->gv[2].chs;
            S.invd = h->gv[2].inv_g;
            S.x = xb;
            S.x_in_host = host_io;
            S.act_out = ab;  // the workspace act (qmlp_forward_debug returns it)
            S.out = out_f32 ? nullptr : ob;
            S.out_f32 = out_f32 ? static_cast<float*>(ob) : nullptr;
            S.part = h->spart;
            S.ticket = h->ticket;
            S.err = h->err;
            S.wait_ns = h->wait_ns;
            S.withhold = h->withhold;
            S.lim_a = h->lim_a;
            if (launch_split(S, h->sp, s) != cudaSuccess) return QMLP_ERR_CUDA;
            continue;
        }
        if (stages == 3 && fitAB && !out_f32) {
            if (launch_gemv_stream(h->fmt, mb, A, &B, h->part, h->part_cap, h->bar, h->err, h->num_sms, s) !=
                cudaSuccess)
                return QMLP_ERR_CUDA;
            continue;
        }
        GemvLaunch L;
        L.fmt = h->fmt;
        L.M = mb;
        L.part = h->part;
        L.part_cap = h->part_cap;
        if (stages & 1) {
            if (fitA) {
                if (launch_gemv_stream(h->fmt, mb, A, nullptr, h->part, h->part_cap, h->bar, h->err, h->num_sms,
                                       s) != cudaSuccess)
                    return QMLP_ERR_CUDA;
            } else {
                L.epi = kEpiSwiGLU;
                L.p0 = h->gv[0];
                L.p1 = h->gv[1];
                L.x = xb;
                L.out = ab;
                L.counters = h->counters;
                if (launch_gemv(L, h->num_sms, s) != cudaSuccess) return QMLP_ERR_CUDA;
            }
        }
        if (stages & 2) {
            if (fitB) {
                if (launch_gemv_stream(h->fmt, mb, B, nullptr, h->part, h->part_cap, h->bar, h->err, h->num_sms,
                                       s) != cudaSuccess)
                    return QMLP_ERR_CUDA;
            } else {
                L.epi = out_f32 ? kEpiRaw : kEpiPlain;
                L.p0 = h->gv[2];
                L.p1 = GemvProj();
                L.x = ab;
                L.out = ob;
                L.counters = h->counters + Ntg;
                if (launch_gemv(L, h->num_sms, s) != cudaSuccess) return QMLP_ERR_CUDA;
            }
        }
    }
    return QMLP_OK;
}

static qmlp_status run_forward(qmlp_t* h, qmlp_path path, const void* x, int M, void* out, cudaStream_t s,
                               bool host_io = false) {
    return run_stages(h, path, 3, x, M, out, s, host_io);
}

// Device address of a host buffer the GPU can read and write in place
// (pinned, mapped into the device address space), else nullptr.
static void* device_alias(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

qmlp_status qmlp_forward_path(qmlp_t* h, qmlp_path path, const void* x, int M, void* out,
                              qmlp_stream_t stream) {
    qmlp_status st = validate_fwd(h, x, M, out, 2, 0);
    if (st != QMLP_OK) return st;
    if (!valid_path(path)) return QMLP_ERR_INVALID_ARG;
    const size_t xb = (size_t)M * h->K * 2;
    if (overlaps(x, xb, out, xb)) return QMLP_ERR_ALIAS;
    if (overlaps(out, xb, h->act, (size_t)h->max_M * h->I * 2)) return QMLP_ERR_ALIAS;
    return run_forward(h, path, x, M, out, reinterpret_cast<cudaStream_t>(stream));
}

qmlp_status qmlp_forward_stage(qmlp_t* h, int stage, qmlp_path path, const void* x, int M, void* out,
                               qmlp_stream_t stream) {
    if (!h) return QMLP_ERR_INVALID_ARG;
    if (!valid_path(path)) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_M) return QMLP_ERR_SHAPE;
    if (stage == 0) {
        if (!x || out) return QMLP_ERR_INVALID_ARG;
        if (!aligned16(x)) return QMLP_ERR_ALIGNMENT;
        if (overlaps(x, (size_t)M * h->K * 2, h->act, (size_t)h->max_M * h->I * 2)) return QMLP_ERR_ALIAS;
        return run_stages(h, path, 1, x, M, nullptr, reinterpret_cast<cudaStream_t>(stream));
    }
    if (stage == 1) {
        if (x || !out) return QMLP_ERR_INVALID_ARG;
        if (!aligned16(out)) return QMLP_ERR_ALIGNMENT;
        if (overlaps(out, (size_t)M * h->K * 2, h->act, (size_t)h->max_M * h->I * 2)) return QMLP_ERR_ALIAS;
        return run_stages(h, path, 2, nullptr, M, out, reinterpret_cast<cudaStream_t>(stream));
    }
    return QMLP_ERR_INVALID_ARG;
}

qmlp_status qmlp_forward(qmlp_t* h, const void* x, int M, void* out, qmlp_stream_t stream) {
    return qmlp_forward_path(h, QMLP_PATH_AUTO, x, M, out, stream);
}

qmlp_status qmlp_forward_debug(qmlp_t* h, qmlp_path path, const void* x, int M, void* act, void* out,
                               qmlp_stream_t stream) {
    qmlp_status st = qmlp_forward_path(h, path, x, M, out, stream);
    if (st != QMLP_OK) return st;
    if (!act) return QMLP_ERR_INVALID_ARG;
    if (!aligned16(act)) return QMLP_ERR_ALIGNMENT;
    const size_t ab = (size_t)M * h->I * 2;
    if (overlaps(act, ab, x, (size_t)M * h->K * 2) || overlaps(act, ab, out, (size_t)M * h->K * 2))
        return QMLP_ERR_ALIAS;
    return cudaMemcpyAsync(act, h->act, ab, cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? QMLP_OK
               : QMLP_ERR_CUDA;
}

qmlp_status qmlp_forward_host(qmlp_t* h, const void* x_host, int M, void* out_host, qmlp_stream_t stream) {
    if (!h || !x_host || !out_host) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_M) return QMLP_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)M * h->K * 2;
    // pinned buffers: the kernels read x and write out in host memory over the
    // coherent CPU-GPU link, with no copy-engine round trips
    void* xd = device_alias(x_host);
    void* od = device_alias(out_host);
    if (xd && od && aligned16(xd) && aligned16(od) && !overlaps(x_host, bytes, out_host, bytes)) {
        // x is fetched once into the handle's device stage (an ordinary
        // launch: the previous call may still read that stage); the output is
        // written in place over the link
        if (fault("launch")) return QMLP_ERR_CUDA;
        const int n16 = (int)(bytes / 16);
        fetch_x_kernel<<<std::min(8, (n16 + 255) / 256), 256, 0, s>>>(static_cast<const uint4*>(xd),
                                                                      static_cast<uint4*>(h->x_stage), n16);
        if (cudaPeekAtLastError() != cudaSuccess) return QMLP_ERR_CUDA;
        qmlp_status st = run_forward(h, QMLP_PATH_AUTO, h->x_stage, M, od, s);
        if (st != QMLP_OK) return st;
        return cudaStreamSynchronize(s) == cudaSuccess ? QMLP_OK : QMLP_ERR_CUDA;
    }
    if (cudaMemcpyAsync(h->x_stage, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return QMLP_ERR_CUDA;
    qmlp_status st = run_forward(h, QMLP_PATH_AUTO, h->x_stage, M, h->out_stage, s);
    if (st != QMLP_OK) return st;
    if (cudaMemcpyAsync(out_host, h->out_stage, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return QMLP_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? QMLP_OK : QMLP_ERR_CUDA;
}

qmlp_status qmlp_debug_project(qmlp_t* h, int which, qmlp_path path, const void* x, int M, float* y,
                               qmlp_stream_t stream) {
    if (!h || !x || !y) return QMLP_ERR_INVALID_ARG;
    if (which < 0 || which > 2) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_M) return QMLP_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(y)) return QMLP_ERR_ALIGNMENT;
    const GemvProj& P = h->gv[which];
    if (overlaps(x, (size_t)M * P.K * 2, y, (size_t)M * P.N * 4)) return QMLP_ERR_ALIAS;
    if (fault("launch")) return QMLP_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (use_gemm(h, path, M)) {
        if (!h->has_gemm) return QMLP_ERR_SHAPE;
        if (path == QMLP_PATH_GEMM_PAIR && M < kPairMinM) return QMLP_ERR_SHAPE;
        if (path == QMLP_PATH_GEMM_DQ && !h->wdec) return QMLP_ERR_SHAPE;
        GemmLaunch g;
        g.wdec = dq_buffer(h, path, M);
        g.wdec_bytes = h->wdec_bytes;
        g.pair = path == QMLP_PATH_GEMM_PAIR || (g.wdec && kDqPair && M >= kPairMinM);
        g.epi = kEpiRaw;
        g.raw_sel = which == 1 ? 1 : 0;
        g.w = which < 2 ? h->gm_gu : h->gm_d;
        g.a = x;
        g.M = M;
        g.out = y;
        g.a16 = h->a16;
        g.sig = h->sig;
        g.err = h->err;
        return launch_gemm(g, h->num_sms, s) == cudaSuccess ? QMLP_OK : QMLP_ERR_CUDA;
    }
    const size_t Ntg = (size_t)(h->I / kTileRows);
    for (int m0 = 0; m0 < M; m0 += kMaxGemvM) {
        const int mb = std::min(kMaxGemvM, M - m0);
        if (gemv_stream_fits(h->fmt, mb, P.K, 1, P.Rr)) {
            GemvStreamPhase A;
            A.epi = kEpiRaw;
            A.p0 = P;
            A.x = static_cast<const uint8_t*>(x) + (size_t)m0 * P.K * 2;
            A.out = y + (size_t)m0 * P.N;
            A.counters = which == 2 ? h->counters + Ntg : h->counters;
            if (launch_gemv_stream(h->fmt, mb, A, nullptr, h->part, h->part_cap, h->bar, h->err, h->num_sms, s) !=
                cudaSuccess)
                return QMLP_ERR_CUDA;
            continue;
        }
        GemvLaunch L;
        L.fmt = h->fmt;
        L.epi = kEpiRaw;
        L.p0 = P;
        L.x = static_cast<const uint8_t*>(x) + (size_t)m0 * P.K * 2;
        L.M = mb;
        L.out = y + (size_t)m0 * P.N;
        L.part = h->part;
        L.part_cap = h->part_cap;
        L.counters = which == 2 ? h->counters + Ntg : h->counters;
        if (launch_gemv(L, h->num_sms, s) != cudaSuccess) return QMLP_ERR_CUDA;
    }
    return QMLP_OK;
}

qmlp_status qmlp_check(qmlp_t* h, qmlp_stream_t stream) {
    if (!h) return QMLP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return QMLP_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QMLP_ERR_CUDA;
    if (v != 0) {
        cudaMemset(h->err, 0, sizeof(int));
        // a launch that gave up may have left the grid-barrier ticket off a
        // multiple of the CTA count: start the count again
        if (h->ticket) cudaMemset(h->ticket, 0, sizeof(unsigned long long));
        return QMLP_ERR_DEVICE_TIMEOUT;
    }
    return QMLP_OK;
}

int qmlp_decode_ctas(qmlp_t* h) { return h ? h->sp.G : 0; }

qmlp_status qmlp_debug_set_wait(qmlp_t* h, uint64_t limit_ns, int withhold_last_step) {
    if (!h) return QMLP_ERR_INVALID_ARG;
    h->wait_ns = limit_ns;
    h->withhold = withhold_last_step != 0;
    return QMLP_OK;
}

int qmlp_debug_bounds_enabled(void) {
#ifdef QMLP_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

qmlp_status qmlp_debug_bounds(int* site, unsigned long long* index) {
    if (!site || !index) return QMLP_ERR_INVALID_ARG;
    *site = 0;
    *index = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return QMLP_ERR_CUDA;
    cudaError_t (*const units[])(unsigned long long*) = {bounds_take_gemv_split, bounds_take_gemm_tc,
                                                          bounds_take_gemv_stream, bounds_take_gemv_dec,
                                                          bounds_take_moe_awq, bounds_take_moe_grouped,
                                                          bounds_take_tp_shard};
    unsigned long long first = 0;
    for (auto take : units) {
        unsigned long long v = 0;
        if (take(&v) != cudaSuccess) return QMLP_ERR_CUDA;
        if (!first) first = v;  // every unit's word is read, and so cleared
    }
    if (!first) return QMLP_OK;
    *site = (int)(first >> 48);
    *index = first & 0xffffffffffffull;
    return QMLP_ERR_DEVICE_BOUNDS;
}

qmlp_status qmlp_debug_bounds_limit(qmlp_t* h, size_t gate_up_bank_bytes) {
    if (!h || !qmlp_debug_bounds_enabled()) return QMLP_ERR_INVALID_ARG;
    h->lim_a = gate_up_bank_bytes;
    return QMLP_OK;
}

qmlp_status qmlp_debug_split(qmlp_t* h, const void* x, const void* act_in, int M, float* g, float* u,
                             float* out_f32, qmlp_stream_t stream) {
    if (!h || !x || !act_in || !g || !u || !out_f32) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_M) return QMLP_ERR_SHAPE;
    if (!h->sp.G || M > split_max_m(h) || !split_fits(h->fmt, M, h->K, h->sp)) return QMLP_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(act_in) || !aligned16(g) || !aligned16(u) || !aligned16(out_f32))
        return QMLP_ERR_ALIGNMENT;
    const size_t xb = (size_t)M * h->K * 2, ab = (size_t)M * h->I * 2, gb = (size_t)M * h->I * 4,
                 ob = (size_t)M * h->K * 4;
    const void* outs[3] = {g, u, out_f32};
    const size_t osz[3] = {gb, gb, ob};
    for (int i = 0; i < 3; ++i) {
        if (overlaps(outs[i], osz[i], x, xb) || overlaps(outs[i], osz[i], act_in, ab)) return QMLP_ERR_ALIAS;
        for (int j = 0; j < i; ++j)
            if (overlaps(outs[i], osz[i], outs[j], osz[j])) return QMLP_ERR_ALIAS;
    }
    if (fault("launch")) return QMLP_ERR_CUDA;
    SplitLaunch S;
    S.fmt = h->fmt;
    S.M = M;
    S.K = h->K;
    S.I = h->I;
    S.gate = h->gv[0];
    S.up = h->gv[1];
    S.wdown = h->wsplit;
    S.chsd = h->gv[2].chs;
    S.invd = h->gv[2].inv_g;
    S.x = x;
    S.act_out = h->act;
    S.out_f32 = out_f32;
    S.act_in = act_in;
    S.dbg_g = g;
    S.dbg_u = u;
    S.part = h->spart;
    S.ticket = h->ticket;
    S.err = h->err;
    S.wait_ns = h->wait_ns;
    S.withhold = h->withhold;
    S.lim_a = h->lim_a;
    return launch_split(S, h->sp, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QMLP_OK
                                                                                          : QMLP_ERR_CUDA;
}

qmlp_status qmlp_forward_partial(qmlp_t* h, const void* x, int M, float* partial, qmlp_stream_t stream) {
    if (!h || !x || !partial) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_M) return QMLP_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(partial)) return QMLP_ERR_ALIGNMENT;
    const size_t pb = (size_t)M * h->K * 4;
    if (overlaps(partial, pb, x, (size_t)M * h->K * 2) || overlaps(partial, pb, h->act, (size_t)h->max_M * h->I * 2))
        return QMLP_ERR_ALIAS;
    return run_stages(h, QMLP_PATH_AUTO, 3, x, M, nullptr, reinterpret_cast<cudaStream_t>(stream), false, partial);
}

qmlp_status qmlp_shard_combine(qmlp_t* h, const float* partials, int nranks, int M, void* out,
                               qmlp_stream_t stream) {
    if (!h || !partials || !out) return QMLP_ERR_INVALID_ARG;
    if (nranks != h->nranks) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_M) return QMLP_ERR_SHAPE;
    if (!aligned16(partials) || !aligned16(out)) return QMLP_ERR_ALIGNMENT;
    if (overlaps(out, (size_t)M * h->K * 2, partials, (size_t)nranks * M * h->K * 4)) return QMLP_ERR_ALIAS;
    if (fault("launch")) return QMLP_ERR_CUDA;
    return launch_shard_combine(h->fmt, partials, nranks, M, h->K, h->gv[2].inv_g, h->gv[2].chs,
                                out, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QMLP_OK
               : QMLP_ERR_CUDA;
}

int qmlp_shard_info(qmlp_t* h, int* rank, int* nranks, int* I_shard) {
    if (!h) return 0;
    if (rank) *rank = h->rank;
    if (nranks) *nranks = h->nranks;
    if (I_shard) *I_shard = h->I;
    return 1;
}

// ---------------------------------------------------------------------------
// routed-expert AWQ
// ---------------------------------------------------------------------------
qmlp_status qmlp_moe_create(qmlp_moe_t** out, const qmlp_moe_desc* d, qmlp_stream_t stream) {
    if (!out) return QMLP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!d || !d->w13 || !d->w13_meta || !d->w2 || !d->w2_meta) return QMLP_ERR_INVALID_ARG;
    if (d->meta != QMLP_META_3B && d->meta != QMLP_META_4B) return QMLP_ERR_INVALID_ARG;
    if (d->E < 1 || d->K < 64 || d->K > 16384 || d->K % 64 || d->I < 32 || d->I > 1024 || d->I % 32)
        return QMLP_ERR_SHAPE;
    int dev = 0, sms = 0;
    qmlp_status st = check_device(&dev, &sms);
    if (st != QMLP_OK) return st;
    qmlp_moe_t* h = new qmlp_moe_t();
    h->E = d->E;
    h->K = d->K;
    h->I = d->I;
    h->meta = d->meta;
    h->device = dev;
    h->num_sms = sms;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t mb = (size_t)d->meta;
    const size_t w13b = (size_t)d->E * 2 * d->I * (d->K / 2), m13b = (size_t)d->E * 2 * d->I * (d->K / 32) * mb;
    const size_t w2b = (size_t)d->E * d->K * (d->I / 2), m2b = (size_t)d->E * d->K * (d->I / 32) * mb;
    void *t0 = nullptr, *t1 = nullptr, *p = nullptr;
    cudaError_t e = cudaSuccess;
    // W13: the warp-block bank of the K-split W13 kernels; W2: lane-sliced codes
    auto stage = [&](const void* src, size_t wbytes, const void* msrc, size_t mbytes, int N, int Kr,
                     uint8_t** wdst, uint8_t** mdst, bool w13) -> qmlp_status {
        if ((e = h->mem.alloc(&t0, wbytes)) != cudaSuccess) return from_cuda(e);
        if ((e = h->mem.alloc(&t1, mbytes)) != cudaSuccess) return from_cuda(e);
        if (cudaMemcpyAsync(t0, src, wbytes, cudaMemcpyDefault, s) != cudaSuccess) return QMLP_ERR_CUDA;
        if (cudaMemcpyAsync(t1, msrc, mbytes, cudaMemcpyDefault, s) != cudaSuccess) return QMLP_ERR_CUDA;
        void *wo = nullptr, *mo = nullptr;
        const size_t wob = w13 ? moe_w13_bank_bytes(d->E, d->I, d->K) : wbytes;
        const size_t mob = w13 ? moe_w13_meta_bank_bytes(d->E, d->I, d->K, d->meta) : mbytes;
        if ((e = h->mem.alloc(&wo, wob)) != cudaSuccess) return from_cuda(e);
        if ((e = h->mem.alloc(&mo, mob)) != cudaSuccess) return from_cuda(e);
        if ((w13 ? repack_moe_w13_blocks(static_cast<uint8_t*>(t0), static_cast<uint8_t*>(t1), d->meta, d->E, d->I,
                                         d->K, static_cast<uint8_t*>(wo), static_cast<uint8_t*>(mo), s)
                 : repack_moe(static_cast<uint8_t*>(t0), static_cast<uint8_t*>(t1), d->meta, d->E, N, Kr,
                              static_cast<uint8_t*>(wo), static_cast<uint8_t*>(mo), s)) != cudaSuccess)
            return QMLP_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return QMLP_ERR_CUDA;
        for (void* q : {t0, t1}) {
            auto it = std::find(h->mem.ptrs.begin(), h->mem.ptrs.end(), q);
            if (it != h->mem.ptrs.end()) {
                cudaFree(q);
                h->mem.ptrs.erase(it);
            }
        }
        *wdst = static_cast<uint8_t*>(wo);
        *mdst = static_cast<uint8_t*>(mo);
        return QMLP_OK;
    };
    st = stage(d->w13, w13b, d->w13_meta, m13b, 2 * d->I, d->K, &h->w13, &h->w13_meta, true);
    if (st == QMLP_OK) st = stage(d->w2, w2b, d->w2_meta, m2b, d->K, d->I, &h->w2, &h->w2_meta, false);
    if (st == QMLP_OK) {
        if ((e = h->mem.alloc(&p, (size_t)16 * d->I * sizeof(__half))) != cudaSuccess) st = from_cuda(e);
        else h->act_ws = static_cast<__half*>(p);
    }
    if (st == QMLP_OK) {
        if ((e = h->mem.alloc(&p, 16)) != cudaSuccess) st = from_cuda(e);
        else {
            h->err = static_cast<int*>(p);
            if (cudaMemsetAsync(p, 0, 16, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
                st = QMLP_ERR_CUDA;
        }
    }
    if (st != QMLP_OK) {
        cudaStreamSynchronize(s);
        h->mem.release();
        delete h;
        return st;
    }
    *out = h;
    return QMLP_OK;
}

void qmlp_moe_destroy(qmlp_moe_t* h) {
    if (!h) return;
    cudaDeviceSynchronize();
    h->mem.release();
    delete h;
}

static qmlp_status moe_run(qmlp_moe_t* h, const void* x, qmlp_dtype xdt, const int32_t* ids, const float* rw,
                           int topk, void* out, void* gu, void* act, void* y, qmlp_stream_t stream) {
    if (!h || !x || !ids || !rw || !out) return QMLP_ERR_INVALID_ARG;
    if (xdt != QMLP_DT_BF16 && xdt != QMLP_DT_FP16) return QMLP_ERR_INVALID_ARG;
    if (topk < 1 || topk > 16) return QMLP_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ids) || !aligned16(rw)) return QMLP_ERR_ALIGNMENT;
    if ((gu && !aligned16(gu)) || (act && !aligned16(act)) || (y && !aligned16(y))) return QMLP_ERR_ALIGNMENT;
    const size_t ob = (size_t)h->K * 2;
    if (overlaps(out, ob, x, (size_t)h->K * 2) || overlaps(out, ob, ids, (size_t)topk * 4) ||
        overlaps(out, ob, rw, (size_t)topk * 4))
        return QMLP_ERR_ALIAS;
    if (fault("launch")) return QMLP_ERR_CUDA;
    MoeLaunch L;
    L.E = h->E;
    L.K = h->K;
    L.I = h->I;
    L.meta_bytes = h->meta;
    L.sliced = 1;  // the handle's banks (repack_moe)
    L.w13 = h->w13;
    L.w13_meta = h->w13_meta;
    L.w2 = h->w2;
    L.w2_meta = h->w2_meta;
    L.x = x;
    L.x_is_bf16 = xdt == QMLP_DT_BF16;
    L.ids = ids;
    L.rw = rw;
    L.topk = topk;
    L.out = static_cast<__half*>(out);
    L.act_ws = h->act_ws;
    L.gu_dbg = static_cast<__half*>(gu);
    L.act_dbg = static_cast<__half*>(act);
    L.y_dbg = static_cast<__half*>(y);
    return launch_moe(L, h->num_sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QMLP_OK
                                                                                          : QMLP_ERR_CUDA;
}

qmlp_status qmlp_moe_m1_forward(qmlp_moe_t* h, const void* x, qmlp_dtype xdt, const int32_t* ids,
                                const float* rw, int topk, void* out, qmlp_stream_t stream) {
    return moe_run(h, x, xdt, ids, rw, topk, out, nullptr, nullptr, nullptr, stream);
}

qmlp_status qmlp_moe_debug_stages(qmlp_moe_t* h, const void* x, qmlp_dtype xdt, const int32_t* ids,
                                  const float* rw, int topk, void* out, void* gu, void* act, void* y,
                                  qmlp_stream_t stream) {
    return moe_run(h, x, xdt, ids, rw, topk, out, gu, act, y, stream);
}

qmlp_status qmlp_moe_reserve(qmlp_moe_t* h, int max_tokens, qmlp_stream_t stream) {
    if (!h) return QMLP_ERR_INVALID_ARG;
    if (max_tokens < 1 || max_tokens > (1 << 20)) return QMLP_ERR_SHAPE;
    if (max_tokens <= h->max_tokens) return QMLP_OK;
    if (h->K > kMoeGroupedMaxK || h->E > kMoeGroupedMaxE) return QMLP_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return QMLP_ERR_CUDA;
    const size_t routes = (size_t)max_tokens * 16;
    void *act = nullptr, *y = nullptr, *rl = nullptr, *gr = nullptr, *ng = nullptr;
    cudaError_t e;
    if ((e = h->mem.alloc(&act, routes * h->I * sizeof(__half))) != cudaSuccess ||
        (e = h->mem.alloc(&y, routes * h->K * sizeof(__half))) != cudaSuccess ||
        (e = h->mem.alloc(&rl, routes * sizeof(int))) != cudaSuccess ||
        (e = h->mem.alloc(&gr, moe_grouped_max_groups((int)routes, h->E) * sizeof(int4))) != cudaSuccess ||
        (e = h->mem.alloc(&ng, 16)) != cudaSuccess) {
        for (void* p : {act, y, rl, gr, ng}) {
            auto it = std::find(h->mem.ptrs.begin(), h->mem.ptrs.end(), p);
            if (p && it != h->mem.ptrs.end()) {
                cudaFree(p);
                h->mem.ptrs.erase(it);
            }
        }
        return from_cuda(e);
    }
    // the previous (smaller) workspace stays owned by the handle until destroy
    h->g_act = static_cast<__half*>(act);
    h->g_y = static_cast<__half*>(y);
    h->g_route = static_cast<int*>(rl);
    h->g_groups = static_cast<int4*>(gr);
    h->g_ngroups = static_cast<int*>(ng);
    h->max_tokens = max_tokens;
    return QMLP_OK;
}

qmlp_status qmlp_moe_forward(qmlp_moe_t* h, const void* x, qmlp_dtype xdt, const int32_t* ids, const float* rw,
                             int topk, int M, void* out, qmlp_stream_t stream) {
    if (!h || !x || !ids || !rw || !out) return QMLP_ERR_INVALID_ARG;
    if (M < 1 || M > h->max_tokens) return QMLP_ERR_SHAPE;
    if (M == 1) return moe_run(h, x, xdt, ids, rw, topk, out, nullptr, nullptr, nullptr, stream);
    if (xdt != QMLP_DT_BF16 && xdt != QMLP_DT_FP16) return QMLP_ERR_INVALID_ARG;
    if (topk < 1 || topk > 16) return QMLP_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ids) || !aligned16(rw)) return QMLP_ERR_ALIGNMENT;
    const size_t xb = (size_t)M * h->K * 2, rb = (size_t)M * topk * 4;
    if (overlaps(out, xb, x, xb) || overlaps(out, xb, ids, rb) || overlaps(out, xb, rw, rb)) return QMLP_ERR_ALIAS;
    if (fault("launch")) return QMLP_ERR_CUDA;
    MoeGroupedLaunch L;
    L.num_sms = h->num_sms;
    L.E = h->E;
    L.K = h->K;
    L.I = h->I;
    L.meta_bytes = h->meta;
    L.M = M;
    L.topk = topk;
    L.w13 = h->w13;
    L.w13_meta = h->w13_meta;
    L.w2 = h->w2;
    L.w2_meta = h->w2_meta;
    L.x = x;
    L.x_is_bf16 = xdt == QMLP_DT_BF16;
    L.ids = ids;
    L.rw = rw;
    L.out = static_cast<__half*>(out);
    L.act_ws = h->g_act;
    L.y_ws = h->g_y;
    L.route_list = h->g_route;
    L.groups = h->g_groups;
    L.n_groups = h->g_ngroups;
    return launch_moe_grouped(L, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QMLP_OK : QMLP_ERR_CUDA;
}

qmlp_status qmlp_moe_check(qmlp_moe_t* h, qmlp_stream_t stream) {
    if (!h) return QMLP_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QMLP_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QMLP_ERR_CUDA;
    if (v != 0) {
        cudaMemset(h->err, 0, sizeof(int));
        return QMLP_ERR_DEVICE_TIMEOUT;
    }
    return QMLP_OK;
}

}  // extern "C"
