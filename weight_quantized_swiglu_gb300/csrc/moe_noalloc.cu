// moe_noalloc.cu -- routed-expert M=1 forward that allocates nothing.
//
// Some callers cannot call cudaMalloc at the point where they run this step:
// an allocator-owning runtime that forbids foreign device allocations, code
// that must not touch the allocator between warm-up and steady state, or a
// context where every device byte is budgeted up front. For them this entry
// point takes the caller's expert banks as they are (device pointers in the
// checkpoint layout, which the routed-expert kernels read directly) and keeps
// its only scratch -- the fp16 SwiGLU intermediate of the routes -- in a
// file-scope device array instead of a handle's workspace.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "qmlp.h"

namespace {

// Scratch limits: up to 16 routes x 1024 intermediate columns of fp16
// (32 KiB). Every GPU that loads the library holds this array until exit.
constexpr int kNoAllocMaxTopk = 16;
constexpr int kNoAllocMaxI = 1024;
static __device__ __align__(256) __half g_moe_act_scratch[kNoAllocMaxTopk * kNoAllocMaxI];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code cannot use the symbol itself as an address). The
// cached address is never refreshed: a device reset (or a primary-context
// teardown) while the library stays loaded is not supported for this entry
// point.
cudaError_t scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_moe_act_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

extern "C" qmlp_status qmlp_moe_m1_forward_noalloc(const qmlp_moe_desc* banks, const void* x, qmlp_dtype xdt,
                                                   const int32_t* expert_ids, const float* router_w, int topk,
                                                   void* out, qmlp_stream_t stream) {
    if (!banks || !banks->w13 || !banks->w13_meta || !banks->w2 || !banks->w2_meta) return QMLP_ERR_INVALID_ARG;
    if (!x || !expert_ids || !router_w || !out) return QMLP_ERR_INVALID_ARG;
    if (banks->meta != QMLP_META_3B && banks->meta != QMLP_META_4B) return QMLP_ERR_INVALID_ARG;
    if (xdt != QMLP_DT_BF16 && xdt != QMLP_DT_FP16) return QMLP_ERR_INVALID_ARG;
    if (banks->E < 1 || banks->K < 64 || banks->K > 16384 || banks->K % 64 || banks->I < 32 || banks->I % 32)
        return QMLP_ERR_SHAPE;
    // sizes beyond the scratch array are rejected, never truncated
    if (banks->I > kNoAllocMaxI || topk < 1 || topk > kNoAllocMaxTopk) return QMLP_ERR_SHAPE;
    if (!aligned16(banks->w13) || !aligned16(banks->w2) || !aligned16(x) || !aligned16(out) ||
        !aligned16(expert_ids) || !aligned16(router_w))
        return QMLP_ERR_ALIGNMENT;
    // out is written while other CTAs still read the inputs and the caller's
    // banks (read in place, never copied): it may overlap none of them
    const size_t ob = (size_t)banks->K * 2, mb = (size_t)banks->meta;
    const size_t E = (size_t)banks->E, K = (size_t)banks->K, I = (size_t)banks->I;
    if (overlaps(out, ob, x, (size_t)banks->K * 2) || overlaps(out, ob, expert_ids, (size_t)topk * 4) ||
        overlaps(out, ob, router_w, (size_t)topk * 4) || overlaps(out, ob, banks->w13, E * 2 * I * (K / 2)) ||
        overlaps(out, ob, banks->w13_meta, E * 2 * I * (K / 32) * mb) ||
        overlaps(out, ob, banks->w2, E * K * (I / 2)) || overlaps(out, ob, banks->w2_meta, E * K * (I / 32) * mb))
        return QMLP_ERR_ALIAS;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return QMLP_ERR_CUDA;
    if (major != 10 || minor != 3) return QMLP_ERR_UNSUPPORTED_ARCH;
    void* scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) return QMLP_ERR_CUDA;

    qmlp::MoeLaunch L;
    L.E = banks->E;
    L.K = banks->K;
    L.I = banks->I;
    L.meta_bytes = banks->meta;
    L.w13 = banks->w13;
    L.w13_meta = banks->w13_meta;
    L.w2 = banks->w2;
    L.w2_meta = banks->w2_meta;
    L.x = x;
    L.x_is_bf16 = xdt == QMLP_DT_BF16;
    L.ids = expert_ids;
    L.rw = router_w;
    L.topk = topk;
    L.out = static_cast<__half*>(out);
    L.act_ws = static_cast<__half*>(scratch);  // every valid route's row is written before it is read
    L.gu_dbg = nullptr;
    L.act_dbg = nullptr;
    L.y_dbg = nullptr;
    return qmlp::launch_moe(L, 0, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QMLP_OK
                                                                                         : QMLP_ERR_CUDA;
}
