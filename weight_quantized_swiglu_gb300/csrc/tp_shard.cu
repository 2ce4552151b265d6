// tp_shard.cu -- the exchange step of the tensor-parallel shard.
//
// vllm.cpp issue "tp>1 fp8w tail-MLP shard host-dequantizes every layer",
// "Proposed fix": with gate/up row-sliced and down column-sliced over the
// intermediate dimension, each rank's down projection is a partial sum over
// its slice of act, and one sum over the ranks gives the hidden output. Each
// rank hands over its fp32 partial without the down factor; once they are
// gathered ([nranks][M][K], rank-major), this kernel adds them in rank order
// -- a fixed order, so every rank that runs it gets the same bytes -- applies
// the down factor once and rounds to bf16, as the single-GPU path does.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace qmlp {
namespace {

constexpr int kCombineThreads = 256;

// Four outputs per thread (16-byte loads of every rank's partial).
__global__ void __launch_bounds__(kCombineThreads) shard_combine_kernel(const float* __restrict__ part,
                                                                        int nranks, int M, int K, int fp8,
                                                                        float invd, const float* __restrict__ chsd,
                                                                        __nv_bfloat16* __restrict__ out) {
    const size_t plane = (size_t)M * K;
    const size_t n4 = plane / 4;
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += (size_t)gridDim.x * blockDim.x) {
        float4 acc = __ldg(reinterpret_cast<const float4*>(part) + q);
        for (int r = 1; r < nranks; ++r) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(part + (size_t)r * plane) + q);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const int o = (int)((q * 4) % (size_t)K);  // K % 16 == 0: the four outputs share a row
        if (!QMLP_INB(o + 3, K, 51)) continue;
        const float4 f = fp8 ? __ldg(reinterpret_cast<const float4*>(chsd + o)) : make_float4(invd, invd, invd, invd);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * f.x, acc.y * f.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * f.z, acc.w * f.w);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&lo);
        w.y = *reinterpret_cast<const uint32_t*>(&hi);
        reinterpret_cast<uint2*>(out)[q] = w;
    }
}

}  // namespace

cudaError_t launch_shard_combine(int fmt, const float* partials, int nranks, int M, int K, float invd,
                                 const float* chsd, void* out, cudaStream_t s) {
    if (nranks < 1 || M < 1 || K % 16 || (fmt == kFP8 && !chsd)) return cudaErrorInvalidValue;
    const size_t n4 = (size_t)M * K / 4;
    const unsigned grid = (unsigned)std::min<size_t>((n4 + kCombineThreads - 1) / kCombineThreads, 4096);
    shard_combine_kernel<<<grid, kCombineThreads, 0, s>>>(partials, nranks, M, K, fmt == kFP8 ? 1 : 0, invd, chsd,
                                                           static_cast<__nv_bfloat16*>(out));
    return cudaPeekAtLastError();
}

QMLP_BOUNDS_UNIT(tp_shard)

}  // namespace qmlp
