// moe_awq.cu -- routed-expert AWQ int4 group-32 MLP for one token (M = 1).
//
// Operation (1Cat-vLLM PR "[Kernel][SM70] Add native-g32 AWQ QPN M1
// operator", "What it does"):
//   W13 stage: routes in router order; for a valid id, h = x . W13[id]^T in
//     fp32, gate/up materialized as fp16 (g = h[:I], u = h[I:]), and the
//     SwiGLU fused into an fp16 intermediate act[r] = fp16(SiLU(g) * u).
//   W2 stage: per route y[r] = fp16(act[r] . W2[id]^T) in fp32, then the
//     ordered fp32 router-weighted sum over routes into the fp16 output.
//     No fp16 atomics: one thread owns each output element and adds the
//     routes in router order.
//   Weights: half_fma(q, scale, bias) of the u4 code q (converted to half
//   exactly), with bias the stored fp16 (4-byte record) or half(-zero*scale)
//   (3-byte record); this is not half((q - zero) * scale).
//   Invalid ids (< 0 or >= E) contribute zero; duplicate ids are separate
//   routes with their own router weights.
//
// GB300 shape of the work: 10 routes x (320 x 2560 + 2560 x 160) weights,
// about 6 MB per call, so the step is latency-bound rather than bandwidth-
// bound. W13 runs one CTA per (route, 8 intermediate columns) with a warp
// per column computing gate and up together (so SiLU(g)*u is formed in the
// warp), W2 one CTA per 16 output rows looping over the routes. Each lane
// streams 8 consecutive k (4 code bytes) per step with coalesced warp
// accesses; products are exact in fp32 (fp16 weight x fp16/bf16 x) and
// every reduction has a fixed order.
#include "common.cuh"
#include "internal.h"

namespace qmlp {
namespace {

constexpr int kW13Cols = 8;           // intermediate columns per W13 CTA (one warp each)
constexpr int kW2Rows = 16;           // output rows per W2 CTA
constexpr int kW2Threads = 256;

// Decode the 8 weights of code word `w` (nibble i = k offset i, low nibble
// first) of one group record into fp32.
template <int MB>
QMLP_DEV void awq_decode8(uint32_t w, const uint8_t* rec, float (&out)[8]) {
    const __half s = __ushort_as_half((unsigned short)(rec[0] | (rec[1] << 8)));
    __half b;
    if (MB == 4) {
        b = __ushort_as_half((unsigned short)(rec[2] | (rec[3] << 8)));
    } else {
        // half(-zero * scale): the product of a 4-bit integer and an fp16 is
        // exact in fp32, so one rounding to fp16 matches half arithmetic.
        b = __float2half_rn(-(float)rec[2] * __half2float(s));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __half q = __ushort2half_rn((unsigned short)((w >> (4 * i)) & 0xF));
        out[i] = __half2float(__hfma(q, s, b));
    }
}

struct Args {
    int E, K, I;
    const uint8_t* w13;
    const uint8_t* w13_meta;
    const uint8_t* w2;
    const uint8_t* w2_meta;
    const void* x;
    int x_is_bf16;
    const int32_t* ids;
    const float* rw;
    int topk;
    __half* out;
    __half* act_ws;
    __half* gu_dbg;
    __half* act_dbg;
    __half* y_dbg;
};

QMLP_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Dot product of the staged fp32 vector xs[0:Kr) with row `row` of expert e
// of a [E, N, Kr] bank, reduced over the warp (every lane gets the sum).
template <int MB>
QMLP_DEV float awq_row_dot(const uint8_t* __restrict__ w, const uint8_t* __restrict__ meta, int N, int Kr,
                           int e, int row, const float* xs, int lane) {
    const size_t rbase = (size_t)e * N + row;
    const uint8_t* wr = w + rbase * (Kr / 2);
    const uint8_t* mr = meta + rbase * (Kr / 32) * MB;
    float acc = 0.0f;
    for (int k0 = lane * 8; k0 < Kr; k0 += 256) {
        const uint32_t code = __ldg(reinterpret_cast<const uint32_t*>(wr + k0 / 2));
        float wv[8];
        awq_decode8<MB>(code, mr + (size_t)(k0 / 32) * MB, wv);
        const float4 xa = *reinterpret_cast<const float4*>(xs + k0);
        const float4 xb = *reinterpret_cast<const float4*>(xs + k0 + 4);
        acc = fmaf(xa.x, wv[0], acc);
        acc = fmaf(xa.y, wv[1], acc);
        acc = fmaf(xa.z, wv[2], acc);
        acc = fmaf(xa.w, wv[3], acc);
        acc = fmaf(xb.x, wv[4], acc);
        acc = fmaf(xb.y, wv[5], acc);
        acc = fmaf(xb.z, wv[6], acc);
        acc = fmaf(xb.w, wv[7], acc);
    }
    return warp_sum(acc);
}

template <int MB>
__global__ void __launch_bounds__(kW13Cols * 32) moe_w13_kernel(const Args a) {
    extern __shared__ __align__(16) float xs[];  // [K]
    const int r = blockIdx.y;
    const int id = a.ids[r];
    if (id < 0 || id >= a.E) return;
    for (int k = threadIdx.x; k < a.K; k += blockDim.x) {
        const unsigned short b = reinterpret_cast<const unsigned short*>(a.x)[k];
        xs[k] = a.x_is_bf16 ? __bfloat162float(__ushort_as_bfloat16(b)) : __half2float(__ushort_as_half(b));
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = blockIdx.x * kW13Cols + warp;
    if (q >= a.I) return;
    const int N13 = 2 * a.I;
    const float hg = awq_row_dot<MB>(a.w13, a.w13_meta, N13, a.K, id, q, xs, lane);
    const float hu = awq_row_dot<MB>(a.w13, a.w13_meta, N13, a.K, id, a.I + q, xs, lane);
    if (lane == 0) {
        const __half g = __float2half_rn(hg), u = __float2half_rn(hu);
        const __half act = __float2half_rn(silu_f32(__half2float(g)) * __half2float(u));
        a.act_ws[(size_t)r * a.I + q] = act;
        if (a.gu_dbg) {
            a.gu_dbg[(size_t)r * N13 + q] = g;
            a.gu_dbg[(size_t)r * N13 + a.I + q] = u;
        }
        if (a.act_dbg) a.act_dbg[(size_t)r * a.I + q] = act;
    }
}

template <int MB>
__global__ void __launch_bounds__(kW2Threads) moe_w2_kernel(const Args a) {
    extern __shared__ __align__(16) float acts[];  // [topk][I]
    __shared__ float ys[16][kW2Rows];
    __shared__ int s_ids[16];
    const int tid = threadIdx.x;
    if (tid < a.topk) s_ids[tid] = a.ids[tid];
    __syncthreads();
    for (int i = tid; i < a.topk * a.I; i += blockDim.x) {
        const int r = i / a.I;
        const int id = s_ids[r];
        acts[i] = (id >= 0 && id < a.E) ? __half2float(a.act_ws[i]) : 0.0f;
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int n0 = blockIdx.x * kW2Rows;
    for (int item = warp; item < a.topk * kW2Rows; item += nw) {
        const int r = item / kW2Rows, j = item - r * kW2Rows;
        const int id = s_ids[r];
        const int n = n0 + j;
        if (id < 0 || id >= a.E || n >= a.K) continue;
        const float v = awq_row_dot<MB>(a.w2, a.w2_meta, a.K, a.I, id, n, acts + (size_t)r * a.I, lane);
        if (lane == 0) {
            const __half y = __float2half_rn(v);
            ys[r][j] = __half2float(y);
            if (a.y_dbg) a.y_dbg[(size_t)r * a.K + n] = y;
        }
    }
    __syncthreads();
    if (tid < kW2Rows && n0 + tid < a.K) {
        float s = 0.0f;
        for (int r = 0; r < a.topk; ++r) {
            const int id = s_ids[r];
            if (id >= 0 && id < a.E) s = fmaf(a.rw[r], ys[r][tid], s);
        }
        a.out[n0 + tid] = __float2half_rn(s);
    }
}

template <int MB>
cudaError_t launch_mb(const Args& a, cudaStream_t s) {
    const size_t smem13 = (size_t)a.K * sizeof(float);
    const size_t smem2 = (size_t)a.topk * a.I * sizeof(float);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(moe_w13_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             16384 * (int)sizeof(float));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(moe_w2_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 16 * 1024 * (int)sizeof(float));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const dim3 g13((a.I + kW13Cols - 1) / kW13Cols, a.topk);
    moe_w13_kernel<MB><<<g13, kW13Cols * 32, smem13, s>>>(a);
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    const dim3 g2((a.K + kW2Rows - 1) / kW2Rows);
    moe_w2_kernel<MB><<<g2, kW2Threads, smem2, s>>>(a);
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t launch_moe(const MoeLaunch& L, int num_sms, cudaStream_t s) {
    (void)num_sms;
    Args a;
    a.E = L.E;
    a.K = L.K;
    a.I = L.I;
    a.w13 = L.w13;
    a.w13_meta = L.w13_meta;
    a.w2 = L.w2;
    a.w2_meta = L.w2_meta;
    a.x = L.x;
    a.x_is_bf16 = L.x_is_bf16;
    a.ids = L.ids;
    a.rw = L.rw;
    a.topk = L.topk;
    a.out = L.out;
    a.act_ws = L.act_ws;
    a.gu_dbg = L.gu_dbg;
    a.act_dbg = L.act_dbg;
    a.y_dbg = L.y_dbg;
    return L.meta_bytes == 4 ? launch_mb<4>(a, s) : launch_mb<3>(a, s);
}

// The banks are consumed in the checkpoint layout ([E, N, Kr/2] codes,
// [E, N, Kr/32] records): a device copy.
cudaError_t repack_moe(const uint8_t* w, const uint8_t* meta, int meta_bytes, int E, int N, int Kr,
                       uint8_t* w_out, uint8_t* meta_out, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(w_out, w, (size_t)E * N * (Kr / 2), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return e;
    return cudaMemcpyAsync(meta_out, meta, (size_t)E * N * (Kr / 32) * meta_bytes, cudaMemcpyDeviceToDevice, s);
}

}  // namespace qmlp
