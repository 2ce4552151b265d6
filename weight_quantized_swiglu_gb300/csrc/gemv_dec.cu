// gemv_dec.cu -- decode-path (M <= 16) weight-quantized GEMV kernels.
//
// Operation: one or two projections of the SwiGLU MLP (vllm.cpp issue
// "tp>1 fp8w tail-MLP shard host-dequantizes every layer", "Proposed fix"),
// y[m, n] = sum_k x[m, k] * W[n, k], with W dequantized on the fly from the
// resident packed bytes:
//   NVFP4 (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented"):
//     W = E2M1(nibble) * E4M3(scale[n, k/16]); the 1/global factor is applied
//     to the fp32 accumulator in the epilogue.
//   FP8 per-channel (same vllm.cpp issue, "Mechanism on the tp>1 path"):
//     W = e4m3fn(byte); scale[n] is applied in the epilogue.
//
// Design (GB300):
//  * HBM-bound streaming: every lane issues 16-byte coalesced loads of
//    packed weights laid out at create time in tensor-core A-fragment order
//    (one warp load = 512 contiguous bytes = a 16-row x 64-k block of NVFP4).
//  * Decode in registers with the hardware E2M1/E4M3 -> f16x2 conversions
//    (exact), the group-16 E4M3 scale applied by one f16x2 multiply (the
//    product has <= 6 significant bits, exact in fp16), then a warp-level
//    m16n8k16 tensor-core MMA with fp32 accumulation. Tokens are the n8
//    operand, so M <= 8 costs one MMA per 256 weights and M <= 16 two.
//  * Activations: each CTA stages its k-slice of x in shared memory as fp16
//    scaled by a per-token power of two 2^sigma chosen from the slice's
//    max|x| (max*2^sigma in [2^14, 2^15)); every bf16 value within 2^29 of
//    the maximum is then exact in fp16, and the accumulator is multiplied by
//    2^-sigma (exact) before it leaves the CTA.
//  * Gate and up are fused: one pass over the staged x feeds both.
//  * Split-K: 8 warps per CTA take interleaved 64-k chunks and reduce through
//    shared memory; when the row tiles alone cannot fill the GPU, the k range
//    is split across CTAs, partial sums go to a workspace and the last CTA of
//    a row tile (atomic arrival counter, reset by that CTA) adds them in a
//    fixed order. No floating-point atomics: results are run-to-run
//    deterministic.
#include <algorithm>

#include "gemv_frag.cuh"

namespace qmlp {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxStageBytes = 64 * 1024;

struct KArgs {
    int Lr, TWr, Rr;
    const uint8_t* wc0;
    const float* chs0;
    float inv0;
    const uint8_t* wc1;
    const float* chs1;
    float inv1;
    const __nv_bfloat16* x;
    int M, K, N, Nt, Kc, ksplit, cps;
    void* out;
    float* part;
    int* counters;
    size_t part_cap;  // index checks: floats of the partial buffer
};

template <int FMT, int NT, int NP, int EPI>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const KArgs a) {
    extern __shared__ __align__(16) uint8_t dyn_smem[];
    uint4* xs = reinterpret_cast<uint4*>(dyn_smem);  // [cps][2][4*M] fragment slots
    __shared__ float red[kWarps][NP][NT][32][4];
    __shared__ int s_maxbits[16];
    __shared__ int s_sig[16];
    __shared__ int s_last;

    const int tid = threadIdx.x;
    const int rt = blockIdx.x;
    const int ks = blockIdx.y;
    const int M = a.M;
    const int c0 = ks * a.cps;
    const int c1 = min(c0 + a.cps, a.Kc);
    const int nch = c1 - c0;
    const int kb = c0 * kChunkK;
    const int ke = min(c1 * kChunkK, a.K);
    const int kpe = c1 * kChunkK;
    const int slots = 4 * M;
    (void)tid;

    stage_x(a.x, M, a.K, kb, ke, kpe, xs, s_maxbits, s_sig);

    // ---- stream weights, decode, MMA ----------------------------------------
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    float acc[NP][NT][4];
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[p][n][i] = 0.0f;

    const size_t tile0 = (size_t)rt * a.Kc + c0;
    ChunkW cur[NP], nxt[NP];
    // every logical record (row tile, k-chunk) this CTA reads exists
    if (!QMLP_INB(tile0 + (nch > 0 ? nch - 1 : 0), (size_t)a.Nt * a.Kc, 25)) return;
    if (warp < nch) {
        cur[0] = load_chunk<FMT>(a.wc0, tile0 + warp, a.Lr, a.TWr, a.Rr, lane);
        if (NP == 2) cur[NP - 1] = load_chunk<FMT>(a.wc1, tile0 + warp, a.Lr, a.TWr, a.Rr, lane);
    }
    for (int cc = warp; cc < nch; cc += kWarps) {
        const bool more = cc + kWarps < nch;
        if (more) {
            nxt[0] = load_chunk<FMT>(a.wc0, tile0 + cc + kWarps, a.Lr, a.TWr, a.Rr, lane);
            if (NP == 2) nxt[NP - 1] = load_chunk<FMT>(a.wc1, tile0 + cc + kWarps, a.Lr, a.TWr, a.Rr, lane);
        }
        uint4 xb[NT][2];
        load_xfrag<NT>(xs, cc, M, slots, g, t, xb);
        mma_chunk<FMT, NT, NP>(cur, xb, acc);
        if (more) {
#pragma unroll
            for (int p = 0; p < NP; ++p) cur[p] = nxt[p];
        }
    }

    // ---- reduce the 8 warps (fixed order) ----------------------------------
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][p][n][lane][i] = acc[p][n][i];
    __syncthreads();

    // value of (projection p, tile row r, token m) in this CTA
    auto cta_value = [&](int p, int r, int m) -> float {
        const int n = m >> 3, mm = m & 7;
        const int ln = (r & 7) * 4 + (mm >> 1);
        const int reg = (r >= 8 ? 2 : 0) + (mm & 1);
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += red[w][p][n][ln][reg];
        return scalbnf(v, -s_sig[m]);
    };

    const int items = kTileRows * M;
    if (a.ksplit > 1) {
        for (int it = tid; it < items; it += kThreads) {
            const int m = it / kTileRows, r = it - m * kTileRows;
            const int row = rt * kTileRows + r;
#pragma unroll
            for (int p = 0; p < NP; ++p)
                if (QMLP_INB(((size_t)(ks * NP + p) * M + m) * a.N + row, a.part_cap, 26))
                    a.part[((size_t)(ks * NP + p) * M + m) * a.N + row] = cta_value(p, r, m);
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = (atomicAdd(&a.counters[rt], 1) == a.ksplit - 1);
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        if (tid == 0) a.counters[rt] = 0;
    }

    for (int it = tid; it < items; it += kThreads) {
        const int m = it / kTileRows, r = it - m * kTileRows;
        const int row = rt * kTileRows + r;
        if (!QMLP_INB(row, a.N, 27)) continue;
        float v[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            if (a.ksplit > 1) {
                float s = 0.0f;
                for (int q = 0; q < a.ksplit; ++q)
                    if (QMLP_INB(((size_t)(q * NP + p) * M + m) * a.N + row, a.part_cap, 26))
                        s += __ldcg(&a.part[((size_t)(q * NP + p) * M + m) * a.N + row]);
                v[p] = s;
            } else {
                v[p] = cta_value(p, r, m);
            }
        }
        if (EPI == kEpiRaw) {
            reinterpret_cast<float*>(a.out)[(size_t)m * a.N + row] = v[0];
        } else {
            const float sg = FMT == kNVFP4 ? a.inv0 : a.chs0[row];
            const float y0 = v[0] * sg;
            float res = y0;
            if (EPI == kEpiSwiGLU) {
                const float su = FMT == kNVFP4 ? a.inv1 : a.chs1[row];
                res = silu_f32(y0) * (v[NP - 1] * su);
            }
            reinterpret_cast<__nv_bfloat16*>(a.out)[(size_t)m * a.N + row] = __float2bfloat16_rn(res);
        }
    }
}

// ---------------------------------------------------------------------------
// Create-time repack into the fragment layout
// ---------------------------------------------------------------------------
// Record position of (row tile rt, chunk c): the row-tile-major stream
// layout (split = false) or the CTA-sliced layout of the I-partitioned MLP.
struct RecPos {
    int Lr, TWr, Rr;        // stream layout
    bool split;
    int Cb, LB;             // CTA-sliced layout (TWr = 16G, Rr = 4)
    __device__ size_t operator()(int rt, int c, int Kc) const {
        if (!split) return gemv_rec_pos((size_t)rt * Kc + c, Lr, TWr, Rr);
        const int b = c / Cb;
        const long u = (long)rt * Cb + c % Cb;
        const int w = (int)(u / LB), k = (int)(u % LB);
        return ((size_t)(k / Rr) * TWr + (size_t)b * 16 + w) * Rr + k % Rr;
    }
};

__global__ void repack_nvfp4_gemv_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ s,
                                         int N, int K, RecPos pos, uint8_t* __restrict__ wc) {
    const int Nt = N / kTileRows, Kc = (K + kChunkK - 1) / kChunkK, G = K / 16, rb = K / 2;
    const size_t total = (size_t)Nt * Kc * 32;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int lane = (int)(idx % 32);
        const size_t tc = idx / 32;
        const int c = (int)(tc % Kc), rt = (int)(tc / Kc);
        const int g = lane >> 2, t = lane & 3;
        const size_t r0 = (size_t)(rt * kTileRows + g), r8 = r0 + 8;
        uint8_t* rec = wc + pos(rt, c, Kc) * kRecNVFP4;
        uint32_t words[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gi = 4 * c + j;
            uint32_t v = 0;
            if (gi < G) {
                v = (uint32_t)w[r0 * rb + 8 * gi + t] | ((uint32_t)w[r8 * rb + 8 * gi + t] << 8) |
                    ((uint32_t)w[r0 * rb + 8 * gi + 4 + t] << 16) |
                    ((uint32_t)w[r8 * rb + 8 * gi + 4 + t] << 24);
            }
            words[j] = v;
        }
        reinterpret_cast<uint4*>(rec)[lane] = make_uint4(words[0], words[1], words[2], words[3]);
        if (t == 0) {
            uint32_t sv[2] = {0, 0};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gi = 4 * c + j;
                if (gi < G) {
                    const uint32_t pair = (uint32_t)s[r0 * G + gi] | ((uint32_t)s[r8 * G + gi] << 8);
                    sv[j >> 1] |= pair << (16 * (j & 1));
                }
            }
            reinterpret_cast<uint2*>(rec + 512)[g] = make_uint2(sv[0], sv[1]);
        }
    }
}

__global__ void repack_fp8_gemv_kernel(const uint8_t* __restrict__ w, int N, int K, RecPos pos,
                                       uint8_t* __restrict__ wc) {
    const int Nt = N / kTileRows, Kc = (K + kChunkK - 1) / kChunkK;
    const size_t total = (size_t)Nt * Kc * 2 * 32;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int lane = (int)(idx % 32);
        const size_t rest = idx / 32;
        const int h = (int)(rest % 2);
        const size_t tc = rest / 2;
        const int c = (int)(tc % Kc), rt = (int)(tc / Kc);
        const int g = lane >> 2, t = lane & 3;
        const size_t r0 = (size_t)(rt * kTileRows + g), r8 = r0 + 8;
        auto B = [&](size_t row, int k) -> uint32_t { return k < K ? (uint32_t)w[row * K + k] : 0u; };
        uint32_t words[4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int k = 16 * (4 * c + 2 * h + jj) + 2 * t;
            words[jj * 2 + 0] = B(r0, k) | (B(r0, k + 1) << 8) | (B(r8, k) << 16) | (B(r8, k + 1) << 24);
            words[jj * 2 + 1] =
                B(r0, k + 8) | (B(r0, k + 9) << 8) | (B(r8, k + 8) << 16) | (B(r8, k + 9) << 24);
        }
        reinterpret_cast<uint4*>(wc + pos(rt, c, Kc) * kRecFP8 + h * 512)[lane] =
            make_uint4(words[0], words[1], words[2], words[3]);
    }
}

struct Plan {
    int ksplit, cps, nt;
    size_t smem;
};

Plan plan_gemv(int Nt, int Kc, int M, int num_sms) {
    Plan p;
    p.nt = M <= 8 ? 1 : 2;
    const int target = 8 * std::max(num_sms, 1);
    int ks = std::max(1, (target + Nt - 1) / Nt);
    const int cap = std::max(1, kMaxStageBytes / (128 * M));
    ks = std::max(ks, (Kc + cap - 1) / cap);
    ks = std::min(ks, Kc);
    p.cps = (Kc + ks - 1) / ks;
    p.ksplit = (Kc + p.cps - 1) / p.cps;
    p.smem = (size_t)p.cps * 128 * M;
    return p;
}

template <int FMT, int NT, int NP, int EPI>
cudaError_t launch_one(const KArgs& a, dim3 grid, size_t smem, cudaStream_t s) {
    auto kern = gemv_kernel<FMT, NT, NP, EPI>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxStageBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaPeekAtLastError();
}

template <int FMT>
cudaError_t dispatch(const KArgs& a, int nt, int epi, dim3 grid, size_t smem, cudaStream_t s) {
    if (epi == kEpiSwiGLU) {
        return nt == 1 ? launch_one<FMT, 1, 2, kEpiSwiGLU>(a, grid, smem, s)
                       : launch_one<FMT, 2, 2, kEpiSwiGLU>(a, grid, smem, s);
    } else if (epi == kEpiPlain) {
        return nt == 1 ? launch_one<FMT, 1, 1, kEpiPlain>(a, grid, smem, s)
                       : launch_one<FMT, 2, 1, kEpiPlain>(a, grid, smem, s);
    }
    return nt == 1 ? launch_one<FMT, 1, 1, kEpiRaw>(a, grid, smem, s)
                   : launch_one<FMT, 2, 1, kEpiRaw>(a, grid, smem, s);
}

}  // namespace

size_t gemv_codes_bytes(int fmt, int N, int K, int Lr, int TWr) {
    (void)N;
    (void)K;
    return (size_t)Lr * TWr * (fmt == kNVFP4 ? kRecNVFP4 : kRecFP8);
}

size_t gemv_part_elems(int K, int I, int num_sms) {
    size_t best = 0;
    for (int M = 1; M <= 16; ++M) {
        const Plan gu = plan_gemv(I / kTileRows, (K + kChunkK - 1) / kChunkK, M, num_sms);
        const Plan dn = plan_gemv(K / kTileRows, (I + kChunkK - 1) / kChunkK, M, num_sms);
        const Plan dg = plan_gemv(I / kTileRows, (K + kChunkK - 1) / kChunkK, M, num_sms);
        if (gu.ksplit > 1) best = std::max(best, (size_t)gu.ksplit * 2 * M * I);
        if (dg.ksplit > 1) best = std::max(best, (size_t)dg.ksplit * M * I);
        if (dn.ksplit > 1) best = std::max(best, (size_t)dn.ksplit * M * K);
    }
    return best;
}

cudaError_t launch_gemv(const GemvLaunch& L, int num_sms, cudaStream_t s) {
    if (L.M < 1 || L.M > 16) return cudaErrorInvalidValue;
    const GemvProj& P = L.p0;
    const Plan pl = plan_gemv(P.Nt, P.Kc, L.M, num_sms);
    const int NP = L.epi == kEpiSwiGLU ? 2 : 1;
    if (pl.ksplit > 1 && (size_t)pl.ksplit * NP * L.M * P.N > L.part_cap) return cudaErrorInvalidValue;
    KArgs a;
    a.Lr = P.Lr;
    a.TWr = P.TWr;
    a.Rr = P.Rr;
    a.wc0 = P.wc;
    a.chs0 = P.chs;
    a.inv0 = P.inv_g;
    a.wc1 = L.p1.wc;
    a.chs1 = L.p1.chs;
    a.inv1 = L.p1.inv_g;
    a.x = reinterpret_cast<const __nv_bfloat16*>(L.x);
    a.M = L.M;
    a.K = P.K;
    a.N = P.N;
    a.Nt = P.Nt;
    a.Kc = P.Kc;
    a.ksplit = pl.ksplit;
    a.cps = pl.cps;
    a.out = L.out;
    a.part = L.part;
    a.part_cap = L.part_cap;
    a.counters = L.counters;
    const dim3 grid(P.Nt, pl.ksplit);
    return L.fmt == kNVFP4 ? dispatch<kNVFP4>(a, pl.nt, L.epi, grid, pl.smem, s)
                           : dispatch<kFP8>(a, pl.nt, L.epi, grid, pl.smem, s);
}

cudaError_t repack_nvfp4_gemv(const uint8_t* w, const uint8_t* scale, int N, int K, int Lr, int TWr, int Rr,
                              uint8_t* wc, cudaStream_t s) {
    repack_nvfp4_gemv_kernel<<<1024, 256, 0, s>>>(w, scale, N, K, RecPos{Lr, TWr, Rr, false, 0, 0}, wc);
    return cudaPeekAtLastError();
}

cudaError_t repack_fp8_gemv(const uint8_t* w, int N, int K, int Lr, int TWr, int Rr, uint8_t* wc, cudaStream_t s) {
    repack_fp8_gemv_kernel<<<1024, 256, 0, s>>>(w, N, K, RecPos{Lr, TWr, Rr, false, 0, 0}, wc);
    return cudaPeekAtLastError();
}

// The CTA-sliced down layout of the I-partitioned MLP (see SplitPlan); the
// padding records past Nt*Cb of each CTA must be zeroed by the caller.
cudaError_t repack_nvfp4_split(const uint8_t* w, const uint8_t* scale, int N, int K, const SplitPlan& P,
                               uint8_t* wc, cudaStream_t s) {
    if (!P.G || (K / kChunkK) != P.G * P.Cb || K % kChunkK) return cudaErrorInvalidValue;
    repack_nvfp4_gemv_kernel<<<1024, 256, 0, s>>>(w, scale, N, K,
                                                  RecPos{P.LB, P.G * 16, P.RB, true, P.Cb, P.LB}, wc);
    return cudaPeekAtLastError();
}

cudaError_t repack_fp8_split(const uint8_t* w, int N, int K, const SplitPlan& P, uint8_t* wc, cudaStream_t s) {
    if (!P.G || (K / kChunkK) != P.G * P.Cb || K % kChunkK) return cudaErrorInvalidValue;
    repack_fp8_gemv_kernel<<<1024, 256, 0, s>>>(w, N, K,
                                                RecPos{P.LB, P.G * 16, P.RB, true, P.Cb, P.LB}, wc);
    return cudaPeekAtLastError();
}

QMLP_BOUNDS_UNIT(gemv_dec)

}  // namespace qmlp
