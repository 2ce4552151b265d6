// gemm_tc.cu -- tensor-core prefill GEMM for NVFP4 and FP8 per-channel
// projections (M >= 17).
//
// Operation (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented" and the
// prefill tile discussion; vllm.cpp issue "tp>1 fp8w tail-MLP shard ...",
// "Proposed fix" for the fused gate/up epilogue):
//   y[m, n] = sum_k a[m, k] * W[n, k],
//   NVFP4: W[n, k] = E2M1(code) * E4M3(scale[n, k/16]), factor c[n] = 1/global
//   FP8:   W[n, k] = e4m3fn(byte),                    factor c[n] = scale[n]
// followed by one of the epilogues
//   SwiGLU: act[m, i] = bf16( SiLU(c_g[i] y_g[m, i]) * (c_u[i] y_u[m, i]) )
//   Plain:  out[m, n] = bf16( c[n] y[m, n] )
//   Raw:    y[m, n] in fp32 (no factor), debug.
//
// GB300 design (sm_103a, one CTA per SM, persistent):
//  * a (bf16 activations) is first rewritten as fp16 x 2^sigma[m] with one
//    power of two per token (sigma puts the row maximum in [2^14, 2^15)), so
//    every bf16 value within 2^29 of the row maximum is held exactly; the
//    epilogue multiplies by 2^-sigma[m]. W = E2M1 x E4M3 has at most six
//    significant bits and lies in [2^-10, 2688]; an e4m3fn value has four
//    and lies in [2^-9, 448]: both exact in fp16. The MMA is therefore an
//    fp16 x fp16 -> fp32 product of the same values the bf16 formulation
//    multiplies.
//  * Tile 128 tokens x 256 weight rows, k-step 64. Warp roles:
//      warp 0      TMA producer: the activation tile (cp.async.bulk.tensor,
//                  128-byte swizzle) and the packed weight block of the step
//                  (one cp.async.bulk: 9 KB NVFP4, 16 KB FP8) into a 5-stage
//                  load ring (TMA and L2 latency is several
//                  MMA steps long);
//      warp 1      TMEM owner and MMA issuer: 4 x tcgen05.mma (M128 N256 K16)
//                  per step into one of two TMEM accumulators (2 x 256 fp32
//                  columns), tcgen05.commit frees the load stage and the
//                  decoded stage;
//      warps 2-5   epilogue: tcgen05.ld of the finished accumulator (warp w
//                  owns TMEM lanes 32*(w%4)..+31 = 32 token rows), scales,
//                  SwiGLU, bf16 stores; overlaps the next tile's main loop;
//      warps 6-13  decoders: the stage's weight block -> fp16 weights
//                  (NVFP4: cvt.rn.f16x2.e2m1x2, then an exact f16x2 multiply
//                  by the group scale; FP8: cvt.rn.f16x2.e4m3x2) written in
//                  the 128-byte swizzled K-major layout the MMA descriptor
//                  reads, into a 3-stage (FP8: 2-stage) ring, so decoding
//                  runs ahead of the MMAs.
//  * Weight block layout (create-time repack): for n-tile j and k-step s a
//    contiguous block: NVFP4 codes [256 rows][32 B] then scales [256 rows]
//    [4 B] (9216 B); FP8 bytes [256 rows][64 B] (16384 B; the per-channel
//    scales stay a float vector read by the epilogue). For gate/up the 256
//    rows of tile j are gate rows 128j..128j+127 followed by up rows
//    128j..128j+127, so one accumulator holds both inputs of 128 SwiGLU
//    outputs per token.
//  * Dequantise-once instance (PRE; the automatic path from 768 tokens): a
//    predecode kernel first writes every weight block of the projection as
//    its bf16 stage image (the swizzled tile the decoders would have written,
//    bf16 instead of fp16: the decoded values are exact in both), once per
//    call instead of once per 128-token tile; the GEMM's load stage is then
//    the bf16 activation tile, loaded by TMA from the input itself (no
//    prescale), plus the 32 KB image (one cp.async.bulk), 4 stages deep, and
//    the MMAs are bf16 x bf16 -> fp32. Warps 6-13 have no work there.
//  * Every wait is bounded (globaltimer); on expiry the kernel records the
//    error, every role leaves its loop, in-flight copies and MMAs are waited
//    for (bounded) and TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace qmlp {
namespace {

constexpr int BM = 128;                 // tokens per tile (TMEM lanes)
constexpr int BN = 256;                 // weight rows per tile (accumulator columns)
constexpr int BK = 64;                  // k per step (one 128-byte swizzle row of fp16)
constexpr int kABytes = BM * BK * 2;    // 16 KB
constexpr int kBBytes = BN * BK * 2;    // 32 KB
constexpr int kRawCodes = BN * BK / 2;  // NVFP4: 8 KB of codes, then 1 KB of scales
// per format: weight block bytes and load-ring depth (activation tile + block)
template <int FMT>
constexpr int raw_bytes() { return FMT == kNVFP4 ? kRawCodes + BN * (BK / 16) : BN * BK; }
// Ring depths (measured at M=8192: NVFP4 3.51 -> 3.39 ms with a third decoded
// stage for a sixth load stage; FP8, whose blocks are 16 KB, keeps 5 + 2).
template <int FMT>
constexpr int lstages() { return 5; }
template <int FMT>
constexpr int bstages() { return FMT == kNVFP4 ? 3 : 2; }
constexpr int kEpiWarps = 4;
constexpr int kMaxSplits = 16;          // split-K ways at most (a split keeps >= 8 k-steps)
constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kThreads = (2 + kEpiWarps + kDecWarps) * 32;  // 448
constexpr int kTmemCols = 2 * BN;                           // two accumulators
constexpr uint64_t kGemmWaitNs = 2000000000ull;             // 2 s

// Dequantise-once instance (PRE): the weights of the call were decoded
// beforehand into their bf16 stage images, so a load stage is the activation
// tile plus a 32 KB decoded tile and there is no decoded ring.
constexpr int kPreStages = 4;

// shared memory map (offsets from a 1024-byte aligned base)
template <int FMT, bool PRE = false>
struct Smem {
    static constexpr int L = PRE ? kPreStages : lstages<FMT>();
    static constexpr int BS = PRE ? 0 : bstages<FMT>();
    static constexpr int R = PRE ? kBBytes : raw_bytes<FMT>();
    static constexpr int A = 0;
    static constexpr int B = A + L * kABytes;
    static constexpr int Raw = B + BS * kBBytes;
    static constexpr int Bar = Raw + L * R;
    // barriers: full[L], empty[L], bfull[B], bempty[B], acc_full[2], acc_empty[2], done
    static constexpr int NumBars = 2 * L + 2 * BS + 5;
    static constexpr int Misc = Bar + NumBars * 8;  // tmem address, abort flag
    static constexpr int Bytes = Misc + 16 + 1024;  // + alignment slack
    static_assert(B % 1024 == 0 && Raw % 16 == 0 && Bar % 8 == 0, "smem layout");
    static_assert(!PRE || (Raw % 1024 == 0 && R % 1024 == 0), "decoded stages sit on the swizzle period");
    static_assert(Bytes <= 227 * 1024, "smem budget");
};

struct Args {
    const uint8_t* tiles;  // weight blocks [Nt][KS][raw_bytes]
    int M, N, Kd;          // tokens, weight rows (projection outputs), contraction length
    int epi;               // kEpiSwiGLU / kEpiPlain / kEpiRaw
    int raw_sel;           // raw on an interleaved gate/up GEMM: 0 gate rows, 1 up rows
    int interleaved;       // tiles hold gate/up halves
    float inv0, inv1;      // NVFP4 global factors (gate, up) or (down, down)
    const float* cs0;      // FP8 per-channel scales: gate (interleaved) or the projection's
    const float* cs1;      // FP8 up scales (interleaved)
    const int* sig;        // [M] per-token prescale exponent
    void* out;             // bf16 [M, N_out] or fp32 [M, N_out]
    int ldo;               // out row length (elements)
    int splits;            // k-range splits per tile (1: the epilogue above; > 1: fp32 partials to ws)
    float* ws;             // [splits][M][N] fp32 partial sums (splits > 1)
    int* err;
    uint64_t limit;        // ns a wait on another role may take before the CTA aborts
    int withhold;          // error-path tests: the producer never loads its last k-step
    size_t tiles_bytes;    // index checks: bytes of the weight blocks
    size_t ws_elems;       // index checks: floats of the split-K partial buffer
    const uint8_t* wdec;   // PRE: decoded stage images [Nt][KS][32 KB]
    size_t wdec_bytes;     // PRE: bytes of wdec (index checks)
};

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N = BN, M = BM.
constexpr uint32_t kIdesc = (1u << 4)                    // D format fp32
                            | (0u << 7) | (0u << 10)     // A, B fp16
                            | ((uint32_t)(BN >> 3) << 17)  // N >> 3
                            | ((uint32_t)(BM >> 4) << 24); // M >> 4

// The same for bf16 A and B (the dequantise-once instance).
constexpr uint32_t kIdescBF16 = kIdesc | (1u << 7) | (1u << 10);

// Decode one (row, 32-k half) item of a packed block into the swizzled fp16
// B tile: 16 code bytes (32 weights, low nibble = even k) and two E4M3
// scales (k 0..15 and 16..31 of the half).
QMLP_DEV void decode_item(const uint8_t* raw, uint8_t* bt, int n, int h, int soff = kRawCodes) {
    const uint4 c = *reinterpret_cast<const uint4*>(raw + n * 32 + h * 16);
    const uint32_t s2 = *reinterpret_cast<const uint16_t*>(raw + soff + n * 4 + h * 2);
    const uint32_t sf = e4m3x2_to_f16x2(s2);
    const uint32_t sa = dup_lo16(sf), sb = dup_hi16(sf);
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    uint8_t* row = bt + n * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t f0, f1, f2, f3;
        e2m1x4_to_f16x2x4(words[j], f0, f1, f2, f3);
        const uint32_t s = j < 2 ? sa : sb;
        uint4 o;
        o.x = hmul2_u32(f0, s);
        o.y = hmul2_u32(f1, s);
        o.z = hmul2_u32(f2, s);
        o.w = hmul2_u32(f3, s);
        const int chunk = (h * 4 + j) ^ (n & 7);
        *reinterpret_cast<uint4*>(row + chunk * 16) = o;
    }
}

// FP8: one (row, 32-k half) item = 32 e4m3fn bytes -> 32 fp16 (exact).
QMLP_DEV void decode_item_fp8(const uint8_t* raw, uint8_t* bt, int n, int h) {
    const uint4 c0 = *reinterpret_cast<const uint4*>(raw + n * 64 + h * 32);
    const uint4 c1 = *reinterpret_cast<const uint4*>(raw + n * 64 + h * 32 + 16);
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint8_t* row = bt + n * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 o;
        e4m3x4_to_f16x2x2(words[2 * j], o.x, o.y);
        e4m3x4_to_f16x2x2(words[2 * j + 1], o.z, o.w);
        const int chunk = (h * 4 + j) ^ (n & 7);
        *reinterpret_cast<uint4*>(row + chunk * 16) = o;
    }
}

// The output factors of accumulator columns col..col+3: four consecutive
// per-channel scales (FP8; the same four for every thread, a broadcast
// load) or the global factor (NVFP4). col is a multiple of 4.
template <int FMT>
QMLP_DEV float4 factor4(const float* cs, float inv, int col) {
    if (FMT == kNVFP4) return make_float4(inv, inv, inv, inv);
    return __ldg(reinterpret_cast<const float4*>(cs + col));
}
QMLP_DEV float f4_at(const float4& f, int e) { return e == 0 ? f.x : e == 1 ? f.y : e == 2 ? f.z : f.w; }

QMLP_DEV uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

// The tile epilogue (no split): accumulator columns of TMEM base `tbase`
// (this thread's lane = token row m) -> SwiGLU act, plain output or raw fp32.
template <int FMT>
QMLP_DEV void store_tile(const Args& a, uint32_t tbase, int m, bool live, int sg, int nt) {
    if (a.epi == kEpiSwiGLU) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
            float g[32], u[32];
            tmem_ld32(tbase + c0, g);
            tmem_ld32(tbase + BN / 2 + c0, u);
            if (live) {
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 fg = factor4<FMT>(a.cs0, a.inv0, nt * (BN / 2) + c0 + j);
                    const float4 fu = factor4<FMT>(a.cs1, a.inv1, nt * (BN / 2) + c0 + j);
                    float r4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float gv = scalbnf(g[j + e], -sg) * f4_at(fg, e);
                        const float uv = scalbnf(u[j + e], -sg) * f4_at(fu, e);
                        r4[e] = silu_f32(gv) * uv;
                    }
                    pk[j / 2] = pack_bf16x2(r4[0], r4[1]);
                    pk[j / 2 + 1] = pack_bf16x2(r4[2], r4[3]);
                }
                uint4* dst = reinterpret_cast<uint4*>(out + (size_t)m * a.ldo + nt * (BN / 2) + c0);
                if (QMLP_INB(nt * (BN / 2) + c0 + 31, a.ldo, 12) && QMLP_INB(m, a.M, 12))
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
        }
    } else if (a.epi == kEpiPlain) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            float y[32];
            tmem_ld32(tbase + c0, y);
            if (live) {
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 f = factor4<FMT>(a.cs0, a.inv0, nt * BN + c0 + j);
                    pk[j / 2] = pack_bf16x2(scalbnf(y[j], -sg) * f.x, scalbnf(y[j + 1], -sg) * f.y);
                    pk[j / 2 + 1] = pack_bf16x2(scalbnf(y[j + 2], -sg) * f.z, scalbnf(y[j + 3], -sg) * f.w);
                }
                uint4* dst = reinterpret_cast<uint4*>(out + (size_t)m * a.ldo + nt * BN + c0);
                if (QMLP_INB(nt * BN + c0 + 31, a.ldo, 12) && QMLP_INB(m, a.M, 12))
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
        }
    } else {
        float* out = reinterpret_cast<float*>(a.out);
        const int cbeg = a.interleaved ? a.raw_sel * (BN / 2) : 0;
        const int cend = a.interleaved ? cbeg + BN / 2 : BN;
        const int ocol = a.interleaved ? nt * (BN / 2) : nt * BN;
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
            float y[32];
            tmem_ld32(tbase + c0, y);
            if (live) {
                float4* dst = reinterpret_cast<float4*>(out + (size_t)m * a.ldo + ocol + (c0 - cbeg));
                if (QMLP_INB(ocol + (c0 - cbeg) + 31, a.ldo, 12) && QMLP_INB(m, a.M, 12))
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    dst[v] = make_float4(scalbnf(y[4 * v], -sg), scalbnf(y[4 * v + 1], -sg),
                                         scalbnf(y[4 * v + 2], -sg), scalbnf(y[4 * v + 3], -sg));
            }
        }
    }
}

template <int FMT, bool SPLIT, bool PRE>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap amap, const Args a) {
    using S = Smem<FMT, PRE>;
    constexpr int kLStages = S::L;
    constexpr int kBStages = S::BS;
    constexpr int kBDiv = kBStages > 0 ? kBStages : 1;  // ring arithmetic (unused by PRE)
    constexpr int kRawBytes = S::R;
    constexpr int kOffA = S::A, kOffB = S::B, kOffRaw = S::Raw, kOffBar = S::Bar, kOffMisc = S::Misc;
    extern __shared__ uint8_t dyn_smem_raw[];
    const uint32_t base_s = (smem_u32(dyn_smem_raw) + 1023u) & ~1023u;
    uint8_t* base = dyn_smem_raw + (base_s - smem_u32(dyn_smem_raw));
    const uint32_t bar0 = base_s + kOffBar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kLStages + s); };
    auto bfull = [&](int b) { return bar0 + 8u * (2 * kLStages + b); };
    auto bempty = [&](int b) { return bar0 + 8u * (2 * kLStages + kBStages + b); };
    auto acc_full = [&](int b) { return bar0 + 8u * (2 * kLStages + 2 * kBStages + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kLStages + 2 * kBStages + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * kLStages + 2 * kBStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Mt = (a.M + BM - 1) / BM;
    const int Nt = a.N / BN;
    const int KS = a.Kd / BK;
    const int tiles = Mt * Nt;
    // (tile, k-range) work units, k-range-minor; the unsplit instance folds
    // to one unit per tile over the whole k range
    const int nsp = SPLIT ? a.splits : 1;
    const int units = tiles * nsp;
    auto ks_begin = [&](int sp) { return SPLIT ? (int)(((long)sp * KS) / nsp) : (sp == 0 ? 0 : KS); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < kBStages; ++b) {
            mbar_init(bfull(b), kDecThreads);
            mbar_init(bempty(b), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kEpiWarps * 32);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&amap)) : "memory");
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const int t = SPLIT ? u / nsp : u, sp = SPLIT ? u % nsp : 0;
                const int nt = t / Mt, mt = t % Mt;
                const uint8_t* blk = a.tiles + (size_t)nt * KS * kRawBytes;
                const int ks1 = ks_begin(sp + 1);
                // error-path tests: the CTA's very last k-step is never loaded
                const int ks_stop = (a.withhold && u + (int)gridDim.x >= units) ? ks1 - 1 : ks1;
                for (int ks = ks_begin(sp); ks < ks_stop; ++ks, ++it) {
                    const int s = it % kLStages;
                    if (it >= kLStages &&
                        !wait_or_abort(empty(s), (uint32_t)((it / kLStages - 1) & 1), abort_flag, a.err, 11, a.limit)) {
                        ok = false;
                        break;
                    }
                    const uint8_t* src;
                    if (PRE) {
                        src = a.wdec + ((size_t)nt * KS + ks) * kRawBytes;
                        if (!QMLP_INB((size_t)(src - a.wdec) + kRawBytes - 1, a.wdec_bytes, 16)) src = a.wdec;
                    } else {
                        src = blk + (size_t)ks * kRawBytes;
                        if (!QMLP_INB((size_t)(src - a.tiles) + kRawBytes - 1, a.tiles_bytes, 11)) src = a.tiles;
                    }
                    mbar_arrive_expect_tx(full(s), kABytes + kRawBytes);
                    tma_load_2d(base_s + kOffA + s * kABytes, &amap, ks * BK, mt * BM, full(s));
                    bulk_g2s(base_s + kOffRaw + s * kRawBytes, src, kRawBytes, full(s));
                }
            }
            // copies still in flight (only after an abort): wait for the last
            // one issued into each stage
            if (!ok) {
                for (int q = it - 1; q >= 0 && q >= it - kLStages; --q)
                    mbar_wait_bounded(full(q % kLStages), (uint32_t)((q / kLStages) & 1), kGemmWaitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true, issued = false;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++tc) {
                const int sp = SPLIT ? u % nsp : 0;
                const int buf = tc & 1, use = tc >> 1;
                if (use > 0 &&
                    !wait_or_abort(acc_empty(buf), (uint32_t)((use - 1) & 1), abort_flag, a.err, 12, a.limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
                const int kb = ks_begin(sp), ke = ks_begin(sp + 1);
                for (int ks = kb; ks < ke; ++ks, ++it) {
                    const int s = it % kLStages, b = it % kBDiv;
                    if (!wait_or_abort(full(s), (uint32_t)((it / kLStages) & 1), abort_flag, a.err, 13, a.limit) ||
                        (!PRE &&
                         !wait_or_abort(bfull(b), (uint32_t)((it / kBDiv) & 1), abort_flag, a.err, 14, a.limit))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base_s + kOffA + s * kABytes;
                    const uint32_t sb = PRE ? base_s + kOffRaw + s * kRawBytes : base_s + kOffB + b * kBBytes;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        umma_f16(d_tmem, smem_desc_sw128(sa + k * 32), smem_desc_sw128(sb + k * 32),
                                 PRE ? kIdescBF16 : kIdesc,
                                 (ks != kb || k != 0) ? 1u : 0u);
                    }
                    issued = true;
                    umma_commit(empty(s));
                    if (!PRE) umma_commit(bempty(b));
                }
                if (!ok) break;
                umma_commit(acc_full(buf));
            }
            // every MMA this thread issued must be finished before TMEM is freed
            if (issued) {
                umma_commit(done_bar);
                mbar_wait_bounded(done_bar, 0, kGemmWaitNs);
            }
        }
    } else if (warp < 2 + kEpiWarps) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int row_in_tile = q * 32 + lane;
        int tc = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++tc) {
            const int t = SPLIT ? u / nsp : u, sp = SPLIT ? u % nsp : 0;
            const int nt = t / Mt, mt = t % Mt;
            const int buf = tc & 1, use = tc >> 1;
            // warp-uniform: the TMEM loads below are .sync.aligned
            const bool ready = wait_or_abort(acc_full(buf), (uint32_t)(use & 1), abort_flag, a.err, 15, a.limit);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const int m = mt * BM + row_in_tile;
            const bool live = m < a.M;
            const int sg = live && a.sig ? a.sig[m] : 0;  // no prescale (null sig): bf16 operands
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
            if (SPLIT) {
                // a k-range of the tile: its fp32 partial, unscaled, in the
                // GEMM's own column order; the reduce kernel adds the splits
                // in order and applies the epilogue
                float* ws = a.ws + ((size_t)sp * a.M + m) * a.N + nt * BN;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    float y[32];
                    tmem_ld32(tbase + c0, y);
                    if (live && QMLP_INB(((size_t)sp * a.M + m) * a.N + nt * BN + c0 + 31, a.ws_elems, 13)) {
                        float4* dst = reinterpret_cast<float4*>(ws + c0);
#pragma unroll
                        for (int v = 0; v < 8; ++v) dst[v] = make_float4(y[4 * v], y[4 * v + 1], y[4 * v + 2], y[4 * v + 3]);
                    }
                }
            } else {
                store_tile<FMT>(a, tbase, m, live, sg, nt);
            }
            tc_fence_before();
            mbar_arrive(acc_empty(buf));
        }
    } else if (!PRE) {
        // ---------------- decoders ----------------
        const int d = threadIdx.x - (2 + kEpiWarps) * 32;  // 0 .. kDecThreads-1
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int sp = SPLIT ? u % nsp : 0;
            const int ks1 = ks_begin(sp + 1);
            for (int ks = ks_begin(sp); ks < ks1; ++ks, ++it) {
                const int s = it % kLStages, b = it % kBDiv;
                if (!wait_or_abort(full(s), (uint32_t)((it / kLStages) & 1), abort_flag, a.err, 16, a.limit) ||
                    (it >= kBDiv &&
                     !wait_or_abort(bempty(b), (uint32_t)((it / kBDiv - 1) & 1), abort_flag, a.err, 17, a.limit))) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = base + kOffRaw + s * kRawBytes;
                uint8_t* bt = base + kOffB + b * kBBytes;
#pragma unroll
                for (int j = 0; j < (BN * 2) / kDecThreads; ++j) {
                    const int item = d + j * kDecThreads;
                    if (FMT == kNVFP4) decode_item(raw, bt, item >> 1, item & 1);
                    else decode_item_fp8(raw, bt, item >> 1, item & 1);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(bfull(b));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair GEMM (tcgen05.mma.cta_group::2), prefill M >= 256.
//
// A cluster of two CTAs computes a 256-token x 256-row tile: CTA r (its rank
// in the cluster) holds tokens [128r, 128r + 128) of the activation tile and
// weight rows [128r, 128r + 128) of the weight tile -- it loads and decodes
// only that half of every weight block -- and its TMEM holds the 128 x 256
// accumulator of its tokens. One thread of rank 0 (the leader) issues the
// MMAs (M = 256, N = 256, K = 16: the tensor cores of both SMs read the A
// half and the B half of their own CTA, each B half serving both), and its
// commits arrive on the barriers of both CTAs (multicast). Rank 1's MMA warp
// forwards to the leader, with one remote mbarrier arrival each, that its A
// stage has landed and its B stage is decoded, and that its epilogue has
// drained an accumulator. Per SM and 64-k step this moves half the decoded
// weight tile through shared memory (decoder stores 16 KB instead of 32 KB,
// tensor-core reads 16 KB of B instead of 32 KB) and halves the decode work.
//
// Dequantise-once instance (PRE, the automatic path from 768 tokens): no
// decoders; the leader's producer thread issues, per k-step, the four TMA
// loads of both CTAs' stages -- each CTA's 128 tokens of the bf16 activation
// tile and its 128 rows of the decoded image (a tensor map over the images as
// 128-byte rows) -- into the shared memory of the CTA they belong to, all
// completing on the leader's barrier (.cta_group::2), so the leader waits on
// one barrier per stage and no stage needs a signal from the peer. Per SM and
// step 32 KB arrive instead of the 48 KB of the single-CTA instance. Copies in
// flight are tracked by the leader's barriers alone.
// ---------------------------------------------------------------------------
constexpr int kBHalf = (BN / 2) * BK * 2;  // 16 KB: 128 decoded weight rows of a 64-k step
constexpr int kDecGroups = 4;              // decoder groups of the pair kernel (one per B stage)

template <int FMT>
constexpr int raw_half() { return raw_bytes<FMT>() / 2; }  // NVFP4: 4096 codes + 512 scales; FP8: 8192

template <int FMT, bool PRE = false>
struct SmemP {
    // load stages: A (16 KB) + the weight half-block (PRE: the 16 KB half of
    // the decoded image). A stage is held from its TMA until the leader's MMA
    // has used it, which now includes the peer's signal: measured at M=8192
    // (NVFP4 / FP8), 3.90 / 3.92 ms with 5 stages, 3.72 / 3.76 with 6.
    static constexpr int L = 6;
    static constexpr int BS = PRE ? 0 : 4;  // decoded half-B stages
    static constexpr int R = PRE ? kBHalf : raw_half<FMT>();
    static constexpr int A = 0;
    static constexpr int B = A + L * kABytes;
    static constexpr int Raw = B + BS * kBHalf;
    static constexpr int Bar = Raw + L * R;
    // full[L], empty[L], bfull[BS], bempty[BS], acc_full[2], acc_empty[2], done,
    // pbfull[BS] (leader: the peer's decoders have filled B stage b -- so its
    // A stage of that step has landed too), pacc[2] (leader: the peer's
    // accumulator is drained)
    static constexpr int NumBars = 2 * L + 3 * BS + 7;
    static constexpr int Misc = Bar + NumBars * 8;
    static constexpr int Bytes = Misc + 16 + 1024;
    static_assert(B % 1024 == 0 && Raw % 16 == 0 && Bar % 8 == 0 && R % 16 == 0, "smem layout");
    static_assert(!PRE || (Raw % 1024 == 0 && R % 1024 == 0), "decoded stages sit on the swizzle period");
    static_assert(Bytes <= 227 * 1024, "smem budget");
};

// Instruction descriptor of the pair MMA: fp32 accumulator, fp16 A and B,
// K-major, N = 256, M = 256 (128 rows in each CTA); and with bf16 A and B.
constexpr uint32_t kIdescPair = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
constexpr uint32_t kIdescPairBF16 = kIdescPair | (1u << 7) | (1u << 10);

QMLP_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
QMLP_DEV void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive once on the mbarrier at the same shared-memory offset in CTA `rank`
// of the cluster.
QMLP_DEV void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(bar), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
// TMA tile load into the shared memory of CTA `rank` of the pair (same
// offset `dst` as in this CTA), completing on this CTA's barrier `bar`
// (.cta_group::2: the barrier may sit in the destination's peer).
QMLP_DEV void tma_load_2d_pair(uint32_t dst, uint32_t rank, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    uint32_t rd;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rd) : "r"(dst), "r"(rank));
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(rd),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Wait for phase `parity` of a barrier that the peer CTA arrives on
// (acquire at cluster scope); false if the abort flag is raised or the wait
// ran out (which raises it and records `code`).
QMLP_DEV bool wait_cluster_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, int code,
                                    uint64_t limit) {
    auto try_once = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        return ok != 0;
    };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!try_once()) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort_flag = 1;
            atomicExch(err, code);
            return false;
        }
    }
    return true;
}

QMLP_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
QMLP_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
QMLP_DEV void umma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` (same offset) in both CTAs of the pair once every
// tcgen05 operation this thread issued so far is complete.
QMLP_DEV void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}

template <int FMT, bool PRE>
__global__ void __launch_bounds__(kThreads, 1) gemm_pair_kernel(const __grid_constant__ CUtensorMap amap,
                                                                const __grid_constant__ CUtensorMap bmap, const Args a) {
    using S = SmemP<FMT, PRE>;
    constexpr int kL = S::L, kBS = S::BS, kR = S::R;
    constexpr int kBSd = kBS > 0 ? kBS : 1;  // ring arithmetic (unused by PRE)
    extern __shared__ uint8_t dyn_smem_raw[];
    // the same offsets in both CTAs: the MMA addresses the peer's halves, and
    // the commits and remote arrivals its barriers, at this CTA's offsets
    const uint32_t base_s = (smem_u32(dyn_smem_raw) + 1023u) & ~1023u;
    uint8_t* base = dyn_smem_raw + (base_s - smem_u32(dyn_smem_raw));
    const uint32_t bar0 = base_s + S::Bar;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kL + s); };
    auto bfull = [&](int b) { return bar0 + 8u * (2 * kL + b); };
    auto bempty = [&](int b) { return bar0 + 8u * (2 * kL + kBS + b); };
    auto acc_full = [&](int b) { return bar0 + 8u * (2 * kL + 2 * kBS + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kL + 2 * kBS + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * kL + 2 * kBS + 4);
    auto pbfull = [&](int b) { return bar0 + 8u * (2 * kL + 2 * kBS + 5 + b); };
    auto pacc = [&](int b) { return bar0 + 8u * (2 * kL + 3 * kBS + 5 + b); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + S::Misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + S::Misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: the leader, 1: its peer
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int Mt2 = (a.M + 2 * BM - 1) / (2 * BM);  // 256-token tiles
    const int Nt = a.N / BN;
    const int KS = a.Kd / BK;
    const int units = Mt2 * Nt;  // n-tile-major, as the single-CTA kernel

    if (threadIdx.x == 0) {
        for (int s = 0; s < kL; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < kBS; ++b) {
            mbar_init(bfull(b), kDecThreads / kDecGroups);
            mbar_init(bempty(b), 1);
            mbar_init(pbfull(b), kDecThreads / kDecGroups);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kEpiWarps * 32);
            mbar_init(pacc(b), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrival or multicast
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer: this CTA's A half and weight half ----------------
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&amap)) : "memory");
            if (PRE) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&bmap)) : "memory");
            int it = 0;
            bool ok = !PRE || rank == 0;  // PRE: the leader loads the stages of both CTAs
            for (int u = pair; u < units && ok; u += npairs) {
                const int nt = u / Mt2, mt2 = u % Mt2;
                const uint8_t* blk = a.tiles + (size_t)nt * KS * raw_bytes<FMT>();
                // error-path tests: the pair's very last k-step is never loaded
                const int ks_stop = (a.withhold && u + npairs >= units) ? KS - 1 : KS;
                for (int ks = 0; ks < ks_stop; ++ks, ++it) {
                    const int s = it % kL;
                    if (it >= kL &&
                        !wait_or_abort(empty(s), (uint32_t)((it / kL - 1) & 1), abort_flag, a.err, 41, a.limit)) {
                        ok = false;
                        break;
                    }
                    if (PRE) {
                        // both CTAs' stage s, on the leader's barrier: tokens
                        // 128 r.. of the tile and rows 128 r.. of the decoded
                        // image (image rows, 128 B each, are the tensor map's
                        // rows; the row swizzle has period 8) into CTA r
                        mbar_arrive_expect_tx(full(s), 2 * (kABytes + kR));
                        const int row = (nt * KS + ks) * BN;
                        const bool in = QMLP_INB(((size_t)row + BN) * 128 - 1, a.wdec_bytes, 16);
#pragma unroll
                        for (uint32_t r = 0; r < 2; ++r) {
                            tma_load_2d_pair(base_s + S::A + s * kABytes, r, &amap, ks * BK, mt2 * 2 * BM + (int)r * BM,
                                             full(s));
                            tma_load_2d_pair(base_s + S::Raw + s * kR, r, &bmap, 0, in ? row + (int)r * (BN / 2) : 0,
                                             full(s));
                        }
                        continue;
                    }
                    mbar_arrive_expect_tx(full(s), kABytes + kR);
                    tma_load_2d(base_s + S::A + s * kABytes, &amap, ks * BK, mt2 * 2 * BM + (int)rank * BM, full(s));
                    const uint8_t* src = blk + (size_t)ks * raw_bytes<FMT>();
                    if (!QMLP_INB((size_t)(src - a.tiles) + raw_bytes<FMT>() - 1, a.tiles_bytes, 15)) src = a.tiles;
                    const uint32_t dst = base_s + S::Raw + s * kR;
                    if (FMT == kNVFP4) {
                        // rows 128 rank.. of the block: their codes, then their scales
                        bulk_g2s(dst, src + rank * (kRawCodes / 2), kRawCodes / 2, full(s));
                        bulk_g2s(dst + kRawCodes / 2, src + kRawCodes + rank * (BN / 2) * 4, (BN / 2) * 4, full(s));
                    } else {
                        bulk_g2s(dst, src + rank * kR, kR, full(s));
                    }
                }
            }
            if (!ok) {
                for (int q = it - 1; q >= 0 && q >= it - kL; --q)
                    mbar_wait_bounded(full(q % kL), (uint32_t)((q / kL) & 1), kGemmWaitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true, issued = false;
            for (int u = pair; u < units && ok; u += npairs, ++tc) {
                const int buf = tc & 1, use = tc >> 1;
                if (rank == 0) {
                    // ---------------- MMA issuer (leader) ----------------
                    if (use > 0 &&
                        (!wait_or_abort(acc_empty(buf), (uint32_t)((use - 1) & 1), abort_flag, a.err, 42, a.limit) ||
                         !wait_cluster_or_abort(pacc(buf), (uint32_t)((use - 1) & 1), abort_flag, a.err, 43,
                                                a.limit))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
                    for (int ks = 0; ks < KS; ++ks, ++it) {
                        const int s = it % kL, b = it % kBSd;
                        const bool ready =
                            wait_or_abort(full(s), (uint32_t)((it / kL) & 1), abort_flag, a.err, 44, a.limit) &&
                            (PRE || (wait_or_abort(bfull(b), (uint32_t)((it / kBSd) & 1), abort_flag, a.err, 45,
                                                   a.limit) &&
                                     wait_cluster_or_abort(pbfull(b), (uint32_t)((it / kBSd) & 1), abort_flag, a.err,
                                                           46, a.limit)));
                        if (!ready) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = base_s + S::A + s * kABytes;
                        const uint32_t sb = PRE ? base_s + S::Raw + s * kR : base_s + S::B + b * kBHalf;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            umma_f16_pair(d_tmem, smem_desc_sw128(sa + k * 32), smem_desc_sw128(sb + k * 32),
                                          PRE ? kIdescPairBF16 : kIdescPair, (ks != 0 || k != 0) ? 1u : 0u);
                        issued = true;
                        umma_commit_pair(empty(s));
                        if (!PRE) umma_commit_pair(bempty(b));
                    }
                    if (!ok) break;
                    umma_commit_pair(acc_full(buf));
                } else {
                    // ---------------- forwarder (peer): accumulator drained ----------------
                    if (use > 0) {
                        if (!wait_or_abort(acc_empty(buf), (uint32_t)((use - 1) & 1), abort_flag, a.err, 47, a.limit)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_remote(pacc(buf), 0);
                    }
                }
            }
            // every MMA that wrote either CTA's TMEM must be finished before
            // TMEM is freed: the leader's last commit reaches both done barriers
            if (rank == 0 && issued) umma_commit_pair(done_bar);
            if (rank != 0 || issued) mbar_wait_bounded(done_bar, 0, kGemmWaitNs);
        }
    } else if (warp < 2 + kEpiWarps) {
        // ---------------- epilogue: this CTA's 128 tokens ----------------
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        int tc = 0;
        for (int u = pair; u < units; u += npairs, ++tc) {
            const int nt = u / Mt2, mt2 = u % Mt2;
            const int buf = tc & 1, use = tc >> 1;
            const bool ready = wait_or_abort(acc_full(buf), (uint32_t)(use & 1), abort_flag, a.err, 50, a.limit);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const int m = mt2 * 2 * BM + (int)rank * BM + row_in_tile;
            const bool live = m < a.M;
            const int sg = live && a.sig ? a.sig[m] : 0;  // no prescale (null sig): bf16 operands
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
            store_tile<FMT>(a, tbase, m, live, sg, nt);
            tc_fence_before();
            mbar_arrive(acc_empty(buf));
        }
    } else if (!PRE) {
        // ---------------- decoders: rows 128 rank.. of each weight block ----------------
        // kDecGroups groups of warps take turns by step, each decoding a whole
        // half-B stage: the peer's arrival on the leader's barrier is a
        // release at cluster scope, and its fence then overlaps the other
        // groups' decoding instead of gating every step (measured at M=8192,
        // NVFP4: 6.65 ms with all decoders on each step, 4.67 with two groups).
        constexpr int kGT = kDecThreads / kDecGroups;  // threads of a group
        constexpr int kItems = (BN / 2) * 2 / kGT;     // (row, 32-k half) items per thread and step
        const int dg = (warp - (2 + kEpiWarps)) / (kDecWarps / kDecGroups);
        const int dt = threadIdx.x - (2 + kEpiWarps) * 32 - dg * kGT;
        static_assert(kBS % kDecGroups == 0 && (BN / 2) * 2 % kGT == 0, "whole stages per group");
        int it = 0;
        bool ok = true;
        for (int u = pair; u < units && ok; u += npairs) {
            for (int ks = 0; ks < KS; ++ks, ++it) {
                if (it % kDecGroups != dg) continue;
                const int s = it % kL, b = it % kBSd;
                if (!wait_or_abort(full(s), (uint32_t)((it / kL) & 1), abort_flag, a.err, 51, a.limit) ||
                    (it >= kBSd &&
                     !wait_or_abort(bempty(b), (uint32_t)((it / kBSd - 1) & 1), abort_flag, a.err, 52, a.limit))) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = base + S::Raw + s * kR;
                uint8_t* bt = base + S::B + b * kBHalf;
#pragma unroll
                for (int j = 0; j < kItems; ++j) {
                    const int item = dt + j * kGT;  // (row, 32-k half)
                    if (FMT == kNVFP4) decode_item(raw, bt, item >> 1, item & 1, kRawCodes / 2);
                    else decode_item_fp8(raw, bt, item >> 1, item & 1);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                // the leader's MMA thread waits on its own decoders and,
                // directly, on the peer's (whose A stage landed before they
                // could read the weight half of the same step)
                if (rank == 0) mbar_arrive(bfull(b));
                else mbar_arrive_remote(pbfull(b), 0);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA leaves (nor frees TMEM) while the other may still address
    // its shared memory or its MMAs run
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// Split-K: out = epilogue( sum over the splits, in split order, of the fp32
// partials ) with the tile epilogue's arithmetic (2^-sigma[m], the factor,
// SiLU for gate/up, bf16). One thread per output element.
template <int FMT>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const Args a) {
    const bool swiglu = a.epi == kEpiSwiGLU;
    const int nout = swiglu ? a.N / 2 : a.N;
    const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long)a.M * nout) return;
    const int m = (int)(idx / nout), n = (int)(idx % nout);
    const int sg = a.sig ? a.sig[m] : 0;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)m * a.ldo + n;
    const size_t plane = (size_t)a.M * a.N;
    const float* ws = a.ws + (size_t)m * a.N;
    if (!QMLP_INB((size_t)m * a.ldo + n, (size_t)a.M * a.ldo, 14)) return;
    if (swiglu) {
        const int col = (n / (BN / 2)) * BN + n % (BN / 2);  // gate column of the interleaved tile
        float g = 0.0f, u = 0.0f;
        for (int sp = 0; sp < a.splits; ++sp) {
            if (!QMLP_INB((size_t)m * a.N + sp * plane + col + BN / 2, a.ws_elems, 14)) break;
            g += ws[sp * plane + col];
            u += ws[sp * plane + col + BN / 2];
        }
        const float fg = FMT == kNVFP4 ? a.inv0 : a.cs0[n], fu = FMT == kNVFP4 ? a.inv1 : a.cs1[n];
        const float gv = scalbnf(g, -sg) * fg, uv = scalbnf(u, -sg) * fu;
        *out = __float2bfloat16_rn(silu_f32(gv) * uv);
    } else {
        float y = 0.0f;
        for (int sp = 0; sp < a.splits; ++sp)
            if (QMLP_INB((size_t)m * a.N + sp * plane + n, a.ws_elems, 14)) y += ws[sp * plane + n];
        const float f = FMT == kNVFP4 ? a.inv0 : a.cs0[n];
        *out = __float2bfloat16_rn(scalbnf(y, -sg) * f);
    }
}

// Dequantise-once prefill: every weight block of a projection -> its decoded
// stage image, a 128-byte swizzled K-major bf16 tile [256 rows][128 B] that
// the GEMM copies into shared memory as it is (the swizzle is the one the
// decoder warps apply: 16-byte chunk c of row n sits at c ^ (n & 7), the
// image being 1024-byte aligned like a stage). Every decoded weight is exact
// in bf16 as in fp16 (NVFP4: E2M1 x E4M3, at most six significant bits in
// [2^-10, 2688]; FP8: four bits in [2^-9, 448]), so the GEMM multiplies the
// bf16 activations as they are. One thread per 16-byte output chunk (eight
// weights of one row): a warp stores 512 contiguous bytes (four rows) and
// loads the 128 packed bytes of those rows.
template <int FMT>
__global__ void __launch_bounds__(256) predecode_kernel(const uint8_t* __restrict__ tiles, long nblk,
                                                        uint8_t* __restrict__ wdec, size_t tiles_bytes,
                                                        size_t wdec_bytes) {
    constexpr int kChunks = BN * 8;  // 16-byte chunks of an image
    const long total = nblk * kChunks;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const long blk = idx / kChunks;
        const int n = (int)(idx % kChunks) >> 3, p = (int)(idx & 7);  // row, stored chunk
        const int l = p ^ (n & 7);                                     // its k-chunk: k = 8 l .. 8 l + 7
        if (!QMLP_INB((blk + 1) * raw_bytes<FMT>() - 1, tiles_bytes, 17) ||
            !QMLP_INB((blk + 1) * kBBytes - 1, wdec_bytes, 17))
            continue;
        const uint8_t* raw = tiles + blk * raw_bytes<FMT>();
        uint32_t h[4];
        if (FMT == kNVFP4) {
            const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(raw + n * 32 + l * 4));
            const uint32_t sf = e4m3x2_to_f16x2(__ldg(raw + kRawCodes + n * 4 + (l >> 1)));
            const uint32_t sc = dup_lo16(sf);
            e2m1x4_to_f16x2x4(w, h[0], h[1], h[2], h[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = hmul2_u32(h[j], sc);  // exact in fp16
        } else {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(raw + n * 64 + l * 8));
            e4m3x4_to_f16x2x2(w.x, h[0], h[1]);
            e4m3x4_to_f16x2x2(w.y, h[2], h[3]);
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
            o[j] = pack_bf16x2(f.x, f.y);  // exact (see above)
        }
        *reinterpret_cast<uint4*>(wdec + blk * kBBytes + n * 128 + p * 16) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// a (bf16 [M, C]) -> a16 (fp16 [M, C]) * 2^sig[m], sig[m] = the exponent
// that brings max|a[m, :]| into [2^14, 2^15). One CTA per row.
__global__ void __launch_bounds__(256) prescale_rows_kernel(const __nv_bfloat16* __restrict__ a, __half* a16,
                                                            int* sig, int M, int C) {
    __shared__ float red[8];
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4* row = reinterpret_cast<const uint4*>(a + (size_t)m * C);
        float mx = 0.0f;
        for (int i = threadIdx.x; i < C / 8; i += blockDim.x) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] << 16)));
                mx = fmaxf(mx, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
        __syncthreads();
        float rmax = 0.0f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) rmax = fmaxf(rmax, red[i]);
        const int e = prescale_exponent(rmax);
        if (threadIdx.x == 0) sig[m] = e;
        uint4* orow = reinterpret_cast<uint4*>(a16 + (size_t)m * C);
        for (int i = threadIdx.x; i < C / 8; i += blockDim.x) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = scalbnf(__uint_as_float(w[j] << 16), e);
                const float hi = scalbnf(__uint_as_float(w[j] & 0xFFFF0000u), e);
                const __half2 h = __floats2half2_rn(lo, hi);
                o[j] = *reinterpret_cast<const uint32_t*>(&h);
            }
            orow[i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();  // red[] is reused by the next row
    }
}

// Create-time repack into the weight-block layout (see the top of the file).
__global__ void repack_gemm_kernel(const uint8_t* __restrict__ w0, const uint8_t* __restrict__ s0,
                                   const uint8_t* __restrict__ w1, const uint8_t* __restrict__ s1, int N, int K,
                                   int interleave, uint8_t* __restrict__ tiles) {
    const int KS = K / BK;
    const long total = (long)(N / BN) * KS * BN;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int r = (int)(idx % BN);
        const long blk = idx / BN;  // = j * KS + ks
        const int ks = (int)(blk % KS);
        const int j = (int)(blk / KS);
        const uint8_t* w;
        const uint8_t* s;
        int row;
        if (interleave) {
            const bool up = r >= BN / 2;
            w = up ? w1 : w0;
            s = up ? s1 : s0;
            row = j * (BN / 2) + (r - (up ? BN / 2 : 0));
        } else {
            w = w0;
            s = s0;
            row = j * BN + r;
        }
        uint8_t* dst = tiles + blk * raw_bytes<kNVFP4>();
        const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)row * (K / 2) + ks * (BK / 2));
        uint4* dc = reinterpret_cast<uint4*>(dst + r * 32);
        dc[0] = src[0];
        dc[1] = src[1];
        *reinterpret_cast<uint32_t*>(dst + kRawCodes + r * 4) =
            *reinterpret_cast<const uint32_t*>(s + (size_t)row * (K / 16) + ks * (BK / 16));
    }
}

// FP8: block row r of (n-tile j, k-step ks) = the 64 e4m3fn bytes of weight
// row `row` at k = 64 ks .. 64 ks + 63 (same row mapping as NVFP4).
__global__ void repack_fp8_gemm_kernel(const uint8_t* __restrict__ w0, const uint8_t* __restrict__ w1, int N, int K,
                                       int interleave, uint8_t* __restrict__ tiles) {
    const int KS = K / BK;
    const long total = (long)(N / BN) * KS * BN;
    for (long idx = (long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int r = (int)(idx % BN);
        const long blk = idx / BN;  // = j * KS + ks
        const int ks = (int)(blk % KS);
        const int j = (int)(blk / KS);
        const uint8_t* w = w0;
        int row = j * BN + r;
        if (interleave) {
            const bool up = r >= BN / 2;
            w = up ? w1 : w0;
            row = j * (BN / 2) + (r - (up ? BN / 2 : 0));
        }
        const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)row * K + ks * BK);
        uint4* dst = reinterpret_cast<uint4*>(tiles + blk * raw_bytes<kFP8>() + r * BK);
#pragma unroll
        for (int v = 0; v < 4; ++v) dst[v] = src[v];
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// The CTA-pair GEMM over `pairs_wanted` clusters of two (fewer if fewer fit at
// once: the pairs loop over the tiles).
template <int FMT, bool PRE>
cudaError_t launch_pair(const CUtensorMap& map, const CUtensorMap& bmap, const Args& a, int pairs_wanted,
                        cudaStream_t s) {
    static int max_pairs = -1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SmemP<FMT, PRE>::Bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (max_pairs < 0) {
        cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<FMT, PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SmemP<FMT, PRE>::Bytes);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(2);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<FMT, PRE>, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_pairs = n;
    }
    cfg.gridDim = dim3((unsigned)(2 * std::min(pairs_wanted, max_pairs)));
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<FMT, PRE>, map, bmap, a);
}

template <int FMT, bool PRE>
cudaError_t launch_inst(const CUtensorMap& map, const Args& a, int grid, cudaStream_t s) {
    static bool attr = false;
    constexpr int bytes = Smem<FMT, PRE>::Bytes;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_kernel<FMT, false, PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_kernel<FMT, true, PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    if (a.splits > 1) gemm_kernel<FMT, true, PRE><<<grid, kThreads, bytes, s>>>(map, a);
    else gemm_kernel<FMT, false, PRE><<<grid, kThreads, bytes, s>>>(map, a);
    return cudaPeekAtLastError();
}

// The projection's weight blocks -> their decoded images in wdec (= a.wdec,
// which the GEMM then only reads).
template <int FMT>
cudaError_t launch_predecode(const Args& a, uint8_t* wdec, int num_sms, cudaStream_t s) {
    const long nblk = (long)(a.N / BN) * (a.Kd / BK);
    const long items = nblk * (BN * 8);
    const int pgrid = (int)std::min<long>((items + 255) / 256, 8L * std::max(num_sms, 1));
    predecode_kernel<FMT><<<pgrid, 256, 0, s>>>(a.tiles, nblk, wdec, a.tiles_bytes, a.wdec_bytes);
    return cudaPeekAtLastError();
}

template <int FMT>
cudaError_t launch_fmt(const CUtensorMap& map, const Args& a, int grid, cudaStream_t s) {
    cudaError_t e = a.wdec ? launch_inst<FMT, true>(map, a, grid, s) : launch_inst<FMT, false>(map, a, grid, s);
    if (e != cudaSuccess || a.splits == 1) return e;
    const long n = (long)a.M * (a.epi == kEpiSwiGLU ? a.N / 2 : a.N);
    splitk_reduce_kernel<FMT><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a);
    return cudaPeekAtLastError();
}

bool gemm_supported(int K, int N) { return K >= BK && K % BK == 0 && N >= BN && N % BN == 0; }

size_t gemm_splitk_ws_elems(int num_sms) { return (size_t)std::max(num_sms, 1) * BM * BN; }

size_t gemm_decoded_bytes(int N, int K) { return (size_t)(N / BN) * (K / BK) * kBBytes; }

cudaError_t launch_gemm_predecode(const GemmProj& P, uint8_t* wdec, size_t wdec_bytes, int num_sms, cudaStream_t s) {
    if (!gemm_supported(P.K, P.N) || !P.tiles || !wdec || wdec_bytes < gemm_decoded_bytes(P.N, P.K))
        return cudaErrorInvalidValue;
    Args a = {};
    a.tiles = P.tiles;
    a.N = P.N;
    a.Kd = P.K;
    a.tiles_bytes = gemm_tiles_bytes(P.fmt, P.N, P.K);
    a.wdec = wdec;
    a.wdec_bytes = gemm_decoded_bytes(P.N, P.K);
    return P.fmt == kFP8 ? launch_predecode<kFP8>(a, wdec, num_sms, s) : launch_predecode<kNVFP4>(a, wdec, num_sms, s);
}

size_t gemm_tiles_bytes(int fmt, int N, int K) {
    return (size_t)(N / BN) * (K / BK) * (fmt == kNVFP4 ? raw_bytes<kNVFP4>() : raw_bytes<kFP8>());
}

cudaError_t repack_nvfp4_gemm(const uint8_t* w0, const uint8_t* s0, const uint8_t* w1, const uint8_t* s1, int N,
                              int K, bool interleave, uint8_t* tiles, cudaStream_t s) {
    if (!gemm_supported(K, N) || (interleave && (!w1 || !s1))) return cudaErrorInvalidValue;
    const long total = (long)(N / BN) * (K / BK) * BN;
    const int grid = (int)std::min<long>((total + 255) / 256, 65535);
    repack_gemm_kernel<<<grid, 256, 0, s>>>(w0, s0, w1, s1, N, K, interleave ? 1 : 0, tiles);
    return cudaPeekAtLastError();
}

cudaError_t repack_fp8_gemm(const uint8_t* w0, const uint8_t* w1, int N, int K, bool interleave, uint8_t* tiles,
                            cudaStream_t s) {
    if (!gemm_supported(K, N) || (interleave && !w1)) return cudaErrorInvalidValue;
    const long total = (long)(N / BN) * (K / BK) * BN;
    const int grid = (int)std::min<long>((total + 255) / 256, 65535);
    repack_fp8_gemm_kernel<<<grid, 256, 0, s>>>(w0, w1, N, K, interleave ? 1 : 0, tiles);
    return cudaPeekAtLastError();
}

cudaError_t launch_gemm(const GemmLaunch& L, int num_sms, cudaStream_t s) {
    const GemmProj& P = L.w;
    if (!gemm_supported(P.K, P.N) || L.M < 1 || !L.a16 || !L.sig) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;

    // dequantise-once: bf16 weight images against the bf16 activations as
    // they are
    const bool dq = L.wdec != nullptr;
    if (dq && L.wdec_bytes < gemm_decoded_bytes(P.N, P.K)) return cudaErrorInvalidValue;

    // 1. per-token fp16 prescale of the activations (decoder-warp GEMMs,
    //    whose decoders write fp16 weights)
    if (!dq) {
        const int pgrid = std::min(L.M, 8 * std::max(num_sms, 1));
        prescale_rows_kernel<<<pgrid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(L.a),
                                                    static_cast<__half*>(L.a16), L.sig, L.M, P.K);
        cudaError_t e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
    }

    // 2. tensor map of the MMA's activations: [M rows, K] row-major, box 64 x
    //    128 (fp16 prescaled, or the bf16 input itself)
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)P.K, (cuuint64_t)L.M};
    const cuuint64_t strides[1] = {(cuuint64_t)P.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BM};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, dq ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            dq ? const_cast<void*>(L.a) : L.a16, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    // 3. the GEMM
    Args a;
    a.tiles = P.tiles;
    a.M = L.M;
    a.N = P.N;
    a.Kd = P.K;
    a.epi = L.epi;
    a.raw_sel = L.raw_sel;
    a.interleaved = P.interleaved ? 1 : 0;
    a.inv0 = P.inv_g0;
    a.inv1 = P.inv_g1;
    a.cs0 = P.cs0;
    a.cs1 = P.cs1;
    if (P.fmt == kFP8 && (!P.cs0 || (P.interleaved && !P.cs1))) return cudaErrorInvalidValue;
    a.sig = dq ? nullptr : L.sig;
    a.out = L.out;
    a.ldo = L.epi == kEpiSwiGLU ? P.N / 2 : (L.epi == kEpiRaw && P.interleaved ? P.N / 2 : P.N);
    a.err = L.err;
    a.limit = L.wait_ns ? L.wait_ns : kGemmWaitNs;
    a.withhold = L.withhold ? 1 : 0;
    a.tiles_bytes = gemm_tiles_bytes(P.fmt, P.N, P.K);
    a.ws_elems = L.ws ? gemm_splitk_ws_elems(num_sms) : 0;
    a.wdec = dq ? L.wdec : nullptr;
    a.wdec_bytes = dq ? gemm_decoded_bytes(P.N, P.K) : 0;
    if (dq && !L.images_ready) {  // the images first
        const cudaError_t e = P.fmt == kFP8 ? launch_predecode<kFP8>(a, L.wdec, num_sms, s)
                                            : launch_predecode<kNVFP4>(a, L.wdec, num_sms, s);
        if (e != cudaSuccess) return e;
    }
    // Split-K when the tiles cannot fill the GPU (small M, or the down
    // projection's few column tiles): each (tile, k-range) unit writes fp32
    // partials and a reduce kernel adds them in split order. The partials
    // never exceed num_sms tiles' worth: splits * tiles <= num_sms.
    const int tiles0 = ((L.M + BM - 1) / BM) * (P.N / BN);
    const int KS = P.K / BK;
    a.splits = 1;
    a.ws = L.ws;
    if (L.ws && L.epi != kEpiRaw && !L.pair && 2 * tiles0 <= num_sms)
        a.splits = std::max(1, std::min(std::min(num_sms / tiles0, KS / 8), kMaxSplits));
    // 256-token tiles on CTA pairs (every weight row decoded once per 256
    // tokens), when asked for
    if (L.pair) {
        if (L.M < kPairMinM) return cudaErrorInvalidValue;
        const int pairs = std::min(((L.M + 2 * BM - 1) / (2 * BM)) * (P.N / BN), std::max(num_sms, 2) / 2);
        if (!dq)
            return P.fmt == kFP8 ? launch_pair<kFP8, false>(map, map, a, pairs, s)
                                 : launch_pair<kNVFP4, false>(map, map, a, pairs, s);
        // the decoded images as rows of 128 bytes, 128-row boxes (a CTA's
        // half of a k-step's image), no swizzle (the images carry it)
        CUtensorMap bmap;
        const cuuint64_t bdims[2] = {128, (cuuint64_t)(a.wdec_bytes / 128)};
        const cuuint64_t bstrides[1] = {128};
        const cuuint32_t bbox[2] = {128, (cuuint32_t)(BN / 2)};
        if (enc(&bmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, L.wdec, bdims, bstrides, bbox, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        return P.fmt == kFP8 ? launch_pair<kFP8, true>(map, bmap, a, pairs, s)
                             : launch_pair<kNVFP4, true>(map, bmap, a, pairs, s);
    }
    const int grid = std::min(tiles0 * a.splits, std::max(num_sms, 1));
    return P.fmt == kFP8 ? launch_fmt<kFP8>(map, a, grid, s) : launch_fmt<kNVFP4>(map, a, grid, s);
}

QMLP_BOUNDS_UNIT(gemm_tc)

}  // namespace qmlp
