// internal.h -- host-side structures shared by the qmlp translation units.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmlp.h"

namespace qmlp {

enum Fmt { kNVFP4 = 1, kFP8 = 2 };

// Rows per tensor-core tile of the GEMV kernels and k per "chunk" (four
// NVFP4 scale groups of 16).
constexpr int kTileRows = 16;
constexpr int kChunkK = 64;

// Epilogue of a GEMV launch.
enum GemvEpi {
    kEpiSwiGLU = 0,  // two projections (gate, up) -> act = bf16(SiLU(g)*u)
    kEpiPlain = 1,   // one projection -> bf16(sigma * acc)
    kEpiRaw = 2      // one projection -> fp32 acc (no scale), debug
};

// One projection [N, K] in the GEMV ("fragment-native") layout.
//  NVFP4: wc = [Nt][Kc][32 lanes][16 B]   E2M1 bytes in mma A-fragment order
//         sc = [Nt][Kc][8 row pairs][8 B] E4M3 scales (row g, row g+8) x 4 groups
//  FP8:   wc = [Nt][Kc][2][32 lanes][16 B] e4m3fn bytes in A-fragment order
//         chs = fp32 [N] per-channel scale
// Nt = N/16 row tiles, Kc = ceil(K/64) chunks (zero padded).
struct GemvProj {
    const uint4* wc = nullptr;
    const uint2* sc = nullptr;
    const float* chs = nullptr;
    float inv_g = 1.0f;
    int N = 0, K = 0, Nt = 0, Kc = 0;
};

struct GemvLaunch {
    int fmt;
    int epi;
    GemvProj p0, p1;         // p1 used by kEpiSwiGLU only
    const void* x;           // bf16 [M, K]
    int M;
    void* out;               // bf16 [M, N] (act or out) or fp32 [M, N] (raw)
    float* part;             // fp32 split-K partials
    size_t part_cap;         // elements available in part
    int* counters;           // >= Nt zeroed ints
};

cudaError_t launch_gemv(const GemvLaunch& L, int num_sms, cudaStream_t s);

// Create-time repack into the GEMV layout. src pointers are device copies of
// the checkpoint layout.
cudaError_t repack_nvfp4_gemv(const uint8_t* w, const uint8_t* scale, int N, int K, uint4* wc,
                              uint2* sc, cudaStream_t s);
cudaError_t repack_fp8_gemv(const uint8_t* w, int N, int K, uint4* wc, cudaStream_t s);
size_t gemv_codes_bytes(int fmt, int N, int K);
size_t gemv_scales_bytes(int fmt, int N, int K);
// Largest split-K partial buffer (fp32 elements) any GEMV launch of a handle
// with these sizes can need for M <= 16.
size_t gemv_part_elems(int K, int I, int num_sms);

// ---------------------------------------------------------------------------
// Tensor-core prefill GEMM (NVFP4, tcgen05)
// ---------------------------------------------------------------------------
struct GemmProj {
    const uint8_t* tiles = nullptr;  // [N/BN][K/BK][BN rows][BK/2 B codes] + scales, see gemm_tc.cu
    float inv_g0 = 1.0f, inv_g1 = 1.0f;  // column halves (gate, up) or both = down
    int N = 0, K = 0;
};
size_t gemm_tiles_bytes(int N, int K);
cudaError_t repack_nvfp4_gemm(const uint8_t* w0, const uint8_t* s0, const uint8_t* w1,
                              const uint8_t* s1, int N, int K, bool interleave, uint8_t* tiles,
                              cudaStream_t s);
struct GemmLaunch {
    int epi;            // kEpiSwiGLU / kEpiPlain / kEpiRaw
    GemmProj w;
    const void* a;      // bf16 [M, K]
    int M;
    void* out;          // bf16 [M, N_out] or fp32 [M, N_out] (raw)
    int* err;           // device error word
};
cudaError_t launch_gemm(const GemmLaunch& L, int num_sms, cudaStream_t s);
bool gemm_supported(int K, int N);

// ---------------------------------------------------------------------------
// Routed-expert AWQ M=1
// ---------------------------------------------------------------------------
struct MoeLaunch {
    int E, K, I, meta_bytes;
    const uint8_t* w13;       // repacked, see moe_awq.cu
    const uint8_t* w13_meta;
    const uint8_t* w2;
    const uint8_t* w2_meta;
    const void* x;
    int x_is_bf16;
    const int32_t* ids;
    const float* rw;
    int topk;
    __half* out;
    __half* act_ws;           // [16][I] workspace
    __half* gu_dbg;           // optional [topk][2I]
    __half* act_dbg;          // optional [topk][I]
    __half* y_dbg;            // optional [topk][K]
};
cudaError_t launch_moe(const MoeLaunch& L, int num_sms, cudaStream_t s);
cudaError_t repack_moe(const uint8_t* w, const uint8_t* meta, int meta_bytes, int E, int N,
                       int Kr, uint8_t* w_out, uint8_t* meta_out, cudaStream_t s);

}  // namespace qmlp
