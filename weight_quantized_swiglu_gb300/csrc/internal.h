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

// One projection [N, K] in the GEMV ("fragment-native") layout: one record
// per 16-row x 64-k chunk, row-tile-major (see gemv_frag.cuh):
//  NVFP4: 576 B = 512 B of E2M1 bytes in mma A-fragment order + 64 B of E4M3
//         scales; FP8: 1024 B of e4m3fn bytes, with chs = fp32 [N] scales.
// Nt = N/16 row tiles, Kc = ceil(K/64) chunks (zero padded).
// Records are stored interleaved for the stream kernel: warp w of TWr
// streaming warps owns the logical records [w*Lr, (w+1)*Lr) (row-tile-major
// order), taken Rr at a time; logical record u = w*Lr + k is stored at
// ((k / Rr) * TWr + w) * Rr + k % Rr, so at step j the 16 warps of a CTA
// find their Rr records each in one contiguous block and the GPU sweeps one
// contiguous window at a time. Lr is a multiple of Rr.
struct GemvProj {
    const uint8_t* wc = nullptr;
    const float* chs = nullptr;
    float inv_g = 1.0f;
    int N = 0, K = 0, Nt = 0, Kc = 0;
    int Lr = 1, TWr = 1, Rr = 1;
};
__host__ __device__ inline size_t gemv_rec_pos(size_t u, int Lr, int TWr, int Rr) {
    const size_t w = u / (size_t)Lr, k = u % (size_t)Lr;
    return ((k / (size_t)Rr) * (size_t)TWr + w) * (size_t)Rr + k % (size_t)Rr;
}
// Streaming warps of the layout on a device with num_sms SMs.
int gemv_layout_warps(int num_sms);

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

// Persistent stream-K GEMV (gemv_stream.cu). One phase = one projection, or
// gate+up with the SwiGLU epilogue; with a second phase the launch is
// cooperative and runs gate/up -> grid barrier -> down.
struct GemvStreamPhase {
    int epi;
    GemvProj p0, p1;
    const void* x;   // bf16 [M, p0.K]
    void* out;       // bf16 or fp32 [M, p0.N]
    int* counters;   // >= p0.Nt zeroed ints
};
bool gemv_stream_fits(int fmt, int M, int K, int np, int R);
size_t gemv_stream_part_elems(int K, int I, int num_sms);
cudaError_t launch_gemv_stream(int fmt, int M, const GemvStreamPhase& A, const GemvStreamPhase* B, float* part,
                               size_t part_cap, unsigned* bar, int* err, int num_sms, cudaStream_t s);

// Create-time repack into the GEMV layout. src pointers are device copies of
// the checkpoint layout.
cudaError_t repack_nvfp4_gemv(const uint8_t* w, const uint8_t* scale, int N, int K, int Lr, int TWr, int Rr,
                              uint8_t* wc, cudaStream_t s);
cudaError_t repack_fp8_gemv(const uint8_t* w, int N, int K, int Lr, int TWr, int Rr, uint8_t* wc, cudaStream_t s);
size_t gemv_codes_bytes(int fmt, int N, int K, int Lr, int TWr);
// Records per warp per step of the layout: gate/up (streamed in pairs) take
// half as many as a projection streamed alone, so one step fills the same
// number of bytes in both cases; FP8 records (1024 B) take half as many as
// NVFP4 ones (576 B), so a step is 32-37 KB for both formats.
__host__ __device__ constexpr int gemv_recs_pair(int fmt) { return fmt == kFP8 ? 1 : 2; }
__host__ __device__ constexpr int gemv_recs_single(int fmt) { return fmt == kFP8 ? 2 : 4; }
// Largest split-K partial buffer (fp32 elements) any GEMV launch of a handle
// with these sizes can need for M <= 16.
size_t gemv_part_elems(int K, int I, int num_sms);

// ---------------------------------------------------------------------------
// I-partitioned fused decode MLP (gemv_split.cu): CTA b of G owns gate/up
// row tiles [T*b, T*(b+1)) and the matching Cb = T/4 down k-chunks.
// ---------------------------------------------------------------------------
struct SplitPlan {
    int G = 0;        // CTAs (0: no plan for this shape / device)
    int T = 0;        // gate/up row tiles per CTA
    int Cb = 0;       // down 64-k chunks per CTA
    int LA = 0;       // gate/up records per warp (= T*Kc/16; the gate/up layout uses Lr = LA, TWr = 16G)
    int LB = 0;       // down records per warp in the CTA-sliced layout (multiple of RB)
    int RA = 0, RB = 0;  // records per warp per step: gate/up pairs, down
    int SA = 0;       // most warps sharing one gate/up tile
};
SplitPlan plan_split(int fmt, int K, int I, int num_sms);
bool split_fits(int fmt, int M, int K, const SplitPlan& P);
size_t split_part_elems(int K, const SplitPlan& P);       // fp32 partials for M <= 16
size_t split_codes_bytes(int fmt, const SplitPlan& P);     // down records, CTA-sliced
// Down projection [K, I] into the CTA-sliced layout: local record u = w*LB + k
// of CTA b (u < Nt*Cb) is (row tile u / Cb, chunk Cb*b + u % Cb), stored at
// ((k / RB) * 16G + 16b + w) * RB + k % RB; records past Nt*Cb are zero.
cudaError_t repack_nvfp4_split(const uint8_t* w, const uint8_t* scale, int N, int K, const SplitPlan& P,
                               uint8_t* wc, cudaStream_t s);
cudaError_t repack_fp8_split(const uint8_t* w, int N, int K, const SplitPlan& P, uint8_t* wc, cudaStream_t s);
struct SplitLaunch {
    int fmt = 0, M = 0, K = 0, I = 0;
    GemvProj gate, up;               // GEMV layout with TWr = 16G, Lr = LA
    const uint8_t* wdown = nullptr;  // CTA-sliced down records
    const float* chsd = nullptr;     // FP8 down per-channel scales
    float invd = 1.0f;               // NVFP4 down 1/global
    const void* x = nullptr;         // bf16 [M, K]
    bool x_in_host = false;          // x is device-mapped host memory: staged with plain loads
    void* act_out = nullptr;         // optional bf16 [M, I]
    void* out = nullptr;             // bf16 [M, K]
    float* out_f32 = nullptr;        // optional fp32 [M, K]: sums without the down factor, written instead of out
    const void* act_in = nullptr;    // optional bf16 [M, I]: the down projection consumes these (debug)
    float* dbg_g = nullptr;          // optional fp32 [M, I]: raw gate dot products (debug; with dbg_u)
    float* dbg_u = nullptr;          // optional fp32 [M, I]: raw up dot products (debug)
    float* part = nullptr;           // >= split_part_elems
    unsigned long long* ticket = nullptr;  // grid-barrier ticket counter (zeroed at create)
    int* err = nullptr;
    uint64_t wait_ns = 0;            // bounded-wait limit (0: the kernel's default of 2 s)
    bool withhold = false;           // error-path tests: the last weight step is never issued
    size_t lim_a = 0;                // index-check tests: bytes of the gate/up banks the checks allow (0: all)
};
cudaError_t launch_split(const SplitLaunch& L, const SplitPlan& P, cudaStream_t s);

// Tensor-parallel combine (tp_shard.cu): out[m, o] = bf16( sigma_d[o] * sum
// over r = 0..nranks-1, in rank order, of partials[r][m][o] ), sigma_d = invd
// (NVFP4) or chsd[o] (FP8).
cudaError_t launch_shard_combine(int fmt, const float* partials, int nranks, int M, int K, float invd,
                                 const float* chsd, void* out, cudaStream_t s);

// ---------------------------------------------------------------------------
// Tensor-core prefill GEMM (NVFP4, tcgen05)
// ---------------------------------------------------------------------------
struct GemmProj {
    int fmt = kNVFP4;                    // kNVFP4 or kFP8
    const uint8_t* tiles = nullptr;      // weight blocks [N/256][K/64][9216 B NVFP4 | 16384 B FP8], see gemm_tc.cu
    float inv_g0 = 1.0f, inv_g1 = 1.0f;  // NVFP4 global factors: (gate, up) when interleaved, else both = down
    const float* cs0 = nullptr;          // FP8 per-channel scales: gate when interleaved, else the projection's
    const float* cs1 = nullptr;          // FP8 up scales when interleaved
    int N = 0, K = 0;                    // N weight rows (2I when interleaved), K contraction length
    bool interleaved = false;            // tile rows = 128 gate rows then the same 128 up rows
};
size_t gemm_tiles_bytes(int fmt, int N, int K);
cudaError_t repack_fp8_gemm(const uint8_t* w0, const uint8_t* w1, int N, int K, bool interleave, uint8_t* tiles,
                            cudaStream_t s);
cudaError_t repack_nvfp4_gemm(const uint8_t* w0, const uint8_t* s0, const uint8_t* w1,
                              const uint8_t* s1, int N, int K, bool interleave, uint8_t* tiles,
                              cudaStream_t s);
struct GemmLaunch {
    int epi = kEpiPlain;  // kEpiSwiGLU / kEpiPlain / kEpiRaw
    int raw_sel = 0;      // kEpiRaw on an interleaved GEMM: 0 = gate rows, 1 = up rows
    GemmProj w;
    const void* a = nullptr;  // bf16 [M, K]
    int M = 0;
    void* out = nullptr;      // bf16 [M, N_out] or fp32 [M, N_out] (raw)
    void* a16 = nullptr;      // workspace fp16 [M, K]: prescaled activations
    int* sig = nullptr;       // workspace [M]: per-token prescale exponents
    int* err = nullptr;       // device error word
    float* ws = nullptr;      // split-K partials, >= gemm_splitk_ws_elems (null: no split-K)
    uint64_t wait_ns = 0;     // bounded-wait limit (0: the kernel's default of 2 s)
    bool withhold = false;    // error-path tests: the last k-step of each CTA is never loaded
    bool pair = false;        // the CTA-pair kernel (M >= kPairMinM; never split-K)
    uint8_t* wdec = nullptr;  // dequantise-once: decoded stage images of w (null: the decoder warps decode)
    size_t wdec_bytes = 0;    // bytes of wdec, >= gemm_decoded_bytes(w.N, w.K)
    bool images_ready = false;  // dequantise-once: wdec already holds w's images (no predecode launch)
};
constexpr int kPairMinM = 256;  // one 256-token tile of a CTA pair
cudaError_t launch_gemm(const GemmLaunch& L, int num_sms, cudaStream_t s);
size_t gemm_splitk_ws_elems(int num_sms);
size_t gemm_decoded_bytes(int N, int K);  // bf16 stage images of an [N, K] projection (2 N K bytes)
// The dequantise-once predecode of projection P into wdec, on its own.
cudaError_t launch_gemm_predecode(const GemmProj& P, uint8_t* wdec, size_t wdec_bytes, int num_sms, cudaStream_t s);
bool gemm_supported(int K, int N);

// ---------------------------------------------------------------------------
// Routed-expert AWQ M=1
// ---------------------------------------------------------------------------
struct MoeLaunch {
    int E, K, I, meta_bytes;
    int sliced = 0;           // 1: the banks are lane-sliced (the handle's copy), 0: checkpoint layout
    const uint8_t* w13;       // see moe_awq.cu
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

// M tokens, routes grouped by expert (see moe_grouped.cu).
constexpr int kMoeGroupedMaxK = 8192;  // x of a group's 8 tokens is staged in shared memory
constexpr int kMoeGroupedMaxE = 8192;  // the routing CTA keeps 4 ints per expert in shared memory
struct MoeGroupedLaunch {
    int E, K, I, meta_bytes, M, topk;
    int num_sms = 0;
    const uint8_t* w13;
    const uint8_t* w13_meta;
    const uint8_t* w2;
    const uint8_t* w2_meta;
    const void* x;                 // [M, K]
    int x_is_bf16;
    const int32_t* ids;            // [M, topk]
    const float* rw;               // [M, topk]
    __half* out;                   // [M, K]
    __half* act_ws;                // [>= M*topk, I]
    __half* y_ws;                  // [>= M*topk, K]
    int* route_list;               // [>= M*topk]
    int4* groups;                  // [>= moe_grouped_max_groups(M*topk, E)]
    int* n_groups;                 // one int
};
size_t moe_grouped_max_groups(int routes, int E);
cudaError_t launch_moe_grouped(const MoeGroupedLaunch& L, cudaStream_t s);
// W13 bank of a handle in warp blocks: the one-token and grouped W13 kernels
// split K over kMoeKSplit warps, and warp ks of row octet o (gate rows
// 8o..8o+7 and the matching up rows) reads one contiguous block per expert.
// Block (e, o, ks) = [q (gate 0 / up 1)][pair p][lane l = 4g + t][16 B]: the
// 16 bytes are chunks c = ks*cpw + 2p and +1 (64 k each, zero past the warp's
// range), 8 bytes per chunk = the 32-bit words lane t picks from the chunk's
// two 16-byte units of row g (byte t of each word of the unit). Metadata:
// block (e, o, ks) = [q][g][the 2*cpw records of those chunks, padded to a
// multiple of 16 bytes, sized for whole batches of 4 chunks: the one-token
// kernel loads a batch's records at once]. Byte counts per block below.
constexpr int kMoeKSplit = 10;
__host__ __device__ inline int moe_w13_cpw(int K) { return (K / 64 + kMoeKSplit - 1) / kMoeKSplit; }
__host__ __device__ inline int moe_w13_pairs(int K) { return (moe_w13_cpw(K) + 1) / 2; }
__host__ __device__ inline size_t moe_w13_block_bytes(int K) { return (size_t)2 * moe_w13_pairs(K) * 512; }
__host__ __device__ inline int moe_w13_meta_stride(int K, int MB) {
    return (2 * ((moe_w13_cpw(K) + 3) / 4 * 4) * MB + 15) / 16 * 16;
}
__host__ __device__ inline size_t moe_w13_meta_block_bytes(int K, int MB) { return (size_t)2 * 8 * moe_w13_meta_stride(K, MB); }
inline size_t moe_w13_bank_bytes(int E, int I, int K) { return (size_t)E * (I / 8) * kMoeKSplit * moe_w13_block_bytes(K); }
inline size_t moe_w13_meta_bank_bytes(int E, int I, int K, int MB) {
    return (size_t)E * (I / 8) * kMoeKSplit * moe_w13_meta_block_bytes(K, MB);
}
// checkpoint W13 codes [E, 2I, K/2] and records [E, 2I, K/32] x MB -> the
// warp-block bank above
cudaError_t repack_moe_w13_blocks(const uint8_t* w, const uint8_t* meta, int meta_bytes, int E, int I, int K,
                                  uint8_t* w_out, uint8_t* meta_out, cudaStream_t s);
cudaError_t repack_moe(const uint8_t* w, const uint8_t* meta, int meta_bytes, int E, int N,
                       int Kr, uint8_t* w_out, uint8_t* meta_out, cudaStream_t s);

// Index checks of a QMLP_DEBUG_BOUNDS build (common.cuh): each translation
// unit's first failed check, (site << 48) | index, or 0; reading clears it.
// The default build returns 0.
cudaError_t bounds_take_gemv_split(unsigned long long* v);
cudaError_t bounds_take_gemm_tc(unsigned long long* v);
cudaError_t bounds_take_gemv_stream(unsigned long long* v);
cudaError_t bounds_take_gemv_dec(unsigned long long* v);
cudaError_t bounds_take_moe_awq(unsigned long long* v);
cudaError_t bounds_take_moe_grouped(unsigned long long* v);
cudaError_t bounds_take_tp_shard(unsigned long long* v);

}  // namespace qmlp
