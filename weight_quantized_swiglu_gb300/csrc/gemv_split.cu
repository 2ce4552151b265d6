// gemv_split.cu -- the whole decode MLP (M <= 16) in one persistent launch,
// with the intermediate dimension partitioned across CTAs.
// Launched with programmatic dependent launch: a CTA may start while the
// previous kernel of the stream still holds SMs (its producer waits for that
// kernel before copying x, its consumers before touching any shared buffer);
// all G <= SMs CTAs, one per SM, are co-resident once it has finished.
//
// Operation (vllm.cpp issue "tp>1 fp8w tail-MLP shard ...", "Proposed fix";
// Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented"):
//   act[m, i] = bf16( SiLU(sg * x[m].Wg[i]) * (su * x[m].Wu[i]) )
//   out[m, n] = bf16( sd * sum_i act[m, i] Wd[n, i] )
// with W decoded on the fly (NVFP4: E2M1 x E4M3, s = 1/global; FP8: e4m3fn,
// s = per-channel scale).
//
// Schedule: CTA b of G owns the T gate/up row tiles [T*b, T*(b+1)) -- the
// act slice i in [16*T*b, 16*T*(b+1)) -- and the matching T*16 columns of
// the down projection. The dependency between the projections is then local
// to the CTA:
//  1. stream gate/up (16 consumer warps, L_A records each, tiles split
//     between warps are combined in shared memory) -> SwiGLU -> the CTA's
//     act slice in shared memory (bf16 values);
//  2. restage the slice as prescaled fp16 fragments, stream the down
//     records of the slice (every output row tile, Cb = T/4 k-chunks) ->
//     the CTA's partial out[m, n] over its slice, fp32, to global memory;
//  3. either (a) one grid-wide barrier (a 64-bit ticket counter: one
//     atomic per CTA), then every CTA reduces a share of the outputs over
//     the G partials in a fixed order and applies the down scale; or (b)
//     the CTA leaves and a small reduce kernel, launched next, does the same
//     sums once this grid has completed. (b) lets the next call's CTAs
//     start as soon as these leave and fill their weight rings before they
//     wait for the reduce kernel: measured faster where the start of a call
//     is HBM-bound (FP8: 44.05 vs 44.97 us at M=1; NVFP4 M=4: 45.8 vs 47.0),
//     slower where the consumers bound it (NVFP4 M=1: 31.0-31.4 vs 30.55 us,
//     the second grid completion is on its critical path), so (a) serves
//     NVFP4 M=1 and (b) everything else.
// The producer warp streams the gate/up records and then the down records
// without a pause (the down weights do not depend on act), one bulk-async
// copy per projection and step into a shared-memory ring, as in
// gemv_stream.cu. No float atomics: every sum has a fixed order.
// Every wait is bounded (globaltimer); on expiry the CTA records the error,
// still arrives at the grid barrier exactly once, waits for its own copies
// in flight and leaves.
#include <algorithm>

#include "gemv_frag.cuh"

namespace qmlp {
namespace {

constexpr int kW = 16;                // consumer warps
constexpr int kCT = kW * 32;          // consumer threads
constexpr int kThr = kCT + 32;        // + one producer warp
constexpr int kDepthMax = 16;
constexpr int kBudget = 220 * 1024;
constexpr int kBars = 2 * kDepthMax * 8 + 16;  // full, empty, x
constexpr uint64_t kLimit = 2000000000ull;  // 2 s: waits for copies known to be in flight
constexpr int kXRawMax = 16 * 1024;  // raw x copied to shared memory up to this size
constexpr int kPreStepsBarrier = 1;          // weight steps issued before the wait on the previous kernel:
constexpr int kPreStepsSep = kDepthMax;      //   schedule (a) / schedule (b) (the whole ring)
constexpr double kSmallCtaBytes = 256.0 * 1024;  // weight bytes a CTA streams in a "small" MLP
constexpr int kRedLoads = 10;                // partials a warp adds per output: G <= 16 * kRedLoads

struct Args {
    // phase A: gate (wc0) and up (wc1), row-tile-major layout over 16*G warps
    const uint8_t* wa0;
    const uint8_t* wa1;
    const float* chs0;
    const float* chs1;
    float inv0, inv1;
    // phase B: down in the CTA-sliced layout
    const uint8_t* wb;
    const float* chsd;
    float invd;
    const __nv_bfloat16* x;    // [M, K]
    __nv_bfloat16* act_out;    // optional [M, I]
    __nv_bfloat16* out;        // [M, K]
    float* out_f32;            // optional [M, K]: the sums in fp32 without the down factor, instead of out
    const __nv_bfloat16* act_in;  // optional [M, I]: phase B consumes these act values (debug)
    float* dbg_g;              // optional [M, I]: gate dot products, fp32, no factor (debug)
    float* dbg_u;              // optional [M, I]: up dot products, likewise
    float* part;               // [G][M][K]
    unsigned long long* ticket;
    int* err;
    int M, K, I;
    int G, T, KcA, LA, Cb, NtD, LB;
    int xs_bytes;              // x staging (phase A) region
    int pa_off, act_off, pb_off;  // byte offsets of the combine / act regions
    int ring_off, slot_bytes, depth;
    int SA;                    // partial slots per gate/up tile
    int xraw_off, xraw_bytes;  // raw bf16 x copied to shared memory (0: staged from global)
    uint64_t limit;            // ns a wait on another role or CTA may take before it gives up
    int withhold;              // error-path tests: the producer never issues the last step
    size_t wa_bytes, wb_bytes; // index checks: bytes of each gate/up bank and of the down bank
    size_t part_elems;         // index checks: floats of the partial buffer
};

struct Ring {
    uint8_t* base;
    uint32_t base_s, full0, empty0;
    uint32_t xbar;  // completion of the x copy
    int slot_bytes, depth;
    uint64_t limit;  // Args::limit
};

// The producer's view of the two phases: step q < steps_a is the gate and up
// blocks of gate/up step q, later steps are down blocks. Step j of CTA b is
// the 16 warps' records R*j..R*j+R-1, contiguous in the interleaved layout.
struct Steps {
    const uint8_t* a0;
    const uint8_t* a1;
    const uint8_t* b;
    size_t stride_a, stride_b;
    uint32_t bytes_a, bytes_b;  // per block
    int steps_a, steps;
    size_t off_a, off_b;        // index checks: offset of this CTA's first block in its bank
    size_t lim_a, lim_b;        // index checks: bank bytes
    const uint8_t* base_a0;     // index checks: bank starts (a failed check copies from there)
    const uint8_t* base_a1;
    const uint8_t* base_b;
};

// Producer (one thread): every step of both phases into the ring, without a
// pause between the phases (the down weights do not depend on act). Returns
// the number of steps issued, or -(issued + 1) after an expired wait.
// (Measured: L2 prefetches of later steps, of both phases or of the down
// steps only, slow the call down by 2-8 us; the bulk copies alone are kept.)
template <int FMT>
QMLP_DEV int produce(const Steps& st, const Ring& r, int* err, int q0, int q1) {
    int slot = q0 % r.depth, round = q0 / r.depth;
    for (int q = q0; q < q1; ++q) {
        if (round > 0 && !mbar_wait_bounded(r.empty0 + 8u * slot, (uint32_t)((round - 1) & 1), r.limit)) {
            atomicExch(err, 24);
            return -(q + 1);
        }
        const uint32_t full = r.full0 + 8u * slot;
        const uint32_t dst = r.base_s + (uint32_t)slot * r.slot_bytes;
        if (q < st.steps_a) {
            const uint8_t* s0 = st.a0 + (size_t)q * st.stride_a;
            const uint8_t* s1 = st.a1 + (size_t)q * st.stride_a;
            if (!QMLP_INB(st.off_a + (size_t)q * st.stride_a + st.bytes_a - 1, st.lim_a, 1)) {
                s0 = st.base_a0;
                s1 = st.base_a1;
            }
            mbar_arrive_expect_tx(full, 2 * st.bytes_a);
            bulk_g2s(dst, s0, st.bytes_a, full);
            bulk_g2s(dst + st.bytes_a, s1, st.bytes_a, full);
        } else {
            const uint8_t* sb = st.b + (size_t)(q - st.steps_a) * st.stride_b;
            if (!QMLP_INB(st.off_b + (size_t)(q - st.steps_a) * st.stride_b + st.bytes_b - 1, st.lim_b, 2))
                sb = st.base_b;
            mbar_arrive_expect_tx(full, st.bytes_b);
            bulk_g2s(dst, sb, st.bytes_b, full);
        }
        if (++slot == r.depth) {
            slot = 0;
            ++round;
        }
    }
    return q1;
}

// 2^-s as a float (exact for every exponent the prescale produces); the
// product v * 2^-s is the correctly rounded v scaled by 2^-s, as scalbnf.
QMLP_DEV float pow2_neg(int s) {
    return (s >= -126 && s <= 126) ? __int_as_float((127 - s) << 23) : scalbnf(1.0f, -s);
}

// Fragment element (p, n, e) of lane (g, t): token m = 8n + 2t + (e & 1),
// row g + 8*(e >> 1). Compact partial layout: [p][m][16 rows] fp32.
template <int NT, int NP>
QMLP_DEV void store_compact(float* dst, int M, const float (&acc)[NP][NT][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = n * 8 + 2 * t + (e & 1);
                if (m < M) dst[(p * M + m) * 16 + g + 8 * (e >> 1)] = acc[p][n][e];
            }
}
template <int NT, int NP>
QMLP_DEV void add_compact(const float* src, int M, float (&v)[NP][NT][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = n * 8 + 2 * t + (e & 1);
                if (m < M) v[p][n][e] += src[(p * M + m) * 16 + g + 8 * (e >> 1)];
            }
}

// Combine a tile's partial through shared memory: store this warp's part in
// its slot, count arrivals; the last of `nc` contributors gets true and the
// slot-ordered sum in `v`.
template <int NT, int NP>
QMLP_DEV bool combine_smem(float* slots, int slot_floats, int slot, int nc, int* cnt, int M, float (&v)[NP][NT][4]) {
    const int lane = threadIdx.x & 31;
    store_compact<NT, NP>(slots + slot * slot_floats, M, v);
    __syncwarp();
    int prev = 0;
    if (lane == 0) {
        __threadfence_block();
        prev = atomicAdd(cnt, 1);
    }
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev != nc - 1) return false;
    __threadfence_block();
    if (lane == 0) *cnt = 0;
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) v[p][n][e] = 0.0f;
    for (int sl = 0; sl < nc; ++sl) add_compact<NT, NP>(slots + sl * slot_floats, M, v);
    return true;
}

// Phase-A epilogue of local tile lt: act = bf16(SiLU(g)*u) into the CTA's
// act slice (and optionally the global act).
template <int FMT, int NT>
QMLP_DEV void epilogue_a(const Args& a, int M, int lt, const float (&v)[2][NT][4], const int* s_sig,
                         float* s_act, int* s_actmax) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int tslice = a.T * 16;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = n * 8 + 2 * t + (e & 1);
            if (m >= M) continue;
            const int r = lt * 16 + g + 8 * (e >> 1);  // row within the CTA's slice
            const int i = blockIdx.x * tslice + r;     // intermediate index
            if (!QMLP_INB((size_t)m * a.I + i, (size_t)a.M * a.I, 4)) continue;
            const float s0 = FMT == kNVFP4 ? a.inv0 : a.chs0[i];
            const float s1 = FMT == kNVFP4 ? a.inv1 : a.chs1[i];
            const float pw = pow2_neg(s_sig[m]);
            const float graw = v[0][n][e] * pw, uraw = v[1][n][e] * pw;
            const float gv = graw * s0;
            const float uv = uraw * s1;
            __nv_bfloat16 act = __float2bfloat16_rn(silu_f32(gv) * uv);
            if (a.dbg_g) {
                a.dbg_g[(size_t)m * a.I + i] = graw;
                a.dbg_u[(size_t)m * a.I + i] = uraw;
            }
            if (a.act_in) act = a.act_in[(size_t)m * a.I + i];
            const float af = __bfloat162float(act);
            s_act[m * tslice + r] = af;
            // running max|act| of the slice (non-negative floats order as
            // their bits): the restage needs no scan of its own
            atomicMax(&s_actmax[m], __float_as_int(fabsf(af)));
            if (a.act_out) a.act_out[(size_t)m * a.I + i] = act;
        }
}

// End of this warp's part of gate/up tile lt: the epilogue when the warp
// covered the whole tile, else the shared-memory combine (the last
// contributor applies the epilogue). Out of line: it runs once per tile
// part, and keeping it out of the streaming loop keeps that loop small.
template <int NT>
struct AccA {
    float v[2][NT][4];
};
template <int FMT, int NT>
__device__ __noinline__ void finish_tile_a(const Args& a, int M, int lt, bool whole, int warp, AccA<NT> acc,
                                           float* s_pa, int pa_floats, int* s_cnta, const int* s_sig, float* s_act,
                                           int* s_actmax) {
    if (whole) {
        epilogue_a<FMT, NT>(a, M, lt, acc.v, s_sig, s_act, s_actmax);
        return;
    }
    const int w0 = (lt * a.KcA) / a.LA, w1 = ((lt + 1) * a.KcA - 1) / a.LA;
    if (combine_smem<NT, 2>(s_pa + (size_t)lt * a.SA * pa_floats, pa_floats, warp - w0, w1 - w0 + 1, &s_cnta[lt], M,
                            acc.v))
        epilogue_a<FMT, NT>(a, M, lt, acc.v, s_sig, s_act, s_actmax);
}

// Phase-B result of down row tile rt over this CTA's slice -> global partial.
template <int NT>
QMLP_DEV void store_part_b(const Args& a, int M, int rt, const float (&v)[1][NT][4], const int* s_sigb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float* dst = a.part + (size_t)blockIdx.x * M * a.K;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = n * 8 + 2 * t + (e & 1);
            if (m < M && QMLP_INB(rt * 16 + g + 8 * (e >> 1), a.K, 5) &&
                QMLP_INB((size_t)blockIdx.x * M * a.K + (size_t)m * a.K + rt * 16 + g + 8 * (e >> 1), a.part_elems, 5))
                dst[(size_t)m * a.K + rt * 16 + g + 8 * (e >> 1)] = v[0][n][e] * pow2_neg(s_sigb[m]);
        }
}

template <int NT, int NP>
QMLP_DEV void zero_acc(float (&acc)[NP][NT][4]);

// x (raw bf16 rows of length K in shared memory) -> prescaled fp16 fragments
// in xs with a single barrier over the consumer threads: every warp finds
// the per-token maxima itself (reading all of x from shared memory), keeps
// the exponents in its own row of sigw, and converts its 1/16 share of the
// 8-element items; k in [K, kpe) is zero. sig (for the epilogue) is written
// by warp 0.
QMLP_DEV void stage_x_local(const uint4* xr, int M, int K, int kpe, uint4* xs, int* sigw, int* sig, int warp) {
    const int lane = threadIdx.x & 31;
    const int k8 = K / 8, p8 = kpe / 8;
    for (int m = 0; m < M; ++m) {
        float mx = 0.0f;
        for (int q = lane; q < k8; q += 32) mx = fmaxf(mx, absmax8(xr[m * k8 + q]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) {
            sigw[m] = prescale_exponent(mx);
            if (warp == 0) sig[m] = sigw[m];
        }
    }
    __syncwarp();
    const int slots = 4 * M;
    for (int it = warp * 32 + lane; it < M * p8; it += kCT) {
        const int m = it / p8, q = it - m * p8;
        stage_store8(xs, slots, m, q * 8, sigw[m], q < k8 ? xr[m * k8 + q] : make_uint4(0, 0, 0, 0));
    }
    named_bar_sync(1, kCT);
}

// One token's x (K raw bf16 values in shared memory) -> prescaled fp16
// fragments in xs with two barriers over the consumer threads: each warp
// writes its max|x| to its own word (no shared initialisation, no atomics),
// then every thread folds the kW words itself (max is order-independent, so
// every thread finds the same exponent) and converts its items (8 values
// each; k in [K, kpe) is zero). Thread 0 also writes sig[0] for the
// epilogue. Needs kpe / 8 <= REGS * kCT. (Written for one token: no index
// division, one fold per thread -- this runs once per call and its
// instruction count is on the critical path.)
template <int REGS>
QMLP_DEV void stage_x_one_token(const uint4* xr, int K, int kpe, uint4* xs, float* wmax, int* sig) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k8 = K / 8, p8 = kpe / 8;
    uint4 v[REGS];
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < REGS; ++i) {
        const int it = tid + i * kCT;
        v[i] = it < k8 ? xr[it] : make_uint4(0, 0, 0, 0);
        mx = fmaxf(mx, absmax8(v[i]));
    }
    // one warp reduction: mx is a non-negative float (fmaxf drops NaN), so
    // its bits order as unsigned integers
    mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
    if (lane == 0) wmax[warp] = mx;
    named_bar_sync(1, kCT);
    mx = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) mx = fmaxf(mx, wmax[w]);
    const int sg = prescale_exponent(mx);
#pragma unroll
    for (int i = 0; i < REGS; ++i) {
        const int it = tid + i * kCT;
        if (it < p8) stage_store8(xs, 4, 0, it * 8, sg, v[i]);
    }
    if (tid == 0) sig[0] = sg;
    named_bar_sync(1, kCT);
}

// 9..16 tokens (see halves_ok): x of pass `pass` as prescaled fp16
// fragments at half-local chunk positions. Chunk position cp < Kc/2 holds
// global chunk (cp % q) + (cp / q) * (Kc/2) + pass * q, q = Kc/4 (the same
// map as half_slot). With find_sig, the per-token exponents are found first
// from all of x (warp m takes token m; M <= kW). Ends with a barrier over the
// consumer threads. Loads go out eight per thread at a time.
// Chunk c (0 <= c < 4q, q = Kc/4) -> its half-local position c mod q + q
// [c >= 2q], with compares: the streaming loop evaluates it per record, and
// a division by the runtime q there cost ~10 instructions per weight group.
QMLP_DEV int half_slot(int c, int q) {
    const bool hi = c >= 2 * q;
    const int cc = hi ? c - 2 * q : c;
    return (cc >= q ? cc - q : cc) + (hi ? q : 0);
}

QMLP_DEV void stage_x_half(const __nv_bfloat16* x, int M, int K, int pass, bool find_sig, uint4* xs, int* s_sig,
                           int warp) {
    const int lane = threadIdx.x & 31;
    const int kca = K / kChunkK, q = kca / 4, h = kca / 2, k8 = K / 8;
    if (find_sig) {
        if (warp < M) {
            const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)warp * K);
            float mx = 0.0f;
#pragma unroll 8
            for (int i = lane; i < k8; i += 32) mx = fmaxf(mx, absmax8(__ldcg(xr + i)));
            mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
            if (lane == 0) s_sig[warp] = prescale_exponent(mx);
        }
        named_bar_sync(1, kCT);
    }
    // item it = (token m, r < per_tok): kept incrementally from one division
    // per 8 items (it advances by kCT, r wraps a few times at most); the
    // chunk position cp < h maps to chunk cp + pass q, plus q for cp >= q
    const int slots = 4 * M, per_tok = h * 8, total = M * per_tok;
    for (int base = threadIdx.x; base < total; base += 8 * kCT) {
        uint4 v[8];
        int mu[8], ru[8];
        int m = base / per_tok, r = base - m * per_tok;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            mu[u] = m;
            ru[u] = r;
            v[u] = make_uint4(0, 0, 0, 0);
            if (base + u * kCT < total) {
                const int cp = r >> 3, e8 = r & 7;
                const int c = cp + pass * q + (cp >= q ? h - q : 0);
                if (QMLP_INB((size_t)m * K + c * kChunkK + e8 * 8 + 7, (size_t)M * K, 8))
                    v[u] = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)m * K + c * kChunkK + e8 * 8));
            }
            r += kCT;
            while (r >= per_tok) {
                r -= per_tok;
                ++m;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (base + u * kCT < total)
                stage_store8(xs, slots, mu[u], (ru[u] >> 3) * kChunkK + (ru[u] & 7) * 8, s_sig[mu[u]], v[u]);
    }
    named_bar_sync(1, kCT);
}

// Phase B when the CTA's slice is CB = 1, 2 or 4 down chunks: every warp's
// range starts on a row-tile boundary (LB is a multiple of 4), a step's 4
// records are 4/CB whole tiles, and the CB activation fragments are the same
// for every record, so they are loaded once and stay in registers. Records
// past the CTA's real ones are zero and their tiles are not stored.
template <int FMT, int NT, bool M1, int CB>
QMLP_DEV bool phase_b_fixed(const Args& a, const Ring& r, int q, int steps, const uint4* xs, const int* s_sigb,
                            int M, int warp) {
    constexpr int rec = rec_bytes<FMT>();
    constexpr int R = gemv_recs_single(FMT);
    static_assert(R % CB == 0, "whole tiles per step");
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    uint4 xb[CB][NT][2];
#pragma unroll
    for (int c = 0; c < CB; ++c) load_xfrag<NT>(xs, c, M, 4 * M, g, t, xb[c]);
    int rt = warp * a.LB / CB;
    int slot = q % r.depth;
    uint32_t parity = (uint32_t)((q / r.depth) & 1);
    for (int j = 0; j < steps; ++j) {
        if (!mbar_wait_bounded(r.full0 + 8u * slot, parity, a.limit)) {
            if (lane == 0) atomicExch(a.err, 22);
            return false;
        }
        const uint8_t* sb = r.base + (uint32_t)slot * (uint32_t)r.slot_bytes + (uint32_t)warp * R * rec;
#pragma unroll
        for (int tt = 0; tt < R / CB; ++tt, ++rt) {
            float acc[1][NT][4];
            zero_acc<NT, 1>(acc);
#pragma unroll
            for (int c = 0; c < CB; ++c) {
                ChunkW w[1];
                w[0] = lds_chunk<FMT>(sb + (tt * CB + c) * rec, lane);
                mma_chunk<FMT, NT, 1, M1>(w, xb[c], acc);
            }
            if (rt < a.NtD) store_part_b<NT>(a, M, rt, acc, s_sigb);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(r.empty0 + 8u * slot);
        if (++slot == r.depth) {
            slot = 0;
            parity ^= 1u;
        }
    }
    return true;
}

template <int NT, int NP>
QMLP_DEV void zero_acc(float (&acc)[NP][NT][4]) {
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[p][n][e] = 0.0f;
}

QMLP_DEV unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// MC: the token count when the instance fixes it (1, 2, 4, 8), else 0 (the
// count is a.M). A fixed count folds the token loops and the x-fragment
// addressing of the streaming loop (measured at 4 tokens: 45.6 -> 43.7 us).
template <int FMT, int NT, int MC, bool SEP>
__global__ void __launch_bounds__(kThr, 1) gemv_split_kernel(const __grid_constant__ Args a) {
    constexpr bool M1 = MC == 1;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_maxbits[16];
    __shared__ int s_sig[16];
    __shared__ int s_sigb[16];
    __shared__ int s_cnta[64];
    __shared__ int s_actmax[16];  // per token: max|act| bits over the CTA's slice
    __shared__ int s_cntb[kW];
    __shared__ int s_sigw[kW][16];
    __shared__ float s_wmax[kW];
    __shared__ int s_fail;
    __shared__ int s_pass;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = MC ? MC : a.M;
    Ring r;
    r.base = smem + a.ring_off;
    r.base_s = smem_u32(r.base);
    r.slot_bytes = a.slot_bytes;
    r.depth = a.depth;
    r.limit = a.limit;
    r.full0 = smem_u32(r.base + (size_t)a.depth * a.slot_bytes);
    r.empty0 = r.full0 + 8u * kDepthMax;
    r.xbar = r.empty0 + 8u * kDepthMax;
    constexpr int kRA = gemv_recs_pair(FMT), kRB = gemv_recs_single(FMT);
    const int stepsA = a.LA / kRA, stepsB = a.LB / kRB;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.depth; ++i) {
            mbar_init(r.full0 + 8u * i, 1);
            mbar_init(r.empty0 + 8u * i, kW);
        }
        mbar_init(r.xbar, 1);
        fence_mbar_init();
        s_fail = 0;
    }
    if (threadIdx.x < 64) s_cnta[threadIdx.x] = 0;
    if (threadIdx.x < 16) s_actmax[threadIdx.x] = 0;
    if (threadIdx.x < kW) s_cntb[threadIdx.x] = 0;
    __syncthreads();  // the last CTA-wide barrier: the producer never waits on the consumers
    // the next kernel's CTAs may start as SMs free up (set-up and launch
    // latency overlap this call's end); they wait before touching its buffers
    pdl_launch_dependents();

    if (warp == kW) {
        if (lane == 0) {
            Steps st;
            const uint32_t rec = rec_bytes<FMT>();
            st.bytes_a = kW * kRA * rec;
            st.bytes_b = kW * kRB * rec;
            st.stride_a = (size_t)a.G * st.bytes_a;
            st.stride_b = (size_t)a.G * st.bytes_b;
            st.a0 = a.wa0 + (size_t)blockIdx.x * st.bytes_a;
            st.a1 = a.wa1 + (size_t)blockIdx.x * st.bytes_a;
            st.b = a.wb + (size_t)blockIdx.x * st.bytes_b;
            st.steps_a = stepsA;
            st.steps = stepsA + stepsB - (a.withhold ? 1 : 0);
            st.off_a = (size_t)blockIdx.x * st.bytes_a;
            st.off_b = (size_t)blockIdx.x * st.bytes_b;
            st.lim_a = a.wa_bytes;
            st.lim_b = a.wb_bytes;
            st.base_a0 = a.wa0;
            st.base_a1 = a.wa1;
            st.base_b = a.wb;
            // The weights do not depend on the previous kernel: the first
            // kPreSteps steps go out before the wait, x right after it, then
            // the rest of the weights. (Measured back to back: one step
            // gains 0.1-0.5 us; two or more delay the x copy behind them.)
            const int pre = min(min(SEP ? kPreStepsSep : kPreStepsBarrier, a.depth), st.steps);
            produce<FMT>(st, r, a.err, 0, pre);
            pdl_wait();
            if (a.xraw_bytes) {
                if (QMLP_INB(a.xraw_bytes - 1, (size_t)a.M * a.K * 2, 3)) {
                    mbar_arrive_expect_tx(r.xbar, a.xraw_bytes);
                    bulk_g2s(smem_u32(smem + a.xraw_off), a.x, a.xraw_bytes, r.xbar);
                } else {
                    mbar_arrive(r.xbar);  // no copy: the barrier still completes
                }
            }
            int q = produce<FMT>(st, r, a.err, pre, st.steps);
            if (a.xraw_bytes) mbar_wait_bounded(r.xbar, 0, kLimit);  // the x copy is never left in flight
            if (q < 0) {
                const int issued = -q - 1;
                for (int qq = issued - 1; qq >= 0 && qq >= issued - a.depth; --qq)
                    mbar_wait_bounded(r.full0 + 8u * (qq % a.depth), (uint32_t)((qq / a.depth) & 1), kLimit);
            }
        }
        return;
    }

    constexpr int rec = rec_bytes<FMT>();
    uint4* xs = reinterpret_cast<uint4*>(smem);
    float* s_pa = reinterpret_cast<float*>(smem + a.pa_off);
    float* s_act = reinterpret_cast<float*>(smem + a.act_off);
    float* s_pb = reinterpret_cast<float*>(smem + a.pb_off);
    const int g = lane >> 2, t = lane & 3;
    bool ok = true;

    // x, act, the partials and the output belong to the previous kernel until
    // it has completed
    pdl_wait();

    // ---------------- phase A: gate/up over this CTA's tiles ----------------
    if (NT == 2) {
        stage_x_half(a.x, M, a.K, 0, true, xs, s_sig, warp);
    } else if (a.xraw_bytes) {
        if (!mbar_wait_bounded(r.xbar, 0, a.limit)) {
            if (lane == 0) atomicExch(a.err, 25);
            ok = false;
        }
        // (after a failed wait x reads as whatever is there; the error word
        // reports the call)
        // one token: warp maxima, two barriers; several: every warp finds
        // the maxima itself and only one barrier remains (measured: 33.4 vs
        // 34.4 us at M=1, 53.2 vs 50.6 us at M=4)
        // a one-token x in shared memory has at most kXRawMax / 2 columns
        // (padded to a chunk: still <= 2 items of 8 per consumer thread)
        static_assert(kXRawMax / 16 <= 2 * kCT && kXRawMax % (2 * kChunkK) == 0, "one-token staging: 2 items");
        if (M1)
            stage_x_one_token<2>(reinterpret_cast<const uint4*>(smem + a.xraw_off), a.K, a.KcA * kChunkK, xs,
                                 s_wmax, s_sig);
        else
            stage_x_local(reinterpret_cast<const uint4*>(smem + a.xraw_off), M, a.K, a.KcA * kChunkK, xs,
                          s_sigw[warp], s_sig, warp);
    } else if (M1 && a.KcA * kChunkK <= 16 * kCT) {
        // one token read in place (host-mapped memory): the same compact
        // staging, its loads in flight together
        stage_x_one_token<2>(reinterpret_cast<const uint4*>(a.x), a.K, a.KcA * kChunkK, xs, s_wmax, s_sig);
    } else {
        stage_x(a.x, M, a.K, 0, a.K, a.KcA * kChunkK, xs, s_maxbits, s_sig, kCT);
    }
    int q = 0;
    {
        const int slots = 4 * M;
        const int pa_floats = 2 * M * 16;
        const uint32_t step_bytes = (uint32_t)kW * kRA * rec;
        float acc[2][NT][4];
        zero_acc<NT, 2>(acc);
        const int u0 = warp * a.LA;  // local record index of this warp's first record
        int lt = u0 / a.KcA, c = u0 % a.KcA, cs = c;
        const int qc = a.KcA / 4;    // 9..16 tokens: the x halves' quarter of Kc
        int slot = 0;
        uint32_t parity = 0;
        int k = 0;
        // 9..16 tokens: the warp's one tile part is combined after the loop
        // (its slots alias the x halves); a warp whose wait gave up still
        // reaches both barriers below
        AccA<NT> pend;
        int pend_lt = -1, pend_whole = 0;
        for (int j = 0; j < stepsA && (ok || NT == 2); ++j) {
            if (NT == 2 && j == stepsA / 2) {
                named_bar_sync(1, kCT);  // every warp is done with the first half of x
                stage_x_half(a.x, M, a.K, 1, false, xs, s_sig, warp);
            }
            if (!ok) continue;
            if (!mbar_wait_bounded(r.full0 + 8u * slot, parity, a.limit)) {
                if (lane == 0) atomicExch(a.err, 21);
                ok = false;
                if (NT == 2) continue;
                break;
            }
            const uint8_t* sb = r.base + (uint32_t)slot * (uint32_t)r.slot_bytes + (uint32_t)warp * kRA * rec;
            for (int kk = 0; kk < kRA; ++kk, ++k, sb += rec) {
                ChunkW w[2];
                w[0] = lds_chunk<FMT>(sb, lane);
                w[1] = lds_chunk<FMT>(sb + step_bytes, lane);
                uint4 xb[NT][2];
                load_xfrag<NT>(xs, NT == 2 ? half_slot(c, qc) : c, M, slots, g, t, xb);
                mma_chunk<FMT, NT, 2, M1>(w, xb, acc);
                if (++c == a.KcA || k == a.LA - 1) {
                    AccA<NT> av;
#pragma unroll
                    for (int p = 0; p < 2; ++p)
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) av.v[p][n][e] = acc[p][n][e];
                    if (NT == 2) {
                        pend = av;
                        pend_lt = lt;
                        pend_whole = cs == 0 && c == a.KcA;
                    } else {
                        finish_tile_a<FMT, NT>(a, M, lt, cs == 0 && c == a.KcA, warp, av, s_pa, pa_floats, s_cnta,
                                               s_sig, s_act, s_actmax);
                    }
                    zero_acc<NT, 2>(acc);
                    ++lt;
                    c = 0;
                    cs = 0;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(r.empty0 + 8u * slot);
            if (++slot == r.depth) {
                slot = 0;
                parity ^= 1u;
            }
        }
        if (NT == 2) {
            named_bar_sync(1, kCT);  // x is no longer read: its region takes the combine slots
            if (pend_lt >= 0)
                finish_tile_a<FMT, NT>(a, M, pend_lt, pend_whole != 0, warp, pend, s_pa, pa_floats, s_cnta, s_sig,
                                       s_act, s_actmax);
        }
        q = stepsA;
    }
    if (!ok && lane == 0) s_fail = 1;
    named_bar_sync(1, kCT);  // the CTA's act slice is complete

    // ---------------- restage act (prescaled fp16 fragments) ----------------
    const int tslice = a.T * 16;
    if (s_fail == 0) {
        // the slice maxima were kept by the epilogues: the items (8 act
        // values each) convert straight away; one barrier
        if (threadIdx.x < M) s_sigb[threadIdx.x] = prescale_exponent(__int_as_float(s_actmax[threadIdx.x]));
        const int slots = 4 * M;
        for (int it = threadIdx.x; it < M * (tslice / 8); it += kCT) {
            const int m = it / (tslice / 8), k8 = (it % (tslice / 8)) * 8;
            const float* src = s_act + m * tslice + k8;
            uint4 v;
            uint32_t* vw = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(src[2 * h], src[2 * h + 1]);  // exact: bf16 values
                vw[h] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            stage_store8(xs, slots, m, k8, prescale_exponent(__int_as_float(s_actmax[m])), v);
        }
        named_bar_sync(1, kCT);
    }

    // ---------------- phase B: down over this CTA's act slice ----------------
    constexpr int kCB4 = kRB % 4 == 0 ? 4 : 1;  // CB = 4 has a fixed path when a step holds whole tiles
    if (s_fail == 0 && (a.Cb == 1 || a.Cb == 2 || (a.Cb == 4 && kRB % 4 == 0))) {
        ok = a.Cb == 1   ? phase_b_fixed<FMT, NT, M1, 1>(a, r, q, stepsB, xs, s_sigb, M, warp)
             : a.Cb == 2 ? phase_b_fixed<FMT, NT, M1, 2>(a, r, q, stepsB, xs, s_sigb, M, warp)
                         : phase_b_fixed<FMT, NT, M1, kCB4>(a, r, q, stepsB, xs, s_sigb, M, warp);
    } else if (s_fail == 0) {
        const int slots = 4 * M;
        const int pb_floats = M * 16;
        float acc[1][NT][4];
        zero_acc<NT, 1>(acc);
        const int nrec = a.NtD * a.Cb;          // real records of the CTA
        const int u0 = warp * a.LB;
        const int n = max(0, min(a.LB, nrec - u0));  // real records of this warp
        int rt = u0 / a.Cb, c = u0 % a.Cb, cs = c;
        int slot = q % r.depth;
        uint32_t parity = (uint32_t)((q / r.depth) & 1);
        int k = 0;
        for (int j = 0; j < stepsB && ok; ++j) {
            if (!mbar_wait_bounded(r.full0 + 8u * slot, parity, a.limit)) {
                if (lane == 0) atomicExch(a.err, 22);
                ok = false;
                break;
            }
            const uint8_t* sb = r.base + (uint32_t)slot * (uint32_t)r.slot_bytes +
                                (uint32_t)warp * kRB * rec;
            const int kend = min(k + kRB, n);
            for (; k < kend; ++k, sb += rec) {
                ChunkW w[1];
                w[0] = lds_chunk<FMT>(sb, lane);
                uint4 xb[NT][2];
                load_xfrag<NT>(xs, c, M, slots, g, t, xb);
                mma_chunk<FMT, NT, 1, M1>(w, xb, acc);
                if (++c == a.Cb || k == n - 1) {
                    if (cs == 0 && c == a.Cb) {
                        store_part_b<NT>(a, M, rt, acc, s_sigb);
                    } else {
                        // a tile split at a warp boundary: two contributors
                        const int wb = (cs == 0) ? warp : warp - 1;  // boundary after warp wb
                        if (combine_smem<NT, 1>(s_pb + (size_t)wb * 2 * pb_floats, pb_floats, cs == 0 ? 0 : 1, 2,
                                                &s_cntb[wb], M, acc))
                            store_part_b<NT>(a, M, rt, acc, s_sigb);
                    }
                    zero_acc<NT, 1>(acc);
                    ++rt;
                    c = 0;
                    cs = 0;
                }
            }
            k = max(k, (j + 1) * kRB);
            __syncwarp();
            if (lane == 0) mbar_arrive(r.empty0 + 8u * slot);
            if (++slot == r.depth) {
                slot = 0;
                parity ^= 1u;
            }
        }
    }
    if (!ok && lane == 0) s_fail = 1;
    // schedule (b): the partials are written (a failed wait is in the error
    // word); the reduce kernel waits for this grid
    if (SEP) return;

    // ---------------- grid barrier (every CTA arrives exactly once) ----------------
    // The CTA barrier orders every consumer thread's partial stores before
    // thread 0's release add (cumulative), and thread 0's acquire poll before
    // the CTA barrier that precedes the reads of the other CTAs' partials.
    named_bar_sync(1, kCT);
    if (threadIdx.x == 0) {
        unsigned long long tk;
        asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(tk) : "l"(a.ticket) : "memory");
        const unsigned long long target = (tk / (unsigned long long)a.G + 1ull) * (unsigned long long)a.G;
        int pass = 1;
        if (tk + 1ull != target) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_u64(a.ticket) < target) {
                if (globaltimer_ns() - t0 > a.limit) {
                    atomicExch(a.err, 23);
                    pass = 0;
                    break;
                }
            }
        }
        s_pass = pass;
    }
    named_bar_sync(1, kCT);
    if (s_pass == 0) return;
    // a CTA that failed still reduces: every partial it could not write is
    // reported through the error word, and outputs are never left unwritten

    // ---------------- reduction over the G partials ----------------
    // The CTA's units (token m, 32 output columns): every warp adds its
    // share of the partials of all of them first (the loads of all units in
    // flight together), one barrier, then a warp per unit adds the 16 warp
    // sums in order. Scratch: the weight ring, idle after phase B (every
    // step issued was consumed, so no copy is in flight).
    const int units_n = (a.K + 31) / 32;
    const int units = M * units_n;
    float* red = reinterpret_cast<float*>(r.base);
    const size_t bstride = (size_t)M * a.K;
    int nu = 0;
    // two units per round; every load of a round is issued before the adds
    // (in the same fixed order), so a round costs one L2 round trip
    for (int u0 = blockIdx.x; u0 < units; u0 += 2 * gridDim.x) {
        const int u1 = u0 + gridDim.x;
        const int n0 = (u0 % units_n) * 32 + lane, n1 = (u1 % units_n) * 32 + lane;
        const bool ok0 = n0 < a.K, ok1 = u1 < units && n1 < a.K;
        const float* src0 = a.part + (size_t)(u0 / units_n) * a.K + n0;
        const float* src1 = a.part + (size_t)(u1 / units_n) * a.K + n1;
        float v0[kRedLoads], v1[kRedLoads];
#pragma unroll
        for (int i = 0; i < kRedLoads; ++i) {
            const int b = warp + i * kW;
            v0[i] = (ok0 && b < a.G &&
                     QMLP_INB((size_t)(u0 / units_n) * a.K + n0 + (size_t)b * bstride, a.part_elems, 6))
                        ? __ldcg(src0 + (size_t)b * bstride)
                        : 0.0f;
            v1[i] = (ok1 && b < a.G &&
                     QMLP_INB((size_t)(u1 / units_n) * a.K + n1 + (size_t)b * bstride, a.part_elems, 6))
                        ? __ldcg(src1 + (size_t)b * bstride)
                        : 0.0f;
        }
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int i = 0; i < kRedLoads; ++i) {
            s0 += v0[i];
            s1 += v1[i];
        }
        red[(nu * kW + warp) * 32 + lane] = s0;
        ++nu;
        if (u1 < units) {
            red[(nu * kW + warp) * 32 + lane] = s1;
            ++nu;
        }
    }
    named_bar_sync(1, kCT);
    for (int i = warp; i < nu; i += kW) {
        const int u = blockIdx.x + i * gridDim.x;
        const int m = u / units_n, n = (u % units_n) * 32 + lane;
        if (n < a.K && QMLP_INB((size_t)m * a.K + n, (size_t)a.M * a.K, 6)) {
            float tot = 0.0f;
#pragma unroll
            for (int w = 0; w < kW; ++w) tot += red[(i * kW + w) * 32 + lane];
            if (a.out_f32) {
                a.out_f32[(size_t)m * a.K + n] = tot;
            } else {
                const float sd = FMT == kNVFP4 ? a.invd : a.chsd[n];
                a.out[(size_t)m * a.K + n] = __float2bfloat16_rn(tot * sd);
            }
        }
    }
}

// ---------------- schedule (b): reduction over the G partials ----------------
// One CTA per output unit (token m, 32 columns): warp w adds the partials
// b = w, w + 8, ... (every load of a lane in flight together), then warp 0
// adds the 8 warp sums in order and applies the down scale: a fixed order.
// Small (256 threads, few registers, 1 KB of shared memory), so it sits
// beside a streaming CTA of the next call on the same SM.
constexpr int kRedThr = 256;
constexpr int kRedWarps = kRedThr / 32;
constexpr int kRedPer = 20;  // partials per lane: G <= kRedWarps * kRedPer
// <= 48 registers a thread: 8 warps x 48 x 32 beside a streaming CTA's
// 17 warps x 96 x 32 stay within the SM's 65536 registers
constexpr int kRedMinBlocks = 5;
static_assert(kW * kRedLoads <= kRedWarps * kRedPer, "every planned G is reducible");

struct RArgs {
    size_t part_elems;  // index checks: floats of the partial buffer
    const float* part;  // [G][M][K]
    const float* chsd;  // FP8 down per-channel scales
    float invd;         // NVFP4 down 1/global
    __nv_bfloat16* out; // [M, K]
    float* out_f32;     // optional [M, K]: fp32 sums without the factor, instead of out
    int G, M, K;
};

template <int FMT>
__global__ void __launch_bounds__(kRedThr, kRedMinBlocks) gemv_split_reduce_kernel(const __grid_constant__ RArgs a) {
    __shared__ float red[kRedWarps][32];
    // the next kernel may start (its streaming CTAs fill their rings) ...
    pdl_launch_dependents();
    // ... while this one waits for every partial of the streaming grid
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units_n = (a.K + 31) / 32, units = a.M * units_n;
    const size_t bstride = (size_t)a.M * a.K;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int m = u / units_n, n = (u % units_n) * 32 + lane;
        const float* src = a.part + (size_t)m * a.K + n;
        float v[kRedPer];
#pragma unroll
        for (int i = 0; i < kRedPer; ++i) {
            const int b = warp + i * kRedWarps;
            v[i] = (n < a.K && b < a.G && QMLP_INB((size_t)m * a.K + n + (size_t)b * bstride, a.part_elems, 7))
                       ? __ldcg(src + (size_t)b * bstride)
                       : 0.0f;
        }
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < kRedPer; ++i) s += v[i];
        red[warp][lane] = s;
        __syncthreads();
        if (warp == 0 && n < a.K && QMLP_INB((size_t)m * a.K + n, (size_t)a.M * a.K, 7)) {
            float tot = 0.0f;
#pragma unroll
            for (int w = 0; w < kRedWarps; ++w) tot += red[w][lane];
            if (a.out_f32) {
                a.out_f32[(size_t)m * a.K + n] = tot;
            } else {
                const float sd = FMT == kNVFP4 ? a.invd : a.chsd[n];
                a.out[(size_t)m * a.K + n] = __float2bfloat16_rn(tot * sd);
            }
        }
        __syncthreads();
    }
}

template <int FMT, int NT, int MC, bool SEP>
cudaError_t launch_t(const Args& a, size_t smem, cudaStream_t s) {
    auto kern = gemv_split_kernel<FMT, NT, MC, SEP>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBudget);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.G);
    cfg.blockDim = dim3(kThr);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // Programmatic dependent launch instead of a cooperative one: a CTA can
    // start (and stream weights) while the previous kernel still holds SMs.
    // All G CTAs are co-resident once it has finished (one CTA per SM, G <=
    // SMs, checked at create); the grid barrier's wait is bounded regardless.
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Schedule (b) with one 8-token column tile: instances with the token count
// fixed for 2, 4 and 8 tokens (and 1 for FP8; NVFP4 at one token takes
// schedule (a)), the general one otherwise.
template <int FMT>
cudaError_t launch_one_tile(const Args& a, size_t smem, int M, cudaStream_t s) {
    if constexpr (FMT == kFP8)
        if (M == 1) return launch_t<FMT, 1, 1, true>(a, smem, s);
    switch (M) {
        case 2: return launch_t<FMT, 1, 2, true>(a, smem, s);
        case 4: return launch_t<FMT, 1, 4, true>(a, smem, s);
        case 8: return launch_t<FMT, 1, 8, true>(a, smem, s);
        default: return launch_t<FMT, 1, 0, true>(a, smem, s);
    }
}

struct Layout {
    int xs, pa, act, pb, xraw, xraw_bytes, ring, slot, depth, sa;
    size_t total;
};

// 9..16 tokens (two 8-token MMA column tiles): x for all of K no longer
// fits beside the ring, so phase A stages it in two halves. This works when
// every gate/up tile is split between exactly two warps at K/2 (LA = Kc/2):
// the first half of the steps then touches only the chunks [0, Kc/4) and
// [Kc/2, 3Kc/4) of every tile, the second half the other two quarters.
bool halves_ok(int fmt, int K, const SplitPlan& P) {
    const int kca = (K + kChunkK - 1) / kChunkK;
    return P.G && K % kChunkK == 0 && kca % 4 == 0 && P.LA * 2 == kca && (P.LA / gemv_recs_pair(fmt)) % 2 == 0;
}

Layout layout_for(int fmt, int M, int K, const SplitPlan& P) {
    Layout L;
    const int kca = (K + kChunkK - 1) / kChunkK;
    const int rec = fmt == kNVFP4 ? kRecNVFP4 : kRecFP8;
    auto al = [](size_t v) { return (int)((v + 127) & ~(size_t)127); };
    L.sa = P.SA;
    if (M > 8) {
        // half of x; the tile combine slots alias it (used only once every
        // warp has finished phase A)
        L.xs = al(std::max((size_t)std::max(kca / 2, P.Cb) * 128 * M, (size_t)P.T * L.sa * 2 * M * 16 * 4));
        L.pa = 0;
        L.act = L.xs;
    } else {
        L.xs = al((size_t)std::max(kca, P.Cb) * 128 * M);
        L.pa = L.xs;
        L.act = L.pa + al((size_t)P.T * L.sa * 2 * M * 16 * 4);
    }
    L.pb = L.act + al((size_t)M * P.T * 16 * 4);
    // split down tiles (two contributors per warp boundary) only on the
    // generic down path: Cb not 1, 2 or 4, or a step not whole tiles
    const int rb = gemv_recs_single(fmt);
    const bool fixed_b = (P.Cb == 1 || P.Cb == 2 || P.Cb == 4) && rb % P.Cb == 0;
    L.xraw = L.pb + (fixed_b ? 0 : al((size_t)kW * 2 * M * 16 * 4));
    L.xraw_bytes = (size_t)M * K * 2 <= (size_t)kXRawMax ? M * K * 2 : 0;
    L.ring = L.xraw + al((size_t)L.xraw_bytes);
    L.slot = std::max(2 * kW * gemv_recs_pair(fmt) * rec, kW * rb * rec);
    const long avail = (long)kBudget - L.ring - kBars - 1024;
    L.depth = avail > 0 ? (int)std::min<long>(kDepthMax, avail / L.slot) : 0;
    L.total = (size_t)L.ring + (size_t)L.depth * L.slot + kBars;
    return L;
}

}  // namespace

SplitPlan plan_split(int fmt, int K, int I, int num_sms) {
    SplitPlan P;
    if (K % 16 || I % 16 || num_sms < 1) return P;
    const int ra = gemv_recs_pair(fmt), rb = gemv_recs_single(fmt);
    const int nta = I / 16, kca = (K + kChunkK - 1) / kChunkK, ntd = K / 16;
    // a small MLP (every CTA streams at most kSmallCtaBytes) is bound by
    // fixed costs, not bandwidth: a few CTAs serve it
    const double wbytes = (double)3 * K * I * (fmt == kNVFP4 ? 9.0 / 16.0 : 1.0);
    for (int T = 4; T <= nta; T += 4) {
        if (nta % T) continue;
        const int G = nta / T;
        if (G > num_sms || G > kW * kRedLoads) continue;
        const bool small = wbytes / G <= kSmallCtaBytes;
        // the smallest T with G <= SMs: the most CTAs; too few CTAs cannot
        // pull the bandwidth (each SM's consumers decode ~1.4x the HBM rate)
        if (4 * G < 3 * num_sms && !small) return P;
        if ((T * kca) % (16 * ra) != 0) {  // gate/up: whole steps, no padding
            if (small) continue;
            return P;
        }
        if (ntd < 16 || T > 64) return P;
        P.G = G;
        P.T = T;
        P.Cb = T / 4;
        P.LA = T * kca / 16;
        const int lb = (ntd * P.Cb + 15) / 16;
        P.LB = (lb + rb - 1) / rb * rb;
        P.RA = ra;
        P.RB = rb;
        P.SA = 1;
        for (int lt = 0; lt < T; ++lt)
            P.SA = std::max(P.SA, ((lt + 1) * kca - 1) / P.LA - (lt * kca) / P.LA + 1);
        return P;
    }
    return P;
}

bool split_fits(int fmt, int M, int K, const SplitPlan& P) {
    if (!P.G || M < 1 || M > 16 || (M > 8 && !halves_ok(fmt, K, P))) return false;
    const Layout L = layout_for(fmt, M, K, P);
    // the in-kernel reduction's scratch (units per CTA x 16 warps x 32
    // floats) lives in the ring
    const size_t units = (size_t)M * ((K + 31) / 32);
    const size_t per_cta = (units + P.G - 1) / P.G;
    return L.depth >= 2 && per_cta * kW * 32 * 4 <= (size_t)L.depth * L.slot;
}

size_t split_part_elems(int K, const SplitPlan& P) { return (size_t)P.G * 16 * K; }

size_t split_codes_bytes(int fmt, const SplitPlan& P) {
    return (size_t)P.G * kW * P.LB * (fmt == kNVFP4 ? kRecNVFP4 : kRecFP8);
}

cudaError_t launch_split(const SplitLaunch& L, const SplitPlan& P, cudaStream_t s) {
    if (!split_fits(L.fmt, L.M, L.K, P)) return cudaErrorInvalidValue;
    if (L.gate.TWr != P.G * kW || L.gate.Lr != P.LA || L.gate.Rr != P.RA || L.up.TWr != P.G * kW ||
        P.RA != gemv_recs_pair(L.fmt) || P.RB != gemv_recs_single(L.fmt))
        return cudaErrorInvalidValue;
    const Layout lay = layout_for(L.fmt, L.M, L.K, P);
    if (P.T > 64) return cudaErrorInvalidValue;
    Args a;
    a.wa0 = L.gate.wc;
    a.wa1 = L.up.wc;
    a.chs0 = L.gate.chs;
    a.chs1 = L.up.chs;
    a.inv0 = L.gate.inv_g;
    a.inv1 = L.up.inv_g;
    a.wb = L.wdown;
    a.chsd = L.chsd;
    a.invd = L.invd;
    a.x = static_cast<const __nv_bfloat16*>(L.x);
    a.act_out = static_cast<__nv_bfloat16*>(L.act_out);
    a.out = static_cast<__nv_bfloat16*>(L.out);
    a.out_f32 = L.out_f32;
    a.act_in = static_cast<const __nv_bfloat16*>(L.act_in);
    a.dbg_g = L.dbg_g;
    a.dbg_u = L.dbg_u;
    a.part = L.part;
    a.ticket = L.ticket;
    a.err = L.err;
    a.M = L.M;
    a.K = L.K;
    a.I = L.I;
    a.G = P.G;
    a.T = P.T;
    a.KcA = (L.K + kChunkK - 1) / kChunkK;
    a.LA = P.LA;
    a.Cb = P.Cb;
    a.NtD = L.K / 16;
    a.LB = P.LB;
    a.xs_bytes = lay.xs;
    a.pa_off = lay.pa;
    a.act_off = lay.act;
    a.pb_off = lay.pb;
    a.ring_off = lay.ring;
    a.slot_bytes = lay.slot;
    a.depth = lay.depth;
    a.SA = lay.sa;
    a.xraw_off = lay.xraw;
    a.limit = L.wait_ns ? L.wait_ns : kLimit;
    a.withhold = L.withhold ? 1 : 0;
    const size_t rec = L.fmt == kNVFP4 ? kRecNVFP4 : kRecFP8;
    a.wa_bytes = L.lim_a ? L.lim_a : (size_t)P.G * kW * P.LA * rec;
    a.wb_bytes = split_codes_bytes(L.fmt, P);
    a.part_elems = split_part_elems(L.K, P);
    // the bulk copy of x needs device memory; host-resident x is staged by loads
    a.xraw_bytes = L.x_in_host ? 0 : lay.xraw_bytes;
    // M <= 8 (split_fits): one 8-token MMA tile. Schedule (a) for NVFP4 at
    // one token, (b) otherwise (see the top of the file).
    if (L.fmt == kNVFP4 && L.M == 1) return launch_t<kNVFP4, 1, 1, false>(a, lay.total, s);
    // 9..16 tokens: two 8-token column tiles, x staged in halves
    cudaError_t e = L.M > 8 ? (L.fmt == kNVFP4 ? launch_t<kNVFP4, 2, 0, true>(a, lay.total, s)
                                                : launch_t<kFP8, 2, 0, true>(a, lay.total, s))
                            : (L.fmt == kNVFP4 ? launch_one_tile<kNVFP4>(a, lay.total, L.M, s)
                                                : launch_one_tile<kFP8>(a, lay.total, L.M, s));
    if (e != cudaSuccess) return e;
    RArgs r;
    r.part_elems = a.part_elems;
    r.part = L.part;
    r.chsd = L.chsd;
    r.invd = L.invd;
    r.out = static_cast<__nv_bfloat16*>(L.out);
    r.out_f32 = L.out_f32;
    r.G = P.G;
    r.M = L.M;
    r.K = L.K;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(L.M * ((L.K + 31) / 32)));
    cfg.blockDim = dim3(kRedThr);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return L.fmt == kNVFP4 ? cudaLaunchKernelEx(&cfg, gemv_split_reduce_kernel<kNVFP4>, r)
                           : cudaLaunchKernelEx(&cfg, gemv_split_reduce_kernel<kFP8>, r);
}

QMLP_BOUNDS_UNIT(gemv_split)

}  // namespace qmlp
