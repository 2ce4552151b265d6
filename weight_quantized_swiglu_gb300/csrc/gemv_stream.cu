// gemv_stream.cu -- persistent stream-K decode GEMV (M <= 16), optionally the
// whole MLP block in one cooperative launch.
//
// Operation: as gemv_dec.cu -- y[m, n] = sum_k x[m,k] W[n,k] with W decoded
// on the fly (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented"; vllm.cpp
// issue "tp>1 fp8w tail-MLP shard ...", "Mechanism on the tp>1 path"), gate
// and up fused with the SwiGLU epilogue (same issue, "Proposed fix").
//
// Schedule (GB300, 152 SMs, HBM-bound): the weight matrix of a phase is a
// flat sequence of W = Nt * Kc chunk records (16 rows x 64 k each,
// contiguous in row-tile-major order). One 16-warp CTA per SM; global warp w
// streams the contiguous record range [w*L, (w+1)*L), L = ceil(W / warps),
// so every warp moves the same bytes.
//  * Records are stored interleaved (see GemvProj): at step j the 16 warps of
//    a CTA need 16 adjacent records, so one producer warp fetches a whole
//    step per projection with a single bulk-async copy (cp.async.bulk, 9 KB
//    for NVFP4) into a ring of shared-memory slots (full/empty mbarriers).
//    Small per-warp copies cap a GB300 at ~2.5 TB/s; step-sized copies reach
//    ~6 TB/s. Bytes in flight cost shared memory, not registers.
//  * The producer starts before the consumers stage x and runs ahead into
//    the next phase (the weights do not depend on x or act), so HBM latency
//    overlaps the staging and the grid barrier.
//  * x[:, 0:K) is staged once per CTA as prescaled fp16 fragments (per-token
//    power of two, exact for every value within 2^29 of the token's max).
//  * A warp that covers a whole 16-row tile applies the epilogue from its
//    MMA accumulators; a tile split between warps is finished by the last
//    warp to arrive (atomic counter, reset by that warp), which adds the
//    per-warp partials in k order. No float atomics: deterministic.
//  * Fused mode runs gate/up+SwiGLU, then a grid-wide barrier (bounded spin;
//    the launch is cooperative so all CTAs are resident), then the down
//    projection; each warp fills its ring with down-projection records
//    before waiting at the barrier.
//  * Every wait is bounded (globaltimer); on expiry the kernel records the
//    error in the handle's error word, waits (bounded) for its own copies
//    still in flight and returns.
#include <algorithm>

#include "gemv_frag.cuh"

namespace qmlp {
namespace {

constexpr int kSWarps = 16;                     // consumer warps
constexpr int kCThreads = kSWarps * 32;         // consumer threads
constexpr int kSThreads = kCThreads + 32;       // + one producer warp
constexpr int kMaxDepth = 16;
constexpr int kSmemBudget = 220 * 1024;
constexpr int kBarBytes = 2 * kMaxDepth * 8;    // full + empty barriers
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

struct PhaseArgs {
    int TWr;                 // warps of the record layout (= warps launched)
    int R;                   // records per warp per step
    const uint8_t* wc0;
    const float* chs0;
    float inv0;
    const uint8_t* wc1;
    const float* chs1;
    float inv1;
    const __nv_bfloat16* x;  // [M, K]
    void* out;               // bf16 [M, N] or fp32 [M, N]
    int* counters;           // [Nt]
    int Nt, Kc, K, N;
    int L;                   // records per warp
    int smax;                // partial slots per row tile
    int depth;               // ring slots per warp
    size_t part_floats;      // index checks: floats of the partial buffer
};

struct StreamArgs {
    PhaseArgs A, B;
    float* part;
    unsigned* bar;  // [2]: arrival count, generation
    int* err;
    int M;
    int xs_bytes;    // activation staging region
    int slot_bytes;  // one ring slot: NP x 16 warps x R records
    int depth;       // ring slots
};

// Epilogue of one 16-row tile from fragment-ordered sums v[(p*NT+n)*4+e]
// (lane (g, t) holds rows g, g+8 x tokens 2t, 2t+1 of each token tile).
template <int FMT, int NT, int NP, int EPI>
__device__ __noinline__ void tile_epilogue(const PhaseArgs* a, int M, int rt, const float* v, const int* s_sig) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = n * 8 + 2 * t + (e & 1);
            if (m >= M) continue;
            const int row = rt * kTileRows + g + (e >= 2 ? 8 : 0);
            if (!QMLP_INB(row, a->N, 24)) continue;
            const float y0 = scalbnf(v[(0 * NT + n) * 4 + e], -s_sig[m]);
            if (EPI == kEpiRaw) {
                reinterpret_cast<float*>(a->out)[(size_t)m * a->N + row] = y0;
            } else {
                const float s0 = FMT == kNVFP4 ? a->inv0 : a->chs0[row];
                float res = y0 * s0;
                if (EPI == kEpiSwiGLU) {
                    const float s1 = FMT == kNVFP4 ? a->inv1 : a->chs1[row];
                    const float y1 = scalbnf(v[((NP - 1) * NT + n) * 4 + e], -s_sig[m]) * s1;
                    res = silu_f32(res) * y1;
                }
                reinterpret_cast<__nv_bfloat16*>(a->out)[(size_t)m * a->N + row] = __float2bfloat16_rn(res);
            }
        }
    }
}

// Partial-sum slot of warp gw in row tile rt: contributors are the warps
// w0..w1 whose record ranges overlap the tile; slot = gw - w0.
QMLP_DEV void tile_contributors(const PhaseArgs* a, int rt, int gw, int* slot, int* ncontrib) {
    const long base = (long)rt * a->Kc;
    const long w0 = base / a->L, w1 = (base + a->Kc - 1) / a->L;
    *slot = (int)(gw - w0);
    *ncontrib = (int)(w1 - w0 + 1);
}

// Store this warp's partial sums of tile rt (no fence: published later).
template <int NT, int NP>
__device__ __noinline__ void write_partial(const PhaseArgs* a, float* part, int rt, int gw, const float* acc) {
    constexpr int Q = NP * NT;
    const int lane = threadIdx.x & 31;
    int slot, nc;
    tile_contributors(a, rt, gw, &slot, &nc);
    float4* dst = reinterpret_cast<float4*>(part) + ((size_t)rt * a->smax + slot) * (Q * 32);
    if (!QMLP_INB(slot, a->smax, 22) ||
        !QMLP_INB((((size_t)rt * a->smax + slot) * (Q * 32) + (Q - 1) * 32 + lane) * 4 + 3, a->part_floats, 22))
        return;
#pragma unroll
    for (int q = 0; q < Q; ++q)
        dst[q * 32 + lane] = make_float4(acc[q * 4 + 0], acc[q * 4 + 1], acc[q * 4 + 2], acc[q * 4 + 3]);
}

// Announce this warp's (already fenced) partials of the row tiles pend[0..npend)
// -- one counter per tile, the atomics issued together from separate lanes --
// and, for each tile where this warp arrived last, add all partials in slot
// (= k) order and apply the epilogue.
template <int FMT, int NT, int NP, int EPI>
__device__ __noinline__ void finish_partials(const PhaseArgs* a, float* part, int M, const int* pend, int npend,
                                             int gw, const int* s_sig) {
    constexpr int Q = NP * NT;
    const int lane = threadIdx.x & 31;
    int prev = -1;
    if (lane < npend) {
        const int rt = lane == 0 ? pend[0] : pend[1];
        unsigned* ctr = reinterpret_cast<unsigned*>(&a->counters[QMLP_INB(rt, a->Nt, 23) ? rt : 0]);
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
    }
    __syncwarp();
    for (int i = 0; i < npend; ++i) {
        const int rt = i == 0 ? pend[0] : pend[1];
        int slot, nc;
        tile_contributors(a, rt, gw, &slot, &nc);
        const int pv = __shfl_sync(0xffffffffu, prev, i);
        if (pv != nc - 1) continue;
        // the acquiring lane saw every partial; order this warp's reads after it
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        if (lane == 0) a->counters[rt] = 0;
        float v[Q * 4];
#pragma unroll
        for (int e = 0; e < Q * 4; ++e) v[e] = 0.0f;
        const float4* src = reinterpret_cast<const float4*>(part) + (size_t)rt * a->smax * (Q * 32);
        for (int sl = 0; sl < nc; ++sl) {
            if (!QMLP_INB((((size_t)rt * a->smax + sl) * (Q * 32) + (Q - 1) * 32 + lane) * 4 + 3, a->part_floats, 23))
                break;
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const float4 f = __ldcg(src + ((size_t)sl * Q + q) * 32 + lane);
                v[q * 4 + 0] += f.x;
                v[q * 4 + 1] += f.y;
                v[q * 4 + 2] += f.z;
                v[q * 4 + 3] += f.w;
            }
        }
        tile_epilogue<FMT, NT, NP, EPI>(a, M, rt, v, s_sig);
    }
}

// Ring bookkeeping: global step index q (counting across phases) uses slot
// q % depth in round q / depth.
struct Ring {
    uint8_t* base;
    uint32_t base_s;   // shared address of slot 0
    uint32_t full0;    // full barriers [depth]
    uint32_t empty0;   // empty barriers [depth]
    int slot_bytes;
    int depth;
};

// Producer warp (lane 0): stream the steps of one phase into the ring.
// Returns the next global step index, or -(q + 1) when the wait before step
// q expired (steps < q were issued).
template <int FMT, int NP>
QMLP_DEV int produce_phase(const PhaseArgs& a, const Ring& r, int q, int* err) {
    constexpr uint32_t rec = rec_bytes<FMT>();
    const uint32_t step_bytes = kSWarps * a.R * rec;
    const int steps = a.L / a.R;
    int slot = q % r.depth;
    int round = q / r.depth;
    const uint8_t* src0 = a.wc0 + (size_t)blockIdx.x * kSWarps * a.R * rec;
    const uint8_t* src1 = a.wc1 + (size_t)blockIdx.x * kSWarps * a.R * rec;
    const size_t stride = (size_t)a.TWr * a.R * rec;  // bytes between consecutive steps
    for (int j = 0; j < steps; ++j, ++q) {
        if (round > 0 && !mbar_wait_bounded(r.empty0 + 8u * slot, (uint32_t)((round - 1) & 1), kWaitLimitNs)) {
            atomicExch(err, 4);
            return -(q + 1);
        }
        const uint32_t full = r.full0 + 8u * slot;
        const uint32_t dst = r.base_s + (uint32_t)slot * r.slot_bytes;
        const uint8_t* s0 = src0 + (size_t)j * stride;
        const uint8_t* s1 = src1 + (size_t)j * stride;
        if (!QMLP_INB((size_t)(s0 - a.wc0) + step_bytes - 1, (size_t)a.TWr * a.L * rec, 21)) {
            s0 = a.wc0;
            s1 = a.wc1;
        }
        mbar_arrive_expect_tx(full, NP * step_bytes);
        bulk_g2s(dst, s0, step_bytes, full);
        if (NP == 2) bulk_g2s(dst + step_bytes, s1, step_bytes, full);
        if (++slot == r.depth) {
            slot = 0;
            ++round;
        }
    }
    return q;
}

// Consumer warp: stream this warp's records of one phase from the ring.
// Returns the next global step index, or -1 after an expired wait.
template <int FMT, int NT, int NP, int EPI, bool M1>
QMLP_DEV int consume_phase(const PhaseArgs* ap, const Ring& r, int q, float* part, int M, int gw, int warp,
                           const uint4* xs, const int* s_sig, int* err) {
    const PhaseArgs& a = *ap;
    constexpr int rec = rec_bytes<FMT>();
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int slots = 4 * M;
    const int R = a.R;
    const long W = (long)a.Nt * a.Kc;
    const long u0 = (long)gw * a.L;
    const int n = u0 < W ? (int)min((long)a.L, W - u0) : 0;  // records of this warp
    const int steps = a.L / R;
    const uint32_t step_bytes = (uint32_t)kSWarps * R * rec;
    const int Kc = a.Kc;
    float acc[NP][NT][4];
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int qq = 0; qq < NT; ++qq)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[p][qq][i] = 0.0f;
    int rt = n > 0 ? (int)(u0 / Kc) : 0, c = n > 0 ? (int)(u0 % Kc) : 0, cs = c;
    int slot = q % r.depth;
    uint32_t parity = (uint32_t)((q / r.depth) & 1);
    const uint32_t warp_off = (uint32_t)warp * R * rec;
    int pend[2] = {0, 0};  // row tiles with an unannounced partial (range start / end)
    int npend = 0;
    int k = 0;  // records of this warp consumed so far
    for (int j = 0; j < steps; ++j) {
        if (!mbar_wait_bounded(r.full0 + 8u * slot, parity, kWaitLimitNs)) {
            if (lane == 0) atomicExch(err, 2);
            return -1;
        }
        const uint8_t* sbase = r.base + (uint32_t)slot * (uint32_t)r.slot_bytes + warp_off;
        const int kend = min(k + R, n);
        for (; k < kend; ++k, sbase += rec) {
            ChunkW w[NP];
#pragma unroll
            for (int p = 0; p < NP; ++p) w[p] = lds_chunk<FMT>(sbase + p * step_bytes, lane);
            uint4 xb[NT][2];
            load_xfrag<NT>(xs, c, M, slots, g, t, xb);
            mma_chunk<FMT, NT, NP, M1>(w, xb, acc);
            if (++c == Kc || k == n - 1) {
                float tmp[NP * NT * 4];
#pragma unroll
                for (int p = 0; p < NP; ++p)
#pragma unroll
                    for (int qq = 0; qq < NT; ++qq)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            tmp[(p * NT + qq) * 4 + e] = acc[p][qq][e];
                            acc[p][qq][e] = 0.0f;
                        }
                if (cs == 0 && c == Kc) {
                    tile_epilogue<FMT, NT, NP, EPI>(ap, M, rt, tmp, s_sig);
                } else {
                    // a tile shared with neighbouring warps: store now, announce
                    // once at the end of the range (one fence per warp)
                    write_partial<NT, NP>(ap, part, rt, gw, tmp);
                    if (npend < 2) pend[npend++] = rt;
                }
                ++rt;
                c = 0;
                cs = 0;
            }
        }
        k = max(k, (j + 1) * R);
        __syncwarp();
        if (lane == 0) mbar_arrive(r.empty0 + 8u * slot);
        if (++slot == r.depth) {
            slot = 0;
            parity ^= 1u;
        }
    }
    if (npend > 0) {
        __threadfence();
        finish_partials<FMT, NT, NP, EPI>(ap, part, M, pend, npend, gw, s_sig);
    }
    return q + steps;
}

// Grid-wide barrier over all (co-resident) CTAs; false if the bounded wait
// ran out (the error word is set).
QMLP_DEV bool grid_barrier(unsigned* bar, int* err) {
    __shared__ int s_ok;
    named_bar_sync(1, kCThreads);
    if (threadIdx.x == 0) {
        volatile unsigned* vgen = bar + 1;
        const unsigned gen = *vgen;
        __threadfence();
        const unsigned arrived = atomicAdd(bar, 1u);
        int ok = 1;
        if (arrived == gridDim.x - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (*vgen == gen) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicExch(err, 3);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    named_bar_sync(1, kCThreads);
    return s_ok != 0;
}

template <int FMT, int NT, int NPA, int EPIA, bool FUSED, bool M1>
__global__ void __launch_bounds__(kSThreads, 1) gemv_stream_kernel(const __grid_constant__ StreamArgs sa) {
    extern __shared__ __align__(128) uint8_t dyn_smem[];
    uint4* xs = reinterpret_cast<uint4*>(dyn_smem);
    __shared__ int s_maxbits[16];
    __shared__ int s_sig[16];
    __shared__ int s_fail;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Ring r;
    r.base = dyn_smem + sa.xs_bytes;
    r.base_s = smem_u32(r.base);
    r.slot_bytes = sa.slot_bytes;
    r.depth = sa.depth;
    r.full0 = smem_u32(r.base + (size_t)sa.depth * sa.slot_bytes);
    r.empty0 = r.full0 + 8u * kMaxDepth;
    if (threadIdx.x == 0) {
        for (int i = 0; i < sa.depth; ++i) {
            mbar_init(r.full0 + 8u * i, 1);
            mbar_init(r.empty0 + 8u * i, kSWarps);
        }
        fence_mbar_init();
        s_fail = 0;
    }
    __syncthreads();  // the last CTA-wide barrier: the producer never waits on consumers' barriers

    if (warp == kSWarps) {
        // ---- producer warp ----
        if (lane == 0) {
            int q = produce_phase<FMT, NPA>(sa.A, r, 0, sa.err);
            if (FUSED && q >= 0) q = produce_phase<FMT, 1>(sa.B, r, q, sa.err);
            // every issued step is waited on by the consumers; after an
            // expired wait, wait (bounded) for the last copy issued into each
            // slot so none is in flight when the CTA leaves
            if (q < 0) {
                const int issued = -q - 1;
                for (int qq = issued - 1; qq >= 0 && qq >= issued - sa.depth; --qq)
                    mbar_wait_bounded(r.full0 + 8u * (int)(qq % sa.depth), (uint32_t)((qq / sa.depth) & 1),
                                      kWaitLimitNs);
            }
        }
        return;
    }

    // ---- consumer warps ----
    const int gw = blockIdx.x * kSWarps + warp;
    const int M = sa.M;
    stage_x(sa.A.x, M, sa.A.K, 0, sa.A.K, sa.A.Kc * kChunkK, xs, s_maxbits, s_sig, kCThreads);
    int q = consume_phase<FMT, NT, NPA, EPIA, M1>(&sa.A, r, 0, sa.part, M, gw, warp, xs, s_sig, sa.err);
    if (FUSED) {
        if (q < 0 && lane == 0) s_fail = 1;
        __threadfence();
        const bool grid_ok = grid_barrier(sa.bar, sa.err);
        if (!grid_ok || s_fail != 0) return;
        stage_x(sa.B.x, M, sa.B.K, 0, sa.B.K, sa.B.Kc * kChunkK, xs, s_maxbits, s_sig, kCThreads);
        consume_phase<FMT, NT, 1, kEpiPlain, M1>(&sa.B, r, q, sa.part, M, gw, warp, xs, s_sig, sa.err);
    }
}

template <int FMT, int NT, int NPA, int EPIA, bool FUSED, bool M1>
cudaError_t launch_t(const StreamArgs& a, size_t smem, int grid, bool coop, cudaStream_t s) {
    auto kern = gemv_stream_kernel<FMT, NT, NPA, EPIA, FUSED, M1>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = coop ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Occupancy of one instantiation at a dynamic shared memory size; the last
// answer is cached (the query costs far more than a launch).
template <int FMT, int NT, int NPA, int EPIA, bool FUSED, bool M1>
cudaError_t occupancy_t(size_t smem, int* blocks) {
    auto kern = gemv_stream_kernel<FMT, NT, NPA, EPIA, FUSED, M1>;
    static bool attr_set = false;
    static size_t cached_smem = ~(size_t)0;
    static int cached_blocks = 0;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (smem == cached_smem) {
        *blocks = cached_blocks;
        return cudaSuccess;
    }
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, kern, kSThreads, smem);
    if (e == cudaSuccess) {
        cached_smem = smem;
        cached_blocks = *blocks;
    }
    return e;
}

// mode: 0 = fused MLP, 1 = gate/up+SwiGLU, 2 = plain, 3 = raw
template <int FMT, int NT, bool M1>
cudaError_t dispatch_t(int mode, const StreamArgs* a, size_t smem, int* blocks, bool query, cudaStream_t s,
                       int grid) {
    switch (mode) {
        case 0:
            return query ? occupancy_t<FMT, NT, 2, kEpiSwiGLU, true, M1>(smem, blocks)
                         : launch_t<FMT, NT, 2, kEpiSwiGLU, true, M1>(*a, smem, grid, true, s);
        case 1:
            return query ? occupancy_t<FMT, NT, 2, kEpiSwiGLU, false, M1>(smem, blocks)
                         : launch_t<FMT, NT, 2, kEpiSwiGLU, false, M1>(*a, smem, grid, false, s);
        case 2:
            return query ? occupancy_t<FMT, NT, 1, kEpiPlain, false, M1>(smem, blocks)
                         : launch_t<FMT, NT, 1, kEpiPlain, false, M1>(*a, smem, grid, false, s);
        default:
            return query ? occupancy_t<FMT, NT, 1, kEpiRaw, false, M1>(smem, blocks)
                         : launch_t<FMT, NT, 1, kEpiRaw, false, M1>(*a, smem, grid, false, s);
    }
}

// nt = token tiles (1: M <= 8, 2: M <= 16); m1 = (M == 1)
cudaError_t dispatch(int fmt, int nt, bool m1, int mode, const StreamArgs* a, size_t smem, int* blocks, bool query,
                     cudaStream_t s, int grid) {
    if (fmt == kNVFP4) {
        if (nt == 2) return dispatch_t<kNVFP4, 2, false>(mode, a, smem, blocks, query, s, grid);
        return m1 ? dispatch_t<kNVFP4, 1, true>(mode, a, smem, blocks, query, s, grid)
                  : dispatch_t<kNVFP4, 1, false>(mode, a, smem, blocks, query, s, grid);
    }
    if (nt == 2) return dispatch_t<kFP8, 2, false>(mode, a, smem, blocks, query, s, grid);
    return m1 ? dispatch_t<kFP8, 1, true>(mode, a, smem, blocks, query, s, grid)
              : dispatch_t<kFP8, 1, false>(mode, a, smem, blocks, query, s, grid);
}

int rec_of(int fmt) { return fmt == kNVFP4 ? kRecNVFP4 : kRecFP8; }

size_t stage_bytes(int M, int K) {
    const size_t b = (size_t)((K + kChunkK - 1) / kChunkK) * 128 * M;
    return (b + 127) & ~(size_t)127;
}

// Ring slots that fit after the staging region for slots of `slot_bytes`.
int depth_for(size_t xs, int slot_bytes) {
    const long avail = (long)kSmemBudget - (long)xs - kBarBytes - 1024;
    if (avail <= 0) return 0;
    return (int)std::min<long>(kMaxDepth, avail / slot_bytes);
}
int slot_bytes_for(int fmt, int np, int R) { return np * kSWarps * R * rec_of(fmt); }

void fill_phase(PhaseArgs& p, const GemvStreamPhase& src, int total_warps, int depth) {
    p.TWr = src.p0.TWr;
    p.R = src.p0.Rr;
    p.wc0 = src.p0.wc;
    p.chs0 = src.p0.chs;
    p.inv0 = src.p0.inv_g;
    p.wc1 = src.p1.wc;
    p.chs1 = src.p1.chs;
    p.inv1 = src.p1.inv_g;
    p.x = reinterpret_cast<const __nv_bfloat16*>(src.x);
    p.out = src.out;
    p.counters = src.counters;
    p.Nt = src.p0.Nt;
    p.Kc = src.p0.Kc;
    p.K = src.p0.K;
    p.N = src.p0.N;
    (void)total_warps;
    p.L = src.p0.Lr;  // the layout fixes the records per warp
    p.smax = (p.Kc + p.L - 1) / p.L + 1;
    p.depth = depth;
}

size_t phase_part_elems(const PhaseArgs& p, int np, int nt) { return (size_t)p.Nt * p.smax * np * nt * 128; }

}  // namespace

int gemv_layout_warps(int num_sms) { return std::max(num_sms, 1) * kSWarps; }

bool gemv_stream_fits(int fmt, int M, int K, int np, int R) {
    if (M < 1 || M > 16) return false;
    return depth_for(stage_bytes(M, K), slot_bytes_for(fmt, np, R)) >= 2;
}

size_t gemv_stream_part_elems(int K, int I, int num_sms) {
    // Nt*smax <= total_warps + 2*Nt (see fill_phase); fragments of 2
    // projections x 2 token tiles, one CTA per SM
    const size_t tw = (size_t)std::max(num_sms, 1) * kSWarps;
    const size_t nt_max = (size_t)std::max(K, I) / kTileRows;
    return (tw + 2 * nt_max + 16) * 2 * 2 * 128;
}

cudaError_t launch_gemv_stream(int fmt, int M, const GemvStreamPhase& A, const GemvStreamPhase* B, float* part,
                               size_t part_cap, unsigned* bar, int* err, int num_sms, cudaStream_t s) {
    if (M < 1 || M > 16) return cudaErrorInvalidValue;
    const int nt = M <= 8 ? 1 : 2;
    const int mode = B ? 0 : (A.epi == kEpiSwiGLU ? 1 : (A.epi == kEpiPlain ? 2 : 3));
    const int npa = A.epi == kEpiSwiGLU ? 2 : 1;
    size_t xs = stage_bytes(M, A.p0.K);
    if (B) xs = std::max(xs, stage_bytes(M, B->p0.K));
    int slot = slot_bytes_for(fmt, npa, A.p0.Rr);
    if (B) slot = std::max(slot, slot_bytes_for(fmt, 1, B->p0.Rr));
    const int depth = depth_for(xs, slot);
    if (depth < 2) return cudaErrorInvalidValue;
    const size_t smem = xs + (size_t)depth * slot + kBarBytes;
    int blocks = 0;
    const bool m1 = M == 1;
    cudaError_t e = dispatch(fmt, nt, m1, mode, nullptr, smem, &blocks, true, s, 0);
    if (e != cudaSuccess) return e;
    if (blocks < 1) return cudaErrorInvalidConfiguration;
    // one CTA per streaming-warp group of the layout (at most one per SM: the
    // rings fill its shared memory, and the fused launch is cooperative)
    const int grid = A.p0.TWr / kSWarps;
    if (grid < 1 || grid > num_sms || A.p0.TWr != grid * kSWarps || (B && B->p0.TWr != grid * kSWarps))
        return cudaErrorInvalidValue;
    StreamArgs a;
    fill_phase(a.A, A, grid * kSWarps, depth);
    size_t need = phase_part_elems(a.A, npa, nt);
    if (B) {
        fill_phase(a.B, *B, grid * kSWarps, depth);
        need = std::max(need, phase_part_elems(a.B, 1, nt));
    } else {
        a.B = a.A;
    }
    if (need > part_cap) return cudaErrorInvalidValue;
    a.A.part_floats = part_cap;
    a.B.part_floats = part_cap;
    a.part = part;
    a.bar = bar;
    a.err = err;
    a.M = M;
    a.xs_bytes = (int)xs;
    a.slot_bytes = slot;
    a.depth = depth;
    return dispatch(fmt, nt, m1, mode, &a, smem, &blocks, false, s, grid);
}

QMLP_BOUNDS_UNIT(gemv_stream)

}  // namespace qmlp
