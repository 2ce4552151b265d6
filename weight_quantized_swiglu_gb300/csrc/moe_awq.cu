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
// GB300 design. 10 routes x (320 x 2560 + 2560 x 160) weights, ~7.7 MB per
// call: a latency problem. The dot products run on the tensor cores
// (mma.sync m16n8k16, fp16 x fp16 -> fp32, the token in column 0), so a
// weight costs ~2 instructions of decode instead of a scalar half_fma,
// conversion and fp32 FMA each, and the work spreads over thousands of
// warps:
//  * A fragments straight from the checkpoint layout: lane (g, t) of a
//    16-row tile needs byte t of every 32-bit word of rows g and g+8 (the k
//    pairs 2t..2t+1 and 8+2t..9+2t of each k16 group). One PRMT copies that
//    byte into both halves of a register, one LOP3 turns it into the fp16
//    pair (1024 + q_lo, 1024 + 16 q_hi), one exact HFMA2 recovers (q_lo,
//    q_hi) and one HFMA2 forms half_fma(q, s, b) for both -- the same
//    single rounding as the scalar definition.
//  * B fragment = the token: x as fp16 (fp16 input as is; bf16 input times a
//    power of two per call, exact for every value within 2^29 of max|x|),
//    the intermediate act as fp16 (exact).
//  * W13: a CTA per (route, 8 gate rows and the matching 8 up rows as one
//    16-row MMA tile); each warp takes the tile over a tenth of K, and the
//    partial sums are added in a fixed order in shared memory.
//  * W2: a CTA per 16 output rows with one warp per route; the fp16 route
//    results are added in router order by one thread per output row.
//  * Programmatic dependent launch: the W2 grid starts while W13 runs, reads
//    the ids and loads its codes and metadata into registers, and only then
//    waits (griddepcontrol.wait) for the intermediate.
//  * Lane-sliced banks (the handle's copy, made at create): every 16-byte
//    unit of a row (4 words, 32 k) is byte-transposed so that byte t of its
//    four words is one aligned 32-bit word at offset 4t -- exactly what lane
//    t's PRMT picks. A lane then loads 4 bytes per unit instead of the whole
//    unit: 4x less register space per chunk, so W13 keeps a warp's 4 chunks
//    in flight at once. The allocation-free entry point reads the banks in
//    the checkpoint layout and uses the same kernels in that layout.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace qmlp {
namespace {

constexpr int kK13 = 10;  // W13 K splits: a CTA has kK13 warps, each on 8 gate + 8 up rows
constexpr int kC13 = 2;   // 64-k chunks a W13 warp loads at once (checkpoint layout)
constexpr int kC13S = 4;  // the same with lane-sliced banks (a fifth of the registers per chunk)
constexpr int kG2 = 10;   // k16 groups a W2 warp loads at once
constexpr int kW2PreMax = 56 * 1024;  // W2's decoded fragments (w2_pre): up to 11 routes of 10 groups
constexpr int kXRegs = 4; // x pairs a W13 thread loads before the ids (K <= 2 * 4 * 320 = 2560 in one go)
// Shared memory of a W13 CTA: x (2K bytes, K <= 16384) needs at most 32 KB;
// the request is 80 KB so that no SM takes a third W13 CTA. Measured: the
// next call's W13 grid launches while the previous W2 CTAs still hold SMs,
// and the free SMs were given three W13 CTAs each (their MMA phase took 2.5
// instead of 1.7 us and set the end of the stage): 8.2 -> 7.3 us per call.
constexpr int kW13Smem = 80 * 1024;

struct Args {
    int E, K, I;
    const uint8_t* w13;
    const uint8_t* w13_meta;
    const uint8_t* w2;
    const uint8_t* w2_meta;
    const void* x;
    int x_is_bf16;
    int meta_al4;  // 4-byte records are 4-byte aligned (one load each)
    const int32_t* ids;
    const float* rw;
    int topk;
    __half* out;
    __half* act_ws;
    __half* gu_dbg;
    __half* act_dbg;
    __half* y_dbg;
    // index checks: bytes of the banks, elements of the act workspace
    size_t w13_bytes, w13_meta_bytes, w2_bytes, w2_meta_bytes, act_elems;
    int w2_pre;  // W2 decodes its A fragments into shared memory before the wait (one batch of groups)
};

// One metadata record (little-endian fp16 scale, then fp16 bias or u8 zero)
// as its raw bytes, low byte first.
template <int MB>
QMLP_DEV uint32_t load_meta(const uint8_t* p, bool al4) {
    if (MB == 4 && al4) return __ldg(reinterpret_cast<const unsigned int*>(p));
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < MB; ++i) v |= (uint32_t)__ldg(p + i) << (8 * i);
    return v;
}

// {scale, scale} and {bias, bias} of a record as f16x2: the bias is stored
// (4-byte) or half(-zero*scale) -- the product of a 4-bit integer and an fp16
// is exact in fp32, so one rounding to fp16 matches half arithmetic.
template <int MB>
QMLP_DEV void meta_sb2(uint32_t m, uint32_t& s2, uint32_t& b2) {
    const uint32_t s = m & 0xFFFFu;
    uint32_t b;
    if (MB == 4) {
        b = m >> 16;
    } else {
        const float bf = -(float)((m >> 16) & 0xFFu) * __half2float(__ushort_as_half((unsigned short)s));
        b = __half_as_ushort(__float2half_rn(bf));
    }
    s2 = s | (s << 16);
    b2 = b | (b << 16);
}

QMLP_DEV uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The byte of word w that `sel` (pair_selector) picks -- two u4 codes, the
// low nibble the earlier k -- to f16x2 {half_fma(q_lo, s, b), half_fma(q_hi, s, b)}.
QMLP_DEV uint32_t awq_pair(uint32_t w, uint32_t sel, uint32_t s2, uint32_t b2) {
    const uint32_t m = __byte_perm(w, 0u, sel);                // [b, 0, b, 0]
    const uint32_t h = (m & 0x00F0000Fu) | 0x64006400u;        // {1024 + q_lo, 1024 + 16 q_hi}
    const uint32_t q = hfma2_u32(h, 0x2C003C00u, 0xD400E400u);  // {q_lo, q_hi} = h * {1, 1/16} - {1024, 64}
    return hfma2_u32(q, s2, b2);
}

// PRMT selector placing byte t of a word in bytes 0 and 2 (bytes 1, 3 zero).
QMLP_DEV uint32_t pair_selector(int t) {
    return (uint32_t)t | (4u << 4) | ((uint32_t)t << 8) | (4u << 12);
}

// ---------------------------------------------------------------------------
// W13 + SwiGLU
// ---------------------------------------------------------------------------
// One W13 CTA: route r, gate rows 8 bx.. and the matching up rows. Returns
// false (the whole CTA, uniformly) for an invalid route, which writes nothing.
template <int MB, bool SL>
QMLP_DEV bool w13_cta(const Args& a, int bx, int r, uint32_t* x16, float (*part)[16], int& s_max) {
    // x does not depend on the route: its loads go out first, all at once
    // (then the ids -> weights round trips run while they are in flight)
    const uint32_t* xin32 = reinterpret_cast<const uint32_t*>(a.x);
    const int K2 = a.K / 2;
    uint32_t xv[kXRegs];
#pragma unroll
    for (int i = 0; i < kXRegs; ++i) {
        const int k2 = threadIdx.x + i * (int)blockDim.x;
        xv[i] = k2 < K2 ? xin32[k2] : 0u;
    }
    const int id = a.ids[r];
    if (id < 0 || id >= a.E) return false;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    // warp = K split; its 16-row MMA tile is gate rows 8*bx.. (rows 0-7) and
    // the matching up rows I + 8*bx.. (rows 8-15), both halves of 8 outputs
    const int ks = warp;
    const int Kc = a.K / 64, gpr = a.K / 32, N = 2 * a.I;
    const int cpw = moe_w13_cpw(a.K);  // chunks per warp
    static_assert(kK13 == kMoeKSplit, "the bank's warp blocks follow the K split");
    const int c0 = ks * cpw, c1 = min(Kc, c0 + cpw);
    const bool al4 = a.meta_al4 != 0;
    const size_t row0 = (size_t)id * N + 8 * bx + g;
    const size_t rows[2] = {row0, row0 + a.I};
    constexpr int kC = SL ? kC13S : kC13;
    static_assert(!SL || kC == 4, "batches of 4 chunks: the bank's metadata slots are sized for them");
    uint4 cw[kC][2][2];      // checkpoint layout: the two 16-byte units of each row's 32-byte chunk
    uint32_t cs[kC][2][2];   // handle's bank: this lane's word of each unit
    uint32_t mw[kC][2][2];
    // the handle's bank: this warp's block (e, octet, split) of codes and
    // its metadata slots (internal.h): per row half, one 16-byte load per
    // chunk pair and two (three for 3-byte records) for a batch's records
    const size_t blk = ((size_t)id * (a.I / 8) + bx) * kMoeKSplit + ks;
    const uint8_t* bcodes = a.w13 + blk * moe_w13_block_bytes(a.K);
    const int np = moe_w13_pairs(a.K);
    const int ms = moe_w13_meta_stride(a.K, MB);
    // every byte this lane reads of the banks lies inside them (one check of
    // the whole range: the offsets inside it are fixed by the layout)
    const bool inb = SL ? (QMLP_INB((blk + 1) * moe_w13_block_bytes(a.K) - 1, a.w13_bytes, 31) &&
                           QMLP_INB((blk + 1) * moe_w13_meta_block_bytes(a.K, MB) - 1, a.w13_meta_bytes, 32))
                        : (QMLP_INB((rows[1] + 1) * (a.K / 2) - 1, a.w13_bytes, 31) &&
                           QMLP_INB((rows[1] + 1) * gpr * MB - 1, a.w13_meta_bytes, 32));
    auto load_batch = [&](int cb) {
        if (!inb) return;
        if (SL) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
#pragma unroll
                for (int pi = 0; pi < kC / 2; ++pi) {
                    const int pp = (cb - c0) / 2 + pi;
                    if (pp < np) {
                        const uint4 u = __ldg(reinterpret_cast<const uint4*>(bcodes + (size_t)(q * np + pp) * 512) +
                                              lane);
                        cs[2 * pi][q][0] = u.x;
                        cs[2 * pi][q][1] = u.y;
                        cs[2 * pi + 1][q][0] = u.z;
                        cs[2 * pi + 1][q][1] = u.w;
                    }
                }
                // records 2(cb - c0) .. 2(cb - c0) + 2kC - 1 of the (q, g) slot
                const uint8_t* slot = a.w13_meta + blk * moe_w13_meta_block_bytes(a.K, MB) + (q * 8 + g) * ms +
                                      (size_t)(cb - c0) * 2 * MB;
                {
                    if (MB == 4) {
                        const uint4 m0 = __ldg(reinterpret_cast<const uint4*>(slot));
                        const uint4 m1 = __ldg(reinterpret_cast<const uint4*>(slot) + 1);
                        const uint32_t mr[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
                        for (int i = 0; i < kC; ++i) {
                            mw[i][q][0] = mr[2 * i];
                            mw[i][q][1] = mr[2 * i + 1];
                        }
                    } else {
                        uint32_t mr[3 * kC / 2 + 1];
#pragma unroll
                        for (int j = 0; j < 3 * kC / 4; ++j) {
                            const uint2 v = __ldg(reinterpret_cast<const uint2*>(slot) + j);
                            mr[2 * j] = v.x;
                            mr[2 * j + 1] = v.y;
                        }
                        mr[3 * kC / 2] = 0u;
#pragma unroll
                        for (int i = 0; i < kC; ++i)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int b = 3 * (2 * i + h);  // record 2i + h starts at byte b
                                mw[i][q][h] = __funnelshift_r(mr[b / 4], mr[b / 4 + 1], 8 * (b % 4)) & 0xFFFFFFu;
                            }
                    }
                }
            }
            return;
        }
#pragma unroll
        for (int i = 0; i < kC; ++i) {
            const int c = cb + i;
            if (c < c1) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint8_t* rowc = a.w13 + rows[q] * (a.K / 2) + c * 32;
                    cw[i][q][0] = __ldg(reinterpret_cast<const uint4*>(rowc));
                    cw[i][q][1] = __ldg(reinterpret_cast<const uint4*>(rowc) + 1);
                    const uint8_t* m = a.w13_meta + (rows[q] * gpr + 2 * c) * MB;
                    mw[i][q][0] = load_meta<MB>(m, al4);
                    mw[i][q][1] = load_meta<MB>(m + MB, al4);
                }
            }
        }
    };
    load_batch(c0);  // issued before x is staged: the two round trips overlap
    if (MB == 4) pdl_launch_dependents();  // see moe_w13_kernel

    // x -> fp16 pairs (bf16: times 2^sig so that max|x| lies in [2^14, 2^15));
    // pairs past kXRegs per thread (K > 2 kXRegs blockDim) are loaded here
    if (threadIdx.x == 0) s_max = 0;
    __syncthreads();
    const int kreg = kXRegs * (int)blockDim.x;
    if (a.x_is_bf16) {
        float mx = 0.0f;
#pragma unroll
        for (int i = 0; i < kXRegs; ++i)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(xv[i] << 16)), fabsf(__uint_as_float(xv[i] & 0xFFFF0000u))));
        for (int k2 = kreg + threadIdx.x; k2 < K2; k2 += blockDim.x) {
            const uint32_t v = xin32[k2];
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(v << 16)), fabsf(__uint_as_float(v & 0xFFFF0000u))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0 && mx > 0.0f) atomicMax(&s_max, __float_as_int(mx));
        __syncthreads();
    }
    const int sig = a.x_is_bf16 ? prescale_exponent(__int_as_float(s_max)) : 0;
    auto to16 = [&](uint32_t v) -> uint32_t {
        if (!a.x_is_bf16) return v;
        const float lo = scalbnf(__uint_as_float(v << 16), sig);
        const float hi = scalbnf(__uint_as_float(v & 0xFFFF0000u), sig);
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    };
#pragma unroll
    for (int i = 0; i < kXRegs; ++i) {
        const int k2 = threadIdx.x + i * (int)blockDim.x;
        if (k2 < K2) x16[k2] = to16(xv[i]);
    }
    for (int k2 = kreg + threadIdx.x; k2 < K2; k2 += blockDim.x) x16[k2] = to16(xin32[k2]);
    __syncthreads();

    const uint32_t sel = pair_selector(t);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    for (int cb = c0; cb < c1; cb += kC) {
        if (cb != c0) load_batch(cb);
#pragma unroll
        for (int i = 0; i < kC; ++i) {
            const int c = cb + i;
            if (c < c1) {
                uint32_t s2[2][2], b2[2][2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    meta_sb2<MB>(mw[i][q][0], s2[q][0], b2[q][0]);
                    meta_sb2<MB>(mw[i][q][1], s2[q][1], b2[q][1]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // k16 group j: AWQ group j/2, words 2j, 2j+1 of the chunk
                    const int h = j >> 1;
                    // B fragment: lanes with g == 0 hold column 0, the token;
                    // the other lanes load the same words (a broadcast, no
                    // branch) into columns 1-7, whose results are never read
                    const int k2 = (c * 64 + 16 * j) / 2 + t;
                    const uint32_t x0 = x16[k2], x1 = x16[k2 + 4];
                    uint32_t f0, f1, f2, f3;  // rows g, g+8 at k 2t.. (words 2j), then at 8+2t.. (words 2j+1)
                    if (SL) {
                        const uint32_t sa = pair_selector(2 * (j & 1)), sb = pair_selector(2 * (j & 1) + 1);
                        f0 = awq_pair(cs[i][0][h], sa, s2[0][h], b2[0][h]);
                        f1 = awq_pair(cs[i][1][h], sa, s2[1][h], b2[1][h]);
                        f2 = awq_pair(cs[i][0][h], sb, s2[0][h], b2[0][h]);
                        f3 = awq_pair(cs[i][1][h], sb, s2[1][h], b2[1][h]);
                    } else {
                        const uint32_t wa0 = (j & 1) ? cw[i][0][h].z : cw[i][0][h].x;
                        const uint32_t wb0 = (j & 1) ? cw[i][0][h].w : cw[i][0][h].y;
                        const uint32_t wa1 = (j & 1) ? cw[i][1][h].z : cw[i][1][h].x;
                        const uint32_t wb1 = (j & 1) ? cw[i][1][h].w : cw[i][1][h].y;
                        f0 = awq_pair(wa0, sel, s2[0][h], b2[0][h]);
                        f1 = awq_pair(wa1, sel, s2[1][h], b2[1][h]);
                        f2 = awq_pair(wb0, sel, s2[0][h], b2[0][h]);
                        f3 = awq_pair(wb1, sel, s2[1][h], b2[1][h]);
                    }
                    mma_f16_16816(d, f0, f1, f2, f3, x0, x1);
                }
            }
        }
    }
    // the token is column 0: lanes t == 0 hold rows g (d[0]) and g+8 (d[2])
    if (t == 0) {
        part[warp][g] = d[0];
        part[warp][g + 8] = d[2];
    }
    __syncthreads();
    if (threadIdx.x < 8) {
        const int j = threadIdx.x;
        float hg = 0.0f, hu = 0.0f;
        for (int w = 0; w < kK13; ++w) {
            hg += part[w][j];
            hu += part[w][8 + j];
        }
        const int q = 8 * bx + j;
        const __half gh = __float2half_rn(scalbnf(hg, -sig)), uh = __float2half_rn(scalbnf(hu, -sig));
        const __half act = __float2half_rn(silu_f32(__half2float(gh)) * __half2float(uh));
        if (QMLP_INB((size_t)r * a.I + q, a.act_elems, 33)) a.act_ws[(size_t)r * a.I + q] = act;
        if (a.gu_dbg) {
            a.gu_dbg[(size_t)r * 2 * a.I + q] = gh;
            a.gu_dbg[(size_t)r * 2 * a.I + a.I + q] = uh;
        }
        if (a.act_dbg) a.act_dbg[(size_t)r * a.I + q] = act;
    }
    return true;
}

template <int MB, bool SL>
__global__ void __launch_bounds__(kK13 * 32) moe_w13_kernel(const Args a) {
    extern __shared__ __align__(16) uint32_t x16[];  // [K/2] fp16 pairs
    __shared__ float part[kK13][16];                // [warp][row of its tile]
    __shared__ int s_max;
    // the ids, x and (through the intermediate) the previous call's W2
    // stage belong to the kernels before this one
    pdl_wait();
    // When the W2 grid may launch (its CTAs load their weights while this
    // grid computes): with 4-byte records once every CTA has issued its own
    // weight loads (inside w13_cta; a CTA of an invalid route leaves before),
    // with 3-byte records at once -- measured at E=512 top-10, hot ids:
    // 7.21 -> 6.77 us (4-byte), 8.00 against 7.80 us had 3-byte records waited.
    if (MB != 4) pdl_launch_dependents();
    w13_cta<MB, SL>(a, blockIdx.x, blockIdx.y, x16, part, s_max);
    if (MB == 4) pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// W2 + ordered router-weighted sum
// ---------------------------------------------------------------------------
// One W2 CTA: output rows 16 bx.., warp r = route r. Launched with
// programmatic dependent launch: the prologue (ids, codes, metadata) overlaps
// the W13 grid, then griddepcontrol.wait makes the intermediate visible.
template <int MB, bool SL>
QMLP_DEV void w2_cta(const Args& a, int bx, float (*ys)[16], float* s_rw, int* s_ok, uint4* frag) {
    const int r = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int n0 = 16 * bx;
    // prologue, overlapping the W13 stage: the ids and router weights (final
    // before W13 released this grid), kept in shared memory for the final
    // sum, and the first batch of codes and metadata
    const int id = r < a.topk ? a.ids[r] : -1;
    const bool valid = id >= 0 && id < a.E;
    if (lane == 0) {
        s_ok[r] = valid ? 1 : 0;
        s_rw[r] = valid ? a.rw[r] : 0.0f;
    }
    const int ng = a.I / 16, gpr = a.I / 32;
    const size_t row0 = (size_t)(valid ? id : 0) * a.K + n0 + g;
    const uint2* c0p = reinterpret_cast<const uint2*>(a.w2 + row0 * (a.I / 2));
    const uint2* c8p = reinterpret_cast<const uint2*>(a.w2 + (row0 + 8) * (a.I / 2));
    const uint8_t* m0p = a.w2_meta + row0 * gpr * MB;
    const uint8_t* m8p = a.w2_meta + (row0 + 8) * gpr * MB;
    const bool al4 = a.meta_al4 != 0;
    // the lane's rows of the banks and its route's act row lie inside them
    const bool inb = QMLP_INB((row0 + 9) * (a.I / 2) - 1, a.w2_bytes, 34) &&
                     QMLP_INB((row0 + 9) * gpr * MB - 1, a.w2_meta_bytes, 34) &&
                     QMLP_INB((size_t)(r + 1) * a.I - 1, a.act_elems, 35);
    uint2 cw[kG2][2];         // checkpoint layout: words 2j, 2j+1 of rows g and g+8 for k16 group j
    uint32_t cs[kG2 / 2][2];  // lane-sliced layout: this lane's 4 bytes of unit j/2 (groups j, j+1)
    uint32_t mw[kG2 / 2][2];  // the AWQ records of the batch
    auto load_batch = [&](int gb) {  // gb is a multiple of kG2 (even)
        if (!inb) return;
        if (SL) {
#pragma unroll
            for (int i = 0; i < kG2 / 2; ++i) {
                if (valid && gb + 2 * i < ng) {
                    cs[i][0] = __ldg(reinterpret_cast<const unsigned int*>(c0p + gb + 2 * i) + t);
                    cs[i][1] = __ldg(reinterpret_cast<const unsigned int*>(c8p + gb + 2 * i) + t);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < kG2; ++i) {
                if (valid && gb + i < ng) {
                    cw[i][0] = __ldg(c0p + gb + i);
                    cw[i][1] = __ldg(c8p + gb + i);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kG2 / 2; ++i) {
            const int ag = gb / 2 + i;
            if (valid && ag < gpr) {
                mw[i][0] = load_meta<MB>(m0p + (size_t)ag * MB, al4);
                mw[i][1] = load_meta<MB>(m8p + (size_t)ag * MB, al4);
            }
        }
    };
    load_batch(0);
    const uint32_t sel = pair_selector(t);
    // With every k16 group in the first batch, the A fragments (which do not
    // depend on act) are decoded before the wait, into this warp's slice of
    // shared memory: after the wait only the MMAs remain.
    const bool pre = a.w2_pre != 0;
    if (pre && valid) {
#pragma unroll
        for (int i = 0; i < kG2; ++i) {
            if (i < ng) {
                uint32_t s0, b0, s8, b8;
                meta_sb2<MB>(mw[i / 2][0], s0, b0);
                meta_sb2<MB>(mw[i / 2][1], s8, b8);
                uint4 f;
                if (SL) {
                    const uint32_t sa = pair_selector(2 * (i & 1)), sb = pair_selector(2 * (i & 1) + 1);
                    f = make_uint4(awq_pair(cs[i / 2][0], sa, s0, b0), awq_pair(cs[i / 2][1], sa, s8, b8),
                                   awq_pair(cs[i / 2][0], sb, s0, b0), awq_pair(cs[i / 2][1], sb, s8, b8));
                } else {
                    f = make_uint4(awq_pair(cw[i][0].x, sel, s0, b0), awq_pair(cw[i][1].x, sel, s8, b8),
                                   awq_pair(cw[i][0].y, sel, s0, b0), awq_pair(cw[i][1].y, sel, s8, b8));
                }
                frag[(r * kG2 + i) * 32 + lane] = f;
            }
        }
        __syncwarp();
    }
    pdl_wait();  // the W13 stage (act) is complete and visible
    const uint32_t* act = reinterpret_cast<const uint32_t*>(a.act_ws + (size_t)r * a.I);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    if (valid && pre) {
        uint32_t av[kG2][2];
#pragma unroll
        for (int i = 0; i < kG2; ++i) {
            av[i][0] = i < ng && inb ? act[8 * i + t] : 0u;
            av[i][1] = i < ng && inb ? act[8 * i + 4 + t] : 0u;
        }
#pragma unroll
        for (int i = 0; i < kG2; ++i) {
            if (i < ng) {
                const uint4 f = frag[(r * kG2 + i) * 32 + lane];
                mma_f16_16816(d, f.x, f.y, f.z, f.w, av[i][0], av[i][1]);
            }
        }
    } else if (valid) {
        for (int gb = 0; gb < ng; gb += kG2) {
            if (gb > 0) load_batch(gb);
            // the batch's act words, all loads at once; B fragment column 0
            // (lanes g == 0) is the token, the other lanes load the same words
            // into columns 1-7, whose results are never read (no branch)
            uint32_t av[kG2][2];
#pragma unroll
            for (int i = 0; i < kG2; ++i) {
                const int j = gb + i;
                av[i][0] = j < ng && inb ? act[8 * j + t] : 0u;
                av[i][1] = j < ng && inb ? act[8 * j + 4 + t] : 0u;
            }
#pragma unroll
            for (int i = 0; i < kG2; ++i) {
                const int j = gb + i;
                if (j < ng) {
                    uint32_t s0, b0, s8, b8;
                    meta_sb2<MB>(mw[i / 2][0], s0, b0);
                    meta_sb2<MB>(mw[i / 2][1], s8, b8);
                    const uint32_t x0 = av[i][0], x1 = av[i][1];
                    if (SL) {
                        const uint32_t sa = pair_selector(2 * (i & 1)), sb = pair_selector(2 * (i & 1) + 1);
                        mma_f16_16816(d, awq_pair(cs[i / 2][0], sa, s0, b0), awq_pair(cs[i / 2][1], sa, s8, b8),
                                      awq_pair(cs[i / 2][0], sb, s0, b0), awq_pair(cs[i / 2][1], sb, s8, b8), x0, x1);
                    } else {
                        mma_f16_16816(d, awq_pair(cw[i][0].x, sel, s0, b0), awq_pair(cw[i][1].x, sel, s8, b8),
                                      awq_pair(cw[i][0].y, sel, s0, b0), awq_pair(cw[i][1].y, sel, s8, b8), x0, x1);
                    }
                }
            }
        }
    }
    if (t == 0) {
        const __half y0 = __float2half_rn(d[0]), y8 = __float2half_rn(d[2]);
        ys[r][g] = __half2float(y0);
        ys[r][g + 8] = __half2float(y8);
        if (a.y_dbg && valid) {
            a.y_dbg[(size_t)r * a.K + n0 + g] = y0;
            a.y_dbg[(size_t)r * a.K + n0 + g + 8] = y8;
        }
    }
    __syncthreads();
    if (threadIdx.x < 16) {
        float s = 0.0f;
        for (int rr = 0; rr < a.topk; ++rr)
            if (s_ok[rr]) s = fmaf(s_rw[rr], ys[rr][threadIdx.x], s);
        if (QMLP_INB(n0 + threadIdx.x, a.K, 36)) a.out[n0 + threadIdx.x] = __float2half_rn(s);
    }
    // only now may the next kernel's CTAs launch: launched while this grid
    // computes, their set-up slowed the W2 warps on the same SMs (measured,
    // E=512 top-10: 7.41 -> 7.22 us hot with the trigger here)
    pdl_launch_dependents();
}

template <int MB, bool SL>
__global__ void __launch_bounds__(16 * 32) moe_w2_kernel(const Args a) {
    extern __shared__ __align__(16) uint4 w2frag[];  // [topk][kG2][32] decoded A fragments (w2_pre)
    __shared__ float ys[16][16];
    __shared__ float s_rw[16];
    __shared__ int s_ok[16];
    w2_cta<MB, SL>(a, blockIdx.x, ys, s_rw, s_ok, w2frag);
}

template <int MB, bool SL>
cudaError_t launch_mb(const Args& a, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(moe_w13_kernel<MB, SL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kW13Smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(moe_w2_kernel<MB, SL>, cudaFuncAttributeMaxDynamicSharedMemorySize, kW2PreMax);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c13 = {};
    c13.gridDim = dim3(a.I / 8, a.topk);
    c13.blockDim = dim3(kK13 * 32);
    c13.dynamicSmemBytes = kW13Smem;
    c13.stream = s;
    c13.attrs = pdl;
    c13.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&c13, moe_w13_kernel<MB, SL>, a);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t c2 = {};
    c2.gridDim = dim3(a.K / 16);
    c2.blockDim = dim3(32 * a.topk);
    c2.dynamicSmemBytes = a.w2_pre ? (size_t)a.topk * kG2 * 32 * sizeof(uint4) : 0;
    c2.stream = s;
    c2.attrs = pdl;
    c2.numAttrs = 1;
    return cudaLaunchKernelEx(&c2, moe_w2_kernel<MB, SL>, a);
}

}  // namespace

cudaError_t launch_moe(const MoeLaunch& L, int num_sms, cudaStream_t s) {
    (void)num_sms;
    if (L.topk < 1 || L.topk > 16 || L.K % 64 || L.I % 32 || L.K > 16384) return cudaErrorInvalidValue;
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
    a.meta_al4 = ((reinterpret_cast<uintptr_t>(L.w13_meta) | reinterpret_cast<uintptr_t>(L.w2_meta)) & 3u) == 0;
    a.ids = L.ids;
    a.rw = L.rw;
    a.topk = L.topk;
    a.out = L.out;
    a.act_ws = L.act_ws;
    a.gu_dbg = L.gu_dbg;
    a.act_dbg = L.act_dbg;
    a.y_dbg = L.y_dbg;
    const int MB = L.meta_bytes;
    a.w13_bytes = L.sliced ? moe_w13_bank_bytes(L.E, L.I, L.K) : (size_t)L.E * 2 * L.I * (L.K / 2);
    a.w13_meta_bytes =
        L.sliced ? moe_w13_meta_bank_bytes(L.E, L.I, L.K, MB) : (size_t)L.E * 2 * L.I * (L.K / 32) * MB;
    a.w2_bytes = (size_t)L.E * L.K * (L.I / 2);
    a.w2_meta_bytes = (size_t)L.E * L.K * (L.I / 32) * MB;
    a.act_elems = (size_t)16 * L.I;
    // the decoded fragments fit beside two W13 CTAs on an SM (one batch of
    // groups: I <= 16 kG2)
    a.w2_pre = L.I / 16 <= kG2 && (size_t)L.topk * kG2 * 32 * sizeof(uint4) <= kW2PreMax;
    if (L.sliced) return L.meta_bytes == 4 ? launch_mb<4, true>(a, s) : launch_mb<3, true>(a, s);
    return L.meta_bytes == 4 ? launch_mb<4, false>(a, s) : launch_mb<3, false>(a, s);
}

namespace {
// Lane-sliced codes: within every 16-byte unit, output word t holds byte t
// of input words 0..3 (a 4x4 byte transpose; units stay in place, so rows
// keep their offsets and every unit its alignment).
__global__ void slice_units_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, size_t units) {
    for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (size_t)gridDim.x * blockDim.x) {
        const uint4 v = in[u];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            o[t] = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) o[t] |= ((w[j] >> (8 * t)) & 0xFFu) << (8 * j);
        }
        out[u] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

namespace {
// One 16-byte item of the W13 warp-block bank (see internal.h) per thread:
// (block, q, pair, lane) -> 4 words, chunk c = c0 + 2p + hh, unit h, word =
// byte t of each of the unit's four checkpoint words.
__global__ void w13_blocks_kernel(const uint8_t* __restrict__ w, int E, int I, int K, uint4* __restrict__ out) {
    const int Kc = K / 64, cpw = moe_w13_cpw(K), np = moe_w13_pairs(K), no = I / 8;
    const size_t items = (size_t)E * no * kMoeKSplit * 2 * np * 32;
    for (size_t it = (size_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (size_t)gridDim.x * blockDim.x) {
        const int l = (int)(it % 32);
        size_t rest = it / 32;
        const int p = (int)(rest % np);
        rest /= np;
        const int q = (int)(rest % 2);
        rest /= 2;
        const int ks = (int)(rest % kMoeKSplit);
        rest /= kMoeKSplit;
        const int o = (int)(rest % no);
        const size_t e = rest / no;
        const int g = l >> 2, t = l & 3;
        const int c0 = ks * cpw, c1 = min(Kc, c0 + cpw);
        const size_t R = (size_t)(q == 0 ? 8 * o + g : I + 8 * o + g);
        const uint8_t* row = w + (e * 2 * I + R) * (K / 2);
        uint32_t o4[4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int c = c0 + 2 * p + hh;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t v = 0;
                if (c < c1) {
                    const uint4 u = *reinterpret_cast<const uint4*>(row + c * 32 + h * 16);
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) v |= ((wd[j] >> (8 * t)) & 0xFFu) << (8 * j);
                }
                o4[hh * 2 + h] = v;
            }
        }
        out[it] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
}

// One (block, q, g) metadata slot per thread: the 2 cpw records of row R's
// chunks of the warp's range, zero past it and in the padding.
__global__ void w13_meta_blocks_kernel(const uint8_t* __restrict__ meta, int MB, int E, int I, int K,
                                       uint8_t* __restrict__ out) {
    const int Kc = K / 64, cpw = moe_w13_cpw(K), gpr = K / 32, no = I / 8, ms = moe_w13_meta_stride(K, MB);
    const size_t slots = (size_t)E * no * kMoeKSplit * 2 * 8;
    for (size_t it = (size_t)blockIdx.x * blockDim.x + threadIdx.x; it < slots; it += (size_t)gridDim.x * blockDim.x) {
        const int g = (int)(it % 8);
        size_t rest = it / 8;
        const int q = (int)(rest % 2);
        rest /= 2;
        const int ks = (int)(rest % kMoeKSplit);
        rest /= kMoeKSplit;
        const int o = (int)(rest % no);
        const size_t e = rest / no;
        const int c0 = ks * cpw, c1 = min(Kc, c0 + cpw);
        const size_t R = (size_t)(q == 0 ? 8 * o + g : I + 8 * o + g);
        const uint8_t* src = meta + ((e * 2 * I + R) * gpr + 2 * (size_t)c0) * MB;
        uint8_t* dst = out + it * ms;
        const int nb = 2 * max(0, c1 - c0) * MB;
        for (int b = 0; b < ms; ++b) dst[b] = b < nb ? src[b] : 0;
    }
}
}  // namespace

cudaError_t repack_moe_w13_blocks(const uint8_t* w, const uint8_t* meta, int meta_bytes, int E, int I, int K,
                                  uint8_t* w_out, uint8_t* meta_out, cudaStream_t s) {
    if (K % 64 || I % 8 || E < 1) return cudaErrorInvalidValue;
    const size_t items = moe_w13_bank_bytes(E, I, K) / 16;
    w13_blocks_kernel<<<(unsigned)std::min<size_t>((items + 255) / 256, 65535), 256, 0, s>>>(
        w, E, I, K, reinterpret_cast<uint4*>(w_out));
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    const size_t slots = (size_t)E * (I / 8) * kMoeKSplit * 16;
    w13_meta_blocks_kernel<<<(unsigned)std::min<size_t>((slots + 255) / 256, 65535), 256, 0, s>>>(
        meta, meta_bytes, E, I, K, meta_out);
    return cudaPeekAtLastError();
}

// The handle's banks: codes lane-sliced ([E, N, Kr/2] bytes, every 16-byte
// unit transposed), records as in the checkpoint ([E, N, Kr/32] records).
cudaError_t repack_moe(const uint8_t* w, const uint8_t* meta, int meta_bytes, int E, int N, int Kr,
                       uint8_t* w_out, uint8_t* meta_out, cudaStream_t s) {
    const size_t bytes = (size_t)E * N * (Kr / 2);
    if (bytes % 16) return cudaErrorInvalidValue;
    const size_t units = bytes / 16;
    const int grid = (int)std::min<size_t>((units + 255) / 256, 65535);
    slice_units_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(w), reinterpret_cast<uint4*>(w_out), units);
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    return cudaMemcpyAsync(meta_out, meta, (size_t)E * N * (Kr / 32) * meta_bytes, cudaMemcpyDeviceToDevice, s);
}

QMLP_BOUNDS_UNIT(moe_awq)

}  // namespace qmlp
