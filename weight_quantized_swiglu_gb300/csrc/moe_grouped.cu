// moe_grouped.cu -- routed-expert AWQ int4 group-32 MLP for M tokens.
//
// Operation: every token t independently computes the one-token routed
// expert step (1Cat-vLLM PR "[Kernel][SM70] Add native-g32 AWQ QPN M1
// operator", "What it does"; the PR leaves grouped decode and prefill out):
//   for each route r of t in router order with 0 <= ids[t, r] < E:
//     h       = x[t] . W13[id]^T in fp32; g, u = fp16(h[:I]), fp16(h[I:])
//     act     = fp16(SiLU(g) * u)
//     y[t, r] = fp16(act . W2[id]^T) in fp32
//   out[t] = fp16( sum over valid r, in router order, of rw[t, r] * y[t, r] )
// with the same half_fma weight decode as the one-token kernels, on the
// handle's lane-sliced banks (byte t of every 4 words is lane t's 32-bit
// word, see moe_awq.cu).
//
// GB300 design: tokens that share an expert share its weight reads.
//  * moe_route_kernel (one CTA): counting sort of the valid routes by
//    expert (shared-memory histogram, scan, scatter) and a list of groups of
//    at most 8 routes with one expert -- 16 once the routes average 8 or
//    more per expert (and K <= 4096), a group then being two sets of MMA
//    columns that share every decoded weight fragment. The order of the
//    routes inside an expert's bucket is whatever the atomics give: it does
//    not matter, because every route is one column of the MMAs below and a
//    column's result depends on nothing else in the group.
//  * moe_w13_grouped_kernel: 2-5 CTAs per group (fewer when there are many
//    groups), each looping over its share of the row octets -- 8 gate rows
//    and the matching 8 up rows as one 16-row MMA tile, so a CTA is only the
//    10 K-split warps, each with one 64-k chunk in flight (64 registers:
//    three CTAs per SM; x staged once per CTA); the group's tokens are the
//    8 (or 2 x 8) columns of the m16n8k16 MMAs (A fragments decoded as in
//    the one-token kernel), each token prescaled by its own power of two;
//    the K split over 10 warps is added in a fixed order.
//  * moe_w2_grouped_kernel: as many CTAs per group, each looping over its
//    share of the 256-row blocks, a warp per 16 rows, the group's act rows
//    as the MMA columns; y is stored as fp16.
//  * moe_combine_kernel: one thread per (token, 8 output elements, one
//    16-byte load per route) adds the token's valid routes in router order
//    (fmaf, fp32), like the one-token W2 stage.
//  * All four are chained with programmatic dependent launch; a grid sized
//    for the worst-case group count exits early past the real count.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace qmlp {
namespace {

constexpr int kGW13 = 10;  // W13 K splits: kGW13 warps per CTA, each on 8 gate + 8 up rows
constexpr int kGC13 = 1;   // 64-k chunks a W13 warp loads at once (lane-sliced banks: 4 bytes per unit and lane)
constexpr int kGG2 = 10;   // k16 groups a W2 warp loads at once
constexpr int kCols = 8;   // routes per MMA (n8); a group holds 8 or 16 routes (NC), 16 as two MMAs per A fragment
constexpr int kWideMaxK = 4096;  // 16-route groups: x of 16 tokens staged in shared memory
constexpr int kRouteThreads = 1024;
constexpr int kMaxCtasPerGroup = 5;  // CTAs per group (each loops over its share of the row octets / 256-row blocks)

struct GArgs {
    int E, K, I, M, topk;
    int gcap;  // routes per group: 8 or 16
    const uint8_t* w13;
    const uint8_t* w13_meta;
    const uint8_t* w2;
    const uint8_t* w2_meta;
    const void* x;  // [M, K]
    int x_is_bf16;
    int meta_al4;
    const int32_t* ids;  // [M, topk]
    const float* rw;     // [M, topk]
    __half* out;         // [M, K]
    __half* act_ws;      // [M * topk, I]
    __half* y_ws;        // [M * topk, K]
    int* route_list;     // [M * topk]: route indices sorted by expert
    int4* groups;        // {expert, first position in route_list, count, 0}
    int* n_groups;
    // index checks: bytes of the banks, the group list's capacity
    size_t w13_bytes, w13_meta_bytes, w2_bytes, w2_meta_bytes;
    int gmax;
};

template <int MB>
QMLP_DEV uint32_t gload_meta(const uint8_t* p, bool al4) {
    if (MB == 4 && al4) return __ldg(reinterpret_cast<const unsigned int*>(p));
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < MB; ++i) v |= (uint32_t)__ldg(p + i) << (8 * i);
    return v;
}

// {scale, scale}, {bias, bias} of one record (bias stored, or half(-zero*scale))
template <int MB>
QMLP_DEV void gmeta_sb2(uint32_t m, uint32_t& s2, uint32_t& b2) {
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

QMLP_DEV uint32_t ghfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The byte of w that `sel` picks (two u4 codes, low nibble = earlier k) ->
// f16x2 {half_fma(q_lo, s, b), half_fma(q_hi, s, b)}: the byte goes to both
// halves, 0x6400 | q is 1024 + q exactly, one exact HFMA2 gives (q_lo, q_hi),
// one HFMA2 the single-rounding half_fma.
QMLP_DEV uint32_t gawq_pair(uint32_t w, uint32_t sel, uint32_t s2, uint32_t b2) {
    const uint32_t m = __byte_perm(w, 0u, sel);
    const uint32_t h = (m & 0x00F0000Fu) | 0x64006400u;
    const uint32_t q = ghfma2(h, 0x2C003C00u, 0xD400E400u);
    return ghfma2(q, s2, b2);
}
QMLP_DEV uint32_t gpair_selector(int t) { return (uint32_t)t | (4u << 4) | ((uint32_t)t << 8) | (4u << 12); }

// ---------------------------------------------------------------------------
// routing: valid routes sorted by expert, groups of <= 8
// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one 64-bit value per thread (kRouteThreads).
QMLP_DEV unsigned long long block_excl_scan(unsigned long long v, unsigned long long* wsum,
                                            unsigned long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        unsigned long long w = wsum[lane];
        unsigned long long wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        wsum[lane] = wi - w;  // exclusive prefix of the warp totals
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    return wsum[warp] + inc - v;
}

__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const GArgs a) {
    extern __shared__ int rsm[];  // cnt[E], off[E], cur[E], goff[E]
    __shared__ unsigned long long wsum[32];
    __shared__ unsigned long long total;
    int* cnt = rsm;
    int* off = cnt + a.E;
    int* cur = off + a.E;
    int* goff = cur + a.E;
    pdl_wait();  // the ids and the workspace belong to the kernels before
    pdl_launch_dependents();
    const int n = a.M * a.topk;
    for (int e = threadIdx.x; e < a.E; e += kRouteThreads) {
        cnt[e] = 0;
        cur[e] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kRouteThreads) {
        const int id = a.ids[i];
        if (id >= 0 && id < a.E) atomicAdd(&cnt[id], 1);
    }
    __syncthreads();
    // a contiguous chunk of experts per thread: routes and groups, scanned
    // together (routes in the high word, groups in the low word)
    const int per = (a.E + kRouteThreads - 1) / kRouteThreads;
    const int e0 = min(a.E, threadIdx.x * per), e1 = min(a.E, e0 + per);
    unsigned long long mine = 0;
    const int gc = a.gcap;
    for (int e = e0; e < e1; ++e) mine += ((unsigned long long)cnt[e] << 32) + (unsigned)((cnt[e] + gc - 1) / gc);
    unsigned long long pre = block_excl_scan(mine, wsum, &total);
    for (int e = e0; e < e1; ++e) {
        off[e] = (int)(pre >> 32);
        goff[e] = (int)(pre & 0xFFFFFFFFull);
        pre += ((unsigned long long)cnt[e] << 32) + (unsigned)((cnt[e] + gc - 1) / gc);
    }
    if (threadIdx.x == 0) *a.n_groups = (int)(total & 0xFFFFFFFFull);
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kRouteThreads) {
        const int id = a.ids[i];
        if (id >= 0 && id < a.E) {
            const int pos = off[id] + atomicAdd(&cur[id], 1);
            if (QMLP_INB(pos, n, 41)) a.route_list[pos] = i;
        }
    }
    for (int e = e0; e < e1; ++e)
        for (int j = 0; j * gc < cnt[e]; ++j)
            if (QMLP_INB(goff[e] + j, a.gmax, 42))
                a.groups[goff[e] + j] = make_int4(e, off[e] + j * gc, min(gc, cnt[e] - j * gc), 0);
}

// ---------------------------------------------------------------------------
// W13 + SwiGLU for a group of routes sharing one expert
// ---------------------------------------------------------------------------
template <int MB, int NC>
__global__ void __launch_bounds__(kGW13 * 32, 3) moe_w13_grouped_kernel(const GArgs a) {
    extern __shared__ __align__(16) uint32_t xs[];  // [NC][K/2 + 4] fp16 pairs (padded: no bank conflicts)
    __shared__ float part[kGW13][16][NC];
    __shared__ int s_route[NC];
    __shared__ int s_max[NC];
    __shared__ int s_sig[NC];
    __shared__ int s_tok[NC];  // slot's token, -1 past the group's routes
    pdl_wait();
    pdl_launch_dependents();
    if ((int)blockIdx.x >= *a.n_groups) return;
    const int4 grp = a.groups[blockIdx.x];
    const int e = grp.x, cnt = grp.z;
    if (!QMLP_INB(e, a.E, 43) || !QMLP_INB(grp.y + cnt - 1, a.M * a.topk, 43) || !QMLP_INB(cnt - 1, NC, 43)) return;
    // a group of more than 8 routes is two MMA column sets on the same A fragments
    const bool two = NC == 16 && cnt > kCols;
    const int ns = two ? 2 * kCols : kCols;  // slots staged
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int ks = warp;
    const int Kc = a.K / 64, gpr = a.K / 32, N = 2 * a.I;
    const int cpw = moe_w13_cpw(a.K);
    static_assert(kGW13 == kMoeKSplit, "the bank's warp blocks follow the K split");
    const int c0 = ks * cpw, c1 = min(Kc, c0 + cpw);
    const bool al4 = a.meta_al4 != 0;
    // this CTA's row octets tp = blockIdx.y, blockIdx.y + gridDim.y, ...:
    // gate rows 8tp..8tp+7 are MMA rows 0-7 and the matching up rows MMA
    // rows 8-15, so one warp's tile holds both halves of 8 SwiGLU outputs
    const int ntp = a.I / 8;
    size_t rows[2];
    auto set_rows = [&](int tp) {
        rows[0] = (size_t)e * N + 8 * tp + g;
        rows[1] = rows[0] + a.I;
    };
    int tp = blockIdx.y;
    set_rows(tp);
    uint32_t cs[kGC13][2][2];  // this lane's 4 bytes of the two 16-byte units of each row's chunk
    uint32_t mw[kGC13][2][2];
    // the handle's W13 bank in warp blocks (internal.h): block (e, octet tp,
    // split ks); chunk c's two words of a row half are 8 adjacent bytes
    const int np = moe_w13_pairs(a.K), ms = moe_w13_meta_stride(a.K, MB);
    auto load_batch = [&](int cb, int octet) {
        const size_t blk = ((size_t)e * (a.I / 8) + octet) * kMoeKSplit + ks;
        const uint8_t* bc = a.w13 + blk * moe_w13_block_bytes(a.K);
        const uint8_t* bm = a.w13_meta + blk * moe_w13_meta_block_bytes(a.K, MB);
        if (!QMLP_INB((blk + 1) * moe_w13_block_bytes(a.K) - 1, a.w13_bytes, 44) ||
            !QMLP_INB((blk + 1) * moe_w13_meta_block_bytes(a.K, MB) - 1, a.w13_meta_bytes, 44))
            return;
#pragma unroll
        for (int i = 0; i < kGC13; ++i) {
            const int c = cb + i;
            if (c < c1) {
                const int cc = c - c0;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint2 u = __ldg(reinterpret_cast<const uint2*>(bc + (size_t)(q * np + cc / 2) * 512 +
                                                                         lane * 16 + (cc % 2) * 8));
                    cs[i][q][0] = u.x;
                    cs[i][q][1] = u.y;
                    const uint8_t* m = bm + (q * 8 + g) * ms + cc * 2 * MB;
                    mw[i][q][0] = gload_meta<MB>(m, al4);
                    mw[i][q][1] = gload_meta<MB>(m + MB, al4);
                }
            }
        }
    };
    load_batch(c0, tp);  // the first codes are in flight while x is staged

    // the group's tokens -> fp16 pairs, each token times its own 2^sig. A
    // thread takes pairs k2 = threadIdx.x + n * blockDim.x of every slot,
    // eight slots' loads in flight together; bf16 input takes one pass for
    // the per-token maxima and one to convert.
    const int xstride = a.K / 2 + 4;
    if (threadIdx.x < NC) {
        const int r = threadIdx.x < cnt ? a.route_list[grp.y + threadIdx.x] : -1;
        s_route[threadIdx.x] = r;
        s_tok[threadIdx.x] = r >= 0 ? r / a.topk : -1;
        s_max[threadIdx.x] = 0;
    }
    __syncthreads();
    const uint32_t* xin = reinterpret_cast<const uint32_t*>(a.x);
    const int kh = a.K / 2;
    // slots [c0, c0 + 8) at pair k2 (zeros past the group's routes)
    auto load_slots = [&](int c0, int k2, uint32_t (&v)[kCols]) {
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
            const int tk = s_tok[c0 + c];
            v[c] = tk >= 0 ? xin[(size_t)tk * kh + k2] : 0u;
        }
    };
    if (a.x_is_bf16) {
#pragma unroll 1
        for (int c0 = 0; c0 < ns; c0 += kCols) {
            float mx[kCols];
#pragma unroll
            for (int c = 0; c < kCols; ++c) mx[c] = 0.0f;
            for (int k2 = threadIdx.x; k2 < kh; k2 += blockDim.x) {
                uint32_t v[kCols];
                load_slots(c0, k2, v);
#pragma unroll
                for (int c = 0; c < kCols; ++c)
                    mx[c] = fmaxf(mx[c], fmaxf(fabsf(__uint_as_float(v[c] << 16)),
                                               fabsf(__uint_as_float(v[c] & 0xFFFF0000u))));
            }
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                float m = mx[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if (lane == 0 && m > 0.0f) atomicMax(&s_max[c0 + c], __float_as_int(m));
            }
        }
        __syncthreads();
    }
    if (threadIdx.x < NC) s_sig[threadIdx.x] = a.x_is_bf16 ? prescale_exponent(__int_as_float(s_max[threadIdx.x])) : 0;
    __syncthreads();
    for (int k2 = threadIdx.x; k2 < kh; k2 += blockDim.x) {
#pragma unroll 1
        for (int c0 = 0; c0 < ns; c0 += kCols) {
            uint32_t v[kCols];
            load_slots(c0, k2, v);
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                uint32_t o = v[c];
                if (a.x_is_bf16) {
                    const int sg = s_sig[c0 + c];
                    const __half2 h = __floats2half2_rn(scalbnf(__uint_as_float(o << 16), sg),
                                                        scalbnf(__uint_as_float(o & 0xFFFF0000u), sg));
                    o = *reinterpret_cast<const uint32_t*>(&h);
                }
                xs[(c0 + c) * xstride + k2] = o;
            }
        }
    }
    __syncthreads();

    const uint32_t* xcol = xs + g * xstride;  // this lane's MMA columns = route slots g and 8 + g
    const uint32_t* xcol1 = xcol + kCols * xstride;
    for (; tp < ntp; tp += gridDim.y) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        float d1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int cb = c0; cb < c1; cb += kGC13) {
            if (cb != c0) load_batch(cb, tp);
#pragma unroll
            for (int i = 0; i < kGC13; ++i) {
                const int c = cb + i;
                if (c < c1) {
                    uint32_t s2[2][2], b2[2][2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        gmeta_sb2<MB>(mw[i][q][0], s2[q][0], b2[q][0]);
                        gmeta_sb2<MB>(mw[i][q][1], s2[q][1], b2[q][1]);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // group j: unit j/2, its words 2(j&1) (k 2t..) and 2(j&1)+1 (k 8+2t..)
                        const int h = j >> 1;
                        const uint32_t sa = gpair_selector(2 * (j & 1)), sb = gpair_selector(2 * (j & 1) + 1);
                        const int k2 = (c * 64 + 16 * j) / 2 + t;
                        const uint32_t a0 = gawq_pair(cs[i][0][h], sa, s2[0][h], b2[0][h]);
                        const uint32_t a1 = gawq_pair(cs[i][1][h], sa, s2[1][h], b2[1][h]);
                        const uint32_t a2 = gawq_pair(cs[i][0][h], sb, s2[0][h], b2[0][h]);
                        const uint32_t a3 = gawq_pair(cs[i][1][h], sb, s2[1][h], b2[1][h]);
                        mma_f16_16816(d, a0, a1, a2, a3, xcol[k2], xcol[k2 + 4]);
                        if (two) mma_f16_16816(d1, a0, a1, a2, a3, xcol1[k2], xcol1[k2 + 4]);
                    }
                }
            }
        }
        // C fragment: (row g, cols 2t, 2t+1) and (row g+8, the same cols)
        part[warp][g][2 * t] = d[0];
        part[warp][g][2 * t + 1] = d[1];
        part[warp][g + 8][2 * t] = d[2];
        part[warp][g + 8][2 * t + 1] = d[3];
        if (two) {
            part[warp][g][kCols + 2 * t] = d1[0];
            part[warp][g][kCols + 2 * t + 1] = d1[1];
            part[warp][g + 8][kCols + 2 * t] = d1[2];
            part[warp][g + 8][kCols + 2 * t + 1] = d1[3];
        }
        // the next octet's first codes go out before the reduction
        if (tp + (int)gridDim.y < ntp) {
            set_rows(tp + gridDim.y);
            load_batch(c0, tp + gridDim.y);
        }
        __syncthreads();
        if (threadIdx.x < 8 * NC) {
            const int j = threadIdx.x / NC, c = threadIdx.x % NC;
            if (c < cnt) {
                float hg = 0.0f, hu = 0.0f;
                for (int w = 0; w < kGW13; ++w) {
                    hg += part[w][j][c];
                    hu += part[w][8 + j][c];
                }
                const int sg = s_sig[c];
                const __half gh = __float2half_rn(scalbnf(hg, -sg)), uh = __float2half_rn(scalbnf(hu, -sg));
                if (QMLP_INB((size_t)s_route[c] * a.I + 8 * tp + j, (size_t)a.M * a.topk * a.I, 45))
                    a.act_ws[(size_t)s_route[c] * a.I + 8 * tp + j] =
                        __float2half_rn(silu_f32(__half2float(gh)) * __half2float(uh));
            }
        }
        __syncthreads();  // part is rewritten by the next octet
    }
}

// ---------------------------------------------------------------------------
// W2 for a group of routes sharing one expert -> y (fp16)
// ---------------------------------------------------------------------------
template <int MB, int NC>
__global__ void __launch_bounds__(16 * 32) moe_w2_grouped_kernel(const GArgs a) {
    extern __shared__ __align__(16) uint32_t acts[];  // [NC][I/2 + 4]
    __shared__ int s_route[NC];
    pdl_wait();
    pdl_launch_dependents();
    if ((int)blockIdx.x >= *a.n_groups) return;
    const int4 grp = a.groups[blockIdx.x];
    const int e = grp.x, cnt = grp.z;
    if (!QMLP_INB(e, a.E, 46) || !QMLP_INB(grp.y + cnt - 1, a.M * a.topk, 46) || !QMLP_INB(cnt - 1, NC, 46)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int astride = a.I / 2 + 4;
    const bool two = NC == 16 && cnt > kCols;  // two MMA column sets on the same A fragments
    if (threadIdx.x < NC) s_route[threadIdx.x] = threadIdx.x < cnt ? a.route_list[grp.y + threadIdx.x] : -1;
    __syncthreads();
    {
        // the group's act rows: a thread takes pairs k2 = threadIdx.x + n * blockDim.x
        // of every slot, eight slots' loads in flight together
        const int ih = a.I / 2;
        const uint32_t* act32 = reinterpret_cast<const uint32_t*>(a.act_ws);
        const int ns = two ? 2 * kCols : kCols;
        for (int k2 = threadIdx.x; k2 < ih; k2 += blockDim.x) {
#pragma unroll 1
            for (int c0 = 0; c0 < ns; c0 += kCols) {
                uint32_t v[kCols];
#pragma unroll
                for (int c = 0; c < kCols; ++c) {
                    const int r = s_route[c0 + c];
                    v[c] = r >= 0 && QMLP_INB((size_t)r * ih + k2, (size_t)a.M * a.topk * ih, 46)
                               ? act32[(size_t)r * ih + k2]
                               : 0u;
                }
#pragma unroll
                for (int c = 0; c < kCols; ++c) acts[(c0 + c) * astride + k2] = v[c];
            }
        }
    }
    __syncthreads();
    const int ng = a.I / 16, gpr = a.I / 32;
    const bool al4 = a.meta_al4 != 0;
    const uint32_t* xcol = acts + g * astride;
    const uint32_t* xcol1 = xcol + kCols * astride;
    // this CTA's 256-row blocks; warps are independent from here (no barrier)
    for (int nb = blockIdx.y; 256 * nb < a.K; nb += gridDim.y) {
    const int n0 = 256 * nb + 16 * warp;
    if (n0 >= a.K) continue;
    const size_t row0 = (size_t)e * a.K + n0 + g;
    const uint2* c0p = reinterpret_cast<const uint2*>(a.w2 + row0 * (a.I / 2));
    const uint2* c8p = reinterpret_cast<const uint2*>(a.w2 + (row0 + 8) * (a.I / 2));
    const uint8_t* m0p = a.w2_meta + row0 * gpr * MB;
    const uint8_t* m8p = a.w2_meta + (row0 + 8) * gpr * MB;
    if (!QMLP_INB((row0 + 9) * (a.I / 2) - 1, a.w2_bytes, 47) || !QMLP_INB((row0 + 9) * gpr * MB - 1, a.w2_meta_bytes, 47))
        continue;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    float d1[4] = {0.f, 0.f, 0.f, 0.f};
    for (int gb = 0; gb < ng; gb += kGG2) {
        uint32_t cs[kGG2 / 2][2];  // this lane's 4 bytes of unit (gb/2 + i): k16 groups gb+2i, gb+2i+1
        uint32_t mw[kGG2 / 2][2];
#pragma unroll
        for (int i = 0; i < kGG2 / 2; ++i) {
            if (gb + 2 * i < ng) {
                cs[i][0] = __ldg(reinterpret_cast<const unsigned int*>(c0p + gb + 2 * i) + t);
                cs[i][1] = __ldg(reinterpret_cast<const unsigned int*>(c8p + gb + 2 * i) + t);
            }
        }
#pragma unroll
        for (int i = 0; i < kGG2 / 2; ++i) {
            const int ag = gb / 2 + i;
            if (ag < gpr) {
                mw[i][0] = gload_meta<MB>(m0p + (size_t)ag * MB, al4);
                mw[i][1] = gload_meta<MB>(m8p + (size_t)ag * MB, al4);
            }
        }
#pragma unroll
        for (int i = 0; i < kGG2; ++i) {
            const int j = gb + i;
            if (j < ng) {
                uint32_t s0, b0, s8, b8;
                gmeta_sb2<MB>(mw[i / 2][0], s0, b0);
                gmeta_sb2<MB>(mw[i / 2][1], s8, b8);
                const uint32_t sa = gpair_selector(2 * (i & 1)), sb = gpair_selector(2 * (i & 1) + 1);
                const uint32_t a0 = gawq_pair(cs[i / 2][0], sa, s0, b0), a1 = gawq_pair(cs[i / 2][1], sa, s8, b8);
                const uint32_t a2 = gawq_pair(cs[i / 2][0], sb, s0, b0), a3 = gawq_pair(cs[i / 2][1], sb, s8, b8);
                mma_f16_16816(d, a0, a1, a2, a3, xcol[8 * j + t], xcol[8 * j + 4 + t]);
                if (two) mma_f16_16816(d1, a0, a1, a2, a3, xcol1[8 * j + t], xcol1[8 * j + 4 + t]);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c = 2 * t + (q & 1), row = n0 + g + 8 * (q >> 1);
        const size_t ycap = (size_t)a.M * a.topk * a.K;
        if (c < cnt && QMLP_INB((size_t)s_route[c] * a.K + row, ycap, 48))
            a.y_ws[(size_t)s_route[c] * a.K + row] = __float2half_rn(d[q]);
        if (two && kCols + c < cnt && QMLP_INB((size_t)s_route[kCols + c] * a.K + row, ycap, 48))
            a.y_ws[(size_t)s_route[kCols + c] * a.K + row] = __float2half_rn(d1[q]);
    }
    }
}

// ---------------------------------------------------------------------------
// ordered router-weighted sum per token
// ---------------------------------------------------------------------------
constexpr int kCombThr = 128;  // combine: threads per CTA, 8 output elements each

__global__ void __launch_bounds__(kCombThr) moe_combine_kernel(const GArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int tok = blockIdx.x, n = 8 * (kCombThr * blockIdx.y + threadIdx.x);
    if (n >= a.K) return;
    // every load first (16 bytes of each route's y row; an invalid route's
    // slot is read and ignored), then the sum in router order per element
    int id[16];
    float w[16];
    uint4 y[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        if (r < a.topk) {
            const int i = tok * a.topk + r;
            id[r] = a.ids[i];
            w[r] = a.rw[i];
            y[r] = QMLP_INB((size_t)i * a.K + n + 7, (size_t)a.M * a.topk * a.K, 49)
                       ? *reinterpret_cast<const uint4*>(a.y_ws + (size_t)i * a.K + n)
                       : make_uint4(0, 0, 0, 0);
        }
    }
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        if (r < a.topk && id[r] >= 0 && id[r] < a.E) {
            const __half* h = reinterpret_cast<const __half*>(&y[r]);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[r], __half2float(h[e]), acc[e]);
        }
    }
    uint4 o;
    __half* oh = reinterpret_cast<__half*>(&o);
#pragma unroll
    for (int e = 0; e < 8; ++e) oh[e] = __float2half_rn(acc[e]);
    if (QMLP_INB((size_t)tok * a.K + n + 7, (size_t)a.M * a.K, 49))
        *reinterpret_cast<uint4*>(a.out + (size_t)tok * a.K + n) = o;
}

cudaLaunchConfig_t pdl_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* at) {
    cudaLaunchConfig_t c = {};
    c.gridDim = grid;
    c.blockDim = block;
    c.dynamicSmemBytes = smem;
    c.stream = s;
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = at;
    c.numAttrs = 1;
    return c;
}

template <int MB, int NC>
cudaError_t launch_grouped_mb(const GArgs& a, int gmax, int cpg, cudaStream_t s) {
    const size_t rsmem = (size_t)4 * a.E * sizeof(int);
    const size_t xsmem = (size_t)NC * (a.K / 2 + 4) * 4;
    const size_t asmem = (size_t)NC * (a.I / 2 + 4) * 4;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kMoeGroupedMaxE * 4 * (int)sizeof(int));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(moe_w13_grouped_kernel<MB, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     NC * ((NC == kCols ? kMoeGroupedMaxK : kWideMaxK) / 2 + 4) * 4);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchAttribute at[1];
    cudaLaunchConfig_t c = pdl_cfg(dim3(1), dim3(kRouteThreads), rsmem, s, at);
    cudaError_t e = cudaLaunchKernelEx(&c, moe_route_kernel, a);
    if (e != cudaSuccess) return e;
    c = pdl_cfg(dim3(gmax, std::min(a.I / 8, cpg)), dim3(kGW13 * 32), xsmem, s, at);
    if ((e = cudaLaunchKernelEx(&c, moe_w13_grouped_kernel<MB, NC>, a)) != cudaSuccess) return e;
    c = pdl_cfg(dim3(gmax, std::min((a.K + 255) / 256, cpg)), dim3(16 * 32), asmem, s, at);
    if ((e = cudaLaunchKernelEx(&c, moe_w2_grouped_kernel<MB, NC>, a)) != cudaSuccess) return e;
    c = pdl_cfg(dim3(a.M, (a.K / 8 + kCombThr - 1) / kCombThr), dim3(kCombThr), 0, s, at);
    return cudaLaunchKernelEx(&c, moe_combine_kernel, a);
}

}  // namespace

size_t moe_grouped_max_groups(int routes, int E) { return (size_t)routes / kCols + 1 + (size_t)std::min(E, routes); }

cudaError_t launch_moe_grouped(const MoeGroupedLaunch& L, cudaStream_t s) {
    if (L.M < 1 || L.topk < 1 || L.topk > 16 || L.K % 64 || L.I % 32 || L.K > kMoeGroupedMaxK ||
        L.E > kMoeGroupedMaxE || L.E < 1)
        return cudaErrorInvalidValue;
    GArgs a;
    a.E = L.E;
    a.K = L.K;
    a.I = L.I;
    a.M = L.M;
    a.topk = L.topk;
    a.w13 = L.w13;
    a.w13_meta = L.w13_meta;
    a.w2 = L.w2;
    a.w2_meta = L.w2_meta;
    a.x = L.x;
    a.x_is_bf16 = L.x_is_bf16;
    a.meta_al4 = ((reinterpret_cast<uintptr_t>(L.w13_meta) | reinterpret_cast<uintptr_t>(L.w2_meta)) & 3u) == 0;
    a.ids = L.ids;
    a.rw = L.rw;
    a.out = L.out;
    a.act_ws = L.act_ws;
    a.y_ws = L.y_ws;
    a.route_list = L.route_list;
    a.groups = L.groups;
    a.n_groups = L.n_groups;
    const int routes = L.M * L.topk;
    const int gmax = (int)moe_grouped_max_groups(routes, L.E);
    a.gmax = gmax;
    a.w13_bytes = moe_w13_bank_bytes(L.E, L.I, L.K);
    a.w13_meta_bytes = moe_w13_meta_bank_bytes(L.E, L.I, L.K, L.meta_bytes);
    a.w2_bytes = (size_t)L.E * L.K * (L.I / 2);
    a.w2_meta_bytes = (size_t)L.E * L.K * (L.I / 32) * L.meta_bytes;
    // 16-route groups once experts average 8 routes or more: each decoded
    // weight fragment then feeds two MMAs
    const bool wide = L.K <= kWideMaxK && routes >= kCols * L.E;
    a.gcap = wide ? 2 * kCols : kCols;
    // CTAs per group: about four waves' worth of CTAs in all, counting the
    // worst-case group count, and at least 2 (measured at E=512 top-10: M=16
    // 64.9 us with 4 per group, 72.1 with 5; M=512 302.9 us with 2, 314.7
    // with 1; with three W13 CTAs per SM, M=512 258 us with 2, 267 with 3,
    // 269 with 4)
    const int sms = std::max(1, L.num_sms);
    const int cpg = std::max(2, std::min(kMaxCtasPerGroup, (4 * sms + gmax - 1) / gmax));
    if (L.meta_bytes == 4)
        return wide ? launch_grouped_mb<4, 2 * kCols>(a, gmax, cpg, s) : launch_grouped_mb<4, kCols>(a, gmax, cpg, s);
    return wide ? launch_grouped_mb<3, 2 * kCols>(a, gmax, cpg, s) : launch_grouped_mb<3, kCols>(a, gmax, cpg, s);
}

QMLP_BOUNDS_UNIT(moe_grouped)

}  // namespace qmlp
