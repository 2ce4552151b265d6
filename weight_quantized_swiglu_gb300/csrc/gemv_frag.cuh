// gemv_frag.cuh -- fragment-layout helpers shared by the GEMV kernels.
//
// Weight layout (built at create time, see gemv_dec.cu), one record per
// chunk u (16 rows x 64 k), records contiguous in row-tile-major order:
//   NVFP4 (576 B): 32 lanes x 16 B of E2M1 bytes, lane (g = lane/4,
//          t = lane%4) holding for each of the 4 k16 groups the bytes of
//          (row g, k 2t..2t+1), (row g+8, same), (row g, k 8+2t..),
//          (row g+8, k 8+2t..) = the m16n8k16 A fragment; then 8 row pairs x
//          8 B of E4M3 scales (row g, row g+8) x 4 groups.
//   FP8 (1024 B): 2 x 32 lanes x 16 B of e4m3fn bytes in the same order.
// Activation staging: x[m, k] as fp16 scaled by 2^sigma[m] in B-fragment
// order, slots [chunk][half][4*M]: slot (m, t) of a half holds the k pairs
// (2t, 2t+1) and (8+2t, 9+2t) of two k16 groups.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace qmlp {

// Weights of one chunk of one projection, as loaded.
struct ChunkW {
    uint4 w0;  // NVFP4: the 4 groups; FP8: groups 0,1
    uint4 w1;  // FP8: groups 2,3
    uint2 s;   // NVFP4 scales
};

constexpr int kRecNVFP4 = 576;
constexpr int kRecFP8 = 1024;
template <int FMT>
constexpr int rec_bytes() { return FMT == kNVFP4 ? kRecNVFP4 : kRecFP8; }

// One chunk record from global memory (streaming loads).
template <int FMT>
QMLP_DEV ChunkW load_chunk(const uint8_t* wc, size_t chunk, int Lr, int TWr, int Rr, int lane) {
    ChunkW c;
    const uint8_t* r = wc + gemv_rec_pos(chunk, Lr, TWr, Rr) * rec_bytes<FMT>();
    if (FMT == kNVFP4) {
        c.w0 = ldg_stream_u4(reinterpret_cast<const uint4*>(r) + lane);
        c.s = ldg_stream_u2(reinterpret_cast<const uint2*>(r + 512) + (lane >> 2));
        c.w1 = make_uint4(0, 0, 0, 0);
    } else {
        c.w0 = ldg_stream_u4(reinterpret_cast<const uint4*>(r) + lane);
        c.w1 = ldg_stream_u4(reinterpret_cast<const uint4*>(r + 512) + lane);
        c.s = make_uint2(0, 0);
    }
    return c;
}

// One chunk record from shared memory.
template <int FMT>
QMLP_DEV ChunkW lds_chunk(const uint8_t* r, int lane) {
    ChunkW c;
    if (FMT == kNVFP4) {
        c.w0 = reinterpret_cast<const uint4*>(r)[lane];
        c.s = reinterpret_cast<const uint2*>(r + 512)[lane >> 2];
        c.w1 = make_uint4(0, 0, 0, 0);
    } else {
        c.w0 = reinterpret_cast<const uint4*>(r)[lane];
        c.w1 = reinterpret_cast<const uint4*>(r + 512)[lane];
        c.s = make_uint2(0, 0);
    }
    return c;
}

QMLP_DEV uint32_t u4_word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Group j (16 k) of a chunk -> the four f16x2 A-fragment registers, exact:
// NVFP4 E2M1 -> f16x2, times the group's E4M3 scale (<= 6 significant bits,
// exact in fp16); FP8 e4m3fn -> f16x2.
template <int FMT>
QMLP_DEV void decode_group(const ChunkW& c, int j, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    if (FMT == kNVFP4) {
        e2m1x4_to_f16x2x4(u4_word(c.w0, j), a0, a1, a2, a3);
        const uint32_t sp = e4m3x2_to_f16x2((j < 2 ? c.s.x : c.s.y) >> (16 * (j & 1)));
        const uint32_t slo = dup_lo16(sp), shi = dup_hi16(sp);
        a0 = hmul2_u32(a0, slo);
        a1 = hmul2_u32(a1, shi);
        a2 = hmul2_u32(a2, slo);
        a3 = hmul2_u32(a3, shi);
    } else {
        const uint4& v = j < 2 ? c.w0 : c.w1;
        const int jj = j & 1;
        e4m3x4_to_f16x2x2(u4_word(v, jj * 2 + 0), a0, a1);
        e4m3x4_to_f16x2x2(u4_word(v, jj * 2 + 1), a2, a3);
    }
}

// Decode + MMA of one chunk for NP projections and NT token tiles.
//  NVFP4: each k16 group is exactly one scale group, so the MMA runs on the
//  raw E2M1 values (exact in fp16) with a zero accumulator and the group's
//  E4M3 scale (rows g and g+8) is applied in fp32 when the group product is
//  added to the running sum: acc += (A_e2m1 * B) * scale. The group
//  products are independent MMAs (no accumulator chain) and the scale costs
//  fp32 FMAs instead of f16 multiplies on the decoded weights.
//  FP8: the whole weight is the e4m3fn value; MMAs accumulate in place and
//  the per-channel scale is applied in the epilogue.
// ONE_TOKEN: M == 1, so only the accumulator elements of token 0 (c0 and
// c2 of lanes with t == 0) carry data; the others are skipped.
template <int FMT, int NT, int NP, bool ONE_TOKEN = false>
QMLP_DEV void mma_chunk(const ChunkW (&w)[NP], const uint4 (&xb)[NT][2], float (&acc)[NP][NT][4]) {
    if (FMT == kNVFP4) {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            // scales of (row g, row g+8) for groups 0..3 as fp32
            uint32_t sp[4];
            e4m3x4_to_f16x2x2(w[p].s.x, sp[0], sp[1]);
            e4m3x4_to_f16x2x2(w[p].s.y, sp[2], sp[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t a0, a1, a2, a3;
                e2m1x4_to_f16x2x4(u4_word(w[p].w0, j), a0, a1, a2, a3);
                const __half2 sh = *reinterpret_cast<const __half2*>(&sp[j]);
                const float s_lo = __low2float(sh), s_hi = __high2float(sh);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint32_t b0 = u4_word(xb[n][j >> 1], (j & 1) * 2 + 0);
                    const uint32_t b1 = u4_word(xb[n][j >> 1], (j & 1) * 2 + 1);
                    float d[4];
                    mma_f16_16816_zc(d, a0, a1, a2, a3, b0, b1);
                    acc[p][n][0] = fmaf(d[0], s_lo, acc[p][n][0]);
                    acc[p][n][2] = fmaf(d[2], s_hi, acc[p][n][2]);
                    if (!ONE_TOKEN) {
                        acc[p][n][1] = fmaf(d[1], s_lo, acc[p][n][1]);
                        acc[p][n][3] = fmaf(d[3], s_hi, acc[p][n][3]);
                    }
                }
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                uint32_t a0, a1, a2, a3;
                decode_group<FMT>(w[p], j, a0, a1, a2, a3);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint32_t b0 = u4_word(xb[n][j >> 1], (j & 1) * 2 + 0);
                    const uint32_t b1 = u4_word(xb[n][j >> 1], (j & 1) * 2 + 1);
                    mma_f16_16816(acc[p][n], a0, a1, a2, a3, b0, b1);
                }
            }
        }
    }
}

template <int NT>
QMLP_DEV void load_xfrag(const uint4* xs, int chunk, int M, int slots, int g, int t, uint4 (&xb)[NT][2]) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int m = n * 8 + g;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            xb[n][h] = m < M ? xs[(size_t)(chunk * 2 + h) * slots + m * 4 + t] : make_uint4(0, 0, 0, 0);
    }
}

// Synchronization of the threads that stage x: the whole CTA, or (when a
// producer warp must not join) the first `nth` threads via a named barrier.
QMLP_DEV void stage_sync(int nth) {
    if (nth == (int)blockDim.x) __syncthreads();
    else named_bar_sync(1, nth);
}

// Stage x[:, kb:kpe) (bf16, row stride ld) as prescaled fp16 fragments with
// the first `nth` threads of the CTA (all of them by default); k >= ke reads
// as zero. sigma[m] = exponent bringing the slice's max|x[m]| into
// [2^14, 2^15). One pass over memory: each thread keeps its (at most
// kStageRegs) 16-byte items in registers between the max and the convert;
// larger slices take a second pass. Ends with a barrier over those threads.
// REGS bounds the unrolled per-thread items: code that runs once per call is
// fetched cold, so a caller that knows its slice is small asks for fewer.
constexpr int kStageRegs = 8;

// 2^e as a float, e in [-126, 127]
QMLP_DEV float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// x * 2^sig as two multiplies by exact powers of two: for every sig the
// prescale produces ([-113, 163]) both halves are normal exponents, so the
// product is exact whenever it is a normal float (as scalbnf) and the fp16
// rounding is the only one; anything smaller rounds to zero in fp16 either way.
QMLP_DEV void stage_store8(uint4* xs, int slots, int m, int kl, int sig, const uint4& v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    const int s1 = sig / 2;
    const float f1 = pow2f(s1), f2 = pow2f(sig - s1);
    const int cc = kl / kChunkK, j = (kl % kChunkK) / 16, reg = (kl % 16) / 8;
    const int half = j >> 1, word = (j & 1) * 2 + reg;
    uint32_t* base = reinterpret_cast<uint32_t*>(xs + (size_t)(cc * 2 + half) * slots + m * 4);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(h[t]);
        const __half2 hh = __floats2half2_rn(f.x * f1 * f2, f.y * f1 * f2);
        base[t * 4 + word] = *reinterpret_cast<const uint32_t*>(&hh);
    }
}

QMLP_DEV float absmax8(const uint4& v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    return mx;
}

// 16 bytes of x: from global memory (L2, no L1 allocation) or, when x was
// first copied into shared memory, a plain load.
QMLP_DEV uint4 ld_x16(const __nv_bfloat16* p, bool smem_src) {
    return smem_src ? *reinterpret_cast<const uint4*>(p) : __ldcg(reinterpret_cast<const uint4*>(p));
}

template <int REGS = kStageRegs>
QMLP_DEV void stage_x(const __nv_bfloat16* x, int M, int ld, int kb, int ke, int kpe, uint4* xs, int* s_maxbits,
                      int* s_sig, int nth = -1, bool smem_src = false) {
    if (nth < 0) nth = blockDim.x;
    const int tid = threadIdx.x;
    const int slots = 4 * M;
    const int real8 = (ke - kb) / 8;
    const int pad8 = (kpe - kb) / 8;
    const int total = M * real8;
    const bool in_regs = total <= REGS * nth;
    uint4 v[REGS];
    if (tid < 16) s_maxbits[tid] = 0;
    // issue every load first (one memory round trip), then reduce
#pragma unroll
    for (int i = 0; i < REGS; ++i) {
        const int it = tid + i * nth;
        v[i] = make_uint4(0, 0, 0, 0);
        if (in_regs && it < total) {
            const int m = it / real8, q = it - m * real8;
            v[i] = ld_x16(x + (size_t)m * ld + kb + q * 8, smem_src);
        }
    }
    stage_sync(nth);
    // per-token max|x| (order-independent, so deterministic): fold per
    // thread, reduce per warp, one shared atomic per warp and token
    for (int m = 0; m < M; ++m) {
        float mx = 0.0f;
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < REGS; ++i) {
                const int it = tid + i * nth;
                if (it < total && it / real8 == m) mx = fmaxf(mx, absmax8(v[i]));
            }
        } else {
            for (int q = tid; q < real8; q += nth)
                mx = fmaxf(mx, absmax8(ld_x16(x + (size_t)m * ld + kb + q * 8, smem_src)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((tid & 31) == 0 && mx > 0.0f) atomicMax(&s_maxbits[m], __float_as_int(mx));
    }
    stage_sync(nth);
    if (tid < M) s_sig[tid] = prescale_exponent(__int_as_float(s_maxbits[tid]));
    stage_sync(nth);
    if (in_regs) {
#pragma unroll
        for (int i = 0; i < REGS; ++i) {
            const int it = tid + i * nth;
            if (it < total) {
                const int m = it / real8, q = it - m * real8;
                stage_store8(xs, slots, m, q * 8, s_sig[m], v[i]);
            }
        }
        // zero padding of the last chunk (k in [ke, kpe))
        const int padn = M * (pad8 - real8);
        for (int it = tid; it < padn; it += nth) {
            const int m = it / (pad8 - real8), q = real8 + it % (pad8 - real8);
            stage_store8(xs, slots, m, q * 8, 0, make_uint4(0, 0, 0, 0));
        }
    } else {
        for (int it = tid; it < M * pad8; it += nth) {
            const int m = it / pad8, q = it - m * pad8;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (q < real8) w = ld_x16(x + (size_t)m * ld + kb + q * 8, smem_src);
            stage_store8(xs, slots, m, q * 8, s_sig[m], w);
        }
    }
    stage_sync(nth);
}

}  // namespace qmlp
