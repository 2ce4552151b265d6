// common.cuh -- device primitives shared by the qmlp kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define QMLP_DEV __device__ __forceinline__

namespace qmlp {

// ---------------------------------------------------------------------------
// Element conversions (exact).
// E2M1 pair -> f16x2: the byte holds the earlier k in its low nibble, which
// lands in the low half (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented").
// ---------------------------------------------------------------------------
QMLP_DEV void e2m1x4_to_f16x2x4(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                uint32_t& h3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.
QMLP_DEV uint32_t e4m3x2_to_f16x2(uint32_t w16) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(r)
        : "r"(w16));
    return r;
}

// Four E4M3 bytes of a word -> two f16x2 (bytes 0,1 -> first; 2,3 -> second).
QMLP_DEV void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

QMLP_DEV uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// {x.lo, x.lo} and {x.hi, x.hi}
QMLP_DEV uint32_t dup_lo16(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
QMLP_DEV uint32_t dup_hi16(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

// ---------------------------------------------------------------------------
// Warp-level tensor-core MMA: D[16x8] += A[16x16] (f16, row) * B[16x8] (f16,
// col), fp32 accumulation.
// ---------------------------------------------------------------------------
QMLP_DEV void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                            uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA on a zero accumulator: d = A * B (independent of any earlier
// MMA, so consecutive groups do not form a dependency chain).
QMLP_DEV void mma_f16_16816_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                               uint32_t b1) {
    const float z = 0.0f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------
// Streaming 16-byte global load: read once, do not keep in L1.
QMLP_DEV uint4 ldg_stream_u4(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
QMLP_DEV uint2 ldg_stream_u2(const uint2* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

QMLP_DEV float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// Exponent that brings max|v| into [2^14, 2^15): fp16 then holds every bf16
// value within 2^29 of the maximum exactly (bf16 has 8 significant bits,
// fp16 11). Zero/non-finite maxima get 0.
// e with maxabs in [2^(e-1), 2^e) read from the IEEE fields: a normal
// float's biased exponent b gives e = b - 126; a subnormal m * 2^-149 gives
// e = (bit length of m) - 149.
QMLP_DEV int prescale_exponent(float maxabs) {
    const int bits = __float_as_int(maxabs);
    if (bits <= 0 || bits >= 0x7f800000) return 0;  // zero, negative, inf, nan
    const int b = bits >> 23;
    const int e = b ? b - 126 : (32 - __clz(bits)) - 149;
    return 15 - e;
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-async (TMA) copies
// ---------------------------------------------------------------------------
QMLP_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

QMLP_DEV void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
QMLP_DEV void mbar_inval(uint32_t bar) { asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory"); }
QMLP_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
QMLP_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
QMLP_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
QMLP_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase `parity` of an mbarrier; gives up after `limit_ns`.
QMLP_DEV bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}
// Bulk copy global -> shared (this CTA), completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
QMLP_DEV void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream start
// its CTAs / wait until the previous kernel has completed and its memory is
// visible (both are no-ops for kernels launched without the attribute).
QMLP_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
QMLP_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier over `nthreads` threads (a multiple of 32) of the CTA.
QMLP_DEV void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
QMLP_DEV void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------------------
// Index checks: a build with -DQMLP_DEBUG_BOUNDS checks the index of every
// global access whose address the kernels compute from layout arithmetic or
// runtime data against the size of its buffer (QMLP_INB); the default build
// compiles the checks away. A failed check records (site << 48 | index) in
// this translation unit's bounds word -- the first failure wins -- and the
// caller skips the access: a load reads zero, a store is dropped, a bulk copy
// is taken from the start of its buffer so that its barrier still completes.
// No check traps. The host reads and clears the words (qmlp_debug_bounds).
// Sites are numbered per file (gemv_split 1-9, gemm_tc 11-19, gemv_stream and
// gemv_dec 21-29, moe_awq 31-39, moe_grouped 41-49, tp_shard 51-59).
// ---------------------------------------------------------------------------
#ifdef QMLP_DEBUG_BOUNDS
static __device__ unsigned long long g_bounds_word;
QMLP_DEV bool bounds_ok(long long idx, long long lim, int site) {
    if (idx >= 0 && idx < lim) return true;
    atomicCAS(&g_bounds_word, 0ull, ((unsigned long long)site << 48) | ((unsigned long long)idx & 0xffffffffffffull));
    return false;
}
#define QMLP_INB(idx, lim, site) (::qmlp::bounds_ok((long long)(idx), (long long)(lim), (site)))
// The unit's host-side reader: returns the word and clears it.
#define QMLP_BOUNDS_UNIT(name)                                                        \
    cudaError_t bounds_take_##name(unsigned long long* v) {                           \
        cudaError_t e = cudaMemcpyFromSymbol(v, g_bounds_word, sizeof(*v));           \
        if (e != cudaSuccess) return e;                                               \
        const unsigned long long z = 0;                                               \
        return cudaMemcpyToSymbol(g_bounds_word, &z, sizeof(z));                      \
    }
#else
#define QMLP_INB(idx, lim, site) true
#define QMLP_BOUNDS_UNIT(name)                              \
    cudaError_t bounds_take_##name(unsigned long long* v) { \
        *v = 0;                                             \
        return cudaSuccess;                                 \
    }
#endif

}  // namespace qmlp
