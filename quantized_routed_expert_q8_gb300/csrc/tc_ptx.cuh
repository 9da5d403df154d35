// Inline-PTX wrappers shared by the tensor-core kernels: mbarriers (bounded
// waits), TMA, tcgen05 descriptors / MMA / commit / fences, packed fp32 pairs,
// and the int8 / 4-bit / 2-bit -> binary16 conversions (exact: every value is a
// small integer).  Written from the PTX ISA's descriptions of the instructions.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {
namespace tc {

// every wait on another role gives up after ~2 s of SM cycles
constexpr long long TIMEOUT_CYCLES = 1LL << 32;

// ------------------------------------------------------------------ PTX ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase (mbarrier.try_wait may suspend the thread for a
// system-dependent time; test_wait never does).  Used by the threads that poll
// several barriers in turn: the TMA producer and the MMA issuer.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware (up to ~20 us) until
// the phase completes instead of spinning on the issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete; false on abort or timeout.  The
// thread may sleep in hardware until the phase completes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_test_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > TIMEOUT_CYCLES) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Two phases (the second only if need2), both probed before either wait.
__device__ __forceinline__ bool mbar_wait2(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2,
                                           bool need2, volatile int* abort_flag) {
    bool d1 = mbar_test_wait(b1, p1);
    bool d2 = !need2 || mbar_test_wait(b2, p2);
    if (d1 && d2) return true;
    long long t0 = clock64();
    while (true) {
        if (!d1) d1 = mbar_try_wait_sleep(b1, p1);
        if (d1 && !d2) d2 = mbar_try_wait_sleep(b2, p2);
        if (d1 && d2) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > TIMEOUT_CYCLES) {
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void tma_2d(const CUtensorMap* m, uint32_t bar, uint32_t dst, int c0,
                                       int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(dst),
        "l"(m), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_3d(const CUtensorMap* m, uint32_t bar, uint32_t dst, int c0,
                                       int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4, %5}], [%2];" ::"r"(dst),
        "l"(m), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_4d(const CUtensorMap* m, uint32_t bar, uint32_t dst, int c0,
                                       int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4, %5, %6}], [%2];" ::"r"(dst),
        "l"(m), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// tcgen05 shared-memory matrix descriptor: no swizzle, K-major core matrices of
// 8 rows x 16 bytes; lbo = byte step between K-adjacent core matrices, sbo =
// byte step between 8-row groups.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version of the tcgen05 family
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M x N.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Four 16-column TMEM loads (columns ta, ta + 16 of one matrix and tb, tb + 16
// of the other) and the wait for them in one statement, so the registers are
// defined only once the data has landed.
__device__ __forceinline__ void tmem_ld16x4_wait(uint32_t ta, uint32_t tb, uint32_t (&r)[4][16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, "
        "%8, %9, %10, %11, %12, %13, %14, %15}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, "
        "%24, %25, %26, %27, %28, %29, %30, %31}, [%65];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32, %33, %34, %35, %36, %37, %38, %39, "
        "%40, %41, %42, %43, %44, %45, %46, %47}, [%66];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%48, %49, %50, %51, %52, %53, %54, %55, "
        "%56, %57, %58, %59, %60, %61, %62, %63}, [%67];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]),
          "=r"(r[0][6]), "=r"(r[0][7]), "=r"(r[0][8]), "=r"(r[0][9]), "=r"(r[0][10]), "=r"(r[0][11]),
          "=r"(r[0][12]), "=r"(r[0][13]), "=r"(r[0][14]), "=r"(r[0][15]), "=r"(r[1][0]), "=r"(r[1][1]),
          "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]), "=r"(r[1][6]), "=r"(r[1][7]),
          "=r"(r[1][8]), "=r"(r[1][9]), "=r"(r[1][10]), "=r"(r[1][11]), "=r"(r[1][12]), "=r"(r[1][13]),
          "=r"(r[1][14]), "=r"(r[1][15]), "=r"(r[2][0]), "=r"(r[2][1]), "=r"(r[2][2]), "=r"(r[2][3]),
          "=r"(r[2][4]), "=r"(r[2][5]), "=r"(r[2][6]), "=r"(r[2][7]), "=r"(r[2][8]), "=r"(r[2][9]),
          "=r"(r[2][10]), "=r"(r[2][11]), "=r"(r[2][12]), "=r"(r[2][13]), "=r"(r[2][14]), "=r"(r[2][15]),
          "=r"(r[3][0]), "=r"(r[3][1]), "=r"(r[3][2]), "=r"(r[3][3]), "=r"(r[3][4]), "=r"(r[3][5]),
          "=r"(r[3][6]), "=r"(r[3][7]), "=r"(r[3][8]), "=r"(r[3][9]), "=r"(r[3][10]), "=r"(r[3][11]),
          "=r"(r[3][12]), "=r"(r[3][13]), "=r"(r[3][14]), "=r"(r[3][15])
        : "r"(ta), "r"(ta + 16), "r"(tb), "r"(tb + 16)
        : "memory");
}

// Packed fp32 pairs in 64-bit registers (two IEEE round-to-nearest operations
// per instruction); element 0 in the low half.
__device__ __forceinline__ uint64_t pk2(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
    uint32_t a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(v));
    lo = __uint_as_float(a);
    hi = __uint_as_float(b);
}
__device__ __forceinline__ uint64_t mul2u(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2u(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// fp16 pair with bits 0x64XX holds 1024 + XX; subtract a constant pair
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    __half2 x = *reinterpret_cast<__half2*>(&a);
    __half2 y = *reinterpret_cast<__half2*>(&b);
    __half2 r = __hsub2(x, y);
    return *reinterpret_cast<uint32_t*>(&r);
}

constexpr uint32_t MAGIC = 0x64646464u;    // 0x64 high bytes: fp16 1024 + low byte
constexpr uint32_t H1152 = 0x64806480u;    // fp16 (1152, 1152)
constexpr uint32_t H1024 = 0x64006400u;    // fp16 (1024, 1024)

// 4 int8 (one word) -> fp16 pairs (q0,q1), (q2,q3), in element order
__device__ __forceinline__ void cvt_i8x4(uint32_t w, uint32_t& h01, uint32_t& h23) {
    uint32_t u = w ^ 0x80808080u;  // q + 128 as unsigned bytes
    h01 = hsub2_bits(prmt(u, MAGIC, 0x4140u), H1152);
    h23 = hsub2_bits(prmt(u, MAGIC, 0x4342u), H1152);
}

// 8 int8 in two words -> fp16 pairs in the order (x0,x4) (x1,x5) (x2,x6) (x3,x7),
// the within-8 order the 4-bit weights unpack to
__device__ __forceinline__ void cvt_i8x8_interleaved(uint32_t a, uint32_t b, uint32_t (&h)[4]) {
    uint32_t ua = a ^ 0x80808080u, ub = b ^ 0x80808080u;
    uint32_t t0 = prmt(ua, ub, 0x5140u), t1 = prmt(ua, ub, 0x7362u);
    h[0] = hsub2_bits(prmt(t0, MAGIC, 0x4140u), H1152);
    h[1] = hsub2_bits(prmt(t0, MAGIC, 0x4342u), H1152);
    h[2] = hsub2_bits(prmt(t1, MAGIC, 0x4140u), H1152);
    h[3] = hsub2_bits(prmt(t1, MAGIC, 0x4342u), H1152);
}

// 8 nibbles (byte j = element 2j low, 2j+1 high) -> (e0,e4) (e1,e5) (e2,e6) (e3,e7)
__device__ __forceinline__ void cvt_u4x8(uint32_t w, uint32_t (&h)[4]) {
    h[0] = hsub2_bits((w & 0x000F000Fu) | H1024, H1024);
    h[1] = hsub2_bits(((w >> 4) & 0x000F000Fu) | H1024, H1024);
    h[2] = hsub2_bits(((w >> 8) & 0x000F000Fu) | H1024, H1024);
    h[3] = hsub2_bits(((w >> 12) & 0x000F000Fu) | H1024, H1024);
}

// 16 2-bit codes c (one word: byte j holds elements 4j..4j+3, element 4j+i in
// bits 2i..2i+1) -> fp16 pairs of c - 2: a = (e0,e4) (e1,e5) (e2,e6) (e3,e7) and
// b = (e8,e12) (e9,e13) (e10,e14) (e11,e15), the within-8 order of the 4-bit path
constexpr uint32_t H1026 = 0x64026402u;  // fp16 (1026, 1026)
__device__ __forceinline__ void cvt_u2x16(uint32_t w, uint32_t (&a)[4], uint32_t (&b)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t t = (w >> (2 * k)) & 0x03030303u;  // codes of elements k, 4+k, 8+k, 12+k
        a[k] = hsub2_bits(prmt(t, MAGIC, 0x4140u), H1026);
        b[k] = hsub2_bits(prmt(t, MAGIC, 0x4342u), H1026);
    }
}

// As cvt_u2x16 for Q2_K: the 16 codes of one sub-block times its scale sc,
// fp16 pairs of c * sc in the same order.  (1024 + c) * sc - 1024 * sc is one
// fused operation whose exact value c * sc <= 45 is representable, so the
// single rounding returns it exactly.
__device__ __forceinline__ void cvt_u2x16_scaled(uint32_t w, uint32_t sc, uint32_t (&a)[4],
                                                 uint32_t (&b)[4]) {
    const __half hs = __uint2half_rn(sc);  // sc <= 15: exact
    const __half2 m2 = __halves2half2(hs, hs);
    const __half hb = __hneg(__hmul(__ushort_as_half((unsigned short)0x6400u), hs));  // -1024 * sc, exact
    const __half2 b2 = __halves2half2(hb, hb);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t t = (w >> (2 * k)) & 0x03030303u;
        uint32_t xa = prmt(t, MAGIC, 0x4140u), xb = prmt(t, MAGIC, 0x4342u);
        __half2 ra = __hfma2(*reinterpret_cast<__half2*>(&xa), m2, b2);
        __half2 rb = __hfma2(*reinterpret_cast<__half2*>(&xb), m2, b2);
        a[k] = *reinterpret_cast<uint32_t*>(&ra);
        b[k] = *reinterpret_cast<uint32_t*>(&rb);
    }
}

// byte offset of (row, 16-byte chunk c) in the fp16 K-major operand layout:
// [row/8][chunk 0..3][row%8][16 B]  (lbo = 128, sbo = 512)
__device__ __forceinline__ uint32_t f16_off(int row, int c) {
    return (uint32_t)((row >> 3) * 512 + c * 128 + (row & 7) * 16);
}

}  // namespace tc
}  // namespace moe
