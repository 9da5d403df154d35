// Stages 4 and 6 on the fifth-generation tensor cores with the block scales
// folded into the operands (tcgen05 with the A operand in tensor memory).
//
// The MMQ product of the pull-request pages ("#439 prefill: a group's expert
// gathers in one launch", "What": the MMQ group's products run on the gathered
// group buffers; "#1368 ...", intro: the q8_1 activations are expert-sorted
// rows) is, for the expert at active position p and its rows r:
//     acc[r, j] = sum over 32-blocks b of  dW[j,b] * dx[r,b] * I_b[r,j]
//                 (+ mW[j,b] * sx[r,b] for Q4_1),    I_b = the block's integer dot,
// which is the plain dot product  sum over k of (dW*qW)[j,k] * (dx*qx)[r,k]
// (+ the m term) of the dequantized values.  A dequantized value d*q -- a
// binary16 d times an integer |q| <= 127 -- has at most 18 significant bits,
// so it splits exactly into a binary16 pair hi + lo: hi = RN(d*q), and
// lo = d*q - hi is formed without error by one fused multiply-add (the
// residual is a multiple of ulp(d) smaller than half an ulp of hi).  Then
//     acc = sum over k of (Wh*Xh + Wl*Xh + Wh*Xl)      (Wl*Xl < 2^-22 relative: dropped)
// is three fp16 MMAs with fp32 accumulation over the whole reduction, held in
// TMEM: the per-block scaling never touches the CUDA cores.  Q2_0 values
// (d times c - 2 in [-2, 1]) are exact in one binary16, so they need two
// MMAs.  The Q4_1 m term, sum over b of mW[j,b] * sx[r,b], is one more MMA per
// 16 blocks over the binary16 (mW, sx) pairs (each product exact in fp32).
// The fp32 result differs from the scalar definition's order of rounding by a
// few units in the last place of fp32.  |d*q| must stay below 65520 (the
// binary16 range): a block beyond it sets MOE_DEV_ERR_RANGE.
//
// One persistent CTA of 23 warps per SM.  A work item is up to 128 tokens of
// one expert times two 128-row weight matrices (gate and up rows j0..j0+127 for
// stage 4; down rows i0..i0+255 for stage 6); items come from an atomic ticket
// over the device-built, longest-first work list.  Roles, connected by
// mbarrier full/empty rings:
//   scheduler (warp 21): takes tickets, publishes items to a 4-entry ring;
//   weight converters (warps 8-15, one per TMEM lane quarter and matrix):
//     lane = weight row, per block the raw row -> binary16 hi and lo of d*q,
//     written to the A stage in TMEM with tcgen05.st;
//   token converters (warps 16-19): lane = token, per block the q8_1 row ->
//     hi and lo, written to the B stage in shared memory (K-major);
//   MMA issuers (warp 20 for matrix 0, warp 22 for matrix 1): per block 2
//     K-steps x 3 terms of (M=128, N=tokens rounded to 16, K=16) into the
//     matrix's half of one 256-column accumulator; each commits on its own,
//     the operand, m-term and accumulator barriers count both, and one
//     issuer's barrier probes and commits overlap the other's MMAs;
//   epilogue (warps 0-7): once per item, the accumulator -> a shared-memory
//     staging buffer (the accumulator is released as soon as it is copied),
//     SiLU(g)*u for stage 4, then one bulk copy per output row; the CMB
//     instantiation (stage 6 with the top-k combine) stores the rows with
//     generic stores instead, counts each row's token down and combines the
//     tokens whose last row the item wrote.
// Every wait is bounded: on timeout the kernel sets MOE_DEV_ERR_TIMEOUT,
// drains what it started and exits.
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "mmq.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace fold {

using namespace tc;

constexpr int BM = 128;   // weight rows per matrix (TMEM lanes)
constexpr int BN = 128;   // tokens per work item at most
constexpr int AS = 3;     // operand stages (A in TMEM, B in shared memory)
constexpr int MS = 2;     // Q4_1 m-term stages
constexpr int MCH = 16;   // blocks per m-term MMA (its K = 16)
constexpr int IR = 4;     // work-item ring

constexpr int EPI_WARPS = 8;
constexpr int WCVT_WARP0 = 8, WCVT_WARPS = 8;    // (lane quarter, matrix)
constexpr int XCVT_WARP0 = 16, XCVT_WARPS = 4;   // 32 tokens each
constexpr int CVT_WARPS = WCVT_WARPS + XCVT_WARPS;
// two MMA issuers, one per matrix (warps 20 and 22), so that one's barrier
// probes and commits overlap the other's MMAs
constexpr int MMA_WARP = 20, SCHED_WARP = 21, MMA_WARP2 = 22, MMA_ISSUERS = 2;
constexpr int THREADS = 23 * 32;

// tensor memory columns
constexpr uint32_t T_ACC = 0;                // [matrix][BN token columns]
constexpr uint32_t T_A = 2 * BN;             // AS x [matrix][hi 16 | lo 16]
constexpr uint32_t T_M = T_A + AS * 64;      // MS x [matrix][8]
static_assert(T_M + MS * 16 <= 512, "tensor memory budget");

// shared memory (offsets from a 1024-byte aligned base)
constexpr int XT = BN * 64;                       // binary16 token tile [128][32]
constexpr int O_B = 0;                            // AS x (Xh, Xl)
constexpr int O_BM = O_B + AS * 2 * XT;           // MS x (sx) [128][16] binary16
constexpr int O_STAGE = O_BM + MS * BN * 32;      // [128 tokens][256] fp32
constexpr int STAGE_W = 2 * BM;                   // floats per staging row
constexpr int O_BAR = O_STAGE + BN * STAGE_W * 4;
constexpr int B_IF = 0, B_IE = IR, B_OF = 2 * IR, B_OE = B_OF + AS, B_MF = B_OE + AS,
              B_ME = B_MF + MS, B_AF = B_ME + MS, B_AE = B_AF + 1, B_EPI = B_AE + 1,
              N_BARS = B_EPI + 1;
constexpr int O_RING = O_BAR + ((N_BARS * 8 + 16 + 15) / 16) * 16;
// down with the combine: [0] count, [1..BN] tokens whose rows are all written
constexpr int O_LIST = O_RING + IR * 16;
constexpr int SMEM = O_LIST + (BN + 1) * 4 + 1024;  // + alignment slack
static_assert(SMEM <= 232448, "shared memory per block");

// binary16 |d| at or above which d*q_max reaches 65520 (overflows binary16)
template <int WT>
struct Range {
    static constexpr float W = WT == MOE_W_Q8_0 ? 65520.0f / 127.0f
                               : WT == MOE_W_Q4_1 ? 65520.0f / 15.0f
                                                  : 65520.0f / 2.0f;
};
constexpr float X_RANGE = 65520.0f / 127.0f;

struct Params {
    const uint8_t* group_base;
    size_t slot_stride;
    size_t mat_off[2];   // byte offsets of the item's two matrices in a record
    size_t q_off, d_off, m_off;  // plane offsets within a matrix
    int row_bytes;       // quant bytes per weight row
    int wrows;           // rows of the weight matrix (scale-plane stride)
    int mat1_row;        // weight row of matrix 1 relative to matrix 0's
    const int4* tiles;
    const int32_t* n_tiles;
    int32_t* ticket;
    int mt_count;        // weight-row tiles per token tile
    int nb;              // 32-blocks of the reduction
    int klen;            // reduction length (q row length)
    int n_out;           // output row length
    const int8_t* xq;    // [R][klen]
    const uint32_t* xds; // [R][nb] (d, s) binary16 pairs
    float* out;          // [R][n_out]
    uint32_t* err;
    // down with the top-k combine: the combined output, the row -> token and
    // token -> row maps, the top-k weights, and the count of rows still to be
    // written for each (token, 256-column block)
    float* comb;           // [T][n_out]
    const int32_t* src;    // [R]
    const int32_t* slot;   // [T*K]
    const float* wts;      // [T*K]
    int32_t* arrivals;     // [T][n_out/256]
    int K, T, R;
    // failure-detection test hook: CTA 0's matrix-0 issuer withholds the
    // operand-release commit of its block stall_idx, so the converters' bounded
    // wait for that stage runs out (MOE_DEV_ERR_TIMEOUT); -1 withholds nothing
    int stall_idx;
};

// ---------------------------------------------------------------- device ---

__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tmem_st16(uint32_t ta, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t ta, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 columns of two TMEM addresses and the wait for them in one statement
__device__ __forceinline__ void tmem_ld16x2_wait(uint32_t ta, uint32_t tb, uint32_t (&r)[2][16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, "
        "%8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, "
        "%24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]),
          "=r"(r[0][6]), "=r"(r[0][7]), "=r"(r[0][8]), "=r"(r[0][9]), "=r"(r[0][10]), "=r"(r[0][11]),
          "=r"(r[0][12]), "=r"(r[0][13]), "=r"(r[0][14]), "=r"(r[0][15]), "=r"(r[1][0]), "=r"(r[1][1]),
          "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]), "=r"(r[1][6]), "=r"(r[1][7]),
          "=r"(r[1][8]), "=r"(r[1][9]), "=r"(r[1][10]), "=r"(r[1][11]), "=r"(r[1][12]), "=r"(r[1][13]),
          "=r"(r[1][14]), "=r"(r[1][15])
        : "r"(ta), "r"(tb)
        : "memory");
}

__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg4(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg2(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// hi = RN(d*q) and lo = d*q - hi (exact) for 16 pairs of binary16 integers q
__device__ __forceinline__ void split16(const uint32_t (&qv)[16], uint32_t d16, uint32_t (&hi)[16],
                                        uint32_t (&lo)[16]) {
    const uint32_t d2u = d16 | (d16 << 16);
    const __half2 d2 = *reinterpret_cast<const __half2*>(&d2u);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const __half2 q = *reinterpret_cast<const __half2*>(&qv[j]);
        const __half2 h = __hmul2(d2, q);
        const __half2 l = __hfma2(d2, q, __hneg2(h));
        hi[j] = *reinterpret_cast<const uint32_t*>(&h);
        lo[j] = *reinterpret_cast<const uint32_t*>(&l);
    }
}

// Raw weight data of one lane's row for one block
template <int WT>
struct WRaw {
    static constexpr int NW = WT == MOE_W_Q8_0 ? 8 : WT == MOE_W_Q4_1 ? 4 : 2;
    uint32_t w[NW];
    uint32_t d;  // binary16 d
};

// Raw token data of one lane's token for one block
struct XRaw {
    uint32_t w[8];
    uint32_t ds;  // (d, s) binary16 pair
};

// Bounded wait for a whole warp; the result is warp-uniform.
__device__ __forceinline__ bool wait_warp(uint32_t b, uint32_t parity, volatile int* abort_flag) {
    bool done = mbar_test_wait(b, parity);
    if (!done) {
        long long t0 = clock64();
        while (true) {
            if (mbar_try_wait_sleep(b, parity)) {
                done = true;
                break;
            }
            if (*abort_flag) break;
            if (clock64() - t0 > TIMEOUT_CYCLES) {
                *abort_flag = 1;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, done);
}

template <int WT, bool GU, bool CMB>
__global__ void __launch_bounds__(THREADS, 1) mmq_fold_kernel(const Params P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = (uint64_t*)(smem + O_BAR);
    uint32_t* tmem_slot = (uint32_t*)(smem + O_BAR + N_BARS * 8);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    int4* ring = (int4*)(smem + O_RING);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    constexpr int NT = WT == MOE_W_Q2_0 ? 2 : 3;  // MMA terms per K-step
    const int nb = P.nb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < IR; ++i) {
            mbar_init(bar(B_IF + i), 1);
            mbar_init(bar(B_IE + i), EPI_WARPS);
        }
        for (int i = 0; i < AS; ++i) {
            mbar_init(bar(B_OF + i), CVT_WARPS);
            mbar_init(bar(B_OE + i), MMA_ISSUERS);
        }
        for (int i = 0; i < MS; ++i) {
            mbar_init(bar(B_MF + i), CVT_WARPS);
            mbar_init(bar(B_ME + i), MMA_ISSUERS);
        }
        mbar_init(bar(B_AF), MMA_ISSUERS);
        mbar_init(bar(B_AE), EPI_WARPS);
        mbar_init(bar(B_EPI), EPI_WARPS);
        *(int*)(smem + O_LIST) = 0;
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // item i of this CTA as (slot, first row, valid rows, first weight row);
    // rows < 0 ends the sequence
    auto item_warp = [&](int i, int4& e) -> bool {
        if (!wait_warp(bar(B_IF + i % IR), (i / IR) & 1, abort_flag)) return false;
        e = ring[i % IR];
        return true;
    };
    if (warp == SCHED_WARP) {
        if (lane == 0) {
            const int n_items = *P.n_tiles * P.mt_count;
            for (int i = 0;; ++i) {
                const int s = i % IR;
                if (i >= IR && !mbar_wait(bar(B_IE + s), ((i / IR) - 1) & 1, abort_flag)) break;
                const int it = atomicAdd(P.ticket, 1);
                int4 e = make_int4(0, 0, -1, 0);
                if (it < n_items) {
                    const int tile = it / P.mt_count, mt = it - tile * P.mt_count;
                    const int4 t = P.tiles[tile];
                    e = make_int4(t.x, t.y, t.z, mt * (GU ? BM : 2 * BM));
                }
                ring[s] = e;
                mbar_arrive(bar(B_IF + s));
                if (e.z < 0) break;
            }
        }
    } else if (warp >= WCVT_WARP0 && warp < WCVT_WARP0 + WCVT_WARPS) {
        // ---- weight converters: warp (quarter q, matrix mat), lane = weight row m.
        // Blocks are fetched two ahead into a ring of three register buffers; the
        // loop is unrolled over the AS operand stages so that every stage index
        // and buffer index is a constant.
        const int q = warp & 3, mat = (warp - WCVT_WARP0) >> 2;
        const int m = q * 32 + lane;
        const uint32_t lanes = tmem + ((uint32_t)(q * 32) << 16);
        using Raw = WRaw<WT>;
        constexpr int BB = WT == MOE_W_Q8_0 ? 32 : WT == MOE_W_Q4_1 ? 16 : 8;  // bytes per row-block
        const size_t dstep = (size_t)P.wrows * 2;                                 // scale plane: next block
        const uint8_t* fq = nullptr;  // fetch position: quant bytes and scale of the next block
        const uint8_t* fd = nullptr;
        auto row_base = [&](const int4& e) {
            return P.group_base + (size_t)e.x * P.slot_stride + P.mat_off[mat];
        };
        auto fset = [&](const int4& e) {
            const uint8_t* base = row_base(e);
            const int j = e.w + m + mat * P.mat1_row;
            fq = base + P.q_off + (size_t)j * P.row_bytes;
            fd = base + P.d_off + (size_t)j * 2;
        };
        auto load = [&](Raw& r) {
            if (WT == MOE_W_Q8_0) {
                const uint4 a0 = ldg16(fq), a1 = ldg16(fq + 16);
                r.w[0] = a0.x; r.w[1] = a0.y; r.w[2] = a0.z; r.w[3] = a0.w;
                r.w[4] = a1.x; r.w[5] = a1.y; r.w[6] = a1.z; r.w[7] = a1.w;
            } else if (WT == MOE_W_Q4_1) {
                const uint4 a0 = ldg16(fq);
                r.w[0] = a0.x; r.w[1] = a0.y; r.w[2] = a0.z; r.w[3] = a0.w;
            } else {
                const uint2 a0 = ldg8(fq);
                r.w[0] = a0.x; r.w[1] = a0.y;
            }
            r.d = ldg2(fd);
        };
        // binary16 pairs of the integer codes, in the K order the token side uses
        auto codes = [&](const Raw& r, uint32_t (&qv)[16]) {
            if (WT == MOE_W_Q8_0) {
#pragma unroll
                for (int k = 0; k < 8; ++k) cvt_i8x4(r.w[k], qv[2 * k], qv[2 * k + 1]);
            } else if (WT == MOE_W_Q4_1) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t h[4];
                    cvt_u4x8(r.w[c], h);
#pragma unroll
                    for (int t = 0; t < 4; ++t) qv[4 * c + t] = h[t];
                }
            } else {
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {
                    uint32_t a[4], bq[4];
                    cvt_u2x16(r.w[w2], a, bq);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        qv[8 * w2 + t] = a[t];
                        qv[8 * w2 + 4 + t] = bq[t];
                    }
                }
            }
        };
        // Q4_1: binary16 m of this lane's row for the 16 blocks of the current
        // chunk, loaded when the chunk starts (zero past the last block)
        uint32_t mreg[MCH / 2];
        auto load_m = [&](const int4& e, int b0) {
            const uint8_t* mp = row_base(e) + P.m_off + (size_t)(e.w + m + mat * P.mat1_row) * 2;
#pragma unroll
            for (int k = 0; k < MCH / 2; ++k) {
                const int b = b0 + 2 * k;
                const uint32_t lo = b < nb ? ldg2(mp + (size_t)b * dstep) : 0u;
                const uint32_t hi = b + 1 < nb ? ldg2(mp + (size_t)(b + 1) * dstep) : 0u;
                mreg[k] = lo | (hi << 16);
            }
        };
        bool range_bad = false;
        int cw = 0;                 // m chunks written
        int fi = 0, fb = 0, pi = 0, pb = 0;
        int4 fe, pe;                // items of the fetch and conversion positions
        bool ok = item_warp(0, pe);
        fe = pe;
        auto fadvance = [&]() -> bool {
            if (++fb < nb) {
                fq += BB;
                fd += dstep;
                return true;
            }
            fb = 0;
            ++fi;
            if (!item_warp(fi, fe)) return false;
            if (fe.z >= 0) fset(fe);
            return true;
        };
        Raw rb[AS];
        if (ok && fe.z >= 0) {
            fset(fe);
            load(rb[0]);
            ok = fadvance();
            if (ok && fe.z >= 0) load(rb[1]);
        }
        static_assert(AS == 3, "the register ring below holds three blocks");
        for (int round = 0; ok && pe.z >= 0; ++round) {
#pragma unroll
            for (int k = 0; k < AS; ++k) {
                if (!ok || pe.z < 0) break;
                if (fe.z >= 0) {
                    if (!(ok = fadvance())) break;
                    if (fe.z >= 0) load(rb[(k + 2) % AS]);
                }
                if (round > 0 && !wait_warp(bar(B_OE + k), (round - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (WT == MOE_W_Q4_1 && pb % MCH == 0) load_m(pe, pb);
                {
                    uint32_t qv[16], hi[16], lo[16];
                    codes(rb[k], qv);
                    range_bad |= __habs(__ushort_as_half((unsigned short)rb[k].d)) >=
                                 __float2half_rn(Range<WT>::W);
                    split16(qv, rb[k].d, hi, lo);
                    const uint32_t ta = lanes + T_A + k * 64 + mat * 32;
                    tmem_st16(ta, hi);
                    if (NT == 3) tmem_st16(ta + 16, lo);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_OF + k));
                if (WT == MOE_W_Q4_1 && (pb % MCH == MCH - 1 || pb == nb - 1)) {
                    const int ms = cw % MS;
                    if (cw >= MS && !wait_warp(bar(B_ME + ms), ((cw / MS) - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_st8(lanes + T_M + ms * 16 + mat * 8, mreg);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_MF + ms));
                    ++cw;
                }
                if (++pb == nb) {
                    pb = 0;
                    ok = item_warp(++pi, pe);
                }
            }
        }
        tmem_wait_st();
        if (__any_sync(0xffffffffu, range_bad) && lane == 0) set_error(P.err, MOE_DEV_ERR_RANGE);
    } else if (warp >= XCVT_WARP0 && warp < XCVT_WARP0 + XCVT_WARPS) {
        // ---- token converters: lane = token n of the item; the same fetch ring
        // and unrolling as the weight converters
        const int n = (warp - XCVT_WARP0) * 32 + lane;
        const int8_t* fq = nullptr;
        const uint32_t* fd = nullptr;
        bool fin = false;  // token n exists in the fetch position's item
        auto fset = [&](const int4& e) {
            fin = n < e.z;
            fq = P.xq + (size_t)(e.y + (fin ? n : 0)) * P.klen;
            fd = P.xds + (size_t)(e.y + (fin ? n : 0)) * P.nb;
        };
        auto load = [&](XRaw& r) {
            if (fin) {
                const uint4 a0 = ldg16(fq), a1 = ldg16(fq + 16);
                r.w[0] = a0.x; r.w[1] = a0.y; r.w[2] = a0.z; r.w[3] = a0.w;
                r.w[4] = a1.x; r.w[5] = a1.y; r.w[6] = a1.z; r.w[7] = a1.w;
                r.ds = ldg4(fd);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) r.w[k] = 0;
                r.ds = 0;
            }
        };
        // Q4_1: binary16 s of this lane's token for the 16 blocks of the current
        // chunk, loaded when the chunk starts (zero past the last block and for
        // padding tokens)
        uint32_t sreg[MCH / 2];
        auto load_s = [&](const int4& e, int b0) {
            const uint32_t* dp = P.xds + (size_t)(e.y + n) * P.nb;
#pragma unroll
            for (int k = 0; k < MCH / 2; ++k) {
                const int b = b0 + 2 * k;
                const uint32_t lo = n < e.z && b < nb ? ldg4(dp + b) >> 16 : 0u;
                const uint32_t hi = n < e.z && b + 1 < nb ? ldg4(dp + b + 1) >> 16 : 0u;
                sreg[k] = lo | (hi << 16);
            }
        };
        bool range_bad = false;
        int cw = 0;
        int fi = 0, fb = 0, pi = 0, pb = 0;
        int4 fe, pe;
        bool ok = item_warp(0, pe);
        fe = pe;
        auto fadvance = [&]() -> bool {
            if (++fb < nb) {
                fq += QK;
                fd += 1;
                return true;
            }
            fb = 0;
            ++fi;
            if (!item_warp(fi, fe)) return false;
            if (fe.z >= 0) fset(fe);
            return true;
        };
        XRaw rb[AS];
        if (ok && fe.z >= 0) {
            fset(fe);
            load(rb[0]);
            ok = fadvance();
            if (ok && fe.z >= 0) load(rb[1]);
        }
        for (int round = 0; ok && pe.z >= 0; ++round) {
#pragma unroll
            for (int k = 0; k < AS; ++k) {
                if (!ok || pe.z < 0) break;
                if (fe.z >= 0) {
                    if (!(ok = fadvance())) break;
                    if (fe.z >= 0) load(rb[(k + 2) % AS]);
                }
                const int ncols = (pe.z + 15) & ~15;
                if (round > 0 && !wait_warp(bar(B_OE + k), (round - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                if (WT == MOE_W_Q4_1 && pb % MCH == 0) load_s(pe, pb);
                if (n < ncols) {
                    uint32_t qv[16], hi[16], lo[16];
                    if (WT == MOE_W_Q8_0) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) cvt_i8x4(rb[k].w[c], qv[2 * c], qv[2 * c + 1]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t h[4];
                            cvt_i8x8_interleaved(rb[k].w[2 * c], rb[k].w[2 * c + 1], h);
#pragma unroll
                            for (int t = 0; t < 4; ++t) qv[4 * c + t] = h[t];
                        }
                    }
                    const uint32_t d16 = rb[k].ds & 0xFFFFu;
                    range_bad |= __habs(__ushort_as_half((unsigned short)d16)) >= __float2half_rn(X_RANGE);
                    split16(qv, d16, hi, lo);
                    uint8_t* xh = smem + O_B + k * 2 * XT;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        *(uint4*)(xh + f16_off(n, c)) = make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
                        *(uint4*)(xh + XT + f16_off(n, c)) =
                            make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_OF + k));
                if (WT == MOE_W_Q4_1 && (pb % MCH == MCH - 1 || pb == nb - 1)) {
                    const int ms = cw % MS;
                    if (cw >= MS && !wait_warp(bar(B_ME + ms), ((cw / MS) - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (n < ncols) {
                        uint8_t* bm = smem + O_BM + ms * BN * 32;
                        const uint32_t o = (uint32_t)((n >> 3) * 256 + (n & 7) * 16);
                        *(uint4*)(bm + o) = make_uint4(sreg[0], sreg[1], sreg[2], sreg[3]);
                        *(uint4*)(bm + o + 128) = make_uint4(sreg[4], sreg[5], sreg[6], sreg[7]);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_MF + ms));
                    ++cw;
                }
                if (++pb == nb) {
                    pb = 0;
                    ok = item_warp(++pi, pe);
                }
            }
        }
        if (__any_sync(0xffffffffu, range_bad) && lane == 0) set_error(P.err, MOE_DEV_ERR_RANGE);
    } else if (warp == MMA_WARP || warp == MMA_WARP2) {
        if (lane == 0) {
            const int mat = warp == MMA_WARP ? 0 : 1;  // this issuer's matrix
            // ---- MMA issuer.  A lean loop: operand descriptors advance by
            // constant offsets, and the next block's operand barrier is probed
            // before this block's MMAs are issued, so the probe's latency
            // overlaps them.
            const uint64_t bdesc0 = sdesc(sbase + O_B, 128, 512);
            const uint32_t a0 = tmem + T_A;
            int cw = 0;
            int s = 0;          // operand stage of the next block
            uint32_t ph = 0;    // bit k: phase parity of stage k's next fill
            int last_bar = -1;
            uint32_t last_par = 0;
            int gblk = 0;  // blocks issued by this thread so far
            for (int i = 0;; ++i) {
                if (!mbar_wait(bar(B_IF + i % IR), (i / IR) & 1, abort_flag)) break;
                const int4 e = ring[i % IR];
                if (e.z < 0) break;
                const int ncols = (e.z + 15) & ~15;
                const uint32_t id = idesc_f16(BM, ncols);
                if (i > 0 && !mbar_wait(bar(B_AE), (i - 1) & 1, abort_flag)) break;
                tc_fence_after();
                bool ready = mbar_test_wait(bar(B_OF + s), (ph >> s) & 1);
                bool ok = true;
                for (int b = 0; b < nb; ++b, ++gblk) {
                    if (!ready && !mbar_wait(bar(B_OF + s), (ph >> s) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int sn = s + 1 == AS ? 0 : s + 1;
                    const uint32_t phn = ph ^ (1u << s);
                    ready = b + 1 < nb && mbar_test_wait(bar(B_OF + sn), (phn >> sn) & 1);
                    const uint64_t bd = bdesc0 + (uint64_t)((s * 2 * XT) >> 4);
                    const uint32_t as = a0 + s * 64;
                    {
                        const uint32_t d = tmem + T_ACC + mat * BN;
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
                            const uint32_t ah = as + mat * 32 + ks * 8;
                            const uint64_t bh = bd + (uint64_t)((ks * 256) >> 4);
                            const uint64_t bl = bh + (uint64_t)(XT >> 4);
                            mma_tmem_a(d, ah, bh, id, (uint32_t)(b | ks));
                            if (NT == 3) mma_tmem_a(d, ah + 16, bh, id, 1u);
                            mma_tmem_a(d, ah, bl, id, 1u);
                        }
                    }
                    if (!(gblk == P.stall_idx && blockIdx.x == 0 && mat == 0))
                        mma_commit(bar(B_OE + s));
                    last_bar = B_OE + s;
                    last_par = (ph >> s) & 1;
                    ph = phn;
                    s = sn;
                    if (WT == MOE_W_Q4_1 && ((b % MCH) == MCH - 1 || b == nb - 1)) {
                        const int ms = cw % MS;
                        if (!mbar_wait(bar(B_MF + ms), (cw / MS) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t bm = sdesc(sbase + O_BM + ms * BN * 32, 128, 256);
                        mma_tmem_a(tmem + T_ACC + mat * BN, tmem + T_M + ms * 16 + mat * 8, bm, id, 1u);
                        mma_commit(bar(B_ME + ms));
                        last_bar = B_ME + ms;
                        last_par = (cw / MS) & 1;
                        ++cw;
                    }
                }
                if (!ok) break;
                mma_commit(bar(B_AF));
            }
            // everything committed must land before TMEM is freed
            if (last_bar >= 0) {
                long long t0 = clock64();
                bool landed = false;
                while (!(landed = mbar_try_wait(bar(last_bar), last_par)) && clock64() - t0 < TIMEOUT_CYCLES) {
                }
                if (!landed) *abort_flag = 1;  // reported as MOE_DEV_ERR_TIMEOUT
            }
        }
    } else if (warp < EPI_WARPS) {
        // ---- epilogue: warp w copies TMEM lane quarter w % 4 (its 32 weight
        // rows) for token half w / 4 into the staging buffer [token][256]
        const int q = warp & 3, hf = warp >> 2;
        const uint32_t lanes = tmem + ((uint32_t)(q * 32) << 16);
        float* st = (float*)(smem + O_STAGE);
        int epi_phase = 0;
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_EPI));
            const bool r = wait_warp(bar(B_EPI), epi_phase & 1, abort_flag);
            ++epi_phase;
            return r;
        };
        for (int i = 0;; ++i) {
            int4 e;
            if (!item_warp(i, e)) break;
            if (e.z < 0) break;
            const int rows = e.z, ncols = (rows + 15) & ~15;
            if (!wait_warp(bar(B_AF), i & 1, abort_flag)) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int n0 = hf * 64 + c * 16;
                if (n0 < ncols) {  // warp-uniform
                    uint32_t v[2][16];
                    tmem_ld16x2_wait(lanes + T_ACC + n0, lanes + T_ACC + BN + n0, v);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        st[(n0 + k) * STAGE_W + q * 32 + lane] = __uint_as_float(v[0][k]);
                        st[(n0 + k) * STAGE_W + BM + q * 32 + lane] = __uint_as_float(v[1][k]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_AE));  // the MMA may overwrite the accumulator
            if (!epi_sync()) break;
            if (GU) {
                const int t = threadIdx.x;  // 0..255
                const int j = t & (BM - 1);
                for (int n = t >> 7; n < rows; n += 2)
                    st[n * STAGE_W + j] = silu_mul(st[n * STAGE_W + j], st[n * STAGE_W + BM + j]);
            }
            if constexpr (CMB) {
                // Down with the top-k combine ("#1282 ...", "What it does"): the y
                // rows by generic 16-byte stores, then every row counts down its
                // (token, 256-column block); the item that writes a token's last
                // row combines it,
                //   out[t, c] = fma chain over k ascending of w[t*K+k] * y[slot[t*K+k], c],
                // the stand-alone combine's arithmetic, whichever item comes last.
                if (!epi_sync()) break;
                const int t = threadIdx.x;  // 0..255
                const int c4 = t & 63;      // 16-byte column of the item's 256 columns
                for (int n = t >> 6; n < rows; n += EPI_WARPS * 32 / 64)
                    reinterpret_cast<float4*>(P.out + (size_t)(e.y + n) * P.n_out + e.w)[c4] =
                        reinterpret_cast<const float4*>(st + n * STAGE_W)[c4];
                __threadfence();  // this thread's y stores, device-wide, before the count
                if (!epi_sync()) break;
                int* list = (int*)(smem + O_LIST);
                const int ncb = P.n_out / (2 * BM), cb = e.w / (2 * BM);
                if (t < rows) {
                    const int tok = P.src[e.y + t];
                    if ((unsigned)tok < (unsigned)P.T) {
                        __threadfence();
                        if (atomicSub(&P.arrivals[(size_t)tok * ncb + cb], 1) == 1) {
                            __threadfence();
                            list[1 + atomicAdd(&list[0], 1)] = tok;
                        }
                    } else {
                        set_error(P.err, MOE_DEV_ERR_BAD_ROWS);
                    }
                }
                if (!epi_sync()) break;
                const int nl = list[0];
                __threadfence();  // the other items' y rows of these tokens
                for (int li = t >> 6; li < nl; li += EPI_WARPS * 32 / 64) {
                    const int tok = list[1 + li];
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int k = 0; k < P.K; ++k) {
                        const int r = P.slot[(size_t)tok * P.K + k];
                        if ((unsigned)r >= (unsigned)P.R) continue;
                        const float wk = P.wts[(size_t)tok * P.K + k];
                        const float4 v = __ldcg(
                            reinterpret_cast<const float4*>(P.out + (size_t)r * P.n_out + e.w) + c4);
                        acc.x = __fmaf_rn(wk, v.x, acc.x);
                        acc.y = __fmaf_rn(wk, v.y, acc.y);
                        acc.z = __fmaf_rn(wk, v.z, acc.z);
                        acc.w = __fmaf_rn(wk, v.w, acc.w);
                    }
                    reinterpret_cast<float4*>(P.comb + (size_t)tok * P.n_out + e.w)[c4] = acc;
                }
                if (!epi_sync()) break;  // the list is read and the staging buffer free
                if (t == 0) list[0] = 0;
            } else {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (!epi_sync()) break;
                if (warp == 0) {
                    const uint32_t bytes = (GU ? BM : 2 * BM) * 4;
                    for (int n = lane; n < rows; n += 32)
                        bulk_s2g(P.out + (size_t)(e.y + n) * P.n_out + e.w,
                                 smem_u32(st + n * STAGE_W), bytes);
                    bulk_commit();
                    bulk_wait_read0();
                }
                if (!epi_sync()) break;  // the staging buffer is free again
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_IE + i % IR));
        }
        if (warp == 0) bulk_wait0();
    }

    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) set_error(P.err, MOE_DEV_ERR_TIMEOUT);
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host ----

constexpr int kMaxDevices = 64;

// Per device: the shared-memory opt-in of each instantiation, and the SM count.
template <int WT, bool GU, bool CMB>
bool kernel_ready(int dev) {
    static std::mutex mu;
    static signed char state[kMaxDevices] = {};  // 0 unknown, 1 ready, -1 failed
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (state[dev] == 0) {
        cudaError_t e = cudaFuncSetAttribute(mmq_fold_kernel<WT, GU, CMB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        state[dev] = e == cudaSuccess ? 1 : -1;
        if (e != cudaSuccess && std::getenv("MOE_DEBUG"))
            std::fprintf(stderr, "moe_q8: mmq_fold smem attribute failed: %s\n", cudaGetErrorString(e));
    }
    return state[dev] == 1;
}

int sm_count(int dev) {
    static std::mutex mu;
    static int sms[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms[dev];
}

template <int WT, bool GU, bool CMB>
int launch(const uint8_t* group_base, size_t slot_stride, int E, const int8_t* xq,
           const uint16_t* xds, int R, int d, int f, float* out, uint8_t* ws, const WsLayout& W,
           const MmqFused& F, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (!kernel_ready<WT, GU, CMB>(dev)) return MOE_ERR_UNSUPPORTED;
    const RecLayout RL = rec_layout(WT, d, f);
    const MatLayout& ML = GU ? RL.gu : RL.dn;
    Params P;
    P.group_base = group_base;
    P.slot_stride = slot_stride;
    P.mat_off[0] = GU ? RL.gate : RL.down;
    P.mat_off[1] = GU ? RL.up : RL.down;
    P.q_off = ML.q;
    P.d_off = ML.d;
    P.m_off = ML.m;
    P.klen = GU ? d : f;
    P.row_bytes = (int)quant_row_bytes(WT, P.klen);
    P.wrows = GU ? f : d;
    P.mat1_row = GU ? 0 : BM;
    P.tiles = (const int4*)(ws + W.tiles);
    int32_t* counters = (int32_t*)(ws + W.counters);
    P.n_tiles = counters + MMQ_COUNTER_NTILES;
    P.ticket = counters + MMQ_COUNTER_TICKET;
    {
        const char* v = std::getenv("MOE_TEST_STALL_BLOCK");  // the test hook, read per launch
        P.stall_idx = v ? std::atoi(v) : -1;
    }
    P.mt_count = GU ? f / BM : d / (2 * BM);
    P.nb = P.klen / QK;
    P.n_out = GU ? f : d;
    P.xq = xq;
    P.xds = reinterpret_cast<const uint32_t*>(xds);
    P.out = out;
    P.err = (uint32_t*)(ws + W.err);
    P.comb = F.comb;
    P.src = F.src;
    P.slot = F.slot;
    P.wts = F.w;
    P.arrivals = F.arrivals;
    P.K = F.K;
    P.T = F.T;
    P.R = R;
    (void)E;
    const long long upper = ((long long)R / BN + E + 1) * P.mt_count;
    const int sms = sm_count(dev);
    const int grid = (int)(upper < sms ? upper : sms);
    mmq_fold_kernel<WT, GU, CMB><<<grid, THREADS, SMEM, stream>>>(P);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess && std::getenv("MOE_DEBUG"))
        std::fprintf(stderr, "moe_q8: mmq_fold launch failed: %s (grid %d, smem %d)\n",
                     cudaGetErrorString(e), grid, SMEM);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace fold

bool mmq_fold_supported(int wtype, int d, int f) {
    if (wtype != MOE_W_Q8_0 && wtype != MOE_W_Q4_1 && wtype != MOE_W_Q2_0) return false;
    return d % 256 == 0 && f % 128 == 0;  // whole 128-row weight tiles
}

int launch_mmq_fold(int wtype, bool gateup, const uint8_t* group_base, size_t slot_stride,
                    const int32_t* active, const int32_t* n_active, const int32_t* offsets, int E,
                    const int8_t* xq, const uint16_t* xds, int R, int d, int f, float* out,
                    uint8_t* ws, const WsLayout& W, const MmqFused& F, cudaStream_t stream) {
    if (F.hq || (F.comb && gateup)) return MOE_ERR_UNSUPPORTED;
    int rc = launch_mmq_tiles(active, n_active, offsets, E, R, fold::BN, ws, W, stream);
    if (rc != MOE_OK) return rc;
#define MOE_FOLD(WT)                                                                             \
    return gateup ? fold::launch<WT, true, false>(group_base, slot_stride, E, xq, xds, R, d, f,  \
                                                  out, ws, W, F, stream)                         \
           : F.comb ? fold::launch<WT, false, true>(group_base, slot_stride, E, xq, xds, R, d, f, \
                                                    out, ws, W, F, stream)                       \
                    : fold::launch<WT, false, false>(group_base, slot_stride, E, xq, xds, R, d,  \
                                                     f, out, ws, W, F, stream)
    if (wtype == MOE_W_Q8_0) MOE_FOLD(MOE_W_Q8_0);
    if (wtype == MOE_W_Q2_0) MOE_FOLD(MOE_W_Q2_0);
    MOE_FOLD(MOE_W_Q4_1);
#undef MOE_FOLD
}

}  // namespace moe
