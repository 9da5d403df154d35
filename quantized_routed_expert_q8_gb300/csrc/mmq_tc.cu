// Stages 4 and 6 on the fifth-generation tensor cores (tcgen05, TMEM, TMA).
//
// The MMQ product of the pull-request pages ("#439 prefill: a group's expert
// gathers in one launch", "What": the MMQ group's products run on the gathered
// group buffers; "#1368 ...", intro: the q8_1 activations are expert-sorted
// rows) is, for the expert at active position p and its rows r:
//     acc[r, j] = sum over 32-blocks b of  dW[j,b] * dx[r,b] * I_b[r,j]
//                 (+ mW[j,b] * sx[r,b] for Q4_1),    I_b = exact int dot of the block.
// sm_103a has no integer tensor-core MMA, so each block's integer dot is formed
// exactly by an fp16 MMA with fp32 accumulation: |q| <= 127 is exact in fp16,
// each product is an integer below 2^14 and a block's sum stays below 2^24,
// so every partial sum the tensor core forms is an exactly representable
// integer.  The per-block fp32 scaling then runs on the CUDA cores in the same
// order as the scalar definition: acc = fma(dW*dx, I_b, acc) (+ fma(mW, sx, acc)).
//
// One persistent CTA of 16 warps per SM (static round-robin over the
// device-built, longest-first work list).  A work item is 128 tokens of one
// expert times two 128-row weight blocks (gate and up rows j0..j0+127 for
// stage 4; down rows i0..i0+255 for stage 6).  The warps split into roles, one
// warpgroup each, connected by mbarrier full/empty rings:
//   producer (warp 12): TMA loads of raw int8 / 4-bit tiles and fp16 scales,
//     4 blocks a stage;
//   converters (warps 8-11): raw tiles -> fp16 operands in the K-major layout
//     the MMA descriptors read, fp16 scales -> fp32;
//   MMA issuer (warp 13): 2 x (M=128, N<=128, K=16) per matrix into one of two
//     TMEM buffers, committed to an mbarrier;
//   epilogue (warps 0-7): warp w reads TMEM lane quarter w % 4 (its weight rows)
//     for column half w / 4 (tokens), scales and accumulates in registers
//     (128 fp32 per thread) and writes the item's outputs.
// setmaxnreg moves registers from the converter/producer warpgroups to the
// epilogue warpgroups.
// The FUSED instantiations change only an item's end: gate/up writes its hidden
// rows as q8_1 (the stand-alone re-quantization's bytes) instead of fp32, and
// down, after its y rows, counts each row's token down and combines the tokens
// whose last row it wrote (the stand-alone combine's bytes).
// Every wait is bounded: on timeout the kernel sets MOE_DEV_ERR_TIMEOUT, drains
// what it started and exits.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "mmq.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BN = 128;      // tokens per work item (TMEM columns per matrix)
constexpr int BM = 128;      // weight rows per matrix (TMEM lanes)
constexpr int KBS = 4;       // 32-blocks per raw stage
constexpr int RS = 3;        // raw stages
constexpr int NFS = 2;       // fp16 operand slots
constexpr int NTB = 2;       // TMEM partial buffers (256 columns each)
constexpr int NSC = 4;       // fp32 scale slots
constexpr int ITEM_RING = 8; // work items kept in shared memory (written by the producer)

// Warp roles, one warpgroup each (a warpgroup puts one warp on every SM
// sub-partition): warpgroups 0-1 scale and accumulate the block partials
// (epilogue), warpgroup 2 converts raw tiles into fp16 operands and fp32
// scales, warpgroup 3 holds the TMA producer (warp 12) and the MMA issuer
// (warp 13).
constexpr int EPI_WARPS = 8;
constexpr int CVT_WARPS = 4;
constexpr int THREADS = 512;
// Register split.  The launch gives every thread LAUNCH_REGS; warpgroups 2-3
// give registers back (setmaxnreg.dec) and warpgroups 0-1 take them
// (setmaxnreg.inc), so both the CTA's total and every sub-partition's share
// stay as launched.
constexpr int LAUNCH_REGS = 128;  // 65536 / 512
constexpr int EPI_REGS = 216;
constexpr int CVT_REGS = 56;
constexpr int AUX_REGS = 24;
static_assert(2 * EPI_REGS + CVT_REGS + AUX_REGS == 4 * LAUNCH_REGS, "register split must balance");
static_assert(THREADS * LAUNCH_REGS <= 65536, "launch registers exceed the register file");

constexpr int F16_A = 2 * BM * 64;  // two 128-row matrices x 32 fp16
constexpr int F16_B = BN * 64;
constexpr int F16_SLOT = F16_A + F16_B;

__host__ __device__ constexpr int cround(int x, int a) { return (x + a - 1) / a * a; }

template <int WT>
struct Lay {
    // Q2_K: a stage's 4 blocks are half of one 256-weight super-block (one d and
    // one dmin per row) and 8 sub-blocks (one sc | mn << 4 byte each per row);
    // its activations are D2S6 (d, s, s_lo, s_hi), 8 bytes a block
    static constexpr bool QK2 = WT == MOE_W_Q2_K;
    // raw weight bytes per row per stage (KBS blocks)
    static constexpr int WROW = WT == MOE_W_Q8_0 ? 128 : (WT == MOE_W_Q2_0 || QK2) ? 32 : 64;
    static constexpr int W_RAW = 2 * BM * WROW;
    static constexpr int X_RAW = BN * 128;
    static constexpr int WS_RAW = QK2 ? 2 * BM * 2 : 2 * KBS * BM * 2;
    static constexpr int WM_RAW = WT == MOE_W_Q4_1 ? WS_RAW : QK2 ? 2 * BM * 2 : 0;
    static constexpr int WC_RAW = QK2 ? 2 * KBS * 2 * BM : 0;
    static constexpr int XS_RAW = BN * KBS * (QK2 ? 8 : 4);
    static constexpr int O_W = 0;
    static constexpr int O_X = W_RAW;
    static constexpr int O_WS = O_X + X_RAW;
    static constexpr int O_WM = O_WS + WS_RAW;
    static constexpr int O_WC = O_WM + WM_RAW;
    static constexpr int O_XS = O_WC + WC_RAW;
    static constexpr int STAGE = cround(O_XS + XS_RAW, 1024);
    static constexpr uint32_t TX = W_RAW + X_RAW + WS_RAW + WM_RAW + WC_RAW + XS_RAW;
    // fp32 scale slot (float offsets): dW [256], mW [256] (Q2_K: the first
    // half's -dmin*mn, then the second half's [256]), dX [128], sX [128]
    // (Q2_K: s_lo, then s_hi [128])
    static constexpr int SC_MW = 2 * BM;
    static constexpr int SC_MW2 = 4 * BM;
    static constexpr int SC_DX = QK2 ? 6 * BM : 4 * BM;
    static constexpr int SC_SX = SC_DX + BN;
    static constexpr int SC_SX2 = SC_SX + BN;
    static constexpr int SC_SLOT = (SC_SX + BN + (QK2 ? BN : 0)) * 4;
    static constexpr int O_F16 = RS * STAGE;
    static constexpr int O_SC = O_F16 + NFS * F16_SLOT;
    static constexpr int O_BAR = O_SC + NSC * SC_SLOT;
    // full/empty pairs of the four rings, plus the epilogue warps' own barrier
    static constexpr int N_BARS = 2 * (RS + NFS + NSC + NTB) + 1;
    static constexpr int O_ITEMS = cround(O_BAR + N_BARS * 8 + 16, 16);
    // down with the combine: [0] count, [1..BN] tokens whose rows are all written
    static constexpr int O_LIST = O_ITEMS + ITEM_RING * 16;
    static constexpr int SMEM = O_LIST + (BN + 1) * 4 + 1024;  // + alignment slack
};


// q8_1 of 16 tokens' 32-value blocks, one value of each per lane (the
// hidden-row re-quantization of "#1368 ...", intro, done in the gate/up
// epilogue): the stand-alone quantizer's operations, d = amax/127 and
// q = round-half-away(v/d) with IEEE division, s = d * sum(q), so the bytes are
// identical.  Token n0 + i is stored if it is below `rows`; lane 0 stores (d, s),
// or with D2S6 (d, s, s_lo, s_hi) -- s_lo from lanes 0-15, s_hi from 16-31 --
// as one 8-byte store (ds_stride then counts 8-byte entries).
template <bool D2S6>
__device__ __forceinline__ void requant16(const float (&v)[16], int n0, int rows, int8_t* q0,
                                          int q_stride, __half2* ds0, int ds_stride, int lane) {
    float amax[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) amax[i] = fmaxf(0.0f, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i) amax[i] = fmaxf(amax[i], __shfl_xor_sync(0xffffffffu, amax[i], o));
    float d[16];
    int qi[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        d[i] = __fdiv_rn(amax[i], 127.0f);
        qi[i] = 0;
        if (d[i] != 0.0f) {  // warp-uniform; a zero d stores an all-zero block
            float x = roundf(__fdiv_rn(v[i], d[i]));
            x = fminf(127.0f, fmaxf(-127.0f, x));
            qi[i] = (int)x;
        }
    }
    int sum[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) sum[i] = qi[i];
    // sums over each 16-lane half first (the D2S6 half sums), then the block
#pragma unroll
    for (int o = 1; o <= 8; o <<= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i) sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], o);
    int hi[16];
    if (D2S6) {
#pragma unroll
        for (int i = 0; i < 16; ++i) hi[i] = __shfl_sync(0xffffffffu, sum[i], 16);
    }
    int lo[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        lo[i] = sum[i];
        sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], 16);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int n = n0 + i;
        if (n < rows) {
            q0[(size_t)n * q_stride] = (int8_t)qi[i];
            if (lane == 0) {
                const __half2 ds =
                    __halves2half2(__float2half_rn(d[i]), __float2half_rn(__fmul_rn(d[i], (float)sum[i])));
                if (D2S6) {
                    const __half2 lh = __halves2half2(__float2half_rn(__fmul_rn(d[i], (float)lo[i])),
                                                      __float2half_rn(__fmul_rn(d[i], (float)hi[i])));
                    uint2 e;
                    e.x = *reinterpret_cast<const uint32_t*>(&ds);
                    e.y = *reinterpret_cast<const uint32_t*>(&lh);
                    reinterpret_cast<uint2*>(ds0)[(size_t)n * ds_stride] = e;
                } else {
                    ds0[(size_t)n * ds_stride] = ds;
                }
            }
        }
    }
}

struct Params {
    const int4* tiles;
    const int32_t* n_tiles;
    int mt_count;  // weight-row tiles per token tile
    int nb;        // 32-blocks of the reduction
    int n_out;     // output row length (f for gate/up, d for down)
    int R;         // rows
    float* out;    // fp32 rows [R][n_out] (gate/up: h, unless hq is set; down: y)
    uint32_t* err;
    // gate/up: q8_1 hidden rows written by the epilogue instead of h
    int8_t* hq;    // [R][f]
    __half2* hds;  // [R][f/32] (d, s); Q2_K: [R][f/32] 8-byte (d, s, s_lo, s_hi)
    // down: the top-k combine of every (token, 256-column block) whose rows are complete
    float* comb;            // [T][d]
    const int32_t* src;     // row -> token
    const int32_t* slot;    // t*K + k -> row
    const float* wts;       // [T*K] top-k weights
    int32_t* arrivals;      // [T][d/256] rows of the token still to be written
    int K, T;
    // failure-detection test hook: CTA 0 withholds the partials commit of its
    // block stall_idx, so its epilogue's bounded wait runs out (MOE_DEV_ERR_TIMEOUT)
    // and every role exits; -1 (the default) withholds nothing
    int stall_idx;
};

struct Item {
    int p, r0, rows, ncols, w0;  // slot, first row, valid rows, MMA N, first weight row
};



template <bool GU>
__device__ __forceinline__ Item load_item(const Params& P, int it) {
    int tile = it / P.mt_count, mt = it - tile * P.mt_count;
    int4 t = P.tiles[tile];
    Item I;
    I.p = t.x;
    I.r0 = t.y;
    I.rows = t.z;
    I.ncols = (t.z + 15) & ~15;
    I.w0 = GU ? mt * BM : mt * 2 * BM;
    return I;
}

template <int WT, bool GU, bool FUSED>
__global__ void __launch_bounds__(THREADS, 1)
    mmq_tc_kernel(const __grid_constant__ CUtensorMap mW, const __grid_constant__ CUtensorMap mWs,
                  const __grid_constant__ CUtensorMap mWm, const __grid_constant__ CUtensorMap mWc,
                  const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mXs,
                  const Params P) {
    using L = Lay<WT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = (uint64_t*)(smem + L::O_BAR);
    uint32_t* tmem_slot = (uint32_t*)(smem + L::O_BAR + L::N_BARS * 8);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    // full/empty pairs: raw stages (TMA -> converters), fp16 operands
    // (converters -> MMA), fp32 scales (converters -> epilogue), TMEM partials
    // (MMA -> epilogue)
    constexpr int B_RAW_FULL = 0, B_RAW_EMPTY = RS;
    constexpr int B_F16_FULL = 2 * RS, B_F16_EMPTY = B_F16_FULL + NFS;
    constexpr int B_SC_FULL = B_F16_EMPTY + NFS, B_SC_EMPTY = B_SC_FULL + NSC;
    constexpr int B_TM_FULL = B_SC_EMPTY + NSC, B_TM_EMPTY = B_TM_FULL + NTB;
    constexpr int B_EPI = B_TM_EMPTY + NTB;  // the epilogue warps meet at an item's end

    const int n_items = *P.n_tiles * P.mt_count;
    if ((int)blockIdx.x >= n_items) return;
    const int my_items = (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;
    const int nb = P.nb;
    const int spi = nb / KBS;  // raw stages per item
    const int total = my_items * nb;
    const int total_stages = my_items * spi;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RS; ++i) {
            mbar_init(bar(B_RAW_FULL + i), 1);
            mbar_init(bar(B_RAW_EMPTY + i), CVT_WARPS);
        }
        for (int i = 0; i < NFS; ++i) {
            mbar_init(bar(B_F16_FULL + i), CVT_WARPS);
            mbar_init(bar(B_F16_EMPTY + i), 1);
        }
        for (int i = 0; i < NSC; ++i) {
            mbar_init(bar(B_SC_FULL + i), CVT_WARPS);
            mbar_init(bar(B_SC_EMPTY + i), EPI_WARPS);
        }
        for (int i = 0; i < NTB; ++i) {
            mbar_init(bar(B_TM_FULL + i), 1);
            mbar_init(bar(B_TM_EMPTY + i), EPI_WARPS);
        }
        mbar_init(bar(B_EPI), EPI_WARPS);
        *(int*)(smem + L::O_LIST) = 0;
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

    int4* ring = (int4*)(smem + L::O_ITEMS);
    // item i as (slot, first row, valid rows, first weight row); written by the
    // producer before the first TMA of the item, read by the other roles after a
    // barrier that orders them after that TMA
    auto item = [&](int i) -> Item {
        const int4 v = ring[i % ITEM_RING];
        Item I;
        I.p = v.x;
        I.r0 = v.y;
        I.rows = v.z;
        I.ncols = (v.z + 15) & ~15;
        I.w0 = v.w;
        return I;
    };
    // bounded wait for a whole warp; the threads may sleep in hardware until the
    // phase completes.  The result is warp-uniform.
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
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
    };

    // As wait_warp for two phases at once: both probes are issued back to back
    // (a probe of a completed phase still costs a shared-memory round trip)
    // and one vote makes the result warp-uniform.
    auto wait_warp2 = [&](uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2) -> bool {
        bool d1 = mbar_test_wait(b1, p1);
        bool d2 = mbar_test_wait(b2, p2);
        if (!(d1 && d2)) {
            long long t0 = clock64();
            while (true) {
                if (!d1) d1 = mbar_try_wait_sleep(b1, p1);
                if (d1 && !d2) d2 = mbar_try_wait_sleep(b2, p2);
                if (d1 && d2) break;
                if (*abort_flag) break;
                if (clock64() - t0 > TIMEOUT_CYCLES) {
                    *abort_flag = 1;
                    break;
                }
            }
        }
        return __all_sync(0xffffffffu, d1 && d2);
    };

    if (warp < EPI_WARPS) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPI_REGS));
        // ---- epilogue: for block idx, warp w reads TMEM lane quarter w % 4 (its
        // 32 weight rows) for column half w / 4 (64 tokens) of both matrices,
        // scales and accumulates in registers
        const int q = warp & 3;         // TMEM lane quarter this warp may access
        const int h = warp >> 2;        // column half
        const int m = q * 32 + lane;    // weight row (TMEM lane) of this thread
        // accumulators: 4 chunks x 16 columns for each matrix, as 8 packed pairs
        uint64_t accA[4][8], accB[4][8];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) accA[c][j] = accB[c][j] = 0ull;
        const uint32_t lanes = tmem + ((uint32_t)(q * 32) << 16);
        // the 8 epilogue warps meet (bounded; false on abort or timeout)
        int epi_phase = 0;
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_EPI));
            const bool ok = wait_warp(bar(B_EPI), epi_phase & 1);
            ++epi_phase;
            return ok;
        };
        // Down with the top-k combine ("#1282 ...", "What it does"), after the
        // item's y stores: every row of the item counts down its (token,
        // 256-column block); the item that writes a token's last row combines it,
        //   out[t, c] = fma chain over k ascending of w[t*K+k] * y[slot[t*K+k], c],
        // the stand-alone combine's arithmetic, so the result is the same whichever
        // item comes last.
        auto combine_item = [&](const Item& I) -> bool {
            int* list = (int*)(smem + L::O_LIST);
            const int et = threadIdx.x;  // 0..255
            const int ncb = P.n_out / (2 * BM), cb = I.w0 / (2 * BM);
            __threadfence();  // this thread's y stores, device-wide, before the count
            if (!epi_sync()) return false;
            if (et < I.rows) {
                const int t = P.src[I.r0 + et];  // the row's token
                if ((unsigned)t < (unsigned)P.T) {
                    __threadfence();
                    if (atomicSub(&P.arrivals[(size_t)t * ncb + cb], 1) == 1) {
                        __threadfence();
                        list[1 + atomicAdd(&list[0], 1)] = t;
                    }
                } else {
                    set_error(P.err, MOE_DEV_ERR_BAD_ROWS);
                }
            }
            if (!epi_sync()) return false;
            const int nl = list[0];
            __threadfence();  // the other items' y rows of these tokens
            // thread: 16-byte column c4 of every fourth listed token
            const int c4 = et & 63;
            for (int li = et >> 6; li < nl; li += EPI_WARPS * 32 / 64) {
                const int t = list[1 + li];
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int k = 0; k < P.K; ++k) {
                    const int r = P.slot[(size_t)t * P.K + k];
                    if ((unsigned)r >= (unsigned)P.R) continue;
                    const float wk = P.wts[(size_t)t * P.K + k];
                    const float4 v =
                        __ldcg(reinterpret_cast<const float4*>(P.out + (size_t)r * P.n_out + I.w0) + c4);
                    acc.x = __fmaf_rn(wk, v.x, acc.x);
                    acc.y = __fmaf_rn(wk, v.y, acc.y);
                    acc.z = __fmaf_rn(wk, v.z, acc.z);
                    acc.w = __fmaf_rn(wk, v.w, acc.w);
                }
                reinterpret_cast<float4*>(P.comb + (size_t)t * P.n_out + I.w0)[c4] = acc;
            }
            if (!epi_sync()) return false;  // the list is read: it may be reset
            if (et == 0) list[0] = 0;
            return true;
        };
        int i = 0, b = 0;  // item and block within the item of idx
        for (int idx = 0; idx < total; ++idx) {
            const int tb = idx % NTB, ss = idx % NSC;
            // warp-uniform decision: the TMEM loads below are warp-collective
            if (!wait_warp2(bar(B_TM_FULL + tb), (idx / NTB) & 1, bar(B_SC_FULL + ss), (idx / NSC) & 1))
                break;
            tc_fence_after();
            const Item I = item(i);
            const int nch = min(4, max(0, (I.ncols - h * 64) / 16));  // active 16-column chunks
            const uint32_t tbase = lanes + tb * 256 + h * 64;
            const float* sc = (const float*)(smem + L::O_SC + ss * L::SC_SLOT);
            constexpr bool HAS_M = WT == MOE_W_Q4_1 || L::QK2;
            const float dA = sc[m], dB = sc[BM + m];
            const float mA = HAS_M ? sc[L::SC_MW + m] : 0.0f;
            const float mB = HAS_M ? sc[L::SC_MW + BM + m] : 0.0f;
            const float nA = L::QK2 ? sc[L::SC_MW2 + m] : 0.0f;
            const float nB = L::QK2 ? sc[L::SC_MW2 + BM + m] : 0.0f;
            const uint64_t dA2 = pk2(__float_as_uint(dA), __float_as_uint(dA));
            const uint64_t dB2 = pk2(__float_as_uint(dB), __float_as_uint(dB));
            const uint64_t mA2 = pk2(__float_as_uint(mA), __float_as_uint(mA));
            const uint64_t mB2 = pk2(__float_as_uint(mB), __float_as_uint(mB));
            const uint64_t nA2 = pk2(__float_as_uint(nA), __float_as_uint(nA));
            const uint64_t nB2 = pk2(__float_as_uint(nB), __float_as_uint(nB));
            // token scales as 16-byte loads (two pairs each, the same address in
            // every lane); a chunk's loads are issued before the work that hides
            // their latency
            const ulonglong2* dX4 = reinterpret_cast<const ulonglong2*>(sc + L::SC_DX + h * 64);
            const ulonglong2* sX4 = reinterpret_cast<const ulonglong2*>(sc + L::SC_SX + h * 64);
            const ulonglong2* tX4 = reinterpret_cast<const ulonglong2*>(sc + L::SC_SX2 + h * 64);
            // Q2_K adds the second half's min term: fma(mW2, s_hi, acc)
            auto scale = [&](int c, const uint32_t(&ra)[16], const uint32_t(&rb)[16],
                             const ulonglong2(&dx)[4], const ulonglong2(&sx)[4],
                             const ulonglong2(&tx)[4]) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint64_t pa = pk2(ra[2 * j], ra[2 * j + 1]);
                    const uint64_t pb = pk2(rb[2 * j], rb[2 * j + 1]);
                    const uint64_t d2 = (j & 1) ? dx[j >> 1].y : dx[j >> 1].x;
                    accA[c][j] = fma2u(mul2u(dA2, d2), pa, accA[c][j]);
                    accB[c][j] = fma2u(mul2u(dB2, d2), pb, accB[c][j]);
                    if (HAS_M) {
                        const uint64_t s2 = (j & 1) ? sx[j >> 1].y : sx[j >> 1].x;
                        accA[c][j] = fma2u(mA2, s2, accA[c][j]);
                        accB[c][j] = fma2u(mB2, s2, accB[c][j]);
                    }
                    if (L::QK2) {
                        const uint64_t t2 = (j & 1) ? tx[j >> 1].y : tx[j >> 1].x;
                        accA[c][j] = fma2u(nA2, t2, accA[c][j]);
                        accB[c][j] = fma2u(nB2, t2, accB[c][j]);
                    }
                }
            };
            auto scales = [&](int c, ulonglong2(&dx)[4], ulonglong2(&sx)[4], ulonglong2(&tx)[4]) {
#pragma unroll
                for (int k = 0; k < 4; ++k) dx[k] = dX4[c * 4 + k];
                if (HAS_M) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) sx[k] = sX4[c * 4 + k];
                }
                if (L::QK2) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) tx[k] = tX4[c * 4 + k];
                }
            };
#pragma unroll
            for (int c2 = 0; c2 < 4; c2 += 2) {
                if (c2 >= nch) continue;
                ulonglong2 dx[4], sx[4], tx[4];
                scales(c2, dx, sx, tx);  // in flight during the TMEM round trip
                // chunks c2 and c2 + 1 of both matrices in one round trip
                uint32_t r[4][16];
                tmem_ld16x4_wait(tbase + c2 * 16, tbase + 128 + c2 * 16, r);
                scale(c2, r[0], r[2], dx, sx, tx);
                if (c2 + 1 < nch) {
                    scales(c2 + 1, dx, sx, tx);
                    scale(c2 + 1, r[1], r[3], dx, sx, tx);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_TM_EMPTY + tb));
                mbar_arrive(bar(B_SC_EMPTY + ss));
            }
            if (b == nb - 1) {
                // item complete: write this thread's row for every valid token
                if constexpr (GU && FUSED) {
                    // h as q8_1: the 32 lanes of this warp hold one 32-column block
                    // of each token; 16 tokens at a time so that their shuffle and
                    // division chains overlap
                    const int kb = (I.w0 + q * 32) / QK;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[16];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float a0, a1, b0, b1;
                            upk2(accA[c][j], a0, a1);
                            upk2(accB[c][j], b0, b1);
                            v[2 * j] = silu_mul(a0, b0);
                            v[2 * j + 1] = silu_mul(a1, b1);
                            accA[c][j] = accB[c][j] = 0ull;
                        }
                        const int n0 = h * 64 + c * 16;
                        // ds entries of row r0, block kb: (d, s) pairs, or 8-byte D2S6 entries
                        __half2* ds0 =
                            L::QK2 ? reinterpret_cast<__half2*>(reinterpret_cast<uint2*>(P.hds) +
                                                                (size_t)I.r0 * (P.n_out / QK) + kb)
                                   : P.hds + (size_t)I.r0 * (P.n_out / QK) + kb;
                        if (n0 < I.rows)  // warp-uniform
                            requant16<L::QK2>(v, n0, I.rows,
                                              P.hq + (size_t)I.r0 * P.n_out + I.w0 + m, P.n_out,
                                              ds0, P.n_out / QK, lane);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float a[2], bb[2];
                            upk2(accA[c][j], a[0], a[1]);
                            upk2(accB[c][j], bb[0], bb[1]);
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int n = h * 64 + c * 16 + 2 * j + e;
                                if (n < I.rows) {
                                    float* o = P.out + (size_t)(I.r0 + n) * P.n_out + I.w0 + m;
                                    if (GU) {
                                        o[0] = silu_mul(a[e], bb[e]);
                                    } else {
                                        o[0] = a[e];
                                        o[BM] = bb[e];
                                    }
                                }
                            }
                            accA[c][j] = accB[c][j] = 0ull;
                        }
                    }
                }
                if constexpr (!GU && FUSED) {
                    if (!combine_item(I)) break;
                }
                b = 0;
                ++i;
            } else {
                ++b;
            }
        }
        // no TMEM load may be outstanding when the CTA frees TMEM
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    } else if (warp < EPI_WARPS + CVT_WARPS) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CVT_REGS));
        // ---- converters: block idx's raw tiles -> fp16 operand slot idx % NFS
        // (the layout the MMA descriptors read) and fp32 scales -> slot idx % NSC
        const int ct = threadIdx.x - EPI_WARPS * 32;  // 0..127
        int ci = 0, cb = 0;                            // item and block within the item of idx
        const int cw = ct >> 5;
        for (int idx = 0; idx < total; ++idx) {
            const int gs = idx / KBS, sl = gs % RS, blk = idx % KBS;
            const int fs = idx % NFS, ss = idx % NSC;
            static_assert(NSC >= NFS, "slot reuse order");
            if (idx >= NSC) {
                if (!wait_warp2(bar(B_F16_EMPTY + fs), ((idx / NFS) - 1) & 1, bar(B_SC_EMPTY + ss),
                                ((idx / NSC) - 1) & 1))
                    break;
            } else if (idx >= NFS && !wait_warp(bar(B_F16_EMPTY + fs), ((idx / NFS) - 1) & 1)) {
                break;
            }
            if (blk == 0 && !wait_warp(bar(B_RAW_FULL + sl), (gs / RS) & 1)) break;
            const Item I = item(ci);  // read after the barrier that orders it
            if (++cb == nb) {
                cb = 0;
                ++ci;
            }
            const uint8_t* st = smem + sl * L::STAGE;
            uint8_t* fa = smem + L::O_F16 + fs * F16_SLOT;
            uint8_t* fbB = fa + F16_A;
            float* sc = (float*)(smem + L::O_SC + ss * L::SC_SLOT);
            // Thread ct's units: weight rows R0 + 64 * rep (Q8_0: both 16-byte
            // halves split over lanes; Q4_1: one 16-byte row ct + 128 * rep) and
            // tokens R0, R0 + 64.  Lanes 0-7 take 8 consecutive rows, lanes 8-15
            // their second halves, lanes 16-31 the next 8 rows, so every 8-lane
            // phase of the 16-byte loads and stores touches 8 distinct bank groups.
            // All shared-memory loads of the block are issued before any conversion.
            const int R0 = cw * 16 + (lane & 7) + 8 * (lane >> 4);
            const int hh = (lane >> 3) & 1;
            const int ch = (blk * 2 + hh) ^ (R0 & 7);  // 128-byte TMA swizzle (R0 + 64 * k alike)
            constexpr int NW = WT == MOE_W_Q8_0 ? 4 : 2;
            uint4 wv[NW];
#pragma unroll
            for (int rep = 0; rep < NW; ++rep) {
                if (WT == MOE_W_Q8_0) {
                    wv[rep] = *(const uint4*)(st + L::O_W + (rep * 64 + R0) * 128 + ch * 16);
                } else if (WT == MOE_W_Q2_0 || L::QK2) {
                    // 2-bit rows are 8 bytes a block, unswizzled: thread ct loads row ct
                    const uint2 v2 = *(const uint2*)(st + L::O_W + (rep * 128 + ct) * 32 + blk * 8);
                    wv[rep] = make_uint4(v2.x, v2.y, 0u, 0u);
                } else {
                    const int R = rep * 128 + ct;
                    wv[rep] = *(const uint4*)(st + L::O_W + R * 64 + ((blk ^ ((R >> 1) & 3)) * 16));
                }
            }
            const bool x0 = cw * 16 < I.ncols, x1 = cw * 16 + 64 < I.ncols;  // tokens R0, R0 + 64
            uint4 xv[2];
            xv[0] = x0 ? *(const uint4*)(st + L::O_X + R0 * 128 + ch * 16) : make_uint4(0, 0, 0, 0);
            xv[1] = x1 ? *(const uint4*)(st + L::O_X + (R0 + 64) * 128 + ch * 16) : make_uint4(0, 0, 0, 0);
            // scales of block blk: dW (and mW) of rows ct, ct + 128; dX, sX of token ct.
            // Q2_K: the stage's super-block d and dmin ([mat][row] for gate/up,
            // [row] for down: rows ct and ct + 128 either way) and the sub-block
            // bytes of the block's two halves ([mat][8][row] / [8][256 rows])
            const int si0 = L::QK2 ? ct : GU ? (blk * BM + ct) : (blk * 2 * BM + ct);
            const int si1 = L::QK2 ? 128 + ct : GU ? ((KBS + blk) * BM + ct) : (blk * 2 * BM + 128 + ct);
            const __half* ws = (const __half*)(st + L::O_WS);
            const __half dw0 = ws[si0], dw1 = ws[si1];
            __half mw0 = __ushort_as_half(0), mw1 = __ushort_as_half(0);
            if (WT == MOE_W_Q4_1 || L::QK2) {
                const __half* wm = (const __half*)(st + L::O_WM);
                mw0 = wm[si0];
                mw1 = wm[si1];
            }
            uint32_t scmn[2][2] = {{0u, 0u}, {0u, 0u}};  // [rep][half]
            if (L::QK2) {
                const uint8_t* wc = st + L::O_WC;
#pragma unroll
                for (int rep = 0; rep < 2; ++rep)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        scmn[rep][hf] = wc[GU ? (rep * 2 * KBS + 2 * blk + hf) * BM + ct
                                              : (2 * blk + hf) * 2 * BM + rep * 128 + ct];
            }
            uint2 xs2;  // (d, s) and, for D2S6, (s_lo, s_hi)
            if (L::QK2) {
                xs2 = ((const uint2*)(st + L::O_XS))[ct * KBS + blk];
            } else {
                xs2.x = ((const uint32_t*)(st + L::O_XS))[ct * KBS + blk];
                xs2.y = 0u;
            }
            const __half2 xs = *reinterpret_cast<const __half2*>(&xs2.x);
            // weights: 256 rows x 32 values of block blk
#pragma unroll
            for (int rep = 0; rep < NW; ++rep) {
                if (WT == MOE_W_Q8_0) {
                    const int R = rep * 64 + R0;
                    uint4 o0, o1;
                    cvt_i8x4(wv[rep].x, o0.x, o0.y);
                    cvt_i8x4(wv[rep].y, o0.z, o0.w);
                    cvt_i8x4(wv[rep].z, o1.x, o1.y);
                    cvt_i8x4(wv[rep].w, o1.z, o1.w);
                    uint8_t* dst = fa + (R >> 7) * (BM * 64);
                    *(uint4*)(dst + f16_off(R & 127, 2 * hh)) = o0;
                    *(uint4*)(dst + f16_off(R & 127, 2 * hh + 1)) = o1;
                } else if (WT == MOE_W_Q2_0 || L::QK2) {
                    const int R = rep * 128 + ct;
                    const uint32_t w2[2] = {wv[rep].x, wv[rep].y};
                    uint8_t* dst = fa + (R >> 7) * (BM * 64);
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {  // elements 16*c2 .. 16*c2 + 15
                        uint32_t a[4], b[4];
                        if (L::QK2)  // Q2_K: c * sc of the half's sub-block
                            cvt_u2x16_scaled(w2[c2], scmn[rep][c2] & 0xFu, a, b);
                        else
                            cvt_u2x16(w2[c2], a, b);
                        *(uint4*)(dst + f16_off(R & 127, 2 * c2)) = make_uint4(a[0], a[1], a[2], a[3]);
                        *(uint4*)(dst + f16_off(R & 127, 2 * c2 + 1)) = make_uint4(b[0], b[1], b[2], b[3]);
                    }
                } else {
                    const int R = rep * 128 + ct;
                    const uint32_t w4[4] = {wv[rep].x, wv[rep].y, wv[rep].z, wv[rep].w};
                    uint8_t* dst = fa + (R >> 7) * (BM * 64);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t hv[4];
                        cvt_u4x8(w4[c], hv);
                        *(uint4*)(dst + f16_off(R & 127, c)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    }
                }
            }
            // activations: tokens R0 and R0 + 64 of the MMA's ncols columns
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (k == 0 ? x0 : x1) {
                    const int n = R0 + 64 * k;
                    uint4 o0, o1;
                    if (WT == MOE_W_Q8_0) {
                        cvt_i8x4(xv[k].x, o0.x, o0.y);
                        cvt_i8x4(xv[k].y, o0.z, o0.w);
                        cvt_i8x4(xv[k].z, o1.x, o1.y);
                        cvt_i8x4(xv[k].w, o1.z, o1.w);
                    } else {
                        uint32_t a[4], b[4];
                        cvt_i8x8_interleaved(xv[k].x, xv[k].y, a);
                        cvt_i8x8_interleaved(xv[k].z, xv[k].w, b);
                        o0 = make_uint4(a[0], a[1], a[2], a[3]);
                        o1 = make_uint4(b[0], b[1], b[2], b[3]);
                    }
                    *(uint4*)(fbB + f16_off(n, 2 * hh)) = o0;
                    *(uint4*)(fbB + f16_off(n, 2 * hh + 1)) = o1;
                }
            }
            // scales as fp32: dW[256], mW[256] (Q2_K: -dmin*mn of each half, exact
            // products), dX[128], sX[128] (Q2_K: s_lo, s_hi)
            sc[ct] = __half2float(dw0);
            sc[128 + ct] = __half2float(dw1);
            if (WT == MOE_W_Q4_1) {
                sc[L::SC_MW + ct] = __half2float(mw0);
                sc[L::SC_MW + 128 + ct] = __half2float(mw1);
            }
            if (L::QK2) {
                const float dm[2] = {__half2float(mw0), __half2float(mw1)};
#pragma unroll
                for (int rep = 0; rep < 2; ++rep) {
                    sc[L::SC_MW + rep * 128 + ct] = -__fmul_rn(dm[rep], (float)(scmn[rep][0] >> 4));
                    sc[L::SC_MW2 + rep * 128 + ct] = -__fmul_rn(dm[rep], (float)(scmn[rep][1] >> 4));
                }
                const __half2 lh = *reinterpret_cast<const __half2*>(&xs2.y);
                sc[L::SC_DX + ct] = __low2float(xs);
                sc[L::SC_SX + ct] = __low2float(lh);
                sc[L::SC_SX2 + ct] = __high2float(lh);
            } else {
                sc[L::SC_DX + ct] = __low2float(xs);
                sc[L::SC_SX + ct] = __high2float(xs);
            }
            // make this thread's fp16 operands visible to the tensor core, then one
            // arrival per warp and barrier
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_F16_FULL + fs));
                mbar_arrive(bar(B_SC_FULL + ss));
                if (blk == KBS - 1) mbar_arrive(bar(B_RAW_EMPTY + sl));
            }
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(AUX_REGS));
        if (warp == EPI_WARPS + CVT_WARPS && lane == 0) {
            // ---- TMA producer: raw int8 / 4-bit tiles and fp16 scales, KBS
            // blocks a stage, RS stages in flight
            int gs = 0;
            for (; gs < total_stages; ++gs) {
                const int sl = gs % RS, u = gs / RS;
                if (u > 0 && !mbar_wait(bar(B_RAW_EMPTY + sl), (u - 1) & 1, abort_flag)) break;
                const int i = gs / spi, s = gs - i * spi;
                if (s == 0) {
                    const Item J = load_item<GU>(P, (int)blockIdx.x + i * (int)gridDim.x);
                    ring[i % ITEM_RING] = make_int4(J.p, J.r0, J.rows, J.w0);
                }
                const Item I = item(i);
                const uint32_t st = sbase + sl * L::STAGE;
                const uint32_t fb = bar(B_RAW_FULL + sl);
                mbar_expect_tx(fb, L::TX);
                // scale-plane coordinate of the stage: its first block, or for
                // Q2_K its super-block (two stages each) and first sub-block
                const int sy = L::QK2 ? s / 2 : s * KBS;
                if (GU) {
                    tma_4d(&mW, fb, st + L::O_W, s * L::WROW, I.w0, 0, I.p);
                    tma_4d(&mWs, fb, st + L::O_WS, I.w0, sy, 0, I.p);
                    if (L::WM_RAW) tma_4d(&mWm, fb, st + L::O_WM, I.w0, sy, 0, I.p);
                    if (L::QK2) tma_4d(&mWc, fb, st + L::O_WC, I.w0, s * 2 * KBS, 0, I.p);
                } else {
                    tma_3d(&mW, fb, st + L::O_W, s * L::WROW, I.w0, I.p);
                    tma_3d(&mWs, fb, st + L::O_WS, I.w0, sy, I.p);
                    if (L::WM_RAW) tma_3d(&mWm, fb, st + L::O_WM, I.w0, sy, I.p);
                    if (L::QK2) tma_3d(&mWc, fb, st + L::O_WC, I.w0, s * 2 * KBS, I.p);
                }
                tma_2d(&mX, fb, st + L::O_X, s * 128, I.r0);
                // activation scales: 4-byte (d, s), or 8-byte D2S6 entries as two words
                tma_2d(&mXs, fb, st + L::O_XS, s * KBS * (L::QK2 ? 2 : 1), I.r0);
            }
            // drain the copies still in flight before the CTA may exit (waits
            // only on the abort path)
            for (int g = (gs > RS ? gs - RS : 0); g < gs; ++g) {
                long long t0 = clock64();
                bool landed = false;
                while (!(landed = mbar_try_wait(bar(B_RAW_FULL + g % RS), (g / RS) & 1)) &&
                       clock64() - t0 < TIMEOUT_CYCLES) {
                }
                if (!landed) *abort_flag = 1;  // reported as MOE_DEV_ERR_TIMEOUT
            }
        } else if (warp == EPI_WARPS + CVT_WARPS + 1 && lane == 0) {
            // ---- MMA issuer: block idx's products into TMEM buffer idx % NTB,
            // 2 x (M=128, N<=128, K=16) per matrix; one commit releases the
            // partials to the epilogue, a second the fp16 slot to the converters
            int idx = 0;
            int mi = 0, mb = 0;  // item and block within the item of idx
            for (; idx < total; ++idx) {
                const int fs = idx % NFS, tb = idx % NTB;
                if (!mbar_wait2(bar(B_F16_FULL + fs), (idx / NFS) & 1, bar(B_TM_EMPTY + tb),
                                ((idx / NTB) - 1) & 1, idx >= NTB, abort_flag))
                    break;
                tc_fence_after();
                const Item I = item(mi);  // read after the barrier that orders it
                if (++mb == nb) {
                    mb = 0;
                    ++mi;
                }
                const uint32_t fa = sbase + L::O_F16 + fs * F16_SLOT;
                const uint32_t fbB = fa + F16_A;
                const uint32_t id = idesc_f16(BM, I.ncols);
#pragma unroll
                for (int mat = 0; mat < 2; ++mat) {
#pragma unroll
                    for (int k16 = 0; k16 < 2; ++k16) {
                        mma_f16(tmem + tb * 256 + mat * 128,
                                sdesc(fa + mat * (BM * 64) + k16 * 256, 128, 512),
                                sdesc(fbB + k16 * 256, 128, 512), id, (uint32_t)k16);
                    }
                }
                if (!(idx == P.stall_idx && blockIdx.x == 0)) mma_commit(bar(B_TM_FULL + tb));
                mma_commit(bar(B_F16_EMPTY + fs));
            }
            // the last committed group must land before TMEM is freed
            if (idx > 0) {
                const int last = idx - 1;
                long long t0 = clock64();
                bool landed = false;
                while (!(landed = mbar_try_wait(bar(B_TM_FULL + last % NTB), (last / NTB) & 1)) &&
                       clock64() - t0 < TIMEOUT_CYCLES) {
                }
                if (!landed) *abort_flag = 1;  // reported as MOE_DEV_ERR_TIMEOUT
            }
        }
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

bool debug() {
    static const bool on = std::getenv("MOE_DEBUG") != nullptr;
    return on;
}

// MOE_TEST_STALL_BLOCK=n: the failure-detection test's hook (Params::stall_idx);
// read at every launch so that a test can set and clear it
int test_stall_idx() {
    const char* v = std::getenv("MOE_TEST_STALL_BLOCK");
    return v ? std::atoi(v) : -1;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
              const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle sw, const char* what) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), (const cuuint64_t*)dims,
                    (const cuuint64_t*)strides, (const cuuint32_t*)box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && debug()) {
        std::fprintf(stderr, "moe_q8: tensor map %s rejected (CUresult %d), rank %d base %p dims",
                     what, (int)r, rank, base);
        for (int i = 0; i < rank; ++i) std::fprintf(stderr, " %llu", (unsigned long long)dims[i]);
        std::fprintf(stderr, " strides");
        for (int i = 0; i + 1 < rank; ++i)
            std::fprintf(stderr, " %llu", (unsigned long long)strides[i]);
        std::fprintf(stderr, " box");
        for (int i = 0; i < rank; ++i) std::fprintf(stderr, " %u", box[i]);
        std::fprintf(stderr, "\n");
    }
    return r == CUDA_SUCCESS;
}

// The register split relies on the launch giving every thread exactly
// LAUNCH_REGS registers (setmaxnreg.inc waits until warpgroup 2 has released
// enough): check the compiled kernel, and opt it into its shared memory, once
// per device (the opt-in is a property of the device's context) before any
// launch there.
constexpr int kMaxDevices = 64;

template <int WT, bool GU, bool FUSED = false>
bool kernel_ready() {
    static std::mutex mu;
    static signed char state[kMaxDevices] = {};  // 0 unknown, 1 ready, -1 unusable
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (state[dev] != 0) return state[dev] == 1;
    state[dev] = -1;
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, mmq_tc_kernel<WT, GU, FUSED>);
    if (e != cudaSuccess) {
        if (debug()) std::fprintf(stderr, "moe_q8: mmq_tc attributes: %s\n", cudaGetErrorString(e));
        return false;
    }
    if (a.numRegs != LAUNCH_REGS || a.maxThreadsPerBlock < THREADS) {
        if (debug())
            std::fprintf(stderr, "moe_q8: mmq_tc built with %d registers / %d threads, want %d / %d\n",
                         a.numRegs, a.maxThreadsPerBlock, LAUNCH_REGS, THREADS);
        return false;
    }
    e = cudaFuncSetAttribute(mmq_tc_kernel<WT, GU, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay<WT>::SMEM);
    if (e != cudaSuccess) {
        if (debug()) std::fprintf(stderr, "moe_q8: smem attribute failed: %s\n", cudaGetErrorString(e));
        return false;
    }
    state[dev] = 1;
    return true;
}

// SM count of the current device, looked up once per device
int device_sms() {
    static std::mutex mu;
    static int sms[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms[dev];
}

template <int WT, bool GU, bool FUSED>
int launch(const uint8_t* group_base, size_t slot_stride, int E, const int8_t* xq,
           const uint16_t* xds, int R, int d, int f, float* out, uint8_t* ws, const WsLayout& W,
           const MmqFused& F, cudaStream_t stream) {
    using L = Lay<WT>;
    const RecLayout RL = rec_layout(WT, d, f);
    const int K = GU ? d : f;          // reduction
    const int rows = GU ? f : d;       // weight rows per matrix
    const MatLayout& ML = GU ? RL.gu : RL.dn;
    const uint8_t* mbase = group_base + (GU ? RL.gate : RL.down);
    const uint64_t S = (uint64_t)E;    // slots addressable in the group buffer
    const uint64_t wrow = (uint64_t)quant_row_bytes(WT, K);
    const CUtensorMapSwizzle wsw = WT == MOE_W_Q8_0   ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : WT == MOE_W_Q4_1 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
    // scale planes: per 32-block [K/32][rows], or Q2_K's per super-block
    // [K/256][rows] (d, dmin) with one stage loading one super-block row
    const uint64_t n_sb = (uint64_t)(K / (L::QK2 ? QKK : QK));
    const uint32_t sbox = L::QK2 ? 1u : (uint32_t)KBS;
    CUtensorMap mW, mWs, mWm, mWc, mX, mXs;
    bool ok = true;
    if (GU) {
        uint64_t dq[4] = {wrow, (uint64_t)rows, 2, S};
        uint64_t sq[3] = {wrow, RL.gu.bytes, slot_stride};
        uint32_t bq[4] = {(uint32_t)L::WROW, BM, 2, 1};
        ok &= make_map(&mW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, mbase + ML.q, dq, sq, bq,
                       wsw, "W (gate/up)");
        uint64_t ds[4] = {(uint64_t)rows, n_sb, 2, S};
        uint64_t ss[3] = {(uint64_t)rows * 2, RL.gu.bytes, slot_stride};
        uint32_t bs[4] = {BM, sbox, 2, 1};
        ok &= make_map(&mWs, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, mbase + ML.d, ds, ss, bs,
                       CU_TENSOR_MAP_SWIZZLE_NONE, "W scales (gate/up)");
        ok &= make_map(&mWm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                       mbase + (L::WM_RAW ? ML.m : ML.d), ds, ss, bs,
                       CU_TENSOR_MAP_SWIZZLE_NONE, "W mins (gate/up)");
        if (L::QK2) {
            uint64_t dc[4] = {(uint64_t)rows, (uint64_t)(K / 16), 2, S};
            uint64_t sc[3] = {(uint64_t)rows, RL.gu.bytes, slot_stride};
            uint32_t bc[4] = {BM, 2 * KBS, 2, 1};
            ok &= make_map(&mWc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, mbase + ML.s, dc, sc, bc,
                           CU_TENSOR_MAP_SWIZZLE_NONE, "W sub-block scales (gate/up)");
        } else {
            mWc = mWs;  // unused
        }
    } else {
        uint64_t dq[3] = {wrow, (uint64_t)rows, S};
        uint64_t sq[2] = {wrow, slot_stride};
        uint32_t bq[3] = {(uint32_t)L::WROW, 2 * BM, 1};
        ok &= make_map(&mW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, mbase + ML.q, dq, sq, bq,
                       wsw, "W (down)");
        uint64_t ds[3] = {(uint64_t)rows, n_sb, S};
        uint64_t ss[2] = {(uint64_t)rows * 2, slot_stride};
        uint32_t bs[3] = {2 * BM, sbox, 1};
        ok &= make_map(&mWs, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, mbase + ML.d, ds, ss, bs,
                       CU_TENSOR_MAP_SWIZZLE_NONE, "W scales (down)");
        ok &= make_map(&mWm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                       mbase + (L::WM_RAW ? ML.m : ML.d), ds, ss, bs,
                       CU_TENSOR_MAP_SWIZZLE_NONE, "W mins (down)");
        if (L::QK2) {
            uint64_t dc[3] = {(uint64_t)rows, (uint64_t)(K / 16), S};
            uint64_t sc[2] = {(uint64_t)rows, slot_stride};
            uint32_t bc[3] = {2 * BM, 2 * KBS, 1};
            ok &= make_map(&mWc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, mbase + ML.s, dc, sc, bc,
                           CU_TENSOR_MAP_SWIZZLE_NONE, "W sub-block scales (down)");
        } else {
            mWc = mWs;  // unused
        }
    }
    {
        uint64_t dx[2] = {(uint64_t)K, (uint64_t)R};
        uint64_t sx[1] = {(uint64_t)K};
        uint32_t bx[2] = {128, BN};
        ok &= make_map(&mX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, xq, dx, sx, bx,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X");
        // (d, s) as one word per block, or D2S6's 8 bytes as two words
        const uint64_t wpb = L::QK2 ? 2 : 1;
        uint64_t dd[2] = {(uint64_t)(K / QK) * wpb, (uint64_t)R};
        uint64_t sd[1] = {(uint64_t)(K / QK) * 4 * wpb};
        uint32_t bd[2] = {(uint32_t)(KBS * wpb), BN};
        ok &= make_map(&mXs, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, xds, dd, sd, bd,
                       CU_TENSOR_MAP_SWIZZLE_NONE, "X scales");
    }
    if (!ok) return MOE_ERR_CUDA;

    if (!kernel_ready<WT, GU, FUSED>()) return MOE_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    Params P;
    P.tiles = (const int4*)(ws + W.tiles);
    P.n_tiles = (const int32_t*)(ws + W.counters) + MMQ_COUNTER_NTILES;
    P.mt_count = GU ? f / BM : d / (2 * BM);
    P.nb = K / QK;
    P.n_out = GU ? f : d;
    P.R = R;
    P.out = out;
    P.err = (uint32_t*)(ws + W.err);
    P.hq = GU ? F.hq : nullptr;
    P.hds = GU ? reinterpret_cast<__half2*>(F.hds) : nullptr;
    P.comb = GU ? nullptr : F.comb;
    P.src = F.src;
    P.slot = F.slot;
    P.wts = F.w;
    P.arrivals = F.arrivals;
    P.K = F.K;
    P.T = F.T;
    P.stall_idx = test_stall_idx();
    long long upper = ((long long)R / BN + E + 1) * P.mt_count;
    int grid = (int)(upper < sms ? upper : sms);
    mmq_tc_kernel<WT, GU, FUSED><<<grid, THREADS, L::SMEM, stream>>>(mW, mWs, mWm, mWc, mX, mXs, P);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess && debug())
        std::fprintf(stderr, "moe_q8: mmq_tc launch failed: %s (grid %d, smem %d)\n",
                     cudaGetErrorString(e), grid, L::SMEM);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace tc

bool mmq_tc_supported(int wtype, bool gateup, int d, int f) {
    if (wtype != MOE_W_Q8_0 && wtype != MOE_W_Q4_1 && wtype != MOE_W_Q2_0 && wtype != MOE_W_Q2_K)
        return false;
    if (d % 256 || f % 128) return false;  // whole 128-row weight tiles, 128-wide K stages
    if (wtype == MOE_W_Q2_K && f % 256) return false;  // whole super-blocks of the down reduction
    if (tc::encode_fn() == nullptr) return false;
    if (wtype == MOE_W_Q8_0)
        return gateup ? tc::kernel_ready<MOE_W_Q8_0, true>() : tc::kernel_ready<MOE_W_Q8_0, false>();
    if (wtype == MOE_W_Q2_0)
        return gateup ? tc::kernel_ready<MOE_W_Q2_0, true>() : tc::kernel_ready<MOE_W_Q2_0, false>();
    if (wtype == MOE_W_Q2_K)
        return gateup ? tc::kernel_ready<MOE_W_Q2_K, true>() : tc::kernel_ready<MOE_W_Q2_K, false>();
    return gateup ? tc::kernel_ready<MOE_W_Q4_1, true>() : tc::kernel_ready<MOE_W_Q4_1, false>();
}

namespace tc {
template <int WT>
int launch_wt(bool gateup, const uint8_t* group_base, size_t slot_stride, int E, const int8_t* xq,
              const uint16_t* xds, int R, int d, int f, float* out, uint8_t* ws,
              const WsLayout& W, const MmqFused& F, cudaStream_t stream) {
    const bool fused = gateup ? F.hq != nullptr : F.comb != nullptr;
    if (gateup)
        return fused ? launch<WT, true, true>(group_base, slot_stride, E, xq, xds, R, d, f, out, ws,
                                              W, F, stream)
                     : launch<WT, true, false>(group_base, slot_stride, E, xq, xds, R, d, f, out,
                                               ws, W, F, stream);
    return fused ? launch<WT, false, true>(group_base, slot_stride, E, xq, xds, R, d, f, out, ws, W,
                                           F, stream)
                 : launch<WT, false, false>(group_base, slot_stride, E, xq, xds, R, d, f, out, ws,
                                            W, F, stream);
}
}  // namespace tc

int launch_mmq_tc(int wtype, bool gateup, const uint8_t* group_base, size_t slot_stride,
                  const int32_t* active, const int32_t* n_active, const int32_t* offsets, int E,
                  const int8_t* xq, const uint16_t* xds, int R, int d, int f, float* out,
                  uint8_t* ws, const WsLayout& W, const MmqFused& F, cudaStream_t stream) {
    int rc = launch_mmq_tiles(active, n_active, offsets, E, R, tc::BN, ws, W, stream);
    if (rc != MOE_OK) return rc;
    if (wtype == MOE_W_Q8_0)
        return tc::launch_wt<MOE_W_Q8_0>(gateup, group_base, slot_stride, E, xq, xds, R, d, f, out,
                                         ws, W, F, stream);
    if (wtype == MOE_W_Q2_0)
        return tc::launch_wt<MOE_W_Q2_0>(gateup, group_base, slot_stride, E, xq, xds, R, d, f, out,
                                         ws, W, F, stream);
    if (wtype == MOE_W_Q2_K)
        return tc::launch_wt<MOE_W_Q2_K>(gateup, group_base, slot_stride, E, xq, xds, R, d, f, out,
                                         ws, W, F, stream);
    return tc::launch_wt<MOE_W_Q4_1>(gateup, group_base, slot_stride, E, xq, xds, R, d, f, out, ws,
                                     W, F, stream);
}

}  // namespace moe
