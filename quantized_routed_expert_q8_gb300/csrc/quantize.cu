// Stages 2 and 5: q8_1 quantization.
//
// "#1368 prefill: quantize each token's MoE input once and scatter it to its k
// rows (the same bytes)", intro: each token row is read and quantized once and
// its blocks are written to all K rows slot[t*K+k]; the per-row gather form
// (row r quantizes token src[r]) and the hidden-row re-quantization (identity
// map) share the block arithmetic.
//
// q8_1 block: d = amax/127, q = round-half-away(x/d), s = d*sum(q); d and s
// stored as binary16; a block whose d is zero is stored as all-zero.  All divisions are IEEE (__fdiv_rn), the product s is a
// single rounding (__fmul_rn), and nothing is flushed to zero, so the bytes
// match any correct implementation of the definition.
//
// D2S6 layout (the rows Q2_K weights read; the pages name it without defining
// it): the same q and (d, s), followed per block by (s_lo, s_hi) = fp16 of d
// times the sums of q over the block's two 16-value halves.
//
// Mapping: one thread per 16 consecutive values (four 16-byte loads), two
// threads per 32-block, amax and sum(q) reduced with one xor shuffle each.  A
// warp covers 512 consecutive values of a row: each thread stores its 16 quants
// as one 16-byte store, so a warp's q stores are 512 contiguous bytes per
// destination row and its (d, s) stores 64 contiguous bytes (128 for D2S6).
// The thread of the first half of a block holds the sum of its own 16 quants,
// which is s_lo, and receives s_hi's sum from the shuffle.
#include "common.cuh"

namespace moe {

enum QuantMode { QUANT_SCATTER = 0, QUANT_GATHER = 1, QUANT_IDENTITY = 2 };

struct Q8Half {
    uint4 q;      // 16 int8 quants
    __half2 ds;   // (d, s), valid in both lanes of the pair
    __half2 lh;   // D2S6 (s_lo, s_hi), valid in the first-half lane
};

// byte permute: result byte i = byte (sel >> 4i) & 7 of {a, b} (a bytes 0-3)
__device__ __forceinline__ uint32_t prmt_bytes(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

template <bool D2S6>
__device__ __forceinline__ Q8Half quantize16(const float4 (&a)[4]) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[4 * i] = a[i].x;
        v[4 * i + 1] = a[i].y;
        v[4 * i + 2] = a[i].z;
        v[4 * i + 3] = a[i].w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    Q8Half r;
    // d == 0 (amax == 0, or an fp32-subnormal amax <= 63 * 2^-149 whose quotient
    // underflows) leaves x / d undefined: such a block is stored as all-zero
    const float d = __fdiv_rn(amax, 127.0f);
    const bool nz = d != 0.0f;
    // q = round-half-away(fp32(v / d)).  With a normal d, qa = RN(v * RN(1/d))
    // is within 3 ulp of the IEEE quotient (|qa| < 127.0001, so within 2.3e-5),
    // hence unless qa lies within 2^-14 of a half-integer, the nearest integer
    // to qa is the rounded quotient, and no tie can occur, so round-to-nearest-
    // even and round-half-away agree.  That integer comes from one addition of
    // M = 1.5 * 2^23: qa + M lies in [2^23, 2^24), where the spacing is 1, so
    // its bits are 0x4B400000 + q (q in [-127, 127]; the low byte is q's int8
    // byte) and (qa + M) - M = q exactly.  A lane whose block has a subnormal d,
    // or one of whose values lies within 2^-14 of a half-integer
    // (|qa - q| >= 0.5 - 2^-14), forms the IEEE quotients instead.
    constexpr float M = 12582912.0f;
    constexpr uint32_t MB = 0x4B400000u;  // bits of M
    const bool fast_ok = d >= 1.17549435e-38f;
    const float rc = fast_ok ? __frcp_rn(d) : 0.0f;
    uint32_t bq[16];  // bits of q + M
    float off = 0.0f;  // max |qa - q|
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float qa = __fmul_rn(v[i], rc);
        const float t = __fadd_rn(qa, M);
        off = fmaxf(off, fabsf(__fsub_rn(qa, __fsub_rn(t, M))));
        bq[i] = __float_as_uint(t);
    }
    const bool slow = nz && (!fast_ok || off >= 0.49993896484375f);
    // a warp-uniform branch (every lane votes; d differs between the blocks of a
    // warp), so that the divisions run only in the rare warps that need them
    if (__any_sync(0xffffffffu, slow)) {
        if (slow) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x = fminf(127.0f, fmaxf(-127.0f, roundf(__fdiv_rn(v[i], d))));
                bq[i] = __float_as_uint(__fadd_rn(x, M));
            }
        }
    }
    if (!nz) {
#pragma unroll
        for (int i = 0; i < 16; ++i) bq[i] = MB;  // q = 0
    }
    // the quants are the low bytes of bq; sum(q) = sum(bq) - 16 * MB (mod 2^32)
    uint32_t w[4], acc = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = prmt_bytes(bq[4 * k], bq[4 * k + 1], 0x0040u);
        const uint32_t hi = prmt_bytes(bq[4 * k + 2], bq[4 * k + 3], 0x0040u);
        w[k] = prmt_bytes(lo, hi, 0x5410u);
        acc += bq[4 * k] + bq[4 * k + 1] + bq[4 * k + 2] + bq[4 * k + 3];
    }
    const int sum = (int)(acc - 16u * MB);
    const int other = __shfl_xor_sync(0xffffffffu, sum, 1);
    const float s = __fmul_rn(d, (float)(sum + other));
    r.q = make_uint4(w[0], w[1], w[2], w[3]);
    r.ds = __halves2half2(__float2half_rn(d), __float2half_rn(s));
    if (D2S6)
        r.lh = __halves2half2(__float2half_rn(__fmul_rn(d, (float)sum)),
                              __float2half_rn(__fmul_rn(d, (float)other)));
    return r;
}

// one block's ds entries: (d, s), or (d, s, s_lo, s_hi) as one 8-byte store
template <bool D2S6>
__device__ __forceinline__ void store_ds(__half2* ds, size_t blk, const Q8Half& b) {
    if (D2S6) {
        uint2 v;
        v.x = *reinterpret_cast<const uint32_t*>(&b.ds);
        v.y = *reinterpret_cast<const uint32_t*>(&b.lh);
        reinterpret_cast<uint2*>(ds)[blk] = v;
    } else {
        ds[blk] = b.ds;
    }
}

// x: [n_src_rows][d]; writes rows of q [R][d] / ds [R][d/32] (x2 for D2S6).
template <int MODE, bool D2S6>
__global__ void __launch_bounds__(256, 4) quantize_q8_1_kernel(
    const float* __restrict__ x, int n_src_rows, int d, int K, const int32_t* __restrict__ map,
    int R, int8_t* __restrict__ q, __half2* __restrict__ ds, long long n_units) {
    const int upr = d / 16;  // units (of 16 values) per row
    const long long stride = (long long)gridDim.x * blockDim.x;
    // round the bound up to a whole warp so every shuffle has all 32 lanes
    const long long bound = (n_units + 31) / 32 * 32;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < bound; u += stride) {
        bool in = u < n_units;
        const long long row = in ? u / upr : 0;
        const int c = in ? (int)(u % upr) * 16 : 0;
        long long srow = row;  // the x row this unit reads
        if (MODE == QUANT_GATHER) {
            const int t = in ? map[row] : -1;
            in = in && (unsigned)t < (unsigned)n_src_rows;
            srow = in ? t : 0;
        }
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in) {
            const float4* p = reinterpret_cast<const float4*>(x + srow * d + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)  // gather rows are re-read K times: keep them cached;
                a[i] = MODE == QUANT_GATHER ? __ldg(p + i) : __ldcs(p + i);  // else stream past L2
        }
        const Q8Half blk = quantize16<D2S6>(a);
        if (!in) continue;
        const bool lead = (threadIdx.x & 1) == 0;
        if (MODE == QUANT_SCATTER) {
            for (int k = 0; k < K; ++k) {
                const int r = map[row * K + k];
                if ((unsigned)r >= (unsigned)R) continue;
                *reinterpret_cast<uint4*>(q + (size_t)r * d + c) = blk.q;
                if (lead) store_ds<D2S6>(ds, (size_t)r * (d / QK) + c / QK, blk);
            }
        } else {
            if (row >= R) continue;
            *reinterpret_cast<uint4*>(q + (size_t)row * d + c) = blk.q;
            if (lead) store_ds<D2S6>(ds, (size_t)row * (d / QK) + c / QK, blk);
        }
    }
}

static int quant_grid(long long n_units) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (n_units + 255) / 256;
    long long cap = (long long)sms * 4;  // 4 resident blocks of 256 per SM (64 registers)
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

int launch_quantize_scatter(const float* x, int T, int d, int K, const int32_t* slot, int R,
                            int8_t* q, uint16_t* ds, bool d2s6, cudaStream_t stream) {
    long long n = (long long)T * (d / 16);
    if (n == 0) return MOE_OK;
    __half2* ds2 = reinterpret_cast<__half2*>(ds);
    if (d2s6)
        quantize_q8_1_kernel<QUANT_SCATTER, true><<<quant_grid(n), 256, 0, stream>>>(
            x, T, d, K, slot, R, q, ds2, n);
    else
        quantize_q8_1_kernel<QUANT_SCATTER, false><<<quant_grid(n), 256, 0, stream>>>(
            x, T, d, K, slot, R, q, ds2, n);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_quantize_gather(const float* x, int T, int d, const int32_t* src, int R, int8_t* q,
                           uint16_t* ds, bool d2s6, cudaStream_t stream) {
    long long n = (long long)R * (d / 16);
    if (n == 0) return MOE_OK;
    __half2* ds2 = reinterpret_cast<__half2*>(ds);
    if (d2s6)
        quantize_q8_1_kernel<QUANT_GATHER, true><<<quant_grid(n), 256, 0, stream>>>(
            x, T, d, 1, src, R, q, ds2, n);
    else
        quantize_q8_1_kernel<QUANT_GATHER, false><<<quant_grid(n), 256, 0, stream>>>(
            x, T, d, 1, src, R, q, ds2, n);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_requant_hidden(const float* h, int R, int f, int8_t* hq, uint16_t* hds, bool d2s6,
                          cudaStream_t stream) {
    long long n = (long long)R * (f / 16);
    if (n == 0) return MOE_OK;
    __half2* ds2 = reinterpret_cast<__half2*>(hds);
    if (d2s6)
        quantize_q8_1_kernel<QUANT_IDENTITY, true><<<quant_grid(n), 256, 0, stream>>>(
            h, R, f, 1, nullptr, R, hq, ds2, n);
    else
        quantize_q8_1_kernel<QUANT_IDENTITY, false><<<quant_grid(n), 256, 0, stream>>>(
            h, R, f, 1, nullptr, R, hq, ds2, n);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
