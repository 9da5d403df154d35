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
    int sum = 0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    // d == 0 (amax == 0, or an fp32-subnormal amax <= 63 * 2^-149 whose quotient
    // underflows) leaves x / d undefined: such a block is stored as all-zero
    const float d = __fdiv_rn(amax, 127.0f);
    // d differs between the blocks of a warp (and is zero in some), so every
    // warp-collective operation below sits outside the branches on d
    const bool nz = d != 0.0f;
    float x[16];
    uint32_t need = 0u;  // values whose quotient must be formed exactly
    if (nz) {
        // q = round-half-away(fp32(v / d)).  With a normal d, qa = v * RN(1/d) is
        // within 3 ulp of the IEEE quotient, and |qa| < 128 puts an ulp at
        // <= 2^-17; so unless qa lies within 2^-14 of a half-integer, rounding qa
        // gives the same integer as rounding the quotient.  Otherwise (and for
        // a subnormal d) the quotient itself is formed with an IEEE division.
        const bool fast_ok = d >= 1.17549435e-38f;
        const float r = fast_ok ? __frcp_rn(d) : 0.0f;
        if (!fast_ok) need = 0xFFFFu;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float qa = __fmul_rn(v[i], r);
            const float fr = fabsf(qa) - truncf(fabsf(qa));
            x[i] = roundf(qa);
            if (fabsf(fr - 0.5f) <= 6.103515625e-05f) need |= 1u << i;
        }
    }
    // a warp-uniform branch (every lane votes), so that the divisions run only
    // in the rare warps that need one; need is zero where d is
    if (__any_sync(0xffffffffu, need != 0u)) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if ((need >> i) & 1u) x[i] = roundf(__fdiv_rn(v[i], d));
    }
    if (nz) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int qi = (int)fminf(127.0f, fmaxf(-127.0f, x[i]));
            sum += qi;
            w[i >> 2] |= (uint32_t)(qi & 0xff) << (8 * (i & 3));
        }
    }
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
