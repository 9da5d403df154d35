// Stages 2 and 5: q8_1 quantization.
//
// "#1368 prefill: quantize each token's MoE input once and scatter it to its k
// rows (the same bytes)", intro: each token row is read and quantized once and
// its blocks are written to all K rows slot[t*K+k]; the per-row gather form
// (row r quantizes token src[r]) and the hidden-row re-quantization (identity
// map) share the block arithmetic.
//
// q8_1 block: d = amax/127, q = round-half-away(x/d), s = d*sum(q); d and s
// stored as binary16.  All divisions are IEEE (__fdiv_rn), the product s is a
// single rounding (__fmul_rn), and nothing is flushed to zero, so the bytes
// match any correct implementation of the definition.
//
// Mapping: one thread per 8 consecutive values (two 16-byte loads), four
// threads per 32-block, amax and sum(q) reduced with two xor shuffles.  A warp
// covers 256 consecutive values of a row: its q stores are 256 contiguous bytes
// per destination row and its (d, s) stores 32 contiguous bytes.
#include "common.cuh"

namespace moe {

enum QuantMode { QUANT_SCATTER = 0, QUANT_GATHER = 1, QUANT_IDENTITY = 2 };

struct Q8Block8 {
    uint2 q;      // 8 int8 quants
    __half2 ds;   // (d, s), valid in every lane of the 4-lane group
};

__device__ __forceinline__ Q8Block8 quantize8(const float4 a, const float4 b) {
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    Q8Block8 r;
    int sum = 0;
    uint32_t lo = 0, hi = 0;
    float d = 0.0f;
    if (amax != 0.0f) {
        d = __fdiv_rn(amax, 127.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float x = roundf(__fdiv_rn(v[i], d));
            x = fminf(127.0f, fmaxf(-127.0f, x));
            int qi = (int)x;
            sum += qi;
            uint32_t byte = (uint32_t)(qi & 0xff);
            if (i < 4) lo |= byte << (8 * i);
            else hi |= byte << (8 * (i - 4));
        }
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    float s = __fmul_rn(d, (float)sum);
    r.q = make_uint2(lo, hi);
    r.ds = __halves2half2(__float2half_rn(d), __float2half_rn(s));
    return r;
}

// x: [n_src_rows][d]; writes rows of q [R][d] / ds [R][d/32].
template <int MODE>
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(
    const float* __restrict__ x, int n_src_rows, int d, int K, const int32_t* __restrict__ map,
    int R, int8_t* __restrict__ q, __half2* __restrict__ ds, long long n_units) {
    const int upr = d / 8;  // units (of 8 values) per row
    const long long stride = (long long)gridDim.x * blockDim.x;
    // round the bound up to a whole warp so every shuffle has all 32 lanes
    const long long bound = (n_units + 31) / 32 * 32;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < bound; u += stride) {
        bool in = u < n_units;
        long long row = in ? u / upr : 0;
        int c = in ? (int)(u % upr) * 8 : 0;
        long long srow = row;  // the x row this unit reads
        if (MODE == QUANT_GATHER) {
            int t = in ? map[row] : -1;
            in = in && (unsigned)t < (unsigned)n_src_rows;
            srow = in ? t : 0;
        }
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (in) {
            const float4* p = reinterpret_cast<const float4*>(x + srow * d + c);
            if (MODE == QUANT_GATHER) {  // rows are re-read K times: keep them cached
                a = __ldg(p);
                b = __ldg(p + 1);
            } else {  // read once: stream past L2
                a = __ldcs(p);
                b = __ldcs(p + 1);
            }
        }
        Q8Block8 blk = quantize8(a, b);
        if (!in) continue;
        bool lead = (threadIdx.x & 3) == 0;
        if (MODE == QUANT_SCATTER) {
            for (int k = 0; k < K; ++k) {
                int r = map[row * K + k];
                if ((unsigned)r >= (unsigned)R) continue;
                *reinterpret_cast<uint2*>(q + (size_t)r * d + c) = blk.q;
                if (lead) ds[(size_t)r * (d / QK) + c / QK] = blk.ds;
            }
        } else {
            if (row >= R) continue;
            *reinterpret_cast<uint2*>(q + (size_t)row * d + c) = blk.q;
            if (lead) ds[(size_t)row * (d / QK) + c / QK] = blk.ds;
        }
    }
}

static int quant_grid(long long n_units) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (n_units + 255) / 256;
    long long cap = (long long)sms * 8;  // 8 resident blocks of 256 per SM
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

int launch_quantize_scatter(const float* x, int T, int d, int K, const int32_t* slot, int R,
                            int8_t* q, uint16_t* ds, cudaStream_t stream) {
    long long n = (long long)T * (d / 8);
    if (n == 0) return MOE_OK;
    quantize_q8_1_kernel<QUANT_SCATTER><<<quant_grid(n), 256, 0, stream>>>(
        x, T, d, K, slot, R, q, reinterpret_cast<__half2*>(ds), n);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_quantize_gather(const float* x, int T, int d, const int32_t* src, int R, int8_t* q,
                           uint16_t* ds, cudaStream_t stream) {
    long long n = (long long)R * (d / 8);
    if (n == 0) return MOE_OK;
    quantize_q8_1_kernel<QUANT_GATHER><<<quant_grid(n), 256, 0, stream>>>(
        x, T, d, 1, src, R, q, reinterpret_cast<__half2*>(ds), n);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_requant_hidden(const float* h, int R, int f, int8_t* hq, uint16_t* hds,
                          cudaStream_t stream) {
    long long n = (long long)R * (f / 8);
    if (n == 0) return MOE_OK;
    quantize_q8_1_kernel<QUANT_IDENTITY><<<quant_grid(n), 256, 0, stream>>>(
        h, R, f, 1, nullptr, R, hq, reinterpret_cast<__half2*>(hds), n);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
