// Stage 7: top-k combine ("#1282 prefill: STRATA_PREFILL_CPU_SHARE=auto ...",
// section "What it does": every row of Dm is weighted by its token's top-k
// weight and a token's rows are summed).
//   out[t, i] = fma chain over k ascending of w[t*K+k] * y[slot[t*K+k], i], from 0.
// One thread per 4 outputs (16-byte loads and stores); a warp reads 512
// contiguous bytes of each of the token's K rows.
#include "common.cuh"
#include "mmq.cuh"

namespace moe {

__global__ void __launch_bounds__(256) combine_topk_kernel(const float4* __restrict__ y, int R,
                                                           const int32_t* __restrict__ slot,
                                                           const float* __restrict__ w, int T,
                                                           int K, int d4,
                                                           float4* __restrict__ out) {
    const long long n = (long long)T * d4;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += stride) {
        long long t = idx / d4;
        int c = (int)(idx % d4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < K; ++k) {
            int r = __ldg(slot + t * K + k);
            if ((unsigned)r >= (unsigned)R) continue;
            float wk = __ldg(w + t * K + k);
            float4 v = __ldcs(y + (size_t)r * d4 + c);
            acc.x = __fmaf_rn(wk, v.x, acc.x);
            acc.y = __fmaf_rn(wk, v.y, acc.y);
            acc.z = __fmaf_rn(wk, v.z, acc.z);
            acc.w = __fmaf_rn(wk, v.w, acc.w);
        }
        __stcs(out + idx, acc);
    }
}

int launch_combine_topk(const float* y, int R, const int32_t* slot, const float* w, int T, int K,
                        int d, float* out, cudaStream_t stream) {
    long long n = (long long)T * (d / 4);
    if (n == 0) return MOE_OK;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (n + 255) / 256, cap = (long long)sms * 8;
    int grid = (int)(blocks < cap ? blocks : cap);
    combine_topk_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(y), R, slot, w,
                                                  T, K, d / 4, reinterpret_cast<float4*>(out));
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Before the down projection with the combine: arrivals[t][cb] = the number of
// valid rows of token t (slot in [0, R)) for every 256-column block cb, and the
// output row of a token with no valid row is zero (no item will combine it).
__global__ void __launch_bounds__(256) combine_arrivals_kernel(const int32_t* __restrict__ slot,
                                                               int T, int K, int R, int ncb,
                                                               int d4, int32_t* __restrict__ arrivals,
                                                               float4* __restrict__ out) {
    const int stride = gridDim.x * blockDim.x;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += stride) {
        int need = 0;
        for (int k = 0; k < K; ++k) need += (unsigned)__ldg(slot + (size_t)t * K + k) < (unsigned)R;
        for (int cb = 0; cb < ncb; ++cb) arrivals[(size_t)t * ncb + cb] = need;
        if (need == 0)
            for (int c = 0; c < d4; ++c) out[(size_t)t * d4 + c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

int launch_combine_arrivals(const int32_t* slot, int T, int K, int R, int d, int32_t* arrivals,
                            float* out, cudaStream_t stream) {
    if (T == 0) return MOE_OK;
    int blocks = (T + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    combine_arrivals_kernel<<<blocks, 256, 0, stream>>>(slot, T, K, R, (d + 255) / 256, d / 4,
                                                        arrivals, reinterpret_cast<float4*>(out));
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
