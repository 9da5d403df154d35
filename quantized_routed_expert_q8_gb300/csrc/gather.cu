// Stage 3: group gather ("#439 prefill: a group's expert gathers in one launch",
// section "What"; "#372 Prompt path: an MMQ group's experts gathered in one
// launch ...", "What changes").  One launch copies up to 16 experts' records into
// their group-buffer slots with blockIdx.y = expert -- the same bytes to the
// same places as one copy per expert.  16-byte vector copies when everything is
// 16-byte aligned, a byte copy otherwise (the pages' unaligned / odd-size
// fallback).
#include "common.cuh"

namespace moe {

struct GroupIds {
    int32_t id[16];
};

// Copy n16 uint4 from src to dst with this block's share of the grid's x extent.
__device__ __forceinline__ void copy_vec(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         size_t n16) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
              d = __ldcs(src + i + 3 * stride);
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = __ldcs(src + i);
}

__device__ __forceinline__ void copy_bytes(const uint8_t* __restrict__ src,
                                           uint8_t* __restrict__ dst, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
}

template <bool VEC>
__global__ void __launch_bounds__(256) group_gather_kernel(const uint8_t* __restrict__ arena,
                                                           size_t rec_bytes, size_t arena_stride,
                                                           GroupIds g, int first_slot,
                                                           uint8_t* __restrict__ buf,
                                                           size_t slot_stride) {
    int j = blockIdx.y;
    const uint8_t* s = arena + (size_t)g.id[j] * arena_stride;
    uint8_t* dd = buf + (size_t)(first_slot + j) * slot_stride;
    if (VEC) copy_vec(reinterpret_cast<const uint4*>(s), reinterpret_cast<uint4*>(dd), rec_bytes / 16);
    else copy_bytes(s, dd, rec_bytes);
}

// The whole layer's groups in one launch: a persistent grid walks the units
// (active position p, 128 KB part of its record) up to the device-side count, so
// that no block is launched for an expert that is not routed.
constexpr size_t PART = 128u << 10;  // bytes of a record one unit copies

__device__ __forceinline__ void copy_range_vec(const uint4* __restrict__ src,
                                               uint4* __restrict__ dst, size_t n16) {
    size_t i = threadIdx.x;
    const size_t st = blockDim.x;
    for (; i + 3 * st < n16; i += 4 * st) {
        uint4 a = __ldcs(src + i), b = __ldcs(src + i + st), c = __ldcs(src + i + 2 * st),
              d = __ldcs(src + i + 3 * st);
        dst[i] = a;
        dst[i + st] = b;
        dst[i + 2 * st] = c;
        dst[i + 3 * st] = d;
    }
    for (; i < n16; i += st) dst[i] = __ldcs(src + i);
}

template <bool VEC>
__global__ void __launch_bounds__(256, 8) group_gather_active_kernel(
    const uint8_t* __restrict__ arena, size_t rec_bytes, size_t arena_stride,
    const int32_t* __restrict__ active, const int32_t* __restrict__ n_active, int max_active,
    uint8_t* __restrict__ base, size_t slot_stride) {
    const int n = min(*n_active, max_active);
    const long long parts = (long long)((rec_bytes + PART - 1) / PART);
    const long long units = (long long)n * parts;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const int p = (int)(u / parts);  // active position
        const size_t off = (size_t)(u % parts) * PART;
        const size_t len = rec_bytes - off < PART ? rec_bytes - off : PART;
        const int e = active[p];
        if (e < 0) continue;
        const uint8_t* s = arena + (size_t)e * arena_stride + off;
        uint8_t* dd = base + (size_t)p * slot_stride + off;
        if (VEC) {
            copy_range_vec(reinterpret_cast<const uint4*>(s), reinterpret_cast<uint4*>(dd), len / 16);
        } else {
            for (size_t i = threadIdx.x; i < len; i += blockDim.x) dd[i] = s[i];
        }
    }
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

static int blocks_per_record(size_t rec_bytes) {
    // ~128 KB per block: enough blocks for HBM bandwidth, few enough to be cheap
    size_t b = (rec_bytes + (128u << 10) - 1) / (128u << 10);
    return (int)(b < 1 ? 1 : (b > 4096 ? 4096 : b));
}

int launch_group_gather(const uint8_t* arena, size_t rec_bytes, size_t arena_stride,
                        const int32_t* ids, int n, int first_slot, uint8_t* buf,
                        size_t slot_stride, cudaStream_t stream) {
    GroupIds g;
    for (int j = 0; j < 16; ++j) g.id[j] = j < n ? ids[j] : 0;
    if (rec_bytes == 0) return MOE_OK;
    bool vec = aligned16(arena) && aligned16(buf) && rec_bytes % 16 == 0 &&
               arena_stride % 16 == 0 && slot_stride % 16 == 0;
    dim3 grid(blocks_per_record(rec_bytes), n);
    if (vec)
        group_gather_kernel<true><<<grid, 256, 0, stream>>>(arena, rec_bytes, arena_stride, g,
                                                            first_slot, buf, slot_stride);
    else
        group_gather_kernel<false><<<grid, 256, 0, stream>>>(arena, rec_bytes, arena_stride, g,
                                                             first_slot, buf, slot_stride);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_group_gather_active(const uint8_t* arena, size_t rec_bytes, size_t arena_stride,
                               const int32_t* active, const int32_t* n_active, int max_active,
                               uint8_t* base, size_t slot_stride, cudaStream_t stream) {
    if (rec_bytes == 0 || max_active <= 0) return MOE_OK;
    bool vec = aligned16(arena) && aligned16(base) && rec_bytes % 16 == 0 &&
               arena_stride % 16 == 0 && slot_stride % 16 == 0;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long units = (long long)max_active * (long long)((rec_bytes + PART - 1) / PART);
    const int grid = (int)(units < (long long)sms * 8 ? units : (long long)sms * 8);  // 8 blocks an SM
    if (vec)
        group_gather_active_kernel<true><<<grid, 256, 0, stream>>>(
            arena, rec_bytes, arena_stride, active, n_active, max_active, base, slot_stride);
    else
        group_gather_active_kernel<false><<<grid, 256, 0, stream>>>(
            arena, rec_bytes, arena_stride, active, n_active, max_active, base, slot_stride);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
