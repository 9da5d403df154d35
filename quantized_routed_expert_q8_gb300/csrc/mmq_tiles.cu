// Work list of the grouped MMQ kernels: one entry per (active expert, row tile).
//
// Built on the device from offsets[] and the active list, so the layer needs no
// host round trip.  Entries are ordered longest-first (LPT): all full tiles,
// then the partial tiles by descending row count, which lets the persistent
// tensor-core kernel hand out the big work items before the ragged tails.
#include "common.cuh"
#include "mmq.cuh"

namespace moe {

__global__ void __launch_bounds__(1024) mmq_tiles_kernel(const int32_t* __restrict__ active,
                                                         const int32_t* __restrict__ n_active,
                                                         const int32_t* __restrict__ offsets,
                                                         int E, int R, int BM,
                                                         int4* __restrict__ tiles,
                                                         int32_t* __restrict__ n_tiles,
                                                         int32_t* __restrict__ ticket,
                                                         int max_tiles, uint32_t* err) {
    __shared__ int s_full, s_bad;
    __shared__ int part_hist[256];  // partial tiles by row count (BM <= 256)
    if (threadIdx.x == 0) {
        s_full = 0;
        s_bad = 0;
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) part_hist[i] = 0;
    __syncthreads();
    int na = min(*n_active, E);
    // pass 1: count full tiles and partial tiles per size
    for (int p = threadIdx.x; p < na; p += blockDim.x) {
        int e = active[p];
        if ((unsigned)e >= (unsigned)E) {
            s_bad = 1;
            continue;
        }
        int lo = offsets[e], hi = offsets[e + 1];
        if (lo < 0 || hi > R || hi < lo) {
            s_bad = 1;
            lo = max(0, min(lo, R));
            hi = max(lo, min(hi, R));
        }
        int cnt = hi - lo;
        atomicAdd(&s_full, cnt / BM);
        if (cnt % BM) atomicAdd(&part_hist[cnt % BM], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // partial tiles start after the full ones, larger remainders first
        int run = s_full;
        for (int rem = BM - 1; rem >= 1; --rem) {
            int c = part_hist[rem];
            part_hist[rem] = run;
            run += c;
        }
        if (s_bad) set_error(err, MOE_DEV_ERR_BAD_ROWS);
        *n_tiles = min(run, max_tiles);
        *ticket = 0;  // the persistent MMQ kernels take work items from here
        s_full = 0;  // reused as the full-tile cursor
    }
    __syncthreads();
    // pass 2: write the entries (order among equal sizes is irrelevant)
    for (int p = threadIdx.x; p < na; p += blockDim.x) {
        int e = active[p];
        if ((unsigned)e >= (unsigned)E) continue;
        int lo = max(0, min(offsets[e], R));
        int hi = max(lo, min(offsets[e + 1], R));
        int cnt = hi - lo;
        int nf = cnt / BM;
        int base = atomicAdd(&s_full, nf);
        for (int i = 0; i < nf && base + i < max_tiles; ++i)
            tiles[base + i] = make_int4(p, lo + i * BM, BM, e);
        if (cnt % BM) {
            int at = atomicAdd(&part_hist[cnt % BM], 1);
            if (at < max_tiles) tiles[at] = make_int4(p, lo + nf * BM, cnt % BM, e);
        }
    }
}

int launch_mmq_tiles(const int32_t* active, const int32_t* n_active, const int32_t* offsets,
                     int E, int R, int BM, uint8_t* ws, const WsLayout& W, cudaStream_t stream) {
    uint32_t* err = (uint32_t*)(ws + W.err);
    int32_t* n_tiles = (int32_t*)(ws + W.counters) + MMQ_COUNTER_NTILES;
    int32_t* ticket = (int32_t*)(ws + W.counters) + MMQ_COUNTER_TICKET;
    int4* tiles = (int4*)(ws + W.tiles);
    mmq_tiles_kernel<<<1, 1024, 0, stream>>>(active, n_active, offsets, E, R, BM, tiles, n_tiles,
                                             ticket, W.max_tiles, err);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
