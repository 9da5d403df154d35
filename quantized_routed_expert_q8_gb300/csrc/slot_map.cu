// Stage 1: the inverse routing map ("#1368 prefill: quantize each token's MoE
// input once and scatter it to its k rows", intro: token t's k-th row is
// slot[t*K+k], the inverse of src).
//
// A stable counting sort in three launches:
//   hist  -- one block per chunk of SLOT_CHUNK (t,k) entries counts its ids;
//   scan  -- one block turns the per-chunk counts into each chunk's first row
//            per expert, writes offsets[] and the ascending active list;
//   rank  -- one warp per chunk walks its entries in order, 32 at a time, and
//            gives equal ids consecutive rows with __match_any_sync.
#include "common.cuh"

namespace moe {

__global__ void __launch_bounds__(256) slot_hist_kernel(const int32_t* __restrict__ ids, int TK,
                                                        int E, int32_t* __restrict__ chunk_counts,
                                                        uint32_t* err) {
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    int c = blockIdx.x;
    int lo = c * SLOT_CHUNK, hi = min(TK, lo + SLOT_CHUNK);
    bool bad = false;
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        int e = ids[i];
        if ((unsigned)e < (unsigned)E) atomicAdd(&hist[e], 1);
        else bad = true;
    }
    if (bad) set_error(err, MOE_DEV_ERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_counts[(size_t)c * E + e] = hist[e];
}

// Block-wide exclusive scan of one int per thread (blockDim == 1024).
__device__ int block_exclusive_scan(int v, int* total) {
    __shared__ int warp_sums[32];
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    int base = warp ? warp_sums[warp - 1] : 0;
    if (total) *total = warp_sums[31];
    __syncthreads();
    return base + x - v;
}

__global__ void __launch_bounds__(1024) slot_scan_kernel(int32_t* __restrict__ chunk_counts,
                                                         int n_chunks, int E,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ active,
                                                         int32_t* __restrict__ n_active) {
    extern __shared__ int32_t tot[];  // [E]
    // per expert: running prefix over chunks (column walk, coalesced across e),
    // 8 chunks' counts loaded at once so that their latencies overlap
    constexpr int CB = 8;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int c0 = 0; c0 < n_chunks; c0 += CB) {
            int v[CB];
#pragma unroll
            for (int j = 0; j < CB; ++j)
                v[j] = c0 + j < n_chunks ? chunk_counts[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < CB; ++j) {
                if (c0 + j < n_chunks) chunk_counts[(size_t)(c0 + j) * E + e] = run;
                run += v[j];
            }
        }
        tot[e] = run;
    }
    __syncthreads();
    // exclusive scan of tot over experts: each thread owns a contiguous run
    int per = (E + blockDim.x - 1) / blockDim.x;
    int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
    int sum = 0, nact = 0;
    for (int e = e0; e < e1; ++e) {
        sum += tot[e];
        nact += tot[e] > 0;
    }
    int total_rows, total_act;
    int base = block_exclusive_scan(sum, &total_rows);
    int abase = block_exclusive_scan(nact, &total_act);
    for (int e = e0; e < e1; ++e) {
        int t = tot[e];
        offsets[e] = base;
        tot[e] = base;  // becomes the expert's first row
        if (t > 0) active[abase++] = e;
        base += t;
    }
    if (threadIdx.x == 0) {
        offsets[E] = total_rows;
        *n_active = total_act;
    }
    for (int e = total_act + threadIdx.x; e < E; e += blockDim.x) active[e] = -1;
    __syncthreads();
    // chunk base rows: expert first row + rows of that expert in earlier chunks
    for (size_t i = threadIdx.x; i < (size_t)n_chunks * E; i += blockDim.x)
        chunk_counts[i] += tot[i % E];
}

__global__ void __launch_bounds__(32) slot_rank_kernel(const int32_t* __restrict__ ids, int TK,
                                                       int K, int E,
                                                       const int32_t* __restrict__ chunk_base,
                                                       int32_t* __restrict__ slot,
                                                       int32_t* __restrict__ src) {
    extern __shared__ int32_t next[];  // [E]
    int c = blockIdx.x, lane = threadIdx.x;
    for (int e = lane; e < E; e += 32) next[e] = chunk_base[(size_t)c * E + e];
    __syncwarp();
    int lo = c * SLOT_CHUNK, hi = min(TK, lo + SLOT_CHUNK);
    unsigned lt = (1u << lane) - 1u;
    // the ids of 8 steps (256 entries) are loaded at once, so that their
    // latencies overlap; the steps then run in order
    constexpr int SB = 8;
    for (int b0 = lo; b0 < hi; b0 += 32 * SB) {
      int eb[SB];
#pragma unroll
      for (int j = 0; j < SB; ++j) {
          const int i = b0 + 32 * j + lane;
          eb[j] = i < hi ? ids[i] : -1;
      }
#pragma unroll
      for (int j = 0; j < SB; ++j) {
        const int i0 = b0 + 32 * j;
        if (i0 >= hi) break;  // warp-uniform
        int i = i0 + lane;
        bool in = i < hi;
        int e = eb[j];
        bool valid = in && (unsigned)e < (unsigned)E;
        int key = valid ? e : E + lane;  // invalid entries match nobody
        unsigned peers = __match_any_sync(0xffffffffu, key);
        int row = -1;
        if (valid) row = next[e] + __popc(peers & lt);
        __syncwarp();
        if (valid && (peers & lt) == 0) next[e] += __popc(peers);  // lowest peer updates
        __syncwarp();
        if (in) {
            slot[i] = row;
            if (valid) src[row] = i / K;
        }
      }
    }
}

int launch_build_slot_map(const int32_t* ids, int T, int K, int E, int32_t* offsets, int32_t* slot,
                          int32_t* src, int32_t* active, int32_t* n_active, uint8_t* ws,
                          cudaStream_t stream) {
    WsLayout W = ws_layout(T, K, E, 0, 0);
    uint32_t* err = (uint32_t*)(ws + W.err);
    int32_t* cc = (int32_t*)(ws + W.chunk_counts);
    int TK = T * K;
    size_t smem = (size_t)E * sizeof(int32_t);
    if (W.n_chunks > 0) {
        slot_hist_kernel<<<W.n_chunks, 256, smem, stream>>>(ids, TK, E, cc, err);
    }
    slot_scan_kernel<<<1, 1024, smem, stream>>>(cc, W.n_chunks, E, offsets, active, n_active);
    if (W.n_chunks > 0) {
        slot_rank_kernel<<<W.n_chunks, 32, smem, stream>>>(ids, TK, K, E, cc, slot, src);
    }
    count_launches(W.n_chunks > 0 ? 3 : 1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
