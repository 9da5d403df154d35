// Shared definitions of the CUDA library: record layout, workspace layout,
// device error word.  Used only by the library's own .cu files.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_q8.h"

namespace moe {

constexpr int QK = 32;    // block width of q8_1, Q8_0, Q4_1 and Q2_0
constexpr int QKK = 256;  // Q2_K super-block width (sixteen 16-weight sub-blocks)

// quant bytes per row of a weight matrix with reduction length k
__host__ __device__ inline size_t quant_row_bytes(int wtype, int k) {
    return (size_t)k / (wtype == MOE_W_Q4_1 ? 2 : (wtype == MOE_W_Q2_0 || wtype == MOE_W_Q2_K) ? 4 : 1);
}

// binary16 entries per 32-block of a q8_1 ds row: (d, s), or (d, s, s_lo, s_hi)
// in the D2S6 layout that Q2_K weights read
__host__ __device__ inline int ds_halves(int wtype) { return wtype == MOE_W_Q2_K ? 4 : 2; }

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// One weight matrix of an expert record: quant plane [rows][K] (Q4_1: two
// values per byte), fp16 d plane [K/32][rows] (block-major, so one block's
// scales for consecutive rows are contiguous), fp16 m plane [K/32][rows] for
// Q4_1 -- each plane 128-byte aligned.  Q2_K: fp16 d and dmin (the m plane)
// [K/256][rows], then the sub-block bytes sc | mn << 4 [K/16][rows] (plane s).
struct MatLayout {
    size_t q, d, m, s, bytes;
};

__host__ __device__ inline MatLayout mat_layout(int wtype, int rows, int k) {
    MatLayout L;
    size_t qb = (size_t)rows * quant_row_bytes(wtype, k);
    size_t sb = (size_t)rows * (size_t)(k / (wtype == MOE_W_Q2_K ? QKK : QK)) * 2;
    const bool has_m = wtype == MOE_W_Q4_1 || wtype == MOE_W_Q2_K;
    L.q = 0;
    L.d = align_up(qb, 128);
    L.m = L.d + align_up(sb, 128);
    L.s = L.m + (has_m ? align_up(sb, 128) : 0);
    L.bytes = L.s + (wtype == MOE_W_Q2_K ? align_up((size_t)rows * (size_t)(k / 16), 128) : 0);
    return L;
}

// gate [f x d], up [f x d], down [d x f]
struct RecLayout {
    size_t gate, up, down, bytes;
    MatLayout gu, dn;
};

__host__ __device__ inline RecLayout rec_layout(int wtype, int d, int f) {
    RecLayout R;
    R.gu = mat_layout(wtype, f, d);
    R.dn = mat_layout(wtype, d, f);
    R.gate = 0;
    R.up = R.gu.bytes;
    R.down = 2 * R.gu.bytes;
    R.bytes = 2 * R.gu.bytes + R.dn.bytes;
    return R;
}

// Workspace: [header 256 B: error word, counters][slot-map chunk counts]
//            [tile list][spare 256 B][combine arrival counters]
// The slot-map and MMQ calls use everything before the arrival counters
// (`core` bytes); the down projection with the combine uses them too.
constexpr int SLOT_CHUNK = 1024;  // (t,k) entries per slot-map chunk
constexpr int MAX_E = 8192;

struct WsLayout {
    size_t err;           // uint32 error word
    size_t counters;      // uint32 counters[48]
    size_t chunk_counts;  // int32 [n_chunks][E]
    size_t tiles;         // int4 [max_tiles]
    size_t arrivals;      // int32 [T][ceil(d/256)]
    size_t core;          // bytes up to the arrival counters
    size_t total;
    int n_chunks;
    int max_tiles;
};

inline WsLayout ws_layout(int T, int K, int E, int d, int f) {
    (void)f;
    WsLayout W;
    long long TK = (long long)T * K;
    W.err = 0;
    W.counters = 64;
    W.chunk_counts = 256;
    W.n_chunks = (int)((TK + SLOT_CHUNK - 1) / SLOT_CHUNK);
    size_t cc = align_up((size_t)W.n_chunks * (size_t)E * 4, 256);
    W.tiles = W.chunk_counts + cc;
    // smallest row tile of any MMQ schedule is 16 rows; one partial tile per expert
    W.max_tiles = (int)(TK / 16 + E + 16);
    W.core = W.tiles + align_up((size_t)W.max_tiles * 16, 256) + 256;
    W.arrivals = W.core;
    W.total = W.core + align_up((size_t)(T > 0 ? T : 0) * (size_t)((d + 255) / 256) * 4, 256);
    return W;
}

// Number of kernels this library has launched (diagnostics for benchmarks).
void count_launches(int n);

__device__ inline void set_error(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

}  // namespace moe
