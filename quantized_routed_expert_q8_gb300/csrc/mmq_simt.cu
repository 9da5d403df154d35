// Stages 4 and 6, portable form: grouped MMQ with CUDA-core integer dot
// products (dp4a).  Used for shapes the tensor-core kernel does not take and as
// its cross-check.
//
// For the expert at active position p and each of its rows r:
//   acc = sum over 32-blocks b ascending of
//         fma(fp32(dW[j,b]) * fp32(dx[r,b]), I_b, acc)  (+ fma(mW[j,b], sx[r,b], acc) for Q4_1)
// (Q2_0: the block dot uses the weight integers c - 2.  Q2_K: the integers
// sc * c with the sub-block scales of the block's two halves, dW the
// super-block d, then fma(-(dmin * mn_lo), s_lo, acc) and fma(-(dmin * mn_hi),
// s_hi, acc) from the D2S6 activation entries)
// with I_b the exact int32 block dot -- the same fp32 operation sequence as the
// scalar definition, so the result does not depend on the tiling.
// Tile: 64 rows x 64 output columns per block of 256 threads, one 32-block of
// the reduction per step; gate/up tiles carry both matrices and apply SiLU(g)*u.
#include "mmq.cuh"

namespace moe {

constexpr int SB_M = 64;  // rows (tokens) per tile
constexpr int SB_N = 64;  // output columns per tile

// 4 Q4_1 bytes (8 nibbles) -> two words of int8 in element order
__device__ __forceinline__ void unpack_q4_pair(uint32_t bytes2, uint32_t& w) {
    uint32_t b0 = bytes2 & 0xff, b1 = (bytes2 >> 8) & 0xff;
    w = (b0 & 0xf) | ((b0 >> 4) << 8) | ((b1 & 0xf) << 16) | ((b1 >> 4) << 24);
}

// one byte of 2-bit codes (4 consecutive elements) -> 4 bytes c in 0..3
__device__ __forceinline__ uint32_t spread_q2_byte(uint32_t x) {
    return (x & 0x3u) | ((x & 0xCu) << 6) | ((x & 0x30u) << 12) | ((x & 0xC0u) << 18);
}

// one Q2_0 byte -> 4 int8 c - 2
__device__ __forceinline__ int unpack_q2_byte(uint32_t x) {
    return (int)__vsub4(spread_q2_byte(x), 0x02020202u);
}

// mw: [2][SB_N] -- the m term of each row (Q4_1: m; Q2_K: -(dmin * mn) of the
// block's two halves)
template <int WT>
__device__ __forceinline__ void load_w_tile(const uint8_t* __restrict__ qplane,
                                            const __half* __restrict__ dplane,
                                            const __half* __restrict__ mplane,
                                            const uint8_t* __restrict__ splane, int k, int j0,
                                            int nrows, int b, int (*ws)[9], float* dw, float* mw,
                                            int tid) {
    // 64 weight rows x 32 values of block b
    if (tid < SB_N) {
        int j = j0 + tid;
        if (j < nrows && WT == MOE_W_Q2_K) {
            // codes times the sub-block scale: at most 3 * 15 per byte, so the
            // 32-bit multiply of four spread bytes carries nothing across bytes
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(qplane + (size_t)j * (k / 4) + b * 8));
            const uint32_t in[2] = {v.x, v.y};
            const int u = b / (QKK / QK);
            const float dmin = __half2float(mplane[(size_t)u * nrows + j]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t scmn = splane[(size_t)(2 * b + h) * nrows + j];
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    ws[tid][4 * h + t] = (int)(spread_q2_byte((in[h] >> (8 * t)) & 0xffu) * (scmn & 0xFu));
                mw[h * SB_N + tid] = -__fmul_rn(dmin, (float)(scmn >> 4));
            }
            dw[tid] = __half2float(dplane[(size_t)u * nrows + j]);
        } else if (j < nrows) {
            if (WT == MOE_W_Q8_0) {
                const uint4* p = reinterpret_cast<const uint4*>(qplane + (size_t)j * k + b * QK);
                uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
                ws[tid][0] = v0.x; ws[tid][1] = v0.y; ws[tid][2] = v0.z; ws[tid][3] = v0.w;
                ws[tid][4] = v1.x; ws[tid][5] = v1.y; ws[tid][6] = v1.z; ws[tid][7] = v1.w;
            } else if (WT == MOE_W_Q2_0) {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>(qplane + (size_t)j * (k / 4) + b * 8));
                const uint32_t in[2] = {v.x, v.y};
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int t = 0; t < 4; ++t) ws[tid][4 * h + t] = unpack_q2_byte((in[h] >> (8 * t)) & 0xffu);
            } else {
                const uint4* p = reinterpret_cast<const uint4*>(qplane + (size_t)j * (k / 2) + b * 16);
                uint4 v = __ldg(p);
                uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t w0, w1;
                    unpack_q4_pair(in[h] & 0xffff, w0);
                    unpack_q4_pair(in[h] >> 16, w1);
                    ws[tid][2 * h] = (int)w0;
                    ws[tid][2 * h + 1] = (int)w1;
                }
            }
            dw[tid] = __half2float(dplane[(size_t)b * nrows + j]);  // block-major scales
            mw[tid] = WT == MOE_W_Q4_1 ? __half2float(mplane[(size_t)b * nrows + j]) : 0.0f;
        } else {
#pragma unroll
            for (int w = 0; w < 8; ++w) ws[tid][w] = 0;
            dw[tid] = 0.0f;
            mw[tid] = 0.0f;
            mw[SB_N + tid] = 0.0f;
        }
    }
}

template <int WT, bool GATEUP>
__global__ void __launch_bounds__(256) mmq_simt_kernel(
    const uint8_t* __restrict__ group_base, size_t slot_stride, size_t off_a, size_t off_b,
    MatLayout L, const int4* __restrict__ tiles, const int32_t* __restrict__ n_tiles,
    const int8_t* __restrict__ xq, const __half2* __restrict__ xds, int k, int n,
    float* __restrict__ out) {
    __shared__ int xs[SB_M][9];
    __shared__ int wa[SB_N][9];
    __shared__ int wb[GATEUP ? SB_N : 1][9];
    // sx: s (Q4_1) or s_lo, s_hi (Q2_K) per row; ma / mb: the m terms per column
    __shared__ float dx[SB_M], sx[2][SB_M], da[SB_N], ma[2][SB_N], db[SB_N], mb[2][SB_N];
    const int tile = blockIdx.y;
    if (tile >= *n_tiles) return;
    const int4 tl = tiles[tile];
    const int p = tl.x, r0 = tl.y, rows = tl.z;
    const int j0 = blockIdx.x * SB_N;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const uint8_t* rec = group_base + (size_t)p * slot_stride;
    const uint8_t* A = rec + off_a;
    const uint8_t* B = rec + off_b;
    const __half* Ad = reinterpret_cast<const __half*>(A + L.d);
    const __half* Am = reinterpret_cast<const __half*>(A + L.m);
    const __half* Bd = reinterpret_cast<const __half*>(B + L.d);
    const __half* Bm = reinterpret_cast<const __half*>(B + L.m);
    const uint8_t* As = A + L.s;
    const uint8_t* Bs = B + L.s;
    float acc_a[4][4], acc_b[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc_a[i][jj] = acc_b[i][jj] = 0.0f;
    const int nb = k / QK;
    for (int b = 0; b < nb; ++b) {
        // activations: 64 rows x 32 bytes (threads 0..127), scales (128..191)
        if (tid < 128) {
            int row = tid >> 1, half = tid & 1;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (row < rows)
                v = __ldg(reinterpret_cast<const uint4*>(xq + (size_t)(r0 + row) * k + b * QK) + half);
            xs[row][half * 4 + 0] = v.x;
            xs[row][half * 4 + 1] = v.y;
            xs[row][half * 4 + 2] = v.z;
            xs[row][half * 4 + 3] = v.w;
        } else if (tid < 192) {
            int row = tid - 128;
            float2 f = make_float2(0.f, 0.f), g = make_float2(0.f, 0.f);
            if (row < rows) {
                if (WT == MOE_W_Q2_K) {  // D2S6: (d, s, s_lo, s_hi)
                    const size_t e = ((size_t)(r0 + row) * nb + b) * 2;
                    f = __half22float2(xds[e]);
                    g = __half22float2(xds[e + 1]);
                } else {
                    f = __half22float2(xds[(size_t)(r0 + row) * nb + b]);
                }
            }
            dx[row] = f.x;
            sx[0][row] = WT == MOE_W_Q2_K ? g.x : f.y;
            sx[1][row] = g.y;
        }
        if (tid >= 192) {
            load_w_tile<WT>(A, Ad, Am, As, k, j0, n, b, wa, da, &ma[0][0], tid - 192);
        }
        if (GATEUP && tid < 64) {
            load_w_tile<WT>(B, Bd, Bm, Bs, k, j0, n, b, wb, db, &mb[0][0], tid);
        }
        __syncthreads();
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int col = tx + 16 * jj;
            int wva[8], wvb[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                wva[w] = wa[col][w];
                wvb[w] = GATEUP ? wb[col][w] : 0;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = ty + 16 * i;
                int Ia = 0, Ib = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    int xv = xs[row][w];
                    Ia = __dp4a(xv, wva[w], Ia);
                    if (GATEUP) Ib = __dp4a(xv, wvb[w], Ib);
                }
                acc_a[i][jj] = __fmaf_rn(__fmul_rn(da[col], dx[row]), (float)Ia, acc_a[i][jj]);
                if (WT == MOE_W_Q4_1 || WT == MOE_W_Q2_K)
                    acc_a[i][jj] = __fmaf_rn(ma[0][col], sx[0][row], acc_a[i][jj]);
                if (WT == MOE_W_Q2_K) acc_a[i][jj] = __fmaf_rn(ma[1][col], sx[1][row], acc_a[i][jj]);
                if (GATEUP) {
                    acc_b[i][jj] = __fmaf_rn(__fmul_rn(db[col], dx[row]), (float)Ib, acc_b[i][jj]);
                    if (WT == MOE_W_Q4_1 || WT == MOE_W_Q2_K)
                        acc_b[i][jj] = __fmaf_rn(mb[0][col], sx[0][row], acc_b[i][jj]);
                    if (WT == MOE_W_Q2_K)
                        acc_b[i][jj] = __fmaf_rn(mb[1][col], sx[1][row], acc_b[i][jj]);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = ty + 16 * i;
        if (row >= rows) continue;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int col = j0 + tx + 16 * jj;
            if (col >= n) continue;
            float v = GATEUP ? silu_mul(acc_a[i][jj], acc_b[i][jj]) : acc_a[i][jj];
            out[(size_t)(r0 + row) * n + col] = v;
        }
    }
}

// gate/up: out = h [R][f]; down: out = y [R][d]
int launch_mmq_simt(int wtype, bool gateup, const uint8_t* group_base, size_t slot_stride,
                    const int32_t* active, const int32_t* n_active, const int32_t* offsets, int E,
                    const int8_t* xq, const uint16_t* xds, int R, int d, int f, float* out,
                    uint8_t* ws, const WsLayout& W, cudaStream_t stream) {
    int rc = launch_mmq_tiles(active, n_active, offsets, E, R, SB_M, ws, W, stream);
    if (rc != MOE_OK) return rc;
    RecLayout RL = rec_layout(wtype, d, f);
    int k = gateup ? d : f;
    int n = gateup ? f : d;
    MatLayout L = gateup ? RL.gu : RL.dn;
    int max_tiles = R / SB_M + E + 1;
    if (max_tiles > W.max_tiles) max_tiles = W.max_tiles;
    if (max_tiles > 65535) return MOE_ERR_UNSUPPORTED;
    dim3 grid((n + SB_N - 1) / SB_N, max_tiles);
    const int4* tiles = (const int4*)(ws + W.tiles);
    const int32_t* n_tiles = (const int32_t*)(ws + W.counters) + MMQ_COUNTER_NTILES;
    const __half2* ds2 = reinterpret_cast<const __half2*>(xds);
    size_t oa = gateup ? RL.gate : RL.down, ob = gateup ? RL.up : RL.down;
#define MOE_SIMT_LAUNCH(WT, GU)                                                                    \
    mmq_simt_kernel<WT, GU><<<grid, 256, 0, stream>>>(group_base, slot_stride, oa, ob, L, tiles, \
                                                      n_tiles, xq, ds2, k, n, out)
    if (wtype == MOE_W_Q8_0) {
        if (gateup) MOE_SIMT_LAUNCH(MOE_W_Q8_0, true);
        else MOE_SIMT_LAUNCH(MOE_W_Q8_0, false);
    } else if (wtype == MOE_W_Q2_0) {
        if (gateup) MOE_SIMT_LAUNCH(MOE_W_Q2_0, true);
        else MOE_SIMT_LAUNCH(MOE_W_Q2_0, false);
    } else if (wtype == MOE_W_Q2_K) {
        if (gateup) MOE_SIMT_LAUNCH(MOE_W_Q2_K, true);
        else MOE_SIMT_LAUNCH(MOE_W_Q2_K, false);
    } else {
        if (gateup) MOE_SIMT_LAUNCH(MOE_W_Q4_1, true);
        else MOE_SIMT_LAUNCH(MOE_W_Q4_1, false);
    }
#undef MOE_SIMT_LAUNCH
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
