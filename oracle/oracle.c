/*
 * Reference oracle for the quantized routed-expert (q8_1 MMQ) MoE prefill layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded CPU
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it.  It shares no code, no
 * header and no table with the CUDA library (quantized_routed_expert_q8_gb300/csrc),
 * and neither side includes the other.
 *
 * Build: plain C11, no fast-math, no FP contraction (-ffp-contract=off), so every
 * fp32 operation below rounds exactly where it is written.
 *
 * Sources (pull-request pages of the "Strata" engine):
 *   [#1368] "prefill: quantize each token's MoE input once and scatter it to its
 *           k rows (the same bytes)" -- intro paragraph (the inverse map
 *           slot[t*K+k] of src), and section "Identity" (scatter == per-row
 *           gather quantization, byte for byte; one all-zero token).
 *   [#439]  "prefill: a group's expert gathers in one launch" -- section "What"
 *           (one launch copies up to 16 experts, blockIdx.y = expert; same bytes
 *           to the same places; unaligned / odd-size fallback; groups may start
 *           mid-group).
 *   [#372]  "Prompt path: an MMQ group's experts gathered in one launch ..." --
 *           "What changes" (gather_native_group copies a group's 16 experts).
 *   [#1282] "prefill: STRATA_PREFILL_CPU_SHARE=auto ..." -- "What it does"
 *           (the combine weights every row of Dm by the token's top-k weight).
 * The pages leave the numeric formats open; this oracle uses the layer's stated
 * workload definition:
 *   q8_1 activations: 32-wide blocks, d = amax/127 stored as fp16,
 *                     q = round-half-away-from-zero(x/d), s = d * sum(q) as fp16.
 *   Q8_0 weights:     32-wide blocks, int8 q, fp16 d, w = d*q.
 *                     (scale planes are block-major: the d of row j, block b
 *                     is entry b*rows + j)
 *   Q4_1 weights:     32-wide blocks, 4-bit unsigned q (two per byte: byte j holds
 *                     element 2j in its low nibble, 2j+1 in its high nibble),
 *                     fp16 d and fp16 m, w = d*q + m; the MMQ uses s for the m term.
 *   Q2_0 weights:     named by "#1368 ..." (section "Identity": the D4 activation
 *                     layout serves Q2_0, Q8_0 and IQ2_XS) but not defined there;
 *                     this library's definition: 32-wide blocks, 2-bit codes c
 *                     (four per byte: element 4j+i of a block in bits 2i..2i+1 of
 *                     byte j), fp16 d, w = d*(c - 2), so the block dot uses the
 *                     integers c - 2 in {-2, -1, 0, 1} and no m term.
 *   Q2_K weights:     named by "#1368 ..." (section "Identity": the D2S6
 *                     activation layout serves Q2_K) but not defined there; this
 *                     library's definition: 256-weight super-blocks, each of
 *                     sixteen 16-weight sub-blocks; 2-bit codes c packed as for
 *                     Q2_0; per super-block fp16 d and fp16 dmin; per sub-block
 *                     one byte holding a 4-bit scale sc (low nibble) and a 4-bit
 *                     min mn (high nibble); w = d*sc*c - dmin*mn.
 *   D2S6 layout:      the pages name it for Q2_K without defining it.  This
 *                     library's reading: the same q8_1 quants and d as above,
 *                     with four fp16 per 32-block, (d, s, s_lo, s_hi), where
 *                     s_lo = d * sum(q[0..15]) and s_hi = d * sum(q[16..31]) (fp32
 *                     d, one fp32 product, rounded to fp16): the Q2_K min term
 *                     needs the activation sum of every 16-weight sub-block.
 *                     The other weight types use (d, s) pairs.
 *   Gate/up product:  h = SiLU(g) * u with SiLU(g) = g / (1 + exp(-g)).
 *
 * Parity pins for every function are in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32   /* block width of q8_1, Q8_0, Q4_1 and Q2_0 */
#define QKK 256 /* Q2_K super-block width */

enum { ORACLE_W_Q8_0 = 0, ORACLE_W_Q4_1 = 1, ORACLE_W_Q2_0 = 2, ORACLE_W_Q2_K = 3 };
enum { ORACLE_LAYOUT_DS = 0, ORACLE_LAYOUT_D2S6 = 1 };

/* quant bytes per row of a matrix with reduction length k */
static size_t quant_row_bytes(int wtype, int k) {
    return (size_t)k / (wtype == ORACLE_W_Q4_1 ? 2u
                        : (wtype == ORACLE_W_Q2_0 || wtype == ORACLE_W_Q2_K) ? 4u : 1u);
}

/* fp16 entries per 32-block in an activation ds row: (d, s) or (d, s, s_lo, s_hi) */
static int ds_per_block(int layout) { return layout == ORACLE_LAYOUT_D2S6 ? 4 : 2; }

/* the activation layout the MMQ of a weight type reads */
static int layout_of(int wtype) {
    return wtype == ORACLE_W_Q2_K ? ORACLE_LAYOUT_D2S6 : ORACLE_LAYOUT_DS;
}

/* ------------------------------------------------------------------------- */
/* IEEE 754 binary16 conversion, written from the format's definition:        */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits, subnormals below  */
/* 2^-14, round to nearest with ties to even, overflow to infinity.           */
/* ------------------------------------------------------------------------- */
uint16_t oracle_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t exp = (x >> 23) & 0xFFu;
    uint32_t man = x & 0x7FFFFFu;
    if (exp == 0xFFu) { /* inf or NaN */
        return (uint16_t)(sign | 0x7C00u | (man ? 0x200u | (man >> 13) : 0u));
    }
    if (exp == 0u) return (uint16_t)sign; /* fp32 zero or subnormal: far below 2^-25 */
    int e = (int)exp - 127 + 15;          /* biased binary16 exponent */
    if (e >= 31) return (uint16_t)(sign | 0x7C00u);
    if (e >= 1) {
        uint32_t h = ((uint32_t)e << 10) | (man >> 13);
        uint32_t rem = man & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u; /* carry may reach inf */
        return (uint16_t)(sign | h);
    }
    /* binary16 subnormal: value = m * 2^(exp-150), unit 2^-24 -> m * 2^(exp-126) */
    uint32_t m = man | 0x800000u;
    int shift = 126 - (int)exp; /* >= 14 here */
    if (shift >= 32) return (uint16_t)sign;
    uint32_t h = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
}

float oracle_f16_to_f32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t exp = ((uint32_t)h >> 10) & 0x1Fu;
    uint32_t man = (uint32_t)h & 0x3FFu;
    uint32_t x;
    if (exp == 0x1Fu) {
        x = sign | 0x7F800000u | (man << 13);
    } else if (exp == 0u) {
        if (man == 0u) {
            x = sign;
        } else { /* subnormal: man * 2^-24, exact in fp32 */
            float v = (float)man * 5.9604644775390625e-08f;
            memcpy(&x, &v, sizeof x);
            x |= sign;
        }
    } else {
        x = sign | ((exp - 15u + 127u) << 23) | (man << 13);
    }
    float f;
    memcpy(&f, &x, sizeof f);
    return f;
}

void oracle_f32_to_f16_array(const float* in, size_t n, uint16_t* out) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}

void oracle_f16_to_f32_array(const uint16_t* in, size_t n, float* out) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(in[i]);
}

/* ------------------------------------------------------------------------- */
/* Expert record layout (this library's own format; the pages do not define  */
/* one).  A record holds three matrices in the order gate [f x d], up [f x d], */
/* down [d x f]; each matrix is the plane of quants (row-major, reduction dim */
/* innermost), then the fp16 d plane [K/32][rows] (block-major), then for     */
/* Q4_1 the fp16 m plane [K/32][rows]; every plane starts on a 128-byte       */
/* boundary.  Q2_K: quants, then fp16 d [K/256][rows], fp16 dmin             */
/* [K/256][rows] and the sub-block byte plane (sc | mn << 4) [K/16][rows].    */
/* ------------------------------------------------------------------------- */
static size_t align128(size_t x) { return (x + 127u) & ~(size_t)127u; }

typedef struct {
    size_t q, d, m, s, bytes; /* plane offsets inside the matrix, matrix size */
} oracle_matrix_layout;

static oracle_matrix_layout matrix_layout(int wtype, int rows, int k) {
    oracle_matrix_layout L;
    size_t qbytes = (size_t)rows * quant_row_bytes(wtype, k);
    size_t sbytes = (size_t)rows * (size_t)(k / (wtype == ORACLE_W_Q2_K ? QKK : QK)) * 2u;
    int has_m = wtype == ORACLE_W_Q4_1 || wtype == ORACLE_W_Q2_K;
    L.q = 0;
    L.d = align128(qbytes);
    L.m = L.d + align128(sbytes);
    L.s = L.m + (has_m ? align128(sbytes) : 0u);
    L.bytes = L.s + (wtype == ORACLE_W_Q2_K ? align128((size_t)rows * (size_t)(k / 16)) : 0u);
    return L;
}

size_t oracle_expert_record_bytes(int wtype, int d, int f) {
    return 2u * matrix_layout(wtype, f, d).bytes + matrix_layout(wtype, d, f).bytes;
}

/* Offsets of gate, up and down inside a record. */
void oracle_record_offsets(int wtype, int d, int f, size_t* gate, size_t* up, size_t* down) {
    size_t g = matrix_layout(wtype, f, d).bytes;
    *gate = 0;
    *up = g;
    *down = 2u * g;
}

/* ------------------------------------------------------------------------- */
/* Stage a1: routing map.  [#1368] intro: token t's k-th row is slot[t*K+k],  */
/* and slot is the inverse of src (src[row] = the token the row reads).       */
/* Rows are expert-sorted; within an expert they follow ascending t*K+k, the  */
/* order a stable counting sort gives.  Ids outside [0,E) are dropped: their  */
/* slot is -1 and they get no row.  Returns the number of dropped ids.        */
/* active[] lists the experts with at least one row, ascending.               */
/* ------------------------------------------------------------------------- */
int oracle_build_slot_map(const int32_t* ids, int T, int K, int E, int32_t* offsets,
                          int32_t* slot, int32_t* src, int32_t* active, int32_t* n_active) {
    int dropped = 0;
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int i = 0; i < T * K; ++i) {
        int e = ids[i];
        if (e < 0 || e >= E) {
            ++dropped;
            continue;
        }
        offsets[e + 1] += 1; /* count, shifted by one for the exclusive scan */
    }
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    /* fill pointer per expert, walking (t, k) in order */
    int na = 0;
    for (int e = 0; e < E; ++e)
        if (offsets[e + 1] > offsets[e]) active[na++] = e;
    *n_active = na;
    for (int e = na; e < E; ++e) active[e] = -1;
    /* next free row of each expert, walking (t, k) in order: a stable
       counting sort, so rows within an expert follow ascending t*K+k */
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) next[e] = offsets[e];
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int i = t * K + k;
            int e = ids[i];
            if (e < 0 || e >= E) {
                slot[i] = -1;
                continue;
            }
            int row = next[e]++;
            slot[i] = row;
            src[row] = t;
        }
    }
    free(next);
    return dropped;
}

/* ------------------------------------------------------------------------- */
/* Stage a2/a5 quantizer: one 32-wide q8_1 block.                             */
/*   amax = max |v_i| (fp32); d = amax / 127 (IEEE); if d == 0 (amax == 0,    */
/*   or amax <= 63 * 2^-149 so that the quotient underflows) then q = 0,       */
/*   d = 0, s = 0; else q_i = round-half-away(v_i / d) (IEEE),                 */
/*   S = sum q_i exactly, stored d_h = fp16(d), s_h = fp16(d * S).            */
/*   Every quantizer below takes the activation layout: ORACLE_LAYOUT_DS      */
/*   ((d, s) per block) or ORACLE_LAYOUT_D2S6 ((d, s, s_lo, s_hi)).           */
/* ------------------------------------------------------------------------- */
/* The quants of one block; returns the fp32 d (0 for an all-zero block). */
static float block_quants(const float* v, int8_t* q) {
    float amax = 0.0f;
    for (int i = 0; i < QK; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    if (d == 0.0f) {  /* x / d is undefined: the block is stored as all-zero */
        for (int i = 0; i < QK; ++i) q[i] = 0;
        return 0.0f;
    }
    for (int i = 0; i < QK; ++i) {
        float r = roundf(v[i] / d);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
    return d;
}

static int sum_quants(const int8_t* q, int from, int to) {
    int sum = 0;
    for (int i = from; i < to; ++i) sum += q[i];
    return sum;
}

void oracle_quantize_block_q8_1(const float* v, int8_t* q, uint16_t* dh, uint16_t* sh) {
    float d = block_quants(v, q);
    *dh = oracle_f32_to_f16(d);
    *sh = oracle_f32_to_f16(d * (float)sum_quants(q, 0, QK));
}

/* The D2S6 reading of the block: e[0..3] = fp16 of d, d*S, d*S_lo, d*S_hi with
   S_lo, S_hi the exact sums of q over elements 0..15 and 16..31. */
void oracle_quantize_block_q8_1_d2s6(const float* v, int8_t* q, uint16_t* e) {
    float d = block_quants(v, q);
    e[0] = oracle_f32_to_f16(d);
    e[1] = oracle_f32_to_f16(d * (float)sum_quants(q, 0, QK));
    e[2] = oracle_f32_to_f16(d * (float)sum_quants(q, 0, QK / 2));
    e[3] = oracle_f32_to_f16(d * (float)sum_quants(q, QK / 2, QK));
}

/* Quantize one row of n values (n % 32 == 0) into q[n] and ds, the row's fp16
   bit patterns, ds_per_block(layout) per block. */
static void quantize_row(const float* x, int n, int8_t* q, uint16_t* ds, int layout) {
    int w = ds_per_block(layout);
    for (int b = 0; b < n / QK; ++b) {
        if (layout == ORACLE_LAYOUT_D2S6)
            oracle_quantize_block_q8_1_d2s6(x + b * QK, q + b * QK, &ds[w * b]);
        else
            oracle_quantize_block_q8_1(x + b * QK, q + b * QK, &ds[w * b], &ds[w * b + 1]);
    }
}

/* [#1368] intro: quantize each token once, write its blocks to all K of its
   rows through the inverse map.  Rows with slot -1 are skipped. */
void oracle_quantize_scatter_q8_1(const float* x, int T, int d, int K, const int32_t* slot,
                                  int8_t* q, uint16_t* ds, int layout) {
    size_t row_ds = (size_t)ds_per_block(layout) * (size_t)(d / QK);
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int r = slot[t * K + k];
            if (r < 0) continue;
            quantize_row(x + (size_t)t * d, d, q + (size_t)r * d, ds + (size_t)r * row_ds, layout);
        }
    }
}

/* [#1368] intro: the per-row gather quantizer, mmq::quantize(x, src, ...):
   row r reads and quantizes token src[r]; the same bytes as the scatter. */
void oracle_quantize_gather_q8_1(const float* x, int d, const int32_t* src, int R, int8_t* q,
                                 uint16_t* ds, int layout) {
    size_t row_ds = (size_t)ds_per_block(layout) * (size_t)(d / QK);
    for (int r = 0; r < R; ++r)
        quantize_row(x + (size_t)src[r] * d, d, q + (size_t)r * d, ds + (size_t)r * row_ds, layout);
}

/* Stage a5: the down-projection q8_1 quantization of the hidden rows
   ([#1368] intro names it as unchanged), identity row map. */
void oracle_requant_hidden_q8_1(const float* h, int R, int f, int8_t* hq, uint16_t* hds,
                                int layout) {
    size_t row_ds = (size_t)ds_per_block(layout) * (size_t)(f / QK);
    for (int r = 0; r < R; ++r)
        quantize_row(h + (size_t)r * f, f, hq + (size_t)r * f, hds + (size_t)r * row_ds, layout);
}

/* ------------------------------------------------------------------------- */
/* Stage a3: group gather.  [#439] "What": copy up to 16 experts' records     */
/* into group-buffer slots first_slot .. first_slot+n-1, the same bytes as    */
/* one copy per expert.                                                       */
/* ------------------------------------------------------------------------- */
void oracle_gather_one(const uint8_t* arena, size_t rec_bytes, size_t arena_stride, int expert,
                       uint8_t* group_buf, size_t slot_stride, int slot) {
    memcpy(group_buf + (size_t)slot * slot_stride, arena + (size_t)expert * arena_stride, rec_bytes);
}

void oracle_group_gather(const uint8_t* arena, size_t rec_bytes, size_t arena_stride,
                         const int32_t* expert_ids, int n, int first_slot, uint8_t* group_buf,
                         size_t slot_stride) {
    for (int j = 0; j < n; ++j)
        oracle_gather_one(arena, rec_bytes, arena_stride, expert_ids[j], group_buf, slot_stride,
                          first_slot + j);
}

/* ------------------------------------------------------------------------- */
/* Stages a4/a6: the MMQ dot of one weight row with one activation row.       */
/*   dot = sum over blocks b ascending of                                      */
/*         fmaf(fp32(dW[b]) * fp32(dX[b]), (float)I_b, acc)                    */
/*         and, for Q4_1, then fmaf(fp32(mW[b]), fp32(sX[b]), acc),            */
/*   with I_b the exact integer sum over the block of qW * qX.                 */
/*   Q2_K (block b lies in super-block u = b/8 and covers the sub-blocks      */
/*   2b and 2b+1): I_b = sc_2b * sum_{i<16} c_i qX_i + sc_2b+1 * sum_{i>=16}   */
/*   c_i qX_i, dW = d_u, and the min term is two more steps,                   */
/*   fmaf(-(dmin_u * mn_2b), s_lo[b], acc) then fmaf(-(dmin_u * mn_2b+1),      */
/*   s_hi[b], acc) (each product dmin * mn is exact in fp32).                  */
/* ------------------------------------------------------------------------- */
typedef struct {
    const uint8_t* q;
    const uint16_t* d;
    const uint16_t* m;
    const uint8_t* s;
    size_t q_row; /* bytes per row of the quant plane */
    int rows;     /* rows of the matrix = stride between blocks of a scale plane */
} wmat;

static wmat weight_matrix(int wtype, const uint8_t* base, int rows, int k) {
    oracle_matrix_layout L = matrix_layout(wtype, rows, k);
    wmat W;
    W.q = base + L.q;
    W.d = (const uint16_t*)(base + L.d);
    W.m = (const uint16_t*)(base + L.m);
    W.s = base + L.s;
    W.q_row = quant_row_bytes(wtype, k);
    W.rows = rows;
    return W;
}

/* 2-bit code of element i of a packed row segment (four per byte, low bits first) */
static int32_t code2(const uint8_t* p, int i) { return (p[i / 4] >> (2 * (i % 4))) & 3; }

/* Weight row j of W against one activation row (quants xq, fp16 entries xds,
   ds_per_block(layout_of(wtype)) per block), reduction length k. */
static float wdot(int wtype, wmat W, int j, const int8_t* xq, const uint16_t* xds, int k) {
    const uint8_t* wq_row = W.q + (size_t)j * W.q_row;
    const size_t rs = (size_t)W.rows; /* block-major scale planes: entry b of row j at b*rows+j */
    const int w = ds_per_block(layout_of(wtype));
    float acc = 0.0f;
    for (int b = 0; b < k / QK; ++b) {
        int32_t I = 0;
        const int8_t* xb = xq + b * QK;
        if (wtype == ORACLE_W_Q8_0) {
            const int8_t* wb = (const int8_t*)wq_row + b * QK;
            for (int i = 0; i < QK; ++i) I += (int32_t)wb[i] * (int32_t)xb[i];
        } else if (wtype == ORACLE_W_Q2_0) {
            const uint8_t* wb = wq_row + b * (QK / 4);
            for (int i = 0; i < QK; ++i) I += (code2(wb, i) - 2) * (int32_t)xb[i];
        } else if (wtype == ORACLE_W_Q2_K) {
            const uint8_t* wb = wq_row + b * (QK / 4);
            for (int h = 0; h < 2; ++h) {
                int32_t sc = W.s[(size_t)(2 * b + h) * rs + j] & 0x0F;
                int32_t part = 0;
                for (int i = 16 * h; i < 16 * h + 16; ++i) part += code2(wb, i) * (int32_t)xb[i];
                I += sc * part;
            }
        } else {
            const uint8_t* wb = wq_row + b * (QK / 2);
            for (int i = 0; i < QK / 2; ++i) {
                int32_t lo = wb[i] & 0x0F, hi = wb[i] >> 4;
                I += lo * (int32_t)xb[2 * i] + hi * (int32_t)xb[2 * i + 1];
            }
        }
        const uint16_t* e = xds + (size_t)w * b; /* this block's activation entries */
        if (wtype == ORACLE_W_Q2_K) {
            const int u = b / (QKK / QK);
            float scale = oracle_f16_to_f32(W.d[(size_t)u * rs + j]) * oracle_f16_to_f32(e[0]);
            acc = fmaf(scale, (float)I, acc);
            const float dmin = oracle_f16_to_f32(W.m[(size_t)u * rs + j]);
            for (int h = 0; h < 2; ++h) {
                int32_t mn = W.s[(size_t)(2 * b + h) * rs + j] >> 4;
                acc = fmaf(-(dmin * (float)mn), oracle_f16_to_f32(e[2 + h]), acc);
            }
            continue;
        }
        float scale = oracle_f16_to_f32(W.d[(size_t)b * rs + j]) * oracle_f16_to_f32(e[0]);
        acc = fmaf(scale, (float)I, acc);
        if (wtype == ORACLE_W_Q4_1)
            acc = fmaf(oracle_f16_to_f32(W.m[(size_t)b * rs + j]), oracle_f16_to_f32(e[1]), acc);
    }
    return acc;
}

/* SiLU(g) * u in fp32, SiLU(g) = g / (1 + exp(-g)). */
static float silu_mul(float g, float u) { return (g / (1.0f + expf(-g))) * u; }

/* Stage a4.  The expert at active position p has its record at
   group_base + p * slot_stride (the gathered group buffers, back to back) and
   rows offsets[e] .. offsets[e+1]-1 of q/ds. */
void oracle_grouped_mmq_gateup(int wtype, const uint8_t* group_base, size_t slot_stride,
                               const int32_t* active, int n_active, const int32_t* offsets,
                               const int8_t* q, const uint16_t* ds, int d, int f, float* h) {
    size_t og, ou, od;
    oracle_record_offsets(wtype, d, f, &og, &ou, &od);
    size_t row_ds = (size_t)ds_per_block(layout_of(wtype)) * (size_t)(d / QK);
    for (int p = 0; p < n_active; ++p) {
        int e = active[p];
        const uint8_t* rec = group_base + (size_t)p * slot_stride;
        wmat G = weight_matrix(wtype, rec + og, f, d);
        wmat U = weight_matrix(wtype, rec + ou, f, d);
        for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
            const int8_t* xq = q + (size_t)r * d;
            const uint16_t* xds = ds + (size_t)r * row_ds;
            for (int j = 0; j < f; ++j) {
                float g = wdot(wtype, G, j, xq, xds, d);
                float u = wdot(wtype, U, j, xq, xds, d);
                h[(size_t)r * f + j] = silu_mul(g, u);
            }
        }
    }
}

/* Stage a6: y[r, i] = MMQ dot of W_down row i with the re-quantized hidden row r. */
void oracle_grouped_mmq_down(int wtype, const uint8_t* group_base, size_t slot_stride,
                             const int32_t* active, int n_active, const int32_t* offsets,
                             const int8_t* hq, const uint16_t* hds, int d, int f, float* y) {
    size_t og, ou, od;
    oracle_record_offsets(wtype, d, f, &og, &ou, &od);
    size_t row_ds = (size_t)ds_per_block(layout_of(wtype)) * (size_t)(f / QK);
    for (int p = 0; p < n_active; ++p) {
        int e = active[p];
        const uint8_t* rec = group_base + (size_t)p * slot_stride;
        wmat D = weight_matrix(wtype, rec + od, d, f);
        for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
            const int8_t* xq = hq + (size_t)r * f;
            const uint16_t* xds = hds + (size_t)r * row_ds;
            for (int i = 0; i < d; ++i) y[(size_t)r * d + i] = wdot(wtype, D, i, xq, xds, f);
        }
    }
}

/* Stage a7: [#1282] "What it does": the combine weights each of a token's rows
   of Dm by its top-k weight and sums them: acc = 0, then for k ascending
   acc = fmaf(w[t,k], y[slot[t*K+k], i], acc).  Dropped rows (slot -1) add 0. */
void oracle_combine_topk(const float* y, const int32_t* slot, const float* w, int T, int K, int d,
                         float* out) {
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < d; ++i) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int r = slot[t * K + k];
                if (r < 0) continue;
                acc = fmaf(w[t * K + k], y[(size_t)r * d + i], acc);
            }
            out[(size_t)t * d + i] = acc;
        }
    }
}
