/*
 * moe_q8.h -- C ABI of the GB300 quantized routed-expert MoE prefill library
 * (libmoe_q8.so, CUDA kernels for sm_103a).
 *
 * One call per stage of a mixture-of-experts layer's prompt (prefill) step:
 *   1. moe_build_slot_map         routing ids -> expert-sorted rows, slot/src maps
 *   2. moe_quantize_scatter_q8_1  quantize each token once, write it to its K rows
 *   3. moe_group_gather[_active]  copy up to 16 routed experts per launch
 *   4. moe_grouped_mmq_gateup     int8 x quantized-weight block dots, SiLU(g)*u
 *   5. moe_requant_hidden_q8_1    q8_1 re-quantization of the hidden rows
 *   6. moe_grouped_mmq_down       down projection
 *   7. moe_combine_topk           weighted sum of each token's K rows
 * and two fused forms (the same results, fewer passes over HBM):
 *   4+5. moe_grouped_mmq_gateup_q8_1   stage 4 writing stage 5's q8_1 rows
 *   6+7. moe_grouped_mmq_down_combine  stage 6 with stage 7 in its epilogue
 *
 * Sources (pull-request pages of the "Strata" engine):
 *   [#1368] "prefill: quantize each token's MoE input once and scatter it to its
 *           k rows (the same bytes)", intro and section "Identity".
 *   [#439]  "prefill: a group's expert gathers in one launch (bit-identical, long
 *           prompts +4%)", section "What".
 *   [#372]  "Prompt path: an MMQ group's experts gathered in one launch, after one
 *           wait, released by one event", "What changes".
 *   [#1282] "prefill: STRATA_PREFILL_CPU_SHARE=auto hands a small chunk's
 *           least-routed experts to the idle CPU pool", "What it does".
 *
 * Conventions shared by every call:
 *   - Pointers are DEVICE pointers owned by the caller unless a parameter says
 *     "host".  No call allocates, frees, synchronizes (except moe_device_error
 *     and moe_layer_forward_streamed, which say what they do) or keeps a
 *     pointer after it returns.  Every call is asynchronous on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - Misuse that the host can see (null pointer with nonzero size, a width that
 *     is not a multiple of 32, a misaligned buffer, too small a workspace, a
 *     group larger than 16) returns an error status before anything is launched.
 *   - A failed launch returns MOE_ERR_CUDA (the CUDA error is left for
 *     cudaGetLastError to report as well).
 *   - Data-dependent problems found on the device never trap: the kernels skip
 *     the offending item, stay in bounds, and set a bit in the workspace's
 *     error word, which moe_device_error reads back.
 *   - Empty inputs (T = 0, R = 0, no active expert) are valid and do nothing
 *     beyond writing the (empty) outputs' headers such as offsets.
 *
 * Formats:
 *   q8_1 activations: 32-wide blocks.  d = amax/127 (fp32, IEEE division),
 *     q = round-half-away-from-zero(x/d) (IEEE division) in int8, S = sum(q);
 *     stored: q plane int8 [rows][width], ds plane [rows][width/32][2] of
 *     binary16 bit patterns (d, s) with s = fp16(d * S).  An all-zero block is
 *     q = 0, d = 0, s = 0.
 *   Expert record (this library's layout): three matrices, gate [f x d], up
 *     [f x d], down [d x f], each stored as: quant plane (rows x K, reduction
 *     dimension innermost; Q8_0 int8; Q4_1 two 4-bit values per byte, byte j of
 *     a block holding element 2j in the low nibble and 2j+1 in the high; Q2_0
 *     four 2-bit codes per byte, byte j of a block holding element 4j+i in bits
 *     2i..2i+1), then the binary16 d plane [K/32][rows] (block-major: the scale
 *     of row j, block b is entry b*rows + j), then for Q4_1 the binary16 m plane
 *     [K/32][rows].  Every plane starts on a 128-byte boundary.  Weight value
 *     w = d*q (Q8_0), d*q + m (Q4_1) or d*(c - 2) (Q2_0, code c in 0..3).  The
 *     pages name Q2_0 ([#1368] "Identity") without defining it; this is the
 *     library's own definition.
 *   Q2_K record matrices (the pages name Q2_K with the D2S6 layout, [#1368]
 *     "Identity", without defining either; this is the library's definition):
 *     K % 256 == 0; 256-weight super-blocks of sixteen 16-weight sub-blocks;
 *     quant plane of 2-bit codes c packed as for Q2_0; then the binary16 d plane
 *     and the binary16 dmin plane, each [K/256][rows] (super-block-major); then
 *     one byte per sub-block, [K/16][rows], holding the 4-bit scale sc in the
 *     low nibble and the 4-bit min mn in the high nibble.  w = d*sc*c - dmin*mn.
 *   D2S6 q8_1 layout (what MOE_W_Q2_K's MMQ reads): the same q plane, and four
 *     binary16 per block, ds [rows][width/32][4] = (d, s, s_lo, s_hi) with
 *     s_lo = fp16(d * sum of q[0..15]) and s_hi = fp16(d * sum of q[16..31])
 *     (fp32 d, one fp32 product) -- the activation sums of the two 16-weight
 *     sub-blocks a 32-block spans, which the Q2_K min term multiplies.
 */
#ifndef MOE_Q8_H
#define MOE_Q8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1, /* null pointer, bad size or count */
    MOE_ERR_ALIGNMENT = -2,   /* a buffer or stride is not aligned as required */
    MOE_ERR_WORKSPACE = -3,   /* ws is null or smaller than moe_workspace_size */
    MOE_ERR_UNSUPPORTED = -4, /* a size outside what the kernels support */
    MOE_ERR_CUDA = -5,        /* a CUDA runtime or launch error */
    MOE_ERR_DEVICE = -6       /* moe_device_error found a device-side error bit */
} moe_status;

typedef enum { MOE_W_Q8_0 = 0, MOE_W_Q4_1 = 1, MOE_W_Q2_0 = 2, MOE_W_Q2_K = 3 } moe_wtype;

/* Device error bits, set in the workspace error word. */
#define MOE_DEV_ERR_BAD_EXPERT_ID 0x1u /* an id outside [0, E): its slot is -1 */
#define MOE_DEV_ERR_BAD_ROWS 0x2u      /* offsets or slot beyond R: rows skipped */
#define MOE_DEV_ERR_TIMEOUT 0x4u       /* a bounded wait inside a kernel gave up */
#define MOE_DEV_ERR_RANGE 0x8u         /* a q8_1 or weight block with |d*q| >= 65520: the
                                          tensor-core MMQ's binary16 operands overflow */

/* Bytes of one expert record (gate, up, down) for the given weight type. */
size_t moe_expert_record_bytes(int wtype, int d, int f);

/* Byte offsets of the gate, up and down matrices inside a record. */
void moe_expert_record_offsets(int wtype, int d, int f, size_t* gate, size_t* up, size_t* down);

/* Workspace bytes the calls that take `ws` need for T tokens, top-K, E experts,
   model width d and expert FFN width f.  The workspace must be 256-byte aligned
   and is reused by every call; its first word is the device error word, which
   must be zero before the first call (moe_workspace_init). */
size_t moe_workspace_size(int T, int K, int E, int d, int f);

/* Zero the workspace header (error word and counters), async on stream. */
int moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 1 -- inverse routing map.  [#1368] intro: token t's k-th row is
 * slot[t*K+k], the inverse of src (src[row] = token of that row).
 *   ids      int32 [T*K], ids[t*K+k] = token t's k-th expert.
 *   offsets  int32 [E+1] out: exclusive prefix sum of per-expert row counts;
 *            expert e owns rows offsets[e] .. offsets[e+1]-1; offsets[E] = R.
 *   slot     int32 [T*K] out: row of (t, k); within an expert rows follow
 *            ascending t*K+k (a stable counting sort).  -1 for a dropped id.
 *   src      int32 [T*K] out: src[row] = t for rows < R (entries >= R untouched).
 *   active   int32 [E] out: experts with at least one row, ascending, then -1.
 *   n_active int32 [1] out.
 * Ids outside [0, E) are dropped and flag MOE_DEV_ERR_BAD_EXPERT_ID.
 * Limits: 1 <= E <= 8192, T*K < 2^31.
 */
int moe_build_slot_map(const int32_t* ids, int T, int K, int E, int32_t* offsets, int32_t* slot,
                       int32_t* src, int32_t* active, int32_t* n_active, void* ws,
                       size_t ws_bytes, void* stream);

/*
 * Stage 2 -- [#1368] intro: quantize each token's row of x once to q8_1 and
 * write the blocks to all K of its rows slot[t*K+k] (the same bytes as the
 * per-row gather quantizer).
 *   x    float [T][d], 16-byte aligned.    slot int32 [T*K].
 *   q    int8 [R][d] out, 16-byte aligned.  ds uint16 [R][d/32][2] out, 4-byte aligned.
 * Rows with slot outside [0, R) are skipped.  d % 32 == 0.  A block whose
 * d = amax/127 is zero in fp32 (amax == 0, or amax <= 63 * 2^-149) is stored
 * as all-zero: x/d is undefined there.
 */
int moe_quantize_scatter_q8_1(const float* x, int T, int d, int K, const int32_t* slot, int R,
                              int8_t* q, uint16_t* ds, void* stream);

/*
 * Stage 2, gather form -- the per-row quantizer the scatter replaces
 * ([#1368] intro, mmq::quantize(x, src, ...)): row r quantizes token src[r].
 * Same layouts and alignment as moe_quantize_scatter_q8_1; src values outside
 * [0, T) leave the row unwritten.
 */
int moe_quantize_gather_q8_1(const float* x, int T, int d, const int32_t* src, int R, int8_t* q,
                             uint16_t* ds, void* stream);

/*
 * Stage 2 (scatter and gather forms) and stage 5 in the D2S6 layout, the q8_1
 * rows that MOE_W_Q2_K's MMQ reads ([#1368] "Identity": the scatter writes
 * the same bytes as the gather in every layout, D2S6 included).  Arguments,
 * row maps and alignment as moe_quantize_scatter_q8_1,
 * moe_quantize_gather_q8_1 and moe_requant_hidden_q8_1, except that ds / hds
 * are uint16 [rows][width/32][4] of (d, s, s_lo, s_hi), 8-byte aligned.  q and
 * (d, s) are byte-identical to the (d, s) layout's.
 */
int moe_quantize_scatter_q8_1_d2s6(const float* x, int T, int d, int K, const int32_t* slot,
                                   int R, int8_t* q, uint16_t* ds, void* stream);
int moe_quantize_gather_q8_1_d2s6(const float* x, int T, int d, const int32_t* src, int R,
                                  int8_t* q, uint16_t* ds, void* stream);
int moe_requant_hidden_q8_1_d2s6(const float* h, int R, int f, int8_t* hq, uint16_t* hds,
                                 void* stream);

/*
 * Stage 3 -- [#439] "What" / [#372] "What changes": one launch copies up to 16
 * experts' records into the group buffer, blockIdx.y = expert; expert j of the
 * call lands in slot first_slot + j.  The same bytes as one copy per expert.
 *   arena        device: expert e's record at arena + e*arena_stride.
 *   expert_ids   HOST int32 [n], 1 <= n <= 16, first_slot + n <= 16.
 *   group_buf    device: slot s at group_buf + s*slot_stride.
 * 16-byte vector copies when arena, group_buf, rec_bytes and both strides are
 * 16-byte aligned; otherwise a byte copy with the same result.  Source and
 * destination must not overlap.
 */
int moe_group_gather(const uint8_t* arena, size_t rec_bytes, size_t arena_stride,
                     const int32_t* expert_ids, int n, int first_slot, uint8_t* group_buf,
                     size_t slot_stride, void* stream);

/*
 * Stage 3 for a whole layer without a host round trip: the groups of 16 active
 * experts (ascending id, as listed by moe_build_slot_map) gathered back to
 * back; the expert at active position p lands at group_base + p*slot_stride.
 * One launch covers every group: a persistent grid walks the (routed expert,
 * 128 KB part of its record) units up to the device-side count, so no block
 * is spent on an expert that is not routed.  The same bytes as the per-group
 * calls.  active and n_active are device pointers; max_active bounds n_active
 * (normally E).
 */
int moe_group_gather_active(const uint8_t* arena, size_t rec_bytes, size_t arena_stride,
                            const int32_t* active, const int32_t* n_active, int max_active,
                            uint8_t* group_base, size_t slot_stride, void* stream);

/*
 * Stage 4 -- grouped quantized matmul, gate and up, then h = SiLU(g) * u.
 * For the expert at active position p (record at group_base + p*slot_stride,
 * expert id e = active[p]) and each of its rows r in [offsets[e], offsets[e+1]):
 *   g[r,j] = sum over blocks b ascending of  dWg[j,b]*dx[r,b]*I_b (+ mWg[j,b]*sx[r,b]
 *            for Q4_1), accumulated in fp32, I_b the exact integer block dot;
 *   u likewise with W_up;  h[r,j] = (g / (1 + exp(-g))) * u.
 *   Q2_K: block b of super-block u = b/8 spans the sub-blocks 2b and 2b+1;
 *   I_b = sc_2b * (sum of c*q over its first 16) + sc_2b+1 * (over its last 16),
 *   the scale is d_u*dx[r,b], and the min term is two more fp32 steps,
 *   fma(-(dmin_u*mn_2b), s_lo[r,b], acc) then fma(-(dmin_u*mn_2b+1), s_hi[r,b], acc).
 *   q int8 [R][d], ds uint16 [R][d/32][2] (stage 2 output; [R][d/32][4] in the
 *   D2S6 layout for MOE_W_Q2_K); h float [R][f] out.
 * group_base and slot_stride must be 128-byte aligned, q, ds and h 16-byte
 * aligned, d % 32 == 0, f % 32 == 0 (Q2_K: d % 256 == 0, f % 256 == 0).  Shapes
 * with d % 256 == 0 and f % 128 == 0 run on the tensor cores; others on a
 * CUDA-core kernel with the same result.  Rows past R are skipped
 * (MOE_DEV_ERR_BAD_ROWS).
 */
int moe_grouped_mmq_gateup(int wtype, const uint8_t* group_base, size_t slot_stride,
                           const int32_t* active, const int32_t* n_active, const int32_t* offsets,
                           int E, const int8_t* q, const uint16_t* ds, int R, int d, int f,
                           float* h, void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 5 -- the down-projection q8_1 quantization of the hidden rows ([#1368]
 * intro calls it unchanged): hq int8 [R][f], hds uint16 [R][f/32][2] from
 * h float [R][f].  Same quantizer as stage 2 with the identity row map.
 * h 16-byte aligned, hq 16-byte aligned, hds 4-byte aligned.
 */
int moe_requant_hidden_q8_1(const float* h, int R, int f, int8_t* hq, uint16_t* hds,
                            void* stream);

/*
 * Stages 4 and 5 in one launch: the gate/up product of stage 4 whose epilogue
 * quantizes the hidden rows to q8_1 itself (stage 5, [#1368] intro, applied to
 * h) instead of writing h.  hq int8 [R][f] and hds uint16 [R][f/32][2] out are
 * byte-identical to moe_grouped_mmq_gateup followed by moe_requant_hidden_q8_1
 * (same fp32 h, same block arithmetic).  The pages name a fused expert path
 * ([#439] rebase note, [#1368] "Identity" tests) without defining it; this is
 * our own fusion.  Tensor-core kernel only: returns MOE_ERR_UNSUPPORTED where
 * moe_grouped_mmq_gateup would take the CUDA-core kernel (d % 256 != 0,
 * f % 128 != 0, or MOE_MMQ_PATH=simt).  hds 4-byte aligned (MOE_W_Q2_K: the
 * D2S6 layout, 8-byte aligned); otherwise as stage 4.
 */
int moe_grouped_mmq_gateup_q8_1(int wtype, const uint8_t* group_base, size_t slot_stride,
                                const int32_t* active, const int32_t* n_active,
                                const int32_t* offsets, int E, const int8_t* q, const uint16_t* ds,
                                int R, int d, int f, int8_t* hq, uint16_t* hds, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * Stage 6 -- grouped quantized matmul, down projection: y[r,i] = sum over
 * blocks b of dWd[i,b]*dh[r,b]*I_b (+ mWd[i,b]*sh[r,b] for Q4_1; Q2_K as in
 * stage 4), fp32.
 *   hq, hds from stage 5 (D2S6 for MOE_W_Q2_K); y float [R][d] out.  Alignment
 *   and shapes as stage 4.
 * Q8_0, Q4_1 and Q2_0 shapes that fit the tensor cores run by default on the
 * folded-scale kernel: each dequantized value d*q is split exactly into two
 * binary16 terms and the whole reduction accumulates in fp32 on the tensor
 * cores, so y differs from the definition's per-block order of roundings by at
 * most a few fp32 units of the sum of |w*x| (the accumulation count times
 * 2^-23, the smallest cross term dropped at 2^-22).  MOE_MMQ_PATH=blockscale
 * selects the per-block-scaling kernel, whose y equals the definition's bit
 * for bit.
 */
int moe_grouped_mmq_down(int wtype, const uint8_t* group_base, size_t slot_stride,
                         const int32_t* active, const int32_t* n_active, const int32_t* offsets,
                         int E, const int8_t* hq, const uint16_t* hds, int R, int d, int f,
                         float* y, void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 7 -- [#1282] "What it does": the combine weights each of a token's
 * rows by its top-k weight:  out[t,i] = sum over k ascending of
 * w[t*K+k] * y[slot[t*K+k], i], accumulated as acc = fma(w, y, acc) from 0.
 * Rows with slot outside [0, R) add nothing.
 *   y float [R][d], 16-byte aligned;  w float [T*K];  out float [T][d] out,
 *   16-byte aligned.  d % 4 == 0.
 */
int moe_combine_topk(const float* y, int R, const int32_t* slot, const float* w, int T, int K,
                     int d, float* out, void* stream);

/*
 * Stages 6 and 7 in one call: the down product of stage 6 (y float [R][d] is
 * written as there) with the combine of stage 7 done in its epilogue.  Each
 * row of a work item counts down its token's arrival counter for the item's
 * 256 output columns (a workspace region, set by a small kernel first); the
 * item that writes a token's last row computes out[t, those columns] with
 * stage 7's arithmetic (fma chain over k ascending from 0), so out is
 * bit-identical to moe_grouped_mmq_down followed by moe_combine_topk whatever
 * the order in which items finish, on the same kernel moe_grouped_mmq_down
 * picks (folded scales by default, per-block scaling under
 * MOE_MMQ_PATH=blockscale).  A token with no valid row gets a zero row.
 *   src [R] and slot [T*K] from stage 1; w float [T*K]; out float [T][d] out,
 *   16-byte aligned; R must equal T*K.  The workspace is the one
 *   moe_workspace_size(T, K, E, d, f) sizes.  Tensor-core shapes only
 *   (MOE_ERR_UNSUPPORTED otherwise, and under MOE_MMQ_PATH=simt); otherwise as
 *   stage 6.
 */
int moe_grouped_mmq_down_combine(int wtype, const uint8_t* group_base, size_t slot_stride,
                                 const int32_t* active, const int32_t* n_active,
                                 const int32_t* offsets, int E, const int8_t* hq,
                                 const uint16_t* hds, int R, int d, int f, const int32_t* src,
                                 const int32_t* slot, const float* w, int T, int K, float* y,
                                 float* out, void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 1 without a workspace.  The pull-request pages have no counterpart of
 * this call; it exists for callers that cannot allocate device memory and so
 * cannot hand the library a workspace -- for example code embedded in a host
 * framework that owns every device allocation, or code that must not trigger
 * cudaMalloc's implicit device synchronization.  It computes exactly what
 * moe_build_slot_map computes (same arguments without ws / ws_bytes) and
 * allocates nothing: its scratch is a file-scope device array of 1 MiB + 256 B
 * that every GPU which loads the library holds until the process exits, and it
 * calls no cudaMalloc or cudaFree.
 *   - Limit: ceil(T*K / 1024) * E <= 262144 (the per-chunk expert counts must
 *     fit the array), e.g. T*K <= 262144 at E = 1024 or T*K <= 524288 at E = 512;
 *     larger sizes return MOE_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up the array's device address with that
 *     device current (cudaGetSymbolAddress); make that first call before any
 *     stream capture.
 *   - Every call shares the one array, which keeps the previous call's
 *     contents: each call clears its header first, and calls that overlap on
 *     the GPU (other streams, or other threads' calls on this device) race --
 *     run them one after another.
 *   - Ids outside [0, E) are dropped (slot -1) as in moe_build_slot_map; the
 *     error word is not reported.
 */
int moe_build_slot_map_noalloc(const int32_t* ids, int T, int K, int E, int32_t* offsets,
                               int32_t* slot, int32_t* src, int32_t* active, int32_t* n_active,
                               void* stream);

/*
 * The whole layer with the expert records in HOST memory (pinned, for example
 * from cudaHostAlloc), streamed to the GPU as the pull-request pages' streamed
 * walk does ([#372] "What changes"; [#439] "Ring-slot safety"):
 *   - copy_stream: each routed expert's record, in ascending id order, is copied
 *     (one cudaMemcpyAsync per record) into the next slot of a device staging
 *     ring of ring_groups x 16 slots; before refilling a slot the copy stream
 *     waits on the event that last released it; a group's last copy records
 *     the group's "staged" event;
 *   - compute_stream: per group of 16 routed experts, one wait on "staged", one
 *     gather launch from the ring into the 16-slot MMQ group buffer, one event
 *     that releases all of the group's ring slots, then the group's stage 4, 5
 *     and 6 calls; stage 7 once at the end.
 * Stages 1-2 run first on compute_stream; the call then synchronizes it once to
 * read the routed experts and their row offsets into b->host_scratch, and
 * returns after enqueuing the rest (asynchronous from there).  The output is
 * bit-identical to the resident layer's (the same kernels on the same bytes).
 * The library pairs 2 x 64 CUDA events with each device on first use and keeps
 * them for the process; calls on one device that overlap must not share a
 * ring_groups slice of them, so run them one after another.
 *   - host_arena: host pointer, record e at e * arena_stride (rec_bytes each).
 *   - ring: device, ring_groups * 16 * slot_stride bytes; group_buf: device,
 *     16 * slot_stride bytes (128-byte aligned, slot_stride % 128 == 0);
 *     group_counts: device int32 [ceil(E / 16)];
 *     host_scratch: pinned host int32 [2 * E + 2 + ceil(E / 16)] (routed experts,
 *     their row offsets, then the per-group expert counts staged for the
 *     device); the caller must not write it while a call is in flight.
 *   - The other buffers as the stage calls document (q, ds for T*K rows of d;
 *     h, hq, hds for T*K rows of f; ds and hds in the D2S6 layout for
 *     MOE_W_Q2_K; y for T*K rows of d; ws of
 *     moe_workspace_size(T, K, E, d, f) bytes).
 *   - ring_groups in [1, 64]; compute_stream != copy_stream.
 */
typedef struct moe_stream_buffers {
    uint8_t* ring;
    uint8_t* group_buf;
    int32_t* group_counts;
    int32_t* offsets;
    int32_t* slot;
    int32_t* src;
    int32_t* active;
    int32_t* n_active;
    int8_t* q;
    uint16_t* ds;
    float* h;
    int8_t* hq;
    uint16_t* hds;
    float* y;
    void* ws;
    size_t ws_bytes;
    int32_t* host_scratch;
} moe_stream_buffers;

int moe_layer_forward_streamed(int wtype, int T, int K, int E, int d, int f, const float* x,
                               const int32_t* ids, const float* w, float* out,
                               const uint8_t* host_arena, size_t rec_bytes, size_t arena_stride,
                               size_t slot_stride, int ring_groups, const moe_stream_buffers* b,
                               void* compute_stream, void* copy_stream);

/* Synchronize `stream`, read the workspace error word into *bits (host) and
   clear it.  Returns MOE_ERR_DEVICE if any bit was set, MOE_OK otherwise. */
int moe_device_error(void* ws, uint32_t* bits, void* stream);

/* Number of kernels the library has launched in this process (a diagnostic
   counter for benchmarks; calls that return early launch nothing). */
unsigned long long moe_launch_count(void);

/* Human-readable text of a moe_status value. */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_Q8_H */
