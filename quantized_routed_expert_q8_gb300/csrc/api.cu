// C ABI of the library (declared in include/moe_q8.h): argument checks on the
// host, then the stage launches.  Nothing here allocates or synchronizes
// except moe_device_error.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "mmq.cuh"

namespace moe {
int launch_build_slot_map(const int32_t*, int, int, int, int32_t*, int32_t*, int32_t*, int32_t*,
                          int32_t*, uint8_t*, cudaStream_t);
int launch_quantize_scatter(const float*, int, int, int, const int32_t*, int, int8_t*, uint16_t*,
                            bool, cudaStream_t);
int launch_quantize_gather(const float*, int, int, const int32_t*, int, int8_t*, uint16_t*, bool,
                           cudaStream_t);
int launch_requant_hidden(const float*, int, int, int8_t*, uint16_t*, bool, cudaStream_t);
int launch_group_gather(const uint8_t*, size_t, size_t, const int32_t*, int, int, uint8_t*, size_t,
                        cudaStream_t);
int launch_group_gather_active(const uint8_t*, size_t, size_t, const int32_t*, const int32_t*, int,
                               uint8_t*, size_t, cudaStream_t);
int launch_combine_topk(const float*, int, const int32_t*, const float*, int, int, int, float*,
                        cudaStream_t);
int launch_mmq_simt(int, bool, const uint8_t*, size_t, const int32_t*, const int32_t*,
                    const int32_t*, int, const int8_t*, const uint16_t*, int, int, int, float*,
                    uint8_t*, const WsLayout&, cudaStream_t);
int launch_mmq_tc(int, bool, const uint8_t*, size_t, const int32_t*, const int32_t*,
                  const int32_t*, int, const int8_t*, const uint16_t*, int, int, int, float*,
                  uint8_t*, const WsLayout&, const MmqFused&, cudaStream_t);
bool mmq_tc_supported(int wtype, bool gateup, int d, int f);
}  // namespace moe

#include <atomic>

namespace moe {
static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace moe

using namespace moe;

namespace {

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool al(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline bool wtype_ok(int w) {
    return w == MOE_W_Q8_0 || w == MOE_W_Q4_1 || w == MOE_W_Q2_0 || w == MOE_W_Q2_K;
}
// reduction widths a weight type's blocks need: 32, or Q2_K's 256-weight super-blocks
inline bool widths_ok(int w, int d, int f) {
    const int b = w == MOE_W_Q2_K ? QKK : QK;
    return d % b == 0 && f % b == 0;
}

// Kernel choice for the grouped MMQ.  Stage 4 (gate/up) runs on the tensor-core
// kernel that forms each block's integer dot exactly and scales it on the CUDA
// cores in the scalar definition's order, so the hidden rows -- which stage 5
// re-quantizes -- equal the definition's values.  Stage 6 (down) runs on the
// folded-scale kernel (binary16 hi + lo operands, whole reduction in TMEM), whose
// result differs from that order by a few fp32 ulps; its output is only
// combined, never re-quantized.
// MOE_MMQ_PATH=simt forces the CUDA-core MMQ (the cross-check of the tensor-core
// paths); =blockscale the per-block-scaling tensor-core kernel for both stages;
// =fold the folded-scale kernel for both stages.
inline bool mmq_path_is(const char* name) {
    const char* v = std::getenv("MOE_MMQ_PATH");
    return v && std::strcmp(v, name) == 0;
}
inline bool force_simt() { return mmq_path_is("simt"); }

// recover the (T, K) the workspace was sized for is not possible; the MMQ and
// slot-map calls size it from their own arguments
int check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (!ws) return MOE_ERR_WORKSPACE;
    if (!al(ws, 256)) return MOE_ERR_ALIGNMENT;
    if (ws_bytes < need) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// F: the fused epilogues (tensor-core kernel only), or null
int mmq_common(int wtype, bool gateup, const uint8_t* group_base, size_t slot_stride,
               const int32_t* active, const int32_t* n_active, const int32_t* offsets, int E,
               const int8_t* xq, const uint16_t* xds, int R, int d, int f, float* out, void* ws,
               size_t ws_bytes, void* stream, const MmqFused* F = nullptr, size_t ws_need = 0) {
    if (!wtype_ok(wtype) || R < 0 || d <= 0 || f <= 0 || E <= 0 || E > MAX_E)
        return MOE_ERR_INVALID_ARG;
    if (!widths_ok(wtype, d, f)) return MOE_ERR_INVALID_ARG;
    if (!active || !n_active || !offsets) return MOE_ERR_INVALID_ARG;
    const bool q8_out = F && F->hq;
    if (R > 0 && (!group_base || !xq || !xds || (!out && !q8_out))) return MOE_ERR_INVALID_ARG;
    if (q8_out && R > 0 && !F->hds) return MOE_ERR_INVALID_ARG;
    if (!al(group_base, 128) || slot_stride % 128) return MOE_ERR_ALIGNMENT;
    if (!al(xq, 16) || !al(xds, 16) || !al(out, 16)) return MOE_ERR_ALIGNMENT;
    if (q8_out && !al(F->hds, ds_halves(wtype) == 4 ? 8 : 4)) return MOE_ERR_ALIGNMENT;
    // the tile list needs R/16 + E entries: size it as if T*K = R
    WsLayout W = ws_layout(R, 1, E, d, f);
    int rc = check_ws(ws, ws_bytes, W.core > ws_need ? W.core : ws_need);
    if (rc) return rc;
    const bool tc = !force_simt() && mmq_tc_supported(wtype, gateup, d, f);
    // the folded-scale kernel takes the down projection's combine, not the
    // gate/up re-quantization
    const bool fold = (!F || (!gateup && F->comb && !F->hq)) && !force_simt() &&
                      !mmq_path_is("blockscale") && (!gateup || mmq_path_is("fold")) &&
                      mmq_fold_supported(wtype, d, f);
    if (F && !tc && !fold) return MOE_ERR_UNSUPPORTED;
    if (R == 0) return MOE_OK;
    uint8_t* w8 = (uint8_t*)ws;
    if (fold)
        return launch_mmq_fold(wtype, gateup, group_base, slot_stride, active, n_active, offsets,
                               E, xq, xds, R, d, f, out, w8, W, F ? *F : MmqFused{}, S(stream));
    if (tc)
        return launch_mmq_tc(wtype, gateup, group_base, slot_stride, active, n_active, offsets, E,
                             xq, xds, R, d, f, out, w8, W, F ? *F : MmqFused{}, S(stream));
    return launch_mmq_simt(wtype, gateup, group_base, slot_stride, active, n_active, offsets, E, xq,
                           xds, R, d, f, out, w8, W, S(stream));
}

}  // namespace

extern "C" {

size_t moe_expert_record_bytes(int wtype, int d, int f) {
    if (!wtype_ok(wtype) || d <= 0 || f <= 0 || !widths_ok(wtype, d, f)) return 0;
    return rec_layout(wtype, d, f).bytes;
}

void moe_expert_record_offsets(int wtype, int d, int f, size_t* gate, size_t* up, size_t* down) {
    RecLayout R = rec_layout(wtype, d, f);
    if (gate) *gate = R.gate;
    if (up) *up = R.up;
    if (down) *down = R.down;
}

size_t moe_workspace_size(int T, int K, int E, int d, int f) {
    if (T < 0 || K < 0 || E <= 0) return 0;
    WsLayout a = ws_layout(T, K, E, d, f);
    return a.total;
}

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < 256) return MOE_ERR_WORKSPACE;
    if (!al(ws, 256)) return MOE_ERR_ALIGNMENT;
    return cudaMemsetAsync(ws, 0, 256, S(stream)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_build_slot_map(const int32_t* ids, int T, int K, int E, int32_t* offsets, int32_t* slot,
                       int32_t* src, int32_t* active, int32_t* n_active, void* ws,
                       size_t ws_bytes, void* stream) {
    if (T < 0 || K < 0 || E <= 0 || E > MAX_E) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    if (!offsets || !active || !n_active) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K > 0 && (!ids || !slot || !src)) return MOE_ERR_INVALID_ARG;
    int rc = check_ws(ws, ws_bytes, ws_layout(T, K, E, 0, 0).total);
    if (rc) return rc;
    return launch_build_slot_map(ids, T, K, E, offsets, slot, src, active, n_active, (uint8_t*)ws,
                                 S(stream));
}

}  // extern "C"

namespace {

int quantize_scatter(const float* x, int T, int d, int K, const int32_t* slot, int R, int8_t* q,
                     uint16_t* ds, bool d2s6, void* stream) {
    if (T < 0 || K < 0 || R < 0 || d <= 0 || d % QK) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K > 0 && (!x || !slot)) return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!q || !ds)) return MOE_ERR_INVALID_ARG;
    if (!al(x, 16) || !al(q, 16) || !al(ds, d2s6 ? 8 : 4)) return MOE_ERR_ALIGNMENT;
    if (T == 0 || K == 0 || R == 0) return MOE_OK;
    return launch_quantize_scatter(x, T, d, K, slot, R, q, ds, d2s6, S(stream));
}

int quantize_gather(const float* x, int T, int d, const int32_t* src, int R, int8_t* q,
                    uint16_t* ds, bool d2s6, void* stream) {
    if (T < 0 || R < 0 || d <= 0 || d % QK) return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!x || !src || !q || !ds)) return MOE_ERR_INVALID_ARG;
    if (!al(x, 16) || !al(q, 16) || !al(ds, d2s6 ? 8 : 4)) return MOE_ERR_ALIGNMENT;
    if (R == 0) return MOE_OK;
    return launch_quantize_gather(x, T, d, src, R, q, ds, d2s6, S(stream));
}

int requant_hidden(const float* h, int R, int f, int8_t* hq, uint16_t* hds, bool d2s6,
                   void* stream) {
    if (R < 0 || f <= 0 || f % QK) return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!h || !hq || !hds)) return MOE_ERR_INVALID_ARG;
    if (!al(h, 16) || !al(hq, 16) || !al(hds, d2s6 ? 8 : 4)) return MOE_ERR_ALIGNMENT;
    if (R == 0) return MOE_OK;
    return launch_requant_hidden(h, R, f, hq, hds, d2s6, S(stream));
}

}  // namespace

extern "C" {

int moe_quantize_scatter_q8_1(const float* x, int T, int d, int K, const int32_t* slot, int R,
                              int8_t* q, uint16_t* ds, void* stream) {
    return quantize_scatter(x, T, d, K, slot, R, q, ds, false, stream);
}

int moe_quantize_scatter_q8_1_d2s6(const float* x, int T, int d, int K, const int32_t* slot,
                                   int R, int8_t* q, uint16_t* ds, void* stream) {
    return quantize_scatter(x, T, d, K, slot, R, q, ds, true, stream);
}

int moe_quantize_gather_q8_1(const float* x, int T, int d, const int32_t* src, int R, int8_t* q,
                             uint16_t* ds, void* stream) {
    return quantize_gather(x, T, d, src, R, q, ds, false, stream);
}

int moe_quantize_gather_q8_1_d2s6(const float* x, int T, int d, const int32_t* src, int R,
                                  int8_t* q, uint16_t* ds, void* stream) {
    return quantize_gather(x, T, d, src, R, q, ds, true, stream);
}

int moe_group_gather(const uint8_t* arena, size_t rec_bytes, size_t arena_stride,
                     const int32_t* expert_ids, int n, int first_slot, uint8_t* group_buf,
                     size_t slot_stride, void* stream) {
    if (n < 1 || n > 16 || first_slot < 0 || first_slot + n > 16) return MOE_ERR_INVALID_ARG;
    if (!arena || !expert_ids || !group_buf) return MOE_ERR_INVALID_ARG;
    if (rec_bytes > arena_stride || rec_bytes > slot_stride) return MOE_ERR_INVALID_ARG;
    for (int j = 0; j < n; ++j)
        if (expert_ids[j] < 0) return MOE_ERR_INVALID_ARG;
    return launch_group_gather(arena, rec_bytes, arena_stride, expert_ids, n, first_slot, group_buf,
                               slot_stride, S(stream));
}

int moe_group_gather_active(const uint8_t* arena, size_t rec_bytes, size_t arena_stride,
                            const int32_t* active, const int32_t* n_active, int max_active,
                            uint8_t* group_base, size_t slot_stride, void* stream) {
    if (max_active < 0 || max_active > MAX_E) return MOE_ERR_INVALID_ARG;
    if (!arena || !active || !n_active || !group_base) return MOE_ERR_INVALID_ARG;
    if (rec_bytes > arena_stride || rec_bytes > slot_stride) return MOE_ERR_INVALID_ARG;
    return launch_group_gather_active(arena, rec_bytes, arena_stride, active, n_active, max_active,
                                      group_base, slot_stride, S(stream));
}

int moe_grouped_mmq_gateup(int wtype, const uint8_t* group_base, size_t slot_stride,
                           const int32_t* active, const int32_t* n_active, const int32_t* offsets,
                           int E, const int8_t* q, const uint16_t* ds, int R, int d, int f,
                           float* h, void* ws, size_t ws_bytes, void* stream) {
    return mmq_common(wtype, true, group_base, slot_stride, active, n_active, offsets, E, q, ds, R,
                      d, f, h, ws, ws_bytes, stream);
}

int moe_grouped_mmq_gateup_q8_1(int wtype, const uint8_t* group_base, size_t slot_stride,
                                const int32_t* active, const int32_t* n_active,
                                const int32_t* offsets, int E, const int8_t* q, const uint16_t* ds,
                                int R, int d, int f, int8_t* hq, uint16_t* hds, void* ws,
                                size_t ws_bytes, void* stream) {
    MmqFused F;
    F.hq = hq;
    F.hds = hds;
    if (R > 0 && (!hq || !hds)) return MOE_ERR_INVALID_ARG;
    return mmq_common(wtype, true, group_base, slot_stride, active, n_active, offsets, E, q, ds, R,
                      d, f, nullptr, ws, ws_bytes, stream, &F);
}

int moe_requant_hidden_q8_1(const float* h, int R, int f, int8_t* hq, uint16_t* hds,
                            void* stream) {
    return requant_hidden(h, R, f, hq, hds, false, stream);
}

int moe_requant_hidden_q8_1_d2s6(const float* h, int R, int f, int8_t* hq, uint16_t* hds,
                                 void* stream) {
    return requant_hidden(h, R, f, hq, hds, true, stream);
}

int moe_grouped_mmq_down(int wtype, const uint8_t* group_base, size_t slot_stride,
                         const int32_t* active, const int32_t* n_active, const int32_t* offsets,
                         int E, const int8_t* hq, const uint16_t* hds, int R, int d, int f,
                         float* y, void* ws, size_t ws_bytes, void* stream) {
    return mmq_common(wtype, false, group_base, slot_stride, active, n_active, offsets, E, hq, hds,
                      R, d, f, y, ws, ws_bytes, stream);
}

int moe_grouped_mmq_down_combine(int wtype, const uint8_t* group_base, size_t slot_stride,
                                 const int32_t* active, const int32_t* n_active,
                                 const int32_t* offsets, int E, const int8_t* hq,
                                 const uint16_t* hds, int R, int d, int f, const int32_t* src,
                                 const int32_t* slot, const float* w, int T, int K, float* y,
                                 float* out, void* ws, size_t ws_bytes, void* stream) {
    if (T < 0 || K <= 0 || (long long)T * K != R) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!out || !slot || !w || !src)) return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!group_base || !hq || !hds || !y)) return MOE_ERR_INVALID_ARG;
    if (d <= 0 || d % 4) return MOE_ERR_INVALID_ARG;
    if (!al(out, 16)) return MOE_ERR_ALIGNMENT;
    const WsLayout W = ws_layout(T, K, E, d, f);
    MmqFused F;
    F.comb = out;
    F.src = src;
    F.slot = slot;
    F.w = w;
    F.arrivals = (int32_t*)((uint8_t*)ws + W.arrivals);
    F.K = K;
    F.T = T;
    // argument and workspace checks first, nothing launched on failure
    int rc = mmq_common(wtype, false, group_base, slot_stride, active, n_active, offsets, E, hq,
                        hds, 0, d, f, y, ws, ws_bytes, stream, &F, W.total);
    if (rc != MOE_OK) return rc;
    rc = launch_combine_arrivals(slot, T, K, R, d, F.arrivals, out, S(stream));
    if (rc != MOE_OK) return rc;
    return mmq_common(wtype, false, group_base, slot_stride, active, n_active, offsets, E, hq, hds,
                      R, d, f, y, ws, ws_bytes, stream, &F, W.total);
}

int moe_combine_topk(const float* y, int R, const int32_t* slot, const float* w, int T, int K,
                     int d, float* out, void* stream) {
    if (T < 0 || K < 0 || R < 0 || d <= 0 || d % 4) return MOE_ERR_INVALID_ARG;
    if (T > 0 && !out) return MOE_ERR_INVALID_ARG;
    if ((long long)T * K > 0 && (!slot || !w)) return MOE_ERR_INVALID_ARG;
    if (R > 0 && !y) return MOE_ERR_INVALID_ARG;
    if (!al(y, 16) || !al(out, 16)) return MOE_ERR_ALIGNMENT;
    if (T == 0) return MOE_OK;
    return launch_combine_topk(y, R, slot, w, T, K, d, out, S(stream));
}

int moe_device_error(void* ws, uint32_t* bits, void* stream) {
    if (!ws || !bits) return MOE_ERR_INVALID_ARG;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, S(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    *bits = v;
    if (v && cudaMemsetAsync(ws, 0, 4, S(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    return v ? MOE_ERR_DEVICE : MOE_OK;
}

unsigned long long moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_ALIGNMENT: return "misaligned buffer or stride";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_UNSUPPORTED: return "unsupported size";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE: return "device-side error flag set";
        default: return "unknown status";
    }
}

}  // extern "C"
