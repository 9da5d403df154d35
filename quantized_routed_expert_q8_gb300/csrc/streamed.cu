// The layer with the expert records in host memory: the streamed walk of the
// pull-request pages ("Prompt path: an MMQ group's experts gathered in one
// launch, after one wait, released by one event", "What changes"; "#439 ...",
// "Ring-slot safety"), on GB300 over NVLink-C2C from pinned host memory.
//
//   copy stream:    for each routed expert in ascending id order, copy its record
//                   into the next staging-ring slot (one cudaMemcpyAsync per
//                   record); before refilling a slot, wait for the event that
//                   released it (used_of[slot]); after a group's last copy,
//                   record the group's `staged` event.
//   compute stream: per group of 16 experts, one wait (on `staged`: the copy
//                   stream is in order, so its last copy covers the others),
//                   one gather launch from the ring slots into the MMQ group
//                   buffer, one `used` event that gives all of the group's ring
//                   slots back; then the group's gate/up, hidden re-quantization
//                   and down products.  The combine runs once at the end.
//
// Only routed experts are streamed, in ascending id order, so no ring entry is
// ever skipped inside an open group.  The host learns which experts are routed
// from one device-to-host copy after the routing map (the call's one
// synchronization: the per-group counts go back from the pinned host scratch
// without another).  Every product runs in the same kernels as the resident
// layer on the same bytes, so the output is bit-identical to it.
#include <mutex>
#include <vector>

#include "common.cuh"

using moe::MAX_E;

namespace {

constexpr int GROUP = 16;
constexpr int MAX_RING_GROUPS = 64;

// Events are created once per device and kept for the process.
struct EventPool {
    cudaEvent_t staged[MAX_RING_GROUPS];
    cudaEvent_t used[MAX_RING_GROUPS];
    bool ready = false;
};
constexpr int kMaxDevices = 64;
std::mutex g_ev_mutex;
EventPool g_pools[kMaxDevices];

int event_pool(EventPool** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_ev_mutex);
    EventPool& p = g_pools[dev];
    if (!p.ready) {
        for (int i = 0; i < MAX_RING_GROUPS; ++i) {
            if (cudaEventCreateWithFlags(&p.staged[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.used[i], cudaEventDisableTiming) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        p.ready = true;
    }
    *out = &p;
    return MOE_OK;
}

}  // namespace

extern "C" int moe_layer_forward_streamed(int wtype, int T, int K, int E, int d, int f,
                                          const float* x, const int32_t* ids, const float* w,
                                          float* out, const uint8_t* host_arena, size_t rec_bytes,
                                          size_t arena_stride, size_t slot_stride, int ring_groups,
                                          const moe_stream_buffers* b, void* compute_stream,
                                          void* copy_stream) {
    if (!b || !host_arena || ring_groups < 1 || ring_groups > MAX_RING_GROUPS)
        return MOE_ERR_INVALID_ARG;
    if (T < 0 || K <= 0 || E <= 0 || E > MAX_E || d <= 0 || f <= 0) return MOE_ERR_INVALID_ARG;
    if (rec_bytes == 0 || rec_bytes > arena_stride || rec_bytes > slot_stride)
        return MOE_ERR_INVALID_ARG;
    if (!b->ring || !b->group_buf || !b->group_counts || !b->host_scratch)
        return MOE_ERR_INVALID_ARG;
    if (compute_stream == copy_stream) return MOE_ERR_INVALID_ARG;  // the walk overlaps them
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(compute_stream);
    cudaStream_t xs = reinterpret_cast<cudaStream_t>(copy_stream);
    const int R = T * K;
    int rc;

    // stages 1 and 2 as in the resident layer
    rc = moe_build_slot_map(ids, T, K, E, b->offsets, b->slot, b->src, b->active, b->n_active,
                            b->ws, b->ws_bytes, compute_stream);
    if (rc != MOE_OK) return rc;
    // Q2_K's MMQ reads the D2S6 layout (d, s, s_lo, s_hi); the others (d, s)
    const bool d2s6 = wtype == MOE_W_Q2_K;
    const int dsw = d2s6 ? 4 : 2;
    rc = (d2s6 ? moe_quantize_scatter_q8_1_d2s6 : moe_quantize_scatter_q8_1)(
        x, T, d, K, b->slot, R, b->q, b->ds, compute_stream);
    if (rc != MOE_OK) return rc;

    // the routed experts and their row ranges, on the host
    int32_t* hs = b->host_scratch;  // [0] n_active, [1..E] active, [E+1..2E+1] offsets
    if (cudaMemcpyAsync(hs, b->n_active, sizeof(int32_t), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaMemcpyAsync(hs + 1, b->active, sizeof(int32_t) * E, cudaMemcpyDeviceToHost, cs) !=
            cudaSuccess ||
        cudaMemcpyAsync(hs + 1 + E, b->offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost,
                        cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int n_active = hs[0];
    const int32_t* active = hs + 1;
    const int32_t* offsets = hs + 1 + E;
    if (n_active < 0 || n_active > E) return MOE_ERR_DEVICE;
    const int n_groups = (n_active + GROUP - 1) / GROUP;

    // per-group expert counts, on the device, for the grouped products; staged in
    // the caller's pinned host_scratch, which no later host write touches before
    // this copy has run (the next call writes it only after its own
    // synchronization of compute_stream), so the copy needs no wait
    int32_t* counts = hs + 2 * E + 2;
    for (int g = 0; g < n_groups; ++g) counts[g] = std::min(GROUP, n_active - g * GROUP);
    if (n_groups > 0 && cudaMemcpyAsync(b->group_counts, counts, sizeof(int32_t) * n_groups,
                                        cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return MOE_ERR_CUDA;

    EventPool* ev = nullptr;
    rc = event_pool(&ev);
    if (rc != MOE_OK) return rc;
    const int ring_slots = ring_groups * GROUP;
    std::vector<int> used_of(ring_slots, -1);  // ring slot -> `used` event that last released it

    for (int g = 0; g < n_groups; ++g) {
        const int n = counts[g];
        const int e_ev = g % ring_groups;
        int slots[GROUP];
        // copy stream: stage the group's records
        for (int j = 0; j < n; ++j) {
            const int p = g * GROUP + j;
            const int s = p % ring_slots;
            slots[j] = s;
            if (used_of[s] >= 0 && cudaStreamWaitEvent(xs, ev->used[used_of[s]], 0) != cudaSuccess)
                return MOE_ERR_CUDA;
            if (cudaMemcpyAsync(b->ring + (size_t)s * slot_stride,
                                host_arena + (size_t)active[p] * arena_stride, rec_bytes,
                                cudaMemcpyHostToDevice, xs) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        if (cudaEventRecord(ev->staged[e_ev], xs) != cudaSuccess) return MOE_ERR_CUDA;
        // compute stream: one wait, one gather, one release
        if (cudaStreamWaitEvent(cs, ev->staged[e_ev], 0) != cudaSuccess) return MOE_ERR_CUDA;
        rc = moe_group_gather(b->ring, rec_bytes, slot_stride, slots, n, 0, b->group_buf,
                              slot_stride, compute_stream);
        if (rc != MOE_OK) return rc;
        if (cudaEventRecord(ev->used[e_ev], cs) != cudaSuccess) return MOE_ERR_CUDA;
        for (int j = 0; j < n; ++j) used_of[slots[j]] = e_ev;
        // the group's products: its experts' rows are contiguous
        const int r0 = offsets[active[g * GROUP]];
        const int r1 = offsets[active[g * GROUP + n - 1] + 1];
        rc = moe_grouped_mmq_gateup(wtype, b->group_buf, slot_stride, b->active + g * GROUP,
                                    b->group_counts + g, b->offsets, E, b->q, b->ds, R, d, f, b->h,
                                    b->ws, b->ws_bytes, compute_stream);
        if (rc != MOE_OK) return rc;
        if (r1 > r0) {
            rc = (d2s6 ? moe_requant_hidden_q8_1_d2s6 : moe_requant_hidden_q8_1)(
                b->h + (size_t)r0 * f, r1 - r0, f, b->hq + (size_t)r0 * f,
                b->hds + (size_t)r0 * (f / 32) * dsw, compute_stream);
            if (rc != MOE_OK) return rc;
        }
        rc = moe_grouped_mmq_down(wtype, b->group_buf, slot_stride, b->active + g * GROUP,
                                  b->group_counts + g, b->offsets, E, b->hq, b->hds, R, d, f, b->y,
                                  b->ws, b->ws_bytes, compute_stream);
        if (rc != MOE_OK) return rc;
    }
    return moe_combine_topk(b->y, R, b->slot, w, T, K, d, out, compute_stream);
}
