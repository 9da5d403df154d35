"""GB300 quantized routed-expert (q8_1 MMQ) MoE prefill layer.

A thin ctypes binding over ``libmoe_q8.so`` (hand-written CUDA for sm_103a; C ABI
in ``include/moe_q8.h``).  Every function has the name of the C entry point it
calls and only marshals arguments: torch tensors in, device pointers and sizes
out, the current CUDA stream unless one is given.  All arithmetic runs in the
library's kernels; there is no CPU fallback -- importing this package on a
machine without the built library raises.

``MoeLayer`` owns the per-layer device buffers and runs the seven stages in
order on one stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_q8.so")

MOE_W_Q8_0 = 0
MOE_W_Q4_1 = 1
MOE_W_Q2_0 = 2
MOE_W_Q2_K = 3
QK = 32


def ds_halves(wtype: int) -> int:
    """binary16 entries per 32-block of a q8_1 ds row for a weight type's MMQ:
    (d, s), or (d, s, s_lo, s_hi) -- the D2S6 layout -- for Q2_K."""
    return 4 if wtype == MOE_W_Q2_K else 2

DEV_ERR_BAD_EXPERT_ID = 0x1
DEV_ERR_BAD_ROWS = 0x2
DEV_ERR_TIMEOUT = 0x4
DEV_ERR_RANGE = 0x8

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_SIGNATURES = {
    "moe_expert_record_bytes": (_Z, [_I, _I, _I]),
    "moe_expert_record_offsets": (None, [_I, _I, _I, _P, _P, _P]),
    "moe_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "moe_workspace_init": (_I, [_P, _Z, _P]),
    "moe_build_slot_map": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_quantize_scatter_q8_1": (_I, [_P, _I, _I, _I, _P, _I, _P, _P, _P]),
    "moe_quantize_gather_q8_1": (_I, [_P, _I, _I, _P, _I, _P, _P, _P]),
    "moe_quantize_scatter_q8_1_d2s6": (_I, [_P, _I, _I, _I, _P, _I, _P, _P, _P]),
    "moe_quantize_gather_q8_1_d2s6": (_I, [_P, _I, _I, _P, _I, _P, _P, _P]),
    "moe_requant_hidden_q8_1_d2s6": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_group_gather": (_I, [_P, _Z, _Z, _P, _I, _I, _P, _Z, _P]),
    "moe_group_gather_active": (_I, [_P, _Z, _Z, _P, _P, _I, _P, _Z, _P]),
    "moe_grouped_mmq_gateup": (_I, [_I, _P, _Z, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_requant_hidden_q8_1": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_grouped_mmq_down": (_I, [_I, _P, _Z, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_combine_topk": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P]),
    "moe_grouped_mmq_gateup_q8_1": (_I, [_I, _P, _Z, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P,
                                         _P, _Z, _P]),
    "moe_grouped_mmq_down_combine": (_I, [_I, _P, _Z, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P,
                                          _P, _I, _I, _P, _P, _P, _Z, _P]),
    "moe_build_slot_map_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_layer_forward_streamed": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _Z, _Z,
                                        _I, _P, _P, _P]),
    "moe_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "moe_launch_count": (ctypes.c_ulonglong, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
}
EXPORTED = tuple(_SIGNATURES)


class MoeError(RuntimeError):
    pass


def lib():
    """Load libmoe_q8.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, name: str):
    if rc != 0:
        msg = lib().moe_status_string(rc).decode()
        raise MoeError(f"{name} failed: {msg} ({rc})")


def _dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors passed to libmoe_q8 must live on the GPU")


# --- sizes ------------------------------------------------------------------

def moe_expert_record_bytes(wtype: int, d: int, f: int) -> int:
    return int(lib().moe_expert_record_bytes(wtype, d, f))


def moe_expert_record_offsets(wtype: int, d: int, f: int):
    g, u, dn = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    lib().moe_expert_record_offsets(wtype, d, f, ctypes.byref(g), ctypes.byref(u), ctypes.byref(dn))
    return g.value, u.value, dn.value


def moe_workspace_size(T: int, K: int, E: int, d: int, f: int) -> int:
    return int(lib().moe_workspace_size(T, K, E, d, f))


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().moe_workspace_init(_p(ws), ws.numel() * ws.element_size(), _s(stream)),
           "moe_workspace_init")


# --- the seven stages ---------------------------------------------------------

def moe_build_slot_map(ids, E, offsets, slot, src, active, n_active, ws, stream=None):
    _dev(ids, offsets, slot, src, active, n_active, ws)
    T, K = ids.shape
    _check(lib().moe_build_slot_map(_p(ids), T, K, E, _p(offsets), _p(slot), _p(src), _p(active),
                                    _p(n_active), _p(ws), ws.numel() * ws.element_size(), _s(stream)),
           "moe_build_slot_map")


def moe_quantize_scatter_q8_1(x, slot, K, R, q, ds, stream=None):
    _dev(x, slot, q, ds)
    T, d = x.shape
    _check(lib().moe_quantize_scatter_q8_1(_p(x), T, d, K, _p(slot), R, _p(q), _p(ds), _s(stream)),
           "moe_quantize_scatter_q8_1")


def moe_quantize_gather_q8_1(x, src, R, q, ds, stream=None):
    _dev(x, src, q, ds)
    T, d = x.shape
    _check(lib().moe_quantize_gather_q8_1(_p(x), T, d, _p(src), R, _p(q), _p(ds), _s(stream)),
           "moe_quantize_gather_q8_1")


def moe_quantize_scatter_q8_1_d2s6(x, slot, K, R, q, ds, stream=None):
    _dev(x, slot, q, ds)
    T, d = x.shape
    _check(lib().moe_quantize_scatter_q8_1_d2s6(_p(x), T, d, K, _p(slot), R, _p(q), _p(ds),
                                                _s(stream)), "moe_quantize_scatter_q8_1_d2s6")


def moe_quantize_gather_q8_1_d2s6(x, src, R, q, ds, stream=None):
    _dev(x, src, q, ds)
    T, d = x.shape
    _check(lib().moe_quantize_gather_q8_1_d2s6(_p(x), T, d, _p(src), R, _p(q), _p(ds),
                                               _s(stream)), "moe_quantize_gather_q8_1_d2s6")


def quantizers(wtype: int):
    """(scatter, gather, requant) entry points whose ds layout the weight type's
    MMQ reads: the D2S6 ones for Q2_K, the (d, s) ones otherwise."""
    if wtype == MOE_W_Q2_K:
        return (moe_quantize_scatter_q8_1_d2s6, moe_quantize_gather_q8_1_d2s6,
                moe_requant_hidden_q8_1_d2s6)
    return moe_quantize_scatter_q8_1, moe_quantize_gather_q8_1, moe_requant_hidden_q8_1


def moe_requant_hidden_q8_1_d2s6(h, R, f, hq, hds, stream=None):
    _dev(h, hq, hds)
    _check(lib().moe_requant_hidden_q8_1_d2s6(_p(h), R, f, _p(hq), _p(hds), _s(stream)),
           "moe_requant_hidden_q8_1_d2s6")


def moe_group_gather(arena, rec_bytes, arena_stride, expert_ids, first_slot, group_buf,
                     slot_stride, stream=None):
    """expert_ids: host sequence of up to 16 ints (kernel parameters)."""
    _dev(arena, group_buf)
    ids = (ctypes.c_int32 * len(expert_ids))(*[int(e) for e in expert_ids])
    _check(lib().moe_group_gather(_p(arena), rec_bytes, arena_stride, ctypes.cast(ids, _P),
                                  len(expert_ids), first_slot, _p(group_buf), slot_stride,
                                  _s(stream)), "moe_group_gather")


def moe_group_gather_active(arena, rec_bytes, arena_stride, active, n_active, max_active,
                            group_base, slot_stride, stream=None):
    _dev(arena, active, n_active, group_base)
    _check(lib().moe_group_gather_active(_p(arena), rec_bytes, arena_stride, _p(active),
                                         _p(n_active), max_active, _p(group_base), slot_stride,
                                         _s(stream)), "moe_group_gather_active")


def moe_grouped_mmq_gateup(wtype, group_base, slot_stride, active, n_active, offsets, E, q, ds, R,
                           d, f, h, ws, stream=None):
    _dev(group_base, active, n_active, offsets, q, ds, h, ws)
    _check(lib().moe_grouped_mmq_gateup(wtype, _p(group_base), slot_stride, _p(active), _p(n_active),
                                        _p(offsets), E, _p(q), _p(ds), R, d, f, _p(h), _p(ws),
                                        ws.numel() * ws.element_size(), _s(stream)),
           "moe_grouped_mmq_gateup")


def moe_requant_hidden_q8_1(h, R, f, hq, hds, stream=None):
    _dev(h, hq, hds)
    _check(lib().moe_requant_hidden_q8_1(_p(h), R, f, _p(hq), _p(hds), _s(stream)),
           "moe_requant_hidden_q8_1")


def moe_grouped_mmq_down(wtype, group_base, slot_stride, active, n_active, offsets, E, hq, hds, R,
                         d, f, y, ws, stream=None):
    _dev(group_base, active, n_active, offsets, hq, hds, y, ws)
    _check(lib().moe_grouped_mmq_down(wtype, _p(group_base), slot_stride, _p(active), _p(n_active),
                                      _p(offsets), E, _p(hq), _p(hds), R, d, f, _p(y), _p(ws),
                                      ws.numel() * ws.element_size(), _s(stream)),
           "moe_grouped_mmq_down")


def moe_combine_topk(y, R, slot, w, T, K, d, out, stream=None):
    _dev(y, slot, w, out)
    _check(lib().moe_combine_topk(_p(y), R, _p(slot), _p(w), T, K, d, _p(out), _s(stream)),
           "moe_combine_topk")


def moe_grouped_mmq_gateup_q8_1(wtype, group_base, slot_stride, active, n_active, offsets, E, q,
                                ds, R, d, f, hq, hds, ws, stream=None):
    _dev(group_base, active, n_active, offsets, q, ds, hq, hds, ws)
    _check(lib().moe_grouped_mmq_gateup_q8_1(wtype, _p(group_base), slot_stride, _p(active),
                                             _p(n_active), _p(offsets), E, _p(q), _p(ds), R, d, f,
                                             _p(hq), _p(hds), _p(ws),
                                             ws.numel() * ws.element_size(), _s(stream)),
           "moe_grouped_mmq_gateup_q8_1")


def moe_grouped_mmq_down_combine(wtype, group_base, slot_stride, active, n_active, offsets, E, hq,
                                 hds, R, d, f, src, slot, w, T, K, y, out, ws, stream=None):
    _dev(group_base, active, n_active, offsets, hq, hds, src, slot, w, y, out, ws)
    _check(lib().moe_grouped_mmq_down_combine(wtype, _p(group_base), slot_stride, _p(active),
                                              _p(n_active), _p(offsets), E, _p(hq), _p(hds), R, d,
                                              f, _p(src), _p(slot), _p(w), T, K, _p(y), _p(out),
                                              _p(ws), ws.numel() * ws.element_size(), _s(stream)),
           "moe_grouped_mmq_down_combine")


def moe_build_slot_map_noalloc(ids, E, offsets, slot, src, active, n_active, stream=None):
    """moe_build_slot_map without a workspace, for callers that cannot allocate
    device memory: the scratch is a fixed device array inside the library (see
    include/moe_q8.h for its limit and its once-per-device set-up)."""
    _dev(ids, offsets, slot, src, active, n_active)
    T, K = ids.shape
    _check(lib().moe_build_slot_map_noalloc(_p(ids), T, K, E, _p(offsets), _p(slot), _p(src),
                                            _p(active), _p(n_active), _s(stream)),
           "moe_build_slot_map_noalloc")


class StreamBuffers(ctypes.Structure):
    """moe_stream_buffers: the device (and one host) buffers of the streamed layer."""
    _fields_ = [(n, _P) for n in ("ring", "group_buf", "group_counts", "offsets", "slot", "src",
                                  "active", "n_active", "q", "ds", "h", "hq", "hds", "y", "ws")]
    _fields_ += [("ws_bytes", _Z), ("host_scratch", _P)]


def moe_layer_forward_streamed(wtype, x, ids, w, out, host_arena, rec_bytes, arena_stride,
                               slot_stride, ring_groups, bufs: "StreamBuffers", E, f,
                               compute_stream=None, copy_stream=None):
    """The whole layer with the expert records in host memory (host_arena: a
    pinned CPU uint8 tensor), streamed through the device ring in bufs."""
    _dev(x, ids, w, out)
    if host_arena.is_cuda:
        raise ValueError("host_arena must be a (pinned) host tensor")
    T, d = x.shape
    K = ids.shape[1]
    _check(lib().moe_layer_forward_streamed(wtype, T, K, E, d, f, _p(x), _p(ids), _p(w), _p(out),
                                            ctypes.c_void_p(host_arena.data_ptr()), rec_bytes,
                                            arena_stride, slot_stride, ring_groups,
                                            ctypes.byref(bufs), _s(compute_stream),
                                            _s(copy_stream)),
           "moe_layer_forward_streamed")


def moe_device_error(ws, stream=None) -> int:
    """Synchronize the stream and return (and clear) the workspace error bits."""
    bits = ctypes.c_uint32(0)
    rc = lib().moe_device_error(_p(ws), ctypes.byref(bits), _s(stream))
    if rc not in (0, -6):
        _check(rc, "moe_device_error")
    return int(bits.value)


def moe_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().moe_launch_count())


# --- one layer -------------------------------------------------------------------

class MoeLayer:
    """Device buffers of one MoE layer for up to ``T_max`` tokens, and the seven
    calls in order.  ``arena`` holds the E expert records (uint8, on the GPU,
    record e at e*arena_stride); it stays resident and is not copied per call
    except by the group gather stage."""

    def __init__(self, wtype, E, d, f, K, T_max, arena, rec_bytes, arena_stride, device=None):
        device = device or arena.device
        self.wtype, self.E, self.d, self.f, self.K, self.T_max = wtype, E, d, f, K, T_max
        self.arena, self.rec_bytes, self.arena_stride = arena, rec_bytes, arena_stride
        self.slot_stride = (rec_bytes + 255) // 256 * 256
        R = T_max * K
        i32 = dict(dtype=torch.int32, device=device)
        self.offsets = torch.zeros(E + 1, **i32)
        self.slot = torch.zeros(max(R, 1), **i32)
        self.src = torch.zeros(max(R, 1), **i32)
        self.active = torch.zeros(E, **i32)
        self.n_active = torch.zeros(1, **i32)
        self.q = torch.zeros((max(R, 1), d), dtype=torch.int8, device=device)
        hw = ds_halves(wtype)
        self.ds = torch.zeros((max(R, 1), d // QK, hw), dtype=torch.int16, device=device)
        self.group_buf = torch.zeros(E * self.slot_stride, dtype=torch.uint8, device=device)
        self.h = torch.zeros((max(R, 1), f), dtype=torch.float32, device=device)
        self.hq = torch.zeros((max(R, 1), f), dtype=torch.int8, device=device)
        self.hds = torch.zeros((max(R, 1), f // QK, hw), dtype=torch.int16, device=device)
        self.y = torch.zeros((max(R, 1), d), dtype=torch.float32, device=device)
        self.out = torch.zeros((max(T_max, 1), d), dtype=torch.float32, device=device)
        ws_bytes = moe_workspace_size(T_max, K, E, d, f)
        self.ws = torch.zeros((ws_bytes + 255) // 256 * 256, dtype=torch.uint8, device=device)
        moe_workspace_init(self.ws)

    def _out_writable(self, stream):
        """Order the stream's next write of the output buffer after the copies back
        of a forward_host call that was not waited for."""
        ev = getattr(self, "_out_free", None)
        if ev is not None:
            (stream if stream is not None else torch.cuda.current_stream()).wait_event(ev)

    def forward(self, x, ids, w, stream=None, fused=False):
        """x f32 [T, d], ids int32 [T, K], w f32 [T, K] on the GPU -> out [T, d]
        (a view of the layer's output buffer).  fused=True runs stages 4+5 and
        6+7 as the two fused calls (same bytes; tensor-core shapes only)."""
        T = x.shape[0]
        self._out_writable(stream)
        assert T <= self.T_max and ids.shape == (T, self.K) and w.shape == (T, self.K)
        K, E, d, f = self.K, self.E, self.d, self.f
        R = T * K
        moe_build_slot_map(ids, E, self.offsets, self.slot, self.src, self.active, self.n_active,
                           self.ws, stream)
        scatter, _, requant = quantizers(self.wtype)
        scatter(x, self.slot, K, R, self.q, self.ds, stream)
        moe_group_gather_active(self.arena, self.rec_bytes, self.arena_stride, self.active,
                                self.n_active, E, self.group_buf, self.slot_stride, stream)
        if fused:
            moe_grouped_mmq_gateup_q8_1(self.wtype, self.group_buf, self.slot_stride, self.active,
                                        self.n_active, self.offsets, E, self.q, self.ds, R, d, f,
                                        self.hq, self.hds, self.ws, stream)
            moe_grouped_mmq_down_combine(self.wtype, self.group_buf, self.slot_stride, self.active,
                                         self.n_active, self.offsets, E, self.hq, self.hds, R, d,
                                         f, self.src, self.slot, w, T, K, self.y, self.out,
                                         self.ws, stream)
            return self.out[:T]
        moe_grouped_mmq_gateup(self.wtype, self.group_buf, self.slot_stride, self.active,
                               self.n_active, self.offsets, E, self.q, self.ds, R, d, f, self.h,
                               self.ws, stream)
        requant(self.h, R, f, self.hq, self.hds, stream)
        moe_grouped_mmq_down(self.wtype, self.group_buf, self.slot_stride, self.active,
                             self.n_active, self.offsets, E, self.hq, self.hds, R, d, f, self.y,
                             self.ws, stream)
        moe_combine_topk(self.y, R, self.slot, w, T, K, d, self.out, stream)
        return self.out[:T]

    def forward_host(self, hx, hids, hw, hout, chunks=4, stream=None, wait=True):
        """As forward, from pinned host inputs hx f32 [T, d], hids i32 [T, K],
        hw f32 [T, K] to the pinned host output hout f32 [T, d], with the
        host-device copies overlapped with the layer: an upload stream copies ids
        and w first, then x in `chunks` token slices, each quantized (stage 2 on
        its tokens) as soon as it has landed while the routing map and the group
        gather run; at the end the combine (stage 7) runs per token slice and a
        download stream copies each slice's output back while the next is
        combined.  The same kernels and bytes as forward.

        The device staging of x, ids and w is double-buffered, so the next call's
        uploads may run during this call's layer, and this call's downloads
        during the next call's layer.  wait=True (default): `stream` (default:
        the current stream) waits for the downloads, so hout is complete once
        the stream reaches the point of return.  wait=False: it does not, and
        the returned event marks hout complete -- calls made back to back then
        overlap one call's copies with another's layer.  Returns that event.
        The uploads start at once, ordered only after the layer that last read
        their staging set: hx, hids and hw must hold their values when the call
        is made (a device-to-host copy that fills them must have completed)."""
        T = hx.shape[0]
        assert T <= self.T_max and hids.shape == (T, self.K) and hw.shape == (T, self.K)
        assert hout.shape == (T, self.d)
        dev = self.group_buf.device
        cs = stream if stream is not None else torch.cuda.current_stream(dev)
        if not hasattr(self, "_h2d"):
            self._h2d = torch.cuda.Stream(device=dev)
            self._d2h = torch.cuda.Stream(device=dev)
            tm = max(self.T_max, 1)
            self._staging = [
                {"x": torch.zeros((tm, self.d), dtype=torch.float32, device=dev),
                 "ids": torch.zeros((tm, self.K), dtype=torch.int32, device=dev),
                 "w": torch.zeros((tm, self.K), dtype=torch.float32, device=dev),
                 "free": None}
                for _ in range(2)]
            self._flip = 0
            self._out_free = None
        st = self._staging[self._flip]
        self._flip ^= 1
        up, dn = self._h2d, self._d2h
        K, E, d, f = self.K, self.E, self.d, self.f
        R = T * K
        # slices of at least 1 MB of x: below that the copies are too short to hide anything
        n = max(1, min(chunks, T, T * self.d * 4 // (1 << 20)))
        bounds = [T * i // n for i in range(n + 1)]
        x_ready = [torch.cuda.Event() for _ in range(n)]
        routing_ready = torch.cuda.Event()
        if st["free"] is not None:
            up.wait_event(st["free"])  # the layer that last read this staging set is done
        dx, dids, dw = st["x"], st["ids"], st["w"]
        with torch.cuda.stream(up):
            dids[:T].copy_(hids, non_blocking=True)
            dw[:T].copy_(hw, non_blocking=True)
            routing_ready.record(up)
            for c in range(n):
                t0, t1 = bounds[c], bounds[c + 1]
                dx[t0:t1].copy_(hx[t0:t1], non_blocking=True)
                x_ready[c].record(up)
        ids, w = dids[:T], dw[:T]
        cs.wait_event(routing_ready)
        moe_build_slot_map(ids, E, self.offsets, self.slot, self.src, self.active, self.n_active,
                           self.ws, cs)
        moe_group_gather_active(self.arena, self.rec_bytes, self.arena_stride, self.active,
                                self.n_active, E, self.group_buf, self.slot_stride, cs)
        scatter, _, requant = quantizers(self.wtype)
        for c in range(n):
            t0, t1 = bounds[c], bounds[c + 1]
            cs.wait_event(x_ready[c])
            if t1 > t0:
                scatter(dx[t0:t1], self.slot[t0 * K:t1 * K], K, R, self.q, self.ds, cs)
        moe_grouped_mmq_gateup(self.wtype, self.group_buf, self.slot_stride, self.active,
                               self.n_active, self.offsets, E, self.q, self.ds, R, d, f, self.h,
                               self.ws, cs)
        requant(self.h, R, f, self.hq, self.hds, cs)
        moe_grouped_mmq_down(self.wtype, self.group_buf, self.slot_stride, self.active,
                             self.n_active, self.offsets, E, self.hq, self.hds, R, d, f, self.y,
                             self.ws, cs)
        if self._out_free is not None:
            cs.wait_event(self._out_free)  # the previous call's downloads have read out
        for c in range(n):
            t0, t1 = bounds[c], bounds[c + 1]
            if t1 > t0:
                moe_combine_topk(self.y, R, self.slot[t0 * K:t1 * K], w[t0:t1], t1 - t0, K, d,
                                 self.out[t0:t1], cs)
            combined = torch.cuda.Event()
            combined.record(cs)
            dn.wait_event(combined)
            with torch.cuda.stream(dn):
                hout[t0:t1].copy_(self.out[t0:t1], non_blocking=True)
        st["free"] = torch.cuda.Event()
        st["free"].record(cs)  # the combine was this staging set's last reader
        done = torch.cuda.Event()
        done.record(dn)
        self._out_free = done
        if wait:
            cs.wait_event(done)
        return done

    def forward_streamed(self, host_arena, x, ids, w, ring_groups=3, stream=None):
        """As forward, with the expert records read from host_arena (pinned host
        memory, record e at e*arena_stride) and streamed through a device ring of
        ring_groups x 16 slots on a copy stream of the layer's own."""
        dev = self.group_buf.device
        if getattr(self, "_ring_groups", None) != ring_groups:
            self.ring = torch.zeros(ring_groups * 16 * self.slot_stride, dtype=torch.uint8,
                                    device=dev)
            self._ring_groups = ring_groups
        if not hasattr(self, "stage_buf"):
            self.stage_buf = torch.zeros(16 * self.slot_stride, dtype=torch.uint8, device=dev)
            self.group_counts = torch.zeros((self.E + 15) // 16, dtype=torch.int32, device=dev)
            n_scratch = 2 * self.E + 2 + (self.E + 15) // 16
            self.host_scratch = torch.zeros(n_scratch, dtype=torch.int32).pin_memory()
            self.copy_stream = torch.cuda.Stream(device=dev)
        b = StreamBuffers()
        for name, t in (("ring", self.ring), ("group_buf", self.stage_buf),
                        ("group_counts", self.group_counts), ("offsets", self.offsets),
                        ("slot", self.slot), ("src", self.src), ("active", self.active),
                        ("n_active", self.n_active), ("q", self.q), ("ds", self.ds),
                        ("h", self.h), ("hq", self.hq), ("hds", self.hds), ("y", self.y),
                        ("ws", self.ws), ("host_scratch", self.host_scratch)):
            setattr(b, name, t.data_ptr())
        b.ws_bytes = self.ws.numel()
        cs = stream if stream is not None else torch.cuda.current_stream(dev)
        self._out_writable(cs)
        moe_layer_forward_streamed(self.wtype, x, ids, w, self.out, host_arena, self.rec_bytes,
                                   self.arena_stride, self.slot_stride, ring_groups, b, self.E,
                                   self.f, cs, self.copy_stream)
        return self.out[:x.shape[0]]
