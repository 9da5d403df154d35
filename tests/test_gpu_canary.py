"""GPU: guard canaries around every device buffer the layer writes.

Each buffer of the layer (routing maps, q8_1 rows, group buffers, h, y, out,
the workspace, the streamed walk's ring) is replaced by a view into a larger
allocation filled with 0xA5, with 4 KB of guard bytes before and after it.
After the seven calls, the fused calls and the streamed walk, every guard byte
must still be 0xA5 (no kernel wrote outside its buffer), and the outputs must
equal those of a layer with zero-initialized buffers (no output depends on
what a buffer held before the call).
"""
import numpy as np
import pytest

import moe_workloads as mw
from tests import helpers as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import quantized_routed_expert_q8_gb300 as m  # noqa: E402

GUARD = 4096
CANARY = 0xA5
BUFFERS = ("offsets", "slot", "src", "active", "n_active", "q", "ds", "group_buf", "h", "hq",
           "hds", "y", "out", "ws")


class Guarded:
    def __init__(self):
        self.raw = []  # (name, raw uint8 tensor, payload bytes)

    def view(self, name, like):
        n = like.numel() * like.element_size()
        raw = torch.full((GUARD + (n + 255) // 256 * 256 + GUARD,), CANARY, dtype=torch.uint8,
                         device=like.device)
        self.raw.append((name, raw, n))
        return raw[GUARD:GUARD + n].view(like.dtype).view(like.shape)

    def check(self):
        for name, raw, n in self.raw:
            head, tail = raw[:GUARD], raw[GUARD + n:]
            assert bool((head == CANARY).all()), f"{name}: write before the buffer"
            assert bool((tail == CANARY).all()), f"{name}: write past the buffer"


def _guard_layer(layer, g, streamed_ring_groups=None):
    for name in BUFFERS:
        setattr(layer, name, g.view(name, getattr(layer, name)))
    m.moe_workspace_init(layer.ws)
    if streamed_ring_groups:
        dev = layer.group_buf.device
        ring = torch.empty(streamed_ring_groups * 16 * layer.slot_stride, dtype=torch.uint8,
                           device=dev)
        layer.ring = g.view("ring", ring)
        layer._ring_groups = streamed_ring_groups
        layer.stage_buf = g.view("stage_buf", torch.empty(16 * layer.slot_stride,
                                                          dtype=torch.uint8, device=dev))
        layer.group_counts = g.view("group_counts", torch.empty((layer.E + 15) // 16,
                                                                dtype=torch.int32, device=dev))
        n_scratch = 2 * layer.E + 2 + (layer.E + 15) // 16
        layer.host_scratch = torch.zeros(n_scratch, dtype=torch.int32).pin_memory()
        layer.copy_stream = torch.cuda.Stream(device=dev)


def _layer(wtype, E, d, f, K, T, arena, rb, stride):
    return m.MoeLayer(wtype, E, d, f, K, T, H.to_dev(arena), rb, stride)


def _run_all(layer, x, ids, w, arena, fused, streamed):
    out = layer.forward(x, ids, w).clone()
    torch.cuda.synchronize()
    # y rows past offsets[E] belong to no expert (dropped ids) and are never written
    n_rows = int(layer.offsets[layer.E].item())
    res = {"out": out, "y": layer.y[:n_rows].clone()}
    if fused:
        res["out_fused"] = layer.forward(x, ids, w, fused=True).clone()
    if streamed:
        res["out_streamed"] = layer.forward_streamed(torch.from_numpy(arena).pin_memory(), x, ids,
                                                     w, ring_groups=1).clone()
    torch.cuda.synchronize()
    res["err"] = m.moe_device_error(layer.ws)
    return res


def _case(wtype, T, K, E, d, f, seed, ids=None, fused=True, streamed=True, wl=None):
    if wl is not None:
        arena, rb, stride = wl.arena, wl.rec_bytes, wl.arena_stride
        x, ids_np, w_np = H.to_dev(wl.x), wl.ids, wl.w
    else:
        arena, rb, stride = mw.expert_arena(wtype, E, d, f, seed)
        x = H.to_dev(mw.normal_f32(seed, 1, T * d).reshape(T, d))
        if ids is None:
            ids_np, w_np = mw.topk_softmax(mw.normal_f32(seed, 2, T * E).reshape(T, E), K)
        else:
            ids_np = ids
            w_np = np.full(ids.shape, 1.0 / ids.shape[1], np.float32)
    ids_d, w_d = H.to_dev(np.ascontiguousarray(ids_np, np.int32)), H.to_dev(np.ascontiguousarray(w_np))
    plain = _layer(wtype, E, d, f, K, T, arena, rb, stride)
    ref = _run_all(plain, x, ids_d, w_d, arena, fused, streamed)
    g = Guarded()
    guarded = _layer(wtype, E, d, f, K, T, arena, rb, stride)
    _guard_layer(guarded, g, 1 if streamed else None)
    got = _run_all(guarded, x, ids_d, w_d, arena, fused, streamed)
    g.check()
    for k in ref:
        if k == "err":
            assert got[k] == ref[k]
        else:
            assert torch.equal(got[k], ref[k]), k


def test_canary_tiny_all_paths():
    _case(mw.Q8_0, 7, 2, 16, 256, 128, 41)


@pytest.mark.parametrize("wtype", [mw.Q4_1, mw.Q2_0, mw.Q2_K])
def test_canary_other_formats(wtype):
    _case(wtype, 300, 4, 40, 256, 256 if wtype == mw.Q2_K else 128, 42)


def test_canary_ragged_and_dropped():
    sizes = [1, 15, 16, 17, 127, 128, 129, 257]
    ids = np.concatenate([np.full(n, e + 1, np.int32) for e, n in enumerate(sizes)])
    ids = np.random.default_rng(9).permutation(ids)
    ids[::29] = 99  # out of range: dropped rows
    _case(mw.Q8_0, ids.size, 1, len(sizes) + 2, 256, 128, 43, ids=ids.reshape(-1, 1))


def test_canary_cuda_core_shape():
    # d = 288, f = 96: the CUDA-core MMQ (the fused calls do not take it)
    _case(mw.Q8_0, 40, 2, 6, 288, 96, 44, fused=False, streamed=True)


def test_canary_many_experts():
    # the 600-token workload: 512 experts of ~12 rows, d = 2048, f = 768
    wl = H.workload(mw.T600.name)
    c = wl.cfg
    _case(c.wtype, c.T, c.K, c.E, c.d, c.f, 0, wl=wl, streamed=False)
