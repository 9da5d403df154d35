"""GPU: the layer with the expert records in pinned host memory, streamed through
the device staging ring (moe_layer_forward_streamed), against the resident layer.

The streamed walk runs the same kernels on the same bytes, group by group, so
its output must equal the resident layer's bit for bit; the ring sizes below
force slot reuse (a ring of one to three groups for up to 32 groups of experts),
which exercises the copy stream's waits on the events that release ring slots.
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


def _layer(wl):
    cfg = wl.cfg
    return m.MoeLayer(cfg.wtype, cfg.E, cfg.d, cfg.f, cfg.K, cfg.T, H.to_dev(wl.arena),
                      wl.rec_bytes, wl.arena_stride)


@pytest.mark.parametrize("name,ring_groups", [(mw.TINY.name, 1), (mw.T600.name, 1),
                                              (mw.T600.name, 3), (mw.T2048.name, 2),
                                              (mw.T2048_Q2K.name, 2)])
def test_streamed_equals_resident(name, ring_groups):
    wl = H.workload(name)
    layer = _layer(wl)
    x, ids, w = H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w)
    ref = layer.forward(x, ids, w).clone()
    assert m.moe_device_error(layer.ws) == 0
    host_arena = torch.from_numpy(wl.arena).pin_memory()
    layer.out.fill_(float("nan"))
    layer.y.fill_(float("nan"))
    got = layer.forward_streamed(host_arena, x, ids, w, ring_groups=ring_groups)
    torch.cuda.synchronize()
    assert m.moe_device_error(layer.ws) == 0
    assert torch.equal(got, ref)
    # and again, reusing the events and the ring
    got2 = layer.forward_streamed(host_arena, x, ids, w, ring_groups=ring_groups).clone()
    torch.cuda.synchronize()
    assert torch.equal(got2, ref)


def test_streamed_rejects_bad_arguments():
    wl = H.workload(mw.TINY.name)
    layer = _layer(wl)
    x, ids, w = H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w)
    with pytest.raises(ValueError):  # a device tensor is not a host arena
        layer.forward_streamed(layer.arena, x, ids, w)
    host_arena = torch.from_numpy(wl.arena).pin_memory()
    with pytest.raises(m.MoeError):
        layer.forward_streamed(host_arena, x, ids, w, ring_groups=0)
    with pytest.raises(m.MoeError):
        layer.forward_streamed(host_arena, x, ids, w, ring_groups=65)
    assert np.isfinite(layer.forward_streamed(host_arena, x, ids, w).cpu().numpy()).all()


@pytest.mark.parametrize("name,chunks", [(mw.TINY.name, 4), (mw.T600.name, 1), (mw.T600.name, 3),
                                         (mw.T2048_Q2K.name, 4), (mw.T8192.name, 4)])
def test_forward_host_equals_forward(name, chunks):
    """MoeLayer.forward_host (pinned host in, pinned host out, copies overlapped
    with the layer on a copy stream, stage 2 and stage 7 per token slice) gives
    the same bytes as forward on device inputs, twice in a row."""
    wl = H.workload(name)
    layer = _layer(wl)
    ref = layer.forward(H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w)).cpu().numpy()
    assert m.moe_device_error(layer.ws) == 0
    hx = torch.from_numpy(wl.x).pin_memory()
    hids = torch.from_numpy(wl.ids).pin_memory()
    hw = torch.from_numpy(wl.w).pin_memory()
    for _ in range(2):
        hout = torch.full((wl.cfg.T, wl.cfg.d), float("nan")).pin_memory()
        layer.out.fill_(float("nan"))
        layer.forward_host(hx, hids, hw, hout, chunks=chunks)
        torch.cuda.current_stream().synchronize()
        assert m.moe_device_error(layer.ws) == 0
        assert np.array_equal(hout.numpy(), ref)


@pytest.mark.parametrize("name", [mw.T600.name, mw.T8192.name])
def test_forward_host_back_to_back(name):
    """Three forward_host calls on different inputs queued back to back without
    waiting (wait=False): the double-buffered staging and the output buffer are
    reused across calls whose copies overlap one another's layers, and every
    call must still give forward's bytes for its own inputs."""
    wl = H.workload(name)
    cfg = wl.cfg
    layer = _layer(wl)
    rev = np.ascontiguousarray
    inputs = [(wl.x, wl.ids, wl.w),
              (rev(wl.x[::-1]), rev(wl.ids[::-1]), rev(wl.w[::-1])),
              ((wl.x * np.float32(0.5)).astype(np.float32), rev(np.roll(wl.ids, 1, axis=1)),
               wl.w)]
    refs = []
    for x, ids, w in inputs:
        refs.append(layer.forward(H.to_dev(x), H.to_dev(ids), H.to_dev(w)).cpu().numpy())
        assert m.moe_device_error(layer.ws) == 0
    assert not np.array_equal(refs[0], refs[1]) and not np.array_equal(refs[0], refs[2])
    host = [tuple(torch.from_numpy(a).pin_memory() for a in inp) for inp in inputs]
    outs = [torch.full((cfg.T, cfg.d), float("nan")).pin_memory() for _ in inputs]
    dev_in = [tuple(H.to_dev(a) for a in inp) for inp in inputs]
    for _ in range(2):
        for o in outs:
            o.fill_(float("nan"))
        events = [layer.forward_host(hx, hids, hw, o, wait=False)
                  for (hx, hids, hw), o in zip(host, outs)]
        # a device-input call queued at once rewrites the output buffer only
        # after the last copy back has read it
        last = layer.forward(*dev_in[0])
        for ev, o, ref in zip(events, outs, refs):
            ev.synchronize()
            assert np.array_equal(o.numpy(), ref)
        assert np.array_equal(last.cpu().numpy(), refs[0])
        torch.cuda.current_stream().synchronize()
        assert m.moe_device_error(layer.ws) == 0
