"""GPU: the two fused calls against the seven-call layer.

moe_grouped_mmq_gateup_q8_1 must write the same q8_1 hidden bytes as the
gate/up product followed by the stand-alone re-quantization, and
moe_grouped_mmq_down_combine the same y rows and the same combined output as
the down product followed by the stand-alone combine, bit for bit: the fused
epilogues run the same arithmetic on the same kernel (by default the
per-block-scaling kernel for gate/up and the folded-scale kernel for down; with
MOE_MMQ_PATH=blockscale the per-block-scaling kernel for both), and the
combine's fixed k order does not depend on which work item finishes a token
last.

Both fused calls are also checked against the oracle itself: the fused layer's
output (the combine written by moe_grouped_mmq_down_combine) within 2e-3
relative L2 per token on every workload, all-zero tokens exactly zero, and the
down + combine call alone on the oracle's own hidden rows.
"""
import os

import numpy as np
import pytest

import moe_workloads as mw
import oracle
from tests import helpers as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import quantized_routed_expert_q8_gb300 as m  # noqa: E402


PATHS = [None, "blockscale"]


class _path:
    """MOE_MMQ_PATH set to path (None: unset) inside the block, restored after."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.old = os.environ.get("MOE_MMQ_PATH")
        if self.path is None:
            os.environ.pop("MOE_MMQ_PATH", None)
        else:
            os.environ["MOE_MMQ_PATH"] = self.path

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop("MOE_MMQ_PATH", None)
        else:
            os.environ["MOE_MMQ_PATH"] = self.old


def _both(layer, x, ids, w, path=None):
    """(unfused, fused) copies of hq, hds, y and out for one input, both with
    MOE_MMQ_PATH=path (None: the default kernels)."""
    res = []
    for fused in (False, True):
        for t in (layer.hq, layer.hds, layer.y, layer.out):
            t.zero_()
        with _path(path):
            out = layer.forward(x, ids, w, fused=fused)
            torch.cuda.synchronize()
        res.append({"hq": layer.hq.clone(), "hds": layer.hds.clone(), "y": layer.y.clone(),
                    "out": out.clone(), "err": m.moe_device_error(layer.ws)})
    return res


def _assert_same(a, b):
    for k in ("hq", "hds", "y", "out"):
        assert torch.equal(a[k], b[k]), k
    assert a["err"] == b["err"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", [mw.TINY.name, mw.T600.name, mw.T2048.name, mw.T2048_Q2.name,
                                  mw.T2048_Q2K.name, mw.T8192.name])
def test_fused_equals_seven_calls(name, path):
    wl = H.workload(name)
    cfg = wl.cfg
    layer = m.MoeLayer(cfg.wtype, cfg.E, cfg.d, cfg.f, cfg.K, cfg.T, H.to_dev(wl.arena),
                       wl.rec_bytes, wl.arena_stride)
    a, b = _both(layer, H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w), path)
    assert a["err"] == 0
    _assert_same(a, b)
    # again: the arrival counters are set afresh by every call
    with _path(path):
        out2 = layer.forward(H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w), fused=True).clone()
        torch.cuda.synchronize()
    assert torch.equal(out2, a["out"])


def _small(wtype, T, ids, seed, E=10, d=256, f=128):
    arena, rb, stride = mw.expert_arena(wtype, E, d, f, seed)
    x = mw.normal_f32(seed, 1, T * d).reshape(T, d)
    w = mw.normal_f32(seed, 2, ids.size).reshape(ids.shape).astype(np.float32)
    layer = m.MoeLayer(wtype, E, d, f, ids.shape[1], T, H.to_dev(arena), rb, stride)
    return layer, H.to_dev(x), H.to_dev(np.ascontiguousarray(ids, np.int32)), H.to_dev(w)


@pytest.mark.parametrize("path", PATHS)
def test_fused_ragged_expert_sizes(path):
    """Experts with 1 .. 257 rows: partial 16-row tiles and 128-token items."""
    sizes = [1, 15, 16, 17, 127, 128, 129, 257]
    ids = np.concatenate([np.full(n, e + 1, np.int32) for e, n in enumerate(sizes)])
    ids = np.random.default_rng(5).permutation(ids).reshape(-1, 1)
    layer, x, idd, w = _small(mw.Q8_0, ids.shape[0], ids, 31)
    a, b = _both(layer, x, idd, w, path)
    assert a["err"] == 0
    _assert_same(a, b)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("wtype", [mw.Q8_0, mw.Q4_1, mw.Q2_0])
def test_fused_dropped_ids(wtype, path):
    """Some of a token's ids are out of range (fewer rows to combine) and some
    tokens have none (a zero output row, whatever the buffer held)."""
    T, K, E = 300, 4, 10
    rng = np.random.default_rng(7)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < 0.2] = E + 3
    ids[::37] = -1
    layer, x, idd, w = _small(wtype, T, ids, 32, E=E)
    a, b = _both(layer, x, idd, w, path)
    assert a["err"] & m.DEV_ERR_BAD_EXPERT_ID
    _assert_same(a, b)
    assert not b["out"][::37].any()
    layer.out.fill_(float("nan"))
    with _path(path):
        out = layer.forward(x, idd, w, fused=True)
        torch.cuda.synchronize()
    assert torch.equal(out, b["out"])


def test_fused_no_routed_expert():
    T, K = 5, 2
    ids = np.full((T, K), 10, np.int32)
    layer, x, idd, w = _small(mw.Q8_0, T, ids, 33)
    layer.out.fill_(float("nan"))
    out = layer.forward(x, idd, w, fused=True)
    torch.cuda.synchronize()
    assert not out.any()
    assert m.moe_device_error(layer.ws) & m.DEV_ERR_BAD_EXPERT_ID


def test_fused_rejects_what_it_cannot_take():
    # d = 288 is no whole tensor-core tile: the fused calls refuse, the seven run
    T, K = 8, 2
    ids = np.tile(np.arange(K, dtype=np.int32), (T, 1))
    layer, x, idd, w = _small(mw.Q8_0, T, ids, 34, E=4, d=288, f=96)
    layer.forward(x, idd, w)
    with pytest.raises(m.MoeError):
        layer.forward(x, idd, w, fused=True)
    # R must be T*K for the combine
    ids = np.tile(np.arange(K, dtype=np.int32), (T, 1))
    layer, x, idd, w = _small(mw.Q8_0, T, ids, 35, E=4)
    layer.forward(x, idd, w)
    with pytest.raises(m.MoeError):
        m.moe_grouped_mmq_down_combine(layer.wtype, layer.group_buf, layer.slot_stride,
                                       layer.active, layer.n_active, layer.offsets, layer.E,
                                       layer.hq, layer.hds, T * K - 1, layer.d, layer.f,
                                       layer.src, layer.slot, w, T, K, layer.y, layer.out,
                                       layer.ws)


@pytest.mark.parametrize("name", [c.name for c in mw.CONFIG_LIST])
def test_fused_layer_matches_oracle(name):
    """MoeLayer.forward(fused=True) -- gate/up writing q8_1 hidden rows, then
    down with the in-kernel combine -- against the oracle's layer: <= 2e-3
    relative L2 per token (the tolerance of the layer output), zero tokens
    exactly zero."""
    wl = H.workload(name)
    cfg = wl.cfg
    layer = m.MoeLayer(cfg.wtype, cfg.E, cfg.d, cfg.f, cfg.K, cfg.T, H.to_dev(wl.arena),
                       wl.rec_bytes, wl.arena_stride)
    layer.out.fill_(float("nan"))
    out = layer.forward(H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w), fused=True)
    out = out.cpu().numpy()
    assert m.moe_device_error(layer.ws) == 0
    assert np.isfinite(out).all()
    err = H.rel_l2_rows(out, H.oracle_layer_all(wl))
    assert err.max() <= 2e-3, (err.max(), int(np.argmax(err)))
    for t in cfg.zero_list():
        assert not out[t].any()


@pytest.mark.parametrize("name", [mw.TINY.name, mw.T600.name, mw.T2048.name, mw.T2048_Q2.name,
                                  mw.T2048_Q2K.name])
def test_down_combine_matches_oracle(name):
    """moe_grouped_mmq_down_combine alone, on hidden rows quantized by the
    oracle: its combined output against the oracle's down product followed by
    the oracle's combine, within 5e-5 relative L2 per token (the stage-level
    bar of the folded-scale down product, which the call runs by default; the
    combine adds K fp32 roundings)."""
    wl = H.workload(name)
    cfg = wl.cfg
    T, K, d, f = cfg.T, cfg.K, cfg.d, cfg.f
    o = oracle.build_slot_map(wl.ids, cfg.E)
    R = int(o["offsets"][cfg.E])
    assert R == T * K
    hid = mw.normal_f32(cfg.seed, 9, R * f, scale=0.05).reshape(R, f)
    hid[::53] = 0.0
    hq, hds = oracle.requant_hidden_q8_1(hid, layout=oracle.layout_of(cfg.wtype))
    layer = m.MoeLayer(cfg.wtype, cfg.E, d, f, K, T, H.to_dev(wl.arena), wl.rec_bytes,
                       wl.arena_stride)
    layer.forward(H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w))  # slot map, group buffers
    w = H.to_dev(wl.w)
    layer.out.fill_(float("nan"))
    m.moe_grouped_mmq_down_combine(layer.wtype, layer.group_buf, layer.slot_stride, layer.active,
                                   layer.n_active, layer.offsets, layer.E, H.to_dev(hq),
                                   H.to_dev(hds.view(np.int16)), R, d, f, layer.src, layer.slot, w,
                                   T, K, layer.y, layer.out, layer.ws)
    out = layer.out[:T].cpu().numpy()
    assert m.moe_device_error(layer.ws) == 0
    toks = H.layer_tokens(cfg)
    rows = o["slot"].reshape(T, K)[toks].reshape(-1)
    y_rows = H.oracle_rows("down", wl, o["offsets"], hq, hds, rows)
    n = len(toks)  # the oracle's combine on the selected tokens' rows, renumbered
    ref = oracle.combine_topk(y_rows, np.arange(n * K, dtype=np.int32), wl.w[toks], n, K, d)
    err = H.rel_l2_rows(out[toks], ref)
    assert err.max() <= 5e-5, (err.max(), toks[np.argmax(err)])
