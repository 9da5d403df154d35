"""GPU edge cases of the whole layer against the CPU oracle: no routed expert at
all, a single token with a single expert, expert row counts straddling the
16-row token tiles and the 128-token items (ragged tails), and a shape the
tensor-core kernel does not take (so the CUDA-core MMQ runs inside the layer)."""
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


def _problem(wtype, T, d, f, E, K, seed, ids=None):
    arena, rb, stride = mw.expert_arena(wtype, E, d, f, seed)
    x = mw.normal_f32(seed, 1, T * d).reshape(T, d)
    if ids is None:
        ids, w = mw.topk_softmax(mw.normal_f32(seed, 2, T * E).reshape(T, E), K)
    else:
        w = np.full(ids.shape, 1.0 / ids.shape[1], np.float32)
    return arena, rb, stride, x, np.ascontiguousarray(ids, np.int32), np.ascontiguousarray(w)


def _run(wtype, E, d, f, arena, rb, stride, x, ids, w, streamed=False):
    T, K = ids.shape
    layer = m.MoeLayer(wtype, E, d, f, K, T, H.to_dev(arena), rb, stride)
    xd, idd, wd = H.to_dev(x), H.to_dev(ids), H.to_dev(w)
    if streamed:
        out = layer.forward_streamed(torch.from_numpy(arena).pin_memory(), xd, idd, wd)
    else:
        out = layer.forward(xd, idd, wd)
    out = out.cpu().numpy()
    return out, m.moe_device_error(layer.ws)


def _oracle(wtype, E, d, f, arena, rb, stride, x, ids, w):
    return oracle.layer_forward(wtype, arena, rb, stride, x, ids, w, E, d, f)["out"]


@pytest.mark.parametrize("streamed", [False, True])
def test_no_routed_expert(streamed):
    """Every id out of range: no expert is active, every output row is zero and
    the device error word reports the dropped ids."""
    E, d, f, T, K = 16, 256, 128, 5, 2
    arena, rb, stride, x, _, w = _problem(mw.Q8_0, T, d, f, E, K, 21)
    ids = np.full((T, K), E, np.int32)
    out, bits = _run(mw.Q8_0, E, d, f, arena, rb, stride, x, ids, w, streamed)
    assert not out.any()
    assert bits & m.DEV_ERR_BAD_EXPERT_ID


@pytest.mark.parametrize("wtype", [mw.Q8_0, mw.Q4_1, mw.Q2_0, mw.Q2_K])
def test_single_token_single_expert(wtype):
    E, d, f = 4, 256, 256 if wtype == mw.Q2_K else 128
    arena, rb, stride, x, _, _ = _problem(wtype, 1, d, f, E, 1, 22)
    ids = np.array([[3]], np.int32)
    w = np.array([[1.0]], np.float32)
    out, bits = _run(wtype, E, d, f, arena, rb, stride, x, ids, w)
    assert bits == 0
    ref = _oracle(wtype, E, d, f, arena, rb, stride, x, ids, w)
    assert H.rel_l2_rows(out, ref).max() <= 2e-3


@pytest.mark.parametrize("streamed", [False, True])
def test_ragged_expert_sizes(streamed):
    """Experts with 1, 15, 16, 17, 127, 128, 129 and 257 rows (K = 1): partial
    16-row tiles and partial 128-token items next to full ones."""
    sizes = [1, 15, 16, 17, 127, 128, 129, 257]
    E, d, f = len(sizes) + 2, 256, 128
    ids = np.concatenate([np.full(n, e + 1, np.int32) for e, n in enumerate(sizes)])
    ids = np.random.default_rng(3).permutation(ids).reshape(-1, 1)
    T = ids.shape[0]
    arena, rb, stride, x, _, w = _problem(mw.Q8_0, T, d, f, E, 1, 23, ids=ids)
    out, bits = _run(mw.Q8_0, E, d, f, arena, rb, stride, x, ids, w, streamed)
    assert bits == 0
    ref = _oracle(mw.Q8_0, E, d, f, arena, rb, stride, x, ids, w)
    assert H.rel_l2_rows(out, ref).max() <= 2e-3


@pytest.mark.parametrize("path", [None, "simt"])
def test_ragged_expert_sizes_q2_k(path, monkeypatch):
    """Q2_K (D2S6 activations) on experts with 1 .. 257 rows, K = 2, three
    super-blocks of d and two of f, on the tensor cores and on the CUDA cores."""
    if path:
        monkeypatch.setenv("MOE_MMQ_PATH", path)
    sizes = [1, 15, 16, 17, 127, 128, 129, 257]
    E, d, f = len(sizes) + 2, 768, 512
    ids = np.concatenate([np.full(n, e + 1, np.int32) for e, n in enumerate(sizes)])
    ids = np.random.default_rng(4).permutation(ids)
    ids = ids[: ids.size // 2 * 2].reshape(-1, 2)
    T = ids.shape[0]
    arena, rb, stride, x, _, w = _problem(mw.Q2_K, T, d, f, E, 2, 25, ids=ids)
    x[5] = 0.0
    out, bits = _run(mw.Q2_K, E, d, f, arena, rb, stride, x, ids, w)
    assert bits == 0
    ref = _oracle(mw.Q2_K, E, d, f, arena, rb, stride, x, ids, w)
    assert H.rel_l2_rows(out, ref).max() <= 2e-3
    assert not out[5].any()


@pytest.mark.parametrize("wtype", [mw.Q8_0, mw.Q4_1, mw.Q2_0])
def test_shape_outside_the_tensor_core_kernel(wtype):
    """d = 288 and f = 96 are not whole tensor-core tiles: the CUDA-core MMQ runs."""
    E, d, f, T, K = 6, 288, 96, 40, 2
    arena, rb, stride, x, ids, w = _problem(wtype, T, d, f, E, K, 24)
    out, bits = _run(wtype, E, d, f, arena, rb, stride, x, ids, w)
    assert bits == 0
    ref = _oracle(wtype, E, d, f, arena, rb, stride, x, ids, w)
    assert H.rel_l2_rows(out, ref).max() <= 2e-3


@pytest.mark.parametrize("wtype,path", [(mw.Q8_0, None), (mw.Q8_0, "simt"), (mw.Q2_K, None)])
def test_maximum_expert_count(wtype, path, monkeypatch):
    """E = 8192, the largest expert count the calls accept, with K = 16 routed
    experts a token: most experts get one or two rows, so every group of 16 and
    every work item is ragged; every token against the oracle, fused and
    streamed forms included where the tensor-core kernel runs."""
    if path:
        monkeypatch.setenv("MOE_MMQ_PATH", path)
    E, K, T = 8192, 16, 400
    d, f = 256, 256 if wtype == mw.Q2_K else 128
    arena, rb, stride, x, ids, w = _problem(wtype, T, d, f, E, K, 31)
    x[17] = 0.0
    out, bits = _run(wtype, E, d, f, arena, rb, stride, x, ids, w)
    assert bits == 0
    ref = _oracle(wtype, E, d, f, arena, rb, stride, x, ids, w)
    assert H.rel_l2_rows(out, ref).max() <= 2e-3
    assert not out[17].any()
    if path is None:
        layer = m.MoeLayer(wtype, E, d, f, K, T, H.to_dev(arena), rb, stride)
        xd, idd, wd = H.to_dev(x), H.to_dev(ids), H.to_dev(w)
        fused = layer.forward(xd, idd, wd, fused=True).cpu().numpy()
        assert m.moe_device_error(layer.ws) == 0
        assert H.rel_l2_rows(fused, ref).max() <= 2e-3
        streamed, _ = _run(wtype, E, d, f, arena, rb, stride, x, ids, w, streamed=True)
        assert np.array_equal(streamed, out)


def test_bounded_wait_reports_timeout(monkeypatch):
    """Failure detection without a fault: MOE_TEST_STALL_BLOCK makes CTA 0 of
    the per-block-scaling MMQ (stage 4) withhold one partials commit and CTA 0 of
    the folded-scale MMQ (stage 6) one operand-release commit, so a bounded wait
    runs out (about 2 s); the kernel sets MOE_DEV_ERR_TIMEOUT, every role exits,
    and the context stays usable: the next calls are exact again."""
    wl = H.workload(mw.TINY.name)
    cfg = wl.cfg
    layer = m.MoeLayer(cfg.wtype, cfg.E, cfg.d, cfg.f, cfg.K, cfg.T, H.to_dev(wl.arena),
                       wl.rec_bytes, wl.arena_stride)
    x, ids, w = H.to_dev(wl.x), H.to_dev(wl.ids), H.to_dev(wl.w)
    ref = layer.forward(x, ids, w).cpu().numpy()
    assert m.moe_device_error(layer.ws) == 0
    R = cfg.T * cfg.K

    def gateup():
        m.moe_grouped_mmq_gateup(layer.wtype, layer.group_buf, layer.slot_stride, layer.active,
                                 layer.n_active, layer.offsets, cfg.E, layer.q, layer.ds, R, cfg.d,
                                 cfg.f, layer.h, layer.ws)

    def down():  # the folded-scale kernel: an operand-release commit withheld
        m.moe_grouped_mmq_down(layer.wtype, layer.group_buf, layer.slot_stride, layer.active,
                               layer.n_active, layer.offsets, cfg.E, layer.hq, layer.hds, R, cfg.d,
                               cfg.f, layer.y, layer.ws)

    for call in (gateup, down):
        monkeypatch.setenv("MOE_TEST_STALL_BLOCK", "0")
        call()
        bits = m.moe_device_error(layer.ws)
        assert bits & m.DEV_ERR_TIMEOUT, call.__name__
        monkeypatch.delenv("MOE_TEST_STALL_BLOCK")
        call()
        assert m.moe_device_error(layer.ws) == 0
    out = layer.forward(x, ids, w).cpu().numpy()
    assert m.moe_device_error(layer.ws) == 0
    assert np.array_equal(out, ref)
