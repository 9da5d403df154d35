"""The workspace-free routing-map call (moe_build_slot_map_noalloc), for callers
that cannot allocate device memory: through the C ABI it must give the same
offsets, slot, src and active list as moe_build_slot_map with a workspace, on
two calls in a row (the second reuses the library's fixed scratch array), and
it must refuse sizes that do not fit that array before launching anything.

This file is collected last so that a failure here stops a -x run only after
every other test has run."""
import ctypes

import numpy as np
import pytest

import moe_workloads as mw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import quantized_routed_expert_q8_gb300 as m  # noqa: E402


def _outputs(T, K, E):
    i32 = dict(dtype=torch.int32, device="cuda")
    R = max(T * K, 1)
    return dict(offsets=torch.full((E + 1,), -9, **i32), slot=torch.full((R,), -9, **i32),
                src=torch.full((R,), -9, **i32), active=torch.full((E,), -9, **i32),
                n_active=torch.full((1,), -9, **i32))


def _with_workspace(ids, E):
    T, K = ids.shape
    o = _outputs(T, K, E)
    n = m.moe_workspace_size(T, K, E, 64, 64)
    ws = torch.zeros((n + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(ws)
    m.moe_build_slot_map(ids, E, o["offsets"], o["slot"], o["src"], o["active"], o["n_active"], ws)
    return o


def _without_workspace(ids, E):
    T, K = ids.shape
    o = _outputs(T, K, E)
    m.moe_build_slot_map_noalloc(ids, E, o["offsets"], o["slot"], o["src"], o["active"],
                                 o["n_active"])
    return o


def _same(a, b, R):
    for k in ("offsets", "active", "n_active"):
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(a["slot"][:R], b["slot"][:R])
    assert torch.equal(a["src"][:R], b["src"][:R])


def test_noalloc_matches_workspace_form_twice():
    cases = []
    wl = mw.make_workload(mw.TINY)
    cases.append((wl.ids, mw.TINY.E))
    rng = np.random.default_rng(17)
    E = 512
    logits = rng.normal(size=(3000, E)).astype(np.float32)
    ids, _ = mw.topk_softmax(logits, 10)
    cases.append((ids, E))
    for ids_h, E in cases:  # two calls in a row, different sizes
        ids = torch.from_numpy(ids_h).cuda()
        T, K = ids.shape
        a = _without_workspace(ids, E)
        b = _with_workspace(ids, E)
        torch.cuda.synchronize()
        _same(a, b, T * K)
    # and once more on the first input, after the larger call left its counts behind
    ids = torch.from_numpy(cases[0][0]).cuda()
    _same(_without_workspace(ids, cases[0][1]), _with_workspace(ids, cases[0][1]), ids.numel())


def test_noalloc_rejects_sizes_beyond_its_array():
    L = m.lib()
    P = ctypes.c_void_p
    # 600 chunks of 1024 entries x 512 experts exceed the 1 MiB count table.  The
    # buffers are real allocations of the declared shape, so a size check that
    # stopped rejecting would not launch on made-up addresses.
    T, K, E = 61440, 10, 512
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    o = _outputs(T, K, E)
    rc = L.moe_build_slot_map_noalloc(P(ids.data_ptr()), T, K, E, P(o["offsets"].data_ptr()),
                                      P(o["slot"].data_ptr()), P(o["src"].data_ptr()),
                                      P(o["active"].data_ptr()), P(o["n_active"].data_ptr()), None)
    assert rc == -4  # MOE_ERR_UNSUPPORTED, before any launch
    torch.cuda.synchronize()
    assert int(o["n_active"].item()) == -9  # nothing was written
