"""Host-side checks of the C ABI (no GPU needed): the built library loads and
exports every function include/moe_q8.h declares, the binding covers them, and
size queries agree with the record layout of the oracle and the generator."""
import ctypes
import os
import re

import pytest

import moe_workloads as mw
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_q8.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from quantized_routed_expert_q8_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_header():
    import quantized_routed_expert_q8_gb300 as m
    assert sorted(m.EXPORTED) == _declared()
    for n in _declared():
        assert callable(getattr(m, n, None)) or n == "moe_status_string", n


@pytest.mark.parametrize("wtype", [0, 1])
def test_record_bytes_agree(lib, wtype):
    import quantized_routed_expert_q8_gb300 as m
    for d, f in ((256, 128), (2048, 768), (96, 64)):
        assert m.moe_expert_record_bytes(wtype, d, f) == oracle.expert_record_bytes(wtype, d, f)
        assert m.moe_expert_record_bytes(wtype, d, f) == mw.record_bytes(wtype, d, f)
        assert m.moe_expert_record_offsets(wtype, d, f) == oracle.record_offsets(wtype, d, f)
    assert m.moe_expert_record_bytes(wtype, 100, 64) == 0  # d not a multiple of 32


def test_record_bytes_agree_q2_k(lib):
    """Q2_K records (super-blocks of 256) agree across the library, the oracle
    and the generator; widths that are not whole super-blocks are refused."""
    import quantized_routed_expert_q8_gb300 as m
    for d, f in ((256, 256), (2048, 768), (512, 1280)):
        assert m.moe_expert_record_bytes(3, d, f) == oracle.expert_record_bytes(3, d, f)
        assert m.moe_expert_record_bytes(3, d, f) == mw.record_bytes(3, d, f)
        assert m.moe_expert_record_offsets(3, d, f) == oracle.record_offsets(3, d, f)
    assert m.moe_expert_record_bytes(3, 2048, 640) == 0  # f not a multiple of 256
    assert m.moe_expert_record_bytes(3, 96, 256) == 0
    assert m.ds_halves(3) == 4 and m.ds_halves(0) == 2


def test_status_strings(lib):
    import quantized_routed_expert_q8_gb300 as m
    L = m.lib()
    for rc in range(0, -7, -1):
        assert L.moe_status_string(rc)
    assert m.moe_workspace_size(8192, 10, 512, 2048, 768) > 0


class _Buffers:
    """Pointers for the rejection tests.  With a GPU present every pointer is a
    real device allocation of 1 MiB (offset by `off` bytes for the misaligned
    cases), so that a host check that stopped rejecting would launch on valid
    memory instead of a made-up address; without a GPU nothing can launch and
    plain aligned integers stand in."""

    def __init__(self):
        self.keep = []
        try:
            import torch
            self.cuda = torch.cuda.is_available()
        except ImportError:
            self.cuda = False

    def __call__(self, off=0):
        if not self.cuda:
            return ctypes.c_void_p(4096 * (len(self.keep) + 1) + off)
        import torch
        t = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
        self.keep.append(t)
        return ctypes.c_void_p(t.data_ptr() + off)


def test_host_checks_reject_before_launch(lib):
    """Host-visible misuse returns an error status before launching anything."""
    import quantized_routed_expert_q8_gb300 as m
    L = m.lib()
    B = _Buffers()

    def P(v):  # v = the alignment the old fake address had; v % 16 == 1 means misaligned
        return B(off=v % 16 if v % 16 else 0)
    # null stream is fine: nothing launches on these paths
    assert L.moe_group_gather(P(16), 16, 16, P(16), 17, 0, P(16), 16, None) == -1
    assert L.moe_group_gather(P(16), 16, 16, P(16), 2, 15, P(16), 16, None) == -1
    assert L.moe_quantize_scatter_q8_1(P(16), 4, 100, 2, P(16), 8, P(16), P(16), None) == -1
    assert L.moe_quantize_scatter_q8_1(P(17), 4, 64, 2, P(16), 8, P(16), P(16), None) == -2
    assert L.moe_build_slot_map(P(16), 4, 2, 8, P(16), P(16), P(16), P(16), P(16), None, 0,
                                None) == -3
    assert L.moe_build_slot_map(P(16), 4, 2, 0, P(16), P(16), P(16), P(16), P(16), P(256), 1 << 20,
                                None) == -1
    assert L.moe_grouped_mmq_gateup(0, P(128), 100, P(16), P(16), P(16), 4, P(16), P(16), 8, 64,
                                    64, P(16), P(256), 1 << 20, None) == -2
    assert L.moe_combine_topk(P(16), 8, P(16), P(16), 2, 2, 6, P(16), None) == -1
    # D2S6 rows: 8-byte (d, s, s_lo, s_hi) entries
    assert L.moe_quantize_scatter_q8_1_d2s6(P(16), 4, 64, 2, P(16), 8, P(16), P(4), None) == -2
    assert L.moe_requant_hidden_q8_1_d2s6(P(16), 4, 64, P(16), P(4), None) == -2
    assert L.moe_quantize_gather_q8_1_d2s6(P(16), 4, 64, P(16), 8, P(16), P(4), None) == -2
    # Q2_K reductions must be whole 256-weight super-blocks
    assert L.moe_grouped_mmq_down(3, P(128), 128, P(16), P(16), P(16), 4, P(16), P(16), 8, 256,
                                  128, P(16), P(256), 1 << 20, None) == -1


def test_fused_calls_reject_before_launch(lib):
    """The fused calls' host checks: R must be T*K, outputs must be present, and
    the workspace must include the combine's arrival counters."""
    import quantized_routed_expert_q8_gb300 as m
    L = m.lib()
    B = _Buffers()

    def P(v):  # misaligned by v % 16 bytes when v is not a multiple of 16
        return B(off=v % 16)
    T, K, E, d, f = 16, 2, 4, 256, 128
    R = T * K
    need = m.moe_workspace_size(T, K, E, d, f)
    core = m.moe_workspace_size(T, K, E, 0, f)
    assert need - core == (T * ((d + 255) // 256) * 4 + 255) // 256 * 256
    args = (0, P(128), 128, P(16), P(16), P(16), E, P(16), P(16))
    # R != T*K, K == 0
    assert L.moe_grouped_mmq_down_combine(*args, R - 1, d, f, P(16), P(16), P(16), T, K, P(16),
                                          P(16), P(256), need, None) == -1
    assert L.moe_grouped_mmq_down_combine(*args, 0, d, f, P(16), P(16), P(16), T, 0, P(16),
                                          P(16), P(256), need, None) == -1
    # no output, misaligned output
    assert L.moe_grouped_mmq_down_combine(*args, R, d, f, P(16), P(16), P(16), T, K, P(16),
                                          None, P(256), need, None) == -1
    assert L.moe_grouped_mmq_down_combine(*args, R, d, f, P(16), P(16), P(16), T, K, P(16),
                                          P(20), P(256), need, None) == -2
    # a workspace sized without the arrival counters
    assert L.moe_grouped_mmq_down_combine(*args, R, d, f, P(16), P(16), P(16), T, K, P(16),
                                          P(16), P(256), core, None) == -3
    # gate/up to q8_1 without its outputs, or with misaligned (d, s) pairs
    assert L.moe_grouped_mmq_gateup_q8_1(*args, R, d, f, None, P(16), P(256), need, None) == -1
    assert L.moe_grouped_mmq_gateup_q8_1(*args, R, d, f, P(16), P(18), P(256), need, None) == -2
