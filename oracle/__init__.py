"""Reference oracle for the quantized routed-expert (q8_1 MMQ) MoE prefill layer.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain single-threaded C statement of
the layer (``oracle/oracle.c``) behind numpy-facing ctypes wrappers.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may load
it.  It shares no code with the CUDA library and never imports it.

Every wrapper takes and returns numpy arrays; fp16 quantities are carried as
``uint16`` bit patterns (``ds`` arrays hold ``(d, s)`` pairs along the last axis,
or ``(d, s, s_lo, s_hi)`` in the D2S6 layout that Q2_K weights read).
The pages and passages each function follows are cited in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

W_Q8_0 = 0
W_Q4_1 = 1
W_Q2_0 = 2
W_Q2_K = 3
QK = 32
LAYOUT_DS = 0
LAYOUT_D2S6 = 1


def layout_of(wtype: int) -> int:
    """The activation layout the MMQ of a weight type reads."""
    return LAYOUT_D2S6 if wtype == W_Q2_K else LAYOUT_DS


def ds_per_block(layout: int) -> int:
    return 4 if layout == LAYOUT_D2S6 else 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C11, no FP contraction)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            Z = ctypes.c_size_t
            sig = {
                "oracle_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
                "oracle_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "oracle_f32_to_f16_array": (None, [P, Z, P]),
                "oracle_f16_to_f32_array": (None, [P, Z, P]),
                "oracle_expert_record_bytes": (Z, [I, I, I]),
                "oracle_record_offsets": (None, [I, I, I, P, P, P]),
                "oracle_build_slot_map": (I, [P, I, I, I, P, P, P, P, P]),
                "oracle_quantize_block_q8_1": (None, [P, P, P, P]),
                "oracle_quantize_block_q8_1_d2s6": (None, [P, P, P]),
                "oracle_quantize_scatter_q8_1": (None, [P, I, I, I, P, P, P, I]),
                "oracle_quantize_gather_q8_1": (None, [P, I, P, I, P, P, I]),
                "oracle_requant_hidden_q8_1": (None, [P, I, I, P, P, I]),
                "oracle_gather_one": (None, [P, Z, Z, I, P, Z, I]),
                "oracle_group_gather": (None, [P, Z, Z, P, I, I, P, Z]),
                "oracle_grouped_mmq_gateup": (None, [I, P, Z, P, I, P, P, P, I, I, P]),
                "oracle_grouped_mmq_down": (None, [I, P, Z, P, I, P, P, P, I, I, P]),
                "oracle_combine_topk": (None, [P, P, P, I, I, I, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --- binary16 -------------------------------------------------------------

def f32_to_f16_bits(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_f32_to_f16_array(_p(x), x.size, _p(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().oracle_f16_to_f32_array(_p(h), h.size, _p(out))
    return out


# --- record layout --------------------------------------------------------

def expert_record_bytes(wtype: int, d: int, f: int) -> int:
    return int(_load().oracle_expert_record_bytes(wtype, d, f))


def record_offsets(wtype: int, d: int, f: int):
    g, u, dn = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _load().oracle_record_offsets(wtype, d, f, ctypes.byref(g), ctypes.byref(u), ctypes.byref(dn))
    return g.value, u.value, dn.value


# --- stages -----------------------------------------------------------------

def build_slot_map(ids, E: int):
    """Stage a1.  ids: int32 [T, K].  Returns dict(offsets, slot, src, active,
    n_active, dropped); slot is [T*K], src is [offsets[E]]."""
    ids = _c(ids, np.int32)
    T, K = ids.shape
    offsets = np.zeros(E + 1, np.int32)
    slot = np.empty(T * K, np.int32)
    src = np.full(max(T * K, 1), -1, np.int32)
    active = np.empty(max(E, 1), np.int32)
    n_active = np.zeros(1, np.int32)
    dropped = _load().oracle_build_slot_map(_p(ids), T, K, E, _p(offsets), _p(slot), _p(src),
                                            _p(active), _p(n_active))
    R = int(offsets[E])
    return dict(offsets=offsets, slot=slot, src=src[:R].copy(), active=active[:E].copy(),
                n_active=int(n_active[0]), dropped=int(dropped))


def quantize_block_q8_1(v):
    v = _c(v, np.float32)
    assert v.shape == (QK,)
    q = np.empty(QK, np.int8)
    dh = np.zeros(1, np.uint16)
    sh = np.zeros(1, np.uint16)
    _load().oracle_quantize_block_q8_1(_p(v), _p(q), _p(dh), _p(sh))
    return q, int(dh[0]), int(sh[0])


def quantize_block_q8_1_d2s6(v):
    """One block in the D2S6 layout: q int8 [32] and (d, s, s_lo, s_hi) fp16 bits."""
    v = _c(v, np.float32)
    assert v.shape == (QK,)
    q = np.empty(QK, np.int8)
    e = np.zeros(4, np.uint16)
    _load().oracle_quantize_block_q8_1_d2s6(_p(v), _p(q), _p(e))
    return q, e


def quantize_scatter_q8_1(x, slot, K: int, R: int, fill: int = 0, layout: int = LAYOUT_DS):
    """Stage a2.  x: f32 [T, d]; slot: int32 [T*K].  Returns q int8 [R, d] and
    ds uint16 [R, d/32, ds_per_block(layout)].  Rows nobody writes keep ``fill``."""
    x = _c(x, np.float32)
    slot = _c(slot, np.int32)
    T, d = x.shape
    q = np.full((R, d), fill, np.int8)
    ds = np.full((R, d // QK, ds_per_block(layout)), fill, np.uint16)
    _load().oracle_quantize_scatter_q8_1(_p(x), T, d, K, _p(slot), _p(q), _p(ds), layout)
    return q, ds


def quantize_gather_q8_1(x, src, layout: int = LAYOUT_DS):
    """Per-row gather quantizer: row r quantizes token src[r]."""
    x = _c(x, np.float32)
    src = _c(src, np.int32)
    d = x.shape[1]
    R = src.shape[0]
    q = np.empty((R, d), np.int8)
    ds = np.empty((R, d // QK, ds_per_block(layout)), np.uint16)
    _load().oracle_quantize_gather_q8_1(_p(x), d, _p(src), R, _p(q), _p(ds), layout)
    return q, ds


def requant_hidden_q8_1(h, layout: int = LAYOUT_DS):
    """Stage a5.  h: f32 [R, f] -> hq int8 [R, f], hds uint16 [R, f/32, ds_per_block(layout)]."""
    h = _c(h, np.float32)
    R, f = h.shape
    hq = np.empty((R, f), np.int8)
    hds = np.empty((R, f // QK, ds_per_block(layout)), np.uint16)
    _load().oracle_requant_hidden_q8_1(_p(h), R, f, _p(hq), _p(hds), layout)
    return hq, hds


def gather_one(arena, rec_bytes, arena_stride, expert, group_buf, slot_stride, slot):
    _load().oracle_gather_one(_p(arena), rec_bytes, arena_stride, int(expert), _p(group_buf),
                              slot_stride, int(slot))


def group_gather(arena, rec_bytes, arena_stride, expert_ids, first_slot, group_buf, slot_stride):
    """Stage a3, in place on group_buf (uint8)."""
    ids = _c(expert_ids, np.int32)
    _load().oracle_group_gather(_p(arena), rec_bytes, arena_stride, _p(ids), len(ids),
                                int(first_slot), _p(group_buf), slot_stride)


def grouped_mmq_gateup(wtype, group_base, slot_stride, active, n_active, offsets, q, ds, d, f):
    """Stage a4.  Returns h f32 [R, f] with R = offsets[-1]."""
    active = _c(active, np.int32)
    offsets = _c(offsets, np.int32)
    q = _c(q, np.int8)
    ds = _c(ds, np.uint16)
    R = int(offsets[-1])
    h = np.zeros((R, f), np.float32)
    _load().oracle_grouped_mmq_gateup(wtype, _p(group_base), slot_stride, _p(active), int(n_active),
                                      _p(offsets), _p(q), _p(ds), d, f, _p(h))
    return h


def grouped_mmq_down(wtype, group_base, slot_stride, active, n_active, offsets, hq, hds, d, f):
    """Stage a6.  Returns y f32 [R, d]."""
    active = _c(active, np.int32)
    offsets = _c(offsets, np.int32)
    hq = _c(hq, np.int8)
    hds = _c(hds, np.uint16)
    R = int(offsets[-1])
    y = np.zeros((R, d), np.float32)
    _load().oracle_grouped_mmq_down(wtype, _p(group_base), slot_stride, _p(active), int(n_active),
                                    _p(offsets), _p(hq), _p(hds), d, f, _p(y))
    return y


def combine_topk(y, slot, w, T, K, d):
    """Stage a7.  Returns out f32 [T, d]."""
    y = _c(y, np.float32)
    slot = _c(slot, np.int32)
    w = _c(w, np.float32)
    out = np.empty((T, d), np.float32)
    if y.size == 0:
        y = np.zeros(1, np.float32)
    _load().oracle_combine_topk(_p(y), _p(slot), _p(w), T, K, d, _p(out))
    return out


def gather_groups(arena, rec_bytes, arena_stride, active, n_active, slot_stride):
    """All groups' buffers back to back: expert at active position p lands at
    p * slot_stride (groups of 16 in ascending expert order)."""
    buf = np.zeros(max(n_active, 1) * slot_stride, np.uint8)
    for g0 in range(0, n_active, 16):
        ids = active[g0:min(g0 + 16, n_active)]
        sub = buf[g0 * slot_stride:]
        group_gather(arena, rec_bytes, arena_stride, ids, 0, sub, slot_stride)
    return buf


def layer_forward(wtype, arena, rec_bytes, arena_stride, x, ids, w, E, d, f, slot_stride=None,
                  gather=True):
    """All seven stages in order; returns a dict of every intermediate.  With
    gather=False stage 3 (a byte copy of the routed records, checked on its own)
    is skipped and the two MMQ stages read every record in place in the arena
    (active position p = expert p): the same values without the copy."""
    x = _c(x, np.float32)
    T = x.shape[0]
    K = ids.shape[1]
    sm = build_slot_map(ids, E)
    R = int(sm["offsets"][E])
    lay = layout_of(wtype)
    q, ds = quantize_scatter_q8_1(x, sm["slot"], K, R, layout=lay)
    if gather:
        slot_stride = slot_stride or rec_bytes
        gb = gather_groups(arena, rec_bytes, arena_stride, sm["active"], sm["n_active"],
                           slot_stride)
        active, n_active = sm["active"], sm["n_active"]
    else:
        gb, slot_stride = arena, arena_stride
        active, n_active = np.arange(E, dtype=np.int32), E
    h = grouped_mmq_gateup(wtype, gb, slot_stride, active, n_active, sm["offsets"], q, ds, d, f)
    hq, hds = requant_hidden_q8_1(h, layout=lay)
    y = grouped_mmq_down(wtype, gb, slot_stride, active, n_active, sm["offsets"], hq, hds, d, f)
    out = combine_topk(y, sm["slot"], w, T, K, d)
    return dict(sm, q=q, ds=ds, group_buf=gb if gather else None, h=h, hq=hq, hds=hds, y=y,
                out=out)
