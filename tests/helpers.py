"""Shared helpers of the GPU parity tests: cached seeded workloads, uploads, and
oracle sub-problems that let the CPU oracle check sampled rows and tokens of the
full-size workloads (each token's output depends only on its own K rows)."""
from __future__ import annotations

import functools

import numpy as np

import moe_workloads as mw
import oracle


@functools.lru_cache(maxsize=5)
def workload(name: str) -> mw.Workload:
    return mw.make_workload(mw.CONFIGS[name])


def to_dev(a, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def u16(t) -> np.ndarray:
    """A device int16 (d, s) tensor as host uint16 bit patterns."""
    return t.cpu().numpy().view(np.uint16)


def sample_rows(offsets: np.ndarray, active: np.ndarray, n_active: int, n: int, seed: int):
    """Rows covering the first and last row of the largest and the smallest
    experts, plus random rows."""
    rng = np.random.default_rng(seed)
    act = active[:n_active]
    cnt = offsets[act + 1] - offsets[act]
    pick = set()
    for e in (act[np.argmax(cnt)], act[np.argmin(cnt)], act[0], act[-1]):
        pick.update([int(offsets[e]), int(offsets[e + 1] - 1)])
    R = int(offsets[-1])
    pick.update(int(r) for r in rng.integers(0, R, max(0, n - len(pick))))
    return np.array(sorted(pick), np.int64)


def oracle_rows(stage: str, wl: mw.Workload, offsets, xq, xds, rows):
    """Oracle stage 'gateup' or 'down' on the listed rows only: the rows are
    packed by expert into a small problem with its own offsets, reading each
    expert's record straight from the arena."""
    cfg = wl.cfg
    rows = np.asarray(rows, np.int64)
    row_exp = np.searchsorted(offsets, rows, side="right") - 1
    experts = np.unique(row_exp)
    order = np.argsort(row_exp, kind="stable")
    rows_s = rows[order]
    counts = np.array([np.sum(row_exp == e) for e in experts])
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    st = wl.arena_stride
    sub = np.concatenate([wl.arena[int(e) * st:(int(e) + 1) * st] for e in experts])
    active = np.arange(len(experts), dtype=np.int32)
    fn = oracle.grouped_mmq_gateup if stage == "gateup" else oracle.grouped_mmq_down
    res = fn(cfg.wtype, sub, st, active, len(experts), offs, xq[rows_s], xds[rows_s], cfg.d, cfg.f)
    out = np.empty_like(res)
    out[order] = res
    return out


def rel_l2_rows(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    num = np.linalg.norm((got.astype(np.float64) - ref.astype(np.float64)), axis=-1)
    den = np.linalg.norm(ref.astype(np.float64), axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1), num)


def layer_tokens(cfg) -> np.ndarray:
    """Tokens the layer tests check against the oracle: all of a small workload;
    for a large one 40 seeded tokens, up to four all-zero tokens and the first
    and last token."""
    if cfg.T <= 600:
        return np.arange(cfg.T)
    rng = np.random.default_rng(cfg.seed)
    return np.unique(np.concatenate([rng.integers(0, cfg.T, 40), cfg.zero_list()[:4],
                                     [0, cfg.T - 1]])).astype(np.int64)


def oracle_layer_tokens(wl: mw.Workload, toks) -> np.ndarray:
    """The oracle's layer output for the listed tokens (each token depends only
    on its own K rows, so the oracle runs on that token subset)."""
    cfg = wl.cfg
    sub = wl.subset(toks)
    return oracle.layer_forward(cfg.wtype, wl.arena, wl.rec_bytes, wl.arena_stride, sub.x,
                                sub.ids, sub.w, cfg.E, cfg.d, cfg.f)["out"]


# ------------------------------------------------ numpy record decoders ----
# Plain numpy decoding of an expert record (independent of the oracle and of
# the CUDA library), shared by the oracle pins and the GPU tolerance bounds.

def _qbytes(wtype, rows, k):
    return rows * k // {mw.Q8_0: 1, mw.Q4_1: 2, mw.Q2_0: 4}[wtype]


def _planes(wtype, rec, off, rows, k):
    """Decode one matrix of a record with numpy (independent of the oracle).
    Q2_0 codes come back as their values c - 2."""
    qb = _qbytes(wtype, rows, k)
    a128 = lambda v: (v + 127) // 128 * 128
    sb = rows * (k // 32) * 2
    base = rec[off:]
    if wtype == mw.Q8_0:
        q = base[:qb].view(np.int8).reshape(rows, k).astype(np.int64)
    elif wtype == mw.Q2_0:
        p = base[:qb].reshape(rows, k // 4).astype(np.int64)
        q = np.empty((rows, k), np.int64)
        for i in range(4):  # element 4j+i sits in bits 2i..2i+1 of byte j
            q[:, i::4] = ((p >> (2 * i)) & 3) - 2
    else:
        p = base[:qb].reshape(rows, k // 2)
        q = np.empty((rows, k), np.int64)
        q[:, 0::2] = p & 0x0F
        q[:, 1::2] = p >> 4
    # scale planes are block-major [k/32][rows]
    dpl = base[a128(qb):a128(qb) + sb].view(np.float16).reshape(k // 32, rows).T.astype(np.float64)
    mpl = None
    if wtype == mw.Q4_1:
        o = a128(qb) + a128(sb)
        mpl = base[o:o + sb].view(np.float16).reshape(k // 32, rows).T.astype(np.float64)
    return q, dpl, mpl


def _dequant_w(q, dpl, mpl):
    w = q.astype(np.float64) * np.repeat(dpl, 32, axis=1)
    if mpl is not None:
        w += np.repeat(mpl, 32, axis=1)
    return w


def _dequant_x(q, ds):
    dx = ds[..., 0].view(np.float16).astype(np.float64)
    return q.astype(np.float64) * np.repeat(dx, 32, axis=1)


def _mat_offsets(wtype, d, f):
    a128 = lambda v: (v + 127) // 128 * 128
    qb = _qbytes(wtype, f, d)
    sb = f * (d // 32) * 2
    g = a128(qb) + a128(sb) * (2 if wtype == mw.Q4_1 else 1)
    return 0, g, 2 * g




def abs_dot_bound(stage: str, wl: mw.Workload, offsets, xq, xds, rows) -> np.ndarray:
    """sum over k of |w_k| * |x_k| (+ sum over blocks of |m| * |s| for Q4_1) for
    every output of the listed rows, with the dequantized weights of each row's
    expert: the magnitude that bounds the rounding error of any summation order
    of one output of stage 'gateup' (gate rows then up rows) or 'down'."""
    cfg = wl.cfg
    d, f = cfg.d, cfg.f
    rows = np.asarray(rows, np.int64)
    row_exp = np.searchsorted(offsets, rows, side="right") - 1
    og, ou, od = _mat_offsets(cfg.wtype, d, f)
    st = wl.arena_stride
    out = []
    xa = np.abs(_dequant_x(xq[rows], xds[rows]))
    sa = np.abs(xds[rows][..., 1].view(np.float16).astype(np.float64))
    for i, r in enumerate(rows):
        e = int(row_exp[i])
        rec = wl.arena[e * st:e * st + wl.rec_bytes]
        mats = [(og, f, d), (ou, f, d)] if stage == "gateup" else [(od, d, f)]
        parts = []
        for off, nr, k in mats:
            q, dpl, mpl = _planes(cfg.wtype, rec, off, nr, k)
            wa = np.abs(_dequant_w(q, dpl, None))
            b = wa @ xa[i]
            if mpl is not None:
                b = b + np.abs(mpl) @ sa[i]
            parts.append(b)
        out.append(np.concatenate(parts))
    return np.array(out)


def mmq_error_bound(cfg, stage: str) -> float:
    """Relative bound (times abs_dot_bound) on |GPU - oracle| for one output of a
    grouped MMQ stage, whatever the tensor-core kernel.  The folded-scale kernel
    accumulates every product in TMEM: 3 MMAs per 16-wide K step (2 for Q2_0,
    whose weights are exact in one binary16) plus one per 16 blocks for the Q4_1
    m term, each fp32 accumulation off by at most one ulp of the running sum
    (which abs_dot_bound bounds), and it drops the lo*lo product (below 2^-22 of
    each term).  The oracle rounds once per block (half an ulp)."""
    k = cfg.d if stage == "gateup" else cfg.f
    nb = k // 32
    n_acc = (2 if cfg.wtype == mw.Q2_0 else 3) * (k // 16)
    if cfg.wtype == mw.Q4_1:
        n_acc += (nb + 15) // 16
    return (n_acc + nb) * 2.0 ** -23 + 2.0 ** -22
