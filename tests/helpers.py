"""Shared helpers of the GPU parity tests: cached seeded workloads, uploads, and
oracle sub-problems that let the CPU oracle check sampled rows and tokens of the
full-size workloads (each token's output depends only on its own K rows), or
every row and token, split over one host thread per core."""
from __future__ import annotations

import concurrent.futures
import functools
import os

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


def oracle_threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _pmap(fn, parts):
    """fn over the parts on one host thread each (the oracle's C calls release
    the interpreter lock), results in order."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(parts), oracle_threads())) as ex:
        return list(ex.map(fn, parts))


def oracle_stage_all(stage: str, wl: mw.Workload, offsets, xq, xds) -> np.ndarray:
    """Oracle stage 'gateup' or 'down' on every row: contiguous row ranges, one
    per host thread, each with its own rebased offsets; the MMQ reads every
    expert's record in place in the arena (active position p = expert p; the
    group gather is a byte copy, checked on its own)."""
    cfg = wl.cfg
    E = cfg.E
    offsets = np.asarray(offsets, np.int64)
    R = int(offsets[E])
    active = np.arange(E, dtype=np.int32)
    fn = oracle.grouped_mmq_gateup if stage == "gateup" else oracle.grouped_mmq_down
    bounds = np.linspace(0, R, min(R, 4 * oracle_threads()) + 1).astype(np.int64) if R else [0, 0]

    def run(k):
        r0, r1 = int(bounds[k]), int(bounds[k + 1])
        off = (np.clip(offsets, r0, r1) - r0).astype(np.int32)
        return fn(cfg.wtype, wl.arena, wl.arena_stride, active, E, off, xq[r0:r1], xds[r0:r1],
                  cfg.d, cfg.f)

    n = (cfg.f if stage == "gateup" else cfg.d)
    if R == 0:
        return np.zeros((0, n), np.float32)
    return np.concatenate(_pmap(run, range(len(bounds) - 1)))


def oracle_layer_all(wl: mw.Workload) -> np.ndarray:
    """The oracle's layer output for every token: contiguous token slices, one
    per host thread (tokens are independent)."""
    cfg = wl.cfg
    parts = [p for p in np.array_split(np.arange(wl.T), min(wl.T, 4 * oracle_threads())) if len(p)]

    def run(p):
        sub = wl.subset(p)
        return oracle.layer_forward(cfg.wtype, wl.arena, wl.rec_bytes, wl.arena_stride, sub.x,
                                    sub.ids, sub.w, cfg.E, cfg.d, cfg.f, gather=False)["out"]

    return np.concatenate(_pmap(run, parts))


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
    return rows * k // {mw.Q8_0: 1, mw.Q4_1: 2, mw.Q2_0: 4, mw.Q2_K: 4}[wtype]


def _a128(v):
    return (v + 127) // 128 * 128


def _codes2(p, rows, k):
    """2-bit codes packed four per byte: element 4j+i in bits 2i..2i+1 of byte j."""
    p = p.reshape(rows, k // 4).astype(np.int64)
    c = np.empty((rows, k), np.int64)
    for i in range(4):
        c[:, i::4] = (p >> (2 * i)) & 3
    return c


def _planes(wtype, rec, off, rows, k):
    """Decode one matrix of a record with numpy (independent of the oracle) into
    (q, dpl, mpl) with w = q * dpl + mpl, each scale plane repeated along k to
    its block width.  Q2_0 codes come back as their values c - 2; Q2_K as
    sc * c, with dpl the super-block d [rows, k/256] and mpl = -dmin * mn
    [rows, k/16]."""
    qb = _qbytes(wtype, rows, k)
    base = rec[off:]
    if wtype == mw.Q2_K:
        sb = rows * (k // 256) * 2
        o = _a128(qb)
        dpl = base[o:o + sb].view(np.float16).reshape(k // 256, rows).T.astype(np.float64)
        o += _a128(sb)
        dmin = base[o:o + sb].view(np.float16).reshape(k // 256, rows).T.astype(np.float64)
        o += _a128(sb)
        scmn = base[o:o + rows * (k // 16)].reshape(k // 16, rows).T.astype(np.int64)
        q = _codes2(base[:qb], rows, k) * np.repeat(scmn & 0x0F, 16, axis=1)
        mpl = -np.repeat(dmin, 16, axis=1) * (scmn >> 4)
        return q, dpl, mpl
    sb = rows * (k // 32) * 2
    if wtype == mw.Q8_0:
        q = base[:qb].view(np.int8).reshape(rows, k).astype(np.int64)
    elif wtype == mw.Q2_0:
        q = _codes2(base[:qb], rows, k) - 2
    else:
        p = base[:qb].reshape(rows, k // 2)
        q = np.empty((rows, k), np.int64)
        q[:, 0::2] = p & 0x0F
        q[:, 1::2] = p >> 4
    # scale planes are block-major [k/32][rows]
    dpl = base[_a128(qb):_a128(qb) + sb].view(np.float16).reshape(k // 32, rows).T.astype(np.float64)
    mpl = None
    if wtype == mw.Q4_1:
        o = _a128(qb) + _a128(sb)
        mpl = base[o:o + sb].view(np.float16).reshape(k // 32, rows).T.astype(np.float64)
    return q, dpl, mpl


def _dequant_w(q, dpl, mpl):
    k = q.shape[1]
    w = q.astype(np.float64) * np.repeat(dpl, k // dpl.shape[1], axis=1)
    if mpl is not None:
        w += np.repeat(mpl, k // mpl.shape[1], axis=1)
    return w


def _dequant_x(q, ds):
    dx = ds[..., 0].view(np.float16).astype(np.float64)
    return q.astype(np.float64) * np.repeat(dx, 32, axis=1)


def _msums(wtype, ds):
    """The activation sums the weight type's m term multiplies: s per 32-block
    (Q4_1) or (s_lo, s_hi) per 32-block, i.e. one per 16 values (Q2_K)."""
    if wtype == mw.Q2_K:
        return ds[..., 2:4].reshape(ds.shape[0], -1).view(np.float16).astype(np.float64)
    return ds[..., 1].view(np.float16).astype(np.float64)


def _mat_offsets(wtype, d, f):
    qb = _qbytes(wtype, f, d)
    if wtype == mw.Q2_K:
        g = _a128(qb) + 2 * _a128(f * (d // 256) * 2) + _a128(f * (d // 16))
    else:
        sb = f * (d // 32) * 2
        g = _a128(qb) + _a128(sb) * (2 if wtype == mw.Q4_1 else 1)
    return 0, g, 2 * g


def abs_dot_bound(stage: str, wl: mw.Workload, offsets, xq, xds, rows) -> np.ndarray:
    """sum over k of |w_k| * |x_k| (+ sum of |m| * |s| over the m term's blocks,
    Q4_1 and Q2_K) for
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
    sa = np.abs(_msums(cfg.wtype, xds[rows]))
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
    whose weights are exact in one binary16) plus one per 16 m-term entries (one
    per block for Q4_1, per 16 values for Q2_K), each fp32 accumulation off by at
    most one ulp of the running sum (which abs_dot_bound bounds), and it drops
    the lo*lo product (below 2^-22 of each term).  The oracle rounds once per
    block step (half an ulp): one step per block, two for Q4_1, three for Q2_K."""
    k = cfg.d if stage == "gateup" else cfg.f
    nb = k // 32
    n_acc = (2 if cfg.wtype == mw.Q2_0 else 3) * (k // 16)
    if cfg.wtype == mw.Q4_1:
        n_acc += (nb + 15) // 16
    if cfg.wtype == mw.Q2_K:
        n_acc += (k // 16 + 15) // 16
    n_oracle = nb * {mw.Q4_1: 2, mw.Q2_K: 3}.get(cfg.wtype, 1)
    return (n_acc + n_oracle) * 2.0 ** -23 + 2.0 ** -22
