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
