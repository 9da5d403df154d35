"""Seeded synthetic workloads for the MoE prefill layer.

Input generation only: token activations ``x``, top-k routing (``ids``, ``w``) and
quantized expert weights packed as expert records.  None of the layer's seven
stages is computed here; the CUDA library's tests and the oracle's tests both
draw their inputs from this module, and it imports neither of them.

Recipe (all seeded, counter-based, independent of thread count):
  x      ~ N(0, 1) fp32 [T, d]            (tensor id 1); listed tokens set to 0.
  logits ~ N(0, 1) fp32 [T, E]            (tensor id 2); the skewed workload adds
           1.5 * ln(k^-1.1) for the expert of Zipf rank k = 1 + pi(e), where pi is
           the permutation sorting uniforms of tensor id 3.
  ids    = top-K experts by logit, descending, ties to the lower id.
  w      = softmax over the K selected logits, in float64, stored fp32.
  weights: gate/up [f, d], down [d, f] per expert ~ N(0, 0.02) (tensor id
           100 + 3e + m), quantized per 32-wide block of the reduction dimension
           to Q8_0 (d = amax/127, q = round(w/d)), Q4_1 (d = (max-min)/15,
           m = min, q = round((w-m)/d) clamped to [0, 15]) or Q2_0 (d = amax/2,
           c = round(w/d) + 2 clamped to [0, 3]); scales stored fp16.  Q2_K packs
           per 256-wide super-block: each 16-wide sub-block j spans [-mn_j, max_j]
           (mn_j = max(0, -min)) in three steps st_j = (max_j + mn_j)/3; d =
           max st_j / 15 and dmin = max mn_j / 15 (fp16); sc_j = round(st_j/d),
           mn'_j = round(mn_j/dmin) in [0, 15]; c = round((w + dmin*mn'_j) /
           (d*sc_j)) clamped to [0, 3].
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gen.c")
LIB = os.path.join(HERE, "libmoe_gen.so")

Q8_0 = 0
Q4_1 = 1
Q2_0 = 2
Q2_K = 3
WTYPE_NAMES = {Q8_0: "q8_0", Q4_1: "q4_1", Q2_0: "q2_0", Q2_K: "q2_k"}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", SRC,
                        "-o", tmp, "-lm", "-lpthread"], check=True)
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            U64, Z, P, I, D = (ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                               ctypes.c_double)
            lib.gen_normal_f32.argtypes = [U64, U64, U64, Z, D, P, I]
            lib.gen_normal_f32.restype = None
            lib.gen_uniform_f64.argtypes = [U64, U64, U64, Z, P]
            lib.gen_uniform_f64.restype = None
            lib.gen_record_bytes.argtypes = [I, I, I]
            lib.gen_record_bytes.restype = Z
            lib.gen_expert_records.argtypes = [I, I, I, I, U64, D, P, Z, I]
            lib.gen_expert_records.restype = None
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_f32(seed: int, tensor_id: int, n: int, scale: float = 1.0, start: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    if n:
        _load().gen_normal_f32(seed, tensor_id, start, n, scale, out.ctypes.data, _threads())
    return out


def uniform_f64(seed: int, tensor_id: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, np.float64)
    if n:
        _load().gen_uniform_f64(seed, tensor_id, start, n, out.ctypes.data)
    return out


def record_bytes(wtype: int, d: int, f: int) -> int:
    return int(_load().gen_record_bytes(wtype, d, f))


def expert_arena(wtype: int, E: int, d: int, f: int, seed: int, sigma: float = 0.02,
                 stride: int | None = None) -> tuple[np.ndarray, int, int]:
    """E quantized expert records; returns (arena uint8 [E*stride], rec_bytes, stride)."""
    rb = record_bytes(wtype, d, f)
    stride = stride or ((rb + 255) // 256) * 256
    arena = np.zeros(E * stride, np.uint8)
    _load().gen_expert_records(wtype, E, d, f, seed, sigma, arena.ctypes.data, stride, _threads())
    return arena, rb, stride


def topk_softmax(logits: np.ndarray, K: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-K ids by logit (descending, ties to the lower id) and softmax weights
    over the K selected logits (float64, stored fp32)."""
    order = np.argsort(-logits, axis=1, kind="stable")[:, :K]
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    sel = np.exp(sel - sel.max(axis=1, keepdims=True))
    w = (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)
    return order.astype(np.int32), w


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    T: int
    d: int
    f: int
    E: int
    K: int
    wtype: int
    seed: int
    routing: str = "normal"  # "normal" or "zipf"
    zero_tokens: tuple = ()
    zero_every: int = 0      # tokens t with (t+1) % zero_every == 0 are all-zero

    def zero_list(self) -> list[int]:
        z = list(self.zero_tokens)
        if self.zero_every:
            z += [t for t in range(self.T) if (t + 1) % self.zero_every == 0]
        return sorted(set(t for t in z if 0 <= t < self.T))

    def describe(self) -> dict:
        return dict(workload=self.name, T=self.T, d=self.d, f=self.f, E=self.E, K=self.K,
                    weights=WTYPE_NAMES[self.wtype], routing=self.routing, seed=hex(self.seed))


CONFIGS = {c.name: c for c in [
    Config("tiny_T7_d256_f128_E16_K2_q8_0", 7, 256, 128, 16, 2, Q8_0, 0x5EED0001,
           zero_tokens=(3,)),
    Config("T600_d2048_f768_E512_K10_q8_0", 600, 2048, 768, 512, 10, Q8_0, 0x5EED0002,
           zero_tokens=(300,)),
    Config("T2048_d2048_f768_E512_K10_q4_1", 2048, 2048, 768, 512, 10, Q4_1, 0x5EED0003),
    Config("T8192_d2048_f768_E512_K10_q8_0_zipf", 8192, 2048, 768, 512, 10, Q8_0, 0x5EED0004,
           routing="zipf"),
    Config("T32768_d2048_f768_E512_K10_q4_1", 32768, 2048, 768, 512, 10, Q4_1, 0x5EED0005,
           zero_every=997),
    Config("T2048_d2048_f768_E512_K10_q2_0", 2048, 2048, 768, 512, 10, Q2_0, 0x5EED0006,
           zero_tokens=(1024,)),
    Config("T2048_d2048_f768_E512_K10_q2_k", 2048, 2048, 768, 512, 10, Q2_K, 0x5EED0007,
           zero_tokens=(1500,)),
]}
CONFIG_LIST = list(CONFIGS.values())
TINY, T600, T2048, T8192, T32768, T2048_Q2, T2048_Q2K = CONFIG_LIST


def routing_logits(cfg: Config, tokens: np.ndarray | None = None) -> np.ndarray:
    """Router logits [T, E] (or for the listed tokens only)."""
    T, E = cfg.T, cfg.E
    if tokens is None:
        logits = normal_f32(cfg.seed, 2, T * E).reshape(T, E)
    else:
        logits = np.stack([normal_f32(cfg.seed, 2, E, start=int(t) * E) for t in tokens]) \
            if len(tokens) else np.zeros((0, E), np.float32)
    if cfg.routing == "zipf":
        perm = np.argsort(uniform_f64(cfg.seed, 3, E), kind="stable")
        rank = np.empty(E, np.int64)
        rank[perm] = np.arange(E)
        bias = 1.5 * np.log((rank + 1.0) ** -1.1)
        logits = (logits.astype(np.float64) + bias[None, :]).astype(np.float32)
    return logits


def activations(cfg: Config, tokens: np.ndarray | None = None) -> np.ndarray:
    d = cfg.d
    if tokens is None:
        x = normal_f32(cfg.seed, 1, cfg.T * d).reshape(cfg.T, d)
        zl = cfg.zero_list()
        if zl:
            x[zl] = 0.0
        return x
    zs = set(cfg.zero_list())
    rows = [np.zeros(d, np.float32) if int(t) in zs else normal_f32(cfg.seed, 1, d, start=int(t) * d)
            for t in tokens]
    return np.stack(rows) if rows else np.zeros((0, d), np.float32)


@dataclasses.dataclass
class Workload:
    cfg: Config
    x: np.ndarray       # f32 [T, d]
    ids: np.ndarray     # int32 [T, K]
    w: np.ndarray       # f32 [T, K]
    arena: np.ndarray   # uint8 [E * arena_stride]
    rec_bytes: int
    arena_stride: int
    tokens: np.ndarray | None = None  # which tokens of cfg these are (None = all)

    @property
    def T(self):
        return self.x.shape[0]

    def subset(self, tokens) -> "Workload":
        tokens = np.asarray(tokens, np.int64)
        return Workload(self.cfg, np.ascontiguousarray(self.x[tokens]),
                        np.ascontiguousarray(self.ids[tokens]), np.ascontiguousarray(self.w[tokens]),
                        self.arena, self.rec_bytes, self.arena_stride, tokens)


def make_workload(cfg: Config | str, tokens=None, arena=None) -> Workload:
    """Generate a workload; with ``tokens`` only those tokens' rows of x and
    routing are drawn (the same values they have in the full workload)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    tok = None if tokens is None else np.asarray(tokens, np.int64)
    x = activations(cfg, tok)
    ids, w = topk_softmax(routing_logits(cfg, tok), cfg.K)
    if arena is None:
        arena = expert_arena(cfg.wtype, cfg.E, cfg.d, cfg.f, cfg.seed)
    a, rb, stride = arena
    return Workload(cfg, x, ids, w, a, rb, stride, tok)
