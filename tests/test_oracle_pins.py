"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks one oracle function against the pages' own invariants, closed
forms, hand-derived golden values, brute force on tiny inputs, or a library
routine computing the same quantity a different way (numpy's IEEE binary16
conversion, a stable argsort, a plain dequantized matrix product).

Pages cited (pull requests of the "Strata" engine):
  #1368 "quantize each token's MoE input once and scatter it to its k rows",
        intro (slot[t*K+k], the inverse of src) and "Identity" (scatter equals
        the per-row gather quantization byte for byte at T = 1, 2, 7, 600, 2099,
        10 of 512 experts, one all-zero token; D2S6 is the layout that
        serves Q2_K, and the Q2_0 / Q2_K names).
  #439  "a group's expert gathers in one launch", "What" (the batch equals one
        copy per expert byte for byte: 1-16 experts, mid-group starts,
        unaligned / odd sizes).
  #1282 "STRATA_PREFILL_CPU_SHARE=auto ...", "What it does" (the combine weights
        each row of Dm by the token's top-k weight).
"""
import os

import numpy as np
import pytest

import moe_workloads as mw
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- binary16 --

def _np_f16_bits(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def test_f16_roundtrip_all_binary16_values():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    back = oracle.f32_to_f16_bits(f[~nan])
    assert np.array_equal(back, h[~nan])


def test_f16_rounding_against_numpy():
    """Round-to-nearest-even at every rounding boundary and on random patterns."""
    rng = np.random.default_rng(1234)
    hi = np.arange(1 << 19, dtype=np.uint32) << np.uint32(13)
    lows = np.array([0, 1, 0x0FFF, 0x1000, 0x1001, 0x1FFF], np.uint32)
    edge = (hi[:, None] | lows[None, :]).ravel()
    # binary16-subnormal results depend on more low bits: sample that band densely
    sub = (rng.integers(102, 113, 1 << 21, dtype=np.uint32) << np.uint32(23)) | \
        rng.integers(0, 1 << 23, 1 << 21, dtype=np.uint32)
    sub |= rng.integers(0, 2, sub.size, dtype=np.uint32) << np.uint32(31)
    rand = rng.integers(0, 1 << 32, 1 << 22, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([edge, sub, rand])
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        ref = _np_f16_bits(x)
    got = oracle.f32_to_f16_bits(x)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- quantizer --

def _golden_blocks(name="q8_1_blocks.txt"):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif key == "x":
                cur["x"] = np.array([float.fromhex(v) if "0x" in v else float(v) for v in vals],
                                    np.float32)
            elif key == "q":
                cur["q"] = np.array([int(v) for v in vals], np.int8)
            else:
                cur[key] = int(vals[0], 16)
    return cases


@pytest.mark.parametrize("case", _golden_blocks(), ids=lambda c: c["name"])
def test_quantizer_golden_blocks(case):
    assert case["x"].shape == (32,)
    q, dh, sh = oracle.quantize_block_q8_1(case["x"])
    assert np.array_equal(q, case["q"])
    assert dh == case["d"]
    assert sh == case["s"]


def test_quantizer_closed_forms_random():
    """Blocks scaled so amax = 127 have d = 1: q is x rounded half away from zero
    and s = fp16(sum q); blocks scaled so amax = 63.5 have d = 0.5, q = round(2x)."""
    rng = np.random.default_rng(7)
    for scale, dval in ((127.0, 1.0), (63.5, 0.5)):
        for _ in range(200):
            v = rng.normal(size=32)
            v = np.round(v / np.abs(v).max() * scale * 4) / 4  # quarter steps -> exact ties
            i = rng.integers(32)
            v[i] = scale * np.sign(v[i] or 1.0)
            v = v.astype(np.float32)
            q, dh, sh = oracle.quantize_block_q8_1(v)
            y = v.astype(np.float64) / dval
            ref = (np.sign(y) * np.floor(np.abs(y) + 0.5)).astype(np.int64)
            assert np.array_equal(q.astype(np.int64), ref)
            assert dh == int(_np_f16_bits(dval))
            assert sh == int(_np_f16_bits(np.float32(dval) * np.float32(ref.sum())))


def test_quantizer_invariants_random():
    rng = np.random.default_rng(8)
    x = (rng.normal(size=(4000, 32)) * rng.lognormal(0, 3, size=(4000, 1))).astype(np.float32)
    x[::97] = 0.0
    for v in x:
        q, dh, sh = oracle.quantize_block_q8_1(v)
        amax = np.abs(v).max()
        if amax == 0:
            assert not q.any() and dh == 0 and sh == 0
            continue
        d32 = np.float32(amax) / np.float32(127)
        # the largest element maps to +-127, all within [-127, 127], |S| <= 4064
        assert np.abs(q).max() == 127 and np.abs(q.astype(int).sum()) <= 4064
        # each q is within half a step of x/d (rounding), ties away from zero
        r = v.astype(np.float64) / np.float64(d32)
        assert np.all(np.abs(r - q) <= 0.5 + 1e-6)
        assert dh == int(_np_f16_bits(d32))
        assert sh == int(_np_f16_bits(d32 * np.float32(q.astype(np.int64).sum())))


@pytest.mark.parametrize("case", _golden_blocks("q8_1_d2s6_blocks.txt"), ids=lambda c: c["name"])
def test_quantizer_d2s6_golden_blocks(case):
    q, e = oracle.quantize_block_q8_1_d2s6(case["x"])
    assert np.array_equal(q, case["q"])
    assert [int(v) for v in e] == [case["d"], case["s"], case["slo"], case["shi"]]


def test_quantizer_d2s6_invariants_random():
    """D2S6 carries the q8_1 block unchanged (quants, d, s equal the (d, s)
    quantizer's) plus the half sums; a block whose second (first) half is zero
    has s_lo == s and s_hi == 0 (s_lo == 0, s_hi == s); a block whose halves are
    negatives of each other has s == 0 and s_lo == -s_hi; and s_lo + s_hi stays
    within the binary16 rounding of s."""
    rng = np.random.default_rng(12)
    x = (rng.normal(size=(3000, 32)) * rng.lognormal(0, 2, size=(3000, 1))).astype(np.float32)
    x[0:500, 16:] = 0.0
    x[500:1000, :16] = 0.0
    x[1000:1500, 16:] = -x[1000:1500, :16]
    for i, v in enumerate(x):
        q, e = oracle.quantize_block_q8_1_d2s6(v)
        q1, dh, sh = oracle.quantize_block_q8_1(v)
        assert np.array_equal(q, q1) and int(e[0]) == dh and int(e[1]) == sh
        f = e.view(np.float16).astype(np.float64)
        if i < 500:
            assert e[2] == e[1] and f[3] == 0.0
        elif i < 1000:
            assert e[3] == e[1] and f[2] == 0.0
        elif i < 1500:
            assert f[1] == 0.0 and f[2] == -f[3]
        assert abs(f[2] + f[3] - f[1]) <= 2 * 2.0 ** -11 * (abs(f[2]) + abs(f[3]) + abs(f[1]))


def test_scatter_equals_gather_identity_d2s6():
    """#1368 Identity for the D2S6 layout: scatter == per-row gather on the
    whole buffer; requant of the gathered token rows gives the same bytes."""
    T, d, K, E = 300, 256, 10, 512
    x = mw.normal_f32(0xD256, 1, T * d).reshape(T, d)
    x[7] = 0.0
    ids, _ = mw.topk_softmax(mw.normal_f32(0xD256, 2, T * E).reshape(T, E), K)
    sm = oracle.build_slot_map(ids, E)
    R = int(sm["offsets"][E])
    L = oracle.LAYOUT_D2S6
    qs, dss = oracle.quantize_scatter_q8_1(x, sm["slot"], K, R, fill=0x55, layout=L)
    qg, dsg = oracle.quantize_gather_q8_1(x, sm["src"], layout=L)
    qh, dsh = oracle.requant_hidden_q8_1(x[sm["src"]], layout=L)
    assert dss.shape == (R, d // 32, 4)
    assert np.array_equal(qs, qg) and np.array_equal(dss, dsg)
    assert np.array_equal(qs, qh) and np.array_equal(dss, dsh)
    q2, ds2 = oracle.quantize_gather_q8_1(x, sm["src"])
    assert np.array_equal(qs, q2) and np.array_equal(dss[..., :2], ds2)


# ------------------------------------------------------------------ slot map --

def _np_slot_map(ids, E):
    """Expert-sorted rows by a stable argsort (library routine); brute force."""
    flat = ids.ravel()
    valid = (flat >= 0) & (flat < E)
    idx = np.nonzero(valid)[0]
    order = idx[np.argsort(flat[idx], kind="stable")]
    slot = np.full(flat.size, -1, np.int64)
    slot[order] = np.arange(order.size)
    K = ids.shape[1]
    src = order // K
    counts = np.bincount(flat[idx], minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    active = np.nonzero(counts)[0]
    return slot, src, offsets, active


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (1, 10, 512), (2, 10, 512), (7, 2, 16), (600, 10, 512),
                                   (2099, 10, 512), (50, 3, 5)])
def test_slot_map_matches_stable_sort(T, K, E):
    rng = np.random.default_rng(T * 1000 + K)
    ids = np.stack([rng.choice(E, K, replace=False) if K <= E else rng.integers(0, E, K)
                    for _ in range(T)]).astype(np.int32)
    sm = oracle.build_slot_map(ids, E)
    slot, src, offsets, active = _np_slot_map(ids, E)
    assert np.array_equal(sm["slot"], slot)
    assert np.array_equal(sm["src"], src)
    assert np.array_equal(sm["offsets"], offsets)
    assert sm["n_active"] == active.size
    assert np.array_equal(sm["active"][:active.size], active)
    # slot and src are inverses (#1368 intro)
    t_of = np.repeat(np.arange(T), K)
    assert np.array_equal(sm["src"][sm["slot"]], t_of)
    assert sm["dropped"] == 0


def test_slot_map_drops_out_of_range_ids():
    ids = np.array([[0, 3], [7, -1], [2, 3], [3, 100]], np.int32)
    sm = oracle.build_slot_map(ids, 4)
    slot, src, offsets, active = _np_slot_map(ids, 4)
    assert sm["dropped"] == 3
    assert np.array_equal(sm["slot"], slot)
    assert list(sm["slot"][[2, 3, 7]]) == [-1, -1, -1]
    assert np.array_equal(sm["offsets"], offsets)
    assert np.array_equal(sm["src"], src)


def test_slot_map_empty():
    sm = oracle.build_slot_map(np.zeros((0, 4), np.int32), 8)
    assert sm["n_active"] == 0 and not sm["offsets"].any()


# ------------------------------------------------------- quantize-scatter ---

@pytest.mark.parametrize("T", [1, 2, 7, 600, 2099])
def test_scatter_equals_gather_identity(T):
    """#1368 Identity: scatter == per-row gather on the whole buffer, 10 of 512
    experts, one all-zero token."""
    d, K, E = 256, 10, 512
    x = mw.normal_f32(0xABC + T, 1, T * d).reshape(T, d)
    x[T // 2] = 0.0
    ids, _ = mw.topk_softmax(mw.normal_f32(0xABC + T, 2, T * E).reshape(T, E), K)
    sm = oracle.build_slot_map(ids, E)
    R = int(sm["offsets"][E])
    assert R == T * K
    qs, dss = oracle.quantize_scatter_q8_1(x, sm["slot"], K, R, fill=0x55)
    qg, dsg = oracle.quantize_gather_q8_1(x, sm["src"])
    assert np.array_equal(qs, qg) and np.array_equal(dss, dsg)
    # the all-zero token's rows are all-zero bytes
    for k in range(K):
        r = sm["slot"][(T // 2) * K + k]
        assert not qs[r].any() and not dss[r].any()


def test_scatter_skips_dropped_rows():
    x = mw.normal_f32(3, 1, 4 * 64).reshape(4, 64)
    ids = np.array([[0, 1], [1, 9], [0, 2], [2, 1]], np.int32)
    sm = oracle.build_slot_map(ids, 3)
    R = int(sm["offsets"][3])
    qs, dss = oracle.quantize_scatter_q8_1(x, sm["slot"], 2, R)
    qg, dsg = oracle.quantize_gather_q8_1(x, sm["src"])
    assert R == 7 and np.array_equal(qs, qg) and np.array_equal(dss, dsg)


# -------------------------------------------------------------- group gather --

@pytest.mark.parametrize("rec", [16 * 37, 16 * 37 + 7, 1, 131])
@pytest.mark.parametrize("arena_off", [0, 3])
def test_group_gather_equals_one_copy_per_expert(rec, arena_off):
    """#439 What: the batch equals one copy per expert, for 1-16 experts, every
    mid-group start, odd sizes and unaligned addresses."""
    rng = np.random.default_rng(rec + arena_off)
    E = 40
    stride = rec + 5
    raw = rng.integers(0, 256, arena_off + E * stride, dtype=np.uint8)
    arena = raw[arena_off:]
    slot_stride = rec + 9
    for n in range(1, 17):
        for first in range(0, 17 - n):
            ids = rng.choice(E, n, replace=False).astype(np.int32)
            a = rng.integers(0, 256, 16 * slot_stride, dtype=np.uint8)
            b = a.copy()
            oracle.group_gather(arena, rec, stride, ids, first, a, slot_stride)
            for j, e in enumerate(ids):
                oracle.gather_one(arena, rec, stride, e, b, slot_stride, first + j)
            assert np.array_equal(a, b)
            # and against plain slicing
            for j, e in enumerate(ids):
                s = (first + j) * slot_stride
                assert np.array_equal(a[s:s + rec], arena[int(e) * stride:int(e) * stride + rec])


# --------------------------------------------------------------------- MMQ ---

from tests.helpers import _dequant_w, _dequant_x, _mat_offsets, _planes, _qbytes  # noqa: E402


def _silu_mul64(g, u):
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


@pytest.mark.parametrize("wtype", [mw.Q8_0, mw.Q4_1, mw.Q2_0, mw.Q2_K])
def test_record_layout_agrees(wtype):
    sizes = ((256, 256), (2048, 768), (512, 1280)) if wtype == mw.Q2_K else \
        ((256, 128), (2048, 768), (96, 64))
    for d, f in sizes:
        assert oracle.expert_record_bytes(wtype, d, f) == mw.record_bytes(wtype, d, f)
        assert oracle.record_offsets(wtype, d, f) == _mat_offsets(wtype, d, f)
    # sizes worked out by hand: 3*f*d*34/32 and 3*f*d*20/32 at d=2048, f=768
    assert oracle.expert_record_bytes(mw.Q8_0, 2048, 768) == 5013504
    assert oracle.expert_record_bytes(mw.Q4_1, 2048, 768) == 2949120
    # Q2_0: 3*f*d*(2/8 + 2/32)
    assert oracle.expert_record_bytes(mw.Q2_0, 2048, 768) == 1474560
    # Q2_K: 3*f*d*(2/8 + 2*2/256 + 1/16)
    assert oracle.expert_record_bytes(mw.Q2_K, 2048, 768) == 1548288


def _small_problem(wtype, T=9, d=128, f=96, E=5, K=2, seed=11):
    arena, rb, stride = mw.expert_arena(wtype, E, d, f, seed)
    x = mw.normal_f32(seed, 1, T * d).reshape(T, d)
    x[2] = 0.0
    ids, w = mw.topk_softmax(mw.normal_f32(seed, 2, T * E).reshape(T, E), K)
    return arena, rb, stride, x, ids, w


@pytest.mark.parametrize("wtype", [mw.Q8_0, mw.Q4_1, mw.Q2_0, mw.Q2_K])
def test_mmq_against_dequantized_matmul(wtype):
    """The block-scaled integer dot equals the product of the dequantized
    matrices (w = d*q (+m), Q2_K w = d*sc*c - dmin*mn; x = d_x*q_x), computed by
    a plain fp64 matmul.  For Q4_1 (Q2_K) the method uses s = fp16(d_x * sum q_x)
    over each 32-block (16-value half) in the m term, so the two differ by at most
    |m| * |s - fp16(d_x) * sum q_x| per block (half)."""
    d, f, E = (512, 256, 5) if wtype == mw.Q2_K else (128, 96, 5)
    arena, rb, stride, x, ids, w = _small_problem(wtype, d=d, f=f, E=E)
    sm = oracle.build_slot_map(ids, E)
    R = int(sm["offsets"][E])
    lay = oracle.layout_of(wtype)
    q, ds = oracle.quantize_scatter_q8_1(x, sm["slot"], ids.shape[1], R, layout=lay)
    gb = oracle.gather_groups(arena, rb, stride, sm["active"], sm["n_active"], rb)
    h = oracle.grouped_mmq_gateup(wtype, gb, rb, sm["active"], sm["n_active"], sm["offsets"], q, ds, d, f)
    hq, hds = oracle.requant_hidden_q8_1(h, layout=lay)
    y = oracle.grouped_mmq_down(wtype, gb, rb, sm["active"], sm["n_active"], sm["offsets"], hq, hds, d, f)
    og, ou, od = _mat_offsets(wtype, d, f)
    xq = _dequant_x(q, ds)
    hx = _dequant_x(hq, hds)
    for p in range(sm["n_active"]):
        e = sm["active"][p]
        rec = gb[p * rb:(p + 1) * rb]
        rows = slice(sm["offsets"][e], sm["offsets"][e + 1])
        Gq, Gd, Gm = _planes(wtype, rec, og, f, d)
        Uq, Ud, Um = _planes(wtype, rec, ou, f, d)
        Dq, Dd, Dm = _planes(wtype, rec, od, d, f)
        g = xq[rows] @ _dequant_w(Gq, Gd, Gm).T
        u = xq[rows] @ _dequant_w(Uq, Ud, Um).T
        yy = hx[rows] @ _dequant_w(Dq, Dd, Dm).T
        # fp32 rounding of ~64 block terms; Q4_1 adds the s rounding bound
        tol_g = 1e-5 * (np.abs(xq[rows]) @ np.abs(_dequant_w(Gq, Gd, Gm)).T) + 1e-30
        tol_u = 1e-5 * (np.abs(xq[rows]) @ np.abs(_dequant_w(Uq, Ud, Um)).T) + 1e-30
        tol_y = 1e-5 * (np.abs(hx[rows]) @ np.abs(_dequant_w(Dq, Dd, Dm)).T) + 1e-30
        if wtype in (mw.Q4_1, mw.Q2_K):
            def sbound(qx, dsx, m):
                dx = dsx[..., 0].view(np.float16).astype(np.float64)
                if wtype == mw.Q2_K:  # (s_lo, s_hi) against each 16-value half
                    sx = dsx[..., 2:4].view(np.float16).astype(np.float64).reshape(qx.shape[0], -1)
                    dx = np.repeat(dx, 2, axis=1)
                    width = 16
                else:
                    sx = dsx[..., 1].view(np.float16).astype(np.float64)
                    width = 32
                err = np.abs(sx - dx * qx.reshape(qx.shape[0], -1, width).sum(-1))
                return err @ np.abs(m).T
            tol_g += sbound(q[rows], ds[rows], Gm)
            tol_u += sbound(q[rows], ds[rows], Um)
            tol_y += sbound(hq[rows], hds[rows], Dm)
        # the oracle exposes only h = SiLU(g) u; check g and u through it with
        # exact fp64 SiLU and a first-order error bound
        href = _silu_mul64(g, u)
        sg = 1.0 / (1.0 + np.exp(-g))
        dh_dg = np.abs(u * (sg + g * sg * (1 - sg)))
        dh_du = np.abs(g * sg)
        tol_h = dh_dg * tol_g + dh_du * tol_u + 4 * np.finfo(np.float32).eps * np.abs(href) + 1e-30
        assert np.all(np.abs(h[rows] - href) <= tol_h)
        assert np.all(np.abs(y[rows] - yy) <= tol_y)


def test_mmq_integer_special_case():
    """All scales 1 (weights d = 1, activation blocks with amax 127): the down
    product is exactly the integer matrix product."""
    d, f, E = 64, 96, 3
    rng = np.random.default_rng(5)
    rb = oracle.expert_record_bytes(mw.Q8_0, d, f)
    og, ou, od = _mat_offsets(mw.Q8_0, d, f)
    recs = np.zeros(E * rb, np.uint8)
    Wd = []
    for e in range(E):
        qd = rng.integers(-127, 128, (d, f)).astype(np.int8)
        qd[:, ::32] = 127  # a 127 in every block keeps the block maximal
        Wd.append(qd.astype(np.int64))
        base = e * rb + od
        recs[base:base + d * f] = qd.ravel().view(np.uint8)
        dpl = np.full(d * (f // 32), 0x3C00, np.uint16).view(np.uint8)
        o = base + ((d * f + 127) // 128) * 128
        recs[o:o + dpl.size] = dpl
    R = 12
    hq = rng.integers(-127, 128, (R, f)).astype(np.int8)
    hq[:, ::32] = -127
    hds = np.zeros((R, f // 32, 2), np.uint16)
    hds[..., 0] = 0x3C00
    offsets = np.array([0, 5, 5, 12], np.int32)
    active = np.array([0, 2], np.int32)
    gb = np.concatenate([recs[0:rb], recs[2 * rb:3 * rb]])
    y = oracle.grouped_mmq_down(mw.Q8_0, gb, rb, active, 2, offsets, hq, hds, d, f)
    ref = np.concatenate([hq[0:5].astype(np.int64) @ Wd[0].T, hq[5:12].astype(np.int64) @ Wd[2].T])
    assert np.array_equal(y.astype(np.float64), ref.astype(np.float64))


def test_silu_closed_forms():
    """h = SiLU(g) * u: through integer-exact g and u (scales 1) the oracle's h
    equals g/(1+exp(-g))*u within 4 fp32 ulp; SiLU(0) = 0."""
    d, f = 32, 32
    rb = oracle.expert_record_bytes(mw.Q8_0, d, f)
    og, ou, od = _mat_offsets(mw.Q8_0, d, f)
    rec = np.zeros(rb, np.uint8)
    rng = np.random.default_rng(9)
    Gq = rng.integers(-3, 4, (f, d)).astype(np.int8)
    Uq = rng.integers(-3, 4, (f, d)).astype(np.int8)
    Gq[0] = 0
    Gq[:, 0] = 0
    Uq[:, 0] = 0
    for off, Q in ((og, Gq), (ou, Uq)):
        rec[off:off + f * d] = Q.ravel().view(np.uint8)
        o = off + ((f * d + 127) // 128) * 128
        rec[o:o + 2 * f] = np.full(f, 0x3C00, np.uint16).view(np.uint8)
    xq = rng.integers(-2, 3, (4, d)).astype(np.int8)
    xq[:, 0] = 127  # amax 127 -> d = 1; column 0 of the weights is zero
    xds = np.zeros((4, 1, 2), np.uint16)
    xds[..., 0] = 0x3C00
    h = oracle.grouped_mmq_gateup(mw.Q8_0, rec, rb, np.array([0], np.int32), 1,
                                  np.array([0, 4], np.int32), xq, xds, d, f)
    g = xq.astype(np.float64) @ Gq.astype(np.float64).T
    u = xq.astype(np.float64) @ Uq.astype(np.float64).T
    ref = _silu_mul64(g, u)
    assert np.all(h[:, 0] == 0.0)
    # 4 ulp, plus fp32's underflow for SiLU of very negative g
    tol = 4 * np.spacing(np.abs(ref).astype(np.float32)) + 1e-36 * np.maximum(1, np.abs(u))
    assert np.all(np.abs(h - ref) <= tol)
    assert np.abs(g).max() > 20  # the range reaches both SiLU tails


# ----------------------------------------------------------------- combine ---

def test_combine_closed_forms():
    rng = np.random.default_rng(3)
    T, K, d = 6, 3, 64
    y = rng.normal(size=(T * K, d)).astype(np.float32)
    slot = rng.permutation(T * K).astype(np.int32)
    # K = 1, w = 1: out is the row itself
    out = oracle.combine_topk(y, slot[:T], np.ones((T, 1), np.float32), T, 1, d)
    assert np.array_equal(out, y[slot[:T]])
    # fp64 weighted sum within the fp32 rounding bound of K fused steps
    w = rng.random((T, K)).astype(np.float32)
    out = oracle.combine_topk(y, slot, w, T, K, d)
    Y = y[slot].reshape(T, K, d).astype(np.float64)
    ref = np.einsum("tk,tkd->td", w.astype(np.float64), Y)
    bound = K * np.finfo(np.float32).eps * np.einsum("tk,tkd->td", np.abs(w), np.abs(Y))
    assert np.all(np.abs(out - ref) <= bound)
    # dropped rows (slot -1) contribute nothing
    slot2 = slot.copy()
    slot2[1] = -1
    out2 = oracle.combine_topk(y, slot2, w, T, K, d)
    w2 = w.copy()
    w2[0, 1] = 0.0
    assert np.allclose(out2, oracle.combine_topk(y, slot, w2, T, K, d), rtol=0, atol=1e-6)


def test_mmq_q2_0_integer_special_case():
    """Q2_0 with every scale 1: the down product is exactly the integer matrix
    product with the weights c - 2, codes packed here by hand (element 4j+i in
    bits 2i..2i+1 of byte j), which pins the code order and the offset."""
    d, f, E = 64, 96, 2
    rng = np.random.default_rng(7)
    rb = oracle.expert_record_bytes(mw.Q2_0, d, f)
    og, ou, od = _mat_offsets(mw.Q2_0, d, f)
    recs = np.zeros(E * rb, np.uint8)
    Wd = []
    for e in range(E):
        c = rng.integers(0, 4, (d, f))
        Wd.append(c - 2)
        packed = np.zeros((d, f // 4), np.uint8)
        for j in range(f // 4):
            for i in range(4):
                packed[:, j] |= (c[:, 4 * j + i] << (2 * i)).astype(np.uint8)
        base = e * rb + od
        recs[base:base + d * f // 4] = packed.ravel()
        dpl = np.full(d * (f // 32), 0x3C00, np.uint16).view(np.uint8)
        o = base + ((d * f // 4 + 127) // 128) * 128
        recs[o:o + dpl.size] = dpl
    R = 9
    hq = rng.integers(-127, 128, (R, f)).astype(np.int8)
    hds = np.zeros((R, f // 32, 2), np.uint16)
    hds[..., 0] = 0x3C00
    offsets = np.array([0, 4, 9], np.int32)
    active = np.array([0, 1], np.int32)
    y = oracle.grouped_mmq_down(mw.Q2_0, recs, rb, active, 2, offsets, hq, hds, d, f)
    ref = np.concatenate([hq[0:4].astype(np.int64) @ Wd[0].T, hq[4:9].astype(np.int64) @ Wd[1].T])
    assert np.array_equal(y.astype(np.float64), ref.astype(np.float64))


def test_mmq_q2_k_integer_special_case():
    """Q2_K with power-of-two scales, packed here by hand: codes as for Q2_0,
    super-block d and dmin planes [k/256][rows], sub-block bytes sc | mn << 4
    [k/16][rows]; activations with d_x = 1 and exact half sums.  Every term is
    then a multiple of 1/2 below 2^23, so the down product equals the exact
    matrix product with the weights d*sc*c - dmin*mn.  Distinct d and dmin per
    super-block and random sc, mn per sub-block pin the plane order, the
    nibbles, the super-block index and the sign and halves of the min term."""
    d, f, E = 64, 512, 2
    rng = np.random.default_rng(17)
    rb = oracle.expert_record_bytes(mw.Q2_K, d, f)
    og, ou, od = _mat_offsets(mw.Q2_K, d, f)
    a128 = lambda v: (v + 127) // 128 * 128
    recs = np.zeros(E * rb, np.uint8)
    Wd = []
    for e in range(E):
        c = rng.integers(0, 4, (d, f))
        sc = rng.integers(0, 16, (d, f // 16))
        mn = rng.integers(0, 16, (d, f // 16))
        dd = rng.choice([1.0, 2.0], (d, f // 256))
        dm = rng.choice([0.5, 4.0], (d, f // 256))
        Wd.append(np.repeat(dd, 256, axis=1) * np.repeat(sc, 16, axis=1) * c
                  - np.repeat(dm, 256, axis=1) * np.repeat(mn, 16, axis=1))
        packed = np.zeros((d, f // 4), np.uint8)
        for j in range(f // 4):
            for i in range(4):
                packed[:, j] |= (c[:, 4 * j + i] << (2 * i)).astype(np.uint8)
        base = e * rb + od
        recs[base:base + d * f // 4] = packed.ravel()
        o = base + a128(d * f // 4)
        sb = d * (f // 256) * 2
        recs[o:o + sb] = dd.T.astype(np.float16).ravel().view(np.uint8)
        o += a128(sb)
        recs[o:o + sb] = dm.T.astype(np.float16).ravel().view(np.uint8)
        o += a128(sb)
        recs[o:o + d * (f // 16)] = (sc | (mn << 4)).T.astype(np.uint8).ravel()
    R = 9
    hq = rng.integers(-127, 128, (R, f)).astype(np.int8)
    halves = hq.astype(np.int64).reshape(R, f // 32, 2, 16).sum(-1)
    hds = np.zeros((R, f // 32, 4), np.uint16)
    hds[..., 0] = 0x3C00
    hds[..., 1] = halves.sum(-1).astype(np.float16).view(np.uint16)
    hds[..., 2:4] = halves.astype(np.float16).view(np.uint16)  # |half| <= 2032: exact
    offsets = np.array([0, 4, 9], np.int32)
    active = np.array([0, 1], np.int32)
    y = oracle.grouped_mmq_down(mw.Q2_K, recs, rb, active, 2, offsets, hq, hds, d, f)
    ref = np.concatenate([hq[0:4].astype(np.float64) @ Wd[0].T, hq[4:9].astype(np.float64) @ Wd[1].T])
    assert np.array_equal(y.astype(np.float64), ref)
    # the numpy decoder of the tests reads the same record the same way
    q, dpl, mpl = _planes(mw.Q2_K, recs[:rb], od, d, f)
    assert np.array_equal(_dequant_w(q, dpl, mpl), Wd[0])


# ------------------------------------------------------------ end to end ---

@pytest.mark.parametrize("wtype", [mw.Q8_0, mw.Q4_1, mw.Q2_0, mw.Q2_K])
def test_layer_end_to_end_tiny(wtype):
    """Tiny layer: the all-zero token gives an exactly zero row, and the whole
    layer agrees with an unquantized fp64 pipeline (dequantized weights, raw
    activations and hidden rows) to within the 8-bit quantization noise."""
    cfg = mw.TINY
    f = 256 if wtype == mw.Q2_K else cfg.f  # Q2_K super-blocks need k % 256 == 0
    cfg = mw.Config(cfg.name, cfg.T, cfg.d, f, cfg.E, cfg.K, wtype, cfg.seed,
                    zero_tokens=cfg.zero_tokens)
    wl = mw.make_workload(cfg)
    r = oracle.layer_forward(wtype, wl.arena, wl.rec_bytes, wl.arena_stride, wl.x, wl.ids, wl.w,
                             cfg.E, cfg.d, cfg.f)
    assert not r["out"][3].any()
    og, ou, od = _mat_offsets(wtype, cfg.d, cfg.f)
    ref = np.zeros((cfg.T, cfg.d))
    for t in range(cfg.T):
        for k in range(cfg.K):
            e = int(wl.ids[t, k])
            rec = wl.arena[e * wl.arena_stride:e * wl.arena_stride + wl.rec_bytes]
            G = _dequant_w(*_planes(wtype, rec, og, cfg.f, cfg.d))
            U = _dequant_w(*_planes(wtype, rec, ou, cfg.f, cfg.d))
            D = _dequant_w(*_planes(wtype, rec, od, cfg.d, cfg.f))
            xv = wl.x[t].astype(np.float64)
            hv = _silu_mul64(G @ xv, U @ xv)
            ref[t] += wl.w[t, k] * (D @ hv)
    for t in range(cfg.T):
        if t == 3:
            continue
        rel = np.linalg.norm(r["out"][t] - ref[t]) / np.linalg.norm(ref[t])
        assert rel < 0.05, (t, rel)


def test_requant_hidden_uses_the_golden_quantizer():
    """Stage a5 quantizes each 32-block of a hidden row exactly like the golden
    hand-derived blocks (identity row map, one row per case)."""
    cases = _golden_blocks()
    h = np.stack([c["x"] for c in cases]).astype(np.float32)
    h = np.concatenate([h, h[::-1]], axis=1)  # two blocks per row
    hq, hds = oracle.requant_hidden_q8_1(h)
    for i, c in enumerate(cases):
        assert np.array_equal(hq[i, :32], c["q"])
        assert hds[i, 0, 0] == c["d"] and hds[i, 0, 1] == c["s"]
        j = len(cases) - 1 - i
        assert np.array_equal(hq[j, 32:], c["q"])
        assert hds[j, 1, 0] == c["d"] and hds[j, 1, 1] == c["s"]
