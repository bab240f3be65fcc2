"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test ties one oracle function to a library routine, a brute-force or
exact-rational computation, a closed form or a hand-derived value, chosen so
that a dropped term, a wrong sign or index or a transposed operand fails.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import synth as S

HERE = os.path.dirname(os.path.abspath(__file__))


def torch_bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
# BF16 rounding
# ----------------------------------------------------------------------------

def test_round_bf16_matches_torch_on_float32_values():
    g = np.random.default_rng(1)
    bits = g.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, 3.3895313892515355e38, 3.4e38,
                         1e-40, -1e-40, 1.1754943508222875e-38, 9.183549615799121e-41], dtype=np.float32)
    x = np.concatenate([x, specials])
    mine = O.round_bf16(x.astype(np.float64))
    ref = torch_bf16_bits_from_f32(x)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all(np.isnan(O.bf16_to_f64(mine[nan])))


def _bruteforce_bf16(x: float) -> int:
    """Nearest BF16 by comparing the two neighbouring BF16 values; ties pick the even pattern."""
    if math.isnan(x):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    ax = abs(x)
    # walk the positive BF16 patterns by binary search on value
    lo, hi = 0, 0x7F80  # 0x7F80 = +inf
    vals = lambda b: O.bf16_to_f64(np.array([b], dtype=np.uint16))[0]
    if ax >= vals(0x7F7F) + (vals(0x7F7F) - vals(0x7F7E)) / 2:
        return sign | 0x7F80
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if vals(mid) <= ax:
            lo = mid
        else:
            hi = mid
    dlo, dhi = ax - vals(lo), vals(hi) - ax
    if dlo < dhi:
        b = lo
    elif dhi < dlo:
        b = hi
    else:
        b = lo if lo % 2 == 0 else hi
    return sign | b


def test_round_bf16_matches_bruteforce_on_float64_values():
    g = np.random.default_rng(2)
    x = np.concatenate([
        g.standard_normal(300) * 10.0 ** g.integers(-40, 38, size=300),
        g.standard_normal(100) * 1e-39,   # subnormal range
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2.0 ** -133 * 0.5, 2.0 ** -133 * 1.5, 2.0 ** -134]),
    ])
    mine = O.round_bf16(x)
    ref = np.array([_bruteforce_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(mine, ref)


# ----------------------------------------------------------------------------
# unpack / dequant
# ----------------------------------------------------------------------------

def test_unpack_hand_patterns():
    words = np.array([[0x76543210, np.uint32(0xFEDCBA98).view(np.int32)]], dtype=np.int64).astype(np.int32)
    q = O.unpack_int4(words)
    assert q.tolist() == [list(range(16))]


def _pack_python(q):
    n, k = q.shape
    out = np.zeros((n, k // 8), dtype=np.int64)
    for r in range(n):
        for w in range(k // 8):
            v = 0
            for i in range(8):
                v |= int(q[r, 8 * w + i]) << (4 * i)
            out[r, w] = v
    return out.astype(np.uint32).view(np.int32)


def test_unpack_round_trip():
    g = np.random.default_rng(3)
    q = g.integers(0, 16, size=(5, 64), dtype=np.uint8)
    assert np.array_equal(O.unpack_int4(_pack_python(q)), q)


def test_dequant_exhaustive_table_vs_torch():
    """All 16 nibbles x all 65536 BF16 scale patterns: one RNE of the exact product."""
    scales = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for q in range(16):
        # one scale per weight: group size 1 for the table
        mine = O.dequant(np.full((65536,), q, dtype=np.uint8), scales, group=1)
        s32 = (scales.astype(np.uint32) << 16).view(np.float32)
        prod32 = np.float32(q - 8) * s32            # exact in float32 (4-bit x 8-bit significands)
        ref = torch_bf16_bits_from_f32(prod32)
        nan = np.isnan(prod32)
        assert np.array_equal(mine[~nan], ref[~nan]), q
        assert np.all(np.isnan(O.bf16_to_f64(mine[nan])))


def test_dequant_groups_of_32_follow_k():
    q = np.full((2, 64), 9, dtype=np.uint8)          # q - 8 = 1 -> W = s
    s = np.array([[0x3F80, 0x4000], [0x4040, 0x4080]], dtype=np.uint16)   # 1, 2 | 3, 4
    w = O.bf16_to_f64(O.dequant(q, s))
    assert np.all(w[0, :32] == 1) and np.all(w[0, 32:] == 2)
    assert np.all(w[1, :32] == 3) and np.all(w[1, 32:] == 4)


# ----------------------------------------------------------------------------
# GEMM: exact rational brute force
# ----------------------------------------------------------------------------

def _frac_to_bf16_bits(x: Fraction) -> int:
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    ax = abs(x)
    e = math.floor(math.log2(ax.numerator) - math.log2(ax.denominator))
    while Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    e = max(e, -126)
    unit = Fraction(2) ** (e - 7)
    m = ax / unit
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = np.float32(float(fl * unit))             # exact: fl < 2**8 + 1 and unit a power of two
    return sign | int(val.view(np.uint32) >> 16)


def test_gemm_matches_exact_rational_bruteforce():
    g = np.random.default_rng(4)
    e_cnt, t, k, kdim, n = 2, 3, 2, 64, 16
    a = S.f32_to_bf16_bits(g.standard_normal((t, kdim)).astype(np.float32))
    qw = g.integers(0, 2 ** 32, size=(e_cnt, n, kdim // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    sc = S.f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(e_cnt, n, kdim // 32)).astype(np.float32))
    ids = np.array([[0, 1], [1, 0], [1, 0]], dtype=np.int32)
    y = O.indexed_gemm(a, ids, lambda e: (qw[e], sc[e]), n)
    af = [[Fraction(float(v)) for v in row] for row in O.bf16_to_f64(a)]
    for f in range(t * k):
        tok, e = f // k, int(ids.reshape(-1)[f])
        for col in range(n):
            acc = Fraction(0)
            for kk in range(kdim):
                word = int(np.uint32(qw[e, col, kk // 8].view(np.uint32)))
                q = (word >> (4 * (kk % 8))) & 0xF
                s = Fraction(float(O.bf16_to_f64(np.array([sc[e, col, kk // 32]]))[0]))
                w_exact = (q - 8) * s
                w_bits = _frac_to_bf16_bits(w_exact)
                w = Fraction(float(O.bf16_to_f64(np.array([w_bits], dtype=np.uint16))[0]))
                acc += af[tok][kk] * w
            assert int(y[f, col]) == _frac_to_bf16_bits(acc), (f, col)


# ----------------------------------------------------------------------------
# hand-derived golden cases
# ----------------------------------------------------------------------------

def _golden():
    with open(os.path.join(HERE, "golden", "closed_form.json")) as fh:
        return {c["name"]: c for c in json.load(fh)["cases"]}


def _pack_rows(q):
    return _pack_python(np.asarray(q, dtype=np.uint8))


def test_golden_ramp_and_parity():
    c = _golden()["ramp_and_parity"]
    kk = np.arange(c["K"])
    q = np.stack([kk % 16, 8 + (kk % 2)]).astype(np.uint8)
    s = O.round_bf16(np.array([c["scale_row0"], c["scale_row1"]]))
    a = O.round_bf16(np.ones((1, c["K"])))
    y = O.indexed_gemm(a, np.array([[0]], dtype=np.int32), lambda e: (_pack_rows(q), s), c["N"])
    assert O.bf16_to_f64(y[0]).tolist() == c["expected"]


def test_golden_dequant_single_rounding():
    c = _golden()["dequant_single_rounding"]
    q = np.full((c["N"], c["K"]), 8, dtype=np.uint8)
    q[:, 0] = c["q_k0"]
    s = np.full((c["N"], c["K"] // 32), c["scale_bits"], dtype=np.uint16)
    a = np.zeros((1, c["K"]))
    a[0, 0] = 1.0
    y = O.indexed_gemm(O.round_bf16(a), np.array([[0]], dtype=np.int32), lambda e: (_pack_rows(q), s), c["N"])
    assert O.bf16_to_f64(y[0]).tolist() == c["expected"]


def test_golden_combine_and_swiglu():
    gd = _golden()
    c = gd["combine_weighted"]
    y = O.round_bf16(np.array([[c["rows"][0]], [c["rows"][1]]]))
    out = O.combine(y, np.array([c["weights"]], dtype=np.float32))
    assert O.bf16_to_f64(out)[0, 0] == c["expected"]
    c = gd["swiglu_unit"]
    h = O.swiglu(O.round_bf16(np.array([[c["gate"], c["up"]]])))
    assert O.bf16_to_f64(h)[0, 0] == c["expected"]


# ----------------------------------------------------------------------------
# invariants
# ----------------------------------------------------------------------------

def _tiny(seed=5, e_cnt=4, t=8, k=2, kdim=128, n=32):
    g = np.random.default_rng(seed)
    a = S.f32_to_bf16_bits(g.standard_normal((t, kdim)).astype(np.float32))
    qw = g.integers(0, 2 ** 32, size=(e_cnt, n, kdim // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    sc = S.f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(e_cnt, n, kdim // 32)).astype(np.float32))
    ids = np.stack([g.permutation(e_cnt)[:k] for _ in range(t)]).astype(np.int32)
    return a, qw, sc, ids


def test_zero_scale_and_zero_point_give_zero():
    a, qw, sc, ids = _tiny()
    y = O.indexed_gemm(a, ids, lambda e: (qw[e], np.zeros_like(sc[e])), 32)
    assert np.all(O.bf16_to_f64(y) == 0)
    eights = np.full_like(qw, np.uint32(0x88888888).view(np.int32))
    y = O.indexed_gemm(a, ids, lambda e: (eights[e], sc[e]), 32)
    assert np.all(O.bf16_to_f64(y) == 0)


def test_identity_like_weights_return_activations():
    g = np.random.default_rng(6)
    kdim = 64
    a = S.f32_to_bf16_bits(g.standard_normal((5, kdim)).astype(np.float32))
    q = np.full((kdim, kdim), 8, dtype=np.uint8)
    np.fill_diagonal(q, 9)
    s = np.full((kdim, kdim // 32), 0x3F80, dtype=np.uint16)   # 1.0
    y = O.indexed_gemm(a, np.zeros((5, 1), dtype=np.int32), lambda e: (_pack_rows(q), s), kdim)
    assert np.array_equal(y, a)


def test_power_of_two_scale_scales_output_exactly():
    a, qw, sc, ids = _tiny()
    y = O.bf16_to_f64(O.indexed_gemm(a, ids, lambda e: (qw[e], sc[e]), 32))
    sc4 = O.round_bf16(O.bf16_to_f64(sc) * 4.0)
    y4 = O.bf16_to_f64(O.indexed_gemm(a, ids, lambda e: (qw[e], sc4[e]), 32))
    assert np.array_equal(y4, 4.0 * y)


def test_expert_permutation_invariance():
    a, qw, sc, ids = _tiny()
    perm = np.array([2, 0, 3, 1])
    inv = np.argsort(perm)
    y = O.indexed_gemm(a, ids, lambda e: (qw[e], sc[e]), 32)
    # relabel: new expert perm[e] holds old expert e's weights
    yp = O.indexed_gemm(a, perm[ids].astype(np.int32), lambda e: (qw[inv[e]], sc[inv[e]]), 32)
    assert np.array_equal(y, yp)


def test_layout_equivalence_indexed_contiguous_masked():
    a, qw, sc, ids = _tiny()
    prov = lambda e: (qw[e], sc[e])
    e_cnt, k = 4, ids.shape[1]
    y = O.indexed_gemm(a, ids, prov, 32)
    row_ids, m_idx = O.contiguous_layout(ids, e_cnt)
    a_pad = O.gather_rows(a, row_ids, k)
    c, valid = O.contiguous_gemm(a_pad, m_idx, prov, 32)
    assert np.array_equal(c[valid], y[row_ids[valid]])
    masked_m, mrows = O.masked_layout(ids, e_cnt, 16)
    a3 = O.gather_rows(a, mrows.reshape(-1), k).reshape(e_cnt, 16, -1)
    cm, mvalid = O.masked_gemm(a3, masked_m, prov, 32)
    assert np.array_equal(cm[mvalid], y[mrows.reshape(-1)[mvalid]])


def test_down_projection_reads_routed_rows():
    """a_per_routed_row: row f reads A[f]; otherwise A[f // top_k]. Swapping them must change results."""
    a, qw, sc, ids = _tiny(t=8, k=2)
    prov = lambda e: (qw[e], sc[e])
    a_rows = np.repeat(a, 2, axis=0)
    y1 = O.indexed_gemm(a, ids, prov, 32)
    y2 = O.indexed_gemm(a_rows, ids, prov, 32, a_per_routed_row=True)
    assert np.array_equal(y1, y2)
    y3 = O.indexed_gemm(a_rows[::-1].copy(), ids, prov, 32, a_per_routed_row=True)
    assert not np.array_equal(y1, y3)


# ----------------------------------------------------------------------------
# align
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("block_m", [1, 8, 16, 32, 128])
def test_align_properties_and_bruteforce(block_m):
    g = np.random.default_rng(7)
    t, k, e_cnt = 37, 3, 9
    ids = np.stack([g.permutation(e_cnt)[:k] for _ in range(t)]).astype(np.int32)
    sorted_ids, expert_ids, npp = O.align(ids, e_cnt, block_m)
    r = t * k
    assert npp == sorted_ids.size == expert_ids.size * block_m
    valid = sorted_ids[sorted_ids < r]
    assert sorted(valid.tolist()) == list(range(r))                 # each (t, j) exactly once
    flat = ids.reshape(-1)
    for b, e in enumerate(expert_ids):
        blk = sorted_ids[b * block_m:(b + 1) * block_m]
        v = blk[blk < r]
        assert np.all(flat[v] == e)                                  # expert-homogeneous
        nv = v.size
        assert np.all(blk[:nv] < r) and np.all(blk[nv:] == r)        # sentinels only at the tail
    # brute-force rebuild: stable sort of flat ids by expert
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(valid, order)
    counts = np.bincount(flat, minlength=e_cnt)
    assert npp == sum(-(-c // block_m) * block_m for c in counts)


def test_contiguous_layout_structure_by_hand():
    """Each expert's rows fill a 128-aligned segment, valid rows first in ascending flat id; padding rows
    carry -1 in both arrays; experts with no rows take no segment. Checked against a layout built by hand
    from per-expert row lists, and on properties (segment starts, counts) that a padding-first or a wrong
    pad size would break."""
    g = np.random.default_rng(11)
    t, k, e_cnt = 70, 3, 7
    used = np.array([0, 1, 2, 3, 5, 6])                             # expert 4 receives no rows
    ids = np.stack([used[g.permutation(used.size)[:k]] for _ in range(t)]).astype(np.int32)
    flat = ids.reshape(-1)
    row_ids, m_idx = O.contiguous_layout(ids, e_cnt)
    # by hand: segment of ceil(c/128)*128 rows per expert with rows, in expert order
    want_rows, want_m = [], []
    for e in range(e_cnt):
        rows = [f for f in range(flat.size) if flat[f] == e]
        if not rows:
            continue
        seg = -(-len(rows) // 128) * 128
        want_rows += rows + [-1] * (seg - len(rows))
        want_m += [e] * len(rows) + [-1] * (seg - len(rows))
    assert np.array_equal(row_ids, np.asarray(want_rows, dtype=np.int32))
    assert np.array_equal(m_idx, np.asarray(want_m, dtype=np.int32))
    assert row_ids.size % 128 == 0
    counts = np.bincount(flat, minlength=e_cnt)
    for s0 in range(0, row_ids.size, 128):                          # segments start at multiples of 128
        seg_m = m_idx[s0:s0 + 128]
        e = seg_m[0]
        assert e >= 0                                               # valid rows come first in a segment
        nv = int((seg_m == e).sum())
        assert np.all(seg_m[:nv] == e) and np.all(seg_m[nv:] == -1)
        assert np.all(row_ids[s0:s0 + nv] >= 0) and np.all(np.diff(row_ids[s0:s0 + nv]) > 0)
    assert np.array_equal(np.bincount(m_idx[m_idx >= 0], minlength=e_cnt), counts)
    assert np.array_equal((row_ids < 0), (m_idx < 0))
    assert row_ids.size == sum(-(-c // 128) * 128 for c in counts)


def test_masked_layout_structure_by_hand():
    """masked_m is the per-expert count; row_ids[e] lists expert e's flat ids in ascending order, then -1."""
    ids = np.array([[2, 0], [0, 1], [2, 1], [1, 0], [3, 2]], dtype=np.int32)
    masked_m, row_ids = O.masked_layout(ids, 5, 4)
    assert masked_m.tolist() == [3, 3, 3, 1, 0]
    assert row_ids.tolist() == [[1, 2, 7, -1], [3, 5, 6, -1], [0, 4, 9, -1], [8, -1, -1, -1], [-1, -1, -1, -1]]
    g = np.random.default_rng(12)
    ids = np.stack([g.permutation(9)[:3] for _ in range(40)]).astype(np.int32)
    masked_m, row_ids = O.masked_layout(ids, 9, 40)
    assert np.array_equal(masked_m, np.bincount(ids.reshape(-1), minlength=9))
    for e in range(9):
        assert np.array_equal(row_ids[e, :masked_m[e]], np.nonzero(ids.reshape(-1) == e)[0])
        assert np.all(row_ids[e, masked_m[e]:] == -1)


def test_masked_layout_overflow_raises():
    ids = np.zeros((5, 1), dtype=np.int32)
    with pytest.raises(ValueError):
        O.masked_layout(ids, 2, 4)


def test_block_m_does_not_change_results():
    a, qw, sc, ids = _tiny()
    prov = lambda e: (qw[e], sc[e])
    y = O.indexed_gemm(a, ids, prov, 32)
    for bm in (1, 8, 64):
        s_ids, _, _ = O.align(ids, 4, bm)
        v = s_ids[s_ids < ids.size]
        # rows computed in aligned order equal rows computed in flat order
        y2 = O.indexed_gemm(a, ids, prov, 32, rows=v)
        assert np.array_equal(y2[v], y[v])


# ----------------------------------------------------------------------------
# epilogues
# ----------------------------------------------------------------------------

def test_swiglu_closed_forms():
    y = O.round_bf16(np.array([[0.0, 16.0, 3.0, 2.0, -7.0, 5.0]]))   # gate [0, 16, 3], up [2, -7, 5]
    h = O.bf16_to_f64(O.swiglu(y))[0]
    assert h[0] == 0.0
    assert h[1] == O.bf16_to_f64(O.round_bf16(np.array([16.0 / (1 + math.exp(-16.0)) * -7.0])))[0]
    assert h[1] == -112.0
    assert h[2] == O.bf16_to_f64(O.round_bf16(np.array([3.0 / (1 + math.exp(-3.0)) * 5.0])))[0]


def test_combine_one_hot_and_convex():
    g = np.random.default_rng(8)
    y = S.f32_to_bf16_bits(g.standard_normal((6, 16)).astype(np.float32))
    w = np.array([[0, 1, 0], [1, 0, 0]], dtype=np.float32)
    out = O.combine(y, w)
    assert np.array_equal(out[0], y[1]) and np.array_equal(out[1], y[3])
    same = np.repeat(y[:1], 3, axis=0)
    out = O.bf16_to_f64(O.combine(same, np.array([[0.2, 0.3, 0.5]], dtype=np.float32)))[0]
    ref = O.bf16_to_f64(y[0])
    ulp = np.abs(ref) * 2.0 ** -7
    assert np.all(np.abs(out - ref) <= ulp)


def test_ffn_sampled_tokens_match_full_chain():
    g = np.random.default_rng(9)
    t, k, e_cnt, hid, inter = 6, 2, 3, 64, 64
    a = S.f32_to_bf16_bits(g.standard_normal((t, hid)).astype(np.float32))
    w1 = [(g.integers(0, 2 ** 32, size=(2 * inter, hid // 8), dtype=np.uint64).astype(np.uint32).view(np.int32),
           S.f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(2 * inter, hid // 32)).astype(np.float32)))
          for _ in range(e_cnt)]
    w2 = [(g.integers(0, 2 ** 32, size=(hid, inter // 8), dtype=np.uint64).astype(np.uint32).view(np.int32),
           S.f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(hid, inter // 32)).astype(np.float32)))
          for _ in range(e_cnt)]
    ids = np.stack([g.permutation(e_cnt)[:k] for _ in range(t)]).astype(np.int32)
    wts = g.uniform(0, 1, size=(t, k)).astype(np.float32)
    full = O.ffn(a, ids, wts, lambda e: w1[e], lambda e: w2[e], 2 * inter, hid)
    part = O.ffn(a, ids, wts, lambda e: w1[e], lambda e: w2[e], 2 * inter, hid, tokens=[1, 4])
    assert np.array_equal(part["out"][[1, 4]], full["out"][[1, 4]])
    # the chain by hand
    y1 = O.indexed_gemm(a, ids, lambda e: w1[e], 2 * inter)
    h = O.swiglu(y1)
    y2 = O.indexed_gemm(h, ids, lambda e: w2[e], hid, a_per_routed_row=True)
    assert np.array_equal(O.combine(y2, wts), full["out"])
