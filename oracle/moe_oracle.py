"""Plain CPU oracle of the W4A16 MoE grouped GEMM.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline leg and reference arm, never by the CUDA library.

Source: the page "vLLM x Novita AI launch Chord: an INT4 MoE operator that
speeds up Kimi K2.x by up to 2.15x" (aihot.vn, called "the Chord page" below).

What the method computes (the Chord page, TL;DR and "Two kernel families"):
a mixture-of-experts GEMM with BF16 activations and INT4 (uint4) weights with
BF16 scales per group of 32 along K.  Per routed row r = (token t, slot j)
with expert e = topk_ids[t, j]:

  1. unpack:  q[e, n, k] = nibble k%8 of word k/8 of qweight[e, n]  (low nibble first)
  2. dequant: W[e, n, k] = bf16_rne((q - 8) * s[e, n, k/32])
              "subtract-then-scale", one BF16 rounding (section "H200 and
              Blackwell indexed decode": fusing it into the nibble extraction
              keeps the unfused BF16 rounding order)
  3. GEMM:    Y[r, n] = bf16_rne(sum_k A[row(r), k] * W[e, n, k])
  4. SwiGLU:  h[r, i] = bf16_rne(silu(Y[r, i]) * Y[r, N/2 + i])      (optional)
  5. combine: out[t, n] = bf16_rne(sum_j w[t, j] * Y_down[t*top_k + j, n]) (optional)

Layouts (the Chord page, section "Grouped SM90 kernels", Figure 3):
  * indexed:    activations unpadded; the routing index carries the padding
                sentinels (sorted_ids per expert, padded to block_m with the
                sentinel R = T*top_k);
  * contiguous: each expert's rows padded to a 128-row boundary (m_indices
                gives the expert per row, -1 on padding rows);
  * masked:     a fixed row budget max_m per expert, masked_m valid counts,
                output flat [E*max_m, N] even for a 3-D input (section "grouped
                operator entry points"); rows past masked_m[e] are ignored.

Readings where the pages are silent:
  * accumulation: the dot product is taken in float64 (np.matmul) and rounded
    once to BF16; the GPU accumulates in FP32 in any order, which the BF16
    output tolerance covers;
  * zero point 8, no per-group zero; gate = first N/2 columns, up = last N/2;
  * intermediate tensors (Y, h, Y_down) are rounded to BF16 where a tensor
    would be materialised; the combine sums in float64 and rounds once;
  * within an expert, routed rows are ordered by ascending flat id t*top_k+j;
    experts with no rows get no blocks / no rows.

BF16 values are carried as uint16 bit patterns throughout.
"""

from __future__ import annotations

from typing import Callable, Dict, Iterable, Optional, Tuple

import numpy as np

__all__ = [
    "bf16_to_f64", "round_bf16", "unpack_int4", "dequant", "dequant_expert",
    "gemm_rows", "align", "contiguous_layout", "masked_layout", "gather_rows",
    "indexed_gemm", "contiguous_gemm", "masked_gemm", "swiglu", "combine", "ffn",
    "GROUP", "ZERO_POINT", "CONTIGUOUS_PAD",
]

GROUP = 32            # scales per 32 consecutive k (the Chord page, TL;DR: "group-32 scales")
ZERO_POINT = 8        # subtract-then-scale offset of uint4 weights
CONTIGUOUS_PAD = 128  # contiguous layout row boundary (the Chord page, Figure 3)

WeightProvider = Callable[[int], Tuple[np.ndarray, np.ndarray]]


# ----------------------------------------------------------------------------
# BF16 arithmetic, written from the IEEE-754 definition
# ----------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 values (exact: BF16 is the top half of binary32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to BF16, nearest with ties to even; return the bit patterns.

    BF16 has 8 significant bits, exponents down to 2**-126 for normal numbers and
    a subnormal spacing of 2**-133; values that round to 2**128 or beyond become
    infinities; NaN maps to the quiet NaN 0x7FC0.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    neg = np.signbit(x)
    with np.errstate(invalid="ignore", over="ignore"):
        mant, expo = np.frexp(ax)                       # ax = mant * 2**expo, mant in [0.5, 1)
        r_normal = np.ldexp(np.rint(np.ldexp(mant, 8)), expo - 8)
        r_sub = np.ldexp(np.rint(np.ldexp(ax, 133)), -133)
        r = np.where(ax >= 2.0 ** -126, r_normal, r_sub)
        r = np.where(r >= 2.0 ** 128, np.inf, r)
        r = np.where(neg, -r, r)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


# ----------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------

def unpack_int4(qweight: np.ndarray) -> np.ndarray:
    """int32 [..., K/8] packed words -> uint8 [..., K]; k = 8w+i sits in bits 4i..4i+3 of word w."""
    w = np.asarray(qweight).view(np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    q = (w[..., :, None] >> shifts) & np.uint32(0xF)
    return q.reshape(*w.shape[:-1], w.shape[-1] * 8).astype(np.uint8)


def dequant(q: np.ndarray, scales: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Subtract-then-scale: bf16_rne((q - 8) * s), s shared by ``group`` consecutive k.

    The Chord page, section "H200 and Blackwell indexed decode". The product is
    formed exactly in float64 and rounded once.
    """
    q = np.asarray(q)
    s = bf16_to_f64(scales)
    s_full = np.repeat(s, group, axis=-1)
    if s_full.shape != q.shape:
        raise ValueError(f"scale shape {scales.shape} does not cover weights {q.shape} in groups of {group}")
    return round_bf16((q.astype(np.float64) - ZERO_POINT) * s_full)


def dequant_expert(qweight: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """One expert: int32 [N, K/8], bf16 [N, K/32] -> bf16 bits [N, K]."""
    return dequant(unpack_int4(qweight), scales)


def gemm_rows(a_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """bf16_rne(A @ W^T) for A [rows, K], W [N, K] (float64 dot products)."""
    a = bf16_to_f64(a_bits)
    w = bf16_to_f64(w_bits)
    return round_bf16(a @ w.T)


# ----------------------------------------------------------------------------
# routing layouts (the Chord page, Figure 3)
# ----------------------------------------------------------------------------

def _rows_of_expert(topk_ids: np.ndarray, num_experts: int):
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= num_experts):
        raise ValueError("expert id out of range")
    return flat, [np.nonzero(flat == e)[0] for e in range(num_experts)]


def align(topk_ids: np.ndarray, num_experts: int, block_m: int):
    """Indexed layout: (sorted_ids, expert_ids, num_post_padded).

    sorted_ids lists, expert by expert, the flat ids t*top_k+j routed to the
    expert in ascending order, padded to a multiple of ``block_m`` with the
    sentinel R = T*top_k; expert_ids[b] is the expert of block b.
    """
    flat, rows = _rows_of_expert(topk_ids, num_experts)
    sentinel = flat.size
    sorted_parts, expert_ids = [], []
    for e, r in enumerate(rows):
        if r.size == 0:
            continue
        nblk = -(-r.size // block_m)
        part = np.full(nblk * block_m, sentinel, dtype=np.int64)
        part[: r.size] = r
        sorted_parts.append(part)
        expert_ids += [e] * nblk
    sorted_ids = np.concatenate(sorted_parts) if sorted_parts else np.zeros(0, dtype=np.int64)
    return sorted_ids.astype(np.int32), np.asarray(expert_ids, dtype=np.int32), int(sorted_ids.size)


def contiguous_layout(topk_ids: np.ndarray, num_experts: int, pad: int = CONTIGUOUS_PAD):
    """Contiguous layout: (row_ids, m_indices) over M_pad rows.

    Each expert's rows take a ``pad``-aligned segment, valid rows first in
    ascending flat id; padding rows have row_id -1 and m_indices -1.
    """
    sorted_ids, expert_ids, m_pad = align(topk_ids, num_experts, pad)
    sentinel = np.asarray(topk_ids).size
    row_ids = np.where(sorted_ids < sentinel, sorted_ids, -1).astype(np.int32)
    m_indices = np.repeat(expert_ids, pad).astype(np.int32)
    m_indices = np.where(row_ids >= 0, m_indices, -1).astype(np.int32)
    return row_ids, m_indices


def masked_layout(topk_ids: np.ndarray, num_experts: int, max_m: int):
    """Masked layout: (masked_m [E], row_ids [E, max_m]) with -1 past each count.

    Raises when an expert holds more than ``max_m`` rows (no valid masked layout).
    """
    _, rows = _rows_of_expert(topk_ids, num_experts)
    masked_m = np.array([r.size for r in rows], dtype=np.int32)
    if masked_m.size and masked_m.max() > max_m:
        raise ValueError("an expert exceeds the masked row budget")
    row_ids = np.full((num_experts, max_m), -1, dtype=np.int32)
    for e, r in enumerate(rows):
        row_ids[e, : r.size] = r
    return masked_m, row_ids


def gather_rows(a_bits: np.ndarray, row_ids: np.ndarray, div: int) -> np.ndarray:
    """dst[i] = a[row_ids[i] // div], zeros where row_ids[i] < 0."""
    ids = np.asarray(row_ids).reshape(-1)
    out = np.zeros((ids.size, a_bits.shape[1]), dtype=np.uint16)
    ok = ids >= 0
    out[ok] = a_bits[ids[ok] // div]
    return out


# ----------------------------------------------------------------------------
# GEMMs per layout
# ----------------------------------------------------------------------------

def _per_expert_gemm(row_src: np.ndarray, row_expert: np.ndarray, a_bits: np.ndarray,
                     weights: WeightProvider, n: int, cache: Optional[Dict[int, np.ndarray]] = None) -> np.ndarray:
    """out[i] = bf16(A[row_src[i]] . W_{row_expert[i]}^T) for rows with row_expert >= 0."""
    out = np.zeros((row_src.size, n), dtype=np.uint16)
    for e in np.unique(row_expert[row_expert >= 0]):
        sel = np.nonzero(row_expert == e)[0]
        if cache is not None and int(e) in cache:
            w = cache[int(e)]
        else:
            w = dequant_expert(*weights(int(e)))
            if cache is not None:
                cache[int(e)] = w
        out[sel] = gemm_rows(a_bits[row_src[sel]], w)
    return out


def indexed_gemm(a_bits: np.ndarray, topk_ids: np.ndarray, weights: WeightProvider, n: int,
                 a_per_routed_row: bool = False, rows: Optional[Iterable[int]] = None,
                 cache: Optional[Dict[int, np.ndarray]] = None) -> np.ndarray:
    """Indexed layout: Y [R, N] with Y[f] = bf16(A[src(f)] . W_e(f)^T), f = t*top_k + j.

    src(f) = f // top_k when A holds one row per token, f itself when A holds one
    row per routed row (the down projection's input). With ``rows`` only those
    flat ids are computed (the others are left zero).
    """
    topk_ids = np.asarray(topk_ids)
    top_k = topk_ids.shape[1]
    flat = topk_ids.reshape(-1).astype(np.int64)
    r_all = flat.size
    want = np.arange(r_all) if rows is None else np.asarray(sorted(set(int(x) for x in rows)), dtype=np.int64)
    src = want if a_per_routed_row else want // top_k
    part = _per_expert_gemm(src, flat[want], a_bits, weights, n, cache)
    out = np.zeros((r_all, n), dtype=np.uint16)
    out[want] = part
    return out


def contiguous_gemm(a_pad_bits: np.ndarray, m_indices: np.ndarray, weights: WeightProvider, n: int,
                    cache: Optional[Dict[int, np.ndarray]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Contiguous layout: (C [M_pad, N], valid rows mask). Padding-row outputs are unspecified (zero here)."""
    m_idx = np.asarray(m_indices, dtype=np.int64)
    src = np.arange(m_idx.size)
    return _per_expert_gemm(src, m_idx, a_pad_bits, weights, n, cache), m_idx >= 0


def masked_gemm(a3_bits: np.ndarray, masked_m: np.ndarray, weights: WeightProvider, n: int,
                cache: Optional[Dict[int, np.ndarray]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Masked layout: (C flat [E*max_m, N], valid rows mask); rows past masked_m[e] are unspecified."""
    e_cnt, max_m, k = a3_bits.shape
    counts = np.asarray(masked_m, dtype=np.int64)
    if counts.max(initial=0) > max_m:
        raise ValueError("masked_m exceeds the row budget")
    row_exp = np.where(np.arange(max_m)[None, :] < counts[:, None], np.arange(e_cnt)[:, None], -1).reshape(-1)
    flat_a = a3_bits.reshape(e_cnt * max_m, k)
    return _per_expert_gemm(np.arange(e_cnt * max_m), row_exp, flat_a, weights, n, cache), row_exp >= 0


# ----------------------------------------------------------------------------
# epilogues
# ----------------------------------------------------------------------------

def swiglu(y_bits: np.ndarray) -> np.ndarray:
    """h = bf16(silu(gate) * up), gate = first N/2 columns of Y, up = last N/2 (BF16 inputs)."""
    n = y_bits.shape[-1]
    if n % 2:
        raise ValueError("SwiGLU needs an even N")
    g = bf16_to_f64(y_bits[..., : n // 2])
    u = bf16_to_f64(y_bits[..., n // 2:])
    with np.errstate(over="ignore"):
        silu = g / (1.0 + np.exp(-g))
    return round_bf16(silu * u)


def combine(y_bits: np.ndarray, topk_weights: np.ndarray) -> np.ndarray:
    """out[t] = bf16(sum_j w[t, j] * Y[t*top_k + j]), j ascending, float64 sum."""
    w = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    t, k = w.shape
    y = bf16_to_f64(y_bits).reshape(t, k, -1)
    acc = np.zeros((t, y.shape[-1]), dtype=np.float64)
    for j in range(k):
        acc += w[:, j: j + 1] * y[:, j, :]
    return round_bf16(acc)


def ffn(a_bits: np.ndarray, topk_ids: np.ndarray, topk_weights: np.ndarray,
        w1: WeightProvider, w2: WeightProvider, n1: int, n2: int,
        tokens: Optional[Iterable[int]] = None) -> Dict[str, np.ndarray]:
    """Full MoE FFN: gate_up -> SwiGLU -> down -> weighted top-k combine.

    With ``tokens`` only those tokens' rows are computed (sampled checks).
    Returns {"y1": [R, n1], "h": [R, n1/2], "y2": [R, n2], "out": [T, n2]}.
    """
    topk_ids = np.asarray(topk_ids)
    t, k = topk_ids.shape
    tok = np.arange(t) if tokens is None else np.asarray(sorted(set(int(x) for x in tokens)))
    rows = (tok[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    y1 = indexed_gemm(a_bits, topk_ids, w1, n1, rows=rows)
    h = np.zeros((t * k, n1 // 2), dtype=np.uint16)
    h[rows] = swiglu(y1[rows])
    y2 = indexed_gemm(h, topk_ids, w2, n2, a_per_routed_row=True, rows=rows)
    out = np.zeros((t, n2), dtype=np.uint16)
    out[tok] = combine(y2.reshape(t, k, n2)[tok].reshape(-1, n2), np.asarray(topk_weights)[tok])
    return {"y1": y1, "h": h, "y2": y2, "out": out}
