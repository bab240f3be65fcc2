"""Helpers shared by the GPU parity tests (inputs from synth, references from oracle)."""

from __future__ import annotations

import numpy as np
import torch

import oracle as O
import synth as S

TOL = 2e-2   # |gpu - ref| <= TOL * (1 + |ref|) on BF16 outputs


def bits_to_dev(bits: np.ndarray, dev) -> torch.Tensor:
    """uint16 BF16 bits -> torch.bfloat16 tensor on dev."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def i32_to_dev(x: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev)


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at each value's magnitude (2**(e - 7) for |v| in [2**e, 2**(e+1)))."""
    v = np.abs(O.bf16_to_f64(bits))
    _, e = np.frexp(v)                       # v = m * 2**e, m in [0.5, 1)
    return np.where(v > 0, np.ldexp(1.0, np.maximum(e - 8, -133)), np.ldexp(1.0, -133))


def combine_slack(y_bits: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """Extra bound on a combined output out[t] = sum_j w[t, j] * y[t*k + j]: one BF16 ulp of each
    rounded intermediate y, times |w|. The intermediate is rounded to BF16 from an FP32 sum whose
    order differs between the GPU and the oracle, so it may land one ulp apart.

    y_bits [T*k, N] (the oracle's intermediate rows), weights [T, k] -> [T, N]."""
    t, k = weights.shape
    u = bf16_ulp(y_bits).reshape(t, k, -1)
    return np.einsum("tk,tkn->tn", np.abs(weights.astype(np.float64)), u)


def assert_close(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str = "", slack=None) -> float:
    """|gpu - ref| <= TOL * (1 + |ref|) (+ slack, where an intermediate BF16 rounding feeds the output)."""
    g = O.bf16_to_f64(gpu_bits)
    r = O.bf16_to_f64(ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - r)
    bound = TOL * (1.0 + np.abs(r))
    if slack is not None:
        bound = bound + slack
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {tuple(idx)}: "
                             f"gpu={g[tuple(idx)]} ref={r[tuple(idx)]}")
    return float((err / (1.0 + np.abs(r))).max(initial=0.0))


def random_weights(rng: np.random.Generator, e: int, n: int, k: int):
    qw = rng.integers(0, 2 ** 32, size=(e, n, k // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    sc = S.f32_to_bf16_bits(rng.uniform(S.SCALE_LO, S.SCALE_HI, size=(e, n, k // 32)).astype(np.float32))
    return qw, sc


def random_acts(rng: np.random.Generator, rows: int, k: int) -> np.ndarray:
    return S.f32_to_bf16_bits(rng.standard_normal((rows, k)).astype(np.float32))


def ids_from_counts(rng: np.random.Generator, counts) -> np.ndarray:
    """top_k = 1 routing in which expert e receives counts[e] tokens (token order shuffled)."""
    ids = np.concatenate([np.full(c, e, dtype=np.int32) for e, c in enumerate(counts)])
    rng.shuffle(ids)
    return ids.reshape(-1, 1)


def distinct_topk(rng: np.random.Generator, t: int, e: int, k: int) -> np.ndarray:
    return np.stack([rng.permutation(e)[:k] for _ in range(t)]).astype(np.int32)


def prepare_dev(qw: np.ndarray, sc: np.ndarray, mode: int, dev):
    import w4a16_int4_mixture_grouped_gb300 as M
    return M.prepare(torch.from_numpy(qw).to(dev), bits_to_dev(sc, dev), mode=mode)


def small_ws(dev):
    """A zeroed header-only workspace (enough for the routing-layout calls)."""
    import w4a16_int4_mixture_grouped_gb300 as M
    ws = torch.zeros(M.WS_HEADER_BYTES, dtype=torch.uint8, device=dev)
    return ws
