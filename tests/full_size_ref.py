"""Oracle references at the full workload sizes, computed per expert in a process pool.

Test infrastructure: calls only ``oracle`` (the arithmetic) and ``synth`` (the
seeded inputs). Nothing here computes a value of the method itself:

* ``dequant_tabulated`` returns exactly ``oracle.dequant``'s values. The
  oracle's dequantisation is a function of the 4-bit code and the 16-bit scale
  pattern alone, so it is evaluated once over that whole domain (16 x 65536
  pairs, by ``oracle.dequant`` itself) and an expert's weights are then looked
  up in that table -- indexing, no arithmetic. A CPU test checks the lookup
  against ``oracle.dequant_expert`` bit for bit.
* ``expert_job`` runs, for one expert, the oracle's GEMM (``oracle.gemm_rows``)
  and SwiGLU (``oracle.swiglu``) on the routed rows a test passes in.

The pool is started with the ``spawn`` method (safe after the parent process
has initialised CUDA).
"""

from __future__ import annotations

import multiprocessing
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

import oracle as O
import synth as S

_TABLE: Optional[np.ndarray] = None


def dequant_table() -> np.ndarray:
    """uint16 [16, 65536]: oracle.dequant(q, scale bits) for every code q and every scale bit pattern."""
    global _TABLE
    if _TABLE is None:
        q = np.repeat(np.arange(16, dtype=np.uint8)[:, None], 65536, axis=1)          # q[i, j] = i
        s = np.repeat(np.arange(65536, dtype=np.uint32).astype(np.uint16)[None, :], 16, axis=0)  # s[i, j] = j
        with np.errstate(invalid="ignore", over="ignore"):
            _TABLE = np.ascontiguousarray(O.dequant(q, s, group=1))   # one scale per weight
    return _TABLE


def dequant_tabulated(qweight: np.ndarray, scales: np.ndarray, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """oracle.dequant_expert(qweight, scales) (bf16 bits [N, K]), or only the given output-channel rows."""
    if rows is not None:
        qweight, scales = qweight[rows], scales[rows]
    q = O.unpack_int4(qweight)                                     # uint8 [n, K]
    s = np.repeat(np.asarray(scales, dtype=np.uint16), O.GROUP, axis=-1)
    return dequant_table()[q, s]


# A task: (key, (activation file, row indices), channels (None: all), kind "gemm" | "swiglu").
# The activation rows are rows `row indices` of a .npy file of BF16 bits [rows, K] (memory-mapped, so the
# pool's processes share one copy). kind "swiglu" takes intermediate channels c of a gate_up weight
# (N = 2I): the GEMM rows c and I + c, then oracle.swiglu of the [rows, 2 * len(c)] result.
Task = Tuple[str, Tuple[str, np.ndarray], Optional[np.ndarray], str]

_ARRAYS: Dict[str, np.ndarray] = {}


def _rows(src) -> np.ndarray:
    path, idx = src
    if path not in _ARRAYS:
        _ARRAYS[path] = np.load(path, mmap_mode="r")
    return np.asarray(_ARRAYS[path][np.asarray(idx, dtype=np.int64)])


def expert_job(spec) -> Tuple[int, Dict[str, np.ndarray]]:
    """spec = (workload name for the weights, "w1" | "w2", expert, [Task]) -> (expert, {key: bf16 bits})."""
    wl_name, which, e, tasks = spec
    wl = S.get_workload(wl_name)
    n, _ = wl.gemm_shape(which)
    qw, sc = S.expert_weights(wl, which, e)
    need_all = any(ch is None for _, _, ch, _ in tasks)
    rows = None
    if not need_all:
        parts = []
        for _, _, ch, kind in tasks:
            parts.append(ch)
            if kind == "swiglu":
                parts.append(ch + n // 2)
        rows = np.unique(np.concatenate(parts))
    w = dequant_tabulated(qw, sc, rows)
    pos = None if rows is None else {int(r): i for i, r in enumerate(rows)}
    out = {}
    # the all-channel tasks share one oracle GEMM over their stacked rows
    full = [(key, _rows(src)) for key, src, ch, _ in tasks if ch is None]
    if full:
        y = O.gemm_rows(np.concatenate([a for _, a in full]), w)
        at = 0
        for key, a in full:
            out[key] = y[at:at + a.shape[0]]
            at += a.shape[0]
    for key, src, ch, kind in tasks:
        if ch is None:
            continue
        want = np.concatenate([ch, ch + n // 2]) if kind == "swiglu" else ch
        idx = want if pos is None else np.array([pos[int(r)] for r in want], dtype=np.int64)
        y = O.gemm_rows(_rows(src), w[idx])
        out[key] = O.swiglu(y) if kind == "swiglu" else y
    return e, out


def make_pool(processes: Optional[int] = None):
    n = processes or min(16, os.cpu_count() or 1)
    return multiprocessing.get_context("spawn").Pool(n)


def run_jobs(pool, specs: Sequence) -> Dict[int, Dict[str, np.ndarray]]:
    """{expert: {key: result}} for per-expert job specs (experts with no task are skipped)."""
    results: Dict[int, Dict[str, np.ndarray]] = {}
    specs = [s for s in specs if s[3]]
    if pool is None:
        for s in specs:
            e, r = expert_job(s)
            results[e] = r
        return results
    for e, r in pool.imap_unordered(expert_job, specs, chunksize=1):
        results[e] = r
    return results


def group_channels(n: int, group: int, per_group: int, seed: int) -> np.ndarray:
    """`per_group` channels of every `group`-channel block of [0, n), the first and last channel included."""
    rng = np.random.default_rng(seed)
    picks = [0, n - 1]
    for g0 in range(0, n, group):
        picks += list(g0 + rng.choice(group, size=min(per_group, group), replace=False))
    return np.unique(np.asarray(picks, dtype=np.int64))


def rows_by_expert(topk_ids: np.ndarray, num_experts: int) -> List[np.ndarray]:
    flat = np.asarray(topk_ids).reshape(-1)
    order = np.argsort(flat, kind="stable")
    bounds = np.searchsorted(flat[order], np.arange(num_experts + 1))
    return [order[bounds[e]:bounds[e + 1]] for e in range(num_experts)]
