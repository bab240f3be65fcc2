"""The full-size reference helpers (tests/full_size_ref.py) on small cases, CPU only.

The GPU parity tests at full size take their references from these helpers;
here the helpers are checked against the oracle's own functions called
directly: the tabulated dequantisation bit for bit against
oracle.dequant_expert, and the per-expert jobs (run in a spawn pool) against
oracle.indexed_gemm / oracle.swiglu on the whole tiny workload.
"""

import os
import tempfile

import numpy as np

import full_size_ref as F
import oracle as O
import synth as S


def test_tabulated_dequant_is_the_oracle_dequant():
    wl = S.get_workload("tiny_indexed")
    for e in (0, 5):
        qw, sc = S.expert_weights(wl, "w1", e)
        assert np.array_equal(F.dequant_tabulated(qw, sc), O.dequant_expert(qw, sc))
        rows = np.array([0, 17, 255])
        assert np.array_equal(F.dequant_tabulated(qw, sc, rows), O.dequant_expert(qw[rows], sc[rows]))
    # every (code, scale) pair, including zero, subnormal, infinite and NaN scales, through one expert-shaped call
    q = np.arange(32, dtype=np.uint32) % 16             # one group of 32 weights: every code twice
    words = np.zeros((65536, 4), dtype=np.uint32)
    for i in range(32):
        words[:, i // 8] |= q[i] << np.uint32(4 * (i % 8))
    scales = np.arange(65536, dtype=np.uint32).astype(np.uint16)[:, None]
    with np.errstate(invalid="ignore", over="ignore"):
        ref = O.dequant_expert(words.view(np.int32), scales)
    got = F.dequant_tabulated(words.view(np.int32), scales)
    assert np.array_equal(got, ref)


def test_expert_jobs_match_the_oracle_on_the_tiny_workload():
    wl = S.get_workload("tiny_indexed")
    ids, _ = S.routing(wl)
    a = S.activations(wl.seed, wl.num_tokens, wl.hidden)
    n, _ = wl.gemm_shape("w1")
    chans = F.group_channels(n // 2, 64, 8, 5)
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "a.npy")
        np.save(path, a)
        rows_e = F.rows_by_expert(ids, wl.num_experts)
        for e, r in enumerate(rows_e):
            assert np.array_equal(r, np.nonzero(ids.reshape(-1) == e)[0])
        specs = [("tiny_indexed", "w1", e,
                  [("all", (path, rows_e[e] // wl.top_k), None, "gemm"),
                   ("sw", (path, rows_e[e] // wl.top_k), chans, "swiglu")])
                 for e in range(wl.num_experts) if rows_e[e].size]
        pool = F.make_pool(2)
        try:
            res = F.run_jobs(pool, specs)
        finally:
            pool.close()
            pool.join()
    y = O.indexed_gemm(a, ids, lambda e: S.expert_weights(wl, "w1", e), n)
    h = O.swiglu(y)
    for e, r in enumerate(rows_e):
        if r.size:
            assert np.array_equal(res[e]["all"], y[r])
            assert np.array_equal(res[e]["sw"], h[r][:, chans])
