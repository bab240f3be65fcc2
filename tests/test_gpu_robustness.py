"""Run-to-run determinism and workspace reuse.

The decode kernel hands units (and, at the end of small calls, k-range parts
of units) out on demand, so which CTA computes a unit changes from run to run
while every output must not: each unit's sums run in a fixed order, the parts
of a cut unit are added in part order, and the combine adds a token's rows in
slot order. Every counter in a workspace is back at zero after a call, so one
workspace serves calls of different shapes, also after a call that recorded a
device error and had its error word cleared.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import (assert_close, bits_to_dev, combine_slack, dev_to_bits, distinct_topk, i32_to_dev, prepare_dev,
                      random_acts, random_weights)

pytestmark = pytest.mark.gpu

M = pytest.importorskip("w4a16_int4_mixture_grouped_gb300") if torch.cuda.is_available() else None
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


@pytest.mark.parametrize("block_m,flags", [(16, 0), (16, "combine"), (32, "combine"), (192, "combine")])
def test_repeated_calls_are_bit_identical(block_m, flags):
    rng = np.random.default_rng(500 + block_m)
    e, t, k, kd, n = 40, 300, 4, 512, 1024
    ids = distinct_topk(rng, t, e, k)
    comb = flags == "combine"
    f = (M.FLAG_COMBINE | M.FLAG_A_PER_ROW) if comb else 0
    a = bits_to_dev(random_acts(rng, t * k if comb else t, kd), DEV)
    qw, sc = random_weights(rng, e, n, kd)
    pw = prepare_dev(qw, sc, 1, DEV)
    w = torch.from_numpy(rng.uniform(0, 1, size=(t, k)).astype(np.float32)).to(DEV) if comb else None
    ws = M.workspace(M.LAYOUT_INDEXED, t, k, e, n, kd, block_m, f, DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, block_m, ws)
    outs = []
    for _ in range(4):
        outs.append(dev_to_bits(M.indexed(a, pw, s_ids, e_ids, npp, t, k, block_m, ws, flags=f, topk_weights=w)))
    assert M.get_device_error(ws) == 0
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_one_workspace_serves_shapes_and_recovers_after_an_index_error():
    rng = np.random.default_rng(600)
    e, kd, n = 24, 256, 512
    qw, sc = random_weights(rng, e, n, kd)
    pw = prepare_dev(qw, sc, 1, DEV)
    t_max, k = 200, 4
    ws = M.workspace(M.LAYOUT_INDEXED, t_max, k, e, n, kd, 16, M.FLAG_COMBINE | M.FLAG_A_PER_ROW, DEV)
    for t in (200, 37, 1, 120):
        ids = distinct_topk(rng, t, e, k)
        h = random_acts(rng, t * k, kd)
        w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
        s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, 16, ws)
        out = M.indexed(bits_to_dev(h, DEV), pw, s_ids, e_ids, npp, t, k, 16, ws,
                        flags=M.FLAG_COMBINE | M.FLAG_A_PER_ROW, topk_weights=torch.from_numpy(w).to(DEV))
        assert M.get_device_error(ws) == 0
        y = O.indexed_gemm(h, ids, lambda x: (qw[x], sc[x]), n, a_per_routed_row=True)
        assert_close(dev_to_bits(out), O.combine(y, w), f"shape t={t}", slack=combine_slack(y, w))
        if t == 37:
            # a call whose expert ids are out of range records an error and skips those blocks
            bad = e_ids.clone()
            bad[0] = e + 5
            M.indexed(bits_to_dev(h, DEV), pw, s_ids, bad, npp, t, k, 16, ws,
                      flags=M.FLAG_COMBINE | M.FLAG_A_PER_ROW, topk_weights=torch.from_numpy(w).to(DEV))
            assert M.get_device_error(ws) == 8
            M.clear_device_error(ws)
