"""moe_w4a16_indexed_routed: the decode GEMM straight from the router's output, in one launch.

Each CTA of the decode kernel builds the align step's block layout in its own
shared memory, so the call must give exactly what moe_w4a16_align followed by
moe_w4a16_indexed gives with the same block size -- compared bit for bit --
and match the oracle. Covered: every block size class, the plain, SwiGLU and
combine epilogues, experts without rows, an expert count that is not a
multiple of 32, the largest expert count and the largest routed row count,
out-of-range ids (skipped and recorded like the align step does), no tokens,
and the host-side refusals.
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


def _both(ids, a_bits, qw, sc, mode, block_m, flags, w=None):
    t, k = ids.shape
    e = qw.shape[0]
    pw = prepare_dev(qw, sc, mode, DEV)
    a = bits_to_dev(a_bits, DEV)
    wd = torch.from_numpy(w).to(DEV) if w is not None else None
    ids_d = i32_to_dev(ids, DEV)
    ws = M.workspace(M.LAYOUT_INDEXED, t, k, e, pw.n, pw.k, block_m, flags, DEV)
    s_ids, e_ids, npp, _ = M.align(ids_d, e, block_m, ws)
    ref = M.indexed(a, pw, s_ids, e_ids, npp, t, k, block_m, ws, flags=flags, topk_weights=wd)
    err_ref = M.get_device_error(ws)
    M.workspace_init(ws)
    outs = []
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        M.indexed_routed(a, pw, ids_d, block_m, ws, flags=flags, topk_weights=wd, out=out)
        outs.append(out)
    err = M.get_device_error(ws)
    return ref, outs, err_ref, err


@pytest.mark.parametrize("block_m", [8, 16, 32])
@pytest.mark.parametrize("epi", ["plain", "swiglu", "combine"])
def test_routed_equals_align_then_indexed(block_m, epi):
    rng = np.random.default_rng(1400 + block_m + len(epi))
    e, t, k, kd = 37, 70, 5, 320
    n = 512
    # experts 3 and 11 receive no rows
    ids = np.stack([rng.permutation(np.setdiff1d(np.arange(e), [3, 11]))[:k] for _ in range(t)]).astype(np.int32)
    qw, sc = random_weights(rng, e, n, kd)
    w = None
    if epi == "combine":
        flags, mode = M.FLAG_COMBINE | M.FLAG_A_PER_ROW, 1
        a_bits = random_acts(rng, t * k, kd)
        w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
        w /= w.sum(axis=1, keepdims=True)
    else:
        flags, mode = (M.FLAG_SWIGLU, 2) if epi == "swiglu" else (0, 1)
        a_bits = random_acts(rng, t, kd)
    ref, outs, err_ref, err = _both(ids, a_bits, qw, sc, mode, block_m, flags, w)
    assert err_ref == 0 and err == 0
    for out in outs:
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "routed call differs from align + indexed"
    # and against the oracle
    y = O.indexed_gemm(a_bits, ids, lambda x: (qw[x], sc[x]), n, a_per_routed_row=(epi == "combine"))
    got = dev_to_bits(outs[0])
    if epi == "combine":
        assert_close(got, O.combine(y, w), "routed combine", slack=combine_slack(y, w))
    elif epi == "swiglu":
        # MODE_GATE_UP packs gate/up pairs; the oracle's gate = first n/2 logical columns
        assert_close(got, O.swiglu(y), "routed swiglu")
    else:
        assert_close(got, y, "routed plain")


@pytest.mark.parametrize("e,t,k", [(1024, 64, 8), (384, 512, 8), (1, 40, 1), (5, 3, 2)])
def test_routed_edge_shapes(e, t, k):
    rng = np.random.default_rng(1500 + e + t)
    kd, n = 256, 256
    ids = distinct_topk(rng, t, e, k)
    qw, sc = random_weights(rng, e, n, kd)
    a_bits = random_acts(rng, t, kd)
    ref, outs, err_ref, err = _both(ids, a_bits, qw, sc, 1, 16, 0)
    assert err_ref == 0 and err == 0
    for out in outs:
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert_close(dev_to_bits(outs[0]), O.indexed_gemm(a_bits, ids, lambda x: (qw[x], sc[x]), n), "routed edge")


def test_routed_out_of_range_ids_are_skipped_and_recorded():
    rng = np.random.default_rng(1600)
    e, t, k, kd, n = 9, 30, 3, 128, 256
    ids = distinct_topk(rng, t, e, k)
    ids[4, 1] = -1
    ids[17, 0] = e
    qw, sc = random_weights(rng, e, n, kd)
    a_bits = random_acts(rng, t, kd)
    ref, outs, err_ref, err = _both(ids, a_bits, qw, sc, 1, 16, 0)
    assert err_ref == 8 and err == 8      # MOE_W4A16_ERR_BAD_INDEX from both paths
    ok = ids.reshape(-1) >= 0
    ok &= ids.reshape(-1) < e
    rows = np.nonzero(ok)[0]
    r_t = torch.from_numpy(rows).to(DEV)
    for out in outs:
        assert torch.equal(out[r_t].view(torch.int16), ref[r_t].view(torch.int16))


def test_routed_refusals_and_no_tokens():
    rng = np.random.default_rng(1700)
    e, kd, n = 8, 64, 256
    qw, sc = random_weights(rng, e, n, kd)
    pw = prepare_dev(qw, sc, 1, DEV)
    ids = i32_to_dev(distinct_topk(rng, 600, e, 8), DEV)            # 4800 routed rows > 4096
    a = torch.zeros((600, kd), dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(M.LAYOUT_INDEXED, 600, 8, e, n, kd, 16, 0, DEV)
    with pytest.raises(M.MoeW4A16Error) as ex:
        M.indexed_routed(a, pw, ids, 16, ws)
    assert ex.value.status == 2
    for flags, bm in ((M.FLAG_A_SORTED, 16), (M.FLAG_OUT_SORTED, 16), (M.FLAG_SPLIT, 32), (0, 64)):
        with pytest.raises(M.MoeW4A16Error) as ex:
            M.indexed_routed(a[:10], pw, ids[:10], bm, ws, flags=flags)
        assert ex.value.status == 1
    empty = torch.zeros((0, 8), dtype=torch.int32, device=DEV)
    out = M.indexed_routed(a[:0], pw, empty, 16, ws)
    assert out.shape == (0, n)
    assert M.get_device_error(ws) == 0
