"""GPU parity, bit-exact parts: dequantised weights, routing layouts, row gather.

Each call goes through the C ABI (python binding) and is compared with the
CPU oracle on the same seeded inputs.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import (bits_to_dev, dev_to_bits, distinct_topk, i32_to_dev, prepare_dev, random_acts, random_weights,
                      small_ws)

pytestmark = pytest.mark.gpu

M = pytest.importorskip("w4a16_int4_mixture_grouped_gb300") if torch.cuda.is_available() else None
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _nan_aware_equal(a: np.ndarray, b: np.ndarray) -> bool:
    fa, fb = O.bf16_to_f64(a), O.bf16_to_f64(b)
    na, nb = np.isnan(fa), np.isnan(fb)
    return bool(np.array_equal(na, nb) and np.array_equal(a[~na], b[~nb]))


@pytest.mark.parametrize("mode", [1, 2])
def test_dequant_check_random_experts_bit_exact(mode):
    rng = np.random.default_rng(11)
    e, n, k = 3, 512, 256
    qw, sc = random_weights(rng, e, n, k)
    pw = prepare_dev(qw, sc, mode, DEV)
    for ex in range(e):
        gpu = dev_to_bits(M.dequant_check(pw, ex))
        ref = O.dequant_expert(qw[ex], sc[ex])
        assert np.array_equal(gpu, ref), f"expert {ex} mode {mode}"


def test_dequant_exhaustive_table_bit_exact():
    """All 16 nibbles x all 65536 BF16 scale patterns through the kernels' dequant routine."""
    n, k = 256, 8192                    # 256 rows x 256 groups = 65536 (row, group) scale slots
    kk = np.arange(k)
    q = np.broadcast_to((kk % 16).astype(np.uint8), (n, k))       # every group of 32 holds q = 0..15 twice
    words = np.zeros((n, k // 8), dtype=np.uint32)
    for i in range(8):
        words |= q[:, i::8].astype(np.uint32) << np.uint32(4 * i)
    sc = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(n, k // 32)
    pw = prepare_dev(words.view(np.int32)[None], sc[None], 1, DEV)
    gpu = dev_to_bits(M.dequant_check(pw, 0))
    ref = O.dequant(q, sc)
    assert _nan_aware_equal(gpu, ref)


@pytest.mark.parametrize("t,k,e,bm", [(64, 2, 8, 16), (37, 3, 9, 1), (300, 8, 64, 32), (1000, 8, 384, 256),
                                      (5, 1, 4, 128), (0, 8, 16, 32)])
def test_align_bit_exact(t, k, e, bm):
    rng = np.random.default_rng(t * 7 + e)
    ids = distinct_topk(rng, t, e, k) if t else np.zeros((0, k), dtype=np.int32)
    ws = small_ws(DEV)
    s_ids, e_ids, npp, counts = M.align(i32_to_dev(ids, DEV), e, bm, ws)
    ref_s, ref_e, ref_n = O.align(ids, e, bm)
    n = int(npp.item())
    assert n == ref_n
    assert np.array_equal(s_ids[:n].cpu().numpy(), ref_s)
    assert np.array_equal(e_ids[: n // bm].cpu().numpy(), ref_e)
    assert np.array_equal(counts.cpu().numpy(), np.bincount(ids.reshape(-1), minlength=e))
    assert M.get_device_error(ws) == 0


def test_align_one_expert_takes_everything():
    ids = np.zeros((513, 1), dtype=np.int32)
    ws = small_ws(DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), 4, 32, ws)
    ref_s, ref_e, ref_n = O.align(ids, 4, 32)
    assert int(npp.item()) == ref_n
    assert np.array_equal(s_ids[:ref_n].cpu().numpy(), ref_s) and np.array_equal(e_ids[: ref_n // 32].cpu().numpy(), ref_e)


def test_contiguous_and_masked_layouts_bit_exact():
    rng = np.random.default_rng(12)
    t, k, e = 200, 4, 16
    ids = distinct_topk(rng, t, e, k)
    ws = small_ws(DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, 128, ws)
    m_idx, row_ids = M.contiguous_layout(s_ids, e_ids, npp, t * k)
    ref_rows, ref_m = O.contiguous_layout(ids, e)
    n = ref_rows.size
    assert np.array_equal(row_ids[:n].cpu().numpy(), ref_rows)
    assert np.array_equal(m_idx[:n].cpu().numpy(), ref_m)
    assert np.all(m_idx[n:].cpu().numpy() == -1) and np.all(row_ids[n:].cpu().numpy() == -1)
    max_m = 80
    mm, mrows = M.masked_layout(i32_to_dev(ids, DEV), e, max_m, ws)
    ref_mm, ref_mrows = O.masked_layout(ids, e, max_m)
    assert np.array_equal(mm.cpu().numpy(), ref_mm)
    assert np.array_equal(mrows.cpu().numpy(), ref_mrows)
    assert M.get_device_error(ws) == 0


def test_gather_rows_exact():
    rng = np.random.default_rng(13)
    a = random_acts(rng, 50, 192)
    row_ids = np.array([3, -1, 49 * 2, 0, 7, -1, 20], dtype=np.int32)
    out = M.gather_rows(bits_to_dev(a, DEV), i32_to_dev(row_ids, DEV), 2)
    assert np.array_equal(dev_to_bits(out), O.gather_rows(a, row_ids, 2))


@pytest.mark.parametrize("row_div", [1, 3])
def test_gather_sorted_exact(row_div):
    rng = np.random.default_rng(14)
    t, k, e, bm, kd = 40, 3, 7, 16, 128
    ids = distinct_topk(rng, t, e, k)
    src = random_acts(rng, t * k if row_div == 1 else t, kd)
    ws = small_ws(DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, bm, ws)
    out = torch.zeros((s_ids.numel(), kd), dtype=torch.bfloat16, device=DEV)
    M.gather_sorted(bits_to_dev(src, DEV), s_ids, npp, t * k, row_div, out=out, ws=ws)
    ref_s, _, n = O.align(ids, e, bm)
    got = dev_to_bits(out)[:n]
    valid = ref_s < t * k
    assert np.array_equal(got[valid], src[ref_s[valid] // row_div])
    assert np.all(got[~valid] == 0)                  # padding slots untouched
    assert M.get_device_error(ws) == 0


def test_device_detects_bad_expert_ids_and_capacity():
    ids = np.array([[0, 1], [2, 99], [1, -3]], dtype=np.int32)
    ws = small_ws(DEV)
    M.align(i32_to_dev(ids, DEV), 4, 8, ws)
    assert M.get_device_error(ws) == 8        # MOE_W4A16_ERR_BAD_INDEX
    M.clear_device_error(ws)
    assert M.get_device_error(ws) == 0
    ids = np.zeros((10, 1), dtype=np.int32)
    M.masked_layout(i32_to_dev(ids, DEV), 2, 4, ws)
    assert M.get_device_error(ws) == 5        # MOE_W4A16_ERR_CAPACITY
