"""GPU parity of the grouped GEMM entry points against the CPU oracle.

Both kernel families (decode: warp MMA; prefill: tcgen05) x the three layouts
x the epilogues, on small shapes that span several tiles and ragged tails,
plus the edge cases of the method: empty experts, one expert holding every
row, rows per expert around the 8/16/32/128/256 tile edges, poison in padding
rows, and device-detected index errors.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import (assert_close, bits_to_dev, combine_slack, dev_to_bits, distinct_topk, i32_to_dev,
                      ids_from_counts, prepare_dev, random_acts, random_weights)

pytestmark = pytest.mark.gpu

M = pytest.importorskip("w4a16_int4_mixture_grouped_gb300") if torch.cuda.is_available() else None
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _indexed_run(a_bits, qw, sc, ids, block_m, mode=1, flags=0, weights=None, a_per_row=False):
    t, k = ids.shape
    e = qw.shape[0]
    pw = prepare_dev(qw, sc, mode, DEV)
    f = flags | (M.FLAG_A_PER_ROW if a_per_row else 0)
    ws = M.workspace(M.LAYOUT_INDEXED, t, k, e, pw.n, pw.k, block_m, f, DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, block_m, ws)
    w_dev = torch.from_numpy(weights).to(DEV) if weights is not None else None
    out = M.indexed(bits_to_dev(a_bits, DEV), pw, s_ids, e_ids, npp, t, k, block_m, ws, flags=f, topk_weights=w_dev)
    code = M.get_device_error(ws)
    assert code == 0, f"device error {code}"
    return dev_to_bits(out)


@pytest.mark.parametrize("block_m", [8, 16, 32, 48, 128, 176, 192])
def test_indexed_plain_matches_oracle(block_m):
    rng = np.random.default_rng(100 + block_m)
    e, t, k, kd, n = 6, 70, 3, 320, 512
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    ids = distinct_topk(rng, t, e, k)
    ref = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n)
    gpu = _indexed_run(a, qw, sc, ids, block_m)
    assert_close(gpu, ref, f"indexed bm={block_m}")


@pytest.mark.parametrize("block_m", [32, 192])
@pytest.mark.parametrize("counts", [[1, 7, 8, 9, 0, 31, 32, 33], [127, 128, 129, 0, 255, 256, 257, 2], [600, 0, 0, 0]])
def test_indexed_tile_edges(block_m, counts):
    rng = np.random.default_rng(sum(counts) + block_m)
    e, kd, n = len(counts), 128, 256
    ids = ids_from_counts(rng, counts)
    a = random_acts(rng, ids.shape[0], kd)
    qw, sc = random_weights(rng, e, n, kd)
    ref = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n)
    gpu = _indexed_run(a, qw, sc, ids, block_m)
    assert_close(gpu, ref, f"edges bm={block_m}")


@pytest.mark.parametrize("block_m", [16, 32, 192])
def test_indexed_gate_up_mode_and_swiglu(block_m):
    rng = np.random.default_rng(7 + block_m)
    e, t, k, kd, n = 5, 90, 2, 256, 512
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    ids = distinct_topk(rng, t, e, k)
    y = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n)
    plain = _indexed_run(a, qw, sc, ids, block_m, mode=2)
    assert_close(plain, y, "gate_up mode plain store")
    h = _indexed_run(a, qw, sc, ids, block_m, mode=2, flags=M.FLAG_SWIGLU)
    assert_close(h, O.swiglu(y), "fused SwiGLU")


@pytest.mark.parametrize("block_m", [16, 32, 128, 192])
def test_indexed_down_with_combine(block_m):
    rng = np.random.default_rng(31 + block_m)
    e, t, k, kd, n = 7, 40, 4, 192, 768
    ids = distinct_topk(rng, t, e, k)
    h = random_acts(rng, t * k, kd)
    qw, sc = random_weights(rng, e, n, kd)
    w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    y = O.indexed_gemm(h, ids, lambda x: (qw[x], sc[x]), n, a_per_routed_row=True)
    ref = O.combine(y, w)
    gpu = _indexed_run(h, qw, sc, ids, block_m, flags=M.FLAG_COMBINE, weights=w, a_per_row=True)
    assert_close(gpu, ref, f"combine bm={block_m}")
    # repeated call reuses the workspace counters
    gpu2 = _indexed_run(h, qw, sc, ids, block_m, flags=M.FLAG_COMBINE, weights=w, a_per_row=True)
    assert np.array_equal(gpu, gpu2)


@pytest.mark.parametrize("block_m", [16, 32, 64, 192])
def test_indexed_sorted_slot_hand_off(block_m):
    """gate_up with OUT_SORTED writes rows at sorted_ids slots; down with A_SORTED reads them there."""
    rng = np.random.default_rng(200 + block_m)
    e, t, k, hid, inter = 6, 50, 3, 256, 256
    a = random_acts(rng, t, hid)
    qw1, sc1 = random_weights(rng, e, 2 * inter, hid)
    qw2, sc2 = random_weights(rng, e, hid, inter)
    ids = distinct_topk(rng, t, e, k)
    w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
    ref = O.ffn(a, ids, w, lambda x: (qw1[x], sc1[x]), lambda x: (qw2[x], sc2[x]), 2 * inter, hid)
    pw1 = prepare_dev(qw1, sc1, 2, DEV)
    pw2 = prepare_dev(qw2, sc2, 1, DEV)
    f1 = M.FLAG_SWIGLU | M.FLAG_OUT_SORTED
    f2 = M.FLAG_COMBINE | M.FLAG_A_SORTED
    ws1 = M.workspace(M.LAYOUT_INDEXED, t, k, e, pw1.n, pw1.k, block_m, f1, DEV)
    ws2 = M.workspace(M.LAYOUT_INDEXED, t, k, e, pw2.n, pw2.k, block_m, f2, DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, block_m, ws1)
    h = M.indexed(bits_to_dev(a, DEV), pw1, s_ids, e_ids, npp, t, k, block_m, ws1, flags=f1)
    n_used = int(npp.item())
    slots = s_ids[:n_used].cpu().numpy()
    valid = slots < t * k
    assert_close(dev_to_bits(h)[:n_used][valid], ref["h"][slots[valid]], f"OUT_SORTED bm={block_m}")
    out = M.indexed(h, pw2, s_ids, e_ids, npp, t, k, block_m, ws2, flags=f2, topk_weights=torch.from_numpy(w).to(DEV))
    assert M.get_device_error(ws1) == 0 and M.get_device_error(ws2) == 0
    assert_close(dev_to_bits(out), ref["out"], f"A_SORTED combine bm={block_m}")


@pytest.mark.parametrize("kernel", ["decode", "prefill"])
def test_contiguous_matches_oracle_and_ignores_poisoned_padding(kernel, monkeypatch):
    monkeypatch.setenv("MOE_W4A16_FORCE_KERNEL", kernel)
    rng = np.random.default_rng(41)
    e, t, k, kd, n = 6, 150, 2, 256, 512
    ids = distinct_topk(rng, t, e, k)
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    row_ids, m_idx = O.contiguous_layout(ids, e)
    a_pad = O.gather_rows(a, row_ids, k)
    a_pad[row_ids < 0] = 0x7FC0                      # NaN in every padding row
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_CONTIGUOUS, t, k, e, n, kd, 0, 0, DEV)
    out = torch.full((a_pad.shape[0], n), 12345.0, dtype=torch.bfloat16, device=DEV)
    M.contiguous(bits_to_dev(a_pad, DEV), i32_to_dev(m_idx, DEV), pw, ws, out=out)
    assert M.get_device_error(ws) == 0
    gpu = dev_to_bits(out)
    ref, valid = O.contiguous_gemm(a_pad, m_idx, lambda x: (qw[x], sc[x]), n)
    assert_close(gpu[valid], ref[valid], f"contiguous {kernel}")
    sentinel = dev_to_bits(torch.full((1,), 12345.0, dtype=torch.bfloat16))[0]
    assert np.all(gpu[~valid] == sentinel), "padding rows were written"


def test_contiguous_runs_of_segments_on_the_tcgen05_kernel(monkeypatch):
    """Each expert's run of 128-row segments is taken in blocks of up to 192 rows: counts around
    the 128 / 192 / 256 / 384 edges, poisoned padding, padding rows left unwritten."""
    monkeypatch.setenv("MOE_W4A16_FORCE_KERNEL", "prefill")
    rng = np.random.default_rng(43)
    counts = [0, 1, 127, 128, 129, 191, 192, 193, 300, 385]
    e, kd, n = len(counts), 192, 256
    ids = ids_from_counts(rng, counts)
    t = ids.shape[0]
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    row_ids, m_idx = O.contiguous_layout(ids, e)
    a_pad = O.gather_rows(a, row_ids, 1)
    a_pad[row_ids < 0] = 0x7FC0
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_CONTIGUOUS, t, 1, e, n, kd, 0, 0, DEV)
    out = torch.full((a_pad.shape[0], n), 12345.0, dtype=torch.bfloat16, device=DEV)
    M.contiguous(bits_to_dev(a_pad, DEV), i32_to_dev(m_idx, DEV), pw, ws, out=out)
    assert M.get_device_error(ws) == 0
    gpu = dev_to_bits(out)
    ref, valid = O.contiguous_gemm(a_pad, m_idx, lambda x: (qw[x], sc[x]), n)
    assert_close(gpu[valid], ref[valid], "contiguous runs of segments")
    sentinel = dev_to_bits(torch.full((1,), 12345.0, dtype=torch.bfloat16))[0]
    assert np.all(gpu[~valid] == sentinel), "padding rows were written"


@pytest.mark.parametrize("kernel", ["decode", "prefill"])
@pytest.mark.parametrize("expected_m", [1, 40, 1000])
def test_masked_matches_oracle_expected_m_only_picks_launch(kernel, expected_m, monkeypatch):
    monkeypatch.setenv("MOE_W4A16_FORCE_KERNEL", kernel)
    rng = np.random.default_rng(51)
    e, t, k, kd, n, max_m = 9, 120, 3, 192, 256, 96
    ids = distinct_topk(rng, t, e, k)
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    masked_m, mrows = O.masked_layout(ids, e, max_m)
    a3 = O.gather_rows(a, mrows.reshape(-1), k).reshape(e, max_m, kd)
    for ex in range(e):
        a3[ex, masked_m[ex]:] = 0x7FC0               # NaN past each count
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_MASKED, t, k, e, n, kd, 0, 0, DEV)
    out = M.masked(bits_to_dev(a3, DEV), i32_to_dev(masked_m, DEV), expected_m, pw, ws)
    assert M.get_device_error(ws) == 0
    ref, valid = O.masked_gemm(a3, masked_m, lambda x: (qw[x], sc[x]), n)
    assert_close(dev_to_bits(out)[valid], ref[valid], f"masked {kernel} em={expected_m}")


@pytest.mark.parametrize("flags", [0, 1])
def test_masked_budget_of_16_rows(flags, monkeypatch):
    """A masked budget of at most 16 rows per expert (the 16-row decode variant), counts 0..16."""
    monkeypatch.setenv("MOE_W4A16_FORCE_KERNEL", "decode")
    rng = np.random.default_rng(55 + flags)
    counts = [16, 0, 5, 9, 16, 1, 13, 8, 0, 15, 2, 16]
    e, kd, n, max_m = len(counts), 320, 512, 16
    ids = ids_from_counts(rng, counts)
    t = ids.shape[0]
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    masked_m, mrows = O.masked_layout(ids, e, max_m)
    a3 = O.gather_rows(a, mrows.reshape(-1), 1).reshape(e, max_m, kd)
    pw = prepare_dev(qw, sc, 2 if flags else 1, DEV)
    ws = M.workspace(M.LAYOUT_MASKED, t, 1, e, n, kd, 0, 0, DEV)
    out = M.masked(bits_to_dev(a3, DEV), i32_to_dev(masked_m, DEV), 6, pw, ws, flags=flags)
    assert M.get_device_error(ws) == 0
    y = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n)
    ref = O.swiglu(y) if flags else y
    valid = mrows.reshape(-1) >= 0
    assert_close(dev_to_bits(out)[valid], ref[mrows.reshape(-1)[valid]], f"masked 16-row budget flags={flags}")


@pytest.mark.parametrize("kernel", ["decode", "prefill"])
def test_masked_swiglu_and_combine(kernel, monkeypatch):
    monkeypatch.setenv("MOE_W4A16_FORCE_KERNEL", kernel)
    rng = np.random.default_rng(61)
    e, t, k, kd, n, max_m = 8, 64, 2, 128, 512, 40
    ids = distinct_topk(rng, t, e, k)
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    masked_m, mrows = O.masked_layout(ids, e, max_m)
    a3 = O.gather_rows(a, mrows.reshape(-1), k).reshape(e, max_m, kd)
    ws = M.workspace(M.LAYOUT_MASKED, t, k, e, n, kd, 0, M.FLAG_COMBINE, DEV)
    y = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n)
    # SwiGLU on a gate_up-mode weight
    pw2 = prepare_dev(qw, sc, 2, DEV)
    h = M.masked(bits_to_dev(a3, DEV), i32_to_dev(masked_m, DEV), 8, pw2, ws, flags=M.FLAG_SWIGLU)
    valid = (mrows.reshape(-1) >= 0)
    assert_close(dev_to_bits(h)[valid], O.swiglu(y)[mrows.reshape(-1)[valid]], f"masked swiglu {kernel}")
    # combine on a plain weight
    w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
    pw1 = prepare_dev(qw, sc, 1, DEV)
    out = M.masked(bits_to_dev(a3, DEV), i32_to_dev(masked_m, DEV), 8, pw1, ws, flags=M.FLAG_COMBINE,
                   row_ids=i32_to_dev(mrows.reshape(-1), DEV), num_tokens=t, top_k=k,
                   topk_weights=torch.from_numpy(w).to(DEV))
    assert M.get_device_error(ws) == 0
    assert_close(dev_to_bits(out), O.combine(y, w), f"masked combine {kernel}")


def test_layout_equivalence_on_gpu():
    """indexed, contiguous and masked give the same valid rows (same kernel family: bit-identical)."""
    rng = np.random.default_rng(71)
    e, t, k, kd, n = 8, 48, 2, 256, 256
    ids = distinct_topk(rng, t, e, k)
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    y_idx = _indexed_run(a, qw, sc, ids, 32)
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_MASKED, t, k, e, n, kd, 0, 0, DEV)
    masked_m, mrows = O.masked_layout(ids, e, 32)
    a3 = O.gather_rows(a, mrows.reshape(-1), k).reshape(e, 32, kd)
    ym = dev_to_bits(M.masked(bits_to_dev(a3, DEV), i32_to_dev(masked_m, DEV), 1, pw, ws))
    v = mrows.reshape(-1) >= 0
    assert np.array_equal(ym[v], y_idx[mrows.reshape(-1)[v]])


def test_empty_routing_is_a_no_op():
    rng = np.random.default_rng(81)
    qw, sc = random_weights(rng, 4, 256, 128)
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_INDEXED, 1, 1, 4, 256, 128, 32, 0, DEV)
    ids = torch.zeros((0, 2), dtype=torch.int32, device=DEV)
    s_ids, e_ids, npp, _ = M.align(ids, 4, 32, ws)
    a = torch.zeros((0, 128), dtype=torch.bfloat16, device=DEV)
    out = M.indexed(a, pw, s_ids, e_ids, npp, 0, 2, 32, ws)
    assert out.shape == (0, 256)
    masked_m = torch.zeros(4, dtype=torch.int32, device=DEV)
    a3 = torch.zeros((4, 16, 128), dtype=torch.bfloat16, device=DEV)
    wsm = M.workspace(M.LAYOUT_MASKED, 1, 1, 4, 256, 128, 0, 0, DEV)
    M.masked(a3, masked_m, 1, pw, wsm)
    assert M.get_device_error(ws) == 0 and M.get_device_error(wsm) == 0


def test_device_index_checks_do_not_fault():
    rng = np.random.default_rng(91)
    qw, sc = random_weights(rng, 4, 256, 128)
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_INDEXED, 8, 1, 4, 256, 128, 32, 0, DEV)
    a = bits_to_dev(random_acts(rng, 8, 128), DEV)
    # masked_m above the budget -> capacity error, no out-of-bounds access
    a3 = torch.zeros((4, 16, 128), dtype=torch.bfloat16, device=DEV)
    wsm = M.workspace(M.LAYOUT_MASKED, 8, 1, 4, 256, 128, 0, 0, DEV)
    M.masked(a3, i32_to_dev(np.array([3, 40, 0, 1]), DEV), 4, pw, wsm)
    assert M.get_device_error(wsm) == 5
    # sorted_ids holding an id past the sentinel and an expert id out of range
    s_ids = i32_to_dev(np.array([0, 1, 99, 8] + [8] * 28), DEV)
    e_ids = i32_to_dev(np.array([7]), DEV)
    npp = i32_to_dev(np.array([32]), DEV)
    M.indexed(a, pw, s_ids, e_ids, npp, 8, 1, 32, ws)
    assert M.get_device_error(ws) == 8
    M.clear_device_error(ws)
    e_ids = i32_to_dev(np.array([1]), DEV)
    M.indexed(a, pw, s_ids, e_ids, npp, 8, 1, 32, ws)
    assert M.get_device_error(ws) == 8
    # the same checks on 16-row blocks (the one-CTA-per-SM decode kernel)
    ws16 = M.workspace(M.LAYOUT_INDEXED, 8, 1, 4, 256, 128, 16, 0, DEV)
    s16 = i32_to_dev(np.array([0, 1, 99, 8] + [8] * 12), DEV)
    npp16 = i32_to_dev(np.array([16]), DEV)
    M.indexed(a, pw, s16, i32_to_dev(np.array([7]), DEV), npp16, 8, 1, 16, ws16)
    assert M.get_device_error(ws16) == 8
    M.clear_device_error(ws16)
    M.indexed(a, pw, s16, i32_to_dev(np.array([1]), DEV), npp16, 8, 1, 16, ws16)
    assert M.get_device_error(ws16) == 8


def test_mode_mismatch_fails_before_launch():
    rng = np.random.default_rng(92)
    qw, sc = random_weights(rng, 2, 256, 64)
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_MASKED, 4, 1, 2, 256, 64, 0, 0, DEV)
    a3 = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device=DEV)
    mm = torch.zeros(2, dtype=torch.int32, device=DEV)
    before = M.launch_count()
    with pytest.raises(M.MoeW4A16Error) as ei:
        M.masked(a3, mm, 1, pw, ws, flags=M.FLAG_SWIGLU)
    assert ei.value.name == "ERR_MODE_MISMATCH"
    assert M.launch_count() == before


@pytest.mark.parametrize("tokens,kernel,block_m,masked_kernel",
                         [(16, 1, 16, 1), (128, 1, 16, 1), (192, 1, 16, 1), (256, 1, 32, 1), (512, 3, 32, 1),
                          (1024, 3, 32, 1), (1152, 3, 32, 3), (1536, 3, 32, 3), (3072, 3, 32, 3), (6096, 3, 32, 3),
                          (6144, 2, 192, 2), (8192, 2, 192, 2)])
def test_plan_picks_family_and_block_from_rows_per_expert(tokens, kernel, block_m, masked_kernel):
    """tok_e = T*top_k/E (384 experts, top-8): decode 16-row blocks up to 4 rows per expert, decode 32-row blocks
    below 8, the split per expert (indexed) from 8 to 127, the tcgen05 family from 128 on; masked calls stay on the
    decode family below 24 rows per expert and split per expert from 24 to 127."""
    s = M.plan(M.LAYOUT_INDEXED, tokens, 8, 384, 4096, 7168)
    assert (s.kernel, s.block_m) == (kernel, block_m)
    assert s.tok_e == -(-tokens * 8 // 384)
    m = M.plan(M.LAYOUT_MASKED, tokens, 8, 384, 4096, 7168, expected_m=s.tok_e)
    assert m.kernel == masked_kernel


@pytest.mark.parametrize("e,t,k,kd,flags,regime", [(30, 100, 4, 448, 0, "all"), (100, 400, 4, 448, 0, "all"),
                                                   (100, 600, 4, 448, 0, "tail"),
                                                   (24, 60, 4, 192, "combine", "all"), (3, 5, 2, 64, 0, "all"),
                                                   (1000, 2100, 8, 64, 0, "none")])
def test_cut_units_match_the_oracle(e, t, k, kd, flags, regime):
    """N=512 (two 256-channel groups), 16-row blocks: a call with at most 304 (row block, group) units cuts every
    unit into k-ranges summed in part order (K chunks 7: parts of 1/2 chunks; 3 chunks: three parts; 1 chunk: one
    part), one with at most 2048 units cuts its last 304 (286 and 398 units here), a larger one none; all match the
    oracle and repeat bit-identically."""
    n, bm = 512, 16
    rng = np.random.default_rng(700 + e + t)
    ids = distinct_topk(rng, t, e, k)
    counts = np.bincount(ids.reshape(-1), minlength=e)
    units = int(np.sum(-(-counts // bm))) * (n // 256)
    assert regime == ("all" if units <= 304 else "tail" if units <= 2048 else "none")
    comb = flags == "combine"
    a = random_acts(rng, t * k if comb else t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    w = rng.uniform(0, 1, size=(t, k)).astype(np.float32) if comb else None
    y = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n, a_per_routed_row=comb)
    f = M.FLAG_COMBINE if comb else 0
    runs = [_indexed_run(a, qw, sc, ids, bm, flags=f, weights=w, a_per_row=comb) for _ in range(3)]
    if comb:
        assert_close(runs[0], O.combine(y, w), f"cut units e={e} t={t} combine", slack=combine_slack(y, w))
    else:
        assert_close(runs[0], y, f"cut units e={e} t={t}")
    for r in runs[1:]:
        assert np.array_equal(r, runs[0])


@pytest.mark.parametrize("flags", [0, 1])
def test_masked_split_matches_oracle(flags):
    """expected_m in 24..127: the masked call splits per expert, experts with at most 32 rows on the decode kernel
    and the others on the tcgen05 kernel (two launches over the same 3-D input, each expert's rows read in place);
    counts around 32 and the 192-row block edges, an expert without rows, NaN past each count (never read); two
    calls are bit-identical."""
    rng = np.random.default_rng(870 + flags)
    counts = [0, 1, 31, 32, 33, 64, 191, 192, 193, 7, 250]
    e, kd, n, max_m = len(counts), 256, 512, 256
    ids = ids_from_counts(rng, counts)
    t = ids.shape[0]
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    masked_m, mrows = O.masked_layout(ids, e, max_m)
    a3 = O.gather_rows(a, mrows.reshape(-1), 1).reshape(e, max_m, kd)
    for ex in range(e):
        a3[ex, masked_m[ex]:] = 0x7FC0
    pw = prepare_dev(qw, sc, 2 if flags else 1, DEV)
    ws = M.workspace(M.LAYOUT_MASKED, t, 1, e, n, kd, 0, 0, DEV)
    assert M.plan(M.LAYOUT_MASKED, t, 1, e, n, kd, expected_m=40).kernel == M.KERNEL_SPLIT
    before = M.launch_count()
    outs = [dev_to_bits(M.masked(bits_to_dev(a3, DEV), i32_to_dev(masked_m, DEV), 40, pw, ws, flags=flags))
            for _ in range(2)]
    assert M.launch_count() - before == 4   # decode + tcgen05 per call
    assert M.get_device_error(ws) == 0
    y = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n)
    ref = O.swiglu(y) if flags else y
    valid = mrows.reshape(-1) >= 0
    assert_close(outs[0][valid], ref[mrows.reshape(-1)[valid]], f"masked split flags={flags}")
    assert np.array_equal(outs[0][valid], outs[1][valid])


SPLIT_COUNTS = [1, 5, 31, 32, 33, 0, 64, 191, 192, 193, 400, 2]


@pytest.mark.parametrize("counts", [SPLIT_COUNTS, [3, 7, 32, 0, 12], [33, 200, 385], [224, 225, 416, 384, 40]])
@pytest.mark.parametrize("block_m", [16, 20, 32])
def test_split_matches_oracle(counts, block_m):
    """FLAG_SPLIT: experts above 32 rows on the tcgen05 kernel (blocks of up to 192 of their rows), the others on
    the decode kernel, and so are the rows of a hot expert past its last full 192-row block when they are at
    most 32 (224, 416: exactly 32; 225: 33 stay on the tcgen05 kernel) and start on a decode block boundary
    (block_m 20: never, everything of a hot expert stays); rows around 32 and the 192-row block edges, no hot
    expert, only hot experts; repeats are bit-identical."""
    rng = np.random.default_rng(800 + sum(counts) + block_m)
    e, kd, n = len(counts), 256, 512
    ids = ids_from_counts(rng, counts)
    a = random_acts(rng, ids.shape[0], kd)
    qw, sc = random_weights(rng, e, n, kd)
    ref = O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), n)
    runs = [_indexed_run(a, qw, sc, ids, block_m, flags=M.FLAG_SPLIT) for _ in range(2)]
    assert_close(runs[0], ref, f"split bm={block_m} counts={counts}")
    assert np.array_equal(runs[0], runs[1])


def test_split_swiglu_out_sorted_and_rows_per_routed_row():
    """SwiGLU into sorted slots (the FFN's gate_up) and A with one row per routed row, top-4 routing."""
    rng = np.random.default_rng(811)
    e, t, k, kd, inter = 40, 300, 4, 192, 256
    # skewed routing: experts 0-2 take 200 rows each, the other 37 about 16 each
    ids = np.stack([np.concatenate([rng.permutation(3)[:2], 3 + rng.permutation(e - 3)[:2]]) for _ in range(t)])
    ids = ids.astype(np.int32)
    qw, sc = random_weights(rng, e, 2 * inter, kd)
    a = random_acts(rng, t, kd)
    pw = prepare_dev(qw, sc, M.MODE_GATE_UP, DEV)
    f = M.FLAG_SPLIT | M.FLAG_SWIGLU | M.FLAG_OUT_SORTED
    ws = M.workspace(M.LAYOUT_INDEXED, t, k, e, pw.n, pw.k, 32, f, DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, 32, ws)
    out = M.indexed(bits_to_dev(a, DEV), pw, s_ids, e_ids, npp, t, k, 32, ws, flags=f)
    assert M.get_device_error(ws) == 0
    h = O.swiglu(O.indexed_gemm(a, ids, lambda x: (qw[x], sc[x]), 2 * inter))
    slots = s_ids.cpu().numpy()[: int(npp.item())]
    valid = slots < t * k
    assert_close(dev_to_bits(out)[: slots.size][valid], h[slots[valid]], "split swiglu out_sorted")
    # A with one row per routed row (the down projection's input, without the combine)
    qw2, sc2 = random_weights(rng, e, 256, kd)
    a2 = random_acts(rng, t * k, kd)
    y2 = _indexed_run(a2, qw2, sc2, ids, 32, flags=M.FLAG_SPLIT, a_per_row=True)
    assert_close(y2, O.indexed_gemm(a2, ids, lambda x: (qw2[x], sc2[x]), 256, a_per_routed_row=True),
                 "split a per routed row")


def test_split_rejects_combine_sorted_input_and_prefill_blocks():
    rng = np.random.default_rng(812)
    qw, sc = random_weights(rng, 3, 256, 64)
    pw = prepare_dev(qw, sc, 1, DEV)
    ids = i32_to_dev(np.array([[0], [1], [2], [1]], dtype=np.int32), DEV)
    for bm, f in [(32, M.FLAG_SPLIT | M.FLAG_COMBINE | M.FLAG_A_PER_ROW), (32, M.FLAG_SPLIT | M.FLAG_A_SORTED),
                  (64, M.FLAG_SPLIT)]:
        with pytest.raises((M.MoeW4A16Error, ValueError)):
            ws = M.workspace(M.LAYOUT_INDEXED, 4, 1, 3, 256, 64, bm, f & ~M.FLAG_A_SORTED, DEV)
            s_ids, e_ids, npp, _ = M.align(ids, 3, bm, ws)
            a_rows = s_ids.numel() if f & M.FLAG_A_SORTED else 4
            w = torch.ones((4, 1), dtype=torch.float32, device=DEV)
            M.indexed(torch.zeros((a_rows, 64), dtype=torch.bfloat16, device=DEV), pw, s_ids, e_ids, npp, 4, 1, bm,
                      ws, flags=f, topk_weights=w if f & M.FLAG_COMBINE else None)
