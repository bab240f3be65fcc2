"""GPU parity at the full workload sizes, in the launch configuration the benchmark times.

Each test builds the benchmark's own arm for a workload (same synthetic inputs,
same plan, same sequence of library calls), runs one step and compares with
the oracle, covering every routed row of every workload:

* every output element: the 64-token, 8-expert GEMM; decode gate_up at 64
  tokens over 384 experts, skewed (indexed and masked, and one 8-way
  tensor-parallel rank's N = 512); decode down + top-8 combine at 128 tokens
  (every token, every channel); the schedule-sweep points with 16, 128 and 512
  tokens under uniform and Zipf routing;
* every routed row on a channel sample holding channels of every 256-channel
  work-unit group: the sweep points with 1536, 4096 and 16384 tokens, and the
  prefill FFN's gate_up + SwiGLU (indexed, contiguous, the tensor-parallel
  rank) on intermediate channels of every group;
* every token on a channel sample of every group: the prefill FFN's down +
  combine call (indexed, contiguous, tensor-parallel rank), made exactly as
  the FFN step makes it, on a synthetic SwiGLU output placed by the oracle's
  routing layout (whose GPU counterpart is checked bit-exact first); the
  tensor-parallel rank's down + combine workload;
* the whole FFN chain on token 0 (gate_up -> SwiGLU -> down -> combine, every
  output channel).

The oracle references are computed per expert in a spawn process pool
(tests/full_size_ref.py: the oracle's dequantisation tabulated over its whole
domain, then its GEMM, SwiGLU and combine).
"""

import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import full_size_ref as F
import oracle as O
import synth as S
from gpu_util import assert_close, combine_slack, dev_to_bits, bits_to_dev

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    M = pytest.importorskip("w4a16_int4_mixture_grouped_gb300")
    import bench as B
    DEV = torch.device("cuda", 0)
else:
    M = B = DEV = None

FULL_SWEEP = (16, 128, 512)
SAMPLED_SWEEP = (1536, 4096, 16384)


@pytest.fixture(scope="module", autouse=True)
def _release_weights():
    """The benchmark caches generated and prepared weights per process; free them after this module."""
    yield
    B.release_weights()


@pytest.fixture(scope="module")
def pool():
    p = F.make_pool()
    yield p
    p.close()
    p.join()


@pytest.fixture(scope="module")
def files():
    """Activation matrices written once as .npy files that the pool's processes map."""
    d = tempfile.mkdtemp(prefix="moe_full_size_")
    saved = {}

    def put(key, arr):
        if key not in saved:
            path = os.path.join(d, f"{key}.npy")
            np.save(path, np.ascontiguousarray(arr))
            saved[key] = path
        return saved[key]

    yield put
    shutil.rmtree(d, ignore_errors=True)


def _arm(name):
    wl, layout = B.resolve(name)
    return B.OurArm(wl, layout, DEV), wl


def _take(out, rows, chans=None):
    """GPU output rows (and channels), as BF16 bits on the host."""
    t = out[torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(out.device)]
    if chans is not None:
        t = t[:, torch.from_numpy(np.asarray(chans, dtype=np.int64)).to(out.device)]
    return dev_to_bits(t)


def _assemble(results, key, rows_e, n_rows, width):
    """Oracle rows per expert -> [n_rows, width] in flat-id order."""
    ref = np.zeros((n_rows, width), dtype=np.uint16)
    filled = np.zeros(n_rows, dtype=bool)
    for e, rows in enumerate(rows_e):
        if rows.size:
            ref[rows] = results[e][key]
            filled[rows] = True
    assert filled.all()
    return ref


def _layout_rows(arm, route):
    """Row of the FFN's intermediate tensor holding each flat id (sorted slot or contiguous row), from the
    GPU's routing layout after checking it bit-exact against the oracle's."""
    wl = arm.wl
    used = int(route[2].item())
    if arm.layout == "indexed":
        s_ref, e_ref, npp_ref = O.align(arm.ids_np, wl.num_experts, arm.ffn.block_m)
        assert used == npp_ref
        assert np.array_equal(route[0][:used].cpu().numpy(), s_ref)
        assert np.array_equal(route[1][: used // arm.ffn.block_m].cpu().numpy(), e_ref)
        slot_ids = s_ref.astype(np.int64)
    else:
        row_ref, m_ref = O.contiguous_layout(arm.ids_np, wl.num_experts)
        assert used == row_ref.size
        assert np.array_equal(route[3][:used].cpu().numpy(), m_ref)
        assert np.array_equal(route[4][:used].cpu().numpy(), row_ref)
        assert (route[3][used:].cpu().numpy() == -1).all() and (route[4][used:].cpu().numpy() == -1).all()
        slot_ids = row_ref.astype(np.int64)
    where = np.full(wl.rows, -1, dtype=np.int64)
    valid = (slot_ids >= 0) & (slot_ids < wl.rows)
    where[slot_ids[valid]] = np.nonzero(valid)[0]
    assert (where >= 0).all()
    return where, used


# ---------------------------------------------------------------------------------------------------------
# the tiny GEMM
# ---------------------------------------------------------------------------------------------------------

def test_tiny_indexed_every_element():
    arm, wl = _arm("tiny_indexed")
    out = arm.step()
    torch.cuda.synchronize()
    n, _ = wl.gemm_shape("w1")
    ref = O.indexed_gemm(arm.a_np, arm.ids_np, lambda e: S.expert_weights(wl, "w1", e), n)
    assert_close(dev_to_bits(out), ref, "tiny indexed, full output")


# ---------------------------------------------------------------------------------------------------------
# gate_up weights (hidden 7168 -> 4096): decode, sweep, prefill FFN gate_up + SwiGLU
# ---------------------------------------------------------------------------------------------------------

def _gate_up_outputs(name, chans):
    """GPU gate_up output of a single-GEMM workload in flat-id order (all channels or `chans`)."""
    arm, wl = _arm(name)
    out = arm.step()
    torch.cuda.synchronize()
    flat = np.arange(wl.rows)
    if arm.layout == "masked":
        masked_m, row_ids = O.masked_layout(arm.ids_np, wl.num_experts, wl.max_m)
        rows = np.empty(wl.rows, dtype=np.int64)
        for e in range(wl.num_experts):
            rows[row_ids[e, : masked_m[e]]] = e * wl.max_m + np.arange(masked_m[e])
        got = _take(out, rows, chans)
    else:
        got = _take(out, flat, chans)
    res = (arm.ids_np, arm.a_np, got)
    del arm, out
    torch.cuda.empty_cache()
    return res


@pytest.fixture(scope="module")
def gate_up_family(pool, files):
    """One pass over the 384 experts of the shared gate_up weights: the GPU outputs of every workload that
    uses them, and the oracle's rows for every routed row (all channels or the channel sample)."""
    n, k = 4096, 7168
    chans = F.group_channels(n, 256, 4, 101)                 # every 256-channel work-unit group
    ichans = F.group_channels(n // 2, 128, 4, 102)           # intermediate channels of every gate/up group
    gpu, cases = {}, []                                      # cases: (oracle key, ids, activations, chans, kind)
    for name in ("decode_gate_up", "decode_gate_up_masked"):
        ids, a, got = _gate_up_outputs(name, None)
        gpu[name] = ("decode_gate_up", got)
    cases.append(("decode_gate_up", ids, a, None, "gemm"))
    for t in FULL_SWEEP + SAMPLED_SWEEP:
        for skew in ("uniform", "zipf"):
            name = f"sweep_gate_up_t{t}_{skew}"
            ch = None if t in FULL_SWEEP else chans
            ids, a, got = _gate_up_outputs(name, ch)
            gpu[name] = (name, got)
            cases.append((name, ids, a, ch, "gemm"))
    for name in ("prefill_ffn", "prefill_ffn_contiguous"):
        arm, wl = _arm(name)
        f = arm.ffn
        route = f.route(arm.ids)
        h = f.gate_up(f.gate_up_input(arm.a, route), route)
        torch.cuda.synchronize()
        where, _ = _layout_rows(arm, route)
        gpu[name] = ("prefill_ffn", _take(h, where, ichans))
        ids, a = arm.ids_np, arm.a_np
        del arm, f, route, h
        torch.cuda.empty_cache()
    cases.append(("prefill_ffn", ids, a, ichans, "swiglu"))

    specs = []
    per_case = [(key, F.rows_by_expert(ids, 384), ids.size, ch, kind) for key, ids, a, ch, kind in cases]
    for e in range(384):
        tasks = []
        for (key, ids, a, ch, kind), (_, rows_e, _, _, _) in zip(cases, per_case):
            if rows_e[e].size:
                tasks.append((key, (files(key + "_a", a), rows_e[e] // ids.shape[1]), ch, kind))
        specs.append(("decode_gate_up", "w1", e, tasks))
    results = F.run_jobs(pool, specs)
    refs = {}
    for key, rows_e, n_rows, ch, kind in per_case:
        width = n if ch is None else ch.size
        refs[key] = _assemble(results, key, rows_e, n_rows, width)
    return gpu, refs


@pytest.mark.parametrize("name", ["decode_gate_up", "decode_gate_up_masked"]
                         + [f"sweep_gate_up_t{t}_{s}" for t in FULL_SWEEP for s in ("uniform", "zipf")])
def test_gate_up_every_element(gate_up_family, name):
    gpu, refs = gate_up_family
    key, got = gpu[name]
    assert got.shape[1] == 4096
    assert_close(got, refs[key], f"{name}: every routed row, every channel")


@pytest.mark.parametrize("name", [f"sweep_gate_up_t{t}_{s}" for t in SAMPLED_SWEEP for s in ("uniform", "zipf")])
def test_gate_up_every_row_channel_sample(gate_up_family, name):
    gpu, refs = gate_up_family
    key, got = gpu[name]
    assert_close(got, refs[key], f"{name}: every routed row, channels of every group")


@pytest.mark.parametrize("name", ["prefill_ffn", "prefill_ffn_contiguous"])
def test_prefill_ffn_swiglu_every_row(gate_up_family, name):
    gpu, refs = gate_up_family
    key, got = gpu[name]
    assert_close(got, refs[key], f"{name}: SwiGLU of every routed row, intermediate channels of every group")


# ---------------------------------------------------------------------------------------------------------
# down weights (2048 -> 7168): decode down + combine, prefill FFN down + combine
# ---------------------------------------------------------------------------------------------------------

def _down_probe(name, chans):
    """The FFN step's down + combine call on a synthetic SwiGLU output (every routed row's input drawn by
    synth.down_input and placed by the oracle's layout), output channels `chans` of every token."""
    arm, wl = _arm(name)
    f = arm.ffn
    route = f.route(arm.ids)
    where, _ = _layout_rows(arm, route)
    h_flat = S.down_input(wl)
    # as many rows as the gate_up call's output: one per sorted slot, or per contiguous-layout row
    h_in = np.zeros((route[0].numel(), wl.intermediate), dtype=np.uint16)
    h_in[where] = h_flat
    out = f.down(bits_to_dev(h_in, DEV), route, arm.wts, arm.out)
    torch.cuda.synchronize()
    got = _take(out, np.arange(wl.num_tokens), chans)
    res = (arm.ids_np, arm.wts_np, h_flat, got)
    del arm, f, route, out
    torch.cuda.empty_cache()
    return res


def _down_refs(pool, files, weights_wl, cases, n):
    """Oracle down rows per case (key, ids, per-routed-row input, chans) in one pass over the experts."""
    per_case = [(key, F.rows_by_expert(ids, 384), ids.size, ch) for key, ids, _, ch in cases]
    specs = []
    for e in range(384):
        tasks = []
        for (key, ids, h, ch), (_, rows_e, _, _) in zip(cases, per_case):
            if rows_e[e].size:
                tasks.append((key, (files(key + "_h", h), rows_e[e]), ch, "gemm"))
        specs.append((weights_wl, "w2", e, tasks))
    results = F.run_jobs(pool, specs)
    return {key: _assemble(results, key, rows_e, n_rows, n if ch is None else ch.size)
            for key, rows_e, n_rows, ch in per_case}


@pytest.fixture(scope="module")
def down_family(pool, files):
    n = 7168
    chans = F.group_channels(n, 256, 3, 201)
    gpu, cases = {}, []
    arm, wl = _arm("decode_down_combine")
    out = arm.step()
    torch.cuda.synchronize()
    gpu["decode_down_combine"] = ("decode_down_combine", dev_to_bits(out))
    cases.append(("decode_down_combine", arm.ids_np, arm.a_np, None))
    wts = {"decode_down_combine": arm.wts_np}
    del arm, out
    torch.cuda.empty_cache()
    for name in ("prefill_ffn", "prefill_ffn_contiguous"):
        ids, w, h, got = _down_probe(name, chans)
        gpu[name] = ("prefill_ffn", got)
    cases.append(("prefill_ffn", ids, h, chans))
    wts["prefill_ffn"] = w
    ys = _down_refs(pool, files, "decode_down_combine", cases, n)
    refs = {key: (O.combine(y, wts[key]), combine_slack(y, wts[key])) for key, y in ys.items()}
    return gpu, refs


def test_decode_down_combine_every_element(down_family):
    gpu, refs = down_family
    key, got = gpu["decode_down_combine"]
    ref, slack = refs[key]
    assert got.shape == (128, 7168)
    assert_close(got, ref, "decode down + combine: every token, every channel", slack=slack)


@pytest.mark.parametrize("name", ["prefill_ffn", "prefill_ffn_contiguous"])
def test_prefill_ffn_down_combine_every_token(down_family, name):
    gpu, refs = down_family
    key, got = gpu[name]
    ref, slack = refs[key]
    assert got.shape[0] == 8192
    assert_close(got, ref, f"{name} down + combine: every token, channels of every group", slack=slack)


# ---------------------------------------------------------------------------------------------------------
# one 8-way tensor-parallel rank (intermediate 256)
# ---------------------------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tp8_family(pool, files):
    gpu, cases = {}, []
    for name in ("tp8_decode_gate_up", "tp8_decode_gate_up_masked"):
        ids, a, got = _gate_up_outputs(name, None)
        gpu[name] = ("tp8_decode_gate_up", got)
    cases.append(("tp8_decode_gate_up", ids, a, None, "gemm"))
    ichans = F.group_channels(256, 128, 16, 301)
    arm, wl = _arm("tp8_prefill_ffn")
    f = arm.ffn
    route = f.route(arm.ids)
    h = f.gate_up(f.gate_up_input(arm.a, route), route)
    torch.cuda.synchronize()
    where, _ = _layout_rows(arm, route)
    gpu["tp8_prefill_ffn"] = ("tp8_prefill_ffn", _take(h, where, ichans))
    cases.append(("tp8_prefill_ffn", arm.ids_np, arm.a_np, ichans, "swiglu"))
    del arm, f, route, h
    torch.cuda.empty_cache()
    per_case = [(key, F.rows_by_expert(ids, 384), ids.size, ch) for key, ids, _, ch, _ in cases]
    specs = []
    for e in range(384):
        tasks = []
        for (key, ids, a, ch, kind), (_, rows_e, _, _) in zip(cases, per_case):
            if rows_e[e].size:
                tasks.append((key, (files(key + "_a", a), rows_e[e] // ids.shape[1]), ch, kind))
        specs.append(("tp8_decode_gate_up", "w1", e, tasks))
    results = F.run_jobs(pool, specs)
    refs = {key: _assemble(results, key, rows_e, n_rows, 512 if ch is None else ch.size)
            for key, rows_e, n_rows, ch in per_case}

    # down (256 -> 7168): the FFN's down + combine call on a synthetic input, and the down-only workload
    chans = F.group_channels(7168, 256, 3, 302)
    down_cases, wts = [], {}
    ids, w, hflat, got = _down_probe("tp8_prefill_ffn", chans)
    gpu["tp8_prefill_ffn_down"] = ("tp8_prefill_ffn_down", got)
    down_cases.append(("tp8_prefill_ffn_down", ids, hflat, chans))
    wts["tp8_prefill_ffn_down"] = w
    arm, wl = _arm("tp8_prefill_down_combine")
    out = arm.step()
    torch.cuda.synchronize()
    gpu["tp8_prefill_down_combine"] = ("tp8_prefill_down_combine", _take(out, np.arange(wl.num_tokens), chans))
    down_cases.append(("tp8_prefill_down_combine", arm.ids_np, arm.a_np, chans))
    wts["tp8_prefill_down_combine"] = arm.wts_np
    del arm, out
    torch.cuda.empty_cache()
    ys = _down_refs(pool, files, "tp8_prefill_down_combine", down_cases, 7168)
    for key, y in ys.items():
        refs[key] = (O.combine(y, wts[key]), combine_slack(y, wts[key]))
    return gpu, refs


@pytest.mark.parametrize("name", ["tp8_decode_gate_up", "tp8_decode_gate_up_masked"])
def test_tp8_decode_gate_up_every_element(tp8_family, name):
    gpu, refs = tp8_family
    key, got = gpu[name]
    assert got.shape[1] == 512
    assert_close(got, refs[key], f"{name}: every routed row, every channel")


def test_tp8_prefill_ffn_swiglu_every_row(tp8_family):
    gpu, refs = tp8_family
    key, got = gpu["tp8_prefill_ffn"]
    assert_close(got, refs[key], "TP8 prefill FFN SwiGLU: every routed row, intermediate channels of both groups")


@pytest.mark.parametrize("name", ["tp8_prefill_ffn_down", "tp8_prefill_down_combine"])
def test_tp8_down_combine_every_token(tp8_family, name):
    gpu, refs = tp8_family
    key, got = gpu[name]
    ref, slack = refs[key]
    assert_close(got, ref, f"{name}: every token, channels of every group", slack=slack)


# ---------------------------------------------------------------------------------------------------------
# the FFN chain end to end
# ---------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["prefill_ffn", "prefill_ffn_contiguous", "tp8_prefill_ffn"])
def test_prefill_ffn_chain_token0(name):
    """gate_up -> SwiGLU -> down -> combine through the FFN step, token 0 against the oracle's own chain
    (every SwiGLU row of token 0's experts, every output channel of token 0)."""
    arm, wl = _arm(name)
    f = arm.ffn
    out = arm.step()
    torch.cuda.synchronize()
    k = wl.top_k
    ids = arm.ids_np
    rows_e = F.rows_by_expert(ids, wl.num_experts)
    y2 = np.zeros((k, wl.hidden), dtype=np.uint16)
    for j in range(k):
        e = int(ids[0, j])
        flat = rows_e[e]
        h = O.swiglu(O.gemm_rows(arm.a_np[flat // k], F.dequant_tabulated(*S.expert_weights(wl, "w1", e))))
        h0 = h[np.searchsorted(flat, j)]               # token 0's row j has flat id j
        y2[j] = O.gemm_rows(h0[None, :], F.dequant_tabulated(*S.expert_weights(wl, "w2", e)))[0]
    ref = O.combine(y2, arm.wts_np[:1])
    assert_close(_take(out, [0]), ref, f"{name} token 0, every channel", slack=combine_slack(y2, arm.wts_np[:1]))
    del arm, f, out
    torch.cuda.empty_cache()
