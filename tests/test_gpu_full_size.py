"""GPU parity at the full workload sizes, in the launch configuration the benchmark times.

Each test builds the benchmark's own arm for a workload (same synthetic inputs,
same plan, same sequence of library calls), runs one step, and compares
outputs with the oracle:

* the 64-token, 8-expert indexed GEMM: every output element;
* decode gate_up, 384 experts, top-8 skewed (indexed and masked layouts),
  at N=4096 and at one 8-way tensor-parallel shard's N=512: every routed
  row of four experts (hottest, median, coldest active, and the expert of
  token 0) on a sample of output channels;
* down + top-8 combine at 128 tokens (decode kernel) and at 8192 tokens with
  K = 256 (one tensor-parallel rank, tcgen05 kernel): 16 tokens on a channel
  sample;
* prefill FFN, 8192 tokens (indexed and contiguous layouts; and the indexed
  layout at the tensor-parallel shard's intermediate 256): the SwiGLU rows
  of every routed row of token 0's eight experts, all intermediate channels,
  then token 0's combined output on a channel sample;
* the gate_up schedule sweep, 16..16384 tokens, uniform and Zipf skew:
  three experts per point on a channel sample.

Weights are generated once per (shape, mode) and kept on the device across
tests. The oracle computes only the sampled outputs, from its own
dequantisation of the same seeded logical weights.
"""

import functools

import numpy as np
import pytest
import torch

import oracle as O
import synth as S
from gpu_util import assert_close, combine_slack, dev_to_bits

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    M = pytest.importorskip("w4a16_int4_mixture_grouped_gb300")
    import bench as B
    DEV = torch.device("cuda", 0)
else:
    M = B = DEV = None

_WEIGHTS = {}


def _cached_upload(wl, which, mode, dev):
    n, k = wl.gemm_shape(which)
    key = (wl.seed, which, n, k, wl.num_experts, mode)
    if key not in _WEIGHTS:
        _WEIGHTS[key] = _orig_upload(wl, which, mode, dev)
    return _WEIGHTS[key]


_orig_upload = B.upload_weights if B is not None else None


@pytest.fixture(scope="module", autouse=True)
def _share_weights():
    B.upload_weights = _cached_upload
    yield
    B.upload_weights = _orig_upload
    _WEIGHTS.clear()
    torch.cuda.empty_cache()


def _arm(name):
    wl, layout = B.resolve(name)
    return B.OurArm(wl, layout, DEV), wl


@functools.lru_cache(maxsize=64)
def _weights_cpu(wl_key, which, e):
    wl = S.get_workload(wl_key)
    return S.expert_weights(wl, which, e)


def _dequant_channels(wl, which, e, chans):
    qw, sc = _weights_cpu(wl.name, which, int(e))
    return O.dequant(O.unpack_int4(qw[chans]), sc[chans])


def _channels(n, count, seed):
    rng = np.random.default_rng(seed)
    c = np.unique(np.concatenate([[0, n - 1], rng.choice(n, size=count, replace=False)]))
    return c.astype(np.int64)


def _rows_of(ids, e):
    return np.nonzero(ids.reshape(-1) == e)[0]


def _gpu_rows(out, rows, chans=None):
    t = out[torch.from_numpy(np.asarray(rows, dtype=np.int64)).to(out.device)]
    if chans is not None:
        t = t[:, torch.from_numpy(chans).to(out.device)]
    return dev_to_bits(t)


def test_tiny_indexed_every_element():
    arm, wl = _arm("tiny_indexed")
    out = arm.step()
    torch.cuda.synchronize()
    n, _ = wl.gemm_shape("w1")
    ref = O.indexed_gemm(arm.a_np, arm.ids_np, lambda e: S.expert_weights(wl, "w1", e), n)
    assert_close(dev_to_bits(out), ref, "tiny indexed, full output")


def _sample_experts(counts, ids):
    active = np.nonzero(counts)[0]
    by_count = active[np.argsort(counts[active], kind="stable")]
    picks = [by_count[-1], by_count[len(by_count) // 2], by_count[0], ids[0, 0]]
    return list(dict.fromkeys(int(e) for e in picks))


@pytest.mark.parametrize("name", ["decode_gate_up", "decode_gate_up_masked", "tp8_decode_gate_up",
                                  "tp8_decode_gate_up_masked"])
def test_decode_gate_up_sampled(name):
    arm, wl = _arm(name)
    out = arm.step()
    torch.cuda.synchronize()
    n, _ = wl.gemm_shape("w1")
    k = wl.top_k
    chans = _channels(n, 384, 11)
    if arm.layout == "masked":
        masked_m, row_ids = O.masked_layout(arm.ids_np, wl.num_experts, wl.max_m)
    for e in _sample_experts(arm.counts, arm.ids_np):
        flat = _rows_of(arm.ids_np, e)
        ref = O.gemm_rows(arm.a_np[flat // k], _dequant_channels(wl, "w1", e, chans))
        if arm.layout == "masked":
            assert masked_m[e] == flat.size and np.array_equal(row_ids[e, : flat.size], flat)
            got = _gpu_rows(out, e * wl.max_m + np.arange(flat.size), chans)
        else:
            got = _gpu_rows(out, flat, chans)
        assert_close(got, ref, f"{name} expert {e} ({flat.size} rows)")


@pytest.mark.parametrize("name", ["decode_down_combine", "tp8_prefill_down_combine"])
def test_down_combine_sampled(name):
    arm, wl = _arm(name)
    out = arm.step()
    torch.cuda.synchronize()
    n, _ = wl.gemm_shape("w2")
    k = wl.top_k
    chans = _channels(n, 512, 12)
    tokens = np.unique(np.concatenate([[0, wl.num_tokens - 1],
                                       np.random.default_rng(13).choice(wl.num_tokens, 14, replace=False)]))
    y = np.zeros((tokens.size * k, chans.size), dtype=np.uint16)
    for i, t in enumerate(tokens):
        for j in range(k):
            e = int(arm.ids_np[t, j])
            y[i * k + j] = O.gemm_rows(arm.a_np[t * k + j][None, :], _dequant_channels(wl, "w2", e, chans))[0]
    ref = O.combine(y, arm.wts_np[tokens])
    slack = combine_slack(y, arm.wts_np[tokens])
    assert_close(_gpu_rows(out, tokens, chans), ref, f"{name}", slack=slack)


@functools.lru_cache(maxsize=2)
def _prefill_token0_reference(base):
    """Oracle SwiGLU rows of every routed row of token 0's experts, and token 0's combined output."""
    wl = S.get_workload(base)
    ids, wts = S.routing(wl)
    a = S.activations(wl.seed, wl.num_tokens, wl.hidden)
    k = wl.top_k
    n2, _ = wl.gemm_shape("w2")
    chans = _channels(n2, 1024, 14)
    h_rows = {}
    y2 = np.zeros((k, chans.size), dtype=np.uint16)
    for j in range(k):
        e = int(ids[0, j])
        flat = _rows_of(ids, e)
        qw, sc = _weights_cpu(wl.name, "w1", e)
        h = O.swiglu(O.gemm_rows(a[flat // k], O.dequant_expert(qw, sc)))
        h_rows[e] = (flat, h)
        h0 = h[np.searchsorted(flat, j)]          # token 0's row j has flat id j
        y2[j] = O.gemm_rows(h0[None, :], _dequant_channels(wl, "w2", e, chans))[0]
    return h_rows, chans, O.combine(y2, wts[:1]), combine_slack(y2, wts[:1])


@pytest.mark.parametrize("name", ["prefill_ffn", "prefill_ffn_contiguous", "tp8_prefill_ffn"])
def test_prefill_ffn_sampled(name):
    arm, wl = _arm(name)
    f = arm.ffn
    route = f.route(arm.ids)
    h = f.gate_up(f.gate_up_input(arm.a, route), route)
    out = f.down(h, route, arm.wts, arm.out)
    torch.cuda.synchronize()
    # row of h holding each flat id: sorted_ids slots (indexed) or contiguous-layout rows
    used = int(route[2].item())                  # valid slots / layout rows: num_post_padded
    slot_ids = (route[0] if arm.layout == "indexed" else route[4])[:used].cpu().numpy().astype(np.int64)
    where = np.full(wl.rows, -1, dtype=np.int64)
    valid = (slot_ids >= 0) & (slot_ids < wl.rows)
    where[slot_ids[valid]] = np.nonzero(valid)[0]
    h_rows, chans, ref0, slack0 = _prefill_token0_reference(wl.name)
    for e, (flat, href) in h_rows.items():
        assert (where[flat] >= 0).all()
        assert_close(_gpu_rows(h, where[flat]), href, f"{name} SwiGLU rows of expert {e}")
    assert_close(_gpu_rows(out, [0], chans), ref0, f"{name} token 0 combined output", slack=slack0)


@pytest.mark.parametrize("skew", ["uniform", "zipf"])
@pytest.mark.parametrize("tokens", S.SWEEP_TOKENS)
def test_sweep_gate_up_sampled(tokens, skew):
    arm, wl = _arm(f"sweep_gate_up_t{tokens}_{skew}")
    out = arm.step()
    torch.cuda.synchronize()
    n, _ = wl.gemm_shape("w1")
    k = wl.top_k
    chans = _channels(n, 256, tokens)
    for e in _sample_experts(arm.counts, arm.ids_np)[:3]:
        flat = _rows_of(arm.ids_np, e)
        ref = O.gemm_rows(arm.a_np[flat // k], _dequant_channels(wl, "w1", e, chans))
        assert_close(_gpu_rows(out, flat, chans), ref, f"sweep t={tokens} {skew} expert {e} ({flat.size} rows)")
