"""The hot path captured in a CUDA graph replays bit-identically to eager launches.

Every step of a MoE layer (routing layout, gathers, both GEMMs with their
epilogues, the combine) is asynchronous on the caller's stream with no host
synchronisation, and every counter the kernels use internally is back at zero
when a call ends, so the whole layer can be captured once and replayed.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits_to_dev, dev_to_bits, distinct_topk, i32_to_dev, prepare_dev, random_acts, random_weights

pytestmark = pytest.mark.gpu

M = pytest.importorskip("w4a16_int4_mixture_grouped_gb300") if torch.cuda.is_available() else None
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _layer(t, e, k, hidden, inter, layout, block_m, seed):
    from w4a16_int4_mixture_grouped_gb300.pipeline import MoEFFN
    rng = np.random.default_rng(seed)
    q1, s1 = random_weights(rng, e, 2 * inter, hidden)
    q2, s2 = random_weights(rng, e, hidden, inter)
    w1 = prepare_dev(q1, s1, 2, DEV)
    w2 = prepare_dev(q2, s2, 1, DEV)
    ffn = MoEFFN(w1, w2, t, k, layout=layout, block_m=block_m)
    a = bits_to_dev(random_acts(rng, t, hidden), DEV)
    ids = i32_to_dev(distinct_topk(rng, t, e, k), DEV)
    wts = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
    wts = torch.from_numpy(wts / wts.sum(axis=1, keepdims=True)).to(DEV)
    return ffn, a, ids, wts


@pytest.mark.parametrize("layout,block_m", [("indexed", 16), ("indexed", 32), ("indexed", 192), ("contiguous", None)])
def test_ffn_layer_graph_replay_matches_eager(layout, block_m):
    t, e, k, hidden, inter = 96, 12, 4, 512, 256
    lay = M.LAYOUT_INDEXED if layout == "indexed" else M.LAYOUT_CONTIGUOUS
    ffn, a, ids, wts = _layer(t, e, k, hidden, inter, lay, block_m, 300 + (block_m or 0))
    eager = ffn.forward(a, ids, wts, out=torch.empty((t, hidden), dtype=torch.bfloat16, device=DEV)).clone()
    torch.cuda.synchronize()
    out = torch.empty((t, hidden), dtype=torch.bfloat16, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ffn.forward(a, ids, wts, out=out)          # warm-up on the capture stream (first-call set-up)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ffn.forward(a, ids, wts, out=out)
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(dev_to_bits(out), dev_to_bits(eager))
    for ws in ffn.workspaces:
        assert M.get_device_error(ws) == 0
