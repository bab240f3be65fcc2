"""A pipeline wait that runs out, and the call after it.

Every wait inside the GEMM kernels is bounded (about two seconds by default).
Here the limit is lowered to zero through the library's diagnostic entry
point, so the first wait for data that has not arrived yet gives up at once,
through ordinary timing: nothing in the kernels is changed or broken, and every
awaited copy does arrive. The kernel then takes its abort path (abort flag
raised, copies in flight drained under the default limit, tensor memory
released) and the workspace error word reads MOE_W4A16_ERR_DEVICE_TIMEOUT.
With the limit restored and the workspace zeroed again, the same calls on the
same workspace match the oracle; the tcgen05 launches after the aborted one
also show that it released its tensor memory.
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
TIMEOUT = 6   # MOE_W4A16_ERR_DEVICE_TIMEOUT


def test_wait_limit_rejects_values_above_the_default():
    with pytest.raises(M.MoeW4A16Error) as ex:
        M.set_wait_limit_ns(M.WAIT_LIMIT_NS + 1)
    assert ex.value.status == 1


@pytest.mark.parametrize("block_m,combine", [(16, True), (32, False), (192, False), (192, True)])
def test_timed_out_wait_reports_and_the_next_call_is_correct(block_m, combine):
    rng = np.random.default_rng(1300 + block_m + combine)
    e, t, k, kd, n = 12, 96, 4, 512, 512
    ids = distinct_topk(rng, t, e, k)
    flags = (M.FLAG_COMBINE | M.FLAG_A_PER_ROW) if combine else 0
    a_bits = random_acts(rng, t * k if combine else t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    pw = prepare_dev(qw, sc, 1, DEV)
    w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    wd = torch.from_numpy(w).to(DEV) if combine else None
    a = bits_to_dev(a_bits, DEV)
    ws = M.workspace(M.LAYOUT_INDEXED, t, k, e, n, kd, block_m, flags, DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, block_m, ws)
    torch.cuda.synchronize()
    try:
        M.set_wait_limit_ns(0)
        M.indexed(a, pw, s_ids, e_ids, npp, t, k, block_m, ws, flags=flags, topk_weights=wd)
        code = M.get_device_error(ws)
    finally:
        M.set_wait_limit_ns(M.WAIT_LIMIT_NS)
    assert code == TIMEOUT, f"expected the timed-out wait to be recorded, got error word {code}"
    # recovery: zero the workspace, then the same call on the same workspace, twice
    M.workspace_init(ws)
    y = O.indexed_gemm(a_bits, ids, lambda x: (qw[x], sc[x]), n, a_per_routed_row=combine)
    for _ in range(2):
        out = M.indexed(a, pw, s_ids, e_ids, npp, t, k, block_m, ws, flags=flags, topk_weights=wd)
        assert M.get_device_error(ws) == 0
        if combine:
            assert_close(dev_to_bits(out), O.combine(y, w), "after a timeout, combine", slack=combine_slack(y, w))
        else:
            assert_close(dev_to_bits(out), y, "after a timeout")
