"""moe_w4a16_indexed_noalloc against moe_w4a16_indexed, through the C-ABI.

The no-allocation entry point serves callers that may not allocate device
memory during a call (a pool that forbids side allocations, a runtime with a
device heap fixed at start-up): it runs the decode kernel with the library's
static scratch array. Each case calls it twice in a row (the second call
reuses the scratch the first one left behind) and compares both outputs with
the workspace entry point's output on the same inputs, within the output
tolerance, and checks the scratch's device error word. The calls are also
checked to allocate nothing (free device memory and torch's allocation count
unchanged), and a call is checked to be correct after the scratch was filled
with garbage, as a call that stopped on a device error could leave it.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import (assert_close, bits_to_dev, dev_to_bits, distinct_topk, i32_to_dev, prepare_dev, random_acts,
                      random_weights)

pytestmark = pytest.mark.gpu

M = pytest.importorskip("w4a16_int4_mixture_grouped_gb300") if torch.cuda.is_available() else None
DEV = torch.device("cuda", 0) if torch.cuda.is_available() else None


def _scratch_error(addr: int) -> int:
    code = ctypes.c_int32(-1)
    st = M.lib.moe_w4a16_get_device_error(ctypes.c_void_p(addr), M._stream(DEV), ctypes.byref(code))
    assert st == 0
    return int(code.value)


def _both(a_bits, qw, sc, ids, block_m, mode, flags, weights=None):
    """(workspace entry output, [two no-alloc outputs]) as BF16 bits."""
    t, k = ids.shape
    e = qw.shape[0]
    pw = prepare_dev(qw, sc, mode, DEV)
    ws = M.workspace(M.LAYOUT_INDEXED, t, k, e, pw.n, pw.k, block_m, flags, DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, block_m, ws)
    a = bits_to_dev(a_bits, DEV)
    w = torch.from_numpy(weights).to(DEV) if weights is not None else None
    ref = M.indexed(a, pw, s_ids, e_ids, npp, t, k, block_m, ws, flags=flags, topk_weights=w)
    assert M.get_device_error(ws) == 0
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    # the first call on the device resolves the scratch address; the ones after it allocate nothing
    M.indexed_noalloc(a, pw, s_ids, e_ids, npp, t, k, block_m, flags=flags, topk_weights=w, out=outs[0])
    torch.cuda.synchronize()
    outs[0].fill_(float("nan"))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(DEV)[0]
    allocs0 = torch.cuda.memory_stats(DEV).get("allocation.all.allocated", 0)
    addrs = []
    for out in outs:
        addr = M.indexed_noalloc(a, pw, s_ids, e_ids, npp, t, k, block_m, flags=flags, topk_weights=w, out=out)
        assert addr != 0 and addr % 256 == 0
        assert _scratch_error(addr) == 0
        addrs.append(addr)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(DEV)[0] == free0, "a no-allocation call changed the free device memory"
    assert torch.cuda.memory_stats(DEV).get("allocation.all.allocated", 0) == allocs0
    assert addrs[0] == addrs[1]
    return dev_to_bits(ref), [dev_to_bits(o) for o in outs]


class _DeviceBytes:
    """A raw device range as a torch tensor (no copy), through the CUDA array interface."""

    def __init__(self, addr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (addr, False),
                                         "version": 3}


@pytest.mark.parametrize("block_m", [8, 32])
def test_noalloc_down_combine_matches_indexed(block_m):
    rng = np.random.default_rng(900 + block_m)
    e, t, k, kd, n = 12, 40, 4, 256, 768
    ids = distinct_topk(rng, t, e, k)
    h = random_acts(rng, t * k, kd)
    qw, sc = random_weights(rng, e, n, kd)
    w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    ref, outs = _both(h, qw, sc, ids, block_m, 1, M.FLAG_COMBINE | M.FLAG_A_PER_ROW, w)
    for i, got in enumerate(outs):
        assert_close(got, ref, f"no-alloc combine call {i}")
    exact = O.combine(O.indexed_gemm(h, ids, lambda x: (qw[x], sc[x]), n, a_per_routed_row=True), w)
    assert_close(outs[1], exact, "no-alloc combine vs oracle")


def test_noalloc_gate_up_swiglu_matches_indexed():
    rng = np.random.default_rng(950)
    e, t, k, kd, n = 9, 33, 3, 320, 512
    a = random_acts(rng, t, kd)
    qw, sc = random_weights(rng, e, n, kd)
    ids = distinct_topk(rng, t, e, k)
    ref, outs = _both(a, qw, sc, ids, 16, 2, M.FLAG_SWIGLU)
    for i, got in enumerate(outs):
        assert_close(got, ref, f"no-alloc swiglu call {i}")


def test_noalloc_rejects_oversize_and_prefill_block():
    rng = np.random.default_rng(960)
    e, kd, n = 4, 64, 1024
    qw, sc = random_weights(rng, e, n, kd)
    pw = prepare_dev(qw, sc, 1, DEV)
    t, k = 3200, 8                      # combine staging 3200*8*1024*2 B + partial tiles > 64 MiB
    need = M.workspace_size(M.LAYOUT_INDEXED, t, k, e, n, kd, 16, M.FLAG_COMBINE | M.FLAG_A_PER_ROW)
    assert need > M.STATIC_SCRATCH_BYTES
    dummy_i = torch.zeros(16, dtype=torch.int32, device=DEV)
    a = torch.zeros((t * k, kd), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros((t, n), dtype=torch.bfloat16, device=DEV)
    w = torch.full((t, k), 0.125, dtype=torch.float32, device=DEV)
    with pytest.raises(M.MoeW4A16Error) as ex:
        M.indexed_noalloc(a, pw, dummy_i, dummy_i, dummy_i, t, k, 16, flags=M.FLAG_COMBINE | M.FLAG_A_PER_ROW,
                          topk_weights=w, out=out)
    assert ex.value.status == 9
    with pytest.raises(M.MoeW4A16Error) as ex:
        M.indexed_noalloc(a[:t], pw, dummy_i, dummy_i, dummy_i, t, k, 64, out=out)
    assert ex.value.status == 1
    # the per-expert split would also run the tcgen05 kernel: refused
    with pytest.raises(M.MoeW4A16Error) as ex:
        M.indexed_noalloc(a[:t], pw, dummy_i, dummy_i, dummy_i, t, k, 32, flags=M.FLAG_SPLIT, out=out)
    assert ex.value.status == 1
    # a call within the limit still runs after the rejections
    ids = distinct_topk(rng, 24, e, 2)
    ref, outs = _both(random_acts(rng, 24, kd), qw, sc, ids, 32, 1, 0)
    for i, got in enumerate(outs):
        assert_close(got, ref, f"no-alloc plain call {i}")


def test_noalloc_correct_after_garbage_scratch():
    """Every byte of the static scratch set to 0xFF (counters at -1, as stale as a call stopped by a device
    error could leave them): the next call still matches the workspace entry point and reports no error."""
    rng = np.random.default_rng(970)
    e, t, k, kd, n = 10, 36, 4, 256, 512
    ids = distinct_topk(rng, t, e, k)
    h = random_acts(rng, t * k, kd)
    qw, sc = random_weights(rng, e, n, kd)
    w = rng.uniform(0, 1, size=(t, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    flags = M.FLAG_COMBINE | M.FLAG_A_PER_ROW
    pw = prepare_dev(qw, sc, 1, DEV)
    ws = M.workspace(M.LAYOUT_INDEXED, t, k, e, n, kd, 16, flags, DEV)
    s_ids, e_ids, npp, _ = M.align(i32_to_dev(ids, DEV), e, 16, ws)
    a = bits_to_dev(h, DEV)
    wd = torch.from_numpy(w).to(DEV)
    ref = M.indexed(a, pw, s_ids, e_ids, npp, t, k, 16, ws, flags=flags, topk_weights=wd)
    out = torch.empty_like(ref)
    addr = M.indexed_noalloc(a, pw, s_ids, e_ids, npp, t, k, 16, flags=flags, topk_weights=wd, out=out)
    torch.cuda.synchronize()
    scratch = torch.as_tensor(_DeviceBytes(addr, M.STATIC_SCRATCH_BYTES), device=DEV)
    assert scratch.data_ptr() == addr
    for _ in range(2):
        scratch.fill_(0xFF)
        out.fill_(float("nan"))
        M.indexed_noalloc(a, pw, s_ids, e_ids, npp, t, k, 16, flags=flags, topk_weights=wd, out=out)
        assert _scratch_error(addr) == 0
        assert_close(dev_to_bits(out), dev_to_bits(ref), "no-alloc call after a garbage-filled scratch")
