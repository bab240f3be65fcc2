"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks reject bad calls before any CUDA work (no GPU needed)."""

import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_w4a16.h")


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_moe_w4a16_build", os.path.join(ROOT, "w4a16_int4_mixture_grouped_gb300", "build.py"))
    B = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(B)
    path = B.build()
    return ctypes.CDLL(path)


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MOE_W4A16_API\s+[\w\s\*]+?\b(moe_w4a16_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for required in ("moe_w4a16_prepare", "moe_w4a16_indexed", "moe_w4a16_contiguous", "moe_w4a16_masked",
                     "moe_w4a16_align", "moe_w4a16_dequant_check"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.moe_w4a16_status_string.restype = ctypes.c_char_p
    for s in range(10):
        assert lib.moe_w4a16_status_string(s)
    assert lib.moe_w4a16_status_string(99) == b"unknown status"
    lib.moe_w4a16_abi_version.restype = ctypes.c_uint32
    assert lib.moe_w4a16_abi_version() == 1


def test_prepare_size_schema_checks(lib):
    f = lib.moe_w4a16_prepare_size
    out = ctypes.c_size_t(0)
    assert f(384, 4096, 7168, 32, 1, ctypes.byref(out)) == 0
    assert out.value == 256 + 384 * (4096 // 128) * (7168 // 64) * 4608
    assert f(8, 256, 512, 64, 1, ctypes.byref(out)) == 2      # group 64: unsupported scheme, fails at load
    assert f(8, 256, 500, 32, 1, ctypes.byref(out)) == 2      # K % 64 != 0
    assert f(8, 200, 512, 32, 1, ctypes.byref(out)) == 2      # N % 256 != 0
    assert f(8, 256, 512, 32, 7, ctypes.byref(out)) == 1      # unknown mode
    assert f(0, 256, 512, 32, 1, ctypes.byref(out)) == 1
    assert f(2000, 256, 512, 32, 1, ctypes.byref(out)) == 1   # more than 1024 experts


def test_align_size_capacity(lib):
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.moe_w4a16_align_size(64, 8, 384, 32, ctypes.byref(a), ctypes.byref(b)) == 0
    cap = 512 + 384 * 31
    cap = -(-cap // 32) * 32
    assert a.value == cap and b.value == cap // 32
    assert lib.moe_w4a16_align_size(64, 8, 384, 257, ctypes.byref(a), ctypes.byref(b)) == 1


def test_workspace_size(lib):
    out = ctypes.c_size_t(0)
    f = lib.moe_w4a16_workspace_size
    # decode-family calls (masked, indexed block_m <= 32): header + the partial tiles of the units the kernel
    # cuts into 4 k-ranges (the last 304 units of a call with at most 2048 units: 304 units x 4 parts x 8
    # warps x 32 lanes x FP32 values, 16 for 16-row blocks, 32 for 32-row blocks and masked calls) + their
    # arrival counters (304 x 8 int32)
    cut16 = 304 * 4 * 8 * 16 * 32 * 4 + 304 * 8 * 4
    cut32 = 304 * 4 * 8 * 32 * 32 * 4 + 304 * 8 * 4
    assert f(2, 128, 8, 384, 7168, 2048, 0, 0, ctypes.byref(out)) == 0 and out.value == 256 + cut32
    assert f(0, 128, 8, 384, 7168, 2048, 32, 0, ctypes.byref(out)) == 0 and out.value == 256 + cut32
    assert f(0, 64, 8, 384, 4096, 7168, 16, 0, ctypes.byref(out)) == 0 and out.value == 256 + cut16
    assert f(0, 64, 8, 384, 512, 7168, 1, 0, ctypes.byref(out)) == 0 and out.value == 256 + cut16
    cap = 64 * 8 + 384 * 63                         # tcgen05 block sizes: gathered rows, no partial tiles
    assert f(0, 64, 8, 384, 512, 7168, 64, 0, ctypes.byref(out)) == 0 and out.value == 256 + cap * 7168 * 2
    # split: + gathered rows [max_sorted, K] + the tcgen05 block table (1 + R/192 + R/33 entries) + expert flags
    # and the decode side's block list (1 + max_blocks int32)
    ms = 4096 + 384 * 31
    cap = 4096 // 192 + 4096 // 33 + 1
    table = -(-((cap + 1) * 16) // 256) * 256
    flags_list = -(-((384 + 1 + ms // 32) * 4) // 256) * 256
    assert f(0, 512, 8, 384, 4096, 7168, 32, 32, ctypes.byref(out)) == 0
    assert out.value == 256 + ms * 7168 * 2 + cut32 + table + flags_list
    # combine: arrival counters + routed-row staging
    assert f(0, 128, 8, 384, 7168, 2048, 32, 2 | 4, ctypes.byref(out)) == 0
    counters = -(-(128 * 28 * 8 * 4) // 256) * 256
    y = -(-(1024 * 7168 * 2) // 256) * 256
    assert out.value == 256 + counters + y + cut32
    # indexed on the tcgen05 family: + gathered activations [max_sorted, K]
    cap = 8192 * 8 + 384 * 255
    cap = -(-cap // 256) * 256
    assert f(0, 8192, 8, 384, 4096, 7168, 256, 1, ctypes.byref(out)) == 0
    assert out.value == 256 + cap * 7168 * 2
    # ... unless A is already in sorted order
    assert f(0, 8192, 8, 384, 7168, 2048, 256, 2 | 8, ctypes.byref(out)) == 0
    counters = -(-(8192 * 28 * 8 * 4) // 256) * 256
    assert out.value == 256 + counters + 65536 * 7168 * 2
    # contiguous: + one int4 per 128-row segment of the largest align-built layout, plus the count
    segs = -(-(8192 * 8 + 384 * 127) // 128)
    assert f(1, 8192, 8, 384, 4096, 7168, 0, 0, ctypes.byref(out)) == 0
    assert out.value == 256 + -(-((segs + 1) * 16) // 256) * 256
    assert f(5, 1, 1, 4, 256, 64, 0, 0, ctypes.byref(out)) == 1    # unknown layout


class Desc(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("mode", ctypes.c_uint32),
                ("num_experts", ctypes.c_uint32), ("n", ctypes.c_uint32), ("k", ctypes.c_uint32),
                ("group_size", ctypes.c_uint32), ("reserved", ctypes.c_uint32), ("bytes", ctypes.c_uint64)]


def _desc(mode=1, e=4, n=256, k=128):
    d = Desc(0x34413457, 1, mode, e, n, k, 32, 0, 0)
    d.bytes = 256 + e * (n // 128) * (k // 64) * 4608
    return d


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails its host-side checks


def _masked(lib, d, flags=0, ws_bytes=1 << 30, k=128, expected_m=1):
    return lib.moe_w4a16_masked(FAKE, ctypes.c_int(d.num_experts), 16, k, FAKE, expected_m, ctypes.byref(d), FAKE,
                                None, 8, 2, None, ctypes.c_uint32(flags), FAKE, FAKE, ctypes.c_size_t(ws_bytes),
                                None)


def test_gemm_host_checks_reject_before_launch(lib):
    d = _desc()
    bad = _desc()
    bad.magic = 0
    assert _masked(lib, bad) == 3                     # not a prepared-weight descriptor
    stale = _desc()
    stale.version = 0
    assert _masked(lib, stale) == 3                   # stale layout version
    assert _masked(lib, d, flags=1) == 3              # SwiGLU needs a gate_up-mode weight
    assert _masked(lib, _desc(mode=2), flags=2) == 3  # combine needs a plain weight
    assert _masked(lib, d, flags=3) == 1              # SwiGLU and combine together
    assert _masked(lib, d, flags=2) == 1              # combine without router weights
    assert _masked(lib, d, k=64) == 1                 # K differs from the prepared weight
    assert _masked(lib, d, ws_bytes=64) == 4          # workspace too small
    assert _masked(lib, d, expected_m=0) == 1         # expected_m must be positive
    assert _masked(lib, d, flags=8) == 1              # sorted-slot flags belong to the indexed layout
    assert _masked(lib, d, flags=4) == 1              # so does A_PER_ROW
    assert _masked(lib, d, flags=64) == 1             # unknown flag bit
    assert _masked(lib, d, flags=32) == 1             # the per-expert split belongs to the indexed layout

    def indexed(flags, block_m=32, weights=None):
        return lib.moe_w4a16_indexed(FAKE, 8, 128, ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, 8, 2, block_m, weights,
                                     ctypes.c_uint32(flags), FAKE, FAKE, ctypes.c_size_t(1 << 30), None)

    assert indexed(32 | 2, weights=FAKE) == 1         # split with the fused combine
    assert indexed(32 | 8) == 1                       # split with an already sorted A
    assert indexed(32, block_m=64) == 1               # split takes the decode kernel's block sizes
    g = _desc()
    g.group_size = 64
    assert _masked(lib, g) == 2


def test_noalloc_rejects_before_any_cuda_call(lib):
    """The static-scratch entry point refuses calls whose scratch exceeds 64 MiB, prefill block sizes and the split."""
    d = _desc(e=4, n=1024, k=64)

    def call(t, k, block_m, flags, desc=d):
        return lib.moe_w4a16_indexed_noalloc(FAKE, t * k, 64, ctypes.byref(desc) if desc else None, FAKE, FAKE, FAKE, FAKE, t, k, block_m, FAKE,
                                             ctypes.c_uint32(flags), FAKE, None, None)

    assert call(3200, 8, 16, 2 | 4) == 9              # counters + 3200*8*1024*2 B + partial tiles > 64 MiB
    assert call(8, 8, 64, 0) == 1                     # block_m above 32 runs the prefill kernel: refused
    assert call(8, 8, 0, 0) == 1
    assert call(8, 8, 16, 0, desc=None) == 1
    assert call(8, 8, 32, 32) == 1                    # the per-expert split would run the tcgen05 kernel


def test_launch_counter_starts_at_zero_without_gpu(lib):
    lib.moe_w4a16_launch_count.restype = ctypes.c_uint64
    assert lib.moe_w4a16_launch_count() == 0


def test_routed_rejects_before_any_cuda_call(lib):
    """The one-launch routed entry point refuses prefill block sizes, the sorted-slot and split flags, more
    routed rows than a CTA's routing table holds, and a missing id array."""
    d = _desc(e=4, n=256, k=128)
    fn = lib.moe_w4a16_indexed_routed
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]

    def call(t, k, block_m, flags=0, ids=FAKE, a_rows=None):
        return fn(FAKE, t if a_rows is None else a_rows, 128, ctypes.byref(d), FAKE, ids, t, k, block_m, None,
                  ctypes.c_uint32(flags), FAKE, FAKE, ctypes.c_size_t(1 << 30), None)

    assert call(8, 2, 64) == 1                        # prefill block size
    assert call(8, 2, 0) == 1
    assert call(8, 2, 16, flags=8) == 1               # A_SORTED
    assert call(8, 2, 16, flags=16) == 1              # OUT_SORTED
    assert call(8, 2, 32, flags=32) == 1              # SPLIT
    assert call(1025, 4, 16) == 2                     # 4100 routed rows > 4096
    assert call(8, 2, 16, ids=None) == 1              # no ids
    assert call(8, 2, 16, a_rows=9) == 1              # A rows must be the token count


def test_binding_constants_match_the_header(lib):
    """Every enum value and size the binding restates equals the header's: a mismatch would pass the wrong flag or
    size through the C ABI without any error."""
    import w4a16_int4_mixture_grouped_gb300 as M
    text = open(HEADER).read()
    vals = {}
    for name, v in re.findall(r"\b(MOE_W4A16_[A-Z0-9_]+)\s*=\s*(\d+)u?\s*[,/\n]", text):
        vals[name] = int(v)
    for name, expr in re.findall(r"#define (MOE_W4A16_[A-Z0-9_]+) \(?([0-9a-fx]+u?(?: << \d+)?)\)?", text):
        vals[name] = eval(expr.replace("ull", "").replace("u", ""))
    expect = {
        "LAYOUT_INDEXED": M.LAYOUT_INDEXED, "LAYOUT_CONTIGUOUS": M.LAYOUT_CONTIGUOUS, "LAYOUT_MASKED": M.LAYOUT_MASKED,
        "MODE_PLAIN": M.MODE_PLAIN, "MODE_GATE_UP": M.MODE_GATE_UP,
        "FLAG_SWIGLU": M.FLAG_SWIGLU, "FLAG_COMBINE": M.FLAG_COMBINE, "FLAG_A_PER_ROW": M.FLAG_A_PER_ROW,
        "FLAG_A_SORTED": M.FLAG_A_SORTED, "FLAG_OUT_SORTED": M.FLAG_OUT_SORTED, "FLAG_SPLIT": M.FLAG_SPLIT,
        "KERNEL_AUTO": M.KERNEL_AUTO, "KERNEL_DECODE": M.KERNEL_DECODE, "KERNEL_PREFILL": M.KERNEL_PREFILL,
        "KERNEL_SPLIT": M.KERNEL_SPLIT, "WS_HEADER_BYTES": M.WS_HEADER_BYTES,
        "STATIC_SCRATCH_BYTES": M.STATIC_SCRATCH_BYTES, "WAIT_LIMIT_NS": M.WAIT_LIMIT_NS,
        "ROUTED_MAX_ROWS": M.ROUTED_MAX_ROWS,
    }
    for name, v in expect.items():
        assert vals["MOE_W4A16_" + name] == v, name
    for code, name in M.STATUS_NAMES.items():
        assert vals["MOE_W4A16_" + name] == code, name
