"""Python binding of the W4A16 MoE grouped-GEMM C ABI (include/moe_w4a16.h).

Argument marshalling only: every function below checks tensor placement and
dtypes, passes raw device pointers and the current CUDA stream to the C
library, and raises MoeW4A16Error on a non-OK status. Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback --
importing this package fails if the compiled library is missing.

Names follow the C entry points without the ``moe_w4a16_`` prefix.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Tuple

import torch

from . import build as _build

LAYOUT_INDEXED, LAYOUT_CONTIGUOUS, LAYOUT_MASKED = 0, 1, 2
MODE_PLAIN, MODE_GATE_UP = 1, 2
FLAG_SWIGLU, FLAG_COMBINE, FLAG_A_PER_ROW, FLAG_A_SORTED, FLAG_OUT_SORTED, FLAG_SPLIT = 1, 2, 4, 8, 16, 32
KERNEL_AUTO, KERNEL_DECODE, KERNEL_PREFILL, KERNEL_SPLIT = 0, 1, 2, 3
WS_HEADER_BYTES = 256
STATIC_SCRATCH_BYTES = 64 << 20   # scratch array of indexed_noalloc, per device

STATUS_NAMES = {
    0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_MODE_MISMATCH", 4: "ERR_WORKSPACE",
    5: "ERR_CAPACITY", 6: "ERR_DEVICE_TIMEOUT", 7: "ERR_CUDA", 8: "ERR_BAD_INDEX",
    9: "ERR_SCRATCH_LIMIT",
}


class MoeW4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.name = STATUS_NAMES.get(self.status, str(status))
        msg = _lib.moe_w4a16_status_string(self.status).decode() if _lib is not None else self.name
        super().__init__(f"{where}: {self.name} ({msg})")


class Desc(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("mode", ctypes.c_uint32),
                ("num_experts", ctypes.c_uint32), ("n", ctypes.c_uint32), ("k", ctypes.c_uint32),
                ("group_size", ctypes.c_uint32), ("reserved", ctypes.c_uint32), ("bytes", ctypes.c_uint64)]


class Schedule(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("block_m", ctypes.c_int32), ("tok_e", ctypes.c_int32),
                ("grid", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_U32 = ctypes.c_uint32

_SIGNATURES = {
    "moe_w4a16_status_string": (ctypes.c_char_p, [_I]),
    "moe_w4a16_abi_version": (ctypes.c_uint32, []),
    "moe_w4a16_launch_count": (ctypes.c_uint64, []),
    "moe_w4a16_prepare_size": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "moe_w4a16_prepare": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _SZ, ctypes.POINTER(Desc), _P]),
    "moe_w4a16_dequant_check": (_I, [ctypes.POINTER(Desc), _P, _I, _P, _P]),
    "moe_w4a16_align_size": (_I, [_I, _I, _I, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "moe_w4a16_align": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_w4a16_contiguous_layout": (_I, [_P, _P, _P, _I, _I, _P, _P, _P]),
    "moe_w4a16_masked_layout": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "moe_w4a16_gather_rows": (_I, [_P, _I, _I, _P, _I, _I, _P, _P, _SZ, _P]),
    "moe_w4a16_gather_sorted": (_I, [_P, _I, _I, _P, _P, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_w4a16_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(Schedule)]),
    "moe_w4a16_workspace_size": (_I, [_I, _I, _I, _I, _I, _I, _I, _U32, ctypes.POINTER(_SZ)]),
    "moe_w4a16_workspace_init": (_I, [_P, _SZ, _P]),
    "moe_w4a16_get_device_error": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_w4a16_clear_device_error": (_I, [_P, _P]),
    "moe_w4a16_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "moe_w4a16_indexed": (_I, [_P, _I, _I, ctypes.POINTER(Desc), _P, _P, _P, _P, _I, _I, _I, _P, _U32, _P, _P, _SZ,
                               _P]),
    "moe_w4a16_contiguous": (_I, [_P, _I, _I, _P, ctypes.POINTER(Desc), _P, _P, _I, _I, _P, _U32, _P, _P, _SZ, _P]),
    "moe_w4a16_masked": (_I, [_P, _I, _I, _I, _P, _I, ctypes.POINTER(Desc), _P, _P, _I, _I, _P, _U32, _P, _P, _SZ,
                              _P]),
    "moe_w4a16_indexed_routed": (_I, [_P, _I, _I, ctypes.POINTER(Desc), _P, _P, _I, _I, _I, _P, _U32, _P, _P, _SZ,
                                      _P]),
    "moe_w4a16_indexed_noalloc": (_I, [_P, _I, _I, ctypes.POINTER(Desc), _P, _P, _P, _P, _I, _I, _I, _P, _U32, _P,
                                       ctypes.POINTER(_P), _P]),
}

_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB_PATH


def _load() -> ctypes.CDLL:
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"the moe_w4a16 CUDA library is not built ({path} missing); "
                          f"run python -m w4a16_int4_mixture_grouped_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
lib = _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MoeW4A16Error(status, where)


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtypes, dev: Optional[torch.device] = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dev is not None and t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
_I32 = (torch.int32,)


# ---------------------------------------------------------------------------
# information
# ---------------------------------------------------------------------------

def status_string(status: int) -> str:
    return _lib.moe_w4a16_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_lib.moe_w4a16_abi_version())


def launch_count() -> int:
    """Kernels launched by the library in this process."""
    return int(_lib.moe_w4a16_launch_count())


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class PreparedWeight:
    buffer: torch.Tensor      # uint8 device buffer
    desc: Desc

    @property
    def num_experts(self) -> int:
        return int(self.desc.num_experts)

    @property
    def n(self) -> int:
        return int(self.desc.n)

    @property
    def k(self) -> int:
        return int(self.desc.k)

    @property
    def mode(self) -> int:
        return int(self.desc.mode)


def prepare_size(num_experts: int, n: int, k: int, group_size: int = 32, mode: int = MODE_PLAIN) -> int:
    out = _SZ(0)
    _check(_lib.moe_w4a16_prepare_size(num_experts, n, k, group_size, mode, ctypes.byref(out)), "prepare_size")
    return int(out.value)


def prepare(qweight: torch.Tensor, scales: torch.Tensor, mode: int = MODE_PLAIN, group_size: int = 32,
            out: Optional[torch.Tensor] = None) -> PreparedWeight:
    """qweight int32 [E, N, K/8] (low nibble first), scales bf16 [E, N, K/32] -> prepared weight."""
    _need(qweight, "qweight", _I32)
    dev = qweight.device
    _need(scales, "scales", _BF16, dev)
    if qweight.dim() != 3 or scales.dim() != 3:
        raise ValueError("qweight and scales must be 3-D [E, N, ...]")
    e, n, kw = qweight.shape
    k = kw * 8
    if tuple(scales.shape) != (e, n, k // group_size if group_size else 0):
        raise ValueError(f"scales shape {tuple(scales.shape)} does not match [E, N, K/{group_size}]")
    nbytes = prepare_size(e, n, k, group_size, mode)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    desc = Desc()
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_prepare(_ptr(qweight), _ptr(scales), e, n, k, group_size, mode, _ptr(out),
                                      out.numel(), ctypes.byref(desc), _stream(dev)), "prepare")
    return PreparedWeight(out, desc)


def dequant_check(pw: PreparedWeight, expert: int) -> torch.Tensor:
    """Expert's dequantised weights, bf16 [N, K], through the GEMM kernels' dequant routine."""
    dev = pw.buffer.device
    out = torch.empty((pw.n, pw.k), dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_dequant_check(ctypes.byref(pw.desc), _ptr(pw.buffer), expert, _ptr(out),
                                            _stream(dev)), "dequant_check")
    return out


# ---------------------------------------------------------------------------
# workspace and errors
# ---------------------------------------------------------------------------

def workspace_size(layout: int, num_tokens: int, top_k: int, num_experts: int, n: int, k: int, block_m: int = 0,
                   flags: int = 0) -> int:
    out = _SZ(0)
    _check(_lib.moe_w4a16_workspace_size(layout, num_tokens, top_k, num_experts, n, k, block_m, flags,
                                         ctypes.byref(out)), "workspace_size")
    return int(out.value)


def workspace(layout: int, num_tokens: int, top_k: int, num_experts: int, n: int, k: int, block_m: int = 0,
              flags: int = 0, device=None) -> torch.Tensor:
    """Allocates (through torch) and zeroes a workspace for the given call shape."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    nbytes = workspace_size(layout, num_tokens, top_k, num_experts, n, k, block_m, flags)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    workspace_init(ws)
    return ws


def workspace_init(ws: torch.Tensor) -> None:
    _need(ws, "ws", (torch.uint8,))
    with torch.cuda.device(ws.device):
        _check(_lib.moe_w4a16_workspace_init(_ptr(ws), ws.numel(), _stream(ws.device)), "workspace_init")


def get_device_error(ws: torch.Tensor) -> int:
    """Synchronises the current stream and returns the device error word (0 = OK)."""
    code = ctypes.c_int32(0)
    with torch.cuda.device(ws.device):
        _check(_lib.moe_w4a16_get_device_error(_ptr(ws), _stream(ws.device), ctypes.byref(code)),
               "get_device_error")
    return int(code.value)


WAIT_LIMIT_NS = 2_000_000_000   # default limit of a device pipeline wait


def set_wait_limit_ns(ns: int, device=None) -> None:
    """Diagnostics and tests: the limit after which a GEMM kernel's pipeline wait gives up, on `device`
    (default WAIT_LIMIT_NS; 0 makes the first wait for data not yet arrived give up at once)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_set_wait_limit_ns(int(ns)), "set_wait_limit_ns")


def clear_device_error(ws: torch.Tensor) -> None:
    with torch.cuda.device(ws.device):
        _check(_lib.moe_w4a16_clear_device_error(_ptr(ws), _stream(ws.device)), "clear_device_error")


# ---------------------------------------------------------------------------
# routing layouts
# ---------------------------------------------------------------------------

def align_size(num_tokens: int, top_k: int, num_experts: int, block_m: int) -> Tuple[int, int]:
    a, b = _SZ(0), _SZ(0)
    _check(_lib.moe_w4a16_align_size(num_tokens, top_k, num_experts, block_m, ctypes.byref(a), ctypes.byref(b)),
           "align_size")
    return int(a.value), int(b.value)


def align(topk_ids: torch.Tensor, num_experts: int, block_m: int, ws: torch.Tensor, with_counts: bool = True):
    """-> (sorted_ids [max_sorted], expert_ids [max_blocks], num_post_padded [1], counts [E] or None)."""
    _need(topk_ids, "topk_ids", _I32)
    dev = topk_ids.device
    t, k = topk_ids.shape
    ms, mb = align_size(t, k, num_experts, block_m)
    sorted_ids = torch.empty(ms, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(mb, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    counts = torch.empty(num_experts, dtype=torch.int32, device=dev) if with_counts else None
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_align(_ptr(topk_ids), t, k, num_experts, block_m, _ptr(sorted_ids), _ptr(expert_ids),
                                    _ptr(npp), _ptr(counts), _ptr(ws), ws.numel(), _stream(dev)), "align")
    return sorted_ids, expert_ids, npp, counts


def contiguous_layout(sorted_ids: torch.Tensor, expert_ids: torch.Tensor, num_post_padded: torch.Tensor,
                      num_rows: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """From an align made with block_m=128 -> (m_indices [M_pad], row_ids [M_pad])."""
    dev = sorted_ids.device
    m_pad = sorted_ids.numel()
    m_idx = torch.empty(m_pad, dtype=torch.int32, device=dev)
    row_ids = torch.empty(m_pad, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_contiguous_layout(_ptr(sorted_ids), _ptr(expert_ids), _ptr(num_post_padded), num_rows,
                                                m_pad, _ptr(m_idx), _ptr(row_ids), _stream(dev)),
               "contiguous_layout")
    return m_idx, row_ids


def masked_layout(topk_ids: torch.Tensor, num_experts: int, max_m: int, ws: torch.Tensor):
    """-> (masked_m [E], row_ids [E, max_m])."""
    _need(topk_ids, "topk_ids", _I32)
    dev = topk_ids.device
    t, k = topk_ids.shape
    masked_m = torch.empty(num_experts, dtype=torch.int32, device=dev)
    row_ids = torch.empty((num_experts, max_m), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_masked_layout(_ptr(topk_ids), t, k, num_experts, max_m, _ptr(masked_m), _ptr(row_ids),
                                            _ptr(ws), ws.numel(), _stream(dev)), "masked_layout")
    return masked_m, row_ids


def gather_rows(src: torch.Tensor, row_ids: torch.Tensor, row_div: int, out: Optional[torch.Tensor] = None,
                ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dst[i] = src[row_ids[i] // row_div] (zeros where row_ids[i] < 0)."""
    _need(src, "src", _BF16)
    dev = src.device
    _need(row_ids, "row_ids", _I32, dev)
    rows, k = src.shape
    n = row_ids.numel()
    if out is None:
        out = torch.empty((n, k), dtype=src.dtype, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_gather_rows(_ptr(src), rows, k, _ptr(row_ids), n, row_div, _ptr(out), _ptr(ws),
                                          0 if ws is None else ws.numel(), _stream(dev)), "gather_rows")
    return out


def gather_sorted(src: torch.Tensor, sorted_ids: torch.Tensor, num_post_padded: torch.Tensor, num_rows: int,
                  row_div: int, out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Rows of src in sorted_ids slot order: out[slot] = src[sorted_ids[slot] // row_div] (padding slots untouched)."""
    _need(src, "src", _BF16)
    dev = src.device
    _need(sorted_ids, "sorted_ids", _I32, dev)
    rows, k = src.shape
    if out is None:
        out = torch.empty((sorted_ids.numel(), k), dtype=src.dtype, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_gather_sorted(_ptr(src), rows, k, _ptr(sorted_ids), _ptr(num_post_padded),
                                            sorted_ids.numel(), num_rows, row_div, _ptr(out), _ptr(ws),
                                            0 if ws is None else ws.numel(), _stream(dev)), "gather_sorted")
    return out


def plan(layout: int, num_tokens: int, top_k: int, num_experts: int, n: int, k: int, expected_m: int = 0) -> Schedule:
    s = Schedule()
    _check(_lib.moe_w4a16_plan(layout, num_tokens, top_k, num_experts, n, k, expected_m, ctypes.byref(s)), "plan")
    return s


# ---------------------------------------------------------------------------
# grouped GEMMs
# ---------------------------------------------------------------------------

def _out_cols(pw: PreparedWeight, flags: int) -> int:
    return pw.n // 2 if flags & FLAG_SWIGLU else pw.n


def indexed(a: torch.Tensor, pw: PreparedWeight, sorted_ids: torch.Tensor, expert_ids: torch.Tensor,
            num_post_padded: torch.Tensor, num_tokens: int, top_k: int, block_m: int, ws: torch.Tensor,
            flags: int = 0, topk_weights: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    dev = pw.buffer.device
    _need(a, "a", _BF16, dev)
    if topk_weights is not None:
        _need(topk_weights, "topk_weights", (torch.float32,), dev)
    if flags & FLAG_COMBINE:
        rows = num_tokens
    elif flags & FLAG_OUT_SORTED:
        rows = sorted_ids.numel()               # one output row per sorted_ids slot
    else:
        rows = num_tokens * top_k
    if out is None:
        out = torch.empty((rows, _out_cols(pw, flags)), dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_indexed(_ptr(a), a.shape[0], a.shape[1], ctypes.byref(pw.desc), _ptr(pw.buffer),
                                      _ptr(sorted_ids), _ptr(expert_ids), _ptr(num_post_padded), num_tokens, top_k,
                                      block_m, _ptr(topk_weights), flags, _ptr(out), _ptr(ws), ws.numel(),
                                      _stream(dev)), "indexed")
    return out


ROUTED_MAX_ROWS = 4096   # routed rows (T * top_k) of one indexed_routed call


def indexed_routed(a: torch.Tensor, pw: PreparedWeight, topk_ids: torch.Tensor, block_m: int, ws: torch.Tensor,
                   flags: int = 0, topk_weights: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """moe_w4a16_indexed_routed: the decode-kernel indexed GEMM from the router's topk_ids [T, top_k] in one
    launch (each CTA builds the align step's block layout itself); same output as align + indexed."""
    dev = pw.buffer.device
    _need(a, "a", _BF16, dev)
    _need(topk_ids, "topk_ids", _I32, dev)
    if topk_weights is not None:
        _need(topk_weights, "topk_weights", (torch.float32,), dev)
    num_tokens, top_k = topk_ids.shape
    rows = num_tokens if flags & FLAG_COMBINE else num_tokens * top_k
    if out is None:
        out = torch.empty((rows, _out_cols(pw, flags)), dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_indexed_routed(_ptr(a), a.shape[0], a.shape[1], ctypes.byref(pw.desc), _ptr(pw.buffer),
                                             _ptr(topk_ids), num_tokens, top_k, block_m, _ptr(topk_weights), flags,
                                             _ptr(out), _ptr(ws), ws.numel(), _stream(dev)), "indexed_routed")
    return out


def indexed_noalloc(a: torch.Tensor, pw: PreparedWeight, sorted_ids: torch.Tensor, expert_ids: torch.Tensor,
                    num_post_padded: torch.Tensor, num_tokens: int, top_k: int, block_m: int, flags: int = 0,
                    topk_weights: Optional[torch.Tensor] = None, out: torch.Tensor = None) -> int:
    """moe_w4a16_indexed_noalloc: the decode-kernel indexed GEMM (block_m <= 32) with the library's static
    scratch instead of a workspace, for callers that may not allocate device memory during the call (so `out`
    is required). Returns the device address of that scratch; its first int32 is the call's error word."""
    dev = pw.buffer.device
    _need(a, "a", _BF16, dev)
    _need(out, "out", _BF16, dev)
    scratch = ctypes.c_void_p(0)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_indexed_noalloc(_ptr(a), a.shape[0], a.shape[1], ctypes.byref(pw.desc),
                                              _ptr(pw.buffer), _ptr(sorted_ids), _ptr(expert_ids),
                                              _ptr(num_post_padded), num_tokens, top_k, block_m, _ptr(topk_weights),
                                              flags, _ptr(out), ctypes.byref(scratch), _stream(dev)),
               "indexed_noalloc")
    return int(scratch.value or 0)


def contiguous(a: torch.Tensor, m_indices: torch.Tensor, pw: PreparedWeight, ws: torch.Tensor, flags: int = 0,
               row_ids: Optional[torch.Tensor] = None, num_tokens: int = 0, top_k: int = 1,
               topk_weights: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    dev = pw.buffer.device
    _need(a, "a", _BF16, dev)
    _need(m_indices, "m_indices", _I32, dev)
    m_pad, k = a.shape
    rows = num_tokens if flags & FLAG_COMBINE else m_pad
    if out is None:
        out = torch.empty((rows, _out_cols(pw, flags)), dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_contiguous(_ptr(a), m_pad, k, _ptr(m_indices), ctypes.byref(pw.desc), _ptr(pw.buffer),
                                         _ptr(row_ids), num_tokens, top_k, _ptr(topk_weights), flags, _ptr(out),
                                         _ptr(ws), ws.numel(), _stream(dev)), "contiguous")
    return out


def masked(a3: torch.Tensor, masked_m: torch.Tensor, expected_m: int, pw: PreparedWeight, ws: torch.Tensor,
           flags: int = 0, row_ids: Optional[torch.Tensor] = None, num_tokens: int = 0, top_k: int = 1,
           topk_weights: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """a3 bf16 [E, max_m, K] -> flat output [E*max_m, N] (or [T, N] with COMBINE)."""
    dev = pw.buffer.device
    _need(a3, "a3", _BF16, dev)
    _need(masked_m, "masked_m", _I32, dev)
    e, max_m, k = a3.shape
    rows = num_tokens if flags & FLAG_COMBINE else e * max_m
    if out is None:
        out = torch.empty((rows, _out_cols(pw, flags)), dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        _check(_lib.moe_w4a16_masked(_ptr(a3), e, max_m, k, _ptr(masked_m), expected_m, ctypes.byref(pw.desc),
                                     _ptr(pw.buffer), _ptr(row_ids), num_tokens, top_k, _ptr(topk_weights), flags,
                                     _ptr(out), _ptr(ws), ws.numel(), _stream(dev)), "masked")
    return out
