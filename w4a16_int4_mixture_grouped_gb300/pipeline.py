"""MoE FFN forward built from the C-ABI calls (sequencing and buffers only).

The hot path of one MoE layer: routing layout -> gate_up GEMM with fused
SwiGLU -> down GEMM with fused weighted top-k combine. Every step is a call
into the CUDA library; this module only allocates buffers (through torch) and
orders the calls on the current stream.

Indexed layout: the gate_up GEMM writes SwiGLU(h) in sorted_ids slot order
(FLAG_OUT_SORTED), so the down GEMM reads its rows consecutively
(FLAG_A_SORTED) and combines them back per token.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import (FLAG_A_SORTED, FLAG_COMBINE, FLAG_OUT_SORTED, FLAG_SPLIT, FLAG_SWIGLU, KERNEL_SPLIT, LAYOUT_CONTIGUOUS,
               LAYOUT_INDEXED, MODE_GATE_UP, MODE_PLAIN, PreparedWeight, align, align_size, contiguous,
               contiguous_layout, gather_rows, gather_sorted, indexed, plan, workspace)

CONTIGUOUS_SEGMENT = 128
DECODE_MAX_BLOCK_M = 32    # indexed calls with block_m above this run the tcgen05 kernel


class MoEFFN:
    """A prepared MoE FFN (gate_up in MODE_GATE_UP, down in MODE_PLAIN) for a fixed token count."""

    def __init__(self, w1: PreparedWeight, w2: PreparedWeight, num_tokens: int, top_k: int,
                 layout: int = LAYOUT_INDEXED, block_m: Optional[int] = None):
        if w1.mode != MODE_GATE_UP or w2.mode != MODE_PLAIN:
            raise ValueError("w1 must be prepared with MODE_GATE_UP and w2 with MODE_PLAIN")
        if w1.num_experts != w2.num_experts or w1.n // 2 != w2.k or w2.n != w1.k:
            raise ValueError("w1 / w2 shapes do not form an FFN")
        self.w1, self.w2 = w1, w2
        self.t, self.top_k, self.layout = num_tokens, top_k, layout
        self.e = w1.num_experts
        self.hidden, self.inter = w1.k, w1.n // 2
        dev = w1.buffer.device
        self.device = dev
        self.r = num_tokens * top_k
        self.a_sorted = None
        if layout == LAYOUT_INDEXED:
            sched = plan(LAYOUT_INDEXED, num_tokens, top_k, self.e, w1.n, w1.k)
            self.block_m = int(block_m if block_m is not None else sched.block_m)
            self.f1 = FLAG_SWIGLU | FLAG_OUT_SORTED
            self.f2 = FLAG_COMBINE | FLAG_A_SORTED
            if block_m is None and sched.kernel == KERNEL_SPLIT:
                # gate_up split per expert (tcgen05 above 32 rows); the down GEMM with its fused
                # combine stays on the decode kernel over the same 32-row layout
                self.f1 |= FLAG_SPLIT
            max_sorted, _ = align_size(num_tokens, top_k, self.e, self.block_m)
            self.h = torch.empty((max_sorted, self.inter), dtype=torch.bfloat16, device=dev)
            if self.block_m > DECODE_MAX_BLOCK_M:
                # the tcgen05 family reads consecutive rows: gather the token rows once, in slot order
                self.f1 |= FLAG_A_SORTED
                self.a_sorted = torch.empty((max_sorted, self.hidden), dtype=torch.bfloat16, device=dev)
        elif layout == LAYOUT_CONTIGUOUS:
            self.block_m = CONTIGUOUS_SEGMENT
            self.f1, self.f2 = FLAG_SWIGLU, FLAG_COMBINE
            self.h = None
        else:
            raise ValueError("MoEFFN runs the indexed or contiguous layout")
        self.ws1 = workspace(layout, num_tokens, top_k, self.e, w1.n, w1.k, self.block_m, self.f1, dev)
        self.ws2 = workspace(layout, num_tokens, top_k, self.e, w2.n, w2.k, self.block_m, self.f2, dev)
        self.out = torch.empty((num_tokens, self.hidden), dtype=torch.bfloat16, device=dev)

    @property
    def workspaces(self):
        return (self.ws1, self.ws2)

    def routing(self, topk_ids: torch.Tensor):
        """The routing layout step (align) for this layer's block size."""
        return align(topk_ids, self.e, self.block_m, self.ws1, with_counts=False)

    def gate_up_input(self, a: torch.Tensor, route) -> torch.Tensor:
        """The gate_up GEMM's activation operand: token rows, sorted rows, or padded contiguous rows."""
        sorted_ids, expert_ids, npp = route[:3]
        if self.layout == LAYOUT_INDEXED:
            if self.a_sorted is None:
                return a
            return gather_sorted(a, sorted_ids, npp, self.r, self.top_k, out=self.a_sorted, ws=self.ws1)
        return gather_rows(a, route[4], self.top_k)

    def gate_up(self, a_in: torch.Tensor, route) -> torch.Tensor:
        sorted_ids, expert_ids, npp = route[:3]
        if self.layout == LAYOUT_INDEXED:
            return indexed(a_in, self.w1, sorted_ids, expert_ids, npp, self.t, self.top_k, self.block_m, self.ws1,
                           flags=self.f1, out=self.h)
        return contiguous(a_in, route[3], self.w1, self.ws1, flags=self.f1)

    def down(self, h: torch.Tensor, route, topk_weights: torch.Tensor, out: torch.Tensor) -> torch.Tensor:
        sorted_ids, expert_ids, npp = route[:3]
        if self.layout == LAYOUT_INDEXED:
            return indexed(h, self.w2, sorted_ids, expert_ids, npp, self.t, self.top_k, self.block_m, self.ws2,
                           flags=self.f2, topk_weights=topk_weights, out=out)
        m_idx, row_ids = route[3], route[4]
        return contiguous(h, m_idx, self.w2, self.ws2, flags=self.f2, row_ids=row_ids, num_tokens=self.t,
                          top_k=self.top_k, topk_weights=topk_weights, out=out)

    def route(self, topk_ids: torch.Tensor):
        sorted_ids, expert_ids, npp, _ = self.routing(topk_ids)
        if self.layout == LAYOUT_INDEXED:
            return (sorted_ids, expert_ids, npp)
        m_idx, row_ids = contiguous_layout(sorted_ids, expert_ids, npp, self.r)
        return (sorted_ids, expert_ids, npp, m_idx, row_ids)

    def forward(self, a: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
        out = self.out if out is None else out
        route = self.route(topk_ids)
        h = self.gate_up(self.gate_up_input(a, route), route)
        return self.down(h, route, topk_weights, out)
