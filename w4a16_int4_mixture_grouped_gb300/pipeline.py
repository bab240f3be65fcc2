"""MoE FFN forward built from the C-ABI calls (sequencing and buffers only).

The hot path of one MoE layer: routing layout -> gate_up GEMM with fused
SwiGLU -> down GEMM with fused weighted top-k combine. Every step is a call
into the CUDA library; this module only allocates buffers (through torch) and
orders the calls on the current stream.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import (FLAG_A_PER_ROW, FLAG_COMBINE, FLAG_SWIGLU, LAYOUT_CONTIGUOUS, LAYOUT_INDEXED, MODE_GATE_UP,
               MODE_PLAIN, PreparedWeight, align, contiguous, contiguous_layout, gather_rows, indexed, plan,
               workspace)

CONTIGUOUS_SEGMENT = 128


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
        r = num_tokens * top_k
        if layout == LAYOUT_INDEXED:
            sched = plan(LAYOUT_INDEXED, num_tokens, top_k, self.e, w1.n, w1.k)
            self.block_m = int(block_m if block_m is not None else sched.block_m)
        elif layout == LAYOUT_CONTIGUOUS:
            self.block_m = CONTIGUOUS_SEGMENT
        else:
            raise ValueError("MoEFFN runs the indexed or contiguous layout")
        self.ws_small = workspace(num_tokens, top_k, w1.n, 0, dev)
        self.ws_down = workspace(num_tokens, top_k, w2.n, FLAG_COMBINE, dev)
        self.h = None
        self.out = torch.empty((num_tokens, self.hidden), dtype=torch.bfloat16, device=dev)
        self.r = r

    def forward(self, a: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
        out = self.out if out is None else out
        sorted_ids, expert_ids, npp, _ = align(topk_ids, self.e, self.block_m, self.ws_small, with_counts=False)
        if self.layout == LAYOUT_INDEXED:
            h = indexed(a, self.w1, sorted_ids, expert_ids, npp, self.t, self.top_k, self.block_m, self.ws_small,
                        flags=FLAG_SWIGLU, out=self.h if self.h is not None and self.h.shape[0] == self.r else None)
            self.h = h
            return indexed(h, self.w2, sorted_ids, expert_ids, npp, self.t, self.top_k, self.block_m, self.ws_down,
                           flags=FLAG_COMBINE | FLAG_A_PER_ROW, topk_weights=topk_weights, out=out)
        m_idx, row_ids = contiguous_layout(sorted_ids, expert_ids, npp, self.r)
        a_pad = gather_rows(a, row_ids, self.top_k)
        h = contiguous(a_pad, m_idx, self.w1, self.ws_small, flags=FLAG_SWIGLU)
        return contiguous(h, m_idx, self.w2, self.ws_down, flags=FLAG_COMBINE, row_ids=row_ids,
                          num_tokens=self.t, top_k=self.top_k, topk_weights=topk_weights, out=out)
