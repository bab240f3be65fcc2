"""Seeded synthetic MoE workloads (inputs only).

Everything here is a random draw or a data-type conversion of a random draw.
Every tensor is produced from a numpy ``Generator`` seeded by a
``SeedSequence`` of (seed, tensor tag, index), so one expert's weights can be
regenerated on its own (the oracle checks sampled experts without building the
whole weight set).

Shapes follow the serving shapes the Chord page ("vLLM x Novita AI Chord:
INT4 MoE operator", TL;DR) is built for: Kimi K2.x MoE layers with 384
experts, top-8 routing, hidden 7168 and intermediate 2048.

Conventions (the logical, caller-facing format):
  * BF16 tensors are carried as ``uint16`` bit patterns.
  * ``qweight``: int32 [N, K/8]; word w of row n holds k = 8w..8w+7, the
    nibble for k = 8w+i in bits 4i..4i+3 (low nibble first).
  * ``scales``: BF16 [N, K/32], one scale per 32 consecutive k of a row.
  * routing: ``topk_ids`` int32 [T, top_k], distinct experts per token;
    ``topk_weights`` float32 [T, top_k].
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "sweep_workload", "get_workload",
    "f32_to_bf16_bits", "rng_for",
    "activations", "expert_qweight", "expert_scales", "expert_weights",
    "all_expert_weights", "routing", "down_input",
    "TAG_A", "TAG_W1", "TAG_W2", "TAG_S1", "TAG_S2", "TAG_ROUTE", "TAG_H",
]

# Tensor tags mixed into the seed sequence.
TAG_A = 1        # activations
TAG_W1 = 2       # gate_up packed weights
TAG_S1 = 3       # gate_up scales
TAG_W2 = 4       # down packed weights
TAG_S2 = 5       # down scales
TAG_ROUTE = 6    # router logits / noise
TAG_H = 7        # down-projection input (gate, up draws)

GROUP = 32
SCALE_LO = 0.005
SCALE_HI = 0.02


def rng_for(seed: int, *tags: int) -> np.random.Generator:
    """A PCG64 generator for (seed, *tags)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed)] + [int(t) for t in tags])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); return the uint16 bits.

    Used only to turn random float draws into BF16 inputs.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    r[nan] = np.uint16(0x7FC0)
    return r


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic MoE workload.

    ``stage`` is "gate_up" (N = 2 * intermediate, K = hidden), "down"
    (N = hidden, K = intermediate, combined over top-k) or "ffn" (both).
    """

    name: str
    num_tokens: int
    num_experts: int
    top_k: int
    hidden: int
    intermediate: int
    stage: str
    routing: str                 # "softmax" | "skewed" | "zipf"
    seed: int = 0
    max_m: int = 0               # masked layout row budget per expert (0: unused)
    hot_experts: int = 48        # skewed routing: size of the hot set
    hot_boost: float = 4.0       # skewed routing: logit boost of the hot set
    capacity: int = 15           # skewed routing: rows per expert at most
    zipf_s: float = 1.2          # zipf routing exponent
    description: str = ""

    @property
    def rows(self) -> int:
        return self.num_tokens * self.top_k

    def gemm_shape(self, which: str) -> Tuple[int, int]:
        """(N, K) of the gate_up ("w1") or down ("w2") GEMM."""
        if which == "w1":
            return 2 * self.intermediate, self.hidden
        if which == "w2":
            return self.hidden, self.intermediate
        raise ValueError(which)


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload(
            name="tiny_indexed", num_tokens=64, num_experts=8, top_k=2, hidden=512, intermediate=128,
            stage="gate_up", routing="softmax",
            description="64 tokens, 8 experts, top-2 softmax routing, K=512, N=256, indexed layout",
        ),
        Workload(
            name="decode_gate_up", num_tokens=64, num_experts=384, top_k=8, hidden=7168, intermediate=2048,
            stage="gate_up", routing="skewed", max_m=16,
            description="decode gate_up: 64 tokens, 384 experts, top-8 skewed routing (1-15 rows per active "
                        "expert), K=7168, N=4096, indexed and masked (16 rows/expert) layouts",
        ),
        Workload(
            name="decode_down_combine", num_tokens=128, num_experts=384, top_k=8, hidden=7168, intermediate=2048,
            stage="down", routing="softmax",
            description="decode down projection with fused top-8 combine: 128 tokens, 384 experts, K=2048, "
                        "N=7168, input SiLU(gate)*up of BF16 normals",
        ),
        Workload(
            name="prefill_ffn", num_tokens=8192, num_experts=384, top_k=8, hidden=7168, intermediate=2048,
            stage="ffn", routing="softmax",
            description="prefill MoE FFN: 8192 tokens, 384 experts, top-8 (about 171 rows/expert), gate_up "
                        "7168->4096, SiLU(gate)*up, down 2048->7168, weighted top-8 combine",
        ),
        # tensor-parallel shards of the same layer (8 ranks: intermediate 2048 / 8 per rank)
        Workload(
            name="tp8_decode_gate_up", num_tokens=64, num_experts=384, top_k=8, hidden=7168, intermediate=256,
            stage="gate_up", routing="skewed", max_m=16,
            description="one rank of an 8-way tensor-parallel decode gate_up: 64 tokens, 384 experts, top-8 "
                        "skewed routing, K=7168, N=512",
        ),
        Workload(
            name="tp8_prefill_down_combine", num_tokens=8192, num_experts=384, top_k=8, hidden=7168,
            intermediate=256, stage="down", routing="softmax",
            description="the down GEMM of one 8-way tensor-parallel prefill rank with fused top-8 combine: "
                        "8192 tokens, 384 experts, K=256, N=7168",
        ),
        Workload(
            name="tp8_prefill_ffn", num_tokens=8192, num_experts=384, top_k=8, hidden=7168, intermediate=256,
            stage="ffn", routing="softmax",
            description="one rank of an 8-way tensor-parallel prefill FFN: 8192 tokens, 384 experts, top-8, "
                        "gate_up 7168->512, SiLU(gate)*up, down 256->7168 (partial sums of the layer's output)",
        ),
    ]
}

SWEEP_TOKENS = (16, 128, 512, 1536, 4096, 16384)


def sweep_workload(num_tokens: int, skew: str) -> Workload:
    """gate_up GEMM at hidden 7168 / intermediate 2048, 384 experts, top-8, uniform or Zipf(1.2) skew."""
    if skew not in ("uniform", "zipf"):
        raise ValueError(skew)
    return Workload(
        name=f"sweep_gate_up_t{num_tokens}_{skew}", num_tokens=num_tokens, num_experts=384, top_k=8,
        hidden=7168, intermediate=2048, stage="gate_up",
        routing="softmax" if skew == "uniform" else "zipf",
        description=f"gate_up sweep point: {num_tokens} tokens, {skew} expert skew",
    )


def get_workload(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep_gate_up_t"):
        rest = name[len("sweep_gate_up_t"):]
        t, skew = rest.split("_", 1)
        return sweep_workload(int(t), skew)
    raise KeyError(name)


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------

def activations(seed: int, rows: int, k: int, tag: int = TAG_A) -> np.ndarray:
    """BF16 bits [rows, k] of N(0, 1) draws."""
    g = rng_for(seed, tag)
    return f32_to_bf16_bits(g.standard_normal((rows, k), dtype=np.float32))


def expert_qweight(seed: int, tag: int, expert: int, n: int, k: int) -> np.ndarray:
    """int32 [n, k/8]: every nibble uniform on 0..15 (a uniform random 32-bit word)."""
    if k % 8:
        raise ValueError("K must be a multiple of 8")
    g = rng_for(seed, tag, expert)
    words = np.frombuffer(g.bytes(n * (k // 8) * 4), dtype="<u4").reshape(n, k // 8)
    return words.view(np.int32).copy()


def expert_scales(seed: int, tag: int, expert: int, n: int, k: int, group: int = GROUP,
                  lo: float = SCALE_LO, hi: float = SCALE_HI) -> np.ndarray:
    """BF16 bits [n, k/group] of U[lo, hi] draws."""
    g = rng_for(seed, tag, expert)
    return f32_to_bf16_bits(g.uniform(lo, hi, size=(n, k // group)).astype(np.float32))


def expert_weights(wl: Workload, which: str, expert: int) -> Tuple[np.ndarray, np.ndarray]:
    """(qweight int32 [N, K/8], scales bf16 bits [N, K/32]) of one expert of ``which`` in {"w1", "w2"}."""
    n, k = wl.gemm_shape(which)
    wt, st = (TAG_W1, TAG_S1) if which == "w1" else (TAG_W2, TAG_S2)
    return expert_qweight(wl.seed, wt, expert, n, k), expert_scales(wl.seed, st, expert, n, k)


def all_expert_weights(wl: Workload, which: str) -> Tuple[np.ndarray, np.ndarray]:
    """Stacked (qweight [E, N, K/8], scales [E, N, K/32]) for every expert."""
    n, k = wl.gemm_shape(which)
    qw = np.empty((wl.num_experts, n, k // 8), dtype=np.int32)
    sc = np.empty((wl.num_experts, n, k // GROUP), dtype=np.uint16)
    for e in range(wl.num_experts):
        qw[e], sc[e] = expert_weights(wl, which, e)
    return qw, sc


def _topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries per row, largest first, ties to the lower index."""
    e = scores.shape[1]
    # lexsort: last key is primary. Sort by -score, then by index ascending.
    idx = np.arange(e)[None, :].repeat(scores.shape[0], 0)
    order = np.lexsort((idx, -scores), axis=1)
    return order[:, :k]


def _softmax(x: np.ndarray) -> np.ndarray:
    m = x.max(axis=1, keepdims=True)
    p = np.exp(x - m)
    return p / p.sum(axis=1, keepdims=True)


def routing(wl: Workload) -> Tuple[np.ndarray, np.ndarray]:
    """(topk_ids int32 [T, top_k], topk_weights float32 [T, top_k]).

    softmax: top-k of softmax(N(0,1) logits), weights renormalised over the top-k.
    skewed:  N(0,1) logits plus ``hot_boost`` on a seeded hot set; tokens in order
             take their best experts that still have room under ``capacity``.
    zipf:    expert i has probability proportional to rank_i^-s over a seeded
             permutation; each token draws top-k distinct experts by Gumbel-top-k.
    """
    t, e, k = wl.num_tokens, wl.num_experts, wl.top_k
    g = rng_for(wl.seed, TAG_ROUTE)
    if wl.routing == "softmax":
        logits = g.standard_normal((t, e))
        p = _softmax(logits)
        ids = _topk_desc(p, k)
    elif wl.routing == "skewed":
        hot = g.choice(e, size=min(wl.hot_experts, e), replace=False)
        logits = g.standard_normal((t, e))
        logits[:, hot] += wl.hot_boost
        p = _softmax(logits)
        order = _topk_desc(p, e)
        counts = np.zeros(e, dtype=np.int64)
        ids = np.empty((t, k), dtype=np.int64)
        for tok in range(t):
            j = 0
            for cand in order[tok]:
                if counts[cand] < wl.capacity:
                    ids[tok, j] = cand
                    counts[cand] += 1
                    j += 1
                    if j == k:
                        break
            if j < k:
                raise RuntimeError("capacity too small for the skewed routing draw")
    elif wl.routing == "zipf":
        perm = g.permutation(e)
        rank = np.empty(e, dtype=np.int64)
        rank[perm] = np.arange(e)
        logp = -wl.zipf_s * np.log(rank + 1.0)
        logp -= np.log(np.exp(logp).sum())
        scores = logp[None, :] + g.gumbel(size=(t, e))
        ids = _topk_desc(scores, k)
        p = np.exp(np.broadcast_to(logp, (t, e)))
    else:
        raise ValueError(wl.routing)
    sel = np.take_along_axis(p, ids, axis=1)
    w = (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids.astype(np.int32), w


def down_input(wl: Workload) -> np.ndarray:
    """BF16 bits [T*top_k, intermediate]: the down projection's input for a down-only workload.

    Drawn as gate * sigmoid(gate) * up of independent BF16 N(0,1) draws, rounded
    to BF16 -- a distribution recipe for the input, not a step under test.
    """
    r, i = wl.rows, wl.intermediate
    g = rng_for(wl.seed, TAG_H)
    gate = f32_to_bf16_bits(g.standard_normal((r, i), dtype=np.float32))
    up = f32_to_bf16_bits(g.standard_normal((r, i), dtype=np.float32))
    gf = (gate.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    uf = (up.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    h = gf / (1.0 + np.exp(-gf)) * uf
    return f32_to_bf16_bits(h.astype(np.float32))


def expert_counts(topk_ids: np.ndarray, num_experts: int) -> np.ndarray:
    return np.bincount(topk_ids.reshape(-1), minlength=num_experts)


__all__.append("expert_counts")
__all__ += ["SWEEP_TOKENS", "SCALE_LO", "SCALE_HI", "GROUP"]
