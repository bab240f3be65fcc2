#!/usr/bin/env python3
"""Benchmark of the W4A16 MoE grouped-GEMM hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one pass of the hot path over one synthetic batch. The default
workload is the prefill MoE FFN (8192 tokens, 384 experts, top-8, hidden 7168,
intermediate 2048, indexed layout): routing align -> gate_up GEMM with fused
SwiGLU -> down GEMM with fused top-8 combine. Other workloads: decode_gate_up,
decode_gate_up_masked, decode_down_combine, prefill_ffn_contiguous,
tiny_indexed, sweep_gate_up_t{16..16384}_{uniform,zipf}.

Prints one JSON line (rank 0). Timing: CUDA events on the launching stream,
warm-up first, inputs larger than L2 (the weights streamed per step exceed
the 129 MB L2), max over ranks. Multi-GPU runs are independent replicas.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth as S  # noqa: E402

METRIC = "W4A16 MoE µs/call, TFLOP/s and weight GB/s vs GB300 roofline (decode+prefill)"
UNIT = "us/call"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CHUNK_BYTES_PER_WEIGHT = 0.5625      # 4-bit weight + a BF16 scale per 32 weights
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

WORKLOAD_ALIASES = {
    "prefill_ffn": ("prefill_ffn", "indexed"),
    "prefill_ffn_contiguous": ("prefill_ffn", "contiguous"),
    "decode_gate_up": ("decode_gate_up", "indexed"),
    "decode_gate_up_masked": ("decode_gate_up", "masked"),
    "decode_down_combine": ("decode_down_combine", "indexed"),
    "tiny_indexed": ("tiny_indexed", "indexed"),
    "tp8_decode_gate_up_masked": ("tp8_decode_gate_up", "masked"),
    # a crossover sweep point in the masked layout, budget above its hottest expert (1428 rows)
    "sweep_gate_up_t1536_zipf_masked": ("sweep_gate_up_t1536_zipf", "masked", 1440),
}


def resolve(name: str):
    if name in WORKLOAD_ALIASES:
        base, layout, *max_m = WORKLOAD_ALIASES[name]
        wl = S.get_workload(base)
        return (dataclasses.replace(wl, max_m=max_m[0]) if max_m else wl), layout
    return S.get_workload(name), "indexed"


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None when the
    summary is missing or the kernel sources changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            rec = json.load(fh).get(workload_name)
        if not rec:
            return None
        h = hashlib.sha256()
        for f in rec["sources"]:
            with open(os.path.join(ROOT, "w4a16_int4_mixture_grouped_gb300", "csrc", f), "rb") as src:
                h.update(src.read())
        return float(rec["dram_bytes_per_launch"]) if h.hexdigest()[:16] == rec["source_sha256"] else None
    except (OSError, KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples every 100 ms; stop() summarises those taken inside the marked windows (all of them when
    no window was marked)."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, t0: float, t1: float):
        """A timed window [t0, t1] in time.perf_counter() seconds."""
        self.windows.append((t0, t1))

    def stop(self, windows=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summary(windows)

    def summary(self, windows=None):
        wins = self.windows if windows is None else windows
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in list(self.lines):
            # a sample describes the 100 ms before it was printed
            if wins and not any(a - 0.1 <= ts <= b + 0.1 for a, b in wins):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm: the CUDA library
# ---------------------------------------------------------------------------

def bits_to_dev(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


# Generated logical weights and prepared weights, shared by every workload of one process with the same
# (seed, GEMM, shape, experts): the decode and sweep gate_up workloads use the prefill FFN's gate_up weights
# prepared in the plain mode, the decode down workload the FFN's down weights.
_LOGICAL = {}
_PREPARED = {}


def _wkey(wl, which, dev):
    n, k = wl.gemm_shape(which)
    return (wl.seed, which, n, k, wl.num_experts, str(dev))


def logical_weights(wl, which: str, dev):
    """Every expert's logical weights (synth), generated once per process straight into device memory."""
    key = _wkey(wl, which, dev)
    if key not in _LOGICAL:
        n, k = wl.gemm_shape(which)
        qw = torch.empty((wl.num_experts, n, k // 8), dtype=torch.int32, device=dev)
        sc = torch.empty((wl.num_experts, n, k // 32), dtype=torch.bfloat16, device=dev)
        for e in range(wl.num_experts):
            q, s = S.expert_weights(wl, which, e)
            qw[e].copy_(torch.from_numpy(q))
            sc[e].copy_(torch.from_numpy(s.view(np.int16)).view(torch.bfloat16))
        _LOGICAL[key] = (qw, sc)
    return _LOGICAL[key]


def upload_weights(wl, which: str, mode: int, dev):
    """The prepared weights of one GEMM of a workload in one mode (cached per process)."""
    import w4a16_int4_mixture_grouped_gb300 as M
    key = _wkey(wl, which, dev) + (mode,)
    if key not in _PREPARED:
        qw, sc = logical_weights(wl, which, dev)
        _PREPARED[key] = M.prepare(qw, sc, mode=mode)
        torch.cuda.synchronize(dev)
    return _PREPARED[key]


def release_weights():
    _LOGICAL.clear()
    _PREPARED.clear()
    torch.cuda.empty_cache()


class OurArm:
    """Holds device inputs and runs one step of the hot path for a workload."""

    def __init__(self, wl, layout: str, dev, block_m: int = 0, routed: bool = True):
        import w4a16_int4_mixture_grouped_gb300 as M
        from w4a16_int4_mixture_grouped_gb300.pipeline import MoEFFN
        self.M, self.wl, self.layout, self.dev = M, wl, layout, dev
        t, e, k = wl.num_tokens, wl.num_experts, wl.top_k
        ids, wts = S.routing(wl)
        self.ids_np, self.wts_np = ids, wts
        self.counts = np.bincount(ids.reshape(-1), minlength=e)
        self.e_active = int((self.counts > 0).sum())
        self.ids = torch.from_numpy(ids).to(dev)
        self.wts = torch.from_numpy(wts).to(dev)
        r = t * k
        self.kind = wl.stage
        if wl.stage == "ffn":
            self.w1 = upload_weights(wl, "w1", M.MODE_GATE_UP, dev)
            self.w2 = upload_weights(wl, "w2", M.MODE_PLAIN, dev)
            self.a_np = S.activations(wl.seed, t, wl.hidden)
            self.a = bits_to_dev(self.a_np, dev)
            self.ffn = MoEFFN(self.w1, self.w2, t, k,
                              layout=M.LAYOUT_INDEXED if layout == "indexed" else M.LAYOUT_CONTIGUOUS)
            self.out = torch.empty((t, wl.hidden), dtype=torch.bfloat16, device=dev)
            n1, k1 = wl.gemm_shape("w1")
            n2, k2 = wl.gemm_shape("w2")
            self.dominant_name = "gate_up GEMM (fused SwiGLU)"
            self.dom_flops = 2.0 * r * k1 * n1
            self.dom_bytes = (self.e_active * CHUNK_BYTES_PER_WEIGHT * k1 * n1 + t * k1 * 2 + r * (n1 // 2) * 2)
            self.flops = self.dom_flops + 2.0 * r * k2 * n2
            self.weight_bytes = self.e_active * CHUNK_BYTES_PER_WEIGHT * (k1 * n1 + k2 * n2)
            self.h2d = self.a_np.nbytes + ids.nbytes + wts.nbytes
            self.d2h = t * wl.hidden * 2
        else:
            which = "w1" if wl.stage == "gate_up" else "w2"
            n, kd = wl.gemm_shape(which)
            self.n, self.kd = n, kd
            self.w = upload_weights(wl, which, M.MODE_PLAIN, dev)
            if wl.stage == "gate_up":
                self.a_np = S.activations(wl.seed, t, kd)
                self.flags = 0
                out_rows = r
                a_rows = t
            else:
                self.a_np = S.down_input(wl)
                self.flags = M.FLAG_COMBINE | M.FLAG_A_PER_ROW
                out_rows = t
                a_rows = r
            self.a = bits_to_dev(self.a_np, dev)
            self.out = torch.empty((out_rows, n), dtype=torch.bfloat16, device=dev)
            sched = M.plan(M.LAYOUT_INDEXED, t, k, e, n, kd)
            self.block_m = int(block_m or sched.block_m)
            self.kernel_family = "decode" if self.block_m <= 32 else "prefill"
            if (not block_m and layout == "indexed" and sched.kernel == M.KERNEL_SPLIT
                    and not self.flags & M.FLAG_COMBINE):
                # experts above 32 rows on the tcgen05 kernel, the others on the decode kernel
                self.kernel_family = "split"
                self.flags |= M.FLAG_SPLIT
            lay = M.LAYOUT_MASKED if layout == "masked" else M.LAYOUT_INDEXED
            self.ws_small = M.workspace(lay, t, k, e, n, kd, self.block_m, 0, dev)
            gemm_flags = self.flags
            self.a_sorted = None
            if self.kernel_family == "prefill" and layout == "indexed":
                gemm_flags = (self.flags & ~M.FLAG_A_PER_ROW) | M.FLAG_A_SORTED
                max_sorted, _ = M.align_size(t, k, e, self.block_m)
                self.a_sorted = torch.empty((max_sorted, kd), dtype=torch.bfloat16, device=dev)
            self.ws = M.workspace(lay, t, k, e, n, kd, self.block_m, gemm_flags, dev)
            # decode-family indexed calls take the router's ids straight: one launch per call (each CTA
            # builds the block layout itself) instead of align + GEMM
            self.routed = (routed and layout == "indexed" and self.kernel_family == "decode" and r <= M.ROUTED_MAX_ROWS)
            written_rows = out_rows   # output rows the GEMM writes (a masked call writes only the valid ones)
            if layout == "masked":
                self.max_m = wl.max_m
                self.expected_m = max(1, int(self.counts[self.counts > 0].mean())) if self.e_active else 1
                # a masked call picks its family itself from expected_m (the split per expert included)
                mk = M.plan(M.LAYOUT_MASKED, t, k, e, n, kd, expected_m=self.expected_m).kernel
                self.kernel_family = {M.KERNEL_DECODE: "decode", M.KERNEL_PREFILL: "prefill",
                                      M.KERNEL_SPLIT: "split"}.get(mk, str(mk))
                self.a3 = torch.empty((e, self.max_m, kd), dtype=torch.bfloat16, device=dev)
                out_rows = e * self.max_m       # flat masked output
                self.out = torch.empty((out_rows, n), dtype=torch.bfloat16, device=dev)
                a_rows = r                      # the GEMM reads each routed row's own copy in the 3-D input
            self.dominant_name = ("gate_up" if wl.stage == "gate_up" else "down+combine") + " GEMM"
            self.dom_flops = 2.0 * r * kd * n
            self.dom_bytes = (self.e_active * CHUNK_BYTES_PER_WEIGHT * kd * n + a_rows * kd * 2
                              + written_rows * n * 2 + (r * n * 4 if self.flags & M.FLAG_COMBINE else 0))
            self.flops = self.dom_flops
            self.weight_bytes = self.e_active * CHUNK_BYTES_PER_WEIGHT * kd * n
            self.h2d = self.a_np.nbytes + ids.nbytes + (wts.nbytes if self.flags else 0)
            self.d2h = out_rows * n * 2
        torch.cuda.synchronize(dev)

    def step(self, ev=None):
        """One pass of the hot path; ev = (start, end) events bracketing the dominant GEMM."""
        M = self.M
        if self.kind == "ffn":
            return self._ffn_step(ev)
        t, k = self.wl.num_tokens, self.wl.top_k
        if self.layout == "masked":
            mm, rows = M.masked_layout(self.ids, self.wl.num_experts, self.max_m, self.ws_small)
            M.gather_rows(self.a, rows.view(-1), k, out=self.a3.view(-1, self.kd))
            if ev:
                ev[0].record()
            M.masked(self.a3, mm, self.expected_m, self.w, self.ws, flags=self.flags, out=self.out)
            if ev:
                ev[1].record()
            return self.out
        if self.routed:
            if ev:
                ev[0].record()
            M.indexed_routed(self.a, self.w, self.ids, self.block_m, self.ws, flags=self.flags,
                             topk_weights=self.wts if self.flags else None, out=self.out)
            if ev:
                ev[1].record()
            return self.out
        s_ids, e_ids, npp, _ = M.align(self.ids, self.wl.num_experts, self.block_m, self.ws_small, with_counts=False)
        a_in, flags = self.a, self.flags
        if self.kernel_family == "prefill":
            # consecutive rows for the tcgen05 kernel: token rows gathered once in slot order
            a_div = 1 if flags & M.FLAG_A_PER_ROW else k
            a_in = M.gather_sorted(self.a, s_ids, npp, t * k, a_div, out=self.a_sorted, ws=self.ws_small)
            flags = (flags & ~M.FLAG_A_PER_ROW) | M.FLAG_A_SORTED
        if ev:
            ev[0].record()
        M.indexed(a_in, self.w, s_ids, e_ids, npp, t, k, self.block_m, self.ws, flags=flags,
                  topk_weights=self.wts if self.flags else None, out=self.out)
        if ev:
            ev[1].record()
        return self.out

    def _ffn_step(self, ev):
        f = self.ffn
        route = f.route(self.ids)
        a_in = f.gate_up_input(self.a, route)
        if ev:
            ev[0].record()
        h = f.gate_up(a_in, route)
        if ev:
            ev[1].record()
        out = f.down(h, route, self.wts, self.out)
        if ev and len(ev) > 2:
            ev[2].record()
        return out

    def flush_l2(self):
        """Writes a buffer twice the L2 size on the current stream (evicts the previous step's lines)."""
        if getattr(self, "_flush_buf", None) is None:
            self._flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=self.dev)
        self._flush_buf.zero_()

    def host_inputs(self):
        """Pinned host inputs (a, ids, wts) and two pinned host outputs."""
        a = torch.from_numpy(self.a_np.view(np.int16)).view(torch.bfloat16).pin_memory()
        ids = torch.from_numpy(self.ids_np).pin_memory()
        wts = torch.from_numpy(self.wts_np).pin_memory()
        outs = [torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        return (a, ids, wts), outs

    def device_set(self):
        """A second set of the step's device inputs and output (double buffering)."""
        return (torch.empty_like(self.a), torch.empty_like(self.ids), torch.empty_like(self.wts),
                torch.empty_like(self.out))

    def use_set(self, dset):
        self.a, self.ids, self.wts, self.out = dset

    def e2e_steps(self, host, outs, steps, dev):
        """`steps` steps through the API from pinned host memory, each with the H2D copy of its inputs
        and the D2H copy of its output. The copies of step i+1 (H2D) and i-1 (D2H) run on two copy
        streams beside the kernels of step i, with double-buffered device inputs and outputs."""
        a, ids, wts = host
        comp = torch.cuda.current_stream(dev)
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        sets = [(self.a, self.ids, self.wts, self.out), self.device_set()]
        in_free = [torch.cuda.Event() for _ in range(2)]
        loaded = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        start = torch.cuda.Event()
        start.record(comp)
        h2d.wait_event(start)
        for i in range(steps):
            b = i % 2
            da, dids, dwts, dout = sets[b]
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(in_free[b])
                da.copy_(a, non_blocking=True)
                dids.copy_(ids, non_blocking=True)
                if self.kind == "ffn" or self.flags:
                    dwts.copy_(wts, non_blocking=True)
                loaded[b].record(h2d)
            comp.wait_event(loaded[b])
            if i >= 2:
                comp.wait_event(out_free[b])
            if needs_l2_flush(self.weight_bytes):
                self.flush_l2()
            self.use_set(sets[b])
            res = self.step()
            in_free[b].record(comp)
            done[b].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(done[b])
                outs[b].copy_(res, non_blocking=True)
                out_free[b].record(d2h)
        comp.wait_stream(d2h)
        self.use_set(sets[0])

    def e2e_serial_steps(self, host, outs, steps):
        """`steps` steps through the API, each one in order on the current stream: the H2D copy of its
        inputs from pinned host memory, the step, the D2H copy of its output (no overlap between steps)."""
        a, ids, wts = host
        for _ in range(steps):
            self.a.copy_(a, non_blocking=True)
            self.ids.copy_(ids, non_blocking=True)
            if self.kind == "ffn" or self.flags:
                self.wts.copy_(wts, non_blocking=True)
            if needs_l2_flush(self.weight_bytes):
                self.flush_l2()
            outs[0].copy_(self.step(), non_blocking=True)


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and reference arm)
# ---------------------------------------------------------------------------

class OracleSample:
    """Times the CPU oracle on slices of the workload and scales to one call.

    A slice is one routed expert with all of its rows and `channels` output
    channels of one GEMM; a call holds E_active * N / channels slices of each
    GEMM it runs. The combine is timed over the sampled rows and scaled by
    tokens. Each part is scaled separately and the parts are summed.
    """

    def __init__(self, wl, channels: int = 128):
        import oracle as O
        self.O, self.wl, self.channels = O, wl, channels
        ids, wts = S.routing(wl)
        self.ids, self.wts = ids, wts
        counts = np.bincount(ids.reshape(-1), minlength=wl.num_experts)
        self.experts = [int(e) for e in np.argsort(-counts, kind="stable") if counts[e] > 0]
        self.next = 0
        self.a = S.activations(wl.seed, wl.num_tokens, wl.hidden) if wl.stage in ("gate_up", "ffn") else None
        self.h = S.down_input(wl) if wl.stage == "down" else None

    def one(self):
        """Runs one slice of every GEMM of the workload; returns (seconds spent, estimated us per call)."""
        O, wl, c = self.O, self.wl, self.channels
        e = self.experts[self.next % len(self.experts)]
        self.next += 1
        rows = np.nonzero(self.ids.reshape(-1) == e)[0]
        local = np.zeros_like(self.ids)              # the slice's rows all go to local expert 0
        e_act = len(self.experts)
        spent, us = 0.0, 0.0
        if wl.stage in ("gate_up", "ffn"):
            n1, _ = wl.gemm_shape("w1")
            q, s = S.expert_weights(wl, "w1", e)
            t0 = time.perf_counter()
            if wl.stage == "ffn":
                sel = np.r_[0:c // 2, n1 // 2:n1 // 2 + c // 2]
                y = O.indexed_gemm(self.a, local, lambda _: (q[sel], s[sel]), c, rows=rows)
                O.swiglu(y[rows])
            else:
                O.indexed_gemm(self.a, local, lambda _: (q[:c], s[:c]), c, rows=rows)
            dt = time.perf_counter() - t0
            spent += dt
            us += dt * e_act * n1 / c * 1e6
        if wl.stage in ("down", "ffn"):
            n2, k2 = wl.gemm_shape("w2")
            q, s = S.expert_weights(wl, "w2", e)
            h = self.h if self.h is not None else np.zeros((self.ids.size, k2), dtype=np.uint16)
            t0 = time.perf_counter()
            O.indexed_gemm(h, local, lambda _: (q[:c], s[:c]), c, a_per_routed_row=True, rows=rows)
            dt = time.perf_counter() - t0
            spent += dt
            us += dt * e_act * n2 / c * 1e6
            tok = np.unique(rows // wl.top_k)
            if tok.size:
                y = np.zeros((tok.size * wl.top_k, c), dtype=np.uint16)
                t0 = time.perf_counter()
                O.combine(y, self.wts[tok])
                dt = time.perf_counter() - t0
                spent += dt
                us += dt * (wl.num_tokens / tok.size) * (n2 / c) * 1e6
        return spent, us

    def measure(self, budget_s: float):
        spent, us = 0.0, []
        while spent < budget_s or not us:
            dt, v = self.one()
            spent += dt
            us.append(v)
        return float(np.mean(us)), spent, len(us)


def sample_text(wl, channels):
    return (f"oracle on slices of {channels} output channels of one routed expert (all of its rows) per GEMM, "
            f"scaled by experts x channel slices per call")


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, wl, layout, world, rank):
    if rank != 0:
        return 0
    samp = OracleSample(wl)
    dt, _ = samp.one()
    steps = args.steps + args.warmup
    budget = 150.0
    if dt * steps > budget:
        samp.channels = max(16, int(128 * budget / (dt * steps)) // 16 * 16)
    for _ in range(args.warmup):
        samp.one()
    vals, spent = [], 0.0
    for _ in range(args.steps):
        d, v_us = samp.one()
        spent += d
        vals.append(v_us)
    v = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, layout, weight_bytes_of(wl)),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample_text(wl, samp.channels) + f"; {args.steps} timed samples, {spent:.1f} s"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129e6
FLUSH_BYTES = 256 << 20


def weight_bytes_of(wl) -> float:
    """Prepared weight bytes one step streams: every active expert's weights and scales, once per GEMM."""
    ids, _ = S.routing(wl)
    e_active = int((np.bincount(ids.reshape(-1), minlength=wl.num_experts) > 0).sum())
    if wl.stage == "ffn":
        shapes = [wl.gemm_shape("w1"), wl.gemm_shape("w2")]
    else:
        shapes = [wl.gemm_shape("w1" if wl.stage == "gate_up" else "w2")]
    return float(e_active * CHUNK_BYTES_PER_WEIGHT * sum(n * k for n, k in shapes))


def needs_l2_flush(weight_bytes: float) -> bool:
    """Workloads whose weights per step do not exceed twice the L2 get an L2 flush before every timed step."""
    return weight_bytes < 2 * L2_BYTES


def config_of(wl, layout, weight_bytes=None):
    if weight_bytes is not None and needs_l2_flush(weight_bytes):
        l2 = (f"L2 flushed before every timed step ({FLUSH_BYTES >> 20} MiB write, outside the step's events; inside "
              f"the e2e region): the {weight_bytes / 1e6:.1f} MB of weights per step would fit in the 129 MB L2")
    else:
        l2 = "inputs larger than L2: the weights streamed per step exceed the 129 MB L2"
    return {"workload": wl.name, "layout": layout, "tokens": wl.num_tokens, "experts": wl.num_experts,
            "top_k": wl.top_k, "hidden": wl.hidden, "intermediate": wl.intermediate, "stage": wl.stage,
            "routing": wl.routing, "seed": wl.seed, "l2": l2}


def time_steps(arm, steps: int, stream, sampler=None):
    """Times `steps` steps of `arm` on `stream` with CUDA events: (ms of all steps, mean µs of the dominant
    GEMM, library launches). Workloads whose weights would fit in twice the L2 get an L2 flush before every
    step, outside the step's own events (the steps' time is then the sum of their events)."""
    import w4a16_int4_mixture_grouped_gb300 as M
    dev = arm.dev
    flush = needs_l2_flush(arm.weight_bytes)
    # FFN steps: a third event after the down GEMM + combine call (the pages sum gate_up and down)
    n_ev = 3 if getattr(arm, "kind", "") == "ffn" else 2
    dom = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(n_ev)) for _ in range(steps)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    launches0 = M.launch_count()
    w0 = time.perf_counter()
    t0.record(stream)
    for i in range(steps):
        if flush:
            arm.flush_l2()
            step_ev[i][0].record(stream)
        arm.step(dom[i])
        if flush:
            step_ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.mark(w0, time.perf_counter())
    launches = M.launch_count() - launches0
    total_ms = sum(a.elapsed_time(b) for a, b in step_ev) if flush else t0.elapsed_time(t1)
    dom_us = float(np.mean([d[0].elapsed_time(d[1]) for d in dom])) * 1e3
    if n_ev == 3:
        arm.down_combine_us = float(np.mean([d[1].elapsed_time(d[2]) for d in dom])) * 1e3
    return total_ms, dom_us, launches


def ffn_kernels(arm, gate_up_us: float):
    """An FFN step's GEMM calls, each timed by events around its own call: gate_up (with SwiGLU), the down GEMM
    call (which also launches the combine pass over the staged rows), and their sum, the pages' convention of
    summing the gate_up and down kernels."""
    return {"gate_up_us": gate_up_us, "down_with_combine_us": arm.down_combine_us,
            "sum_us": gate_up_us + arm.down_combine_us,
            "what": "events around the gate_up call and around the down call; the down call is the down GEMM "
                    "followed by the combine pass it launches"}


def keep_busy(arm, seconds: float):
    """Untimed steps for `seconds`, so the timed steps do not start on a GPU that idled."""
    until = time.perf_counter() + seconds
    while time.perf_counter() < until:
        for _ in range(4):
            arm.step()
        torch.cuda.synchronize(arm.dev)


def roofline_of(arm, dom_us: float, peaks, peaks_src: str):
    """The dominant kernel against its binding roofline: the larger of its algorithmic bytes at the measured
    HBM copy bandwidth and its flops at the measured burst BF16 rate (the kernel is timed alone per step, in a
    run of milliseconds; the sustained rate is reported beside it)."""
    t_hbm = arm.dom_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tensor = arm.dom_flops / (peaks["bf16_tflops"] * 1e12)
    if t_tensor >= t_hbm:
        achieved = arm.dom_flops / (dom_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "sustained": {"peak": peaks["bf16_tflops_sustained"],
                              "frac": achieved / peaks["bf16_tflops_sustained"]},
                "peak_source": f"{peaks_src} bf16_tflops (burst)"}
    else:
        achieved = arm.dom_bytes / (dom_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peaks_src} hbm_gbs"}
    roof.update({"traffic": None, "kernel": arm.dominant_name, "kernel_us": dom_us,
                 "algorithmic": {"flops": arm.dom_flops, "bytes": arm.dom_bytes},
                 "bound_us": {"hbm": t_hbm * 1e6, "tensor": t_tensor * 1e6}})
    return roof


# Workloads timed beside the headline in the same run: the decode gate_up (indexed and masked), the decode
# down + combine, one tensor-parallel rank's decode gate_up, the prefill FFN in the contiguous layout and the
# gate_up schedule sweep.
REGIMES = (["decode_gate_up", "decode_gate_up_masked", "decode_down_combine", "tp8_decode_gate_up",
            "prefill_ffn_contiguous"]
           + [f"sweep_gate_up_t{t}_{skew}" for t in S.SWEEP_TOKENS for skew in ("uniform", "zipf")]
           + ["sweep_gate_up_t1536_zipf_masked"])


# decode workloads also timed as align + GEMM (two launches) beside the one-launch routed call
TWO_LAUNCH_TOO = ("decode_gate_up", "decode_down_combine", "tp8_decode_gate_up")


def host_overhead(arm, calls: int = 200):
    """Host time to issue one GEMM call of an indexed single-GEMM workload, GPU busy behind it: through the
    Python binding, and through the C entry point alone with pre-marshalled ctypes arguments."""
    import ctypes
    import w4a16_int4_mixture_grouped_gb300 as M
    t, k = arm.wl.num_tokens, arm.wl.top_k
    s_ids, e_ids, npp, _ = M.align(arm.ids, arm.wl.num_experts, arm.block_m, arm.ws_small, with_counts=False)
    kwargs = dict(flags=arm.flags, topk_weights=arm.wts if arm.flags else None, out=arm.out)
    M.indexed(arm.a, arm.w, s_ids, e_ids, npp, t, k, arm.block_m, arm.ws, **kwargs)
    torch.cuda.synchronize(arm.dev)
    w0 = time.perf_counter()
    for _ in range(calls):
        M.indexed(arm.a, arm.w, s_ids, e_ids, npp, t, k, arm.block_m, arm.ws, **kwargs)
    binding = (time.perf_counter() - w0) / calls
    torch.cuda.synchronize(arm.dev)
    P = ctypes.c_void_p
    args = (P(arm.a.data_ptr()), arm.a.shape[0], arm.a.shape[1], ctypes.byref(arm.w.desc), P(arm.w.buffer.data_ptr()),
            P(s_ids.data_ptr()), P(e_ids.data_ptr()), P(npp.data_ptr()), t, k, arm.block_m,
            P(arm.wts.data_ptr() if arm.flags else 0), arm.flags, P(arm.out.data_ptr()), P(arm.ws.data_ptr()),
            arm.ws.numel(), P(torch.cuda.current_stream(arm.dev).cuda_stream))
    fn = M.lib.moe_w4a16_indexed
    w0 = time.perf_counter()
    for _ in range(calls):
        if fn(*args) != 0:
            raise RuntimeError("moe_w4a16_indexed failed")
    c_abi = (time.perf_counter() - w0) / calls
    torch.cuda.synchronize(arm.dev)
    w0 = time.perf_counter()
    for _ in range(calls):
        M.indexed_routed(arm.a, arm.w, arm.ids, arm.block_m, arm.ws, **kwargs)
    routed = (time.perf_counter() - w0) / calls
    torch.cuda.synchronize(arm.dev)
    return {"binding_us": binding * 1e6, "c_abi_us": c_abi * 1e6, "routed_binding_us": routed * 1e6, "calls": calls,
            "workload": arm.wl.name,
            "what": "host wall time per GEMM call (argument checks, memoised plan, launch), GPU busy behind it: "
                    "indexed GEMM through the binding and through the C entry point alone, and the one-launch "
                    "routed GEMM through the binding"}


def measure_regimes(names, dev, steps: int, warmup: int, peaks, peaks_src, sampler):
    out = {}
    for name in names:
        wl, layout = resolve(name)
        arm = OurArm(wl, layout, dev)
        for _ in range(warmup):
            arm.step()
        keep_busy(arm, 0.05)
        total_ms, dom_us, launches = time_steps(arm, steps, torch.cuda.current_stream(dev), sampler)
        rec = {"us_per_call": total_ms * 1e3 / steps, "steps": steps, "layout": layout, "tokens": wl.num_tokens,
               "routing": wl.routing, "active_experts": arm.e_active, "gpu_launches": launches,
               "l2": "flushed before every step" if needs_l2_flush(arm.weight_bytes) else "weights exceed L2"}
        if getattr(arm, "kernel_family", None):
            rec["kernel_family"] = arm.kernel_family + (" (routed, one launch)" if getattr(arm, "routed", False) else "")
            rec["block_m"] = arm.block_m
        rec["roofline"] = roofline_of(arm, dom_us, peaks, peaks_src)
        traffic = recorded_traffic(name)
        rec["roofline"]["traffic"] = traffic
        if name == "decode_gate_up":
            rec["host_overhead"] = host_overhead(arm)
        if getattr(arm, "down_combine_us", None) is not None:
            rec["ffn_kernels"] = ffn_kernels(arm, dom_us)
        if getattr(arm, "routed", False) and name in TWO_LAUNCH_TOO:
            # the same workload as align + GEMM (two launches): its GEMM alone against the roofline
            del arm
            arm2 = OurArm(wl, layout, dev, routed=False)
            for _ in range(warmup):
                arm2.step()
            t_ms, d_us, n_l = time_steps(arm2, steps, torch.cuda.current_stream(dev), sampler)
            r2 = roofline_of(arm2, d_us, peaks, peaks_src)
            rec["two_launch"] = {"us_per_call": t_ms * 1e3 / steps, "gpu_launches": n_l, "kernel_us": d_us,
                                 "frac": r2["frac"], "achieved": r2["achieved"], "unit": r2["unit"],
                                 "what": "align kernel + indexed GEMM; kernel_us and frac are the GEMM's alone"}
            arm = arm2
        out[name] = rec
        del arm
        torch.cuda.empty_cache()
    return out


def oracle_cpu_baseline(wl, budget_s: float, single_core: bool):
    """The oracle timed on a bounded sample of the workload, on all host cores or on one (a child process
    pinned to one core with one BLAS thread)."""
    if not single_core:
        samp = OracleSample(wl)
        v, spent, n = samp.measure(budget_s)
        return {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                "sample": sample_text(wl, samp.channels) + f"; {n} slices, {spent:.1f} s"}
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", wl.name,
           "--cpu-budget", str(budget_s)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s * 4 + 120)
        rec = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.TimeoutExpired, ValueError, IndexError) as exc:
        return {"unavailable": f"single-core oracle run failed: {exc}"}
    return rec


def oracle_sample_main(args):
    """Child process of oracle_cpu_baseline(single_core=True): pins itself to one core and prints one line."""
    try:
        cpu = sorted(os.sched_getaffinity(0))[0]
        os.sched_setaffinity(0, {cpu})
    except (AttributeError, OSError):
        pass
    wl = resolve(args.workload)[0]
    samp = OracleSample(wl)
    v, spent, n = samp.measure(args.cpu_budget)
    print(json.dumps({"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                      "sample": sample_text(wl, samp.channels) + f"; {n} slices, {spent:.1f} s, one core"}))
    return 0


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="prefill_ffn")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-regimes", action="store_true", help="time only the headline workload")
    p.add_argument("--regime-steps", type=int, default=10, help="timed steps of each workload beside the headline")
    p.add_argument("--layout", default="", choices=["", "indexed", "masked"],
                   help="override the layout of a single-GEMM workload")
    p.add_argument("--max-m", type=int, default=0, help="masked row budget per expert with --layout masked")
    p.add_argument("--block-m", type=int, default=0,
                   help="indexed rows per block of a single-GEMM workload instead of the plan's (schedule sweeps)")
    p.add_argument("--no-routed", action="store_true",
                   help="decode-family indexed workloads: align + GEMM instead of the one-launch routed GEMM")
    p.add_argument("--tokens", type=int, default=0, help="override the workload's token count (profiling cases)")
    p.add_argument("--experts", type=int, default=0, help="override the workload's expert count (profiling cases)")
    p.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    args = p.parse_args(argv)
    if args.oracle_sample:
        return oracle_sample_main(args)
    if args.warmup < 3:
        args.warmup = 3
    wl, layout = resolve(args.workload)
    custom = bool(args.tokens or args.experts or args.layout or args.block_m)
    if args.tokens or args.experts:
        t = args.tokens or wl.num_tokens
        e = args.experts or wl.num_experts
        wl = dataclasses.replace(wl, name=f"{wl.name}_t{t}_e{e}", num_tokens=t, num_experts=e,
                                 hot_experts=min(wl.hot_experts, e))
    if args.layout:
        layout = args.layout
        if layout == "masked" and args.max_m:
            wl = dataclasses.replace(wl, max_m=args.max_m)
    world, rank, local = dist_setup(args.gpus)

    if args.impl == "reference":
        return run_reference(args, wl, layout, world, rank)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peaks_src = load_peaks()
    arm = OurArm(wl, layout, dev, block_m=args.block_m, routed=not args.no_routed)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        arm.step()
    torch.cuda.synchronize(dev)

    # device-timed region: inputs resident in HBM
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    # keep the GPU under load while the clock sampler starts, so the timed steps do not begin
    # on a GPU that idled (untimed steps, on top of the warm-up)
    keep_busy(arm, 0.2)
    barrier(world)
    total_ms, dom_us, launches = time_steps(arm, args.steps, stream, sampler)
    head_window = list(sampler.windows)
    barrier(world)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = total_ms * 1e3 / (args.steps * world)

    # end to end through the API with host buffers (every step's copies inside the timed region): each step
    # serially on one stream (the per-call figure), and pipelined with the neighbouring steps' copies
    host, host_outs = arm.host_inputs()
    e_steps = max(3, min(args.steps, 20))
    e2e = {"unit": UNIT, "h2d_bytes_per_step": int(arm.h2d), "d2h_bytes_per_step": int(arm.d2h), "steps": e_steps}
    for mode in ("serial", "pipelined"):
        run = (lambda n: arm.e2e_serial_steps(host, host_outs, n)) if mode == "serial" else \
            (lambda n: arm.e2e_steps(host, host_outs, n, dev))
        run(3)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(e_steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e[mode] = e_ms * 1e3 / (e_steps * world)
    e2e["value"] = e2e["serial"]
    e2e["what"] = ("value: each step's H2D copies, kernels and D2H copy in order on one stream (serial); "
                   "pipelined: H2D of step i+1 and D2H of step i-1 on two copy streams beside step i")

    roof = roofline_of(arm, dom_us, peaks, peaks_src)
    # DRAM bytes per launch from the committed ncu capture of this kernel and workload (null if stale or absent)
    roof["traffic"] = recorded_traffic(args.workload) if not custom else None
    config = config_of(wl, layout, arm.weight_bytes)
    if getattr(arm, "block_m", None) and layout == "indexed":
        config["block_m"] = arm.block_m
        config["kernel"] = arm.kernel_family + (" (routed, one launch)" if getattr(arm, "routed", False) else "")

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": config,
        "throughput": {"tflops": arm.flops / (ms_per_step * 1e-3) / 1e12,
                       "weight_gbs": arm.weight_bytes / (ms_per_step * 1e-3) / 1e9,
                       "active_experts": arm.e_active},
        "roofline": roof,
        "e2e": e2e,
        "clocks": None,
        "gpu_launches": int(launches),
    }
    if getattr(arm, "down_combine_us", None) is not None:
        line["ffn_kernels"] = ffn_kernels(arm, dom_us)
    del arm
    torch.cuda.empty_cache()
    if not args.no_regimes and not custom and args.workload == "prefill_ffn":
        line["regimes"] = measure_regimes(REGIMES, dev, args.regime_steps, 3, peaks, peaks_src, sampler)
    release_weights()
    sampler.stop()
    line["clocks"] = sampler.summary(head_window)
    if "regimes" in line:
        line["regimes_clocks"] = sampler.summary(sampler.windows[len(head_window):])
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_cpu_baseline(wl, args.cpu_budget, single_core=False)
        if not custom:
            line["cpu_baseline"]["single_core"] = oracle_cpu_baseline(wl, args.cpu_budget / 2, single_core=True)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
