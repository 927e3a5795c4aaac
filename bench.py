#!/usr/bin/env python3
"""Benchmark of the multi-adapter LoRA projection on GB300.

One step = one lora_proj_apply (or lora_moe_down_apply, ...) call over one
batch: every kernel of the call (routing, shrink, base product, expand-fold).

Default (--config suite): the headline is the prefill workload (8192 rows,
W [14336 x 4096] bf16, 8 rank-64 rsLoRA adapters), the largest one; its
timed region is exactly K steps, each a CUDA-graph replay of one call between
its own pair of events, and value = rows / the median step time. Under
"configs" the line carries prefill, decode, QKV and MoE (--extended: also the
gated MLP input, the decode MoE gather, the stack and the embedding gather),
each timed over max(K, 100) calls (median and min), beside the same calls
with every slot -1 (the base product alone), an end-to-end rate through the
C ABI with host copies, the roofline of the median call and the oracle on
the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config suite|NAME] [--extended]
                  [--impl ours|reference]

N > 1 (under torchrun): every rank runs an independent replica on its own GPU
(the projection shards by rows with no exchange); value = all ranks' rows /
the slowest rank's median step. Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-projection rows/s at 1 GB300; achieved HBM GB/s / tensor TFLOPS vs peak"
L2_BYTES = 129 * 1024 * 1024

DESCRIBE = {
    "tiny": "tiny: 8 rows x W[256x256] bf16, 4 adapters r=8 alpha=16",
    "decode": "decode: 64 rows x W[4096x4096] bf16, 16 adapters r in {8,16,32,64} pool R=64, "
              "alpha=2r, 10% rows slot -1",
    "qkv": "fused QKV: 256 rows x W[6144x4096] (q4096+k1024+v1024) bf16, 32 adapters r=16, "
           "Zipf(1.1) slots, 5% rows -1, adapter scales {0,0.5,1} alpha=32",
    "prefill": "prefill gate/up: 8192 rows (8 seqs x 1024) x W[14336x4096] bf16, 8 adapters r=64 "
               "rsLoRA alpha=16",
    "moe": "MoE down: 8 experts W_e[4096x14336] bf16, 512 tokens top-2 = 1024 slot-rows, "
           "4 adapters/expert r=16 alpha=32",
    "embed": "token embedding gather: 64 tokens of E[32000x4096] bf16, 16 adapters r in "
             "{8,16,32,64} pool R=64, alpha=2r, 10% rows slot -1",
    "embed_prefill": "token embedding gather: 4096 tokens of E[32000x4096] bf16, 16 adapters r in "
                     "{8,16,32,64} pool R=64, alpha=2r, 10% rows slot -1",
    "gate_up": "gated MLP input: 8192 rows (8 seqs x 1024) x fused W[14336x4096] bf16 = gate 7168 | up 7168, "
               "8 adapters r=64 rsLoRA alpha=16 (B rows split the same way), act = silu(gate) * up",
    "gate_up_decode": "gated MLP input: 64 rows x fused W[4096x4096] bf16 = gate 2048 | up 2048, 16 adapters "
                      "r in {8,16,32,64} pool R=64, alpha=2r, 10% rows slot -1, act = silu(gate) * up",
    "moe_gather": "decode MoE down with top-2 combine: 64 tokens x top-2 = 128 slot-rows in token order, "
                  "8 experts W_e[4096x14336] bf16 named per slot-row, 4 adapters/expert r=16 alpha=32, "
                  "combine = softmax of the top-2 logits",
    "stack": "several adapters per slot: 64 rows x W[4096x4096] bf16, 8 slots each a stack of 1-3 adapters "
             "r in {8,16,32} (ranks summing to <= pool R=64), alpha=2r, adapter scales {0.5,1}, one member "
             "at scale 0, 10% rows slot -1",
}
BOUND = {"tiny": "hbm", "decode": "hbm", "qkv": "hbm", "prefill": "tensor", "moe": "hbm",
         "embed": "hbm", "embed_prefill": "hbm", "gate_up": "tensor", "gate_up_decode": "hbm",
         "stack": "hbm", "moe_gather": "hbm"}
GATE_UP = {"gate_up": "prefill", "gate_up_decode": "decode"}  # the projection workload each one reads
EMBED_ROWS = {"embed": 64, "embed_prefill": 4096}
# --small: the same kernels on fewer rows, for profiler captures only (never a bench line)
SMALL = {"prefill": {"seq_len": 256}, "moe": {"tokens": 128}}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained",
                                                                          d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------
# algorithmic bytes / flops of one call (true ranks, touched slots only)
# ----------------------------------------------------------------------------

def _scale_on(ad):
    if ad is None or ad.adapter_scale == 0.0:
        return False
    return True


def proj_algorithmic(wl):
    M, K, N = wl.M, wl.K, wl.N
    byts = N * K * 2 + M * K * 2 + M * N * 2 + M * 4
    flops = 2.0 * M * N * K
    touched = set()
    for i in range(M):
        s = int(wl.seq_slot[i])
        if 0 <= s < wl.max_loras and _scale_on(wl.adapters[s]):
            r = wl.adapters[s].rank
            flops += 2.0 * r * (K + N)
            touched.add(s)
    for s in touched:
        r = wl.adapters[s].rank
        byts += (r * K + N * r) * 2
    return float(byts), float(flops)


def embed_algorithmic(wl):
    """E rows read, y rows written, tokens and slots, plus each adapted row's
    B row and each touched slot's A (true ranks)."""
    M, n = wl.M, wl.n_embd
    byts = 2.0 * M * n * 2 + M * 4 * 2
    flops = 0.0
    touched = set()
    for i in range(M):
        s = int(wl.seq_slot[i])
        if 0 <= s < wl.max_loras and _scale_on(wl.adapters[s]):
            r = wl.adapters[s].rank
            byts += r * 2
            flops += 2.0 * r * n
            touched.add(s)
    for s in touched:
        byts += wl.adapters[s].rank * n * 2
    return float(byts), float(flops)


def moe_gather_algorithmic(wl):
    """W of every expert a slot-row names, x, y [tokens][N], indices, slots
    and combine weights, plus each expert's touched adapters at true rank."""
    T, K, N = wl.T, wl.K, wl.N
    byts = T * K * 2 + (T // wl.top_k) * N * 2 + T * 4 * 3
    flops = 2.0 * T * N * K
    for e in range(wl.E):
        rows = np.nonzero(wl.indices == e)[0]
        if len(rows) == 0:
            continue
        byts += N * K * 2
        touched = set()
        for j in rows:
            s = int(wl.seq_slot[j])
            if 0 <= s < wl.max_loras and _scale_on(wl.adapters[e][s]):
                flops += 2.0 * wl.adapters[e][s].rank * (K + N)
                touched.add(s)
        for s in touched:
            r = wl.adapters[e][s].rank
            byts += (r * K + N * r) * 2
    return float(byts), float(flops)


def stack_algorithmic(wl):
    """W + x + y + seq_slot, plus A and B of every member (scale not 0, true
    rank) of the slots the batch touches; flops 2MNK + per adapted row the
    members' 2 r (K + N)."""
    M, K, N = wl.M, wl.K, wl.N
    byts = N * K * 2 + M * K * 2 + M * N * 2 + M * 4
    flops = 2.0 * M * N * K
    touched = set()
    for i in range(M):
        s = int(wl.seq_slot[i])
        if 0 <= s < wl.max_loras:
            ms = [m for m in wl.stacks[s] if m.adapter_scale != 0.0]
            flops += sum(2.0 * m.rank * (K + N) for m in ms)
            if ms:
                touched.add(s)
    for s in touched:
        byts += sum((m.rank * K + N * m.rank) * 2 for m in wl.stacks[s] if m.adapter_scale != 0.0)
    return float(byts), float(flops)


def gate_up_algorithmic(wl):
    """The fused projection's bytes and flops with act [M][I] written instead
    of y [M][2I] (the halves are an intermediate)."""
    byts, flops = proj_algorithmic(wl)
    return byts - wl.M * wl.N * 2 + wl.M * (wl.N // 2) * 2, flops


def moe_algorithmic(wl):
    T, K, N = wl.T, wl.K, wl.N
    byts = T * K * 2 + T * N * 2 + T * 4 + (wl.E + 1) * 4
    flops = 2.0 * T * N * K
    for e in range(wl.E):
        a, b = int(wl.expert_offsets[e]), int(wl.expert_offsets[e + 1])
        if b > a:
            byts += N * K * 2
        touched = set()
        for j in range(a, b):
            s = int(wl.seq_slot[j])
            if 0 <= s < wl.max_loras and _scale_on(wl.adapters[e][s]):
                flops += 2.0 * wl.adapters[e][s].rank * (K + N)
                touched.add(s)
        for s in touched:
            r = wl.adapters[e][s].rank
            byts += (r * K + N * r) * 2
    return float(byts), float(flops)


# ----------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

# the sources each timed kernel is compiled from (a recorded DRAM figure holds
# while these are unchanged)
KERNEL_SOURCES = {
    "dec_kernel": ["lora_dec.cu", "ptx.cuh", "vec.cuh", "lora_internal.cuh"],
    "tc_kernel": ["lora_tc.cu", "shrink.cuh", "shrink_tc.cuh", "ptx.cuh", "vec.cuh", "lora_internal.cuh"],
    "simt_kernel": ["lora_simt.cu", "shrink.cuh", "vec.cuh", "lora_internal.cuh"],
    "embed_kernel": ["lora_embed.cu", "ptx.cuh", "lora_internal.cuh"],
}


def source_sha(kernel):
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "rank_delta_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(cdir, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config, kernel):
    """dram bytes per launch from a committed ncu capture, if the kernel's sources are unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(config)
    if not ent or ent.get("kernel") != kernel or ent.get("source_sha") != source_sha(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ProjSet:
    """One buffer set: its own copy of W, pool/tables, x, y and workspace."""

    def __init__(self, wl, th, rd, torch):
        self.x = th.to_device_bf16(wl.x)
        self.W = th.to_device_bf16(wl.W)
        self.slots = torch.from_numpy(wl.seq_slot.astype(np.int32)).cuda()
        self.route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
        self.route.pack_all(wl.adapters)
        self.y = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")
        self.ws = th.workspace(rd.lora_proj_workspace_bytes(wl.M, self.route.rt, PROJ_PATH[0]))
        self.bytes = (self.W.numel() * 2 + self.route.pool_bytes + self.x.numel() * 2 +
                      self.y.numel() * 2)

    def step(self, wl, rd, stream, x=None, slots=None, y=None):
        x = self.x if x is None else x
        slots = self.slots if slots is None else slots
        y = self.y if y is None else y
        rd.lora_proj_apply(x, x.stride(0), self.W, wl.M, wl.K, wl.N, slots, self.route.rt, y,
                           y.stride(0), self.ws, self.ws.numel(), stream, path=PROJ_PATH[0])


class MoeSet:
    def __init__(self, wl, th, rd, torch):
        self.x = th.to_device_bf16(wl.x)
        self.W = [th.to_device_bf16(w) for w in wl.W]
        self.off = torch.from_numpy(wl.expert_offsets.astype(np.int32)).cuda()
        self.slots = torch.from_numpy(wl.seq_slot.astype(np.int32)).cuda()
        self.routes = []
        for e in range(wl.E):
            r = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
            r.pack_all(wl.adapters[e])
            self.routes.append(r)
        self.rts = [r.rt for r in self.routes]
        self.y = torch.empty((wl.T, wl.N), dtype=torch.bfloat16, device="cuda")
        self.ws = th.workspace(rd.lora_moe_workspace_bytes(wl.E, wl.T, self.rts))
        self.bytes = (sum(w.numel() for w in self.W) * 2 + sum(r.pool_bytes for r in self.routes)
                      + self.x.numel() * 2 + self.y.numel() * 2)

    def step(self, wl, rd, stream, x=None, slots=None, y=None):
        x = self.x if x is None else x
        slots = self.slots if slots is None else slots
        y = self.y if y is None else y
        rd.lora_moe_down_apply(x, x.stride(0), self.W, self.off, wl.E, wl.T, wl.K, wl.N, slots,
                               self.rts, y, y.stride(0), self.ws, self.ws.numel(), stream)


class EmbedSet:
    """One buffer set of the embedding gather: its own E table, pool, tokens,
    slots, y and workspace (`like`: copy E from this set instead of the host)."""

    def __init__(self, wl, th, rd, torch, like=None):
        self.E = like.E.clone() if like is not None else th.to_device_bf16(wl.E)
        self.x = torch.from_numpy(wl.tokens.astype(np.int32)).cuda()  # the step's input: tokens
        self.slots = torch.from_numpy(wl.seq_slot.astype(np.int32)).cuda()
        self.route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.n_embd, wl.vocab, embed=True)
        # each adapter's flipped pair on the device once, packed from there into every set
        if like is None:
            self.pairs = [None if ad is None else
                          (th.to_device_bf16(ad.B), th.to_device_bf16(np.ascontiguousarray(ad.A.T)))
                          for ad in wl.adapters]
        else:
            self.pairs = like.pairs
        for s, ad in enumerate(wl.adapters):
            if ad is not None:
                rows, cols = self.pairs[s]
                rd.lora_embed_pool_pack(self.route.rt, s, rows, cols, ad.rank, ad.alpha,
                                        ad.use_rslora, ad.adapter_scale)
        self.y = torch.empty((wl.M, wl.n_embd), dtype=torch.bfloat16, device="cuda")
        self.ws = th.workspace(rd.lora_embed_workspace_bytes(wl.M, self.route.rt))
        # what one step touches (the rotation has to cover L2 with these)
        self.bytes = embed_algorithmic(wl)[0]

    def step(self, wl, rd, stream, x=None, slots=None, y=None):
        x = self.x if x is None else x
        slots = self.slots if slots is None else slots
        y = self.y if y is None else y
        rd.lora_embed_apply(x, self.E, wl.M, wl.vocab, wl.n_embd, slots, self.route.rt, y,
                            y.stride(0), self.ws, self.ws.numel(), stream)


class MoeGatherSet:
    """One buffer set of the decode MoE fold with the top-k combine."""

    def __init__(self, wl, th, rd, torch):
        self.x = th.to_device_bf16(wl.x)
        self.W = [th.to_device_bf16(w) for w in wl.W]
        self.idx = torch.from_numpy(wl.indices.astype(np.int32)).cuda()
        self.slots = torch.from_numpy(wl.seq_slot.astype(np.int32)).cuda()
        self.combine = torch.from_numpy(wl.combine.astype(np.float32)).cuda()
        self.routes = []
        for e in range(wl.E):
            r = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
            r.pack_all(wl.adapters[e])
            self.routes.append(r)
        self.rts = [r.rt for r in self.routes]
        self.y = torch.empty((wl.T // wl.top_k, wl.N), dtype=torch.bfloat16, device="cuda")
        self.ws = th.workspace(rd.lora_moe_gather_workspace_bytes(wl.E, wl.T, self.rts))
        self.bytes = (sum(w.numel() for w in self.W) * 2 + sum(r.pool_bytes for r in self.routes)
                      + self.x.numel() * 2 + self.y.numel() * 2)

    def step(self, wl, rd, stream, x=None, slots=None, y=None):
        x = self.x if x is None else x
        slots = self.slots if slots is None else slots
        y = self.y if y is None else y
        rd.lora_moe_gather_apply(x, x.stride(0), self.W, self.idx, wl.E, wl.T, wl.K, wl.N, slots, self.rts,
                                 self.combine, wl.top_k, y, y.stride(0), self.ws, self.ws.numel(), stream)


class StackSet(ProjSet):
    """A projection buffer set whose slots each hold a stack of adapters."""

    def __init__(self, wl, th, rd, torch):
        self.x = th.to_device_bf16(wl.x)
        self.W = th.to_device_bf16(wl.W)
        self.slots = torch.from_numpy(wl.seq_slot.astype(np.int32)).cuda()
        self.route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
        for s, st in enumerate(wl.stacks):
            self.route.pack_stack(s, st)
        self.y = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")
        self.ws = th.workspace(rd.lora_proj_workspace_bytes(wl.M, self.route.rt, PROJ_PATH[0]))
        self.bytes = (self.W.numel() * 2 + self.route.pool_bytes + self.x.numel() * 2 +
                      self.y.numel() * 2)


class GateUpSet(ProjSet):
    """A projection buffer set whose output is act [M][I]."""

    def __init__(self, wl, th, rd, torch):
        super().__init__(wl, th, rd, torch)
        self.I = wl.N // 2
        self.y = torch.empty((wl.M, self.I), dtype=torch.bfloat16, device="cuda")
        self.ws = th.workspace(rd.lora_gate_up_workspace_bytes(wl.M, self.route.rt))
        self.bytes = (self.W.numel() * 2 + self.route.pool_bytes + self.x.numel() * 2 +
                      self.y.numel() * 2 + self.ws.numel())

    def step(self, wl, rd, stream, x=None, slots=None, y=None):
        x = self.x if x is None else x
        slots = self.slots if slots is None else slots
        y = self.y if y is None else y
        rd.lora_gate_up_apply(x, x.stride(0), self.W, wl.M, wl.K, self.I, slots, self.route.rt, y,
                              y.stride(0), self.ws, self.ws.numel(), stream)


def max_over_ranks(ms: float, world: int, device: str) -> float:
    """The slowest rank's time: every rank runs an independent replica, so the
    job ends when the last one does."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(rows: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job rows/s: all ranks' rows over the slowest rank's time."""
    return rows * steps * world / (elapsed_ms / 1e3)


# kernels one call launches: the one-launch kernel (opt-in path) one; the
# tensor-core path the routing sort, then one fused launch (shrink tiles or
# units, base, expand-fold, split-K sum); the CUDA-core path (<= 16 rows) the
# sort, a shrink launch and the GEMV; the embedding gather the sort and one
# launch. Projection and gated calls ask the library's plan (lora_proj_plan),
# which also says whether a gated call needs the separate activation kernel.
LAUNCHES_DEC, LAUNCHES_TC, LAUNCHES_SIMT, LAUNCHES_EMBED = 1, 2, 3, 2
DEC_MAX_ROWS = 256


def launches_per_call(config, rows, kernel, rd=None, rt=None):
    if kernel == "embed_kernel":
        return LAUNCHES_EMBED
    if config == "moe_gather":  # expert sort + row copy, the grouped fold, the combine
        return LAUNCHES_TC + 2
    if kernel == "dec_kernel":
        return LAUNCHES_DEC
    if rd is not None and rt is not None and config not in ("moe",):
        return rd.lora_proj_plan(rows, rt, config in GATE_UP, PROJ_PATH[0])["kernels"]
    if config in GATE_UP: # the projection, then (at most) the activation kernel
        return launches_per_call(GATE_UP[config], rows, kernel) + 1
    if kernel == "simt_kernel":
        return LAUNCHES_SIMT
    return LAUNCHES_TC


def make_workload(config, small=False):
    import workloads
    if config in EMBED_ROWS:
        return workloads.embed(M=EMBED_ROWS[config])
    if config == "stack":
        return workloads.stacked()
    if config == "moe_gather":
        return workloads.moe_gather()
    if config in GATE_UP:
        base = GATE_UP[config]
        return workloads.make(base, **(SMALL.get(base, {}) if small else {}))
    return workloads.make(config, **(SMALL.get(config, {}) if small else {}))


SET_OF = {"moe": MoeSet, "stack": StackSet, "moe_gather": MoeGatherSet, "gate_up": GateUpSet,
          "gate_up_decode": GateUpSet, "embed": EmbedSet, "embed_prefill": EmbedSet}
# the configs of the default run: the headline (the largest workload, whose
# contraction is tensor-bound) first, then the other workloads with targets
SUITE = ["prefill", "decode", "qkv", "moe"]
EXTENDED = ["gate_up", "gate_up_decode", "moe_gather", "stack", "embed", "embed_prefill"]
MIN_CALLS = 100
STEADY_CALLS = 10  # calls per steady-state graph (calls under a millisecond)
PROJ_PATH = [0]    # lora_proj_apply path of the projection workloads (--path)


def algorithmic(config, wl):
    if config in EMBED_ROWS:
        return embed_algorithmic(wl)
    if config == "stack":
        return stack_algorithmic(wl)
    if config == "moe_gather":
        return moe_gather_algorithmic(wl)
    if config in GATE_UP:
        return gate_up_algorithmic(wl)
    if config == "moe":
        return moe_algorithmic(wl)
    return proj_algorithmic(wl)


def rows_of(config, wl):
    return wl.T if config in ("moe", "moe_gather") else wl.M


def config_dict(config, rows, world, small=False):
    """The workload description both arms print (the same keys and values)."""
    return {
        "workload": DESCRIBE[config] + (" [--small profiling case, not the benchmark]"
                                        if small and GATE_UP.get(config, config) in SMALL else ""),
        "rows_per_step": rows,
        "parallelism": f"replicas x{world} (rows shard, no collective)",
        "l2": "buffer sets rotate so one pass over them touches >= 3x L2 (129 MB); inputs of prefill and "
              "MoE exceed L2 on their own",
        "timing": "configs: value = rows / median per-call time in steady state (100 replays of one CUDA "
                  "graph of back-to-back calls, the buffer sets in turn, each replay between two CUDA events "
                  "on the launching stream); the isolated single-call latency beside it. Headline: exactly "
                  "K steps, each its own graph replay between events, value = rows / median step time",
    }


def kernel_of(config, rows):
    if config in EMBED_ROWS:
        return "embed_kernel"
    if config in ("moe", "moe_gather"):
        return "tc_kernel"
    if rows <= 16 and PROJ_PATH[0] == 0:
        return "simt_kernel"
    return "dec_kernel" if rows <= DEC_MAX_ROWS and PROJ_PATH[0] == 3 else "tc_kernel"


def per_call_us(torch, graphs, n, stream, world=1, barrier=False):
    """Device time of n single-call graph replays, each between its own pair
    of events (3 untimed replays first); a barrier and a synchronize on both
    sides of the timed replays."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(3):
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    if barrier and world > 1:
        torch.distributed.barrier()
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            graphs[i % len(graphs)].replay()
            b.record(stream)
    torch.cuda.synchronize()
    if barrier and world > 1:
        torch.distributed.barrier()
    return [a.elapsed_time(b) * 1e3 for a, b in evs]


def steady_us(torch, graph, calls, samples, stream):
    """Per-call device time in steady state: `samples` replays of one graph of
    `calls` back-to-back calls, each replay between its own pair of events (3
    untimed replays first); a sample is the replay's time / calls."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(samples)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 / calls for a, b in evs]


def summary(us):
    s = sorted(us)
    return {"calls": len(s), "median_us": s[len(s) // 2], "min_us": s[0],
            "mean_us": sum(s) / len(s), "max_us": s[-1]}


class Bench:
    """Device buffers, graphs and timings of one workload."""

    def __init__(self, config, args, world, small=False):
        import torch
        import rank_delta_gb300 as rd
        from rank_delta_gb300 import torch_helpers as th
        self.torch, self.rd, self.th = torch, rd, th
        self.config, self.args, self.world, self.small = config, args, world, small
        self.wl = make_workload(config, small)
        self.rows = rows_of(config, self.wl)
        self.algo_bytes, self.algo_flops = algorithmic(config, self.wl)
        Set = SET_OF.get(config, ProjSet)
        first = Set(self.wl, th, rd, torch)
        self.nsets = max(1, int(np.ceil(3 * L2_BYTES / first.bytes)))
        if config in EMBED_ROWS:
            self.sets = [first] + [EmbedSet(self.wl, th, rd, torch, like=first) for _ in range(self.nsets - 1)]
        else:
            self.sets = [first] + [Set(self.wl, th, rd, torch) for _ in range(self.nsets - 1)]
        self.set_bytes = first.bytes
        self.stream = torch.cuda.Stream()
        self.stream.wait_stream(torch.cuda.current_stream())
        self.base_slots = [torch.full_like(s.slots, -1) for s in self.sets]

    def graphs(self, base=False):
        torch, wl, rd = self.torch, self.wl, self.rd
        with torch.cuda.stream(self.stream):
            for i in range(self.args.warmup):
                k = i % self.nsets
                self.sets[k].step(wl, rd, self.stream, slots=self.base_slots[k] if base else None)
        torch.cuda.synchronize()
        gs = []
        for k in range(self.nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.sets[k].step(wl, rd, torch.cuda.current_stream(),
                                  slots=self.base_slots[k] if base else None)
            gs.append(g)
        return gs

    def steady_graph(self, calls, base=False):
        """One graph of `calls` back-to-back calls, the buffer sets in turn."""
        torch, wl, rd = self.torch, self.wl, self.rd
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(calls):
                k = i % self.nsets
                self.sets[k].step(wl, rd, torch.cuda.current_stream(),
                                  slots=self.base_slots[k] if base else None)
        return g

    def e2e(self, steps):
        """Rows/s end to end through the C ABI: every step copies its own
        inputs (pinned host x -- tokens for the embedding -- and seq_slot) to
        the device, makes the call and reads its result back to pinned host
        memory. The copies of step i+1 and the read-back of step i run on
        their own streams beside the call of step i; the K steps are one CUDA
        graph, replayed once untimed and once timed."""
        torch, wl, rd, sets, nsets = self.torch, self.wl, self.rd, self.sets, self.nsets
        cap = self.stream
        nio = max(2, nsets)
        x_h = sets[0].x.cpu().pin_memory()
        s_h = sets[0].slots.cpu().pin_memory()
        y_hs = [torch.empty(sets[0].y.shape, dtype=torch.bfloat16).pin_memory() for _ in range(nio)]
        xs = [torch.empty_like(sets[0].x) for _ in range(nio)]
        ss = [torch.empty_like(sets[0].slots) for _ in range(nio)]
        ys = [torch.empty_like(sets[0].y) for _ in range(nio)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        in_ev = [torch.cuda.Event() for _ in range(nio)]
        comp_ev = [torch.cuda.Event() for _ in range(nio)]
        out_ev = [torch.cuda.Event() for _ in range(nio)]

        def run(n, main):
            for i in range(n):
                k, j = i % nsets, i % nio
                with torch.cuda.stream(s_in):
                    if i >= nio:
                        s_in.wait_event(comp_ev[j])  # step i - nio has read xs[j], ss[j]
                    xs[j].copy_(x_h, non_blocking=True)
                    ss[j].copy_(s_h, non_blocking=True)
                    in_ev[j].record(s_in)
                main.wait_event(in_ev[j])
                if i >= nio:
                    main.wait_event(out_ev[j])  # step i - nio's y is back on the host
                sets[k].step(wl, rd, main, x=xs[j], slots=ss[j], y=ys[j])
                comp_ev[j].record(main)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_ev[j])
                    y_hs[j].copy_(ys[j], non_blocking=True)
                    out_ev[j].record(s_out)

        with torch.cuda.stream(cap):
            s_in.wait_stream(cap)
            s_out.wait_stream(cap)
            run(self.args.warmup, cap)
            cap.wait_stream(s_in)
            cap.wait_stream(s_out)
        torch.cuda.synchronize()
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=cap):
            main = torch.cuda.current_stream()
            s_in.wait_stream(main)
            s_out.wait_stream(main)
            run(steps, main)
            main.wait_stream(s_in)
            main.wait_stream(s_out)
        with torch.cuda.stream(cap):
            g2.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cap):
            e0.record(cap)
            g2.replay()
            e1.record(cap)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), self.world, "cuda")
        return {"value": job_rate(self.rows, steps, self.world, ms), "unit": "rows/s",
                "h2d_bytes_per_step": int(x_h.numel() * x_h.element_size() + s_h.numel() * 4),
                "d2h_bytes_per_step": int(y_hs[0].numel() * 2),
                "how": "one CUDA graph of the K steps: each step copies its own inputs from pinned host "
                       "memory and reads its result back to pinned host memory, the copies on two streams "
                       "beside the neighbouring calls"}

    def roofline(self, call_us):
        return roofline_of(self.config, self.rows, self.algo_bytes, self.algo_flops, call_us)


def roofline_of(config, rows, algo_bytes, algo_flops, call_us):
    """Achieved bytes (HBM-bound workloads) or flops (tensor-bound) per call
    over the call time, against the measured peak: the HBM copy figure, or
    the bf16 burst figure (one call is a sub-millisecond kernel timed alone)."""
    hbm, tf_burst, _tf_sus, peak_kind = load_peaks()
    bound = BOUND[config]
    s = call_us / 1e6
    if bound == "hbm":
        achieved, peak, unit = algo_bytes / s / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = algo_flops / s / 1e12, tf_burst, "TFLOP/s"
    kernel = kernel_of(config, rows)
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": recorded_traffic(config, kernel),
            "kernel": f"{kernel} (timed as the whole call, every launch of it)",
            "algorithmic_bytes_per_call": algo_bytes, "algorithmic_flops_per_call": algo_flops,
            "peak_source": (f"{peak_kind} {'HBM copy' if bound == 'hbm' else 'bf16 burst'} "
                            f"({'MEASURED_PEAKS.json' if peak_kind == 'measured' else 'MEASURED_PEAKS.json absent'})"),
            "call_us": call_us}


def measure(b, want_cpu=True):
    """One workload: per-call times of max(K, 100) calls (median, min), the
    same calls with every slot -1 (base only), the end-to-end rate, the
    roofline of the median call, and the oracle on the host cores."""
    torch, args, world, config = b.torch, b.args, b.world, b.config
    n = max(args.steps, MIN_CALLS)
    iso = summary(per_call_us(torch, b.graphs(), n, b.stream))
    calls = STEADY_CALLS if iso["median_us"] < 1000.0 else 1
    full = summary(steady_us(torch, b.steady_graph(calls), calls, n, b.stream))
    b.graphs(base=True)  # warm-up of the base-only calls
    base = summary(steady_us(torch, b.steady_graph(calls, base=True), calls, n, b.stream))
    med = max_over_ranks(full["median_us"], world, "cuda")
    ent = {
        "value": b.rows * world / (med / 1e6), "unit": "rows/s", "ms_per_step": med / 1e3,
        "per_call": dict(full, how=f"steady state: {n} replays of one CUDA graph of {calls} back-to-back "
                                   f"calls (the buffer sets in turn), each replay between its own events; "
                                   f"a sample is the replay time / {calls}"),
        "per_call_isolated": dict(iso, how="each call its own single-call graph replay between its own "
                                           "events: the latency of one call, the graph launch (about 5 us "
                                           "on this GPU) included"),
        "base_only": dict(base, how="steady state as per_call, every slot -1 (no adapter applied)",
                          delta_share=1.0 - base["median_us"] / full["median_us"]),
        "roofline": b.roofline(med),
        "e2e": b.e2e(args.steps),
        "gpu_launches_per_call": launches_per_call(config, b.rows, kernel_of(config, b.rows), b.rd,
                                                   getattr(getattr(b.sets[0], "route", None), "rt", None)),
        "status_flags": b.rd.lora_status_get(b.sets[0].ws),
        "config": config_dict(config, b.rows, world, b.small),
    }
    if want_cpu:
        ent["cpu_baseline"] = oracle_rate(b.wl, config, budget_s=8.0, cap_s=20.0)
    return ent


def run_ours(args, rank, world, local_rank):
    import torch
    import rank_delta_gb300 as rd
    from rank_delta_gb300 import build as rdbuild

    if rank == 0:
        rdbuild.build()
    if world > 1:
        torch.distributed.barrier()
    rd.lib()
    torch.cuda.set_device(local_rank)
    suite = args.config == "suite"
    head = "prefill" if suite else args.config
    rest = ([c for c in SUITE if c != head] + (EXTENDED if args.extended else [])) if suite else []
    want_cpu = world == 1 and not args.no_cpu_baseline

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    hb = Bench(head, args, world, args.small)
    # the timed region: exactly K steps, each its own graph replay between events
    us = per_call_us(torch, hb.graphs(), args.steps, hb.stream, world, barrier=True)
    med = max_over_ranks(sorted(us)[len(us) // 2], world, "cuda")
    head_ent = measure(hb, want_cpu)
    del hb
    torch.cuda.empty_cache()
    configs = {head: head_ent}
    for c in rest:
        bc = Bench(c, args, world)
        configs[c] = measure(bc, want_cpu)
        del bc
        torch.cuda.empty_cache()
    clk = clocks.stop()
    rows = head_ent["config"]["rows_per_step"]
    ra = head_ent["roofline"]
    out = {
        "metric": METRIC,
        "value": rows * world / (med / 1e6),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": med / 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the workload, no dataset)",
        "config": head_ent["config"],
        "clocks": clk,
        "e2e": head_ent["e2e"],
        "gpu_launches": head_ent["gpu_launches_per_call"] * args.steps,
        "roofline": dict(roofline_of(head, rows, ra["algorithmic_bytes_per_call"],
                                     ra["algorithmic_flops_per_call"], med),
                         per_call_timed_region=summary(us)),
        "status_flags": head_ent["status_flags"],
        "configs": configs,
    }
    if want_cpu:
        out["cpu_baseline"] = head_ent["cpu_baseline"]
    return out


# ----------------------------------------------------------------------------
# oracle timing (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------

def oracle_rate(wl, config, budget_s=12.0, cap_s=30.0):
    """Oracle rows/s on a bounded sample of the workload (whole rows, all columns)."""
    import oracle
    oracle.build()
    is_moe = config == "moe"
    rows_total = wl.T if config in ("moe", "moe_gather") else wl.M
    if config in EMBED_ROWS:
        def fn(w, rows):
            return oracle.embed(w.tokens[rows], w.E, w.seq_slot[rows], w.adapters)
    elif config in GATE_UP:
        def fn(w, rows):
            return oracle.gate_up(w.x, w.W, w.seq_slot, w.adapters, rows=rows)
    elif config == "stack":
        def fn(w, rows):
            return oracle.proj_stack(w.x, w.W, w.seq_slot, w.stacks, rows=rows)
    elif config == "moe_gather":
        def fn(w, rows):  # the sampled slot-rows (the fp32 combine of pairs is left out)
            return oracle.moe_gather(w.x[rows], w.W, w.indices[rows], w.seq_slot[rows], w.adapters)
    else:
        fn = oracle.workload_moe if is_moe else oracle.workload_proj
    # calibrate on a few rows, then size the sample to ~budget_s
    n0 = min(rows_total, 2)
    idx = np.arange(n0, dtype=np.int32)
    t = time.perf_counter()
    fn(wl, rows=idx)
    dt = max(time.perf_counter() - t, 1e-6)
    n = int(min(rows_total, max(n0, budget_s / (dt / n0))))
    rng = np.random.default_rng(0)
    idx = np.sort(rng.choice(rows_total, size=n, replace=False)).astype(np.int32)
    done, t = 0, time.perf_counter()
    while True:
        fn(wl, rows=idx)
        done += n
        el = time.perf_counter() - t
        if el >= min(budget_s, cap_s) or el + el / (done / n) > cap_s:
            break
    threads = oracle.max_threads()
    # the same loops on one core, over a short sample of the same rows
    oracle.set_threads(1)
    try:
        m = min(n, 2)
        done1, t1 = 0, time.perf_counter()
        while True:
            fn(wl, rows=idx[:m])
            done1 += m
            el1 = time.perf_counter() - t1
            if el1 >= min(3.0, budget_s / 4):
                break
    finally:
        oracle.set_threads(threads)
    return {"value": done / el, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "single_core_value": done1 / el1,
            "sample": f"{n} of {rows_total} rows (all "
                      f"{wl.n_embd if config in EMBED_ROWS else (wl.N // 2 if config in GATE_UP else wl.N)} "
                      f"output columns each), "
                      f"{done // n} pass(es), {el:.1f} s of fp32 C loops"}


def run_reference(args, rank, world):
    """The reference arm: the oracle (plain fp32 C loops) on the host cores,
    on the headline workload -- each step a bounded sample of it -- plus one
    bounded sample of every other workload of the run."""
    if rank != 0:
        return
    suite = args.config == "suite"
    head = "prefill" if suite else args.config
    rest = ([c for c in SUITE if c != head] + (EXTENDED if args.extended else [])) if suite else []
    wl = make_workload(head, args.small)
    rows = rows_of(head, wl)
    per = []
    cpu = None
    steps = max(1, args.steps)
    for _ in range(steps):
        cpu = oracle_rate(wl, head, budget_s=max(1.5, 40.0 / steps), cap_s=max(3.0, 60.0 / steps))
        per.append(cpu["value"])
    value = float(np.median(per))
    cpu["value"] = value
    configs = {head: {"value": value, "unit": "rows/s", "ms_per_step": rows / value * 1e3}}
    for c in rest:
        w = make_workload(c)
        r = oracle_rate(w, c, budget_s=5.0, cap_s=10.0)
        configs[c] = {"value": r["value"], "unit": "rows/s", "ms_per_step": rows_of(c, w) / r["value"] * 1e3,
                      "cpu_baseline": r}
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rows / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload, no dataset)",
        "config": config_dict(head, rows, world, args.small),
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "configs": configs,
        "note": "the reference is the CPU oracle (plain fp32 loops); no reference code exists to install",
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="suite", choices=["suite"] + sorted(DESCRIBE),
                    help="suite (default): prefill as the headline, decode, qkv and moe under 'configs'")
    ap.add_argument("--extended", action="store_true",
                    help="with the suite: also gate_up, gate_up_decode, moe_gather, stack, embed, embed_prefill")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "tc", "tc_one"],
                    help="lora_proj_apply path of the projection workloads (default: the library's choice)")
    ap.add_argument("--small", action="store_true",
                    help="profiling case: prefill 2048 rows, MoE 128 tokens (not the benchmarked workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    PROJ_PATH[0] = {"auto": 0, "tc": 2, "tc_one": 3}[args.path]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
