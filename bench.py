#!/usr/bin/env python3
"""Benchmark of the multi-adapter LoRA projection on GB300.

One step = one lora_proj_apply (or lora_moe_down_apply) call over one batch:
the routing sort, the shrink, the base product and the fused expand-fold.
--config embed / embed_prefill time lora_embed_apply instead (the token
embedding row gather with the adapted rows: routing sort + one launch).
Default workload: the decode batch (64 rows, W [4096 x 4096] bf16, 16
adapters of ranks {8,16,32,64} in a rank-64 pool, 10% rows without adapter).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

N > 1 (under torchrun): every rank runs an independent replica on its own GPU
(the projection shards by rows with no exchange); value = all ranks' rows /
the slowest rank's time. Prints one JSON line on rank 0.
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
    "tc_kernel": ["lora_tc.cu", "shrink.cuh", "ptx.cuh", "vec.cuh", "lora_internal.cuh"],
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
        self.ws = th.workspace(rd.lora_proj_workspace_bytes(wl.M, self.route.rt))
        self.bytes = (self.W.numel() * 2 + self.route.pool_bytes + self.x.numel() * 2 +
                      self.y.numel() * 2)

    def step(self, wl, rd, stream, x=None, slots=None, y=None):
        x = self.x if x is None else x
        slots = self.slots if slots is None else slots
        y = self.y if y is None else y
        rd.lora_proj_apply(x, x.stride(0), self.W, wl.M, wl.K, wl.N, slots, self.route.rt, y,
                           y.stride(0), self.ws, self.ws.numel(), stream)


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
        self.ws = th.workspace(rd.lora_proj_workspace_bytes(wl.M, self.route.rt))
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


# kernels one call launches: the routing sort, then one fused tensor-core launch
# (shrink + base + expand-fold), with a tensor-core shrink launch between the
# two from 2048 projection rows; the CUDA-core path (<= 16 rows) runs the sort,
# a shrink launch and the GEMV; the embedding gather runs the sort and one launch
LAUNCHES_TC, LAUNCHES_SIMT, LAUNCHES_EMBED = 2, 3, 2
TC_SHRINK_MIN_ROWS = 2048


def launches_per_call(config, rows, kernel):
    if kernel == "embed_kernel":
        return LAUNCHES_EMBED
    if config == "moe_gather":  # expert sort + row copy, the grouped fold, the combine
        return LAUNCHES_TC + 2
    if config in GATE_UP: # the projection, then the activation kernel
        return launches_per_call(GATE_UP[config], rows, kernel) + 1
    if kernel == "simt_kernel":
        return LAUNCHES_SIMT
    if config != "moe" and rows >= TC_SHRINK_MIN_ROWS:
        return LAUNCHES_TC + 1
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


def run_ours(args, rank, world, local_rank):
    import torch
    import workloads
    import rank_delta_gb300 as rd
    from rank_delta_gb300 import build as rdbuild
    from rank_delta_gb300 import torch_helpers as th

    if rank == 0:
        rdbuild.build()
    if world > 1:
        torch.distributed.barrier()
    rd.lib()
    torch.cuda.set_device(local_rank)
    wl = make_workload(args.config, args.small)
    is_moe = args.config == "moe"
    slot_rows = args.config in ("moe", "moe_gather")
    is_embed = args.config in EMBED_ROWS
    rows = wl.T if slot_rows else wl.M
    is_gate_up = args.config in GATE_UP
    if is_embed:
        algo_bytes, algo_flops = embed_algorithmic(wl)
    elif args.config == "stack":
        algo_bytes, algo_flops = stack_algorithmic(wl)
    elif args.config == "moe_gather":
        algo_bytes, algo_flops = moe_gather_algorithmic(wl)
    elif is_gate_up:
        algo_bytes, algo_flops = gate_up_algorithmic(wl)
    else:
        algo_bytes, algo_flops = moe_algorithmic(wl) if is_moe else proj_algorithmic(wl)
    Set = MoeSet if is_moe else (EmbedSet if is_embed else (GateUpSet if is_gate_up else ProjSet))
    if args.config == "stack":
        Set = StackSet
    if args.config == "moe_gather":
        Set = MoeGatherSet
    first = Set(wl, th, rd, torch)
    nsets = max(1, int(np.ceil(3 * L2_BYTES / first.bytes)))
    if is_embed:
        sets = [first] + [EmbedSet(wl, th, rd, torch, like=first) for _ in range(nsets - 1)]
    else:
        sets = [first] + [Set(wl, th, rd, torch) for _ in range(nsets - 1)]
    stream = torch.cuda.current_stream()

    # The timed region replays one CUDA graph holding the K steps (each step's
    # kernels as graph nodes, buffer sets rotating), so the device time is the
    # kernels' own and not the host's enqueue rate.
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for i in range(args.warmup):
            sets[i % nsets].step(wl, rd, cap)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(args.steps):
            sets[i % nsets].step(wl, rd, torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        graph.replay()  # one untimed replay: the graph's own first-launch costs
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        t_start.record(cap)
        graph.replay()
        t_end.record(cap)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # keep replaying ~1 s so the clock sampler sees the GPU under the same load
    t_keep = time.time()
    with torch.cuda.stream(cap):
        while time.time() - t_keep < 1.0:
            graph.replay()
            torch.cuda.synchronize()
    clk = clocks.stop()

    elapsed_ms = t_start.elapsed_time(t_end)
    call_ms = elapsed_ms / args.steps
    elapsed_ms = max_over_ranks(elapsed_ms, world, "cuda")
    ms_per_step = elapsed_ms / args.steps
    value = job_rate(rows, args.steps, world, elapsed_ms)
    status = rd.lora_status_get(sets[0].ws)

    # end to end through the C ABI: every step copies its own inputs (pinned
    # host x -- tokens for the embedding -- and seq_slot) to the device, makes
    # the call, and reads its result back to pinned host memory. The copies of
    # step i+1 and the read-back of step i run on their own streams beside the
    # call of step i (buffer set i % nsets; events order each set's reuse), as
    # a serving loop would overlap them.
    # input/output buffers of the steps in flight: at least two, so that one
    # step's copies can overlap another's call even with one weight set
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

    def e2e_steps(n, main):
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

    # eager warm-up, then the K steps as one CUDA graph (copy nodes from and to
    # pinned host memory, the calls' kernels), replayed once untimed and once
    # timed, so the host's enqueue rate does not set the number
    with torch.cuda.stream(cap):
        s_in.wait_stream(cap)
        s_out.wait_stream(cap)
        e2e_steps(args.warmup, cap)
        cap.wait_stream(s_in)
        cap.wait_stream(s_out)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=cap):
        main = torch.cuda.current_stream()
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        e2e_steps(args.steps, main)
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
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
    e2e_value = job_rate(rows, args.steps, world, e2e_ms)

    # per-call device times: one graph per buffer set holding a single call,
    # each replay between two events on the launching stream, 100 replays
    # after 3 untimed ones; the median and the minimum are reported beside the
    # mean of the timed region (a failure here only drops these figures)
    try:
        one = []
        for k in range(nsets):
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=cap):
                sets[k].step(wl, rd, torch.cuda.current_stream())
            one.append(g1)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(100)]
        with torch.cuda.stream(cap):
            for i in range(3):
                one[i % nsets].replay()
            for i, (a, b) in enumerate(evs):
                a.record(cap)
                one[i % nsets].replay()
                b.record(cap)
        torch.cuda.synchronize()
        us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
        per_call = {"calls": len(us), "median_us": us[len(us) // 2], "min_us": us[0],
                    "how": "one graph of a single call per buffer set, events around each replay "
                           "(includes the graph's own launch gap, so above the mean of the K-step graph)"}
    except Exception as ex:  # noqa: BLE001
        per_call = {"error": f"{type(ex).__name__}: {ex}"[:200]}

    hbm, tf_burst, tf_sus, peak_kind = load_peaks()
    avg_call_s = call_ms / 1e3
    bound = BOUND[args.config]
    if bound == "hbm":
        achieved = algo_bytes / avg_call_s / 1e9
        peak, unit = hbm, "GB/s"
    else:
        achieved = algo_flops / avg_call_s / 1e12
        # a contraction timed over a long back-to-back loop runs in the
        # power-capped regime the sustained figure was measured in; a short
        # one is compared with the burst figure
        long_loop = elapsed_ms >= 100.0
        peak, unit = (tf_sus if long_loop else tf_burst), "TFLOP/s"
        peak_kind = (f"{peak_kind} sustained (timed region {elapsed_ms:.0f} ms of back-to-back calls; "
                     f"{achieved / tf_burst:.3f} of the burst {tf_burst})" if long_loop else
                     f"{peak_kind} burst")
    if is_embed:
        kernel = "embed_kernel"
    else:
        kernel = "tc_kernel" if (is_moe or rows > 16) else "simt_kernel"
    traffic = recorded_traffic(args.config, kernel)
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the workload, no dataset)",
        "config": {
            "workload": DESCRIBE[args.config] + (" [--small profiling case, not the benchmark]"
                                                 if args.small and GATE_UP.get(args.config, args.config) in SMALL
                                                 else ""),
            "rows_per_step": rows,
            "parallelism": f"replicas x{world} (rows shard, no collective)",
            "l2": f"rotating {nsets} buffer sets of {first.bytes / 1e6:.1f} MB "
                  f"{'touched per step ' if is_embed else ''}(>= 3x L2)",
            "timing": "CUDA events around one replay of a graph of the K steps",
        },
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "rows/s",
                "h2d_bytes_per_step": int(x_h.numel() * x_h.element_size() + s_h.numel() * 4),
                "d2h_bytes_per_step": int(y_hs[0].numel() * 2),
                "how": "one CUDA graph of the K steps: each step copies its own inputs from pinned host "
                       "memory and reads its result back to pinned host memory, the copies on two streams "
                       "beside the neighbouring calls"},
        "gpu_launches": launches_per_call(args.config, rows, kernel) * args.steps,
        "roofline": {
            "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic,
            "kernel": f"{kernel} (timed as the whole call: routing sort + {kernel}, graph replay)",
            "algorithmic_bytes_per_call": algo_bytes, "algorithmic_flops_per_call": algo_flops,
            "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind.startswith("measured") else
                            f"{peak_kind} (MEASURED_PEAKS.json absent)"),
            "call_us": call_ms * 1e3,
            "per_call": per_call,
        },
        "status_flags": status,
    }
    return out, wl


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
    if rank != 0:
        return
    wl = make_workload(args.config)
    per = []
    cpu = None
    for _ in range(args.warmup):
        pass
    for _ in range(max(1, args.steps)):
        cpu = oracle_rate(wl, args.config, budget_s=max(2.0, 60.0 / max(1, args.steps)),
                          cap_s=max(4.0, 90.0 / max(1, args.steps)))
        per.append(cpu["value"])
    value = float(np.median(per))
    rows = wl.T if args.config in ("moe", "moe_gather") else wl.M
    cpu["value"] = value
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rows / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)",
        "config": {"workload": DESCRIBE[args.config], "rows_per_step": rows,
                   "note": "the reference is the CPU oracle (plain fp32 loops), no reference code "
                           "exists to install"},
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="decode", choices=sorted(DESCRIBE))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true",
                    help="profiling case: prefill 2048 rows, MoE 128 tokens (not the benchmarked workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
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
    out, wl = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = oracle_rate(wl, args.config)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
