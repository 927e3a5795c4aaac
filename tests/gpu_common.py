"""Shared helpers of the GPU tests: run the CUDA path through the C ABI on a
workload and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import rank_delta_gb300 as rd
from rank_delta_gb300 import torch_helpers as th

# Tolerance for adapted rows: |gpu - oracle| <= ATOL + RTOL * |oracle|,
# element-wise (bf16 inputs, fp32 accumulation, bf16 output).
ATOL = 2e-2
RTOL = 1e-2

SENTINEL = 0x7FC1  # a NaN bf16 pattern: any output the kernels fail to write stays NaN


def assert_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str = ""):
    g = th.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    o = np.asarray(ref, dtype=np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU outputs (unwritten?)"
    err = np.abs(g - o)
    bad = err > ATOL + RTOL * np.abs(o)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"first at {tuple(i)}: gpu {g[tuple(i)]} oracle {o[tuple(i)]}; "
                             f"max abs err {err.max():.4g}")
    big = np.abs(o) >= 1.0
    rel = (err[big] / np.abs(o[big])).max() if big.any() else 0.0
    return float(err.max()), float(rel)


class ProjRun:
    """Device-resident copy of a ProjWorkload with its route packed."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        self.x = th.to_device_bf16(wl.x, device)
        self.W = th.to_device_bf16(wl.W, device)
        self.slots = torch.from_numpy(np.ascontiguousarray(wl.seq_slot, np.int32)).to(device)
        self.route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N, device)
        self.route.pack_all(wl.adapters)
        # sized for every path (the one-launch kernel's workspace is the larger)
        self.ws = th.workspace(rd.lora_proj_workspace_bytes(wl.M, self.route.rt, rd.LORA_PATH_TC_ONE), device)
        self.device = device

    def apply(self, slots=None, path=rd.LORA_PATH_AUTO, x=None, rows=None, ws_bytes=None):
        wl = self.wl
        x = self.x if x is None else x
        M = x.shape[0]
        s = self.slots if slots is None else slots
        y = torch.full((M, wl.N), 0, dtype=torch.int16, device=self.device)
        y.fill_(SENTINEL)
        y = y.view(torch.bfloat16)
        ws = self.ws if M <= wl.M else th.workspace(rd.lora_proj_workspace_bytes(M, self.route.rt,
                                                                                   rd.LORA_PATH_TC_ONE))
        rd.lora_proj_apply(x, x.stride(0), self.W, M, wl.K, wl.N, s, self.route.rt, y, y.stride(0),
                           ws, ws.numel() if ws_bytes is None else ws_bytes, None, path)
        torch.cuda.synchronize()
        self.last_status = rd.lora_status_get(ws)
        return th.to_numpy_bf16(y)


class EmbedRun:
    """Device-resident copy of an EmbedWorkload with its embedding route packed."""

    def __init__(self, wl, device="cuda", flipped=False):
        self.wl = wl
        self.E = th.to_device_bf16(wl.E, device)
        self.tokens = torch.from_numpy(np.ascontiguousarray(wl.tokens, np.int32)).to(device)
        self.slots = torch.from_numpy(np.ascontiguousarray(wl.seq_slot, np.int32)).to(device)
        self.route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.n_embd, wl.vocab, device,
                                    embed=True)
        for s, ad in enumerate(wl.adapters):
            if ad is not None:
                if flipped:
                    self.route.pack_flipped(s, ad)
                else:
                    self.route.pack(s, ad)
        self.ws = th.workspace(rd.lora_embed_workspace_bytes(wl.M, self.route.rt), device)
        self.device = device

    def apply(self, tokens=None, slots=None, y_stride=None):
        wl = self.wl
        tok = self.tokens if tokens is None else tokens
        s = self.slots if slots is None else slots
        M = tok.shape[0]
        ys = wl.n_embd if y_stride is None else y_stride
        y = torch.full((M, ys), SENTINEL, dtype=torch.int16, device=self.device)
        ws = self.ws if M <= wl.M else th.workspace(rd.lora_embed_workspace_bytes(M, self.route.rt))
        rd.lora_embed_apply(tok, self.E, M, wl.vocab, wl.n_embd, s, self.route.rt, y, ys, ws,
                            ws.numel())
        torch.cuda.synchronize()
        self.last_status = rd.lora_status_get(ws)
        return th.to_numpy_bf16(y.view(torch.bfloat16)[:, :wl.n_embd])
