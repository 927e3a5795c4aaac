"""Device-memory plumbing with PyTorch for callers of the C ABI (tests, bench).

Only allocation and copies live here; every step of the projection runs in
the CUDA library through the binding in ``rank_delta_gb300``.
"""
from __future__ import annotations

import numpy as np
import torch

import rank_delta_gb300 as rd


def to_device_bf16(u16: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bits (numpy) -> torch.bfloat16 tensor on `device`."""
    a = np.ascontiguousarray(u16, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def to_numpy_bf16(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 tensor -> uint16 bits (numpy, host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class DeviceRoute:
    """A route whose pool and tables are torch allocations on one device.

    ``embed=True`` makes a token-embedding route: n_in is n_embd and n_out is
    the vocabulary (the adapted matrix is [vocab][n_embd]).
    """

    def __init__(self, max_loras: int, max_rank: int, n_in: int, n_out: int, device="cuda",
                 stream=None, embed: bool = False):
        self.L, self.R, self.K, self.N = max_loras, max_rank, n_in, n_out
        self.pool_bytes = rd.lora_pool_bytes(max_loras, max_rank, n_in, n_out)
        self.table_bytes = rd.lora_route_table_bytes(max_loras)
        self.pool = torch.empty(self.pool_bytes, dtype=torch.uint8, device=device)
        self.tables = torch.empty(self.table_bytes, dtype=torch.uint8, device=device)
        self.rt = rd.lora_route()
        if embed:
            rd.lora_embed_route_init(self.rt, self.pool, self.pool_bytes, self.tables,
                                     self.table_bytes, max_loras, max_rank, n_out, n_in, stream)
        else:
            rd.lora_route_init(self.rt, self.pool, self.pool_bytes, self.tables, self.table_bytes,
                               max_loras, max_rank, n_in, n_out, stream)

    def pack_flipped(self, slot: int, adapter, stream=None) -> None:
        """Pack a ``workloads.Adapter`` of an embedding route through the
        flipped pair: rows = B [vocab][rank], cols = A^T [n_embd][rank]."""
        rd.lora_embed_pool_pack(self.rt, slot, np.ascontiguousarray(adapter.B),
                                np.ascontiguousarray(np.asarray(adapter.A).T), adapter.rank,
                                adapter.alpha, adapter.use_rslora, adapter.adapter_scale, stream)

    def pack(self, slot: int, adapter, stream=None) -> None:
        """Pack a ``workloads.Adapter`` (host bf16 bits) into `slot`."""
        rd.lora_pool_pack(self.rt, slot, np.ascontiguousarray(adapter.A),
                          np.ascontiguousarray(adapter.B), adapter.rank, adapter.alpha,
                          adapter.use_rslora, adapter.adapter_scale, stream)

    def pack_stack(self, slot: int, members, stream=None) -> None:
        """Pack a list of ``workloads.Adapter`` into `slot` as one stack."""
        rd.lora_pool_pack_stack(self.rt, slot, [np.ascontiguousarray(m.A) for m in members],
                                [np.ascontiguousarray(m.B) for m in members], [m.rank for m in members],
                                [m.alpha for m in members], [m.use_rslora for m in members],
                                [m.adapter_scale for m in members], stream)

    def pack_all(self, adapters, stream=None) -> None:
        for s, ad in enumerate(adapters):
            if ad is not None:
                self.pack(s, ad, stream)

    def scale_table(self) -> np.ndarray:
        n = self.L
        off = self.rt.scale_table - self.tables.data_ptr()
        return self.tables[off:off + 4 * n].cpu().numpy().view(np.float32).copy()
