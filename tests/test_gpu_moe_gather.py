"""Decode-path MoE fold keyed by per-slot-row expert indices, with top-k
combine weights: CUDA path vs the oracle and vs the grouped fold, through the
C ABI (GPU only).

Without weights each slot-row must equal, byte for byte, the grouped fold
(lora_moe_down_apply) of the same rows sorted by expert; rows with no delta
equal the GPU's own all-(-1) run. With weights the token row is a weighted
sum of slot-rows, so the tolerance is the projection's carried through it:
|gpu - oracle| <= 2e-2 + 1e-2 * sum_i w_i |v_i|.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from rank_delta_gb300 import torch_helpers as th
from tests.gpu_common import ATOL, RTOL, SENTINEL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return rd.lib()


class GatherRun:
    def __init__(self, wl):
        self.wl = wl
        self.x = th.to_device_bf16(wl.x)
        self.W = [th.to_device_bf16(w) for w in wl.W]
        self.idx = torch.from_numpy(np.ascontiguousarray(wl.indices, np.int32)).cuda()
        self.slots = torch.from_numpy(np.ascontiguousarray(wl.seq_slot, np.int32)).cuda()
        self.comb = torch.from_numpy(np.ascontiguousarray(wl.combine, np.float32)).cuda()
        self.routes = []
        for e in range(wl.E):
            r = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
            r.pack_all(wl.adapters[e])
            self.routes.append(r)
        self.rts = [r.rt for r in self.routes]
        self.ws = th.workspace(rd.lora_moe_gather_workspace_bytes(wl.E, wl.T, self.rts))

    def apply(self, combine=True, idx=None, slots=None):
        wl = self.wl
        rows = wl.T // wl.top_k if combine else wl.T
        y = torch.full((rows, wl.N), SENTINEL, dtype=torch.int16, device="cuda")
        rd.lora_moe_gather_apply(self.x, self.x.stride(0), self.W, self.idx if idx is None else idx, wl.E,
                                 wl.T, wl.K, wl.N, self.slots if slots is None else slots, self.rts,
                                 self.comb if combine else None, wl.top_k, y, wl.N, self.ws, self.ws.numel())
        torch.cuda.synchronize()
        self.last_status = rd.lora_status_get(self.ws)
        return th.to_numpy_bf16(y.view(torch.bfloat16))

    def grouped(self, order):
        """lora_moe_down_apply on the rows sorted by expert (stably)."""
        wl = self.wl
        o = torch.from_numpy(order.astype(np.int64)).cuda()
        xs = self.x[o].contiguous()
        ss = self.slots[o].contiguous()
        offs = np.zeros(wl.E + 1, dtype=np.int32)
        offs[1:] = np.cumsum(np.bincount(wl.indices, minlength=wl.E))
        d_off = torch.from_numpy(offs).cuda()
        y = torch.full((wl.T, wl.N), SENTINEL, dtype=torch.int16, device="cuda")
        ws = th.workspace(rd.lora_moe_workspace_bytes(wl.E, wl.T, self.rts))
        rd.lora_moe_down_apply(xs, xs.stride(0), self.W, d_off, wl.E, wl.T, wl.K, wl.N, ss, self.rts, y, wl.N,
                               ws, ws.numel())
        torch.cuda.synchronize()
        return th.to_numpy_bf16(y.view(torch.bfloat16))


def assert_close_combined(gpu_bits, wl, rows_f32, what):
    """rows_f32: the oracle's slot-row values [T][N]."""
    w = wl.combine.astype(np.float64)[:, None]
    v = rows_f32.astype(np.float64)
    ok_rows = ((wl.indices >= 0) & (wl.indices < wl.E))[:, None]
    wv = np.where(ok_rows, w * v, 0.0)
    ref = wv.reshape(-1, wl.top_k, wl.N).sum(axis=1)
    tol = ATOL + RTOL * np.abs(wv).reshape(-1, wl.top_k, wl.N).sum(axis=1)
    g = th.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU outputs"
    bad = np.abs(g - ref) > tol
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[0])


@pytest.fixture(scope="module")
def small():
    return GatherRun(workloads.moe_gather(seed=61, tokens=40, E=5, top_k=2, K=512, N=384, rank=16))


def test_gather_rows_equal_the_grouped_fold(small):
    wl = small.wl
    rows = small.apply(combine=False)
    assert small.last_status == 0
    order = np.argsort(wl.indices, kind="stable")
    grouped = small.grouped(order)
    assert np.array_equal(rows[order], grouped)
    assert_close(rows, oracle.workload_moe_gather(wl, with_combine=False), "gather rows")


def test_gather_combined_matches_oracle(small):
    wl = small.wl
    y = small.apply(combine=True)
    assert_close_combined(y, wl, oracle.workload_moe_gather(wl, with_combine=False), "gather combined")


def test_gather_no_delta_rows_are_base_bytes(small):
    wl = small.wl
    rows = small.apply(combine=False)
    base = small.apply(combine=False, slots=torch.full_like(small.slots, -1))
    nod = np.where((wl.seq_slot < 0) | (wl.seq_slot >= wl.max_loras))[0]
    assert nod.size
    assert np.array_equal(rows[nod], base[nod])


def test_gather_expert_out_of_range_adds_nothing(small):
    wl = small.wl
    idx = wl.indices.copy()
    idx[[3, 10]] = [wl.E, -1]
    rows = small.apply(combine=False, idx=torch.from_numpy(idx).cuda())
    assert small.last_status & rd.LORA_FLAG_EXPERT_RANGE
    assert not rows[3].any() and not rows[10].any()
    ref = oracle.moe_gather(wl.x, wl.W, idx, wl.seq_slot, wl.adapters)
    keep = np.setdiff1d(np.arange(wl.T), [3, 10])
    assert_close(rows[keep], ref[keep], "gather with bad indices")
    y = small.apply(combine=True, idx=torch.from_numpy(idx).cuda())
    wl2 = workloads.MoeGatherWorkload(**{**wl.__dict__, "indices": idx})
    assert_close_combined(y, wl2, ref, "gather combined with bad indices")


def test_gather_decode_shapes_sampled():
    wl = workloads.moe_gather()  # 64 tokens top-2, 8 experts of [4096][14336]
    run = GatherRun(wl)
    y = run.apply(combine=True)
    assert run.last_status == 0
    rows = oracle.workload_moe_gather(wl, with_combine=False)
    assert_close_combined(y, wl, rows, "gather decode")


def test_gather_top1_and_ragged_shapes():
    wl = workloads.moe_gather(seed=62, tokens=33, E=3, top_k=1, K=200, N=100, rank=8)
    run = GatherRun(wl)
    y = run.apply(combine=True)
    assert_close_combined(y, wl, oracle.workload_moe_gather(wl, with_combine=False), "gather top-1")
