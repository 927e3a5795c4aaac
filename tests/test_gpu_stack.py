"""Several adapters on one matrix (a slot holding a stack of adapters,
ferrox-core weight_matrix/lora.rs LoraStack) on the GPU, through the C ABI,
against the oracle's stack sum (GPU only).

Tolerance as everywhere: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| per element;
rows with no delta are byte-identical to the GPU's own base-only run.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from rank_delta_gb300 import torch_helpers as th
from tests.gpu_common import SENTINEL, assert_close

pytestmark = pytest.mark.gpu

PATHS = [rd.LORA_PATH_SIMT, rd.LORA_PATH_TC]


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return rd.lib()


class StackRun:
    """Device-resident copy of a StackWorkload, every slot packed as a stack."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        self.x = th.to_device_bf16(wl.x, device)
        self.W = th.to_device_bf16(wl.W, device)
        self.slots = torch.from_numpy(np.ascontiguousarray(wl.seq_slot, np.int32)).to(device)
        self.route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N, device)
        for s, st in enumerate(wl.stacks):
            self.route.pack_stack(s, st)
        self.ws = th.workspace(rd.lora_proj_workspace_bytes(wl.M, self.route.rt), device)

    def apply(self, slots=None, path=rd.LORA_PATH_AUTO):
        wl = self.wl
        s = self.slots if slots is None else slots
        y = torch.full((wl.M, wl.N), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        rd.lora_proj_apply(self.x, self.x.stride(0), self.W, wl.M, wl.K, wl.N, s, self.route.rt, y,
                           y.stride(0), self.ws, self.ws.numel(), None, path)
        torch.cuda.synchronize()
        assert rd.lora_status_get(self.ws) == 0
        return th.to_numpy_bf16(y)

    def base(self, path=rd.LORA_PATH_AUTO):
        return self.apply(slots=torch.full_like(self.slots, -1), path=path)


@pytest.fixture(scope="module")
def stack64():
    return StackRun(workloads.stacked(seed=7, M=64, K=1024, N=2048, L=8, R=64))


@pytest.fixture(scope="module")
def stack64_ref(stack64):
    wl = stack64.wl
    return oracle.proj_stack(wl.x, wl.W, wl.seq_slot, wl.stacks)


@pytest.mark.parametrize("path", PATHS)
def test_stack_matches_oracle(stack64, stack64_ref, path):
    y = stack64.apply(path=path)
    assert_close(y, stack64_ref, f"stack path {path}")
    none = stack64.wl.seq_slot < 0
    base = stack64.base(path=path)
    assert none.any()
    assert np.array_equal(y[none], base[none])
    assert not np.array_equal(y[~none], base[~none])


def test_stack_of_one_is_the_single_pack(stack64):
    """On the tensor-core path a one-member stack and lora_pool_pack of that
    adapter give the same bytes (the rank factor is the adapter's scale, the
    slot scale 1, and s * 1 == 1 * s)."""
    wl = stack64.wl
    single = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
    one = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
    for s, st in enumerate(wl.stacks):
        m = [a for a in st if a.adapter_scale != 0.0][0]
        single.pack(s, m)
        one.pack_stack(s, [m])
    ys = []
    for route in (single, one):
        y = torch.full((wl.M, wl.N), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        rd.lora_proj_apply(stack64.x, wl.K, stack64.W, wl.M, wl.K, wl.N, stack64.slots, route.rt, y, wl.N,
                           stack64.ws, stack64.ws.numel(), None, rd.LORA_PATH_TC)
        torch.cuda.synchronize()
        ys.append(th.to_numpy_bf16(y))
    assert np.array_equal(ys[0], ys[1])


def test_stack_set_scale_multiplies_the_whole_stack(stack64):
    wl = stack64.wl
    s0 = int(wl.seq_slot[wl.seq_slot >= 0][0])
    rows = wl.seq_slot == s0
    try:
        rd.lora_set_scale(stack64.route.rt, s0, 0.0)
        y0 = stack64.apply(path=rd.LORA_PATH_TC)
        assert np.array_equal(y0[rows], stack64.base(path=rd.LORA_PATH_TC)[rows])
        rd.lora_set_scale(stack64.route.rt, s0, 2.0)
        y2 = stack64.apply(path=rd.LORA_PATH_TC)
        doubled = [list(st) for st in wl.stacks]
        doubled[s0] = [workloads.Adapter(m.A, m.B, m.rank, m.alpha, m.use_rslora, 2.0 * m.adapter_scale)
                       for m in wl.stacks[s0]]
        ref = oracle.proj_stack(wl.x, wl.W, wl.seq_slot, doubled)
        assert_close(y2[rows], ref[rows], "stack at scale 2")
    finally:
        rd.lora_set_scale(stack64.route.rt, s0, 1.0)


def test_stack_with_every_scale_zero_is_an_empty_slot(stack64):
    wl = stack64.wl
    route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
    for s, st in enumerate(wl.stacks):
        route.pack_stack(s, [workloads.Adapter(m.A, m.B, m.rank, m.alpha, m.use_rslora, 0.0) for m in st]
                         if s == 0 else st)
    y = torch.full((wl.M, wl.N), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    rd.lora_proj_apply(stack64.x, wl.K, stack64.W, wl.M, wl.K, wl.N, stack64.slots, route.rt, y, wl.N,
                       stack64.ws, stack64.ws.numel(), None, rd.LORA_PATH_TC)
    torch.cuda.synchronize()
    y = th.to_numpy_bf16(y)
    rows = wl.seq_slot == 0
    assert rows.any()
    assert np.array_equal(y[rows], stack64.base(path=rd.LORA_PATH_TC)[rows])


def test_stack_large_batch_tensor_core_shrink():
    """From 2048 rows h comes from the tensor-core shrink tiles inside the
    projection launch."""
    wl = workloads.stacked(seed=8, M=2048, K=512, N=384, L=6, R=64)
    run = StackRun(wl)
    y = run.apply()
    rows = np.random.default_rng(0).choice(wl.M, size=96, replace=False)
    ref = oracle.proj_stack(wl.x, wl.W, wl.seq_slot, wl.stacks, rows=rows)
    assert_close(y[rows], ref, "stack 2048 rows")
    none = wl.seq_slot < 0
    assert np.array_equal(y[none], run.base()[none])


@pytest.mark.parametrize("path", PATHS)
def test_stack_filling_the_pool_rank_with_odd_ranks(path):
    """Members of ranks 3, 5 and 8 (16 = the pool rank) and 1 + 7 on another
    slot: member boundaries off the 8-wide vectors, the pool rank used up."""
    base = workloads.stacked(seed=9, M=40, K=512, N=384, L=3, R=16, zero_member_slot=-1)
    rng = np.random.default_rng(1)

    def member(r, sc):
        A = workloads.f32_to_bf16(rng.uniform(-0.05, 0.05, (r, base.K)).astype(np.float32))
        B = workloads.f32_to_bf16((rng.standard_normal((base.N, r)) * 0.1).astype(np.float32))
        return workloads.Adapter(A, B, r, 2.0 * r, False, sc)

    stacks = [[member(3, 1.0), member(5, 0.5), member(8, 1.0)], [member(1, 1.0), member(7, 0.5)],
              [member(16, 1.0)]]
    wl = workloads.StackWorkload("odd", 9, base.M, base.K, base.N, 3, 16, base.W, base.x, base.seq_slot, stacks)
    run = StackRun(wl)
    y = run.apply(path=path)
    assert_close(y, oracle.proj_stack(wl.x, wl.W, wl.seq_slot, wl.stacks), "odd-rank stacks")


def test_stack_replaces_a_single_adapter_in_place(stack64, stack64_ref):
    """Packing a stack over a slot that held one adapter (and back) takes
    effect for the applies enqueued after it."""
    wl = stack64.wl
    s0 = int(wl.seq_slot[wl.seq_slot >= 0][0])
    rows = wl.seq_slot == s0
    single = wl.stacks[s0][0]
    try:
        stack64.route.pack(s0, single)
        y1 = stack64.apply(path=rd.LORA_PATH_TC)
        one = [list(st) for st in wl.stacks]
        one[s0] = [single]
        assert_close(y1[rows], oracle.proj_stack(wl.x, wl.W, wl.seq_slot, one)[rows], "single in a stack slot")
    finally:
        stack64.route.pack_stack(s0, wl.stacks[s0])
    y2 = stack64.apply(path=rd.LORA_PATH_TC)
    assert_close(y2, stack64_ref, "stack packed again")
