"""The full-size workloads through the C ABI in the launch configuration the
bench times, every output row and column checked against the oracle, plus
properties that hold at any size (GPU only).

The oracle's outputs of the large workloads are computed once per module and
shared by the tests that read them (about 20 s for the prefill batch on the
host cores)."""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from rank_delta_gb300 import torch_helpers as th
from tests.gpu_common import SENTINEL, ProjRun, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available()
    return rd.lib()


def assert_all_rows(y, ref, what):
    """Every row and column within tolerance; the message names the row count."""
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    assert_close(y, ref, f"{what} (all {y.shape[0]} rows x {y.shape[1]} columns)")


@pytest.fixture(scope="module")
def qkv():
    return ProjRun(workloads.make("qkv"))


PATHS = [rd.LORA_PATH_AUTO, rd.LORA_PATH_TC_ONE]


@pytest.mark.parametrize("path", PATHS)
def test_qkv_matches_oracle_on_every_row(qkv, path):
    y = qkv.apply(path=path)
    assert qkv.last_status == 0
    assert_all_rows(y, oracle.workload_proj(qkv.wl), "qkv")


@pytest.mark.parametrize("path", PATHS)
def test_qkv_fused_equals_three_split_calls(qkv, path):
    """One A per adapter, B rows split q/k/v: the fused call's bytes equal the
    stacked split calls' bytes (frink lora_attach.rs module doc)."""
    wl = qkv.wl
    fused = qkv.apply(path=path)
    parts = []
    row0 = 0
    for n in wl.splits:
        sub = workloads.ProjWorkload(
            f"qkv{row0}", wl.seed, wl.M, wl.K, n, wl.max_loras, wl.max_rank,
            np.ascontiguousarray(wl.W[row0:row0 + n]), wl.x, wl.seq_slot,
            [workloads.Adapter(a.A, np.ascontiguousarray(a.B[row0:row0 + n]), a.rank, a.alpha,
                               a.use_rslora, a.adapter_scale) for a in wl.adapters])
        parts.append(ProjRun(sub).apply(path=path))
        row0 += n
    assert np.array_equal(fused, np.concatenate(parts, axis=1))


@pytest.mark.parametrize("path", PATHS)
def test_qkv_no_delta_rows_are_base_bytes(qkv, path):
    wl = qkv.wl
    y = qkv.apply(path=path)
    base = qkv.apply(slots=torch.full_like(qkv.slots, -1), path=path)
    scales = np.array([oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale)
                       for a in wl.adapters])
    none = (wl.seq_slot < 0) | (scales[np.maximum(wl.seq_slot, 0)] == 0.0)
    assert none.sum() > int((wl.seq_slot < 0).sum())  # includes zero-scale adapters
    assert np.array_equal(y[none], base[none])


@pytest.mark.parametrize("path", PATHS)
def test_gated_q_fused_equals_split_and_matches_oracle(path):
    """A gated query projection, output [q | gate] twice the query width,
    one A per adapter and B rows split q / gate (spark_model lora_delta.rs,
    the attention weight holder's gated q width): the fused call matches the
    oracle on every row and its bytes equal the two split calls'."""
    wl = workloads.make("gated_q")
    run = ProjRun(wl)
    fused = run.apply(path=path)
    assert run.last_status == 0
    assert_all_rows(fused, oracle.workload_proj(wl), "gated q [q | gate]")
    parts, runs, row0 = [], [], 0
    for n in wl.splits:
        sub = workloads.ProjWorkload(
            f"gq{row0}", wl.seed, wl.M, wl.K, n, wl.max_loras, wl.max_rank,
            np.ascontiguousarray(wl.W[row0:row0 + n]), wl.x, wl.seq_slot,
            [workloads.Adapter(a.A, np.ascontiguousarray(a.B[row0:row0 + n]), a.rank, a.alpha,
                               a.use_rslora, a.adapter_scale) for a in wl.adapters])
        sr = ProjRun(sub)
        parts.append(sr.apply(path=path))
        runs.append(sr)
        row0 += n
    # bytes agree when the fused and the split calls take the same kernel
    plans = {rd.lora_proj_plan(wl.M, r.route.rt, path=path)["path"] for r in [run] + runs}
    if path == rd.LORA_PATH_AUTO:
        assert plans == {rd.LORA_PLAN_TC}
    if len(plans) == 1:
        assert np.array_equal(fused, np.concatenate(parts, axis=1))
    else:  # the one-launch path: 8192 outputs need more CTAs than SMs, 4096 fit
        assert plans == {rd.LORA_PLAN_TC, rd.LORA_PLAN_ONE_LAUNCH}, plans
        assert_all_rows(np.concatenate(parts, axis=1), oracle.workload_proj(wl), "gated q split calls")


def test_one_launch_path_with_the_default_workspace_is_the_tensor_core_path(qkv):
    """LORA_PATH_TC_ONE given only the default path's workspace runs the
    tensor-core path instead: the same bytes as LORA_PATH_TC."""
    need = rd.lora_proj_workspace_bytes(qkv.wl.M, qkv.route.rt)
    assert need < rd.lora_proj_workspace_bytes(qkv.wl.M, qkv.route.rt, rd.LORA_PATH_TC_ONE)
    y_tc = qkv.apply(path=rd.LORA_PATH_TC)
    y_one = qkv.apply(path=rd.LORA_PATH_TC_ONE, ws_bytes=need)
    assert qkv.last_status == 0
    assert np.array_equal(y_one, y_tc)


@pytest.fixture(scope="module")
def prefill():
    run = ProjRun(workloads.make("prefill"))
    return run, oracle.workload_proj(run.wl)


def test_prefill_matches_oracle_on_every_row(prefill):
    run, ref = prefill
    y = run.apply()
    assert run.last_status == 0
    assert_all_rows(y, ref, "prefill")
    wl = run.wl
    perm, seg = rd.lora_proj_routing(run.ws, wl.M, wl.max_loras)
    operm, oseg = oracle.slot_sort(wl.seq_slot, wl.max_loras)
    assert np.array_equal(perm, operm) and np.array_equal(seg, oseg)


def test_prefill_sequences_without_adapter_are_base_bytes(prefill):
    """Two of the eight sequences switched to slot -1: their rows are the
    base-only call's bytes, the other sequences still match the oracle."""
    run, ref = prefill
    wl = run.wl
    slots = wl.seq_slot.copy()
    off = (slots == 2) | (slots == 5)
    slots[off] = -1
    y = run.apply(slots=torch.from_numpy(slots.astype(np.int32)).cuda())
    base = run.apply(slots=torch.full_like(run.slots, -1))
    assert np.array_equal(y[off], base[off])
    keep = ~off
    assert_close(y[keep], ref[keep], f"prefill with two sequences off ({int(keep.sum())} adapted rows)")


class MoeRun:
    def __init__(self, wl, device="cuda"):
        self.wl = wl
        self.x = th.to_device_bf16(wl.x, device)
        self.W = [th.to_device_bf16(w, device) for w in wl.W]
        self.off = torch.from_numpy(wl.expert_offsets.astype(np.int32)).to(device)
        self.slots = torch.from_numpy(wl.seq_slot.astype(np.int32)).to(device)
        self.routes = []
        for e in range(wl.E):
            r = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N, device)
            r.pack_all(wl.adapters[e])
            self.routes.append(r)
        self.rts = [r.rt for r in self.routes]
        self.ws = th.workspace(rd.lora_moe_workspace_bytes(wl.E, wl.T, self.rts), device)

    def apply(self, slots=None, off=None):
        wl = self.wl
        y = torch.empty((wl.T, wl.N), dtype=torch.int16, device="cuda")
        y.fill_(SENTINEL)
        y = y.view(torch.bfloat16)
        rd.lora_moe_down_apply(self.x, self.x.stride(0), self.W, self.off if off is None else off,
                               wl.E, wl.T, wl.K, wl.N, self.slots if slots is None else slots,
                               self.rts, y, y.stride(0), self.ws, self.ws.numel())
        torch.cuda.synchronize()
        self.last_status = rd.lora_status_get(self.ws)
        return th.to_numpy_bf16(y)


def test_moe_matches_oracle_on_every_slot_row():
    run = MoeRun(workloads.make("moe"))
    y = run.apply()
    assert run.last_status == 0
    wl = run.wl
    assert_all_rows(y, oracle.workload_moe(wl), "moe")
    base = run.apply(slots=torch.full_like(run.slots, -1))
    none = wl.seq_slot < 0
    assert np.array_equal(y[none], base[none])


def test_small_moe_matches_oracle_everywhere():
    wl = workloads.synth.moe(seed=9, tokens=96, E=5, top_k=2, K=256, N=192, n_adapters=3, rank=8)
    run = MoeRun(wl)
    y = run.apply()
    assert run.last_status == 0
    assert_close(y, oracle.workload_moe(wl), "small moe")


@pytest.mark.parametrize("n_adapters,rank", [(4, 16), (8, 32)])
def test_paired_moe_tiles_match_oracle_everywhere(n_adapters, rank):
    """Per-expert tiles of 128 rows or more run as feature-tile pairs (two W
    boxes per x box, one K loop into both accumulators). With 64 feature
    tiles most CTAs take two pairs, and the second waits for both
    accumulators of the first; with 8 adapters of rank 32 a tile's expand
    takes several rounds, so the pair's second tile stages its own s * h
    instead of reusing the first one's."""
    wl = workloads.synth.moe(seed=20 + rank, tokens=512, E=8, top_k=2, K=1024, N=8192,
                             n_adapters=n_adapters, rank=rank)
    run = MoeRun(wl)
    y = run.apply()
    assert run.last_status == 0
    assert_close(y, oracle.workload_moe(wl), f"paired moe, {n_adapters} adapters of rank {rank}")
    base = run.apply(slots=torch.full_like(run.slots, -1))
    none = wl.seq_slot < 0
    assert np.array_equal(y[none], base[none])


def test_moe_bad_offsets_are_flagged():
    wl = workloads.synth.moe(seed=10, tokens=32, E=3, top_k=2, K=64, N=64, n_adapters=2, rank=8)
    run = MoeRun(wl)
    bad = torch.tensor([0, 40, 20, 64], dtype=torch.int32, device="cuda")
    run.apply(off=bad)
    assert run.last_status & rd.LORA_FLAG_BAD_OFFSETS
