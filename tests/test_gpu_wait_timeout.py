"""A bounded device wait that runs out (GPU only; nothing faults or hangs).

The one-launch kernel of up to 256 rows hands the partial h of every CTA to
the others through flags in the workspace, and each CTA that adds a delta
waits, with a time limit, for all of them. Through the test hook the limit is
cut to 200 us and the wait made to include a flag no CTA ever writes, so it
runs out: the call must return, report LORA_FLAG_WAIT_TIMEOUT, and give the
base product (the delta skipped) -- and the next normal call on the same
workspace must be correct and clean (spark_model `lora_delta.rs`,
`LoraKernels`: the kernels bail out loudly instead of running on with
half-built state).
"""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from tests.gpu_common import ProjRun, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available()
    return rd.lib()


@pytest.mark.parametrize("name", ["decode", "qkv"])
def test_exchange_wait_runs_out_then_the_next_call_is_correct(name):
    run = ProjRun(workloads.make(name))
    one = rd.LORA_PATH_TC_ONE
    base = run.apply(slots=torch.full_like(run.slots, -1), path=one)
    assert run.last_status == 0
    rd.lora_test_wait_hook(200_000, 1)
    try:
        y = run.apply(path=one)
        flags = run.last_status
    finally:
        rd.lora_test_wait_hook(0, 0)
    assert flags & rd.LORA_FLAG_WAIT_TIMEOUT, f"{name}: status {flags:#x}"
    assert np.array_equal(y, base), f"{name}: a timed-out call must leave the base product"
    y2 = run.apply(path=one)
    assert run.last_status == 0, f"{name}: the next call reports {run.last_status:#x}"
    assert_close(y2, oracle.workload_proj(run.wl), f"{name} after a timed-out call")


def test_split_k_wait_runs_out_then_the_next_call_is_correct():
    """The tensor-core path's split-K sum waits (bounded) for every K part of
    its tile; with the hook the wait also counts a part that never comes, so
    it runs out: the call returns with LORA_FLAG_WAIT_TIMEOUT, and the next
    normal call on the same workspace is correct and clean."""
    run = ProjRun(workloads.make("decode"))  # 64 rows: four K parts per tile
    tc = rd.LORA_PATH_TC
    run.apply(path=tc)
    assert run.last_status == 0
    rd.lora_test_wait_hook(200_000, 1)
    try:
        run.apply(path=tc)
        flags = run.last_status
    finally:
        rd.lora_test_wait_hook(0, 0)
    assert flags & rd.LORA_FLAG_WAIT_TIMEOUT, f"status {flags:#x}"
    y = run.apply(path=tc)
    assert run.last_status == 0, f"the next call reports {run.last_status:#x}"
    assert_close(y, oracle.workload_proj(run.wl), "decode after a timed-out split-K wait")


def test_shrink_tile_wait_runs_out_then_the_next_call_is_correct():
    """From 2048 rows the projection launch computes h in tensor-core shrink
    tiles of 128 rows and the epilogue waits (bounded) for the tiles of its
    rows before staging s * h; with the hook that wait also counts a
    publication that never comes, so it runs out: the call returns with
    LORA_FLAG_WAIT_TIMEOUT, and the next normal call on the same workspace is
    correct and clean."""
    wl = workloads.random_small(seed=2150, M=2100, K=200, N=136, L=5, R=24)
    run = ProjRun(wl)
    tc = rd.LORA_PATH_TC
    run.apply(path=tc)
    assert run.last_status == 0
    rd.lora_test_wait_hook(200_000, 1)
    try:
        run.apply(path=tc)
        flags = run.last_status
    finally:
        rd.lora_test_wait_hook(0, 0)
    assert flags & rd.LORA_FLAG_WAIT_TIMEOUT, f"status {flags:#x}"
    y = run.apply(path=tc)
    assert run.last_status == 0, f"the next call reports {run.last_status:#x}"
    assert_close(y, oracle.workload_proj(wl), "2100 rows after a timed-out shrink-tile wait")
