"""lora_proj_apply_static_ws: the entry point for callers that cannot allocate
device memory (a plugin whose host framework owns all device memory and gives
it no allocator, or a service that must not grow device memory once it is
running). It takes no workspace and uses the scratch array built into the
library instead.

Checked here through the C ABI: two calls in a row, with different routing,
each give the bytes lora_proj_apply gives on the same inputs (the same
kernels with the same order of sums, so any difference would be a scratch
region read wrongly or reused too early); a decode call followed by a
2048-row prefill-shaped call (the tensor-core shrink layout of the scratch)
gives the bytes of the workspace entry too; and a batch whose scratch need
exceeds the built-in size is refused with a message naming both sizes. This file is collected last on
purpose; it builds everything it uses, so it also passes on its own.
"""
import numpy as np
import pytest
import torch

import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from rank_delta_gb300 import torch_helpers as th
from tests.gpu_common import SENTINEL, ProjRun

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available()
    return rd.lib()


def static_apply(run, slots):
    wl = run.wl
    y = torch.empty((wl.M, wl.N), dtype=torch.int16, device="cuda")
    y.fill_(SENTINEL)
    y = y.view(torch.bfloat16)
    rd.lora_proj_apply_static_ws(run.x, run.x.stride(0), run.W, wl.M, wl.K, wl.N, slots,
                                 run.route.rt, y, y.stride(0))
    torch.cuda.synchronize()
    return th.to_numpy_bf16(y)


@pytest.mark.parametrize("name", ["decode", "tiny"])
def test_static_scratch_matches_workspace_entry_on_two_calls(name):
    run = ProjRun(workloads.make(name))
    rng = np.random.default_rng(11)
    other = rng.integers(-1, run.wl.max_loras, size=run.wl.M).astype(np.int32)
    for slots in (run.slots, torch.from_numpy(other).cuda()):
        want = run.apply(slots=slots)
        got = static_apply(run, slots)
        assert np.array_equal(got, want), f"{name}: static scratch differs from the workspace entry"


def test_static_scratch_decode_then_prefill_shaped_batch():
    dec = ProjRun(workloads.make("decode"))
    pre = ProjRun(workloads.make("prefill", seq_len=256))  # 2048 rows, 8 sequences
    assert pre.wl.M == 2048
    need = rd.lora_proj_workspace_bytes(pre.wl.M, pre.route.rt)
    assert need <= rd.LORA_STATIC_WS_BYTES
    for run in (dec, pre):
        got = static_apply(run, run.slots)
        want = run.apply()
        assert np.array_equal(got, want), f"{run.wl.name}: static scratch differs from the workspace entry"


def test_static_scratch_refuses_batches_beyond_its_size():
    run = ProjRun(workloads.make("tiny"))
    M = 1 << 20  # h alone needs M * max_rank * 4 bytes, far past the built-in size
    need = rd.lora_proj_workspace_bytes(M, run.route.rt)
    assert need > rd.LORA_STATIC_WS_BYTES
    with pytest.raises(rd.LoraError) as ei:
        rd.lora_proj_apply_static_ws(run.x, run.x.stride(0), run.W, M, run.wl.K, run.wl.N,
                                     run.slots, run.route.rt, run.x, run.wl.N)
    assert ei.value.code == rd.LORA_ERR_UNSUPPORTED
    assert str(need) in ei.value.message and str(rd.LORA_STATIC_WS_BYTES) in ei.value.message
