"""Gated MLP input through a fused [gate|up] projection: CUDA path vs the
oracle, through the C ABI (GPU only).

act = silu(g) * u with g, u the two halves of the fused projection. The
projection's tolerance, tol(v) = 2e-2 + 1e-2 |v|, carried through silu(g) * u
to first order plus the same bound on act itself:

    |gpu - oracle| <= tol(act) + |silu'(g) u| tol(g) + |silu(g)| tol(u) + tol(g) tol(u)

(g, u, act the oracle's fp32 values; |silu'| <= 1.1). Rows with no delta
equal the GPU's own all-(-1) run byte for byte.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from rank_delta_gb300 import torch_helpers as th
from tests.gpu_common import ATOL, RTOL, SENTINEL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return rd.lib()


class GateUpRun:
    def __init__(self, wl):
        self.wl = wl
        self.I = wl.N // 2
        self.x = th.to_device_bf16(wl.x)
        self.W = th.to_device_bf16(wl.W)
        self.slots = torch.from_numpy(np.ascontiguousarray(wl.seq_slot, np.int32)).cuda()
        self.route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.K, wl.N)
        self.route.pack_all(wl.adapters)
        self.ws = th.workspace(rd.lora_gate_up_workspace_bytes(wl.M, self.route.rt, rd.LORA_PATH_TC_ONE))

    def apply(self, slots=None, act_stride=None, path=rd.LORA_PATH_AUTO):
        wl, I = self.wl, self.I
        st = I if act_stride is None else act_stride
        act = torch.full((wl.M, st), SENTINEL, dtype=torch.int16, device="cuda")
        rd.lora_gate_up_apply(self.x, self.x.stride(0), self.W, wl.M, wl.K, I,
                              self.slots if slots is None else slots, self.route.rt, act, st, self.ws,
                              self.ws.numel(), path=path)
        torch.cuda.synchronize()
        self.last_status = rd.lora_status_get(self.ws)
        return th.to_numpy_bf16(act.view(torch.bfloat16)[:, :I])


def assert_close_act(gpu_bits, y, I, what):
    """y: the oracle's fp32 projection [rows][2I]."""
    g = y[:, :I].astype(np.float64)
    u = y[:, I:2 * I].astype(np.float64)
    sig = 1.0 / (1.0 + np.exp(-np.clip(g, -80, 80)))
    act = g * sig * u
    dsilu = sig * (1.0 + g * (1.0 - sig))
    tg, tu = ATOL + RTOL * np.abs(g), ATOL + RTOL * np.abs(u)
    tol = ATOL + RTOL * np.abs(act) + np.abs(dsilu * u) * tg + np.abs(g * sig) * tu + 1.1 * tg * tu
    a = th.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    assert a.shape == act.shape
    assert np.all(np.isfinite(a)), f"{what}: non-finite GPU outputs (unwritten?)"
    bad = np.abs(a - act) > tol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first at {i}: "
                             f"gpu {a[i]} oracle {act[i]} tol {tol[i]}")
    # the oracle's own act agrees with the fp64 form above
    assert np.allclose(oracle.silu_mul(y.astype(np.float32), I), act, rtol=1e-5, atol=1e-6)


def _no_delta_rows(wl):
    sc = [0.0 if a is None else oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale)
          for a in wl.adapters]
    return [i for i in range(wl.M) if not (0 <= wl.seq_slot[i] < wl.max_loras) or sc[wl.seq_slot[i]] == 0.0]


@pytest.mark.parametrize("M,K,I,L,R", [
    (9, 64, 24, 3, 16),     # CUDA-core path, I a multiple of 8
    (37, 128, 100, 4, 8),   # tensor-core path, I not a multiple of 8 (scalar activation)
    (300, 256, 136, 5, 32), # several token tiles
    (48, 128, 64, 4, 16),   # K and I multiples of 64: the one-launch kernel's fused act
    (300, 256, 128, 5, 32), # several token tiles, K and I multiples of 64: act from the tensor-core drain
    (700, 192, 64, 6, 16),  # three token tiles, a partial last one
])
@pytest.mark.parametrize("path", [rd.LORA_PATH_AUTO, rd.LORA_PATH_TC_ONE])
def test_gate_up_matches_oracle(M, K, I, L, R, path):
    wl = workloads.random_small(40 + M, M=M, K=K, N=2 * I, L=L, R=R)
    run = GateUpRun(wl)
    act = run.apply(path=path)
    assert run.last_status == 0
    assert_close_act(act, oracle.proj(wl.x, wl.W, wl.seq_slot, wl.adapters), I, f"gate_up {M}x{K}x{I}")


@pytest.mark.parametrize("path", [rd.LORA_PATH_AUTO, rd.LORA_PATH_TC_ONE])
def test_gate_up_decode_shapes_and_no_delta_rows(path):
    wl = workloads.make("decode")  # W [4096][4096] read as gate 2048 | up 2048
    run = GateUpRun(wl)
    act = run.apply(path=path)
    assert run.last_status == 0
    assert_close_act(act, oracle.proj(wl.x, wl.W, wl.seq_slot, wl.adapters), run.I, "gate_up decode")
    base = run.apply(slots=torch.full_like(run.slots, -1), path=path)
    rows = _no_delta_rows(wl)
    assert rows
    assert np.array_equal(act[rows], base[rows])


def test_gate_up_decode_shapes_strided_act_from_the_split_k_sum():
    """64 rows on K 4096: four K parts whose sum forms act, written into rows
    of a wider act buffer; the columns past I keep their sentinel."""
    wl = workloads.make("decode")
    run = GateUpRun(wl)
    st = run.I + 24
    wide = torch.full((wl.M, st), SENTINEL, dtype=torch.int16, device="cuda")
    rd.lora_gate_up_apply(run.x, run.x.stride(0), run.W, wl.M, wl.K, run.I, run.slots, run.route.rt, wide, st,
                          run.ws, run.ws.numel())
    torch.cuda.synchronize()
    assert rd.lora_status_get(run.ws) == 0
    bits = wide.cpu().numpy().view(np.uint16)
    assert (bits[:, run.I:] == np.uint16(SENTINEL & 0xFFFF)).all()
    assert_close_act(bits[:, :run.I], oracle.proj(wl.x, wl.W, wl.seq_slot, wl.adapters), run.I,
                     "gate_up decode, act stride I + 24")


def test_gate_up_prefill_shapes_every_token_tile():
    """act from the tensor-core drain (W read as 64 gate + 64 up rows per
    tile): one row of every 256-row token tile at a different offset in each,
    and every row of one whole tile."""
    wl = workloads.make("prefill")  # W [14336][4096]: gate 7168 | up 7168, 8192 rows
    run = GateUpRun(wl)
    act = run.apply()
    assert run.last_status == 0
    tiles = wl.M // 256
    one = [t * 256 + (37 * t + 11) % 256 for t in range(tiles)]
    whole = list(range(5 * 256, 6 * 256))
    rows = np.array(sorted(set(one) | set(whole)), dtype=np.int32)
    ref = oracle.proj(wl.x, wl.W, wl.seq_slot, wl.adapters, rows=rows)
    assert_close_act(act[rows], ref, run.I,
                     f"gate_up prefill ({len(rows)} rows: one per token tile and all of tile 5)")


@pytest.mark.parametrize("path", [rd.LORA_PATH_AUTO, rd.LORA_PATH_TC_ONE])
def test_gate_up_strided_output(path):
    wl = workloads.random_small(77, M=20, K=64, N=2 * 40, L=2, R=8)
    run = GateUpRun(wl)
    a = run.apply(act_stride=48, path=path)
    assert run.last_status == 0
    assert_close_act(a, oracle.proj(wl.x, wl.W, wl.seq_slot, wl.adapters), 40, "gate_up strided")
