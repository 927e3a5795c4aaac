"""Embedding row gather with the adapted rows: CUDA path vs the oracle,
through the C ABI (GPU only).

Rows with no delta (slot -1, slot >= max_loras, scale 0, empty slot) must be
the E row byte for byte; a token outside the vocabulary gives a zero row;
adapted rows are within |gpu - oracle| <= 2e-2 + 1e-2 |oracle|.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from rank_delta_gb300 import torch_helpers as th
from tests.gpu_common import EmbedRun, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return rd.lib()


def _check(run, y, tokens=None, slots=None, scales=None):
    wl = run.wl
    tok = wl.tokens if tokens is None else tokens
    ss = wl.seq_slot if slots is None else slots
    ref = oracle.embed(tok, wl.E, ss, wl.adapters, scales=scales)
    assert_close(y, ref, wl.name)
    # no-delta rows: the E row's bytes exactly
    sc = scales if scales is not None else [
        oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale) if a is not None else 0.0
        for a in wl.adapters]
    for i in range(len(tok)):
        t, s = int(tok[i]), int(ss[i])
        if not (0 <= t < wl.vocab):
            assert not y[i].any(), i
        elif s < 0 or s >= wl.max_loras or sc[s] == 0.0:
            assert np.array_equal(y[i], wl.E[t]), i
    return ref


@pytest.fixture(scope="module")
def embed_run():
    return EmbedRun(workloads.embed())


def test_embed_decode_batch_matches_oracle(embed_run):
    y = embed_run.apply()
    assert embed_run.last_status == 0
    _check(embed_run, y)


@pytest.mark.parametrize("M,vocab,n_embd,L,R,ranks", [
    (37, 1000, 200, 5, 24, [8, 24, 16, 1, 3]),   # ragged feature tile, rank not a multiple of 16
    (3000, 5000, 384, 4, 64, [64, 8, 32, 16]),   # several chunks per slot
    (300, 2000, 136, 3, 256, [256, 100, 17]),    # four k blocks, ragged ranks
    (1, 64, 8, 1, 8, [8]),                       # one row, one narrow tile
    (5000, 3000, 256, 6, 16, [16, 8, 16, 4, 12, 16]),  # past the in-kernel sort: routing kernel
    (300, 2000, 256, 100, 64, None),             # more slots than the in-kernel sort takes
])
def test_embed_ragged_shapes_match_oracle(M, vocab, n_embd, L, R, ranks):
    wl = workloads.embed(seed=M + n_embd, M=M, vocab=vocab, n_embd=n_embd, L=L, R=R, ranks=ranks)
    run = EmbedRun(wl)
    y = run.apply()
    assert run.last_status == 0
    _check(run, y)


def test_embed_full_size_prefill_samples_match_oracle():
    wl = workloads.embed(seed=9, M=4096)
    run = EmbedRun(wl)
    y = run.apply()
    assert run.last_status == 0
    rows = np.concatenate([np.arange(0, 4096, 97), np.where(wl.seq_slot < 0)[0][:8]])
    ref = oracle.embed(wl.tokens[rows], wl.E, wl.seq_slot[rows], wl.adapters)
    assert_close(y[rows], ref, "embed 4096 rows (sampled)")


def test_embed_flipped_pack_equals_module_layout_pack():
    wl = workloads.embed(seed=11, M=90, vocab=3000, n_embd=512, L=6, R=32, ranks=[32, 8, 16, 24, 32, 1])
    a = EmbedRun(wl)
    b = EmbedRun(wl, flipped=True)
    assert torch.equal(a.route.pool, b.route.pool)
    assert np.array_equal(a.apply(), b.apply())


def test_embed_device_pack_transposes_like_host_pack():
    wl = workloads.embed(seed=12, M=16, vocab=700, n_embd=264, L=2, R=40, ranks=[40, 13])
    host = EmbedRun(wl)
    route = th.DeviceRoute(wl.max_loras, wl.max_rank, wl.n_embd, wl.vocab, embed=True)
    for s, ad in enumerate(wl.adapters):
        rd.lora_pool_pack(route.rt, s, th.to_device_bf16(ad.A), th.to_device_bf16(ad.B), ad.rank,
                          ad.alpha, ad.use_rslora, ad.adapter_scale)
    torch.cuda.synchronize()
    assert torch.equal(host.route.pool, route.pool)


@pytest.mark.parametrize("M", [50, 4500])  # in-kernel sort / routing kernel
def test_embed_out_of_range_tokens_and_slots(M):
    wl = workloads.embed(seed=13, M=M, vocab=900, n_embd=256, L=4, R=16, ranks=[16, 8, 16, 4])
    run = EmbedRun(wl)
    tok = wl.tokens.copy()
    tok[[3, 17]] = [wl.vocab, -5]
    ss = wl.seq_slot.copy()
    ss[[5, 6]] = [wl.max_loras, wl.max_loras + 100]
    y = run.apply(tokens=torch.from_numpy(tok).cuda(), slots=torch.from_numpy(ss).cuda())
    assert run.last_status == rd.LORA_FLAG_TOKEN_RANGE | rd.LORA_FLAG_SLOT_RANGE
    _check(run, y, tokens=tok, slots=ss)


def test_embed_scale_zero_gives_the_embedding_rows():
    wl = workloads.embed(seed=14, M=64, vocab=1200, n_embd=640, L=3, R=16, ranks=[16, 16, 8])
    run = EmbedRun(wl)
    rd.lora_set_scale(run.route.rt, 1, 0.0)
    sc = [oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale) for a in wl.adapters]
    sc[1] = 0.0
    y = run.apply()
    _check(run, y, scales=sc)
    rd.lora_pool_unpack(run.route.rt, 2)
    sc[2] = 0.0
    _check(run, run.apply(), scales=sc)


def test_embed_batch_equals_single_rows(embed_run):
    y = embed_run.apply()
    for i in [0, 5, 31, 63]:
        one = embed_run.apply(tokens=embed_run.tokens[i:i + 1], slots=embed_run.slots[i:i + 1])
        assert np.array_equal(one[0], y[i]), i


def test_embed_strided_output_and_empty_batch(embed_run):
    wl = embed_run.wl
    y = embed_run.apply(y_stride=wl.n_embd + 64)
    _check(embed_run, y)
    empty = torch.empty(0, dtype=torch.int32, device="cuda")
    rd.lora_embed_apply(empty, embed_run.E, 0, wl.vocab, wl.n_embd, empty, embed_run.route.rt,
                        0, wl.n_embd, embed_run.ws, embed_run.ws.numel())


def test_embed_route_is_refused_by_the_projection_and_back(embed_run):
    wl = embed_run.wl
    with pytest.raises(rd.LoraError) as e:
        rd.lora_proj_apply(embed_run.E, wl.n_embd, embed_run.E, 1, wl.n_embd, wl.vocab,
                           embed_run.slots, embed_run.route.rt, embed_run.E, wl.vocab,
                           embed_run.ws, embed_run.ws.numel())
    assert e.value.code == rd.LORA_ERR_UNSUPPORTED
    proj = th.DeviceRoute(2, 8, wl.n_embd, wl.vocab)
    with pytest.raises(rd.LoraError) as e:
        rd.lora_embed_apply(embed_run.tokens, embed_run.E, 4, wl.vocab, wl.n_embd, embed_run.slots,
                            proj.rt, embed_run.E, wl.n_embd, embed_run.ws, embed_run.ws.numel())
    assert e.value.code == rd.LORA_ERR_UNSUPPORTED
