"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, sizes follow the pool layout, and host argument errors are refused
with messages naming the dimensions -- before any CUDA call is made."""
import ctypes
import os
import re

import numpy as np
import pytest

import rank_delta_gb300 as rd
from rank_delta_gb300 import build as rdbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rank_delta.h")
MAGIC = 0x6C6F72615F727431  # the value lora_route_init stamps into a route


@pytest.fixture(scope="module", autouse=True)
def built():
    rdbuild.build()
    return rd.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(lora_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 15, names
    lib = ctypes.CDLL(rd.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(rd.exported_symbols()) == names


def test_pool_bytes_layout():
    # slot = A [R][K] then B [N][R], bf16
    assert rd.lora_pool_bytes(16, 64, 4096, 4096) == 16 * (64 * 4096 + 4096 * 64) * 2
    assert rd.lora_pool_bytes(32, 16, 4096, 6144) == 32 * (16 * 4096 + 6144 * 16) * 2
    assert rd.lora_pool_bytes(0, 64, 4096, 4096) == 0
    assert rd.lora_route_table_bytes(16) >= 16 * (8 + 8 + 4 + 4 + 4)
    assert rd.lora_route_table_bytes(0) == 0


def fake_route(L=4, R=8, K=256, N=256, kind=rd.LORA_ROUTE_PROJ):
    rt = rd.lora_route()
    rt.pool = rt.a_table = rt.b_table = rt.scale_table = rt.factor_table = rt.rank_table = 256
    rt.n_in, rt.n_out, rt.max_rank, rt.max_loras, rt.magic = K, N, R, L, MAGIC
    rt.kind = kind
    return rt


def expect(code, fn, *args, contains=()):
    with pytest.raises(rd.LoraError) as ei:
        fn(*args)
    assert ei.value.code == code, ei.value
    for c in contains:
        assert c in ei.value.message, ei.value.message
    return ei.value.message


def test_route_init_refusals():
    rt = rd.lora_route()
    expect(rd.LORA_ERR_NULL, rd.lora_route_init, rt, 0, 0, 0, 0, 4, 8, 256, 256)
    expect(rd.LORA_ERR_SHAPE, rd.lora_route_init, rt, 256, 1 << 20, 256, 4096, 0, 8, 256, 256)
    expect(rd.LORA_ERR_UNSUPPORTED, rd.lora_route_init, rt, 256, 1 << 30, 256, 1 << 20, 4, 12, 256, 256,
           contains=("max_rank 12",))
    expect(rd.LORA_ERR_ALIGN, rd.lora_route_init, rt, 256, 1 << 30, 256, 1 << 20, 4, 8, 250, 256)
    msg = expect(rd.LORA_ERR_WORKSPACE, rd.lora_route_init, rt, 256, 100, 256, 1 << 20, 4, 8, 256, 256)
    assert "4 slots" in msg and "[256 x 256]" in msg


def test_uninitialised_route_is_refused():
    rt = rd.lora_route()
    expect(rd.LORA_ERR_NOT_INIT, rd.lora_set_scale, rt, 0, 1.0)
    expect(rd.LORA_ERR_NOT_INIT, rd.lora_pool_unpack, rt, 0)


def test_pack_refuses_bad_rank_naming_every_dimension():
    rt = fake_route(L=4, R=8, K=256, N=128)
    A = np.zeros((16, 256), np.uint16)
    B = np.zeros((128, 16), np.uint16)
    msg = expect(rd.LORA_ERR_SHAPE, rd.lora_pool_pack, rt, 0, A, B, 16, 1.0, False, 1.0)
    for part in ("rank 16", "n_out 128", "n_in 256", "max_rank 8", "4096", "2048"):
        assert part in msg, (part, msg)
    expect(rd.LORA_ERR_SHAPE, rd.lora_pool_pack, rt, 0, A, B, 0, 1.0, False, 1.0)


def test_slot_out_of_range_names_the_range():
    rt = fake_route(L=4)
    A = np.zeros((8, 256), np.uint16)
    B = np.zeros((256, 8), np.uint16)
    expect(rd.LORA_ERR_RANGE, rd.lora_pool_pack, rt, 4, A, B, 8, 1.0, False, 1.0,
           contains=("slot 4", "4 slot"))
    expect(rd.LORA_ERR_RANGE, rd.lora_set_scale, rt, 7, 1.0, contains=("slot 7", "[0, 4)"))
    expect(rd.LORA_ERR_RANGE, rd.lora_set_scale, rt, -1, 1.0)
    expect(rd.LORA_ERR_RANGE, rd.lora_pool_unpack, rt, 9)


def test_apply_argument_checks():
    rt = fake_route(L=4, R=8, K=256, N=256)
    ws_need = rd.lora_proj_workspace_bytes(8, rt)
    assert ws_need > 0
    good = dict(x=4096, x_stride=256, W=8192, M=8, K=256, N=256, seq_slot=4096, rt=rt, y=4096,
                y_stride=256, ws=1 << 20, ws_bytes=ws_need)

    def call(**kw):
        a = dict(good, **kw)
        return lambda: rd.lora_proj_apply(a["x"], a["x_stride"], a["W"], a["M"], a["K"], a["N"], a["seq_slot"],
                           a["rt"], a["y"], a["y_stride"], a["ws"], a["ws_bytes"])

    expect(rd.LORA_ERR_SHAPE, call(K=512), contains=("K 512", "n_in 256"))
    expect(rd.LORA_ERR_NULL, call(x=0))
    expect(rd.LORA_ERR_NULL, call(W=0))
    expect(rd.LORA_ERR_ALIGN, call(x=4098))
    expect(rd.LORA_ERR_ALIGN, call(x_stride=260))
    expect(rd.LORA_ERR_SHAPE, call(y_stride=100))
    expect(rd.LORA_ERR_WORKSPACE, call(ws_bytes=ws_need - 1))
    expect(rd.LORA_ERR_ALIGN, call(ws=(1 << 20) + 16))
    expect(rd.LORA_ERR_RANGE, lambda: rd.lora_proj_apply(4096, 256, 8192, 8, 256, 256, 4096, rt,
                                                         4096, 256, 1 << 20, ws_need, path=9))
    # M = 0 is a no-op that launches nothing
    rd.lora_proj_apply(0, 256, 0, 0, 256, 256, 0, rt, 0, 256, 0, 0)


def test_moe_argument_checks():
    rts = [fake_route(L=4, R=16, K=512, N=256) for _ in range(3)]
    need = rd.lora_moe_workspace_bytes(3, 100, rts)
    assert need > 0
    expect(rd.LORA_ERR_UNSUPPORTED, rd.lora_moe_down_apply, 4096, 512, [8192] * 17, 4096, 17, 100,
           512, 256, 4096, [fake_route(L=4, R=16, K=512, N=256)] * 17, 4096, 256, 1 << 20, need)
    bad = [fake_route(L=4, R=16, K=512, N=256), fake_route(L=4, R=8, K=512, N=256),
           fake_route(L=4, R=16, K=512, N=256)]
    expect(rd.LORA_ERR_SHAPE, rd.lora_moe_down_apply, 4096, 512, [8192] * 3, 4096, 3, 100, 512, 256,
           4096, bad, 4096, 256, 1 << 20, need, contains=("expert 1",))
    expect(rd.LORA_ERR_NULL, rd.lora_moe_down_apply, 4096, 512, [8192, 0, 8192], 4096, 3, 100, 512,
           256, 4096, rts, 4096, 256, 1 << 20, need, contains=("W_e[1]",))


def test_build_seq_slot_host_helper():
    # metrale lora/slot_math.rs build_seq_slot_host: negative -> active; padding -> -1
    out = rd.lora_build_seq_slot([3, -1, 0, -5], 6, 2)
    assert out.tolist() == [3, 2, 0, 2, -1, -1]
    assert rd.lora_build_seq_slot([], 3, 1).tolist() == [-1, -1, -1]
    expect(rd.LORA_ERR_SHAPE, rd.lora_build_seq_slot, [1, 2, 3], 2, 0)


def test_set_scales_refuses_an_unknown_id_naming_the_range():
    rt = fake_route(L=4)
    expect(rd.LORA_ERR_RANGE, rd.lora_set_scales, rt, [(1, 0.5), (9, 1.0)],
           contains=("id 9", "4 slot"))
    expect(rd.LORA_ERR_RANGE, rd.lora_set_scales, rt, [(-1, 0.5)], contains=("id -1",))


def _victim_by_the_rules(cache):
    """The promotion rule restated: first unfilled slot in order; else the
    ref_count == 0 slot with the smallest last_used (first on a tie); else full."""
    for slot, filled, _, _ in cache:
        if not filled:
            return slot
    free = [(last, i) for i, (_, _, refs, last) in enumerate(cache) if refs == 0]
    if not free:
        return None
    return cache[min(free)[1]][0]


def test_select_victim_slot_follows_the_promotion_rules():
    assert rd.lora_select_victim_slot([(3, True, 0, 5), (7, False, 0, 0), (9, False, 2, 0)]) == 7
    assert rd.lora_select_victim_slot([(3, True, 1, 1), (5, True, 0, 10), (6, True, 0, 4),
                                       (8, True, 0, 4)]) == 6
    expect(rd.LORA_ERR_POOL_FULL, rd.lora_select_victim_slot, [(1, True, 1, 0), (2, True, 3, 0)])
    expect(rd.LORA_ERR_POOL_FULL, rd.lora_select_victim_slot, [])
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(1, 9))
        cache = [(int(s), bool(rng.random() < 0.8), int(rng.integers(0, 2)), int(rng.integers(0, 6)))
                 for s in rng.permutation(16)[:n]]
        want = _victim_by_the_rules(cache)
        if want is None:
            expect(rd.LORA_ERR_POOL_FULL, rd.lora_select_victim_slot, cache)
        else:
            assert rd.lora_select_victim_slot(cache) == want, cache


def test_embed_argument_checks():
    # an embedding route: the adapted matrix is [vocab 1000][n_embd 256]
    rt = fake_route(L=4, R=16, K=256, N=1000, kind=rd.LORA_ROUTE_EMBED)
    need = rd.lora_embed_workspace_bytes(8, rt)
    assert need > 0
    assert rd.lora_embed_workspace_bytes(8, fake_route()) == 0  # a projection route

    def call(**kw):
        a = dict(dict(tokens=4096, E=8192, M=8, vocab=1000, n_embd=256, seq_slot=4096, rt=rt,
                      y=4096, y_stride=256, ws=1 << 20, ws_bytes=need), **kw)
        return lambda: rd.lora_embed_apply(a["tokens"], a["E"], a["M"], a["vocab"], a["n_embd"],
                                           a["seq_slot"], a["rt"], a["y"], a["y_stride"], a["ws"],
                                           a["ws_bytes"])

    expect(rd.LORA_ERR_SHAPE, call(vocab=999), contains=("vocab 999", "vocab 1000", "n_embd 256"))
    expect(rd.LORA_ERR_NULL, call(tokens=0))
    expect(rd.LORA_ERR_NULL, call(E=0))
    expect(rd.LORA_ERR_ALIGN, call(E=8200))
    expect(rd.LORA_ERR_ALIGN, call(y=4100))
    expect(rd.LORA_ERR_ALIGN, call(y_stride=260))
    expect(rd.LORA_ERR_ALIGN, call(y_stride=128))
    expect(rd.LORA_ERR_UNSUPPORTED, call(rt=fake_route(K=256, N=1000)), contains=("embedding",))
    # and the projection calls refuse an embedding route
    expect(rd.LORA_ERR_UNSUPPORTED, rd.lora_proj_apply, 4096, 256, 8192, 8, 256, 1000, 4096, rt,
           4096, 1000, 1 << 20, 1 << 20, contains=("token-embedding",))
    expect(rd.LORA_ERR_UNSUPPORTED, rd.lora_embed_pool_pack, fake_route(), 0,
           np.zeros((256, 8), np.uint16), np.zeros((256, 8), np.uint16), 8, 1.0, False, 1.0)
    expect(rd.LORA_ERR_RANGE, rd.lora_embed_pool_pack, rt, 4, np.zeros((1000, 8), np.uint16),
           np.zeros((256, 8), np.uint16), 8, 1.0, False, 1.0, contains=("slot 4",))
    expect(rd.LORA_ERR_SHAPE, rd.lora_embed_pool_pack, rt, 0, np.zeros((1000, 32), np.uint16),
           np.zeros((256, 32), np.uint16), 32, 1.0, False, 1.0, contains=("max_rank 16",))
    # M = 0 is a no-op that launches nothing
    rd.lora_embed_apply(0, 0, 0, 1000, 256, 0, rt, 0, 256, 0, 0)


def test_embed_route_init_refusals_name_the_call():
    rt = rd.lora_route()
    expect(rd.LORA_ERR_ALIGN, rd.lora_embed_route_init, rt, 256, 1 << 30, 256, 1 << 20, 4, 8, 1000,
           250, contains=("lora_embed_route_init", "250"))
    msg = expect(rd.LORA_ERR_WORKSPACE, rd.lora_embed_route_init, rt, 256, 100, 256, 1 << 20, 4, 8,
                 1000, 256)
    assert "[1000 x 256]" in msg


def test_gate_up_argument_checks():
    rt = fake_route(L=4, R=8, K=256, N=512)
    need = rd.lora_gate_up_workspace_bytes(8, rt)
    assert need >= rd.lora_proj_workspace_bytes(8, rt) + 8 * 512 * 2
    assert rd.lora_gate_up_workspace_bytes(8, fake_route(N=511)) == 0

    def call(**kw):
        a = dict(dict(x=4096, x_stride=256, W=8192, M=8, K=256, I=256, seq_slot=4096, rt=rt, act=4096,
                      act_stride=256, ws=1 << 20, ws_bytes=need), **kw)
        return lambda: rd.lora_gate_up_apply(a["x"], a["x_stride"], a["W"], a["M"], a["K"], a["I"],
                                             a["seq_slot"], a["rt"], a["act"], a["act_stride"], a["ws"],
                                             a["ws_bytes"])

    expect(rd.LORA_ERR_SHAPE, call(I=200), contains=("I 200", "n_out 512"))
    expect(rd.LORA_ERR_NULL, call(act=0))
    expect(rd.LORA_ERR_SHAPE, call(act_stride=100))
    expect(rd.LORA_ERR_WORKSPACE, call(ws_bytes=need - 1))
    expect(rd.LORA_ERR_UNSUPPORTED, call(rt=fake_route(K=256, N=512, kind=rd.LORA_ROUTE_EMBED)))
    rd.lora_gate_up_apply(0, 256, 0, 0, 256, 256, 0, rt, 0, 256, 0, 0)  # M = 0: nothing


def test_moe_gather_argument_checks():
    rts = [fake_route(L=4, R=16, K=512, N=256) for _ in range(3)]
    need = rd.lora_moe_gather_workspace_bytes(3, 100, rts)
    assert need >= rd.lora_moe_workspace_bytes(3, 100, rts) + 100 * (512 + 256) * 2
    args = dict(x=4096, x_stride=512, W=[8192] * 3, idx=4096, E=3, T=100, K=512, N=256, slots=4096, rts=rts,
                comb=4096, top_k=2, y=4096, y_stride=256, ws=1 << 20, wsb=need)

    def call(**kw):
        a = dict(args, **kw)
        return lambda: rd.lora_moe_gather_apply(a["x"], a["x_stride"], a["W"], a["idx"], a["E"], a["T"], a["K"],
                                                a["N"], a["slots"], a["rts"], a["comb"], a["top_k"], a["y"],
                                                a["y_stride"], a["ws"], a["wsb"])

    expect(rd.LORA_ERR_SHAPE, call(top_k=3), contains=("top_k 3", "T 100"))
    expect(rd.LORA_ERR_UNSUPPORTED, call(T=rd.LORA_GATHER_MAX_ROWS + 2), contains=("8192",))
    expect(rd.LORA_ERR_NULL, call(idx=0))
    expect(rd.LORA_ERR_WORKSPACE, call(wsb=need - 1))
    expect(rd.LORA_ERR_SHAPE, call(K=256), contains=("expert 0",))
    expect(rd.LORA_ERR_UNSUPPORTED, call(E=17))


def test_pack_stack_refusals_name_the_problem():
    rt = fake_route(L=4, R=16, K=64, N=32)
    A = np.zeros((8, 64), np.uint16)
    B = np.zeros((32, 8), np.uint16)
    expect(rd.LORA_ERR_RANGE, rd.lora_pool_pack_stack, rt, 4, [A], [B], [8], [16.0], [0], [1.0],
           contains=("slot 4", "4 slot"))
    # three members of rank 8 at nonzero scale: 24 > max_rank 16
    expect(rd.LORA_ERR_SHAPE, rd.lora_pool_pack_stack, rt, 0, [A, A, A], [B, B, B], [8, 8, 8],
           [16.0] * 3, [0] * 3, [1.0] * 3, contains=("sum to 24", "max_rank 16"))
    expect(rd.LORA_ERR_SHAPE, rd.lora_pool_pack_stack, rt, 0, [A], [B], [0], [16.0], [0], [1.0],
           contains=("rank 0",))
    expect(rd.LORA_ERR_NULL, rd.lora_pool_pack_stack, rt, 0, [A, 0], [B, B], [8, 8], [16.0] * 2,
           [0] * 2, [1.0] * 2, contains=("member 1",))
    emb = fake_route(kind=rd.LORA_ROUTE_EMBED)
    expect(rd.LORA_ERR_UNSUPPORTED, rd.lora_pool_pack_stack, emb, 0, [A], [B], [8], [16.0], [0], [1.0])


def test_workspace_sizes_by_path():
    """The one-launch path sizes its own exchange workspace for up to 256 rows;
    every other path, and larger batches, the general one."""
    rt = fake_route(L=32, R=16, K=4096, N=6144)
    for M in (17, 64, 256):
        base = rd.lora_proj_workspace_bytes(M, rt)
        one = rd.lora_proj_workspace_bytes(M, rt, rd.LORA_PATH_TC_ONE)
        assert one >= base > 0
        assert rd.lora_proj_workspace_bytes(M, rt, rd.LORA_PATH_TC) == base
        assert rd.lora_proj_workspace_bytes(M, rt, rd.LORA_PATH_SIMT) == base
        gu = rd.lora_gate_up_workspace_bytes(M, rt)
        assert rd.lora_gate_up_workspace_bytes(M, rt, rd.LORA_PATH_TC_ONE) - gu == (one + 255) // 256 * 256 - (base + 255) // 256 * 256
    # fused QKV at 256 rows: the cooperative launch's K-part tiles make it larger
    assert rd.lora_proj_workspace_bytes(256, rt, rd.LORA_PATH_TC_ONE) > rd.lora_proj_workspace_bytes(256, rt)
    assert rd.lora_proj_workspace_bytes(300, rt, rd.LORA_PATH_TC_ONE) == rd.lora_proj_workspace_bytes(300, rt)


def test_static_workspace_refuses_calls_that_outgrow_it():
    rt = fake_route(L=16, R=64, K=4096, N=4096)
    M = 20000
    need = rd.lora_proj_workspace_bytes(M, rt)
    assert need > rd.LORA_STATIC_WS_BYTES
    msg = expect(rd.LORA_ERR_UNSUPPORTED, rd.lora_proj_apply_static_ws, 4096, 4096, 8192, M, 4096, 4096,
                 4096, rt, 4096, 4096)
    for part in (f"{M} rows", "max_rank 64", "16 slots", str(need), str(rd.LORA_STATIC_WS_BYTES)):
        assert part in msg, (part, msg)
    # the decode shapes fit the built-in array
    assert rd.lora_proj_workspace_bytes(64, rt) <= rd.LORA_STATIC_WS_BYTES
