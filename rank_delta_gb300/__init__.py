"""Python binding of the rank_delta C ABI (include/rank_delta.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, takes device pointers as ints or as objects with
``data_ptr()`` (torch tensors), and raises :class:`LoraError` with the
library's message on a non-zero status. All compute runs in the CUDA library
``_build/librank_delta.so``; there is no other implementation to fall back
on, so importing this package fails loudly when the library is missing
(build it with ``rank_delta_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librank_delta.so")

LORA_OK = 0
LORA_ERR_NULL = 1
LORA_ERR_SHAPE = 2
LORA_ERR_RANGE = 3
LORA_ERR_ALIGN = 4
LORA_ERR_WORKSPACE = 5
LORA_ERR_CUDA = 6
LORA_ERR_UNSUPPORTED = 7
LORA_ERR_NOT_INIT = 8
LORA_ERR_POOL_FULL = 9

LORA_FLAG_SLOT_RANGE = 1 << 0
LORA_FLAG_WAIT_TIMEOUT = 1 << 1
LORA_FLAG_BAD_OFFSETS = 1 << 2
LORA_FLAG_TOKEN_RANGE = 1 << 3
LORA_FLAG_EXPERT_RANGE = 1 << 4
LORA_GATHER_MAX_ROWS = 8192

LORA_ROUTE_PROJ = 0
LORA_ROUTE_EMBED = 1

LORA_PATH_AUTO = 0
LORA_PATH_SIMT = 1
LORA_PATH_TC = 2
LORA_PATH_TC_ONE = 3

LORA_MAX_EXPERTS = 16
LORA_STATIC_WS_BYTES = 8 << 20
LORA_COMP_STRIDE = 256


LORA_PLAN_SIMT = 1
LORA_PLAN_TC = 2
LORA_PLAN_ONE_LAUNCH = 3


class lora_plan_info(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int32),
        ("kernels", ctypes.c_int32),
        ("cluster_size", ctypes.c_int32),
        ("clusters_needed", ctypes.c_int32),
        ("clusters_resident", ctypes.c_int32),
        ("smem_per_cta", ctypes.c_int32),
    ]


class LoraError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code
        self.message = message


class lora_route(ctypes.Structure):
    _fields_ = [
        ("pool", ctypes.c_void_p),
        ("a_table", ctypes.c_void_p),
        ("b_table", ctypes.c_void_p),
        ("scale_table", ctypes.c_void_p),
        ("factor_table", ctypes.c_void_p),
        ("rank_table", ctypes.c_void_p),
        ("comp_table", ctypes.c_void_p),
        ("n_in", ctypes.c_int32),
        ("n_out", ctypes.c_int32),
        ("max_rank", ctypes.c_int32),
        ("max_loras", ctypes.c_int32),
        ("kind", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("magic", ctypes.c_uint64),
    ]


class lora_slot_view(ctypes.Structure):
    _fields_ = [
        ("slot", ctypes.c_int32),
        ("filled", ctypes.c_int32),
        ("ref_count", ctypes.c_int32),
        ("pad", ctypes.c_int32),
        ("last_used", ctypes.c_uint64),
    ]


_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_f = ctypes.c_float
_rtp = ctypes.POINTER(lora_route)
_i32p = ctypes.POINTER(ctypes.c_int32)

# name -> (restype, argtypes)
_SIGNATURES = {
    "lora_pool_bytes": (_sz, [_i, _i, _i, _i]),
    "lora_route_table_bytes": (_sz, [_i]),
    "lora_route_init": (_i, [_rtp, _vp, _sz, _vp, _sz, _i, _i, _i, _i, _vp]),
    "lora_pool_pack": (_i, [_rtp, _i, _vp, _vp, _i, _f, _i, _f, _vp]),
    "lora_pool_pack_stack": (_i, [_rtp, _i, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32p,
                                  ctypes.POINTER(ctypes.c_float), _i32p, ctypes.POINTER(ctypes.c_float), _vp]),
    "lora_pool_unpack": (_i, [_rtp, _i, _vp]),
    "lora_set_scale": (_i, [_rtp, _i, _f, _vp]),
    "lora_set_scales": (_i, [_rtp, _i32p, ctypes.POINTER(ctypes.c_float), _i, _vp]),
    "lora_select_victim_slot": (_i, [ctypes.POINTER(lora_slot_view), _i, _i32p]),
    "lora_proj_workspace_bytes": (_sz, [_i, _rtp]),
    "lora_proj_workspace_bytes_ex": (_sz, [_i, _rtp, _i]),
    "lora_proj_apply": (_i, [_vp, _i64, _vp, _i, _i, _i, _vp, _rtp, _vp, _i64, _vp, _sz, _vp]),
    "lora_proj_apply_ex": (_i, [_vp, _i64, _vp, _i, _i, _i, _vp, _rtp, _vp, _i64, _vp, _sz, _i,
                                _vp]),
    "lora_proj_apply_static_ws": (_i, [_vp, _i64, _vp, _i, _i, _i, _vp, _rtp, _vp, _i64, _vp]),
    "lora_gate_up_workspace_bytes": (_sz, [_i, _rtp]),
    "lora_gate_up_workspace_bytes_ex": (_sz, [_i, _rtp, _i]),
    "lora_gate_up_apply": (_i, [_vp, _i64, _vp, _i, _i, _i, _vp, _rtp, _vp, _i64, _vp, _sz, _vp]),
    "lora_gate_up_apply_ex": (_i, [_vp, _i64, _vp, _i, _i, _i, _vp, _rtp, _vp, _i64, _vp, _sz, _i, _vp]),
    "lora_moe_workspace_bytes": (_sz, [_i, _i, _rtp]),
    "lora_moe_gather_workspace_bytes": (_sz, [_i, _i, _rtp]),
    "lora_moe_gather_apply": (_i, [_vp, _i64, ctypes.POINTER(_vp), _vp, _i, _i, _i, _i, _vp, _rtp,
                                   _vp, _i, _vp, _i64, _vp, _sz, _vp]),
    "lora_moe_down_apply": (_i, [_vp, _i64, ctypes.POINTER(_vp), _vp, _i, _i, _i, _i, _vp, _rtp,
                                 _vp, _i64, _vp, _sz, _vp]),
    "lora_embed_route_init": (_i, [_rtp, _vp, _sz, _vp, _sz, _i, _i, _i, _i, _vp]),
    "lora_embed_pool_pack": (_i, [_rtp, _i, _vp, _vp, _i, _f, _i, _f, _vp]),
    "lora_embed_workspace_bytes": (_sz, [_i, _rtp]),
    "lora_embed_apply": (_i, [_vp, _vp, _i, _i, _i, _vp, _rtp, _vp, _i64, _vp, _sz, _vp]),
    "lora_status_get": (_i, [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]),
    "lora_test_wait_hook": (None, [ctypes.c_uint64, _i]),
    "lora_proj_plan": (_i, [_i, _rtp, _i, _i, ctypes.POINTER(lora_plan_info)]),
    "lora_proj_routing": (_i, [_vp, _i, _i, _i32p, _i32p, _vp]),
    "lora_last_error": (ctypes.c_char_p, []),
    "lora_build_seq_slot": (_i, [_i32p, _i, _i, _i, _i32p]),
}

_lib = None


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"rank_delta CUDA library not built: {LIB_PATH} is missing "
                              "(run rank_delta_gb300.build.build())")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def exported_symbols():
    return list(_SIGNATURES)


def _ptr(v) -> int:
    if v is None:
        return 0
    if hasattr(v, "data_ptr"):
        return int(v.data_ptr())
    return int(v)


def _stream(s) -> int:
    if s is None:
        return 0
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    return int(s)


def _check(code: int) -> None:
    if code != LORA_OK:
        raise LoraError(code, lib().lora_last_error().decode())


def lora_last_error() -> str:
    return lib().lora_last_error().decode()


def lora_pool_bytes(max_loras: int, max_rank: int, n_in: int, n_out: int) -> int:
    return int(lib().lora_pool_bytes(max_loras, max_rank, n_in, n_out))


def lora_route_table_bytes(max_loras: int) -> int:
    return int(lib().lora_route_table_bytes(max_loras))


def lora_route_init(rt: lora_route, pool, pool_bytes: int, tables, table_bytes: int,
                    max_loras: int, max_rank: int, n_in: int, n_out: int, stream=None) -> None:
    _check(lib().lora_route_init(ctypes.byref(rt), _ptr(pool), pool_bytes, _ptr(tables),
                                 table_bytes, max_loras, max_rank, n_in, n_out, _stream(stream)))


def lora_pool_pack(rt: lora_route, slot: int, A, B, rank: int, alpha: float, use_rslora: bool,
                   adapter_scale: float, stream=None) -> None:
    """A and B: device pointers/tensors or host numpy arrays (bf16 bits)."""
    a = A.ctypes.data if hasattr(A, "ctypes") else _ptr(A)
    b = B.ctypes.data if hasattr(B, "ctypes") else _ptr(B)
    _check(lib().lora_pool_pack(ctypes.byref(rt), slot, a, b, rank, alpha, int(bool(use_rslora)),
                                adapter_scale, _stream(stream)))


def lora_pool_pack_stack(rt: lora_route, slot: int, As, Bs, ranks, alphas, use_rslora, adapter_scales,
                         stream=None) -> None:
    """Several adapters in one slot. As / Bs: lists of device pointers/tensors
    or host numpy arrays (bf16 bits); the other arguments are lists of the
    members' rank, alpha, rule and runtime scale."""
    n = len(As)
    keep = [ctypes.c_void_p(a.ctypes.data if hasattr(a, "ctypes") else _ptr(a)) for a in As]
    keep_b = [ctypes.c_void_p(b.ctypes.data if hasattr(b, "ctypes") else _ptr(b)) for b in Bs]
    pa = (ctypes.c_void_p * max(n, 1))(*keep)
    pb = (ctypes.c_void_p * max(n, 1))(*keep_b)
    rk = (ctypes.c_int32 * max(n, 1))(*[int(r) for r in ranks])
    al = (ctypes.c_float * max(n, 1))(*[float(a) for a in alphas])
    rs = (ctypes.c_int32 * max(n, 1))(*[int(bool(r)) for r in use_rslora])
    sc = (ctypes.c_float * max(n, 1))(*[float(v) for v in adapter_scales])
    _check(lib().lora_pool_pack_stack(ctypes.byref(rt), slot, n, pa, pb, rk, al, rs, sc, _stream(stream)))


def lora_pool_unpack(rt: lora_route, slot: int, stream=None) -> None:
    _check(lib().lora_pool_unpack(ctypes.byref(rt), slot, _stream(stream)))


def lora_set_scale(rt: lora_route, slot: int, adapter_scale: float, stream=None) -> None:
    _check(lib().lora_set_scale(ctypes.byref(rt), slot, adapter_scale, _stream(stream)))


def lora_set_scales(rt: lora_route, scales, stream=None) -> None:
    """scales: (slot, adapter_scale) pairs; every slot not listed gets 0."""
    import numpy as np
    ids = np.ascontiguousarray([int(i) for i, _ in scales], dtype=np.int32)
    sc = np.ascontiguousarray([float(v) for _, v in scales], dtype=np.float32)
    _check(lib().lora_set_scales(ctypes.byref(rt), ids.ctypes.data_as(_i32p),
                                 sc.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), len(ids),
                                 _stream(stream)))


def lora_select_victim_slot(cache) -> int:
    """cache: (slot, filled, ref_count, last_used) tuples; returns the slot a
    promotion overwrites, or raises LoraError(LORA_ERR_POOL_FULL)."""
    arr = (lora_slot_view * max(1, len(cache)))()
    for i, (slot, filled, ref_count, last_used) in enumerate(cache):
        arr[i] = lora_slot_view(int(slot), int(bool(filled)), int(ref_count), 0, int(last_used))
    out = ctypes.c_int32(-1)
    _check(lib().lora_select_victim_slot(arr, len(cache), ctypes.byref(out)))
    return int(out.value)


def lora_proj_workspace_bytes(M: int, rt: lora_route, path: int = LORA_PATH_AUTO) -> int:
    if path == LORA_PATH_AUTO:
        return int(lib().lora_proj_workspace_bytes(M, ctypes.byref(rt)))
    return int(lib().lora_proj_workspace_bytes_ex(M, ctypes.byref(rt), path))


def lora_proj_apply(x, x_stride: int, W, M: int, K: int, N: int, seq_slot, rt: lora_route, y,
                    y_stride: int, ws, ws_bytes: int, stream=None, path: int = LORA_PATH_AUTO):
    if path == LORA_PATH_AUTO:
        code = lib().lora_proj_apply(_ptr(x), x_stride, _ptr(W), M, K, N, _ptr(seq_slot),
                                     ctypes.byref(rt), _ptr(y), y_stride, _ptr(ws), ws_bytes,
                                     _stream(stream))
    else:
        code = lib().lora_proj_apply_ex(_ptr(x), x_stride, _ptr(W), M, K, N, _ptr(seq_slot),
                                        ctypes.byref(rt), _ptr(y), y_stride, _ptr(ws), ws_bytes,
                                        path, _stream(stream))
    _check(code)


def lora_proj_apply_static_ws(x, x_stride: int, W, M: int, K: int, N: int, seq_slot,
                              rt: lora_route, y, y_stride: int, stream=None) -> None:
    """lora_proj_apply without a workspace argument, for callers that cannot
    allocate device memory: the library's built-in scratch array is used."""
    _check(lib().lora_proj_apply_static_ws(_ptr(x), x_stride, _ptr(W), M, K, N, _ptr(seq_slot),
                                           ctypes.byref(rt), _ptr(y), y_stride, _stream(stream)))


def lora_gate_up_workspace_bytes(M: int, rt: lora_route, path: int = LORA_PATH_AUTO) -> int:
    if path == LORA_PATH_AUTO:
        return int(lib().lora_gate_up_workspace_bytes(M, ctypes.byref(rt)))
    return int(lib().lora_gate_up_workspace_bytes_ex(M, ctypes.byref(rt), path))


def lora_gate_up_apply(x, x_stride: int, W, M: int, K: int, I: int, seq_slot, rt: lora_route, act,
                       act_stride: int, ws, ws_bytes: int, stream=None, path: int = LORA_PATH_AUTO) -> None:
    if path == LORA_PATH_AUTO:
        code = lib().lora_gate_up_apply(_ptr(x), x_stride, _ptr(W), M, K, I, _ptr(seq_slot),
                                        ctypes.byref(rt), _ptr(act), act_stride, _ptr(ws), ws_bytes,
                                        _stream(stream))
    else:
        code = lib().lora_gate_up_apply_ex(_ptr(x), x_stride, _ptr(W), M, K, I, _ptr(seq_slot),
                                           ctypes.byref(rt), _ptr(act), act_stride, _ptr(ws), ws_bytes,
                                           path, _stream(stream))
    _check(code)


def lora_moe_workspace_bytes(E: int, T: int, rts) -> int:
    arr = (lora_route * E)(*rts)
    return int(lib().lora_moe_workspace_bytes(E, T, arr))


def lora_moe_down_apply(x, x_stride: int, W_e, expert_offsets, E: int, T: int, K: int, N: int,
                        seq_slot, rts, y, y_stride: int, ws, ws_bytes: int, stream=None) -> None:
    wp = (_vp * E)(*[_ptr(w) for w in W_e])
    arr = (lora_route * E)(*rts)
    _check(lib().lora_moe_down_apply(_ptr(x), x_stride, wp, _ptr(expert_offsets), E, T, K, N,
                                     _ptr(seq_slot), arr, _ptr(y), y_stride, _ptr(ws), ws_bytes,
                                     _stream(stream)))


def lora_embed_route_init(rt: lora_route, pool, pool_bytes: int, tables, table_bytes: int,
                          max_loras: int, max_rank: int, vocab: int, n_embd: int, stream=None) -> None:
    _check(lib().lora_embed_route_init(ctypes.byref(rt), _ptr(pool), pool_bytes, _ptr(tables),
                                       table_bytes, max_loras, max_rank, vocab, n_embd,
                                       _stream(stream)))


def lora_embed_pool_pack(rt: lora_route, slot: int, rows, cols, rank: int, alpha: float,
                         use_rslora: bool, adapter_scale: float, stream=None) -> None:
    """The flipped pair: rows [vocab][rank], cols [n_embd][rank] (device
    pointers/tensors or host numpy arrays of bf16 bits)."""
    r = rows.ctypes.data if hasattr(rows, "ctypes") else _ptr(rows)
    c = cols.ctypes.data if hasattr(cols, "ctypes") else _ptr(cols)
    _check(lib().lora_embed_pool_pack(ctypes.byref(rt), slot, r, c, rank, alpha,
                                      int(bool(use_rslora)), adapter_scale, _stream(stream)))


def lora_embed_workspace_bytes(M: int, rt: lora_route) -> int:
    return int(lib().lora_embed_workspace_bytes(M, ctypes.byref(rt)))


def lora_embed_apply(tokens, E, M: int, vocab: int, n_embd: int, seq_slot, rt: lora_route, y,
                     y_stride: int, ws, ws_bytes: int, stream=None) -> None:
    _check(lib().lora_embed_apply(_ptr(tokens), _ptr(E), M, vocab, n_embd, _ptr(seq_slot),
                                  ctypes.byref(rt), _ptr(y), y_stride, _ptr(ws), ws_bytes,
                                  _stream(stream)))


def lora_moe_gather_workspace_bytes(E: int, T: int, rts) -> int:
    arr = (lora_route * E)(*rts)
    return int(lib().lora_moe_gather_workspace_bytes(E, T, arr))


def lora_moe_gather_apply(x, x_stride: int, W_e, indices, E: int, T: int, K: int, N: int, seq_slot, rts,
                          combine, top_k: int, y, y_stride: int, ws, ws_bytes: int, stream=None) -> None:
    wp = (_vp * E)(*[_ptr(w) for w in W_e])
    arr = (lora_route * E)(*rts)
    _check(lib().lora_moe_gather_apply(_ptr(x), x_stride, wp, _ptr(indices), E, T, K, N, _ptr(seq_slot), arr,
                                       _ptr(combine), top_k, _ptr(y), y_stride, _ptr(ws), ws_bytes,
                                       _stream(stream)))


def lora_status_get(ws, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(lib().lora_status_get(_ptr(ws), ctypes.byref(out), _stream(stream)))
    return int(out.value)


def lora_proj_plan(M: int, rt, gated: bool = False, path: int = LORA_PATH_AUTO) -> dict:
    """Which kernels a projection call of M rows on route `rt` and `path`
    takes on the current device (plan, launches, cluster shape and residency)."""
    info = lora_plan_info()
    _check(lib().lora_proj_plan(int(M), ctypes.byref(rt), int(bool(gated)), int(path), ctypes.byref(info)))
    return {f: int(getattr(info, f)) for f, _ in lora_plan_info._fields_}


def lora_test_wait_hook(wait_ns: int, extra_flags: int) -> None:
    """Test hook: bounded device waits give up after wait_ns and wait for
    extra_flags flags nothing writes (0, 0 restores normal operation)."""
    lib().lora_test_wait_hook(int(wait_ns), int(extra_flags))


def lora_proj_routing(ws, M: int, max_loras: int, stream=None):
    import numpy as np
    perm = np.zeros(max(M, 1), dtype=np.int32)
    seg = np.zeros(max_loras + 2, dtype=np.int32)
    _check(lib().lora_proj_routing(_ptr(ws), M, max_loras,
                                   perm.ctypes.data_as(_i32p), seg.ctypes.data_as(_i32p),
                                   _stream(stream)))
    return perm[:M], seg


def lora_build_seq_slot(adapter_slots, padded_n: int, active: int):
    import numpy as np
    a = np.ascontiguousarray(adapter_slots, dtype=np.int32)
    out = np.zeros(max(padded_n, 1), dtype=np.int32)
    _check(lib().lora_build_seq_slot(a.ctypes.data_as(_i32p), a.shape[0], padded_n, active,
                                     out.ctypes.data_as(_i32p)))
    return out[:padded_n]
