"""Oracle for the multi-adapter LoRA projection -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` leg may import this package. The product path never does:
the CUDA library has no CPU fallback.

This is a thin ctypes wrapper around ``lora_oracle.c`` (plain fp32 loops,
OpenMP over rows). It shares no code with the CUDA path; the only thing both
sides share is the seeded input generator in ``workloads/``.

Every function here is pinned by ``tests/test_oracle_pins.py`` against things
other than itself: fp64 brute force of the materialised ``(W + s B A) x``,
byte identities (scale 0 and slot -1 equal the base-only product; a fused
q/k/v call equals the three split calls; zero-padded rank equals true rank),
closed forms (rsLoRA vs alpha/r at power-of-four ranks; linearity in the
adapter scale) and the worked examples under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)


def build(force: bool = False) -> str:
    """Compile lora_oracle.c with gcc (plain -O2, no fused multiply-add)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.oracle_set_threads.restype = None
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_scale.restype = ctypes.c_float
            lib.oracle_scale.argtypes = [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_float]
            lib.oracle_slot_sort.restype = None
            lib.oracle_slot_sort.argtypes = [_i32p, ctypes.c_int, ctypes.c_int, _i32p, _i32p]
            lib.oracle_proj.restype = None
            lib.oracle_proj.argtypes = [
                _u16p, ctypes.c_int64, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _i32p, ctypes.c_int, ctypes.POINTER(_u16p), ctypes.POINTER(_u16p), _i32p, _f32p,
                _i32p, ctypes.c_int, _i32p, ctypes.c_int, _f32p]
            lib.oracle_moe.restype = None
            lib.oracle_moe.argtypes = [
                _u16p, ctypes.c_int64, ctypes.POINTER(_u16p), _i32p, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, ctypes.POINTER(_u16p),
                ctypes.POINTER(_u16p), _i32p, _f32p, _i32p, ctypes.c_int, _i32p, ctypes.c_int,
                _f32p]
            lib.oracle_moe_slot_sort.restype = None
            lib.oracle_moe_slot_sort.argtypes = [_i32p, ctypes.c_int, _i32p, ctypes.c_int,
                                                 _i32p, _i32p]
            lib.oracle_embed.restype = None
            lib.oracle_embed.argtypes = [
                _i32p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int,
                ctypes.POINTER(_u16p), ctypes.POINTER(_u16p), _i32p, _f32p, _f32p]
            lib.oracle_moe_gather.restype = None
            lib.oracle_moe_gather.argtypes = [
                _u16p, ctypes.c_int64, ctypes.POINTER(_u16p), _i32p, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, ctypes.POINTER(_u16p),
                ctypes.POINTER(_u16p), _i32p, _f32p, _f32p, ctypes.c_int, _f32p]
            lib.oracle_proj_stack.restype = None
            lib.oracle_proj_stack.argtypes = [
                _u16p, ctypes.c_int64, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _i32p, ctypes.c_int, _i32p, ctypes.POINTER(_u16p), ctypes.POINTER(_u16p), _i32p,
                _f32p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, _f32p]
            lib.oracle_silu_mul.restype = None
            lib.oracle_silu_mul.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, _f32p]
            _lib = lib
    return _lib


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def set_threads(n: int) -> None:
    """Threads of the oracle's OpenMP loops (timing only; results do not depend on it)."""
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def scale(alpha: float, rank: int, use_rslora: bool, adapter_scale: float) -> float:
    """Effective scale of one adapter (fp32)."""
    return float(_load().oracle_scale(ctypes.c_float(alpha), int(rank), int(bool(use_rslora)),
                                      ctypes.c_float(adapter_scale)))


def slot_sort(seq_slot: np.ndarray, max_loras: int):
    """Stable grouping of rows by slot -> (perm [M], seg_off [L+2])."""
    s = np.ascontiguousarray(seq_slot, dtype=np.int32)
    perm = np.empty(s.shape[0], dtype=np.int32)
    seg = np.empty(max_loras + 2, dtype=np.int32)
    _load().oracle_slot_sort(_p(s, _i32p), s.shape[0], max_loras, _p(perm, _i32p), _p(seg, _i32p))
    return perm, seg


class _Tables:
    """Per-slot pointer/rank/scale arrays for the C oracle (keeps buffers alive)."""

    def __init__(self, adapters: Sequence, scales: Optional[Sequence[float]] = None):
        self.keep = []
        n = len(adapters)
        self.A = (_u16p * max(n, 1))()
        self.B = (_u16p * max(n, 1))()
        self.rank = np.zeros(max(n, 1), dtype=np.int32)
        self.scale = np.zeros(max(n, 1), dtype=np.float32)
        for s, ad in enumerate(adapters):
            if ad is None:
                self.A[s] = _u16p()
                self.B[s] = _u16p()
                continue
            a = np.ascontiguousarray(ad.A, dtype=np.uint16)
            b = np.ascontiguousarray(ad.B, dtype=np.uint16)
            self.keep += [a, b]
            self.A[s] = _p(a, _u16p)
            self.B[s] = _p(b, _u16p)
            self.rank[s] = ad.rank
            if scales is not None:
                self.scale[s] = np.float32(scales[s])
            else:
                self.scale[s] = np.float32(scale(ad.alpha, ad.rank, ad.use_rslora, ad.adapter_scale))


def _idx(v, n):
    if v is None:
        return None, n
    a = np.ascontiguousarray(v, dtype=np.int32)
    return a, a.shape[0]


def proj(x: np.ndarray, W: np.ndarray, seq_slot: np.ndarray, adapters: Sequence,
         rows=None, cols=None, scales: Optional[Sequence[float]] = None) -> np.ndarray:
    """y = W x + s B (A x) per row, fp32, for the selected rows x columns.

    ``x`` [M][K] and ``W`` [N][K] are bf16 bits (uint16); ``adapters[s]`` is a
    ``workloads.Adapter`` at its true rank (or None). ``scales`` overrides the
    per-slot effective scale (default: :func:`scale` of each adapter).
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    ss = np.ascontiguousarray(seq_slot, dtype=np.int32)
    M, K = x.shape
    N = W.shape[0]
    assert W.shape[1] == K and ss.shape[0] == M
    t = _Tables(adapters, scales)
    r, nr = _idx(rows, M)
    c, nc = _idx(cols, N)
    y = np.empty((nr, nc), dtype=np.float32)
    _load().oracle_proj(_p(x, _u16p), K, _p(W, _u16p), M, K, N, _p(ss, _i32p), len(adapters),
                        t.A, t.B, _p(t.rank, _i32p), _p(t.scale, _f32p),
                        _p(r, _i32p) if r is not None else None, nr,
                        _p(c, _i32p) if c is not None else None, nc, _p(y, _f32p))
    return y


def proj_stack(x: np.ndarray, W: np.ndarray, seq_slot: np.ndarray, stacks: Sequence,
               rows=None, cols=None) -> np.ndarray:
    """y = W x + sum_m s_m B_m (A_m x) per row over the members of the row's
    slot, in order, fp32 (ferrox ``LoraStack::add_to``).

    ``stacks[s]`` is a list of ``workloads.Adapter`` (empty or None: no
    members); each member's scale is :func:`scale` of its own alpha, rank,
    rule and adapter scale.
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    ss = np.ascontiguousarray(seq_slot, dtype=np.int32)
    M, K = x.shape
    N = W.shape[0]
    assert W.shape[1] == K and ss.shape[0] == M
    L = len(stacks)
    members = []
    off = np.zeros(L + 1, dtype=np.int32)
    for s_, st in enumerate(stacks):
        members += list(st or [])
        off[s_ + 1] = len(members)
    t = _Tables(members)
    r, nr = _idx(rows, M)
    c, nc = _idx(cols, N)
    y = np.empty((nr, nc), dtype=np.float32)
    _load().oracle_proj_stack(_p(x, _u16p), K, _p(W, _u16p), M, K, N, _p(ss, _i32p), L,
                              _p(off, _i32p), t.A, t.B, _p(t.rank, _i32p), _p(t.scale, _f32p),
                              _p(r, _i32p) if r is not None else None, nr,
                              _p(c, _i32p) if c is not None else None, nc, _p(y, _f32p))
    return y


def moe(x: np.ndarray, W: List[np.ndarray], expert_offsets: np.ndarray, seq_slot: np.ndarray,
        adapters: Sequence[Sequence], rows=None, cols=None) -> np.ndarray:
    """MoE expert down projection: slot-row j uses its expert's W and adapters."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, K = x.shape
    E = len(W)
    N = W[0].shape[0]
    L = len(adapters[0])
    Ws = [np.ascontiguousarray(w, dtype=np.uint16) for w in W]
    Wp = (_u16p * E)(*[_p(w, _u16p) for w in Ws])
    flat = [ad for per_e in adapters for ad in per_e]
    t = _Tables(flat)
    off = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    ss = np.ascontiguousarray(seq_slot, dtype=np.int32)
    r, nr = _idx(rows, T)
    c, nc = _idx(cols, N)
    y = np.empty((nr, nc), dtype=np.float32)
    _load().oracle_moe(_p(x, _u16p), K, Wp, _p(off, _i32p), E, T, K, N, _p(ss, _i32p), L,
                       t.A, t.B, _p(t.rank, _i32p), _p(t.scale, _f32p),
                       _p(r, _i32p) if r is not None else None, nr,
                       _p(c, _i32p) if c is not None else None, nc, _p(y, _f32p))
    return y


def moe_gather(x: np.ndarray, W: List[np.ndarray], indices: np.ndarray, seq_slot: np.ndarray,
               adapters: Sequence[Sequence], combine: Optional[np.ndarray] = None,
               top_k: int = 1) -> np.ndarray:
    """Decode-path MoE fold keyed by a per-slot-row expert index; with combine
    weights, each token's top_k slot-rows summed with their weights."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, K = x.shape
    E = len(W)
    N = W[0].shape[0]
    L = len(adapters[0])
    Ws = [np.ascontiguousarray(w, dtype=np.uint16) for w in W]
    Wp = (_u16p * E)(*[_p(w, _u16p) for w in Ws])
    t = _Tables([ad for per_e in adapters for ad in per_e])
    idx = np.ascontiguousarray(indices, dtype=np.int32)
    ss = np.ascontiguousarray(seq_slot, dtype=np.int32)
    if combine is None:
        y = np.empty((T, N), dtype=np.float32)
        cw = None
    else:
        assert T % top_k == 0
        y = np.empty((T // top_k, N), dtype=np.float32)
        cw = np.ascontiguousarray(combine, dtype=np.float32)
    _load().oracle_moe_gather(_p(x, _u16p), K, Wp, _p(idx, _i32p), E, T, K, N, _p(ss, _i32p), L,
                              t.A, t.B, _p(t.rank, _i32p), _p(t.scale, _f32p),
                              _p(cw, _f32p) if cw is not None else None, int(top_k), _p(y, _f32p))
    return y


def workload_moe_gather(wl, with_combine: bool = True) -> np.ndarray:
    """Oracle output for a ``workloads.MoeGatherWorkload``."""
    return moe_gather(wl.x, wl.W, wl.indices, wl.seq_slot, wl.adapters,
                      combine=wl.combine if with_combine else None, top_k=wl.top_k)


def moe_slot_sort(expert_offsets: np.ndarray, seq_slot: np.ndarray, max_loras: int):
    """Stable grouping of slot-rows by (expert, slot) -> (perm, seg_off [E*(L+1)+1])."""
    off = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    ss = np.ascontiguousarray(seq_slot, dtype=np.int32)
    E = off.shape[0] - 1
    perm = np.empty(int(off[-1]), dtype=np.int32)
    seg = np.empty(E * (max_loras + 1) + 1, dtype=np.int32)
    _load().oracle_moe_slot_sort(_p(off, _i32p), E, _p(ss, _i32p), max_loras,
                                 _p(perm, _i32p), _p(seg, _i32p))
    return perm, seg


def embed(tokens: np.ndarray, E: np.ndarray, seq_slot: np.ndarray, adapters: Sequence,
          scales: Optional[Sequence[float]] = None) -> np.ndarray:
    """Row gather of the adapted matrix: y[i] = E[t_i] + s B[t_i] A, fp32.

    ``E`` [vocab][n_embd] bf16 bits; ``adapters[s]`` holds ``A`` [rank][n_embd]
    and ``B`` [vocab][rank] (the layouts of the adapted matrix, rows = vocab).
    """
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    E = np.ascontiguousarray(E, dtype=np.uint16)
    ss = np.ascontiguousarray(seq_slot, dtype=np.int32)
    vocab, n_embd = E.shape
    M = tok.shape[0]
    assert ss.shape[0] == M
    t = _Tables(adapters, scales)
    y = np.empty((M, n_embd), dtype=np.float32)
    _load().oracle_embed(_p(tok, _i32p), _p(E, _u16p), M, vocab, n_embd, _p(ss, _i32p),
                         len(adapters), t.A, t.B, _p(t.rank, _i32p), _p(t.scale, _f32p),
                         _p(y, _f32p))
    return y


def silu_mul(y: np.ndarray, I: int) -> np.ndarray:
    """act = silu(y[:, :I]) * y[:, I:2I] in fp32 (y: fp32 [M][2I] projection output)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    M = y.shape[0]
    assert y.shape[1] >= 2 * I
    act = np.empty((M, I), dtype=np.float32)
    _load().oracle_silu_mul(_p(y, _f32p), M, I, y.shape[1], _p(act, _f32p))
    return act


def gate_up(x: np.ndarray, W: np.ndarray, seq_slot: np.ndarray, adapters: Sequence,
            rows=None, scales: Optional[Sequence[float]] = None) -> np.ndarray:
    """Gated MLP input: the fused [gate|up] projection (W [2I][K], adapters'
    B [2I][r]) followed by silu(gate) * up, fp32 [rows][I]."""
    I = W.shape[0] // 2
    y = proj(x, W, seq_slot, adapters, rows=rows, scales=scales)
    return silu_mul(y, I)


def workload_embed(wl) -> np.ndarray:
    """Oracle output for a ``workloads.EmbedWorkload``."""
    return embed(wl.tokens, wl.E, wl.seq_slot, wl.adapters)


def workload_proj(wl, rows=None, cols=None) -> np.ndarray:
    """Oracle output for a ``workloads.ProjWorkload``."""
    return proj(wl.x, wl.W, wl.seq_slot, wl.adapters, rows=rows, cols=cols)


def workload_moe(wl, rows=None, cols=None) -> np.ndarray:
    """Oracle output for a ``workloads.MoeWorkload``."""
    return moe(wl.x, wl.W, wl.expert_offsets, wl.seq_slot, wl.adapters, rows=rows, cols=cols)


class _use_library:
    """Test hook: run the wrapper against another build of lora_oracle.c.

    Used only by tests/test_oracle_mutants.py to show that the pins reject a
    copy of the oracle with a planted mistake.
    """

    def __init__(self, so_path: str):
        self.path = so_path

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_scale", "oracle_slot_sort", "oracle_proj", "oracle_moe",
                     "oracle_moe_slot_sort", "oracle_embed", "oracle_silu_mul", "oracle_moe_gather",
                     "oracle_proj_stack"):
            src = getattr(self.saved, name)
            dst = getattr(lib, name)
            dst.restype = src.restype
            dst.argtypes = src.argtypes
        _lib = lib
        return lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False
