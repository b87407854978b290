"""fp64 CPU oracle for paged-KV decode / verify attention and the LSE merge.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the package smoke
check and by the benchmark's CPU-baseline / reference leg, never by the
product library.  The arithmetic lives in ``oracle.c`` (plain C, fp64); this
file compiles it with gcc and marshals numpy arrays through ctypes.  It
shares no code with the CUDA path.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
things other than itself (library decoders, closed forms, a NumPy dense
brute force, invariants).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"bf16": 0, "int8": 1, "nvfp4": 2, "fp8": 3}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (plain gcc)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Cache(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("k_global", ctypes.c_float), ("v_global", ctypes.c_float)]


def _load(path):
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    for fn in ("oracle_bf16_value", "oracle_fp16_value"):
        getattr(L, fn).restype = ctypes.c_double
        getattr(L, fn).argtypes = [ctypes.c_uint16]
    for fn in ("oracle_e4m3_value", "oracle_e2m1_value"):
        getattr(L, fn).restype = ctypes.c_double
        getattr(L, fn).argtypes = [ctypes.c_uint8]
    L.oracle_gather.restype = None
    L.oracle_gather.argtypes = [P, P, i32, P, i32, i32, P, P]
    L.oracle_attend.restype = ctypes.c_int
    L.oracle_attend.argtypes = [P, P, i32, i32, i32, P, i32, P, P, P,
                                ctypes.c_double, P, P, P, i32, i32]
    L.oracle_merge.restype = None
    L.oracle_merge.argtypes = [P, P, i32, i32, i32, P, P]
    L.oracle_append.restype = ctypes.c_int
    L.oracle_append.argtypes = [P, P, P, i32, P]
    L.oracle_block_means.restype = None
    L.oracle_block_means.argtypes = [P, P, i32, P, i32, i32, i32, P]
    L.oracle_sparse_select.restype = None
    L.oracle_sparse_select.argtypes = [P, i32, i32, i32, i32, P, P, i32, i32, P, P]
    L.oracle_attend_sparse.restype = None
    L.oracle_attend_sparse.argtypes = [P, P, i32, i32, P, i32, P, P, i32, i32, ctypes.c_double,
                                       P, P]
    return L


_override = None


def use_library(path):
    """Point this module at another build of oracle.c (used only by the
    mutation test, which compiles deliberately broken copies); None restores
    the real one."""
    global _override
    _override = None if path is None else _load(path)


def lib():
    global _lib
    if _override is not None:
        return _override
    with _lock:
        if _lib is None:
            build()
            _lib = _load(_LIB)
    return _lib



def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class HostCache:
    """Keeps the numpy arrays alive while the C struct points into them."""

    def __init__(self, dtype, k_cache, v_cache, k_scale=None, v_scale=None,
                 k_global=1.0, v_global=1.0, block_size=16):
        self.arrays = [np.ascontiguousarray(a) if a is not None else None
                       for a in (k_cache, v_cache, k_scale, v_scale)]
        k, v, ks, vs = self.arrays
        nb, hkv = k.shape[0], k.shape[1]
        D = k.shape[3] * (2 if dtype == "nvfp4" else 1)
        self.head_dim = D
        self.num_kv_heads = hkv
        self.struct = _Cache(DTYPES[dtype], nb, block_size, hkv, D, _ptr(k), _ptr(v),
                             _ptr(ks), _ptr(vs), k_global, v_global)

    @classmethod
    def from_host_arrays(cls, h: dict, dtype, k_global=1.0, v_global=1.0):
        return cls(dtype, h["k_cache"], h["v_cache"], h.get("k_scale"), h.get("v_scale"),
                   k_global, v_global)


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(bits)


def fp16_value(bits: int) -> float:
    return lib().oracle_fp16_value(bits)


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def gather(cache: HostCache, block_tables, seq_lens, max_len: int):
    """-> (k, v) fp32 [B, Hkv, max_len, D], zeros past seq_len."""
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = t.shape[0]
    shape = (B, cache.num_kv_heads, max_len, cache.head_dim)
    k = np.zeros(shape, np.float32)
    v = np.zeros(shape, np.float32)
    lib().oracle_gather(ctypes.byref(cache.struct), _ptr(t), t.shape[1], _ptr(sl), B, max_len,
                        _ptr(k), _ptr(v))
    return k, v


def attend(cache: HostCache, q_bits, block_tables, seq_lens, scale: float, *,
           key_begin=None, key_end=None, items=None, nthreads: int | None = None):
    """Exact fp64 attention.  q_bits: uint16 bf16 bits [B, Q, Hq, D].
    Returns (out fp64 [B, Q, Hq, D], lse fp64 [B, Q, Hq]).  With `items`
    (int array of (b, kv_head) pairs) only those rows are computed and the
    rest stay NaN."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    B, Q, Hq, D = q.shape
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    kb = None if key_begin is None else np.ascontiguousarray(key_begin, dtype=np.int32)
    ke = None if key_end is None else np.ascontiguousarray(key_end, dtype=np.int32)
    out = np.full((B, Q, Hq, D), np.nan)
    lse = np.full((B, Q, Hq), np.nan)
    it = None if items is None else np.ascontiguousarray(items, dtype=np.int32).reshape(-1, 2)
    n_it = 0 if it is None else it.shape[0]
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    lib().oracle_attend(ctypes.byref(cache.struct), _ptr(q), B, Q, Hq, _ptr(t), t.shape[1],
                        _ptr(sl), _ptr(kb), _ptr(ke), float(scale), _ptr(out), _ptr(lse),
                        _ptr(it), n_it, int(nthreads))
    return out, lse


def merge(part_o, part_lse):
    """part_o [S, R, D] fp64, part_lse [S, R] fp64 -> (out [R, D], lse [R])."""
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    S, R, D = po.shape
    out = np.zeros((R, D))
    lse = np.zeros(R)
    lib().oracle_merge(_ptr(po), _ptr(pl), S, R, D, _ptr(out), _ptr(lse))
    return out, lse


def append(cache: HostCache, k_bits, v_bits, slot_mapping) -> int:
    """Quantise-on-write of new tokens into the cache arrays, in place.
    k_bits / v_bits: uint16 bf16 bits [T, Hkv, D]; slot_mapping int64 [T]
    (-1 = padded row, nothing written).  Returns the number of rows skipped
    for a slot outside [-1, num_blocks * 16)."""
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = sm.shape[0]
    assert k.shape == v.shape and k.shape[0] == T
    assert k.shape[1:] == (cache.num_kv_heads, cache.head_dim)
    for a in cache.arrays:
        assert a is None or a.flags.writeable
    return lib().oracle_append(ctypes.byref(cache.struct), _ptr(k), _ptr(v), T, _ptr(sm))


def block_means(cache: HostCache, block_tables, seq_lens, sparse_block: int, max_nsb: int):
    """Mean dequantised key of every sparse block: fp64 [B, max_nsb, Hkv, D]."""
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = t.shape[0]
    means = np.zeros((B, max_nsb, cache.num_kv_heads, cache.head_dim))
    lib().oracle_block_means(ctypes.byref(cache.struct), _ptr(t), t.shape[1], _ptr(sl), B,
                             int(sparse_block), int(max_nsb), _ptr(means))
    return means


def sparse_select(q_bits, num_kv_heads: int, means, nsb, top_k: int):
    """q_bits uint16 bf16 [B, 1, Hq, D]; means fp64 [B, max_nsb, Hkv, D];
    nsb int [B].  Returns (scores fp64 [B, Hkv, max_nsb], sel int32
    [B, Hkv, top_k] ascending, -1 padded)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    B, Q, Hq, D = q.shape
    assert Q == 1
    m = np.ascontiguousarray(means, dtype=np.float64)
    n = np.ascontiguousarray(nsb, dtype=np.int32)
    max_nsb = m.shape[1]
    scores = np.zeros((B, num_kv_heads, max_nsb))
    sel = np.zeros((B, num_kv_heads, top_k), np.int32)
    lib().oracle_sparse_select(_ptr(q), B, Hq, int(num_kv_heads), D, _ptr(m), _ptr(n), max_nsb,
                               int(top_k), _ptr(scores), _ptr(sel))
    return scores, sel


def attend_sparse(cache: HostCache, q_bits, block_tables, seq_lens, sel, sparse_block: int,
                  scale: float):
    """Exact decode attention over the selected sparse blocks of each kv
    head.  Returns (out fp64 [B, 1, Hq, D], lse fp64 [B, 1, Hq])."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    B, Q, Hq, D = q.shape
    assert Q == 1
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    s = np.ascontiguousarray(sel, dtype=np.int32)
    k = s.shape[2]
    out = np.zeros((B, 1, Hq, D))
    lse = np.zeros((B, 1, Hq))
    lib().oracle_attend_sparse(ctypes.byref(cache.struct), _ptr(q), B, Hq, _ptr(t), t.shape[1],
                               _ptr(sl), _ptr(s), k, int(sparse_block), float(scale), _ptr(out),
                               _ptr(lse))
    return out, lse


def wo_project(out, w_bits):
    """Output projection of decode attention ("vLLM Fork with focus on GB10
    Homelabs", "Roadmap": fused attention + W_O GEMV):
    y[b, n] = sum_k o[b, k] * W[k, n], o the attention output of all query
    heads flattened (k = head * D + d), W bf16 bits [Hq * D, N].  fp64."""
    o = np.asarray(out, dtype=np.float64)
    B = o.shape[0]
    o = o.reshape(B, -1)
    w = (np.ascontiguousarray(w_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    assert w.shape[0] == o.shape[1]
    return o @ w.astype(np.float64)


def attend_workload(wl, *, items=None, nthreads=None, key_begin=None, key_end=None):
    """Convenience: run the oracle on a `workloads.Workload`."""
    from paged_kv_decode_07_gb300.workloads import host_arrays
    h = host_arrays(wl)
    cache = HostCache.from_host_arrays(h, wl.dtype, wl.k_global, wl.v_global)
    return attend(cache, h["q"], h["block_tables"], h["seq_lens"], wl.softmax_scale,
                  items=items, nthreads=nthreads, key_begin=key_begin, key_end=key_end)
