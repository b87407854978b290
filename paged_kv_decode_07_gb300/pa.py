"""ctypes binding of the C ABI in include/pa.h (argument marshalling only).

Every step of the attention runs in libpa.so's CUDA kernels; this module
only turns torch tensors into pointers and sizes, picks the current CUDA
stream, and allocates outputs / workspace with torch when the caller does
not pass them.  There is no fallback: if libpa.so is missing or a call
fails, it raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_WORKSPACE_TOO_SMALL = -3
PA_ERR_CUDA = -4

PA_KV_BF16, PA_KV_INT8, PA_KV_NVFP4, PA_KV_FP8 = 0, 1, 2, 3
DTYPE_CODES = {"bf16": PA_KV_BF16, "int8": PA_KV_INT8, "nvfp4": PA_KV_NVFP4, "fp8": PA_KV_FP8}

PA_ERRF_BAD_BLOCK_ID = 0x1
PA_ERRF_LEN_OVER_CAPACITY = 0x2
PA_ERRF_NEG_LEN = 0x4
PA_ERRF_LEN_LT_QLEN = 0x8
PA_ERRF_WAIT_TIMEOUT = 0x10
PA_ERRF_PLAN_OVERFLOW = 0x20
PA_ERRF_BAD_SLOT = 0x40

PA_TEST_EXPIRE_WAIT = 0x1

EXPORTED = ("pa_workspace_bytes", "pa_decode", "pa_verify", "pa_merge", "pa_dequant_gather",
            "pa_append_kv", "pa_block_means", "pa_sparse_workspace_bytes", "pa_decode_sparse",
            "pa_decode_wo_workspace_bytes", "pa_decode_wo",
            "pa_read_error", "pa_status_string", "pa_version")


class PaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


class _KvCache(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("k_global_scale", ctypes.c_float), ("v_global_scale", ctypes.c_float)]


class _Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("q_len", ctypes.c_int32), ("q", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("block_table_stride", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("max_seq_len", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("out", ctypes.c_void_p),
                ("out_fp32", ctypes.c_int32), ("lse_out", ctypes.c_void_p)]


class _Sparse(ctypes.Structure):
    _fields_ = [("sparse_block", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("max_sparse_blocks", ctypes.c_int32), ("means", ctypes.c_void_p),
                ("selected", ctypes.c_void_p)]


class _Wo(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("hidden", ctypes.c_int32), ("y", ctypes.c_void_p),
                ("y_fp32", ctypes.c_int32), ("k_split", ctypes.c_int32)]


class _Options(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("split_blocks", ctypes.c_int32),
                ("target_items", ctypes.c_int32), ("event_begin", ctypes.c_void_p),
                ("event_end", ctypes.c_void_p), ("test_flags", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return LIB_PATH


def lib():
    """Loads libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        P, i32 = ctypes.c_void_p, ctypes.c_int32
        L.pa_workspace_bytes.restype = ctypes.c_size_t
        L.pa_workspace_bytes.argtypes = [P, P, P]
        for fn in ("pa_decode", "pa_verify"):
            getattr(L, fn).restype = ctypes.c_int
            getattr(L, fn).argtypes = [P, P, P, P, ctypes.c_size_t, P]
        L.pa_merge.restype = ctypes.c_int
        L.pa_merge.argtypes = [P, P, i32, i32, i32, P, i32, P, P]
        L.pa_dequant_gather.restype = ctypes.c_int
        L.pa_dequant_gather.argtypes = [P, P, i32, P, i32, i32, P, P, P, P]
        L.pa_block_means.restype = ctypes.c_int
        L.pa_block_means.argtypes = [P, P, i32, P, P, i32, i32, i32, i32, P, P, P]
        L.pa_sparse_workspace_bytes.restype = ctypes.c_size_t
        L.pa_sparse_workspace_bytes.argtypes = [P, P, P, P]
        L.pa_decode_sparse.restype = ctypes.c_int
        L.pa_decode_sparse.argtypes = [P, P, P, P, P, ctypes.c_size_t, P]
        L.pa_decode_wo_workspace_bytes.restype = ctypes.c_size_t
        L.pa_decode_wo_workspace_bytes.argtypes = [P, P, P, P]
        L.pa_decode_wo.restype = ctypes.c_int
        L.pa_decode_wo.argtypes = [P, P, P, P, P, ctypes.c_size_t, P]
        L.pa_append_kv.restype = ctypes.c_int
        L.pa_append_kv.argtypes = [P, P, P, i32, P, P, P]
        L.pa_read_error.restype = ctypes.c_int
        L.pa_read_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_status_string.argtypes = [ctypes.c_int]
        L.pa_version.restype = ctypes.c_int
        L.pa_version.argtypes = []
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class KvCache:
    """The paged KV pool (tensors on the device)."""
    dtype: str
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    k_global: float = 1.0
    v_global: float = 1.0
    block_size: int = 16

    @classmethod
    def from_workload(cls, wl):
        return cls(wl.dtype, wl.k_cache, wl.v_cache, wl.k_scale, wl.v_scale, wl.k_global,
                   wl.v_global)

    @property
    def head_dim(self) -> int:
        return int(self.k_cache.shape[3]) * (2 if self.dtype == "nvfp4" else 1)

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_cache.shape[1])

    def struct(self) -> _KvCache:
        return _KvCache(DTYPE_CODES[self.dtype], int(self.k_cache.shape[0]), self.block_size,
                        self.num_kv_heads, self.head_dim, _ptr(self.k_cache), _ptr(self.v_cache),
                        _ptr(self.k_scale), _ptr(self.v_scale), float(self.k_global),
                        float(self.v_global))


def _options(kernel=0, split_blocks=0, target_items=0, events=None, test_flags=0):
    eb = ee = None
    if events is not None:
        eb = ctypes.c_void_p(events[0].cuda_event)
        ee = ctypes.c_void_p(events[1].cuda_event)
    return _Options(int(kernel), int(split_blocks), int(target_items), eb, ee, int(test_flags))


def _problem(kv: KvCache, q, block_tables, seq_lens, softmax_scale, out, lse, max_seq_len):
    B, Q, Hq, D = q.shape
    return _Problem(B, Hq, Q, _ptr(q), _ptr(block_tables), int(block_tables.shape[1]),
                    _ptr(seq_lens), int(max_seq_len), float(softmax_scale), _ptr(out),
                    1 if out.dtype == torch.float32 else 0, _ptr(lse))


def workspace_bytes(kv: KvCache, batch: int, q_len: int, num_q_heads: int, max_seq_len: int,
                    kernel=0, split_blocks=0, target_items=0) -> int:
    p = _Problem(batch, num_q_heads, q_len, None, None, 1, None, int(max_seq_len), 1.0, None, 0,
                 None)
    o = _options(kernel, split_blocks, target_items)
    return int(lib().pa_workspace_bytes(ctypes.byref(kv.struct()), ctypes.byref(p), ctypes.byref(o)))


def _attend(fn_name, kv, q, block_tables, seq_lens, softmax_scale, *, out=None, out_fp32=False,
            return_lse=False, max_seq_len=None, workspace=None, kernel=0, split_blocks=0,
            target_items=0, events=None, stream=None, test_flags=0):
    B, Q, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Q, Hq, D), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=q.device)
    lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    if max_seq_len is None:
        max_seq_len = int(block_tables.shape[1]) * kv.block_size
    opts = _options(kernel, split_blocks, target_items, events, test_flags)
    kvs = kv.struct()
    prob = _problem(kv, q, block_tables, seq_lens, softmax_scale, out, lse, max_seq_len)
    need = int(lib().pa_workspace_bytes(ctypes.byref(kvs), ctypes.byref(prob), ctypes.byref(opts)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = getattr(lib(), fn_name)(ctypes.byref(kvs), ctypes.byref(prob), ctypes.byref(opts),
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    if st != PA_OK:
        raise PaError(fn_name, st)
    return (out, lse, workspace) if return_lse else (out, workspace)


def decode(kv: KvCache, q, block_tables, seq_lens, softmax_scale, **kw):
    """q bf16 [B, 1, Hq, D] -> (out [B, 1, Hq, D], [lse,] workspace)."""
    return _attend("pa_decode", kv, q, block_tables, seq_lens, softmax_scale, **kw)


def verify(kv: KvCache, q, block_tables, seq_lens, softmax_scale, **kw):
    """q bf16 [B, Q, Hq, D] (Q new tokens, causal) -> (out, [lse,] workspace)."""
    return _attend("pa_verify", kv, q, block_tables, seq_lens, softmax_scale, **kw)


def merge(part_out: torch.Tensor, part_lse: torch.Tensor, *, out_fp32=False, return_lse=False,
          stream=None):
    """part_out fp32 [S, R, D], part_lse fp32 [S, R] -> out [R, D] (+ lse [R])."""
    S, R, D = part_out.shape
    out = torch.empty((R, D), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                      device=part_out.device)
    lse = torch.empty((R,), dtype=torch.float32, device=part_out.device) if return_lse else None
    st = lib().pa_merge(_ptr(part_out), _ptr(part_lse), S, R, D, _ptr(out), 1 if out_fp32 else 0,
                        _ptr(lse), _stream(stream))
    if st != PA_OK:
        raise PaError("pa_merge", st)
    return (out, lse) if return_lse else out


def dequant_gather(kv: KvCache, block_tables, seq_lens, max_len: int, workspace=None, stream=None):
    """-> (k, v) fp32 [B, Hkv, max_len, D] through the table, dequantised."""
    B = int(block_tables.shape[0])
    shape = (B, kv.num_kv_heads, max_len, kv.head_dim)
    k = torch.empty(shape, dtype=torch.float32, device=kv.k_cache.device)
    v = torch.empty(shape, dtype=torch.float32, device=kv.k_cache.device)
    st = lib().pa_dequant_gather(ctypes.byref(kv.struct()), _ptr(block_tables),
                                 int(block_tables.shape[1]), _ptr(seq_lens), B, int(max_len),
                                 _ptr(k), _ptr(v), _ptr(workspace), _stream(stream))
    if st != PA_OK:
        raise PaError("pa_dequant_gather", st)
    return k, v


def block_means(kv: KvCache, block_tables, seq_lens, sparse_block: int, max_sparse_blocks: int,
                first=None, count=0, means=None, workspace=None, stream=None):
    """Mean keys of sparse blocks first[b] .. first[b] + count - 1 (count 0 =
    all) of every sequence, fp32 [B, max_sparse_blocks, Hkv, D] (other
    entries untouched; a new tensor starts at 0)."""
    B = int(block_tables.shape[0])
    if means is None:
        means = torch.zeros((B, max_sparse_blocks, kv.num_kv_heads, kv.head_dim),
                            dtype=torch.float32, device=kv.k_cache.device)
    st = lib().pa_block_means(ctypes.byref(kv.struct()), _ptr(block_tables),
                              int(block_tables.shape[1]), _ptr(seq_lens), _ptr(first),
                              int(count), B, int(sparse_block), int(max_sparse_blocks), _ptr(means),
                              _ptr(workspace), _stream(stream))
    if st != PA_OK:
        raise PaError("pa_block_means", st)
    return means


def _sparse(means, sparse_block, top_k, selected):
    return _Sparse(int(sparse_block), int(top_k), int(means.shape[1]), _ptr(means), _ptr(selected))


def sparse_workspace_bytes(kv: KvCache, batch: int, num_q_heads: int, max_seq_len: int, means,
                           sparse_block: int, top_k: int, kernel=0) -> int:
    p = _Problem(batch, num_q_heads, 1, None, None, 1, None, int(max_seq_len), 1.0, None, 0, None)
    sp = _sparse(means, sparse_block, top_k, None)
    o = _options(kernel)
    return int(lib().pa_sparse_workspace_bytes(ctypes.byref(kv.struct()), ctypes.byref(p),
                                               ctypes.byref(sp), ctypes.byref(o)))


def decode_sparse(kv: KvCache, q, block_tables, seq_lens, softmax_scale, means, sparse_block: int,
                  top_k: int, *, out=None, out_fp32=False, return_lse=False, return_selected=False,
                  max_seq_len=None, workspace=None, kernel=0, split_blocks=0, target_items=0,
                  events=None, stream=None):
    """Block-sparse decode: q bf16 [B, 1, Hq, D]; means from block_means.
    Returns (out, [lse,] [selected int32 [B, Hkv, top_k],] workspace)."""
    B, Q, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Q, Hq, D), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=q.device)
    lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    sel = (torch.empty((B, kv.num_kv_heads, top_k), dtype=torch.int32, device=q.device)
           if return_selected else None)
    if max_seq_len is None:
        max_seq_len = min(int(block_tables.shape[1]) * kv.block_size,
                          int(means.shape[1]) * int(sparse_block))
    opts = _options(kernel, split_blocks, target_items, events)
    kvs = kv.struct()
    prob = _problem(kv, q, block_tables, seq_lens, softmax_scale, out, lse, max_seq_len)
    sp = _sparse(means, sparse_block, top_k, sel)
    need = int(lib().pa_sparse_workspace_bytes(ctypes.byref(kvs), ctypes.byref(prob),
                                               ctypes.byref(sp), ctypes.byref(opts)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().pa_decode_sparse(ctypes.byref(kvs), ctypes.byref(prob), ctypes.byref(sp),
                                ctypes.byref(opts), _ptr(workspace), workspace.numel(),
                                _stream(stream))
    if st != PA_OK:
        raise PaError("pa_decode_sparse", st)
    res = [out]
    if return_lse:
        res.append(lse)
    if return_selected:
        res.append(sel)
    res.append(workspace)
    return tuple(res)


def decode_wo(kv: KvCache, q, block_tables, seq_lens, softmax_scale, w_o, *, y=None,
              y_fp32=False, out=None, return_lse=False, k_split=0, max_seq_len=None,
              workspace=None, kernel=0, split_blocks=0, target_items=0, events=None,
              stream=None):
    """Attention (q_len 1: decode, > 1: verify) and the output projection
    y = o . W_O in one call.  w_o bf16 [Hq * D, hidden]; returns (y
    [B * Q, hidden], [lse,] workspace); `out` (fp32 [B, Q, Hq, D]) receives o."""
    B, Q, Hq, D = q.shape
    hidden = int(w_o.shape[1])
    assert w_o.dtype == torch.bfloat16 and w_o.is_contiguous() and int(w_o.shape[0]) == Hq * D
    if y is None:
        y = torch.empty((B * Q, hidden), dtype=torch.float32 if y_fp32 else torch.bfloat16,
                        device=q.device)
    y_fp32 = y.dtype == torch.float32
    if out is not None:
        assert out.dtype == torch.float32
    lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=q.device) if return_lse else None
    if max_seq_len is None:
        max_seq_len = int(block_tables.shape[1]) * kv.block_size
    opts = _options(kernel, split_blocks, target_items, events)
    kvs = kv.struct()
    prob = _Problem(B, Hq, Q, _ptr(q), _ptr(block_tables), int(block_tables.shape[1]),
                    _ptr(seq_lens), int(max_seq_len), float(softmax_scale), _ptr(out), 1,
                    _ptr(lse))
    wo = _Wo(_ptr(w_o), hidden, _ptr(y), 1 if y_fp32 else 0, int(k_split))
    need = int(lib().pa_decode_wo_workspace_bytes(ctypes.byref(kvs), ctypes.byref(prob),
                                                  ctypes.byref(wo), ctypes.byref(opts)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().pa_decode_wo(ctypes.byref(kvs), ctypes.byref(prob), ctypes.byref(wo),
                            ctypes.byref(opts), _ptr(workspace), workspace.numel(),
                            _stream(stream))
    if st != PA_OK:
        raise PaError("pa_decode_wo", st)
    return (y, lse, workspace) if return_lse else (y, workspace)


def append_kv(kv: KvCache, k_new, v_new, slot_mapping, workspace=None, stream=None):
    """Quantise-on-write of new tokens into the pool (in place).  k_new /
    v_new bf16 [T, Hkv, D]; slot_mapping int64 [T] (-1 = padded row)."""
    T = int(slot_mapping.shape[0])
    if T:
        assert k_new.dtype == torch.bfloat16 and v_new.dtype == torch.bfloat16
        assert slot_mapping.dtype == torch.int64
        assert tuple(k_new.shape) == (T, kv.num_kv_heads, kv.head_dim) == tuple(v_new.shape)
        assert k_new.is_contiguous() and v_new.is_contiguous() and slot_mapping.is_contiguous()
    st = lib().pa_append_kv(ctypes.byref(kv.struct()), _ptr(k_new), _ptr(v_new), T,
                            _ptr(slot_mapping), _ptr(workspace), _stream(stream))
    if st != PA_OK:
        raise PaError("pa_append_kv", st)


def read_error(workspace: torch.Tensor, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    st = lib().pa_read_error(_ptr(workspace), ctypes.byref(flags), _stream(stream))
    if st != PA_OK:
        raise PaError("pa_read_error", st)
    return int(flags.value)


def header(workspace: torch.Tensor):
    """(err, num_items, split_blocks, slots, resident) from the workspace
    header; resident is the count of CTAs the planner rounded the items to
    (0 when it did not round)."""
    h = workspace[:32].view(torch.int32).cpu().tolist()
    return tuple(h[:5])
