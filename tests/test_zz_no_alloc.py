"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Callers such as plugins that only receive their input and output buffers,
or code inside a framework that owns every device allocation, cannot hand
pa_decode a workspace.  pa_decode_noalloc keeps that workspace in a fixed
device array inside the library instead.  This test calls it through the C
ABI twice in a row (different inputs, so the second call runs on whatever
the first left in the shared array) and checks each result against the
fp64 oracle, with the tolerance the other GPU tests use, and against
pa_decode's.  It also checks that refused calls (a problem beyond the
array's size, a q_len pa_decode does not take, a missing output) return
pa_decode's status codes and leave the output untouched.  It lives in its
own file, collected last, and passes alone or after the other tests.
"""
import ctypes

import pytest
import torch

from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import MAX_ABS, REL_L2, compare, oracle_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _fn():
    L = pa.lib()
    f = L.pa_decode_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f


def _noalloc(wl, out):
    kv = pa.KvCache.from_workload(wl)
    prob = pa._problem(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale, out, None,
                       max(wl.max_seq_len(), 1))
    kvs = kv.struct()
    return _fn()(ctypes.byref(kvs), ctypes.byref(prob),
                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(a, b):
    d = (a.double() - b.double())
    rel = d.norm() / b.double().norm().clamp(min=1e-30)
    return float(d.abs().max()) <= MAX_ABS and float(rel) <= REL_L2


def test_noalloc_matches_oracle_twice():
    cases = [("int8_b32_l1k_32k_d256", [3001, 17, 1024, 1, 5000]),
             ("bf16_skewed_b256_l16_128k_d256", [16, 20000, 100, 0, 777])]
    for name, lens in cases:
        wl = W.make_workload(name, device=DEV, seq_lens=lens)
        ref, _ = pa.decode(pa.KvCache.from_workload(wl), wl.q, wl.block_tables, wl.seq_lens,
                           wl.softmax_scale, out_fp32=True, max_seq_len=max(lens))
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(wl, out)
        torch.cuda.synchronize()
        assert st == pa.PA_OK, pa.status_string(st)
        oracle_out, _ = oracle_rows(wl)
        compare(out, oracle_out, f"{name} (no-alloc entry point)")
        assert _close(out, ref), name


def test_noalloc_refuses_problems_beyond_its_scratch():
    wl = W.make_workload("int8_b32_l1k_32k_d256", device=DEV, seq_lens=[64])
    big_B = 4096                       # 4096 sequences need far more than 16 MiB of partials
    q = torch.zeros((big_B, 1, wl.Hq, wl.D), dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros((big_B, 4), dtype=torch.int32, device=DEV)
    lens = torch.full((big_B,), 64, dtype=torch.int32, device=DEV)
    out = torch.empty((big_B, 1, wl.Hq, wl.D), dtype=torch.bfloat16, device=DEV)
    big = W.Workload(**{**wl.__dict__, "B": big_B, "q": q, "block_tables": tables,
                        "seq_lens": lens})
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    assert _noalloc(big, out) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all(), "a refused call wrote its output"


def test_noalloc_refused_arguments_launch_nothing():
    """pa_decode's own status codes come back for bad arguments, and the
    output buffer is left as it was."""
    wl = W.make_workload("int8_b32_l1k_32k_d256", device=DEV, seq_lens=[300, 40], Q=2)
    out = torch.full((wl.B, 2, wl.Hq, wl.D), float("nan"), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    assert _noalloc(wl, out) == pa.PA_ERR_UNSUPPORTED      # q_len 2: decode takes q_len 1
    wl1 = W.make_workload("int8_b32_l1k_32k_d256", device=DEV, seq_lens=[300, 40])
    kv = pa.KvCache.from_workload(wl1)
    prob = pa._problem(kv, wl1.q, wl1.block_tables, wl1.seq_lens, wl1.softmax_scale, out, None,
                       300)
    prob.out = None                                        # no output buffer
    st = _fn()(ctypes.byref(kv.struct()), ctypes.byref(prob),
               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(out).all(), "a refused call wrote its output"
