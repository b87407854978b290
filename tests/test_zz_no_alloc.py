"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Callers such as plugins that only receive their input and output buffers,
or code inside a framework that owns every device allocation, cannot hand
pa_decode a workspace.  pa_decode_noalloc keeps that workspace in a fixed
device array inside the library instead.  This test calls it through the C
ABI twice in a row (different inputs, so the second call runs on whatever
the first left in the shared array) and checks each result against
pa_decode's with the tolerance the other GPU tests use; it also checks the
size limit is refused on the host.  It lives in its own file, collected
last, and passes alone or after the other tests.
"""
import ctypes

import pytest
import torch

from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import MAX_ABS, REL_L2

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


def test_noalloc_matches_pa_decode_twice():
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
    assert _noalloc(big, out) == pa.PA_ERR_WORKSPACE_TOO_SMALL
