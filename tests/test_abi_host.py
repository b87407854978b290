"""C ABI checks that need no GPU: the library builds and loads, exports
every entry point include/pa.h declares, and rejects bad arguments on the
host (negative pa_status, nothing launched)."""
import ctypes
import os
import re

import pytest

from paged_kv_decode_07_gb300 import build as pabuild
from paged_kv_decode_07_gb300 import pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    pabuild.build()
    return pa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_api():
    fns = declared_functions()
    for name in ("pa_decode", "pa_verify", "pa_merge", "pa_workspace_bytes",
                 "pa_dequant_gather", "pa_append_kv", "pa_read_error", "pa_status_string"):
        assert name in fns


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(pa.EXPORTED) <= set(declared_functions())


def test_status_strings(L):
    assert pa.status_string(0) == "PA_OK"
    assert pa.status_string(-1) == "PA_ERR_INVALID_ARG"
    assert pa.status_string(-3) == "PA_ERR_WORKSPACE_TOO_SMALL"
    assert L.pa_version() >= 100


FAKE = 1 << 20   # a 16-byte aligned non-null address; never dereferenced on the host


def kv_struct(dtype=0, D=256, hkv=4, nb=128, bs=16, scales=True):
    s = pa._KvCache(dtype, nb, bs, hkv, D, FAKE, FAKE, FAKE if scales else None,
                    FAKE if scales else None, 1.0, 1.0)
    return s


def prob_struct(B=2, Hq=24, Q=1, stride=8, max_len=100, out=FAKE, q=FAKE):
    return pa._Problem(B, Hq, Q, q, FAKE, stride, FAKE, max_len, 0.0625, out, 0, None)


def call(L, fn, kv, p, ws=FAKE, ws_bytes=1 << 30, opts=None):
    o = opts if opts is not None else pa._Options(0, 0, 0, None, None)
    return getattr(L, fn)(ctypes.byref(kv), ctypes.byref(p), ctypes.byref(o),
                          ctypes.c_void_p(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("fn", ["pa_decode", "pa_verify"])
def test_invalid_arguments_are_rejected_on_the_host(L, fn):
    assert call(L, fn, kv_struct(D=96), prob_struct()) == pa.PA_ERR_UNSUPPORTED
    assert call(L, fn, kv_struct(bs=32), prob_struct()) == pa.PA_ERR_UNSUPPORTED
    assert call(L, fn, kv_struct(dtype=7), prob_struct()) == pa.PA_ERR_INVALID_ARG
    assert call(L, fn, kv_struct(dtype=1, scales=False), prob_struct()) == pa.PA_ERR_INVALID_ARG
    assert call(L, fn, kv_struct(), prob_struct(Hq=25)) == pa.PA_ERR_INVALID_ARG     # Hq % Hkv
    assert call(L, fn, kv_struct(hkv=1), prob_struct(Hq=16)) == pa.PA_ERR_UNSUPPORTED  # G > 8
    assert call(L, fn, kv_struct(), prob_struct(q=None)) == pa.PA_ERR_INVALID_ARG
    assert call(L, fn, kv_struct(), prob_struct(out=FAKE + 2)) == pa.PA_ERR_INVALID_ARG  # align
    assert call(L, fn, kv_struct(), prob_struct(stride=0)) == pa.PA_ERR_INVALID_ARG
    assert call(L, fn, kv_struct(), prob_struct(B=-1)) == pa.PA_ERR_INVALID_ARG
    assert call(L, fn, kv_struct(), prob_struct(), ws=None) == pa.PA_ERR_INVALID_ARG
    assert call(L, fn, kv_struct(), prob_struct(), ws_bytes=64) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    bad_opts = pa._Options(6, 0, 0, None, None)
    assert call(L, fn, kv_struct(), prob_struct(), opts=bad_opts) == pa.PA_ERR_INVALID_ARG
    # an empty batch is a no-op
    assert call(L, fn, kv_struct(), prob_struct(B=0)) == pa.PA_OK


def test_q_len_limits(L):
    assert call(L, "pa_decode", kv_struct(), prob_struct(Q=2)) == pa.PA_ERR_UNSUPPORTED
    assert call(L, "pa_verify", kv_struct(), prob_struct(Q=17)) == pa.PA_ERR_UNSUPPORTED


def test_workspace_bytes_bounds(L):
    kv = kv_struct()
    small = L.pa_workspace_bytes(ctypes.byref(kv), ctypes.byref(prob_struct(max_len=1000)), None)
    big = L.pa_workspace_bytes(ctypes.byref(kv), ctypes.byref(prob_struct(B=256, max_len=131072)),
                               None)
    assert 0 < small <= big
    assert big < 256 << 20          # partials stay a small fraction of the KV pool
    # forced tiny partitions need more
    o = pa._Options(0, 1, 0, None, None)
    forced = L.pa_workspace_bytes(ctypes.byref(kv), ctypes.byref(prob_struct(max_len=1000)),
                                  ctypes.byref(o))
    assert forced > 0
    # invalid arguments -> 0
    assert L.pa_workspace_bytes(ctypes.byref(kv_struct(D=96)), ctypes.byref(prob_struct()), None) == 0


def test_merge_and_gather_argument_checks(L):
    assert L.pa_merge(None, None, 1, 4, 6, ctypes.c_void_p(FAKE), 0, None, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_merge(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1, 0, 8,
                      ctypes.c_void_p(FAKE), 0, None, None) == pa.PA_OK
    kv = kv_struct()
    assert L.pa_dequant_gather(ctypes.byref(kv), None, 8, ctypes.c_void_p(FAKE), 2, 10,
                               ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), None,
                               None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_read_error(None, None, None) == pa.PA_ERR_INVALID_ARG


def test_append_argument_checks(L):
    F = ctypes.c_void_p(FAKE)
    kv = kv_struct(dtype=1)
    ap = L.pa_append_kv
    assert ap(ctypes.byref(kv), F, F, -1, F, None, None) == pa.PA_ERR_INVALID_ARG
    assert ap(ctypes.byref(kv), None, F, 4, F, None, None) == pa.PA_ERR_INVALID_ARG
    assert ap(ctypes.byref(kv), F, F, 4, None, None, None) == pa.PA_ERR_INVALID_ARG
    assert ap(ctypes.byref(kv), F, ctypes.c_void_p(FAKE + 8), 4, F, None,
              None) == pa.PA_ERR_INVALID_ARG                           # v_new misaligned
    assert ap(ctypes.byref(kv), F, F, 4, ctypes.c_void_p(FAKE + 4), None,
              None) == pa.PA_ERR_INVALID_ARG                           # slot_mapping misaligned
    assert ap(ctypes.byref(kv_struct(dtype=1, D=96)), F, F, 4, F, None,
              None) == pa.PA_ERR_UNSUPPORTED
    assert ap(ctypes.byref(kv_struct(dtype=2, scales=False)), F, F, 4, F, None,
              None) == pa.PA_ERR_INVALID_ARG                           # NVFP4 without scales
    assert ap(None, F, F, 4, F, None, None) == pa.PA_ERR_INVALID_ARG
    assert ap(ctypes.byref(kv), None, None, 0, None, None, None) == pa.PA_OK   # nothing to do


def test_sparse_argument_checks(L):
    F = ctypes.c_void_p(FAKE)
    kv = kv_struct(dtype=1)
    sp = pa._Sparse(64, 256, 4096, FAKE, None)
    p = prob_struct(B=4, Hq=24, stride=16384, max_len=262144)
    o = pa._Options(0, 0, 0, None, None)
    ws = L.pa_sparse_workspace_bytes(ctypes.byref(kv), ctypes.byref(p), ctypes.byref(sp),
                                     ctypes.byref(o))
    assert ws > 0
    for bad in (pa._Sparse(24, 256, 4096, FAKE, None),      # not a multiple of 16
                pa._Sparse(64, 0, 4096, FAKE, None),        # top_k < 1
                pa._Sparse(64, 256, 5000, FAKE, None),      # more than 4096 sparse blocks
                pa._Sparse(64, 256, 100, FAKE, None)):      # max_seq_len beyond the means
        assert L.pa_sparse_workspace_bytes(ctypes.byref(kv), ctypes.byref(p), ctypes.byref(bad),
                                           ctypes.byref(o)) == 0
    # verify-length queries are not supported by the sparse path
    p2 = prob_struct(B=4, Hq=24, Q=2, stride=16384, max_len=262144)
    assert L.pa_decode_sparse(ctypes.byref(kv), ctypes.byref(p2), ctypes.byref(sp), None, F,
                              1 << 30, None) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_decode_sparse(ctypes.byref(kv), ctypes.byref(p), None, None, F, 1 << 30,
                              None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_decode_sparse(ctypes.byref(kv), ctypes.byref(p), ctypes.byref(sp), None, F,
                              16, None) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    bm = L.pa_block_means
    assert bm(ctypes.byref(kv), F, 8, F, None, 0, 2, 64, 0, F, None, None) == pa.PA_ERR_INVALID_ARG
    assert bm(ctypes.byref(kv), F, 8, F, None, -1, 2, 64, 8, F, None, None) == pa.PA_ERR_INVALID_ARG
    assert bm(ctypes.byref(kv), F, 8, F, None, 0, 2, 40, 8, F, None, None) == pa.PA_ERR_UNSUPPORTED
    assert bm(ctypes.byref(kv), None, 8, F, None, 0, 2, 64, 8, F, None, None) == pa.PA_ERR_INVALID_ARG
    assert bm(ctypes.byref(kv), F, 8, F, None, 0, 0, 64, 8, F, None, None) == pa.PA_OK


def test_wo_argument_checks(L):
    F = ctypes.c_void_p(FAKE)
    kv = kv_struct(dtype=1)
    p = prob_struct(B=32, Hq=24, stride=2048, max_len=32768, out=None)
    o = pa._Options(0, 0, 0, None, None)
    wo = pa._Wo(FAKE, 5120, FAKE, 0, 0)
    ws = L.pa_decode_wo_workspace_bytes(ctypes.byref(kv), ctypes.byref(p), ctypes.byref(wo),
                                        ctypes.byref(o))
    # at least o in fp32 (32 x 6144 x 4) on top of the attention workspace
    assert ws >= 32 * 6144 * 4 + L.pa_workspace_bytes(ctypes.byref(kv), ctypes.byref(p),
                                                      ctypes.byref(o))
    for bad in (pa._Wo(FAKE, 100, FAKE, 0, 0),      # hidden not a multiple of 8
                pa._Wo(FAKE, 5120, FAKE, 0, -1)):   # negative split
        assert L.pa_decode_wo_workspace_bytes(ctypes.byref(kv), ctypes.byref(p), ctypes.byref(bad),
                                              ctypes.byref(o)) == 0
    assert L.pa_decode_wo(ctypes.byref(kv), ctypes.byref(p), None, None, F, 1 << 30,
                          None) == pa.PA_ERR_INVALID_ARG
    p_bf16_out = prob_struct(B=32, Hq=24, stride=2048, max_len=32768)   # out given, not fp32
    assert L.pa_decode_wo(ctypes.byref(kv), ctypes.byref(p_bf16_out), ctypes.byref(wo), None, F,
                          1 << 30, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_decode_wo(ctypes.byref(kv), ctypes.byref(p), ctypes.byref(wo), None, F, 64,
                          None) == pa.PA_ERR_WORKSPACE_TOO_SMALL


def test_test_flags_are_checked_on_the_host(L):
    """PA_TEST_EXPIRE_WAIT is built into the tensor-core decode kernel only;
    other kernels and unknown bits are refused before anything is launched."""
    def opts(kernel, flags):
        return pa._Options(kernel, 0, 0, None, None, flags)
    assert call(L, "pa_decode", kv_struct(), prob_struct(), opts=opts(0, 0x2)) == pa.PA_ERR_INVALID_ARG
    assert call(L, "pa_decode", kv_struct(), prob_struct(),
                opts=opts(1, pa.PA_TEST_EXPIRE_WAIT)) == pa.PA_ERR_UNSUPPORTED
    assert call(L, "pa_verify", kv_struct(dtype=2), prob_struct(Q=8),
                opts=opts(0, pa.PA_TEST_EXPIRE_WAIT)) == pa.PA_ERR_UNSUPPORTED    # tcgen05 verify
    assert call(L, "pa_verify", kv_struct(dtype=1), prob_struct(Q=8),
                opts=opts(2, pa.PA_TEST_EXPIRE_WAIT)) == pa.PA_ERR_UNSUPPORTED    # dense tiles


def test_single_launch_kernel_choice_is_checked_on_the_host(L):
    """kernel 5 (single-launch decode) takes pa_decode only; 6 is unknown."""
    def opts(kernel):
        return pa._Options(kernel, 0, 0, None, None, 0)
    assert call(L, "pa_verify", kv_struct(), prob_struct(Q=2), opts=opts(5)) == pa.PA_ERR_UNSUPPORTED
    assert call(L, "pa_verify", kv_struct(), prob_struct(Q=1), opts=opts(5)) == pa.PA_ERR_UNSUPPORTED
    assert call(L, "pa_decode", kv_struct(), prob_struct(), opts=opts(6)) == pa.PA_ERR_INVALID_ARG
    assert call(L, "pa_decode", kv_struct(), prob_struct(), opts=opts(5), ws=None) == pa.PA_ERR_INVALID_ARG
    assert call(L, "pa_decode", kv_struct(), prob_struct(), opts=opts(5),
                ws_bytes=128) == pa.PA_ERR_WORKSPACE_TOO_SMALL


def test_group_sizes_without_a_kernel_are_refused(L):
    """G = 3 (or 5, 7) query heads per kv head has no kernel instantiation: refused on the host."""
    for Hq, hkv in ((12, 4), (20, 4), (28, 4)):
        assert call(L, "pa_decode", kv_struct(hkv=hkv), prob_struct(Hq=Hq)) == pa.PA_ERR_UNSUPPORTED
