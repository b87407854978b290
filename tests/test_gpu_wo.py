"""GPU parity of attention + output projection (pa_decode_wo through the C
ABI) against the oracle: y = o . W_O with o the exact attention output.

Tolerance: W_O ~ N(0, 1/K) keeps |y| on the scale of |o|, and y's error is
o's error carried through W (the bf16 hi + lo split of o adds < 2^-16
relative), so y is held to the same 2e-3 / 1e-3 as the attention output.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import compare, oracle_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = {"bf16": "bf16_skewed_b256_l16_128k_d256", "int8": "int8_b32_l1k_32k_d256",
         "fp8": "fp8_b32_l1k_32k_d256", "nvfp4": "nvfp4_b4_l262k_d256"}
LENS = [1500, 33, 700, 1, 4000]


def w_o(K, N, seed=11):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(K, N, generator=g) / np.sqrt(K)).to(torch.bfloat16)


def run_wo(wl, w, fn="decode", **kw):
    kv = pa.KvCache.from_workload(wl)
    o = torch.empty((wl.B, wl.Q, wl.Hq, wl.D), dtype=torch.float32, device=DEV)
    y, ws = pa.decode_wo(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale, w.to(DEV),
                         out=o, max_seq_len=max(wl.max_seq_len(), 1), **kw)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    return y, o


def w_bits(w):
    return w.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("hidden", [5120, 200])
@pytest.mark.parametrize("dt", ["bf16", "int8", "fp8", "nvfp4"])
def test_decode_wo_parity(dt, hidden):
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=LENS)
    w = w_o(wl.Hq * wl.D, hidden)
    y, o = run_wo(wl, w, y_fp32=True)
    ref_o, _ = oracle_rows(wl)
    compare(o, ref_o, f"o {dt}")
    ref_y = oracle.wo_project(ref_o, w_bits(w))
    compare(y, ref_y, f"y {dt} N={hidden}")


@pytest.mark.parametrize("k_split", [1, 3, 0])
def test_split_settings_agree_and_repeat_bitwise(k_split):
    wl = W.make_workload(NAMES["int8"], device=DEV, seq_lens=LENS)
    w = w_o(wl.Hq * wl.D, 1024)
    y1, _ = run_wo(wl, w, y_fp32=True, k_split=k_split)
    y2, _ = run_wo(wl, w, y_fp32=True, k_split=k_split)
    assert torch.equal(y1, y2)
    ref_o, _ = oracle_rows(wl)
    compare(y1, oracle.wo_project(ref_o, w_bits(w)), f"split {k_split}")
    yb, _ = run_wo(wl, w, y_fp32=False, k_split=k_split)
    assert torch.equal(yb.view(torch.int16), y1.to(torch.bfloat16).view(torch.int16))


def test_verify_wo_rows_per_query_token():
    wl = W.make_workload("nvfp4_verify_q8_b4_ctx64k_d256", device=DEV, seq_lens=[900, 8, 3000])
    w = w_o(wl.Hq * wl.D, 640)
    y, o = run_wo(wl, w, y_fp32=True)
    ref_o, _ = oracle_rows(wl)
    compare(o, ref_o, "verify o")
    assert y.shape == (wl.B * wl.Q, 640)
    compare(y, oracle.wo_project(ref_o.reshape(wl.B * wl.Q, 1, wl.Hq, wl.D), w_bits(w)),
            "verify y")


def test_more_than_64_rows_and_head_dim_128():
    lens = [int(x) for x in np.random.default_rng(4).integers(1, 300, size=70)]
    wl = W.make_workload(NAMES["bf16"], device=DEV, seq_lens=lens, Hq=8, Hkv=2, D=128)
    w = w_o(wl.Hq * wl.D, 384)
    y, _ = run_wo(wl, w, y_fp32=True)
    ref_o, _ = oracle_rows(wl)
    compare(y, oracle.wo_project(ref_o, w_bits(w)), "70 rows")


def test_full_size_decode_wo_sampled_rows():
    wl = W.make_workload(NAMES["int8"], device=DEV)
    w = w_o(wl.Hq * wl.D, 5120)
    y, o = run_wo(wl, w, y_fp32=True)
    bs = [0, 7, wl.B - 1]
    ref_o, _ = oracle_rows(wl, bs)
    compare(o[bs], ref_o, "full o")
    # y of the sampled rows from the GPU's own o must equal the oracle product of it,
    # and y from the oracle's o within the tolerance
    compare(y[bs], oracle.wo_project(ref_o, w_bits(w)), "full y")
