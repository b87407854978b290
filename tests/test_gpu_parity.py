"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

* every workload at reduced sizes that span several partitions and ragged
  tails, compared element by element (fp32 output within the tolerance;
  bf16 output equal to bf16_RNE of the fp32 output; LSE);
* every workload at full size in the benchmark's launch configuration,
  every sequence compared with the oracle (in chunks of sequences);
* the dequant-only debug kernel bit-exact against the oracle's gather;
* GQA group sizes and head dims the library supports.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import bf16_matches_fp32, compare, compare_lse, oracle_rows, run

pytestmark = pytest.mark.gpu
DEV = "cuda"

REDUCED = {
    "bf16_b1_l1000_d128": dict(),                                    # full size (tiny)
    "int8_b32_l1k_32k_d256": dict(seq_lens=[1024, 3001, 1500, 2047, 17, 4101, 1, 16]),
    "nvfp4_b4_l262k_d256": dict(seq_lens=[8195, 5000]),
    "nvfp4_verify_q8_b4_ctx64k_d256": dict(seq_lens=[4104, 1008, 8, 9]),
    "fp8_b32_l1k_32k_d256": dict(seq_lens=[1024, 3001, 1500, 2047, 17, 4101, 1, 16]),
    "fp8_verify_q8_b4_ctx64k_d256": dict(seq_lens=[4104, 1008, 8, 9]),
    "bf16_skewed_b256_l16_128k_d256": dict(seq_lens=[16, 17, 100, 1000, 5000, 20000, 31, 64,
                                                     2048, 0, 130, 7777]),
}


def _fn(wl):
    return "verify" if wl.Q > 1 else "decode"


def _kernels(dtype, q_len=1):
    """0 = auto; 1 = CUDA-core kernel; 2 = tensor-core kernel (verify: dense
    tile); 3 = tensor-core kernel with verify as one unit per query token;
    4 = tcgen05 verify (NVFP4 / FP8, q_len > 1); 5 = single-launch decode
    (one thread-block cluster per sequence and kv head, q_len 1)."""
    if dtype in ("nvfp4", "fp8") and q_len > 1:
        return [0, 1, 2, 3, 4]
    if q_len > 1:
        return [0, 1, 2, 3]
    return [0, 1, 2, 3, 5]


REDUCED_CASES = [(n, k) for n in REDUCED
                 for k in _kernels(W.spec(n)["dtype"], W.spec(n).get("Q", 1))]


@pytest.mark.parametrize("name,kernel", REDUCED_CASES)
def test_reduced_parity(name, kernel):
    wl = W.make_workload(name, device=DEV, **REDUCED[name])
    o32, lse, ws = run(wl, _fn(wl), out_fp32=True, return_lse=True, kernel=kernel)
    ob, _ = run(wl, _fn(wl), kernel=kernel)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, name)
    compare_lse(lse, ref_l, name)
    assert bf16_matches_fp32(ob, o32), "bf16 output is not RNE of the fp32 output"


FULL_NAMES = ("int8_b32_l1k_32k_d256", "nvfp4_b4_l262k_d256", "nvfp4_verify_q8_b4_ctx64k_d256",
              "fp8_b32_l1k_32k_d256", "fp8_verify_q8_b4_ctx64k_d256",
              "bf16_skewed_b256_l16_128k_d256")

# auto kernel for every workload; bf16 also on both of its kernels explicitly
FULL_CASES = [(n, 0) for n in FULL_NAMES] + [("bf16_skewed_b256_l16_128k_d256", 1),
                                              ("bf16_skewed_b256_l16_128k_d256", 2)]
# sequences per oracle call: bounds the host copy of the pool (the skewed
# batch holds 15 GB of KV)
ORACLE_CHUNK = 32
_full_ref = {}   # workload name -> oracle (out, lse) of every sequence, shared by its cases


def _full_reference(wl):
    if wl.name not in _full_ref:
        outs, lses = [], []
        for c0 in range(0, wl.B, ORACLE_CHUNK):
            o, l = oracle_rows(wl, list(range(c0, min(wl.B, c0 + ORACLE_CHUNK))))
            outs.append(o)
            lses.append(l)
        _full_ref[wl.name] = (np.concatenate(outs), np.concatenate(lses))
    return _full_ref[wl.name]


@pytest.mark.parametrize("name,kernel", FULL_CASES)
def test_full_size_parity(name, kernel):
    """Every workload at its full size in the benchmark's launch
    configuration (one call over the whole batch, so the split-K plan and the
    merge act on all of it); EVERY sequence is compared element by element
    with the oracle, in chunks of sequences."""
    wl = W.make_workload(name, device=DEV)
    o32, lse, ws = run(wl, _fn(wl), out_fp32=True, return_lse=True, kernel=kernel)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    o32, lse = o32.cpu(), lse.cpu()
    ref_o, ref_l = _full_reference(wl)
    for c0 in range(0, wl.B, ORACLE_CHUNK):
        bs = slice(c0, min(wl.B, c0 + ORACLE_CHUNK))
        what = f"{name} kernel {kernel} sequences {c0}..{bs.stop - 1}"
        compare(o32[bs], ref_o[bs], what)
        compare_lse(lse[bs], ref_l[bs], what)
    del wl
    torch.cuda.empty_cache()


DECODE_NAMES = {"bf16": "bf16_skewed_b256_l16_128k_d256", "int8": "int8_b32_l1k_32k_d256",
                "nvfp4": "nvfp4_b4_l262k_d256", "fp8": "fp8_b32_l1k_32k_d256"}
VERIFY_NAMES = {"nvfp4": "nvfp4_verify_q8_b4_ctx64k_d256", "int8": "int8_b32_l1k_32k_d256",
                "fp8": "fp8_verify_q8_b4_ctx64k_d256"}


@pytest.mark.parametrize("dt", ["bf16", "int8", "nvfp4", "fp8"])
def test_dequant_gather_bit_exact(dt):
    name = DECODE_NAMES[dt]
    lens = [33, 1, 200, 16, 0, 47]
    wl = W.make_workload(name, device=DEV, seq_lens=lens)
    kv = pa.KvCache.from_workload(wl)
    maxl = max(lens) + 5
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    k, v = pa.dequant_gather(kv, wl.block_tables, wl.seq_lens, maxl, workspace=ws)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    h = W.host_arrays(wl)
    cache = oracle.HostCache.from_host_arrays(h, wl.dtype, wl.k_global, wl.v_global)
    rk, rv = oracle.gather(cache, h["block_tables"], h["seq_lens"], maxl)
    kg, vg = k.cpu().numpy(), v.cpu().numpy()
    assert np.array_equal(kg.view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(vg.view(np.uint32), rv.view(np.uint32))


@pytest.mark.parametrize("dt,kernel", [(d, k) for d in ("bf16", "int8", "nvfp4", "fp8")
                                       for k in (1, 2, 5)])
@pytest.mark.parametrize("shape", [(8, 8, 128), (16, 8, 128), (12, 2, 256), (4, 4, 256),
                                   (32, 4, 256), (2, 1, 128)])
def test_gqa_and_head_dim_variants(dt, kernel, shape):
    Hq, Hkv, D = shape
    wl = W.make_workload(DECODE_NAMES[dt], device=DEV, seq_lens=[700, 33, 1], Hq=Hq, Hkv=Hkv,
                         D=D)
    o32, lse, _ = run(wl, out_fp32=True, return_lse=True, kernel=kernel)
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, f"{dt} {shape}")
    compare_lse(lse, ref_l, f"{dt} {shape}")


@pytest.mark.parametrize("Q", [2, 5, 8, 16])
@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
@pytest.mark.parametrize("dt", ["nvfp4", "int8", "fp8"])
def test_verify_q_lens(Q, kernel, dt):
    if kernel == 4 and dt == "int8":
        pytest.skip("the tcgen05 verify kernel takes NVFP4 and FP8")
    wl = W.make_workload(VERIFY_NAMES[dt], device=DEV, seq_lens=[900, Q, 33, 3000], Q=Q)
    o32, lse, _ = run(wl, "verify", out_fp32=True, return_lse=True, kernel=kernel)
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, f"verify Q={Q}")
    compare_lse(lse, ref_l, f"verify Q={Q}")


def test_merge_entry_point_matches_oracle():
    g = torch.Generator(device="cpu").manual_seed(9)
    S, R, D = 7, 50, 256
    po = torch.randn(S, R, D, generator=g)
    pl = torch.randn(S, R, generator=g) * 3
    pl[2, :10] = -float("inf")
    pl[:, 20] = -float("inf")                  # an all-empty row
    out, lse = pa.merge(po.to(DEV), pl.to(DEV), out_fp32=True, return_lse=True)
    ref_o, ref_l = oracle.merge(po.double().numpy(), pl.double().numpy())
    np.testing.assert_allclose(out.cpu().double().numpy(), ref_o, atol=1e-5, rtol=0)
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(lse.cpu().double().numpy()[fin], ref_l[fin], atol=1e-5)
    assert (lse.cpu().numpy()[~fin] == -np.inf).all()
    ob = pa.merge(po.to(DEV), pl.to(DEV))
    assert bf16_matches_fp32(ob, out)


@pytest.mark.parametrize("split", [5, 13, 21, 1 << 20])
@pytest.mark.parametrize("name", ["nvfp4_verify_q8_b4_ctx64k_d256", "fp8_verify_q8_b4_ctx64k_d256"])
def test_umma_verify_many_items_per_cta(name, split):
    """tcgen05 verify with partitions of `split` blocks: every CTA walks
    several items whose last 128-token tile is partial (5, 13, 21 blocks) or
    one long item per (sequence, kv head); each must match the oracle."""
    wl = W.make_workload(name, device=DEV, seq_lens=[4104, 3001, 777, 9, 2048, 1500])
    o32, lse, ws = run(wl, "verify", out_fp32=True, return_lse=True, kernel=4, split_blocks=split)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, f"{name} split {split}")
    compare_lse(lse, ref_l, f"{name} split {split}")


@pytest.mark.parametrize("name", ["nvfp4_verify_q8_b4_ctx64k_d256", "fp8_verify_q8_b4_ctx64k_d256"])
def test_umma_verify_full_size(name):
    """tcgen05 verify (selected explicitly) at the full workload size in the
    benchmark's launch configuration, every sequence against the oracle."""
    wl = W.make_workload(name, device=DEV)
    o32, lse, ws = run(wl, "verify", out_fp32=True, return_lse=True, kernel=4)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, name)
    compare_lse(lse, ref_l, name)
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dt", ["bf16", "int8", "nvfp4", "fp8"])
def test_small_problem_runs_as_one_launch(dt):
    """Auto mode sends a problem whose sequences have at most 1,024 keys
    (and whose clusters fit on the GPU at once) to the single-launch
    decode: no plan is written (the header's item count stays 0), and the
    result matches the oracle, including a padded row and a one-key row."""
    lens = [1000, 1, 0, 1024]   # 4 sequences x 4 kv heads x clusters of 8 = 128 CTAs
    wl = W.make_workload(DECODE_NAMES[dt], device=DEV, seq_lens=lens)
    o32, lse, ws = run(wl, out_fp32=True, return_lse=True)
    ob, ws2 = run(wl)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    assert pa.header(ws)[1] == 0, "planned: the single-launch path was not taken"
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, f"{dt} single launch")
    compare_lse(lse, ref_l, f"{dt} single launch")
    assert bf16_matches_fp32(ob, o32), "bf16 output is not RNE of the fp32 output"


def test_single_launch_reports_bad_lengths():
    """Length errors of the single-launch path reach the header: a sequence
    longer than its table's capacity is clamped and flagged."""
    wl = W.make_workload("bf16_b1_l1000_d128", device=DEV, seq_lens=[300, 200])
    seq = wl.seq_lens.clone()
    seq[1] = wl.block_tables.shape[1] * 16 + 40
    kv = pa.KvCache.from_workload(wl)
    out, ws = pa.decode(kv, wl.q, wl.block_tables, seq, wl.softmax_scale, kernel=5,
                        max_seq_len=300)
    torch.cuda.synchronize()
    assert pa.read_error(ws) & pa.PA_ERRF_LEN_OVER_CAPACITY
