"""GPU invariants and device-side error handling (no fault is ever
provoked: bad inputs are ones the kernels check and skip, with a sticky
flag in the workspace header).

* physical-block permutation gives bitwise-identical output;
* run-to-run bitwise determinism (no float atomics);
* forced single partition, forced tiny partitions and auto agree;
* equal-length batches are planned in whole rounds of resident CTAs;
* padded rows (seq_len 0) give 0 and lse -inf;
* an out-of-range block id is skipped and flagged; a length beyond the
  table's capacity is clamped and flagged; verify rows shorter than q_len
  are flagged;
* the split-K merge through pa_merge of two half-pool calls equals the
  single call (the context-parallel shard-and-merge plan, on one GPU).
"""
import numpy as np
import pytest
import torch

from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import compare, oracle_rows, run

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = {"bf16": "bf16_skewed_b256_l16_128k_d256", "int8": "int8_b32_l1k_32k_d256",
         "nvfp4": "nvfp4_b4_l262k_d256", "fp8": "fp8_b32_l1k_32k_d256"}
VERIFY_NAMES = {"nvfp4": "nvfp4_verify_q8_b4_ctx64k_d256", "int8": "int8_b32_l1k_32k_d256",
                "fp8": "fp8_verify_q8_b4_ctx64k_d256"}
# (dtype, kernel): 1 = CUDA-core kernel, 2 = tensor-core kernel
DK = [("bf16", 1), ("bf16", 2), ("int8", 1), ("int8", 2), ("nvfp4", 1), ("nvfp4", 2), ("fp8", 1),
      ("fp8", 2)]
LENS = [3000, 17, 1, 900, 0, 4099]


@pytest.mark.parametrize("dt,kernel", DK)
def test_block_permutation_bitwise(dt, kernel):
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=LENS)
    wp = W.permute_pool(wl, seed=3)
    a, _ = run(wl, out_fp32=True, kernel=kernel)
    b, _ = run(wp, out_fp32=True, kernel=kernel)
    assert torch.equal(a, b)


@pytest.mark.parametrize("dt,kernel", DK)
def test_determinism_bitwise(dt, kernel):
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=LENS)
    a, la, _ = run(wl, out_fp32=True, return_lse=True, kernel=kernel)
    b, lb, _ = run(wl, out_fp32=True, return_lse=True, kernel=kernel)
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("dt,kernel", DK)
def test_split_settings_agree(dt, kernel):
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=LENS)
    ref, _ = oracle_rows(wl)
    auto, _ = run(wl, out_fp32=True, kernel=kernel)
    single, ws1 = run(wl, out_fp32=True, split_blocks=1 << 20, kernel=kernel)
    tiny, ws2 = run(wl, out_fp32=True, split_blocks=1, kernel=kernel)
    few, _ = run(wl, out_fp32=True, target_items=7, kernel=kernel)
    for o, tag in ((auto, "auto"), (single, "single"), (tiny, "tiny"), (few, "few")):
        compare(o, ref, f"{dt} {tag}")
    assert pa.header(ws1)[3] == 0            # no partial slots when nothing splits
    assert pa.header(ws2)[3] > 0


# the library's item target and shortest partition in auto mode: the plan
# before any rounding
DEFAULT_TARGET, MIN_SPLIT = 1184, 8


@pytest.mark.parametrize("dt", ["int8", "nvfp4"])
def test_equal_lengths_fill_whole_rounds(dt):
    """Equal-length sequences: the planner grows the partitions until the
    items fill whole rounds of the decode kernel's resident CTAs (no more
    rounds than the unrounded plan fills completely, each as full as the
    partition granularity allows); one sequence a block shorter keeps the
    unrounded plan.  Results stay those of the oracle."""
    L = 32768
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=[L] * 4)
    o, ws = run(wl, out_fp32=True)
    _, n_items, split, _, res = pa.header(ws)
    per = wl.B * wl.Hkv                        # items per partition index
    nb = L // 16
    w0 = max(MIN_SPLIT, -(-nb * per // DEFAULT_TARGET))
    items0 = per * -(-nb // w0)
    assert res > 0 and items0 > res, (res, items0)
    assert n_items == per * -(-nb // split)
    assert n_items <= items0 // res * res, (n_items, items0, res)
    rounds = -(-n_items // res)
    assert rounds * res - per < n_items, (n_items, rounds, res, per)
    ref, _ = oracle_rows(wl, bs=[0, 3])
    compare(o[[0, 3]], ref, f"{dt} rounded plan")

    wl2 = W.make_workload(NAMES[dt], device=DEV, seq_lens=[L] * 3 + [L - 16])
    _, ws2 = run(wl2, out_fp32=True)
    h2 = pa.header(ws2)
    assert h2[4] == 0
    assert h2[2] == max(MIN_SPLIT, -(-(4 * nb - 1) * wl.Hkv // DEFAULT_TARGET))


def test_padded_rows_zero_and_neg_inf():
    wl = W.make_workload(NAMES["int8"], device=DEV, seq_lens=[0, 40, 0, 0])
    o, lse, ws = run(wl, out_fp32=True, return_lse=True)
    assert not o[0].any() and not o[2].any() and not o[3].any()
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[3]).all()
    assert torch.isfinite(lse[1]).all()
    assert pa.read_error(ws) == 0


@pytest.mark.parametrize("dt,kernel", DK)
def test_bad_block_id_is_skipped_and_flagged(dt, kernel):
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=[400, 50])
    NB = wl.num_blocks
    bad = wl.block_tables.clone()
    bad[0, 3] = -5            # a middle block of sequence 0
    bad[1, 1] = NB + 7        # a block past the end of the pool
    wl_bad = W.Workload(**{**wl.__dict__, "block_tables": bad})
    o, ws = run(wl_bad, out_fp32=True, kernel=kernel)
    torch.cuda.synchronize()
    assert pa.read_error(ws) & pa.PA_ERRF_BAD_BLOCK_ID
    # expected: attention over the keys without those blocks (decode has no
    # positions, so removing a block and shortening the sequence is the same)
    tab = wl.block_tables.clone()
    tab[0, 3:-1] = wl.block_tables[0, 4:].clone()
    tab[1, 1:-1] = wl.block_tables[1, 2:].clone()
    exp_wl = W.Workload(**{**wl.__dict__, "block_tables": tab,
                           "seq_lens": torch.tensor([400 - 16, 50 - 16], dtype=torch.int32,
                                                    device=DEV)})
    ref, _ = oracle_rows(exp_wl)
    compare(o, ref, "bad block skipped")


def test_length_over_capacity_clamped_and_flagged():
    wl = W.make_workload(NAMES["bf16"], device=DEV, seq_lens=[64, 20])
    over = W.Workload(**{**wl.__dict__, "seq_lens": torch.tensor([64 + 16 * 9, 20],
                                                                 dtype=torch.int32, device=DEV)})
    o, ws = run(over, out_fp32=True)
    torch.cuda.synchronize()
    assert pa.read_error(ws) & pa.PA_ERRF_LEN_OVER_CAPACITY
    ref, _ = oracle_rows(wl)       # capacity is 4 blocks = 64 keys
    compare(o, ref, "clamped")


def test_verify_row_shorter_than_q_len_flagged():
    wl = W.make_workload("nvfp4_verify_q8_b4_ctx64k_d256", device=DEV, seq_lens=[100, 5])
    o, ws = run(wl, "verify", out_fp32=True)
    torch.cuda.synchronize()
    assert pa.read_error(ws) & pa.PA_ERRF_LEN_LT_QLEN


def test_two_shards_merged_equal_single_call():
    """Context-parallel plan on one GPU: the blocks of every sequence are
    split between two calls (each sees half of the table), each returns
    fp32 output + LSE, and pa_merge combines them."""
    wl = W.make_workload(NAMES["bf16"], device=DEV, seq_lens=[3000, 1000, 17])
    lens = wl.seq_lens.cpu()
    nblk = (lens + 15) // 16
    half = nblk // 2
    B, stride = wl.block_tables.shape
    t1 = torch.full_like(wl.block_tables, -1)
    t2 = torch.full_like(wl.block_tables, -1)
    l1 = torch.zeros(B, dtype=torch.int32)
    l2 = torch.zeros(B, dtype=torch.int32)
    for b in range(B):
        h = int(half[b])
        t1[b, :h] = wl.block_tables[b, :h]
        l1[b] = h * 16
        t2[b, : int(nblk[b]) - h] = wl.block_tables[b, h: int(nblk[b])]
        l2[b] = int(lens[b]) - h * 16
    parts = []
    for t, l in ((t1, l1), (t2, l2)):
        w = W.Workload(**{**wl.__dict__, "block_tables": t, "seq_lens": l.to(DEV)})
        o, lse, _ = run(w, out_fp32=True, return_lse=True)
        parts.append((o, lse))
    po = torch.stack([p[0].reshape(-1, wl.D) for p in parts])
    pl = torch.stack([p[1].reshape(-1) for p in parts])
    merged = pa.merge(po.contiguous(), pl.contiguous(), out_fp32=True)
    full, _ = run(wl, out_fp32=True)
    np.testing.assert_allclose(merged.cpu().numpy(), full.reshape(-1, wl.D).cpu().numpy(),
                               atol=2e-5, rtol=0)


@pytest.mark.parametrize("kernel", [2, 4])
@pytest.mark.parametrize("dt", ["nvfp4", "int8", "fp8"])
def test_dense_verify_invariants(dt, kernel):
    """Dense-tile verify (mma.sync kernel 2, tcgen05 kernel 4): bitwise
    block-permutation invariance and determinism; forced single / tiny
    partitions agree with the oracle; a bad block id is skipped and
    flagged."""
    if kernel == 4 and dt == "int8":
        pytest.skip("the tcgen05 verify kernel takes NVFP4 and FP8")
    wl = W.make_workload(VERIFY_NAMES[dt], device=DEV, seq_lens=[1500, 8, 300], Q=8)
    a, la, ws = run(wl, "verify", out_fp32=True, return_lse=True, kernel=kernel)
    b, lb, _ = run(wl, "verify", out_fp32=True, return_lse=True, kernel=kernel)
    assert torch.equal(a, b) and torch.equal(la, lb)
    c, _ = run(W.permute_pool(wl, seed=5), "verify", out_fp32=True, kernel=kernel)
    assert torch.equal(a, c)
    ref, _ = oracle_rows(wl)
    for kw in (dict(split_blocks=1 << 20), dict(split_blocks=1), dict(target_items=5)):
        o, _ = run(wl, "verify", out_fp32=True, kernel=kernel, **kw)
        compare(o, ref, f"dense verify {dt} {kw}")
    bad = wl.block_tables.clone()
    bad[0, 7] = -1
    o, ws = run(W.Workload(**{**wl.__dict__, "block_tables": bad}), "verify", out_fp32=True,
                kernel=kernel)
    torch.cuda.synchronize()
    assert pa.read_error(ws) & pa.PA_ERRF_BAD_BLOCK_ID
    assert torch.isfinite(o).all()
