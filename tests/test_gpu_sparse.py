"""GPU parity of block-sparse decode (pa_block_means, pa_decode_sparse
through the C ABI) against the oracle.

* mean keys of every sparse block, and a refresh of only the last one;
* the selection: top_k by score, ties to the lower index -- several answers
  are right when two scores are within rounding, so the kernel's choice is
  checked for validity against the oracle's fp64 scores (and must equal the
  oracle's choice wherever the k-th and (k+1)-th scores are apart);
* the attention over the kernel's selection against the oracle's exact
  attention over the same blocks; with top_k >= every block it is dense
  attention;
* the full-size workload, sampled sequences.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import compact_host, compare, compare_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"
SB = 64
NAMES = {"bf16": "bf16_skewed_b256_l16_128k_d256", "int8": "int8_sparse_b8_l262k_k256_d256",
         "fp8": "fp8_b32_l1k_32k_d256", "nvfp4": "nvfp4_b4_l262k_d256"}
LENS = [3000, 700, 64, 1, 0, 1000, 129]


def _nsb(lens):
    return [(int(L) + SB - 1) // SB for L in lens]


def _means(wl, max_nsb, first=None, count=0, means=None):
    kv = pa.KvCache.from_workload(wl)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    m = pa.block_means(kv, wl.block_tables, wl.seq_lens, SB, max_nsb, first=first, count=count,
                       means=means,
                       workspace=ws)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    return m


def check_selection(sel, scores, nsb, k, what):
    """sel int32 [B, H, k] from the kernel; scores fp64 [B, H, M] from the oracle."""
    for b in range(sel.shape[0]):
        n = min(k, nsb[b])
        for h in range(sel.shape[1]):
            got = sel[b, h]
            chosen = got[:n]
            assert (got[n:] == -1).all(), what
            assert (np.diff(chosen) > 0).all() and (chosen >= 0).all() and (chosen < nsb[b]).all()
            if n == nsb[b]:
                continue
            s = scores[b, h, : nsb[b]]
            rest = np.setdiff1d(np.arange(nsb[b]), chosen)
            tol = 1e-4 * (1.0 + np.abs(s).max())
            assert s[chosen].min() >= s[rest].max() - tol, f"{what}: b {b} h {h}"
            order = np.lexsort((np.arange(nsb[b]), -s))
            if s[order[n - 1]] - s[order[n]] > tol:      # a clear gap: the choice is unique
                assert np.array_equal(chosen, np.sort(order[:n])), f"{what}: b {b} h {h}"


@pytest.mark.parametrize("dt", ["bf16", "int8", "fp8", "nvfp4"])
def test_block_means_and_last_block_refresh(dt):
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=LENS)
    nsb = _nsb(LENS)
    M = max(nsb)
    m = _means(wl, M).cpu().numpy()
    cache, tab, lens, _ = compact_host(wl, list(range(wl.B)))
    ref = oracle.block_means(cache, tab, lens, SB, M)
    for b in range(wl.B):
        np.testing.assert_allclose(m[b, : nsb[b]], ref[b, : nsb[b]], rtol=1e-5, atol=1e-6)
    # refresh of each sequence's last sparse block only: the rest is untouched
    first = torch.tensor([max(n - 1, 0) for n in nsb], dtype=torch.int32, device=DEV)
    sentinel = torch.full_like(torch.from_numpy(m), float("nan")).to(DEV)
    m2 = _means(wl, M, first=first, count=1, means=sentinel).cpu().numpy()
    for b in range(wl.B):
        if nsb[b] == 0:
            continue
        assert np.isnan(m2[b, : nsb[b] - 1]).all()
        np.testing.assert_allclose(m2[b, nsb[b] - 1], ref[b, nsb[b] - 1], rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("top_k", [1, 3, 20, 100])
@pytest.mark.parametrize("dt", ["bf16", "int8", "fp8", "nvfp4"])
def test_sparse_decode_parity(dt, top_k):
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=LENS)
    nsb = _nsb(LENS)
    M = max(nsb)
    means = _means(wl, M)
    kv = pa.KvCache.from_workload(wl)
    o, lse, sel, ws = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale,
                                       means, SB, top_k, out_fp32=True, return_lse=True,
                                       return_selected=True)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    sel = sel.cpu().numpy()
    cache, tab, lens, qb = compact_host(wl, list(range(wl.B)))
    ref_means = oracle.block_means(cache, tab, lens, SB, M)
    scores, _ = oracle.sparse_select(qb, wl.Hkv, ref_means, np.array(nsb, np.int32), top_k)
    check_selection(sel, scores, nsb, top_k, f"{dt} k={top_k}")
    ref_o, ref_l = oracle.attend_sparse(cache, qb, tab, lens, sel, SB, wl.softmax_scale)
    compare(o, ref_o, f"sparse {dt} k={top_k}")
    compare_lse(lse, ref_l, f"sparse {dt} k={top_k}")
    if top_k >= M:   # every block: dense attention
        dense_o, dense_l = oracle.attend(cache, qb, tab, lens, wl.softmax_scale)
        compare(o, dense_o, f"sparse=dense {dt}")
        compare_lse(lse, dense_l, f"sparse=dense {dt}")


def test_full_size_sparse_sampled():
    name = "int8_sparse_b8_l262k_k256_d256"
    spec = W.spec(name)
    wl = W.make_workload(name, device=DEV)
    M = (wl.max_seq_len() + SB - 1) // SB
    means = _means(wl, M)
    kv = pa.KvCache.from_workload(wl)
    o, lse, sel, ws = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale,
                                       means, SB, spec["top_k"], out_fp32=True, return_lse=True,
                                       return_selected=True)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    for b in (0, wl.B - 1):
        cache, tab, lens, qb = compact_host(wl, [b])
        nsb = _nsb(lens)
        ref_means = oracle.block_means(cache, tab, lens, SB, M)
        np.testing.assert_allclose(means[b].cpu().numpy(), ref_means[0], rtol=1e-5, atol=1e-6)
        scores, _ = oracle.sparse_select(qb, wl.Hkv, ref_means, np.array(nsb, np.int32),
                                         spec["top_k"])
        s = sel[b:b + 1].cpu().numpy()
        check_selection(s, scores, nsb, spec["top_k"], f"full b {b}")
        ref_o, ref_l = oracle.attend_sparse(cache, qb, tab, lens, s, SB, wl.softmax_scale)
        compare(o[b:b + 1], ref_o, f"full sparse b {b}")
        compare_lse(lse[b:b + 1], ref_l, f"full sparse b {b}")


def test_selection_ties_go_to_the_lower_index():
    """Three sparse blocks with the same mean key score exactly alike; the
    top two must be the two lowest indices."""
    wl = W.make_workload(NAMES["int8"], device=DEV, seq_lens=[640, 640])
    M = 10
    g = torch.Generator(device="cpu").manual_seed(3)
    means = (torch.randn(wl.B, M, wl.Hkv, wl.D, generator=g) * 0.01).to(DEV)
    G = wl.Hq // wl.Hkv
    for h in range(wl.Hkv):
        direction = wl.q[:, 0, h * G].float()                # [B, D]
        for j in (2, 5, 7):
            means[:, j, h] = 10.0 * direction
    kv = pa.KvCache.from_workload(wl)
    _, sel, _ = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale,
                                 means.contiguous(), SB, 2, return_selected=True)
    assert (sel.cpu() == torch.tensor([2, 5], dtype=torch.int32)).all()
    _, sel, _ = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale,
                                 means.contiguous(), SB, 3, return_selected=True)
    assert (sel.cpu() == torch.tensor([2, 5, 7], dtype=torch.int32)).all()


def test_selection_when_every_score_is_equal():
    """Every sparse block has the same mean key, so every score is the same
    number: the top k are blocks 0 .. k - 1 (ties to the lower index), for a
    k below, at and above the number of blocks."""
    wl = W.make_workload(NAMES["int8"], device=DEV, seq_lens=[1280, 1000])
    M = 20
    g = torch.Generator(device="cpu").manual_seed(5)
    row = torch.randn(wl.D, generator=g)
    means = row.expand(wl.B, M, wl.Hkv, wl.D).contiguous().to(DEV)
    kv = pa.KvCache.from_workload(wl)
    nsb = _nsb([1280, 1000])
    for k in (1, 7, 16, 20, 25):
        _, sel, _ = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale,
                                     means, SB, k, return_selected=True)
        sel = sel.cpu().numpy()
        for b in range(wl.B):
            n = min(k, nsb[b])
            for h in range(wl.Hkv):
                assert np.array_equal(sel[b, h, :n], np.arange(n)), (k, b, h)
                assert (sel[b, h, n:] == -1).all(), (k, b, h)


def test_selection_with_negative_and_mixed_sign_scores():
    """Scores of both signs and all negative: the order of the sign-folded
    keys must be the order of the scores."""
    wl = W.make_workload(NAMES["int8"], device=DEV, seq_lens=[1280, 1280])
    M = 20
    G = wl.Hq // wl.Hkv
    g = torch.Generator(device="cpu").manual_seed(9)
    coef = torch.randn(wl.B, M, wl.Hkv, generator=g)
    coef[1] = -coef[1].abs() - 0.5                          # sequence 1: every score negative
    kv = pa.KvCache.from_workload(wl)
    means = torch.empty(wl.B, M, wl.Hkv, wl.D)
    qf = wl.q[:, 0].float().cpu()                            # [B, Hq, D]
    for b in range(wl.B):
        for h in range(wl.Hkv):
            # nearly along every head of the group, so each head's dot has
            # the sign of coef and so has the score (their max)
            direction = qf[b, h * G:(h + 1) * G].sum(0)
            direction = direction / direction.norm()
            means[b, :, h] = coef[b, :, h, None] * direction
    means = means.to(DEV).contiguous()
    k = 6
    _, sel, _ = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale,
                                 means, SB, k, return_selected=True)
    _, _, _, qb = compact_host(wl, list(range(wl.B)))
    scores, _ = oracle.sparse_select(qb, wl.Hkv, means.cpu().numpy().astype(np.float64),
                                     np.array(_nsb([1280, 1280]), np.int32), k)
    assert (scores[1, :, :20] < 0).all() and (scores[0, :, :20] > 0).any()
    check_selection(sel.cpu().numpy(), scores, _nsb([1280, 1280]), k, "mixed signs")


@pytest.mark.parametrize("dt,Hq,Hkv,D", [("int8", 8, 2, 128), ("nvfp4", 8, 4, 128),
                                         ("bf16", 8, 8, 256)])
def test_sparse_other_head_shapes(dt, Hq, Hkv, D):
    """Head dim 128 (half the float4 per lane in the score kernel) and group
    sizes 4, 2 and 1."""
    lens = [2000, 65, 640, 1]
    wl = W.make_workload(NAMES[dt], device=DEV, seq_lens=lens, Hq=Hq, Hkv=Hkv, D=D)
    nsb = _nsb(lens)
    M = max(nsb)
    means = _means(wl, M)
    kv = pa.KvCache.from_workload(wl)
    top_k = 5
    o, lse, sel, ws = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale,
                                       means, SB, top_k, out_fp32=True, return_lse=True,
                                       return_selected=True)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    sel = sel.cpu().numpy()
    cache, tab, lens_h, qb = compact_host(wl, list(range(wl.B)))
    ref_means = oracle.block_means(cache, tab, lens_h, SB, M)
    scores, _ = oracle.sparse_select(qb, wl.Hkv, ref_means, np.array(nsb, np.int32), top_k)
    check_selection(sel, scores, nsb, top_k, f"{dt} Hq={Hq} Hkv={Hkv} D={D}")
    ref_o, ref_l = oracle.attend_sparse(cache, qb, tab, lens_h, sel, SB, wl.softmax_scale)
    compare(o, ref_o, f"sparse {dt} D={D}")
    compare_lse(lse, ref_l, f"sparse {dt} D={D}")
