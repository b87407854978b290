"""Pins for the oracle's block-sparse decode against things other than
itself ("vLLM-SM70", "Known limitations": sparse-decode selection over
per-block mean keys, 64-token blocks).

* block means against numpy means of the (separately pinned) gathered keys;
* selection against a numpy brute force (library sort), ties to the lower
  index, a block aligned with the query is chosen;
* sparse attention with every block selected equals dense attention, and
  with fewer blocks equals a numpy softmax over the selected tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_07_gb300 import workloads as W

SB = 64
NAMES = {"bf16": "bf16_skewed_b256_l16_128k_d256", "int8": "int8_b32_l1k_32k_d256",
         "fp8": "fp8_b32_l1k_32k_d256", "nvfp4": "nvfp4_b4_l262k_d256"}
LENS = [300, 64, 1, 130, 257]


def _setup(dt, lens=LENS, Hq=None, Hkv=None, D=None):
    kw = {k: v for k, v in dict(Hq=Hq, Hkv=Hkv, D=D).items() if v is not None}
    wl = W.make_workload(NAMES[dt], seq_lens=lens, **kw)
    h = W.host_arrays(wl)
    cache = oracle.HostCache.from_host_arrays(h, wl.dtype, wl.k_global, wl.v_global)
    return wl, h, cache


def _nsb(lens):
    return np.array([(L + SB - 1) // SB for L in lens], np.int32)


@pytest.mark.parametrize("dt", ["int8", "nvfp4"])
def test_block_means_match_numpy_mean_of_gathered_keys(dt):
    wl, h, cache = _setup(dt, Hq=8, Hkv=2, D=128)
    nsb = _nsb(LENS)
    M = int(nsb.max())
    means = oracle.block_means(cache, h["block_tables"], h["seq_lens"], SB, M)
    k, _ = oracle.gather(cache, h["block_tables"], h["seq_lens"], max(LENS))
    for b, L in enumerate(LENS):
        for j in range(M):
            lo, hi = j * SB, min((j + 1) * SB, L)
            ref = k[b, :, lo:hi].astype(np.float64).mean(axis=1) if lo < hi else 0.0
            np.testing.assert_allclose(means[b, j], ref, rtol=0, atol=1e-12)


def _numpy_select(q, means, nsb, k, Hkv):
    B, _, Hq, D = q.shape
    G = Hq // Hkv
    qf = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).double().numpy()[:, 0]
    qf = qf.reshape(B, Hkv, G, D)
    scores = np.einsum("bhgd,bjhd->bhgj", qf, means).max(axis=2)      # [B, Hkv, max_nsb]
    sel = np.full((B, Hkv, k), -1, np.int32)
    for b in range(B):
        for h in range(Hkv):
            order = np.lexsort((np.arange(nsb[b]), -scores[b, h, : nsb[b]]))[:k]
            chosen = np.sort(order)
            sel[b, h, : len(chosen)] = chosen
    return scores, sel


def test_select_matches_numpy_brute_force():
    rng = np.random.default_rng(5)
    B, Hkv, G, D, M = 5, 3, 4, 32, 40
    q = torch.randn(B, 1, Hkv * G, D, generator=torch.Generator().manual_seed(1))
    qb = q.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    means = rng.standard_normal((B, M, Hkv, D))
    nsb = np.array([40, 7, 0, 1, 23], np.int32)
    for k in (1, 5, 8, 64):
        scores, sel = oracle.sparse_select(qb, Hkv, means, nsb, k)
        ref_s, ref_sel = _numpy_select(qb, means, nsb, k, Hkv)
        for b in range(B):
            n = nsb[b]
            np.testing.assert_allclose(scores[b, :, :n], ref_s[b, :, :n], rtol=1e-12, atol=1e-12)
            assert np.all(np.isneginf(scores[b, :, n:]))
        assert np.array_equal(sel, ref_sel), k


def test_select_ties_go_to_the_lower_index():
    B, Hkv, G, D, M = 1, 1, 2, 8, 6
    q = np.zeros((B, 1, Hkv * G, D), np.float32)
    q[0, 0, :, 0] = 1.0
    qb = torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    means = np.zeros((B, M, Hkv, D))
    means[0, [1, 3, 4], 0, 0] = 2.0        # three blocks tie for the top score
    means[0, 5, 0, 0] = 1.0
    nsb = np.array([M], np.int32)
    _, sel = oracle.sparse_select(qb, Hkv, means, nsb, 1)
    assert sel[0, 0].tolist() == [1]
    _, sel = oracle.sparse_select(qb, Hkv, means, nsb, 2)
    assert sel[0, 0].tolist() == [1, 3]
    _, sel = oracle.sparse_select(qb, Hkv, means, nsb, 4)
    assert sel[0, 0].tolist() == [1, 3, 4, 5]


def test_block_aligned_with_the_query_is_selected():
    wl, h, cache = _setup("bf16", lens=[640], Hq=4, Hkv=1, D=128)
    # keys of sparse block 6 all equal to e_0 * 4; the query points along e_0
    k = h["k_cache"]
    tab = h["block_tables"][0]
    for t in range(6 * SB, 7 * SB):
        row = np.zeros(128, np.float32)
        row[0] = 4.0
        k[tab[t // 16], 0, t % 16] = torch.from_numpy(row).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
    cache = oracle.HostCache.from_host_arrays(h, wl.dtype)
    q = np.zeros((1, 1, 4, 128), np.float32)
    q[..., 0] = 3.0
    qb = torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    means = oracle.block_means(cache, h["block_tables"], h["seq_lens"], SB, 10)
    _, sel = oracle.sparse_select(qb, 1, means, np.array([10], np.int32), 1)
    assert sel[0, 0].tolist() == [6]


@pytest.mark.parametrize("dt", ["bf16", "int8", "fp8", "nvfp4"])
def test_sparse_attention_with_every_block_equals_dense(dt):
    wl, h, cache = _setup(dt)
    nsb = _nsb(LENS)
    M = int(nsb.max())
    sel = np.full((wl.B, wl.Hkv, M), -1, np.int32)
    for b in range(wl.B):
        sel[b, :, : nsb[b]] = np.arange(nsb[b])
    o, lse = oracle.attend_sparse(cache, h["q"], h["block_tables"], h["seq_lens"], sel, SB,
                                  wl.softmax_scale)
    ref_o, ref_l = oracle.attend(cache, h["q"], h["block_tables"], h["seq_lens"],
                                 wl.softmax_scale, nthreads=1)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dt", ["int8", "nvfp4"])
def test_sparse_attention_matches_numpy_softmax_over_selected_tokens(dt):
    wl, h, cache = _setup(dt, Hq=6, Hkv=2, D=128)
    nsb = _nsb(LENS)
    M = int(nsb.max())
    rng = np.random.default_rng(2)
    k_sel = 2
    sel = np.full((wl.B, wl.Hkv, k_sel), -1, np.int32)
    for b in range(wl.B):
        for hh in range(wl.Hkv):
            c = np.sort(rng.permutation(nsb[b])[:k_sel])
            sel[b, hh, : len(c)] = c
    o, lse = oracle.attend_sparse(cache, h["q"], h["block_tables"], h["seq_lens"], sel, SB,
                                  wl.softmax_scale)
    kk, vv = oracle.gather(cache, h["block_tables"], h["seq_lens"], max(LENS))
    qf = torch.from_numpy(h["q"].view(np.int16)).view(torch.bfloat16).double().numpy()
    G = wl.Hq // wl.Hkv
    for b, L in enumerate(LENS):
        for hh in range(wl.Hkv):
            toks = [t for j in sel[b, hh] if j >= 0 for t in range(j * SB, min((j + 1) * SB, L))]
            for g in range(G):
                qh = hh * G + g
                s = wl.softmax_scale * kk[b, hh, toks].astype(np.float64) @ qf[b, 0, qh]
                w = np.exp(s - s.max())
                ref = (w[:, None] * vv[b, hh, toks].astype(np.float64)).sum(0) / w.sum()
                np.testing.assert_allclose(o[b, 0, qh], ref, rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[b, 0, qh], s.max() + np.log(w.sum()), atol=1e-12)
