"""Pins for the fp64 oracle against things other than itself.

* format decoders: exhaustive comparison with library decoders (torch bf16
  and float8_e4m3fn, numpy float16) and the OCP E2M1 value table;
* gather + dequant: bit-exact against an independent NumPy decode that uses
  those library decoders and its own nibble unpacking;
* attention: closed forms (seq_len 1, equal scores, constant V, hand-derived
  golden cases), a NumPy fp64 dense brute force on tiny inputs, invariants
  (physical-block permutation, split + merge = unsplit, verify = per-query
  decode with truncated lengths), padded rows.

Definition followed: PagedAttention decode (Kwon et al., cited on "vLLM
Fork with focus on GB10 Homelabs", "About"), exact softmax ("vLLM-SM70",
"Why"), NVFP4 / int8 KV formats ("vLLM All-NVFP4 DFlash2 for Blackwell",
"What makes this stack different"; "vLLM-SM70", "Why").
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_07_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# OCP Microscaling spec, FP4 E2M1 magnitudes for codes 0..7
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ----------------------------------------------------------------- formats

def test_bf16_decoder_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_fp16_decoder_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_value(int(b)) for b in bits])
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_e4m3_decoder_exhaustive():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    # anchors of the format: max 448, min normal 2^-6, min subnormal 2^-9
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x38) == 1.0
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_e2m1_decoder_table():
    for c in range(16):
        mag = E2M1_TABLE[c & 7]
        want = -mag if c & 8 else mag
        assert oracle.e2m1_value(c) == want, c


# ---------------------------------------------------- encoders (inputs side)

def test_e4m3_encoder_roundtrip_every_finite_code():
    codes = torch.arange(0, 127, dtype=torch.int32)
    vals = torch.tensor([oracle.e4m3_value(int(c)) for c in codes], dtype=torch.float32)
    enc = W.e4m3_encode_rne_satfinite(vals)
    assert torch.equal(enc.to(torch.int32), codes)


def test_e4m3_encoder_matches_library_cast():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.rand(20000, generator=g) * 447.0,
                   torch.rand(20000, generator=g) * 2.0 ** -5,
                   torch.tensor([0.0, 2.0 ** -10, 3 * 2.0 ** -10, 232.0, 17.0, 447.9])])
    ours = W.e4m3_encode_rne_satfinite(x)
    lib = x.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(ours, lib)
    assert int(W.e4m3_encode_rne_satfinite(torch.tensor([448.0, 1e6]))[1]) == 0x7E


def test_e2m1_encoder_grid_and_ties():
    grid = torch.tensor(E2M1_TABLE)
    assert torch.equal(W.e2m1_encode_rne(grid), torch.arange(8, dtype=torch.uint8))
    assert torch.equal(W.e2m1_encode_rne(-grid[1:]), torch.arange(9, 16, dtype=torch.uint8))
    ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert W.e2m1_encode_rne(ties).tolist() == [0, 2, 2, 4, 4, 6, 6]
    assert W.e2m1_encode_rne(torch.tensor([7.0, 100.0])).tolist() == [7, 7]
    # rounding error at most half a grid step
    y = torch.rand(10000, generator=torch.Generator().manual_seed(1)) * 6.0
    dec = torch.tensor(E2M1_TABLE)[W.e2m1_encode_rne(y).long()]
    steps = torch.tensor([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0, 2.0])
    assert bool(((dec - y).abs() <= steps[W.e2m1_encode_rne(y).long()] / 2 + 1e-7).all())


def test_int8_quantiser_bounds():
    x = torch.randn(64, 256, generator=torch.Generator().manual_seed(2))
    c, s16 = W.quantize_int8_rows(x)
    assert int(c.abs().max()) <= 127
    s = s16.float().unsqueeze(-1)
    err = (c.float() * s - x).abs()
    assert bool((err <= s * 0.5 + 1e-6 + (x.abs() - 127 * s).clamp(min=0)).all())


def test_fp8_quantiser_on_grid_roundtrip_and_sign():
    g = 0.25
    codes = torch.arange(0, 256, dtype=torch.int64)
    codes = codes[(codes & 0x7F) != 0x7F]            # no NaN
    vals = torch.from_numpy(codes.to(torch.uint8).numpy()).view(torch.float8_e4m3fn).float() * g
    enc = W.quantize_fp8(vals, g)
    dec = torch.from_numpy(enc.numpy()).view(torch.float8_e4m3fn).float() * g
    assert torch.equal(dec, vals)                   # +-0 compare equal
    big = W.quantize_fp8(torch.tensor([1e9, -1e9]), g)
    assert big.tolist() == [0x7E, 0xFE]


def test_nvfp4_quantiser_on_grid_roundtrip():
    # values exactly e2m1 * e4m3(s) * g with the block amax = 6 s g round-trip
    g = 0.5
    gen = torch.Generator().manual_seed(5)
    s_codes = torch.randint(0x30, 0x50, (32,), generator=gen)
    s_vals = torch.tensor([oracle.e4m3_value(int(c)) for c in s_codes], dtype=torch.float32)
    codes = torch.randint(0, 16, (32, 16), generator=gen)
    codes[:, 0] = 7                                   # amax = 6 in every block
    mags = torch.tensor(E2M1_TABLE)[(codes & 7)]
    vals = torch.where(codes >= 8, -mags, mags) * s_vals.unsqueeze(1) * g
    packed, sc = W.quantize_nvfp4_rows(vals.reshape(2, 256), g)
    assert torch.equal(sc.flatten().long(), s_codes)
    lo, hi = (packed & 0xF).long(), (packed >> 4).long()
    un = torch.stack([lo, hi], dim=-1).reshape(32, 16)
    # +0 / -0 both decode to zero; compare magnitudes and nonzero signs
    same = (un == codes) | (((un & 7) == 0) & ((codes & 7) == 0))
    assert bool(same.all())


# ------------------------------------------------ independent NumPy decode

def np_decode(wl, which):
    """fp32 [NB, Hkv, 16, D] decoded with library decoders (not the oracle)."""
    h = W.host_arrays(wl)
    data = h["k_cache" if which == 0 else "v_cache"]
    sc = h["k_scale" if which == 0 else "v_scale"]
    if wl.dtype == "bf16":
        return torch.from_numpy(data.view(np.int16)).view(torch.bfloat16).float().numpy()
    if wl.dtype == "int8":
        with np.errstate(invalid="ignore", over="ignore"):   # poisoned slots
            return data.astype(np.float32) * sc.view(np.float16).astype(np.float32)[..., None]
    if wl.dtype == "fp8":
        e = torch.from_numpy(data).view(torch.float8_e4m3fn).float().numpy()
        g = np.float32(wl.k_global if which == 0 else wl.v_global)
        with np.errstate(invalid="ignore"):
            return e * g
    lo = (data & 0xF).astype(np.int64)
    hi = (data >> 4).astype(np.int64)
    codes = np.stack([lo, hi], axis=-1).reshape(*data.shape[:-1], data.shape[-1] * 2)
    mag = np.array(E2M1_TABLE)[codes & 7]
    e2m1 = np.where(codes >= 8, -mag, mag)
    s = torch.from_numpy(sc).view(torch.float8_e4m3fn).double().numpy()
    s = np.repeat(s, 16, axis=-1)
    g = np.float32(wl.k_global if which == 0 else wl.v_global)
    return (e2m1 * s).astype(np.float32) * g


def np_dense_kv(wl):
    """per (b, kvh): dense K, V [L, D] fp64 for valid tokens."""
    Kd, Vd = np_decode(wl, 0), np_decode(wl, 1)
    tab = wl.block_tables.numpy()
    out = []
    for b, L in enumerate(wl.seq_lens.tolist()):
        t = np.arange(L)
        blk = tab[b, t // 16]
        out.append((Kd[blk, :, t % 16, :].astype(np.float64), Vd[blk, :, t % 16, :].astype(np.float64)))
    return out


def brute_force(wl):
    qf = wl.q.double().numpy()
    G = wl.Hq // wl.Hkv
    out = np.zeros((wl.B, wl.Q, wl.Hq, wl.D))
    lse = np.full((wl.B, wl.Q, wl.Hq), -np.inf)
    for b, (K, V) in enumerate(np_dense_kv(wl)):
        L = int(wl.seq_lens[b])
        for i in range(wl.Q):
            n = L - wl.Q + 1 + i if L else 0
            for h in range(wl.Hq):
                if n <= 0:
                    continue
                s = wl.softmax_scale * (K[:n, h // G, :] @ qf[b, i, h])
                m = s.max()
                w = np.exp(s - m)
                out[b, i, h] = (w @ V[:n, h // G, :]) / w.sum()
                lse[b, i, h] = m + np.log(w.sum())
    return out, lse


SMALL = {
    "bf16": ("bf16_b1_l1000_d128", [37, 1, 64, 16]),
    "int8": ("int8_b32_l1k_32k_d256", [33, 17, 1, 50]),
    "nvfp4": ("nvfp4_b4_l262k_d256", [40, 16, 1, 29]),
    "fp8": ("fp8_b32_l1k_32k_d256", [21, 1, 48, 17]),
}
ALL = ["bf16", "int8", "nvfp4", "fp8"]


@pytest.mark.parametrize("dt", ALL)
def test_gather_bit_exact_vs_numpy_decode(dt):
    name, lens = SMALL[dt]
    wl = W.make_workload(name, seq_lens=lens)
    h = W.host_arrays(wl)
    cache = oracle.HostCache.from_host_arrays(h, wl.dtype, wl.k_global, wl.v_global)
    maxl = max(lens) + 3
    k, v = oracle.gather(cache, h["block_tables"], h["seq_lens"], maxl)
    for b, (K, V) in enumerate(np_dense_kv(wl)):
        L = lens[b]
        assert np.array_equal(k[b, :, :L, :], K.transpose(1, 0, 2).astype(np.float32))
        assert np.array_equal(v[b, :, :L, :], V.transpose(1, 0, 2).astype(np.float32))
        assert not k[b, :, L:, :].any() and not v[b, :, L:, :].any()


@pytest.mark.parametrize("dt", ALL)
@pytest.mark.parametrize("Q", [1, 3])
def test_attention_matches_dense_brute_force(dt, Q):
    name, lens = SMALL[dt]
    lens = [max(L, Q) for L in lens]
    wl = W.make_workload(name, seq_lens=lens, Q=Q)
    out, lse = oracle.attend_workload(wl)
    ref_o, ref_l = brute_force(wl)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dt", ALL)
def test_seq_len_one_returns_that_value(dt):
    name, _ = SMALL[dt]
    wl = W.make_workload(name, seq_lens=[1, 1])
    out, lse = oracle.attend_workload(wl)
    V = np_decode(wl, 1)
    G = wl.Hq // wl.Hkv
    for b in range(2):
        blk = int(wl.block_tables[b, 0])
        for h in range(wl.Hq):
            assert np.array_equal(out[b, 0, h], V[blk, h // G, 0].astype(np.float64))
    # single key: lse is the score itself
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("dt", ALL)
def test_zero_query_gives_mean_of_v(dt):
    name, lens = SMALL[dt]
    wl = W.make_workload(name, seq_lens=lens)
    wl.q.zero_()
    out, lse = oracle.attend_workload(wl)
    G = wl.Hq // wl.Hkv
    for b, (_, V) in enumerate(np_dense_kv(wl)):
        L = lens[b]
        for h in range(wl.Hq):
            np.testing.assert_allclose(out[b, 0, h], V[:, h // G, :].mean(axis=0), atol=1e-12)
            assert abs(lse[b, 0, h] - math.log(L)) < 1e-12


def test_constant_v_gives_that_constant():
    wl = W.make_workload("bf16_b1_l1000_d128", seq_lens=[300, 7], kv_values="const_v")
    out, _ = oracle.attend_workload(wl)
    V = np_decode(wl, 1)
    G = wl.Hq // wl.Hkv
    for b in range(2):
        blk = int(wl.block_tables[b, 0])
        for h in range(wl.Hq):
            np.testing.assert_allclose(out[b, 0, h], V[blk, h // G, 0], atol=1e-12)


@pytest.mark.parametrize("dt", ALL)
def test_physical_block_permutation_is_bitwise_invariant(dt):
    name, lens = SMALL[dt]
    wl = W.make_workload(name, seq_lens=lens)
    wp = W.permute_pool(wl, seed=11)
    assert not torch.equal(wl.block_tables, wp.block_tables)
    o1, l1 = oracle.attend_workload(wl)
    o2, l2 = oracle.attend_workload(wp)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("dt", ALL)
def test_split_and_merge_equals_unsplit(dt):
    name, _ = SMALL[dt]
    lens = [200, 97, 16]
    wl = W.make_workload(name, seq_lens=lens)
    full_o, full_l = oracle.attend_workload(wl)
    cuts = [[0, 64, 150, 200], [0, 16, 97, 97], [0, 0, 5, 16]]   # includes an empty part
    parts_o, parts_l = [], []
    for p in range(3):
        kb = [c[p] for c in cuts]
        ke = [c[p + 1] for c in cuts]
        o, l = oracle.attend_workload(wl, key_begin=kb, key_end=ke)
        parts_o.append(o.reshape(-1, wl.D))
        parts_l.append(l.reshape(-1))
    mo, ml = oracle.merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(mo, full_o.reshape(-1, wl.D), atol=1e-12, rtol=0)
    np.testing.assert_allclose(ml, full_l.reshape(-1), atol=1e-12, rtol=0)


def test_verify_equals_truncated_decodes():
    lens = [60, 33]
    Q = 5
    wl = W.make_workload("nvfp4_verify_q8_b4_ctx64k_d256", seq_lens=lens, Q=Q)
    vo, vl = oracle.attend_workload(wl)
    h = W.host_arrays(wl)
    cache = oracle.HostCache.from_host_arrays(h, wl.dtype, wl.k_global, wl.v_global)
    for i in range(Q):
        trunc = np.array([L - Q + 1 + i for L in lens], np.int32)
        o, l = oracle.attend(cache, h["q"][:, i:i + 1], h["block_tables"], trunc, wl.softmax_scale)
        assert np.array_equal(o[:, 0], vo[:, i]) and np.array_equal(l[:, 0], vl[:, i])


def test_padded_rows_give_zero_and_neg_inf():
    wl = W.make_workload("int8_b32_l1k_32k_d256", seq_lens=[0, 20, 0])
    out, lse = oracle.attend_workload(wl)
    assert not out[0].any() and not out[2].any()
    assert np.isneginf(lse[0]).all() and np.isneginf(lse[2]).all()
    assert np.isfinite(lse[1]).all()


def test_merge_ignores_empty_partials_and_handles_all_empty():
    o = np.random.default_rng(0).normal(size=(3, 2, 4))
    l = np.array([[0.5, -np.inf], [-np.inf, -np.inf], [1.5, -np.inf]])
    mo, ml = oracle.merge(o, l)
    w = np.exp(np.array([0.5, 1.5]) - 1.5)
    np.testing.assert_allclose(mo[0], (w[0] * o[0, 0] + w[1] * o[2, 0]) / w.sum(), atol=1e-15)
    assert abs(ml[0] - (1.5 + math.log(w.sum()))) < 1e-15
    assert not mo[1].any() and np.isneginf(ml[1])


def _golden_arrays(case):
    D = case["head_dim"]
    L = case["seq_len"]

    def pad(rows, n):
        a = np.zeros((n, D), np.float32)
        for i, r in enumerate(rows):
            a[i, : len(r)] = r
        return a

    k = pad(case["k"], 16)
    v = pad(case["v"], 16)
    q = pad(case["q"], case["q_len"])
    bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kc = bits(k).reshape(1, 1, 16, D)
    vc = bits(v).reshape(1, 1, 16, D)
    qb = bits(q).reshape(1, case["q_len"], 1, D)
    return kc, vc, qb, L


def test_golden_closed_form_examples():
    with open(os.path.join(GOLDEN, "closed_form_examples.json")) as f:
        cases = json.load(f)["cases"]
    consts = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln7": math.log(7)}
    for case in cases:
        kc, vc, qb, L = _golden_arrays(case)
        cache = oracle.HostCache("bf16", kc, vc)
        out, lse = oracle.attend(cache, qb, np.zeros((1, 1), np.int32), np.array([L], np.int32),
                                 consts[case["scale_expr"]])
        for i, exp_o in enumerate(case["expected_out"]):
            np.testing.assert_allclose(out[0, i, 0, : len(exp_o)], exp_o, atol=1e-14)
            assert not out[0, i, 0, len(exp_o):].any()
            assert abs(lse[0, i, 0] - consts[case["expected_lse_expr"][i]]) < 1e-14
