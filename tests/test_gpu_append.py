"""GPU parity of the KV append (quantise-on-write, pa_append_kv through the
C ABI) against the oracle's append: every byte of the pool -- codes,
scales, and the bytes that must stay untouched -- is compared bit for bit.

* every format at reduced size with padded rows (slot -1) and out-of-range
  slots (skipped, PA_ERRF_BAD_SLOT), head dims 256 and 128;
* rows built on every rounding tie, saturation and signed zero of the
  formats;
* the full-size workload of the benchmark, checked on sampled tokens;
* append then decode: new tokens written at the end of each sequence and
  attended over, against the oracle's append + attention.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import compare, compare_lse, run

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTS = ["bf16", "int8", "fp8", "nvfp4"]


def kv_of(aw, device_arrays):
    k, v, ks, vs = device_arrays
    return pa.KvCache(aw.dtype, k, v, ks, vs, aw.k_global, aw.v_global)


def gpu_append(aw, slots=None, ws=True):
    arrs = [None if t is None else t.clone() for t in
            (aw.k_cache, aw.v_cache, aw.k_scale, aw.v_scale)]
    kv = kv_of(aw, arrs)
    w = torch.zeros(256, dtype=torch.uint8, device=DEV) if ws else None
    pa.append_kv(kv, aw.k_new, aw.v_new, aw.slot_mapping if slots is None else slots, workspace=w)
    torch.cuda.synchronize()
    return arrs, (pa.read_error(w) if ws else 0)


def oracle_append(aw, slots=None):
    h = W.append_host_arrays(aw)
    c = oracle.HostCache(aw.dtype, h["k_cache"], h["v_cache"], h["k_scale"], h["v_scale"],
                         aw.k_global, aw.v_global)
    sm = h["slot_mapping"] if slots is None else slots.cpu().numpy()
    bad = oracle.append(c, h["k_new"], h["v_new"], sm)
    return c.arrays, bad


def as_bits(t):
    if t is None:
        return None
    t = t.cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def assert_pool_equal(gpu_arrays, ref_arrays):
    for name, g, r in zip(("k", "v", "k_scale", "v_scale"), gpu_arrays, ref_arrays):
        if g is None:
            assert r is None
            continue
        gb = as_bits(g)
        if not np.array_equal(gb, r):
            diff = np.argwhere(gb != r)
            raise AssertionError(f"{name}: {len(diff)} bytes differ, first at {diff[0].tolist()}: "
                                 f"gpu {gb[tuple(diff[0])]} oracle {r[tuple(diff[0])]}")


@pytest.mark.parametrize("D", [256, 128])
@pytest.mark.parametrize("dt", DTS)
def test_append_bit_exact_with_padded_and_bad_slots(dt, D):
    aw = W.make_append_workload(f"append_{dt}_t64k_d256", device=DEV, T=1500, D=D)
    slots = aw.slot_mapping.clone()
    slots[7] = -5                          # below -1: skipped, flagged
    slots[400] = aw.num_blocks * 16 + 3    # past the pool: skipped, flagged
    arrs, flags = gpu_append(aw, slots)
    ref, bad = oracle_append(aw, slots)
    assert bad == 2
    assert flags & pa.PA_ERRF_BAD_SLOT
    assert_pool_equal(arrs, ref)


@pytest.mark.parametrize("dt", DTS)
def test_append_without_bad_slots_sets_no_flag(dt):
    aw = W.make_append_workload(f"append_{dt}_t64k_d256", device=DEV, T=300)
    arrs, flags = gpu_append(aw)
    assert flags == 0
    assert_pool_equal(arrs, oracle_append(aw)[0])


@pytest.mark.parametrize("dt", DTS)
def test_append_row_count_not_a_multiple_of_the_warp_tile(dt):
    # 7 tokens x 3 kv heads = 21 rows: the last warp holds a partial tile
    aw = W.make_append_workload(f"append_{dt}_t64k_d256", device=DEV, T=7, Hkv=3, D=128)
    arrs, flags = gpu_append(aw)
    assert flags == 0
    assert_pool_equal(arrs, oracle_append(aw)[0])


def _tie_rows():
    """Rows on the formats' rounding ties (g = 1 for FP8 and NVFP4)."""
    e2m1 = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
            -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, 0.0,
            9984.0, 1344.0, 224.0] + [0.0] * 13
    e4m3 = [1.0625, 1.1875, 1.0, 1.125, 0.5 * 2.0 ** -9, 1.5 * 2.0 ** -9, 2.0 ** -9,
            2.5 * 2.0 ** -9, 7.5 * 2.0 ** -9, 448.0, 464.0, 500.0, 2.0 ** 100, -1000.0, -1.0625,
            -(2.0 ** -11), -0.0, 240.0, 248.0, 0.0]
    int8 = [15.875, 0.0625, 0.1875, 0.3125, -0.0625, -0.1875, 1.5625, -15.875]
    rows = []
    for r in (e2m1, e4m3, int8):
        rows.append(torch.tensor(r + [0.0] * (256 - len(r))))
    return torch.stack(rows)            # [3, 256]


@pytest.mark.parametrize("dt", DTS)
def test_append_rounding_ties(dt):
    aw = W.make_append_workload(f"append_{dt}_t64k_d256", device=DEV, T=16, Hkv=3)
    x = _tie_rows().to(torch.bfloat16)
    assert torch.equal(x.float(), _tie_rows())       # every value is exact in bf16
    k = x.unsqueeze(0).repeat(16, 1, 1).contiguous()
    aw.k_new = k.to(DEV)
    aw.v_new = (-k).contiguous().to(DEV)
    aw.k_global = aw.v_global = 1.0
    aw.slot_mapping = torch.arange(16, dtype=torch.int64, device=DEV) * 3   # distinct slots
    arrs, flags = gpu_append(aw)
    assert flags == 0
    assert_pool_equal(arrs, oracle_append(aw)[0])


@pytest.mark.parametrize("dt", DTS)
def test_full_size_append_sampled(dt):
    """The benchmark's workload (65,536 tokens) in one call; the oracle
    re-encodes a sample of the tokens into a copy of the starting pool and
    those rows must match; every padded row's target stays untouched."""
    aw = W.make_append_workload(f"append_{dt}_t64k_d256", device=DEV)
    arrs, flags = gpu_append(aw)
    assert flags == 0
    g = torch.Generator().manual_seed(3)
    picks = torch.randperm(aw.T, generator=g)[:600].sort().values
    picks = torch.cat([picks, torch.tensor([0, aw.T - 1])])
    sm = aw.slot_mapping.cpu()
    sub = W.AppendWorkload(**{**aw.__dict__, "T": len(picks), "k_new": aw.k_new[picks.to(DEV)],
                              "v_new": aw.v_new[picks.to(DEV)],
                              "slot_mapping": sm[picks].to(DEV)})
    ref, bad = oracle_append(sub)
    assert bad == 0
    rows = sm[picks]
    rows = rows[rows >= 0]
    blk, off = (rows // 16).numpy(), (rows % 16).numpy()
    for g_arr, r_arr in zip(arrs, ref):
        if g_arr is None:
            continue
        gb = as_bits(g_arr)
        assert np.array_equal(gb[blk, :, off], r_arr[blk, :, off])
    # slots no valid row names keep their starting bytes
    written = np.zeros((aw.num_blocks, 16), bool)
    v = sm[sm >= 0]
    written[(v // 16).numpy(), (v % 16).numpy()] = True
    before = as_bits(aw.k_cache)
    after = as_bits(arrs[0])
    assert np.array_equal(after[~written[:, None, :].repeat(aw.Hkv, 1)],
                          before[~written[:, None, :].repeat(aw.Hkv, 1)])


@pytest.mark.parametrize("dt", DTS)
def test_append_then_decode(dt):
    """Decode step: one new token per sequence is appended at position L
    (its slot from the block table), then attention runs over L + 1 keys;
    a padded row (slot -1) writes nothing."""
    name = {"bf16": "bf16_skewed_b256_l16_128k_d256", "int8": "int8_b32_l1k_32k_d256",
            "fp8": "fp8_b32_l1k_32k_d256", "nvfp4": "nvfp4_b4_l262k_d256"}[dt]
    lens = [1000, 37, 555, 3001, 200]       # none a multiple of 16: room in the last block
    wl = W.make_workload(name, device=DEV, seq_lens=[L + 1 for L in lens])
    B = wl.B
    g = torch.Generator().manual_seed(4)
    k_new = torch.randn(B, wl.Hkv, wl.D, generator=g).to(torch.bfloat16).to(DEV)
    v_new = torch.randn(B, wl.Hkv, wl.D, generator=g).to(torch.bfloat16).to(DEV)
    tab = wl.block_tables.cpu()
    slots = torch.tensor([int(tab[b, L // 16]) * 16 + L % 16 for b, L in enumerate(lens)],
                         dtype=torch.int64)
    slots[4] = -1                           # padded row: sequence 4 keeps its old key L
    kv = pa.KvCache.from_workload(wl)
    h = W.host_arrays(wl)                   # host copy before the append
    pa.append_kv(kv, k_new, v_new, slots.to(DEV))
    o, lse, ws = run(wl, out_fp32=True, return_lse=True)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    cache = oracle.HostCache.from_host_arrays(h, wl.dtype, wl.k_global, wl.v_global)
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)   # noqa: E731
    assert oracle.append(cache, bits(k_new), bits(v_new), slots.numpy()) == 0
    ref_o, ref_l = oracle.attend(cache, h["q"], h["block_tables"], h["seq_lens"],
                                 wl.softmax_scale)
    compare(o, ref_o, f"append+decode {dt}")
    compare_lse(lse, ref_l, f"append+decode {dt}")
