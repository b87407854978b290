"""Pins for the oracle's quantise-on-write KV append against things other
than itself.

* library conversions: the FP8 encoder against torch's float -> float8_e4m3fn
  conversion over every bf16 value in range, the int8 scale against numpy's
  float32 -> float16 conversion over every positive bf16 row maximum;
* hand-derived codes from the OCP E2M1 / E4M3 definitions at every
  round-to-nearest-even tie, saturation and the sign of zero;
* the generator's encoders (an independent, vectorised implementation of
  the same formats) on random rows of several magnitudes;
* on-grid values round-trip exactly through the oracle's own (separately
  pinned) decoder; int8 codes stay within half a scale step;
* padded rows (slot -1) write nothing and out-of-range slots are skipped
  and counted ("vLLM-SM70", "Known limitations": padded drafter rows that
  wrote K/V into other requests' slots).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_07_gb300 import workloads as W

H, D, NB = 2, 128, 8


def empty_cache(dt, k_global=1.0, v_global=1.0, nb=NB, h=H, d=D, fill=None):
    """A host pool of `nb` blocks; `fill` = byte value every array starts with."""
    rng = np.random.default_rng(11)

    def arr(shape, dtype):
        if fill is None:
            return np.zeros(shape, dtype)
        return rng.integers(0, 256, size=shape, dtype=np.uint8).view(dtype).reshape(shape) \
            if np.dtype(dtype).itemsize == 1 else \
            rng.integers(0, 65536, size=shape, dtype=np.uint16).view(dtype).reshape(shape)

    if dt == "bf16":
        k, v, ks, vs = arr((nb, h, 16, d), np.uint16), arr((nb, h, 16, d), np.uint16), None, None
    elif dt == "int8":
        k, v = arr((nb, h, 16, d), np.int8), arr((nb, h, 16, d), np.int8)
        ks, vs = arr((nb, h, 16), np.uint16), arr((nb, h, 16), np.uint16)
    elif dt == "fp8":
        k, v, ks, vs = arr((nb, h, 16, d), np.uint8), arr((nb, h, 16, d), np.uint8), None, None
    else:
        k, v = arr((nb, h, 16, d // 2), np.uint8), arr((nb, h, 16, d // 2), np.uint8)
        ks, vs = arr((nb, h, 16, d // 16), np.uint8), arr((nb, h, 16, d // 16), np.uint8)
    return oracle.HostCache(dt, k, v, ks, vs, k_global, v_global)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def append_rows(dt, rows_k, rows_v=None, k_global=1.0, v_global=1.0):
    """Append rows [T, H, D] (bf16-representable fp32) at slots 0..T-1."""
    rows_v = rows_k if rows_v is None else rows_v
    T = rows_k.shape[0]
    c = empty_cache(dt, k_global, v_global, nb=(T + 15) // 16, h=rows_k.shape[1],
                    d=rows_k.shape[2])
    bad = oracle.append(c, bf16_bits(rows_k), bf16_bits(rows_v), np.arange(T, dtype=np.int64))
    assert bad == 0
    return c


def row_codes(c, which, t, h=0):
    blk, off = divmod(t, 16)
    data = c.arrays[which][blk, h, off]
    sc = c.arrays[2 + which]
    return data, (None if sc is None else sc[blk, h, off])


# ------------------------------------------------------- library conversions

def test_fp8_encoder_matches_torch_float8_over_all_bf16_in_range():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    x = x[torch.isfinite(x) & (x.abs() <= 448.0)]
    n = (x.numel() // D) * D
    x = x[:n]
    rows = x.reshape(-1, 1, D)
    c = append_rows("fp8", rows)
    got = c.arrays[0].reshape(-1, D)[: rows.shape[0]].reshape(-1)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where((ref & 0x7F) == 0, 0, ref)        # zero magnitude is written +0
    assert np.array_equal(got, ref)


def test_int8_scale_matches_numpy_float16_over_all_bf16_maxima():
    bits = np.arange(1, 0x7F80, dtype=np.uint16)      # every positive finite bf16
    a = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    rows = torch.zeros(a.numel(), 1, 16)
    rows[:, 0, 0] = a
    ratio = a.numpy().astype(np.float32) / np.float32(127.0)
    with np.errstate(over="ignore"):
        ref = ratio.astype(np.float16).view(np.uint16)
    c = empty_cache("int8", nb=(a.numel() + 15) // 16, h=1, d=16)
    bad = oracle.append(c, bf16_bits(rows), bf16_bits(rows), np.arange(a.numel(), dtype=np.int64))
    assert bad == 0
    got = c.arrays[2].reshape(-1)[: a.numel()]
    assert np.array_equal(got, ref)


# ------------------------------------------------------- hand-derived codes

def test_e2m1_ties_saturation_and_signed_zero():
    # g = 1 and a block maximum of 6 give block scale 1.0 (E4M3 code 0x38),
    # so each element is rounded onto the E2M1 grid {0,.5,1,1.5,2,3,4,6} as is.
    ties = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
            -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, 0.0]
    ties_codes = [7, 0, 2, 2, 4, 4, 6, 6, 8, 10, 10, 12, 12, 14, 14, 0]
    plain = [6.0, 0.2, 0.3, 0.7, 0.8, 1.2, 1.3, 1.7, 1.8, 2.4, 2.6, 3.4, 3.6, 4.9, 5.1, 5.9]
    plain_codes = [7, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6, 7, 7]
    # amax 9984 > 448 * 6: the block scale saturates at 448 (0x7E); 9984 / 448
    # = 22.3 saturates at 6; 1344 / 448 = 3 and 224 / 448 = 0.5 are on the grid
    sat = [9984.0, 1344.0, 224.0] + [0.0] * 13
    sat_codes = [7, 5, 1] + [0] * 13
    zero = [0.0] * 16
    row = torch.tensor([ties + plain + sat + zero] * 2).reshape(1, 1, 128)
    c = append_rows("nvfp4", row, k_global=1.0)
    data, sc = row_codes(c, 0, 0)
    codes = np.stack([data & 0xF, data >> 4], axis=-1).reshape(-1)
    assert codes[:64].tolist() == ties_codes + plain_codes + sat_codes + [0] * 16
    assert sc[:4].tolist() == [0x38, 0x38, 0x7E, 0x00]


def test_e4m3_ties_subnormals_saturation_and_sign():
    # g = 1: y = x.  E4M3 near 1: 1.0 (0x38), 1.125 (0x39), 1.25 (0x3A);
    # subnormals m * 2^-9 (code m).  Ties go to the even code.
    cases = [(1.0625, 0x38), (1.1875, 0x3A), (1.0, 0x38), (1.125, 0x39),
             (0.5 * 2.0 ** -9, 0x00), (1.5 * 2.0 ** -9, 0x02), (2.0 ** -9, 0x01),
             (2.5 * 2.0 ** -9, 0x02), (7.5 * 2.0 ** -9, 0x08),   # 0x08 = 2^-6, first normal
             (448.0, 0x7E), (464.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E),
             (-1000.0, 0xFE), (-1.0625, 0xB8), (-(2.0 ** -11), 0x00), (-0.0, 0x00),
             (240.0, 0x77), (248.0, 0x78), (0.0, 0x00)]
    vals = [v for v, _ in cases] + [0.0] * (D - len(cases))
    c = append_rows("fp8", torch.tensor(vals).reshape(1, 1, D))
    data, _ = row_codes(c, 0, 0)
    assert data[: len(cases)].tolist() == [code for _, code in cases]


def test_int8_ties_round_half_even():
    # row maximum 15.875 = 127 / 8 gives s = fp16(0.125) exactly; x / s = k + 1/2
    # rounds to the even integer; a negative value keeps its sign
    vals = [15.875, 0.0625, 0.1875, 0.3125, -0.0625, -0.1875, 1.5625, -15.875]
    ref = [127, 0, 2, 2, 0, -2, 12, -127]
    c = append_rows("int8", torch.tensor(vals + [0.0] * (D - len(vals))).reshape(1, 1, D))
    data, s = row_codes(c, 0, 0)
    assert s == 0x3000                                 # fp16 0.125
    assert data[: len(vals)].tolist() == ref


# ------------------------------------------------- the generator's encoders

def _random_rows(T, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, D, generator=g)
    mags = torch.tensor([1.0, 1e-3, 1e3, 1e-6])[torch.arange(T) % 4].view(T, 1, 1)
    return (x * mags).to(torch.bfloat16).float()


@pytest.mark.parametrize("dt", ["bf16", "int8", "fp8", "nvfp4"])
def test_append_matches_generator_encoders(dt):
    T = 40
    xk, xv = _random_rows(T, 1), _random_rows(T, 2)
    gk = float(torch.tensor(float(xk.abs().max()) / (448.0 * (6.0 if dt == "nvfp4" else 1.0)),
                            dtype=torch.float32))
    gv = gk * 0.75
    c = empty_cache(dt, gk, gv, nb=6)
    slots = np.random.default_rng(3).permutation(6 * 16)[:T].astype(np.int64)
    slots[[5, 17]] = -1
    assert oracle.append(c, bf16_bits(xk), bf16_bits(xv), slots) == 0
    for t in range(T):
        if slots[t] < 0:
            continue
        for which, x, g in ((0, xk, gk), (1, xv, gv)):
            for h in range(H):
                data, sc = row_codes(c, which, int(slots[t]), h)
                row = x[t, h]
                if dt == "bf16":
                    assert np.array_equal(data, bf16_bits(row))
                elif dt == "int8":
                    codes, s16 = W.quantize_int8_rows(row[None])
                    assert np.array_equal(data, codes[0].numpy())
                    assert sc == int(s16[0].view(torch.int16)) & 0xFFFF
                elif dt == "fp8":
                    assert np.array_equal(data, W.quantize_fp8(row, g).numpy())
                else:
                    codes, s8 = W.quantize_nvfp4_rows(row[None], g)
                    assert np.array_equal(data, codes[0].numpy())
                    assert np.array_equal(sc, s8[0].numpy())


# -------------------------------------------------------- round trips, bounds

def _decode_slots(c, T):
    tables = np.arange((T + 15) // 16, dtype=np.int32)[None]
    k, v = oracle.gather(c, tables, np.array([T], np.int32), T)
    return k[0], v[0]          # [H, T, D]


def test_on_grid_values_round_trip():
    # int8: s = 1/8 (row max 127/8), x = k/8
    k8 = torch.arange(-127, 129, dtype=torch.float32)[:D] / 8.0
    k8[0] = 15.875
    c = append_rows("int8", k8.reshape(1, 1, D))
    assert np.array_equal(_decode_slots(c, 1)[0][0, 0], k8.numpy())
    # FP8: x = e4m3 * g with g = 2^-4, every finite code
    e = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    e = e[(e & 0x7F) != 0x7F].view(torch.float8_e4m3fn).float()
    x = (e * 2.0 ** -4).reshape(-1, 1, 127 * 2 // 2)
    xf = torch.cat([x.reshape(-1), torch.zeros(2 * D - x.numel())]).reshape(2, 1, D)
    c = append_rows("fp8", xf, k_global=2.0 ** -4)
    got = _decode_slots(c, 2)[0][0]
    assert np.array_equal(got, xf[:, 0].numpy())
    # NVFP4: x = e2m1 * s * g with g = 1/2 and a 6 in every block (amax = 6 s g)
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    blocks = []
    for j, s in enumerate([1.0, 0.375, 2.5, 0.0625, 14.0, 1.125, 0.75, 3.0]):
        vals = torch.cat([grid, -grid.flip(0)])
        vals = vals[torch.randperm(16, generator=torch.Generator().manual_seed(j))]
        vals[0] = 6.0
        blocks.append(vals * s * 0.5)
    xn = torch.cat(blocks).reshape(1, 1, D)
    c = append_rows("nvfp4", xn, k_global=0.5)
    assert np.array_equal(_decode_slots(c, 1)[0][0, 0], xn[0, 0].numpy())


def test_int8_codes_within_half_a_step():
    # rows of magnitude 1e-6 are left out: their scale underflows fp16 (to 0
    # or a subnormal), which the format cannot help
    x = _random_rows(16, 7)
    x[3::4] = (x[3::4] * 1e6).to(torch.bfloat16).float()
    c = append_rows("int8", x)
    k, _ = _decode_slots(c, 16)
    for t in range(16):
        for h in range(H):
            data, s16 = row_codes(c, 0, t, h)
            s = float(np.array([s16], np.uint16).view(np.float16)[0])
            err = np.abs(k[h, t].astype(np.float64) - x[t, h].double().numpy())
            assert np.all(np.abs(data.astype(np.int64)) <= 127)
            assert s > 0 and np.all(err <= s / 2)


# ----------------------------------------------------------- slots

@pytest.mark.parametrize("dt", ["int8", "nvfp4", "fp8", "bf16"])
def test_padded_rows_write_nothing_bad_slots_counted(dt):
    c = empty_cache(dt, 0.01, 0.02, fill=True)
    before = [None if a is None else a.copy() for a in c.arrays]
    x = _random_rows(6, 9)
    slots = np.array([-1, 37, -2, NB * 16, 100, -1], np.int64)
    assert oracle.append(c, bf16_bits(x), bf16_bits(x), slots) == 2
    # the same two tokens alone give the same rows
    ref = empty_cache(dt, 0.01, 0.02, fill=True)
    assert oracle.append(ref, bf16_bits(x[[1, 4]]), bf16_bits(x[[1, 4]]),
                         np.array([37, 100], np.int64)) == 0
    for a, b, r in zip(c.arrays, before, ref.arrays):
        if a is None:
            continue
        changed = np.zeros(a.shape[:3], bool)
        for s in (37, 100):
            changed[s // 16, :, s % 16] = True
        assert np.array_equal(a[~changed], b[~changed])       # nothing else touched
        assert np.array_equal(a[changed], r[changed])
