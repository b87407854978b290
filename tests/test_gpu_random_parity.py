"""Randomised parity sweep: many small problems with random format, head
shape, q_len, lengths (including 0, 1, block-boundary and ragged values),
pool layout, split size and kernel choice, each compared element by element
with the fp64 oracle at the shared tolerance.  The seeds are fixed, so a
failure reproduces; the cases are small enough that the whole sweep runs in
well under a minute."""
import random

import pytest
import torch

from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import bf16_matches_fp32, compare, compare_lse, oracle_rows, run

pytestmark = pytest.mark.gpu
DEV = "cuda"

BASE = {"bf16": "bf16_skewed_b256_l16_128k_d256", "int8": "int8_b32_l1k_32k_d256",
        "nvfp4": "nvfp4_b4_l262k_d256", "fp8": "fp8_b32_l1k_32k_d256"}
SHAPES = [(24, 4, 256), (8, 2, 128), (16, 2, 256), (24, 12, 128), (4, 4, 256), (32, 4, 128),
          (8, 8, 256), (2, 1, 128)]


def case(seed):
    rng = random.Random(seed)
    dt = rng.choice(list(BASE))
    Hq, Hkv, D = rng.choice(SHAPES)
    verify = rng.random() < 0.35
    Q = rng.choice([2, 3, 5, 8, 16]) if verify else 1
    B = rng.randint(1, 6)
    lens = []
    for _ in range(B):
        kind = rng.random()
        if kind < 0.1:
            L = 0
        elif kind < 0.25:
            L = rng.choice([1, 15, 16, 17, 31, 32, 33, 127, 128, 129])
        else:
            L = rng.randint(1, 3000)
        if verify and L:
            L = max(L, Q)
        lens.append(L)
    kernels = [0, 1, 2, 3] + ([4] if verify and dt in ("nvfp4", "fp8") and D == 256 else []) \
        + ([5] if not verify else [])
    kernel = rng.choice(kernels)
    split = rng.choice([0, 0, 1, 3, 8, 1 << 20])
    return dict(dt=dt, shape=(Hq, Hkv, D), Q=Q, lens=lens, kernel=kernel, split=split)


@pytest.mark.parametrize("seed", range(48))
def test_random_case_matches_oracle(seed):
    c = case(seed)
    Hq, Hkv, D = c["shape"]
    wl = W.make_workload(BASE[c["dt"]], device=DEV, seq_lens=c["lens"], Q=c["Q"], Hq=Hq, Hkv=Hkv,
                         D=D, seed=5000 + seed)
    fn = "verify" if c["Q"] > 1 else "decode"
    kw = dict(kernel=c["kernel"])
    if c["split"] and c["kernel"] != 5:
        kw["split_blocks"] = c["split"]
    try:
        o32, lse, ws = run(wl, fn, out_fp32=True, return_lse=True, **kw)
    except pa.PaError as e:   # a kernel that does not take this shape says so on the host
        assert e.status == pa.PA_ERR_UNSUPPORTED, (c, e)
        pytest.skip(f"unsupported combination {c}")
    ob, _ = run(wl, fn, **kw)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0, c
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, str(c))
    compare_lse(lse, ref_l, str(c))
    assert bf16_matches_fp32(ob, o32), c
