"""Seeded synthetic inputs for paged-KV decode and speculative-verify attention.

Both sides of every parity check consume what this module makes: the CUDA
library through its C ABI and the fp64 oracle under ``oracle/``.  It holds
none of the attention method itself.  The storage formats' *encoders* live
here because writing a cache is how the inputs are produced; *decoding* a
cache is the method's first step and is written twice, independently, in
the CUDA kernels and in the oracle.

Workloads follow the shapes of the pages' serving stacks: GQA heads, head
dim 256, contexts up to 262K tokens ("vLLM All-NVFP4 DFlash2 for Blackwell",
"What makes this stack different"), 8-token speculative verify (same
section, DFlash2 K=7), int8 KV ("vLLM-SM70", "Why"), and PagedAttention's
block-table pool (Kwon et al., cited in "vLLM Fork with focus on GB10
Homelabs", "About").

Readings of points the pages leave open (all documented in the design
notes): cache layout [num_blocks, Hkv, 16, D]; int8 scale per (token, kv
head) = fp16_RNE(max|x| / 127); NVFP4 global scale per tensor =
amax(valid) / (6 * 448), block scale = E4M3_RNE_satfinite(amax16 / (6 g)),
codes = E2M1 round-to-nearest-even of x / (s g); element 2i in the low
nibble; seq_lens count every key including the Q new tokens; seed = 1000 +
workload id; unused slots and pool blocks are poisoned.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

BLOCK_SIZE = 16

# name -> recipe.  `lens` is the seq_len recipe, `pool` the block-table recipe.
WORKLOADS = {
    "bf16_b1_l1000_d128": dict(
        id=1, dtype="bf16", B=1, Q=1, Hq=8, Hkv=2, D=128,
        lens=("fixed", 1000), pool=("permuted_subset", 128)),
    "int8_b32_l1k_32k_d256": dict(
        id=2, dtype="int8", B=32, Q=1, Hq=24, Hkv=4, D=256,
        lens=("uniform", 1024, 32768), pool=("shuffled",)),
    "nvfp4_b4_l262k_d256": dict(
        id=3, dtype="nvfp4", B=4, Q=1, Hq=24, Hkv=4, D=256,
        lens=("fixed", 262144), pool=("shuffled",)),
    "nvfp4_verify_q8_b4_ctx64k_d256": dict(
        id=4, dtype="nvfp4", B=4, Q=8, Hq=24, Hkv=4, D=256,
        lens=("fixed", 65536 + 8), pool=("shuffled",)),
    "fp8_b32_l1k_32k_d256": dict(
        id=6, dtype="fp8", B=32, Q=1, Hq=24, Hkv=4, D=256,
        lens=("uniform", 1024, 32768), pool=("shuffled",)),
    "fp8_verify_q8_b4_ctx64k_d256": dict(
        id=7, dtype="fp8", B=4, Q=8, Hq=24, Hkv=4, D=256,
        lens=("fixed", 65536 + 8), pool=("shuffled",)),
    # block-sparse decode: 64-token sparse blocks, 256 of them attended
    # per (sequence, kv head) = 16,384 of 262,144 keys
    "int8_sparse_b8_l262k_k256_d256": dict(
        id=12, dtype="int8", B=8, Q=1, Hq=24, Hkv=4, D=256,
        lens=("fixed", 262144), pool=("shuffled",), sparse_block=64, top_k=256),
    "bf16_skewed_b256_l16_128k_d256": dict(
        id=5, dtype="bf16", B=256, Q=1, Hq=24, Hkv=4, D=256,
        lens=("loguniform", 16, 131072), pool=("interleaved",)),
}

E4M3_MAX = 448.0
E2M1_MAX = 6.0
BF16_NAN_BITS = 0x7FC0


def workload_names():
    return list(WORKLOADS)


def spec(name: str) -> dict:
    return dict(WORKLOADS[name], name=name)


# --------------------------------------------------------------------------
# format encoders (input production only)
# --------------------------------------------------------------------------

def e4m3_encode_rne_satfinite(a: torch.Tensor) -> torch.Tensor:
    """Non-negative fp32 -> OCP FP8 E4M3 code (bias 7, 3 mantissa bits,
    max 448, min subnormal 2^-9), round-to-nearest-even, saturating to 448.
    Returns uint8 codes (sign bit always 0)."""
    a = a.float().clamp(min=0.0)
    sat = a >= E4M3_MAX
    _, ex = torch.frexp(torch.where(a > 0, a, torch.ones_like(a)))
    e = ex.to(torch.int32) - 1                       # a in [2^e, 2^(e+1))
    e = torch.clamp(e, min=-6)                       # subnormals share 2^-6 binade
    quantum = torch.ldexp(torch.ones_like(a), (e - 3).to(torch.int32))
    qv = torch.round(a / quantum).to(torch.int32)   # half-to-even; exact division
    # mantissa overflow to the next binade
    carry = qv >= 16
    e = torch.where(carry, e + 1, e)
    qv = torch.where(carry, qv // 2, qv)
    normal = qv >= 8
    code = torch.where(normal, ((e + 7) << 3) | (qv - 8), qv)
    code = torch.where(sat, torch.full_like(code, 0x7E), code)
    code = torch.clamp(code, max=0x7E)
    return code.to(torch.uint8)


def e2m1_encode_rne(y: torch.Tensor) -> torch.Tensor:
    """fp32 -> FP4 E2M1 code (values {0, .5, 1, 1.5, 2, 3, 4, 6}, bit 3 =
    sign), round-to-nearest-even with ties to the even mantissa, saturating
    at 6.  Returns uint8 codes in [0, 16)."""
    a = y.float().abs()
    # magnitude code thresholds: ties resolve toward the even code
    code = torch.zeros_like(a, dtype=torch.int32)
    code = torch.where(a > 0.25, 1, code)
    code = torch.where(a >= 0.75, 2, code)
    code = torch.where(a > 1.25, 3, code)
    code = torch.where(a >= 1.75, 4, code)
    code = torch.where(a > 2.5, 5, code)
    code = torch.where(a >= 3.5, 6, code)
    code = torch.where(a > 5.0, 7, code)
    sign = (y.float() < 0) | ((y.float() == 0) & torch.signbit(y.float()))
    code = code | (sign.to(torch.int32) << 3)
    return code.to(torch.uint8)


_E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3_values(device) -> torch.Tensor:
    """fp32 value of every non-negative E4M3 code 0..127 (127 = NaN), used by
    the encoder to know which scale it wrote."""
    c = torch.arange(128, device=device, dtype=torch.int32)
    e = c >> 3
    m = c & 7
    sub = torch.ldexp(m.float(), torch.full_like(c, -9))
    nor = torch.ldexp((m + 8).float(), e - 10)
    v = torch.where(e == 0, sub, nor)
    v[127] = float("nan")
    return v


def quantize_int8_rows(x: torch.Tensor):
    """x [..., D] fp32 -> (codes int8 [..., D], scale fp16 [...]) with
    s = fp16_RNE(max|x| / 127), code = clamp(rint(x / s), -127, 127)."""
    amax = x.abs().amax(dim=-1)
    s16 = (amax / 127.0).to(torch.float16)
    s = s16.float().unsqueeze(-1)
    safe = torch.where(s > 0, s, torch.ones_like(s))
    code = torch.round(x / safe).clamp(-127, 127)
    code = torch.where(s > 0, code, torch.zeros_like(code))
    return code.to(torch.int8), s16


def quantize_fp8(x: torch.Tensor, g: float) -> torch.Tensor:
    """x fp32, g fp32 per-tensor scale -> E4M3 codes (uint8) of x / g,
    round-to-nearest-even, saturating at 448, sign in bit 7."""
    g32 = torch.tensor(g, dtype=torch.float32, device=x.device)
    y = x / g32 if g > 0 else torch.zeros_like(x)
    code = e4m3_encode_rne_satfinite(y.abs())
    neg = (y < 0) & (code != 0)
    return (code | (neg.to(torch.uint8) << 7)).to(torch.uint8)


def quantize_nvfp4_rows(x: torch.Tensor, g: float):
    """x [..., D] fp32, g fp32 global scale -> (packed codes uint8 [..., D/2],
    block scales uint8 (E4M3) [..., D/16]).  Element 2i is the low nibble."""
    shp = x.shape
    D = shp[-1]
    xb = x.reshape(*shp[:-1], D // 16, 16)
    amax = xb.abs().amax(dim=-1)
    g32 = torch.tensor(g, dtype=torch.float32, device=x.device)
    denom = g32 * torch.tensor(6.0, dtype=torch.float32, device=x.device)
    s_code = e4m3_encode_rne_satfinite(amax / denom if g > 0 else torch.zeros_like(amax))
    s_val = _e4m3_values(x.device)[s_code.long()]
    sg = (s_val * g32).unsqueeze(-1)
    safe = torch.where(sg > 0, sg, torch.ones_like(sg))
    y = torch.where(sg > 0, xb / safe, torch.zeros_like(xb))
    codes = e2m1_encode_rne(y).reshape(*shp[:-1], D)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).to(torch.uint8)
    return packed, s_code


# --------------------------------------------------------------------------
# workload construction
# --------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    dtype: str                     # "bf16" | "int8" | "nvfp4" | "fp8"
    B: int
    Q: int
    Hq: int
    Hkv: int
    D: int
    seed: int
    seq_lens: torch.Tensor         # int32 [B]
    block_tables: torch.Tensor     # int32 [B, stride]
    q: torch.Tensor                # bf16 [B, Q, Hq, D]
    k_cache: torch.Tensor          # bf16/int8/fp8 [NB,Hkv,16,D] or uint8 [NB,Hkv,16,D/2]
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor] = None   # fp16 [NB,Hkv,16] | uint8 [NB,Hkv,16,D/16]
    v_scale: Optional[torch.Tensor] = None
    k_global: float = 1.0
    v_global: float = 1.0
    softmax_scale: float = 1.0
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def stride(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.long().sum().item())

    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.B else 0


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_seq_lens(recipe, B: int, gen: torch.Generator) -> torch.Tensor:
    kind = recipe[0]
    if kind == "fixed":
        return torch.full((B,), int(recipe[1]), dtype=torch.int32)
    if kind == "uniform":
        lo, hi = int(recipe[1]), int(recipe[2])
        return torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64).to(torch.int32)
    if kind == "loguniform":
        lo, hi = math.log(recipe[1]), math.log(recipe[2])
        u = torch.rand((B,), generator=gen, dtype=torch.float64)
        return torch.round(torch.exp(lo + (hi - lo) * u)).to(torch.int32)
    if kind == "list":
        return torch.tensor(list(recipe[1]), dtype=torch.int32)
    raise ValueError(kind)


def make_block_tables(pool_recipe, seq_lens: torch.Tensor, gen: torch.Generator,
                      stride: Optional[int] = None):
    """Returns (tables int32 [B, stride], num_blocks).  Unused table entries
    are -1 (never read for t < seq_len)."""
    nblk = [(int(L) + BLOCK_SIZE - 1) // BLOCK_SIZE for L in seq_lens.tolist()]
    B = len(nblk)
    need = sum(nblk)
    if stride is None:
        stride = max(nblk) if nblk else 1
        stride = max(stride, 1)
    tables = torch.full((B, stride), -1, dtype=torch.int32)
    kind = pool_recipe[0]
    if kind == "permuted_subset":
        pool = int(pool_recipe[1])
        assert need <= pool
        perm = torch.randperm(pool, generator=gen).to(torch.int32)
        pos = 0
        for b in range(B):
            tables[b, : nblk[b]] = perm[pos: pos + nblk[b]]
            pos += nblk[b]
        return tables, pool
    if kind == "shuffled":
        perm = torch.randperm(max(need, 1), generator=gen).to(torch.int32)
        pos = 0
        for b in range(B):
            tables[b, : nblk[b]] = perm[pos: pos + nblk[b]]
            pos += nblk[b]
        return tables, max(need, 1)
    if kind == "interleaved":
        # append order: step j hands block j to every sequence still growing,
        # in sequence order; ids are consecutive.
        nb = torch.tensor(nblk, dtype=torch.int64)
        maxb = int(nb.max().item()) if B else 0
        nxt = 0
        for j in range(maxb):
            rows = torch.nonzero(nb > j).flatten()
            n = rows.numel()
            tables[rows, j] = torch.arange(nxt, nxt + n, dtype=torch.int32)
            nxt += n
        return tables, max(nxt, 1)
    raise ValueError(kind)


def _valid_counts(tables: torch.Tensor, seq_lens: torch.Tensor, num_blocks: int) -> torch.Tensor:
    """valid slots per physical block (0 for blocks no sequence uses)."""
    vc = torch.zeros(num_blocks, dtype=torch.int32)
    for b, L in enumerate(seq_lens.tolist()):
        n = (L + BLOCK_SIZE - 1) // BLOCK_SIZE
        if n == 0:
            continue
        ids = tables[b, :n].long()
        cnt = torch.full((n,), BLOCK_SIZE, dtype=torch.int32)
        cnt[-1] = L - (n - 1) * BLOCK_SIZE
        vc[ids] = cnt
    return vc


def _normal_chunk(seed: int, tag: int, chunk: int, shape, device) -> torch.Tensor:
    g = _dev_gen((seed * 1000003 + tag * 7919 + chunk) % (2**62), device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _rand_bytes(seed: int, tag: int, chunk: int, shape, device, dtype=torch.uint8, hi=256):
    g = _dev_gen((seed * 1000003 + tag * 7919 + chunk + 17) % (2**62), device)
    return torch.randint(0, hi, shape, generator=g, device=device, dtype=torch.int64).to(dtype)


def make_workload(name: str, device="cpu", *, B: Optional[int] = None,
                  seq_lens: Optional[Sequence[int]] = None, Q: Optional[int] = None,
                  seed: Optional[int] = None, poison: bool = True,
                  chunk_blocks: int = 2048, kv_values: Optional[str] = None,
                  Hq: Optional[int] = None, Hkv: Optional[int] = None,
                  D: Optional[int] = None) -> Workload:
    """Builds a workload by its recipe name.  `B`, `seq_lens` and `Q`
    override the recipe for reduced-size parity cases (same distributions
    and structure); `Hq`, `Hkv`, `D` override the head shape.  `kv_values` = "const_v" makes every valid V row of a
    kv head the same vector (closed-form test input)."""
    s = spec(name)
    seed = 1000 + s["id"] if seed is None else seed
    Bv = s["B"] if B is None else B
    Qv = s["Q"] if Q is None else Q
    gen = _cpu_gen(seed)
    if seq_lens is not None:
        lens = torch.tensor(list(seq_lens), dtype=torch.int32)
        Bv = lens.numel()
    else:
        lens = make_seq_lens(s["lens"], Bv, gen)
    pool = s["pool"]
    if pool[0] == "permuted_subset":
        need = sum((int(L) + 15) // 16 for L in lens.tolist())
        pool = ("permuted_subset", max(int(pool[1]), need))
    tables, NB = make_block_tables(pool, lens, gen)
    Hq = s["Hq"] if Hq is None else Hq
    Hkv = s["Hkv"] if Hkv is None else Hkv
    D = s["D"] if D is None else D
    dt = s["dtype"]
    dev = torch.device(device)

    qg = _dev_gen(seed * 31 + 1, dev)
    q = torch.randn((Bv, Qv, Hq, D), generator=qg, device=dev, dtype=torch.float32).to(torch.bfloat16)

    vcount = _valid_counts(tables, lens, NB).to(dev)
    slot = torch.arange(BLOCK_SIZE, device=dev, dtype=torch.int32)

    def valid_mask(b0, b1):
        return (slot.view(1, BLOCK_SIZE) < vcount[b0:b1].view(-1, 1))  # [n,16]

    chunks = [(b0, min(NB, b0 + chunk_blocks)) for b0 in range(0, NB, chunk_blocks)]
    shape_full = (Hkv, BLOCK_SIZE, D)

    def gen_x(tag, ci, b0, b1):
        x = _normal_chunk(seed, tag, ci, (b1 - b0,) + shape_full, dev)
        if kv_values == "const_v" and tag == 2:
            base = _normal_chunk(seed, 99, 0, (1, Hkv, 1, D), dev)
            x = base.expand_as(x).contiguous()
        return x

    wl_kwargs = {}
    if dt == "bf16":
        caches = []
        for tag in (1, 2):
            out = torch.empty((NB,) + shape_full, dtype=torch.bfloat16, device=dev)
            for ci, (b0, b1) in enumerate(chunks):
                x = gen_x(tag, ci, b0, b1).to(torch.bfloat16)
                if poison:
                    m = valid_mask(b0, b1).view(-1, 1, BLOCK_SIZE, 1)
                    nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16, device=dev).view(torch.bfloat16)
                    x = torch.where(m, x, nan)
                out[b0:b1] = x
            caches.append(out)
        k, v = caches
    elif dt == "int8":
        caches, scales = [], []
        for tag in (1, 2):
            out = torch.empty((NB,) + shape_full, dtype=torch.int8, device=dev)
            sc = torch.empty((NB, Hkv, BLOCK_SIZE), dtype=torch.float16, device=dev)
            for ci, (b0, b1) in enumerate(chunks):
                x = gen_x(tag, ci, b0, b1)
                c, s16 = quantize_int8_rows(x)
                if poison:
                    m = valid_mask(b0, b1).view(-1, 1, BLOCK_SIZE)
                    junk_c = _rand_bytes(seed, tag + 10, ci, c.shape, dev, torch.int64).sub(128).to(torch.int8)
                    junk_s = _rand_bytes(seed, tag + 20, ci, s16.shape, dev, torch.int64, hi=65536)
                    junk_s = junk_s.to(torch.int32).to(torch.int16).view(torch.float16)
                    c = torch.where(m.unsqueeze(-1), c, junk_c)
                    s16 = torch.where(m, s16, junk_s)
                out[b0:b1] = c
                sc[b0:b1] = s16
            caches.append(out)
            scales.append(sc)
        k, v = caches
        wl_kwargs = dict(k_scale=scales[0], v_scale=scales[1])
    elif dt == "nvfp4":
        # pass 1: per-tensor amax over valid elements
        amaxes = []
        for tag in (1, 2):
            am = torch.zeros((), dtype=torch.float32, device=dev)
            for ci, (b0, b1) in enumerate(chunks):
                x = gen_x(tag, ci, b0, b1)
                m = valid_mask(b0, b1).view(-1, 1, BLOCK_SIZE, 1)
                am = torch.maximum(am, torch.where(m, x.abs(), torch.zeros_like(x)).amax())
            amaxes.append(float(am.item()))
        gs = [float(torch.tensor(a / (E2M1_MAX * E4M3_MAX), dtype=torch.float32)) for a in amaxes]
        caches, scales = [], []
        for ti, tag in enumerate((1, 2)):
            out = torch.empty((NB, Hkv, BLOCK_SIZE, D // 2), dtype=torch.uint8, device=dev)
            sc = torch.empty((NB, Hkv, BLOCK_SIZE, D // 16), dtype=torch.uint8, device=dev)
            for ci, (b0, b1) in enumerate(chunks):
                x = gen_x(tag, ci, b0, b1)
                c, s8 = quantize_nvfp4_rows(x, gs[ti])
                if poison:
                    m = valid_mask(b0, b1).view(-1, 1, BLOCK_SIZE, 1)
                    c = torch.where(m, c, _rand_bytes(seed, tag + 10, ci, c.shape, dev))
                    s8 = torch.where(m, s8, _rand_bytes(seed, tag + 20, ci, s8.shape, dev))
                out[b0:b1] = c
                sc[b0:b1] = s8
            caches.append(out)
            scales.append(sc)
        k, v = caches
        wl_kwargs = dict(k_scale=scales[0], v_scale=scales[1], k_global=gs[0], v_global=gs[1])
    elif dt == "fp8":
        amaxes = []
        for tag in (1, 2):
            am = torch.zeros((), dtype=torch.float32, device=dev)
            for ci, (b0, b1) in enumerate(chunks):
                x = gen_x(tag, ci, b0, b1)
                m = valid_mask(b0, b1).view(-1, 1, BLOCK_SIZE, 1)
                am = torch.maximum(am, torch.where(m, x.abs(), torch.zeros_like(x)).amax())
            amaxes.append(float(am.item()))
        gs = [float(torch.tensor(a / E4M3_MAX, dtype=torch.float32)) for a in amaxes]
        caches = []
        for ti, tag in enumerate((1, 2)):
            out = torch.empty((NB,) + shape_full, dtype=torch.uint8, device=dev)
            for ci, (b0, b1) in enumerate(chunks):
                c = quantize_fp8(gen_x(tag, ci, b0, b1), gs[ti])
                if poison:
                    m = valid_mask(b0, b1).view(-1, 1, BLOCK_SIZE, 1)
                    c = torch.where(m, c, _rand_bytes(seed, tag + 10, ci, c.shape, dev))
                out[b0:b1] = c
            caches.append(out)
        k, v = caches
        wl_kwargs = dict(k_global=gs[0], v_global=gs[1])
    else:
        raise ValueError(dt)

    return Workload(
        name=name, dtype=dt, B=Bv, Q=Qv, Hq=Hq, Hkv=Hkv, D=D, seed=seed,
        seq_lens=lens.to(dev), block_tables=tables.to(dev), q=q,
        k_cache=k, v_cache=v, softmax_scale=1.0 / math.sqrt(D),
        meta=dict(recipe=s, num_blocks=NB), **wl_kwargs)


def permute_pool(wl: Workload, seed: int = 7) -> Workload:
    """Same logical KV, physical blocks relabelled by a random permutation
    (tables rewritten accordingly).  Attention must not change."""
    NB = wl.num_blocks
    g = _cpu_gen(seed)
    perm = torch.randperm(NB, generator=g)           # new id of old block i
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(NB)
    dev = wl.k_cache.device
    idx = inv.to(dev)

    def re(t):
        return None if t is None else t[idx].contiguous()

    tables = wl.block_tables.clone()
    valid = tables >= 0
    tables[valid] = perm.to(dev).to(torch.int32)[tables[valid].long()]
    return Workload(
        name=wl.name + "+perm", dtype=wl.dtype, B=wl.B, Q=wl.Q, Hq=wl.Hq, Hkv=wl.Hkv,
        D=wl.D, seed=wl.seed, seq_lens=wl.seq_lens, block_tables=tables, q=wl.q,
        k_cache=re(wl.k_cache), v_cache=re(wl.v_cache), k_scale=re(wl.k_scale),
        v_scale=re(wl.v_scale), k_global=wl.k_global, v_global=wl.v_global,
        softmax_scale=wl.softmax_scale, meta=dict(wl.meta))


def host_arrays(wl: Workload) -> dict:
    """numpy views of every input, as the oracle reads them (raw bits for
    bf16/fp16/E4M3 so that the oracle does its own decoding)."""
    def np_bits(t):
        if t is None:
            return None
        t = t.detach().cpu().contiguous()
        if t.dtype in (torch.bfloat16, torch.float16):
            return t.view(torch.int16).numpy().view("uint16")
        return t.numpy()
    return dict(
        q=np_bits(wl.q), k_cache=np_bits(wl.k_cache), v_cache=np_bits(wl.v_cache),
        k_scale=np_bits(wl.k_scale), v_scale=np_bits(wl.v_scale),
        block_tables=wl.block_tables.cpu().numpy(), seq_lens=wl.seq_lens.cpu().numpy())


# --------------------------------------------------------------------------
# KV append (quantise-on-write) workloads
# --------------------------------------------------------------------------

# T new tokens of `seq` tokens per sequence (a prefill chunk per sequence),
# Hkv 4 / D 256 like the decode workloads; every `pad_every`-th row is a
# padded row (slot -1).  Seeds 1000 + id.
APPEND_WORKLOADS = {
    f"append_{dt}_t64k_d256": dict(id=8 + i, dtype=dt, T=65536, seq=4096, Hkv=4, D=256,
                                   pad_every=61)
    for i, dt in enumerate(("bf16", "int8", "fp8", "nvfp4"))
}


@dataclass
class AppendWorkload:
    name: str
    dtype: str
    T: int
    Hkv: int
    D: int
    seed: int
    k_new: torch.Tensor            # bf16 [T, Hkv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor     # int64 [T], -1 = padded row
    k_cache: torch.Tensor          # the pool before the append (random bytes)
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    k_global: float = 1.0
    v_global: float = 1.0

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def valid_rows(self) -> int:
        return int((self.slot_mapping >= 0).sum().item())


def make_append_workload(name: str, device="cpu", *, T: Optional[int] = None,
                         seed: Optional[int] = None, D: Optional[int] = None,
                         Hkv: Optional[int] = None, dtype: Optional[str] = None) -> AppendWorkload:
    """New K / V rows N(0, 1) (rows of magnitude 1e-3 and 1e3 mixed in, one in
    eight each), bf16; sequences of `seq` tokens whose blocks come from a
    shuffled pool, each token at its block and offset; padded rows -1.  The
    pool starts as random bytes so that untouched bytes can be checked.
    NVFP4 / FP8 per-tensor scales: amax / (6 * 448) and amax / 448 of the new
    rows, in fp32."""
    sp = APPEND_WORKLOADS[name]
    dt = dtype or sp["dtype"]
    T = sp["T"] if T is None else T
    D = D or sp["D"]
    Hkv = Hkv or sp["Hkv"]
    seed = 1000 + sp["id"] if seed is None else seed
    g = _cpu_gen(seed)
    seq = sp["seq"]
    lens = [min(seq, T - s) for s in range(0, T, seq)]
    nblk = [(L + BLOCK_SIZE - 1) // BLOCK_SIZE for L in lens]
    NB = max(sum(nblk) + 8, 1)
    perm = torch.randperm(NB, generator=g)
    slots = []
    pos = 0
    for L, n in zip(lens, nblk):
        blocks = perm[pos: pos + n]
        pos += n
        t = torch.arange(L)
        slots.append(blocks[t // BLOCK_SIZE] * BLOCK_SIZE + t % BLOCK_SIZE)
    slot_mapping = torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64)
    if T:
        slot_mapping[sp["pad_every"] - 1:: sp["pad_every"]] = -1
    slot_mapping = slot_mapping.to(torch.int64)

    def rows(tag):
        x = torch.randn((T, Hkv, D), generator=_cpu_gen(seed * 31 + tag), dtype=torch.float32)
        mag = torch.ones(T)
        mag[3::8] = 1e-3
        mag[5::8] = 1e3
        return (x * mag.view(T, 1, 1)).to(torch.bfloat16)

    k_new, v_new = rows(1), rows(2)
    gl = []
    for x in (k_new, v_new):
        amax = float(x.float().abs().max()) if T else 0.0
        den = E4M3_MAX * (E2M1_MAX if dt == "nvfp4" else 1.0)
        gl.append(float(torch.tensor(amax / den, dtype=torch.float32)))

    def pool(shape, dtype, tag):
        b = torch.randint(0, 256, shape + (torch.empty(0, dtype=dtype).element_size(),),
                          generator=_cpu_gen(seed * 131 + tag), dtype=torch.int64)
        return b.to(torch.uint8).view(dtype).reshape(shape)

    base = (NB, Hkv, BLOCK_SIZE)
    ks = vs = None
    if dt == "bf16":
        kc, vc = pool(base + (D,), torch.bfloat16, 1), pool(base + (D,), torch.bfloat16, 2)
    elif dt == "int8":
        kc, vc = pool(base + (D,), torch.int8, 1), pool(base + (D,), torch.int8, 2)
        ks, vs = pool(base, torch.float16, 3), pool(base, torch.float16, 4)
    elif dt == "fp8":
        kc, vc = pool(base + (D,), torch.uint8, 1), pool(base + (D,), torch.uint8, 2)
    elif dt == "nvfp4":
        kc, vc = pool(base + (D // 2,), torch.uint8, 1), pool(base + (D // 2,), torch.uint8, 2)
        ks, vs = pool(base + (D // 16,), torch.uint8, 3), pool(base + (D // 16,), torch.uint8, 4)
    else:
        raise ValueError(dt)

    def dev(t):
        return None if t is None else t.to(device)

    return AppendWorkload(
        name=name, dtype=dt, T=T, Hkv=Hkv, D=D, seed=seed, k_new=dev(k_new), v_new=dev(v_new),
        slot_mapping=dev(slot_mapping), k_cache=dev(kc), v_cache=dev(vc), k_scale=dev(ks),
        v_scale=dev(vs), k_global=gl[0] if dt in ("fp8", "nvfp4") else 1.0,
        v_global=gl[1] if dt in ("fp8", "nvfp4") else 1.0)


def append_host_arrays(aw: AppendWorkload) -> dict:
    """numpy copies (raw bits) of the pool and the new rows, as the oracle reads them."""
    def np_bits(t):
        if t is None:
            return None
        t = t.detach().cpu().contiguous().clone()
        if t.dtype in (torch.bfloat16, torch.float16):
            return t.view(torch.int16).numpy().view("uint16")
        return t.numpy()
    return dict(k_cache=np_bits(aw.k_cache), v_cache=np_bits(aw.v_cache),
                k_scale=np_bits(aw.k_scale), v_scale=np_bits(aw.v_scale),
                k_new=np_bits(aw.k_new), v_new=np_bits(aw.v_new),
                slot_mapping=aw.slot_mapping.cpu().numpy())
