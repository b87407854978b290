#!/usr/bin/env python3
"""Benchmark of paged-KV decode attention on GB300.

One step = one pa_decode call (device planner -> attention kernel -> LSE
merge) over one batch of the largest synthetic workload: the skewed
continuous batch of 256 sequences with seq_lens log-uniform in [16,
131072] (about 3.7 M keys), 24 query / 4 kv heads, head dim 256, bf16 KV
whose blocks are interleaved across sequences in one pool (append order),
bf16 q and out.  Inputs are resident in HBM when timing starts; the KV pool
(~15 GB) is far larger than the 129 MB L2, so every step streams it from
HBM.

Prints ONE JSON line (rank 0).  Metric: achieved algorithmic HBM GB/s
(KV codes + scales of every valid token, table entries, q and out, divided
by the step time), with KV tokens/s and % of the measured copy bandwidth
beside it.  The same line carries `per_config`: every other workload of
the problem statement (the 1 MB bf16 case, the int8 1K-32K batch, the
NVFP4 262K decode, the NVFP4 8-token verify and the FP8 decode / verify)
timed the same way, each with its kernel time, step time, µs per call and
roofline fraction.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the headline workload instead (the baseline arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "bf16_skewed_b256_l16_128k_d256"
# the other workloads timed on the same line (`per_config`)
PER_CONFIG = ("bf16_b1_l1000_d128", "int8_b32_l1k_32k_d256", "nvfp4_b4_l262k_d256",
              "nvfp4_verify_q8_b4_ctx64k_d256", "fp8_b32_l1k_32k_d256",
              "fp8_verify_q8_b4_ctx64k_d256")
L2_BYTES = 129 << 20
# pools smaller than this are rotated over copies whose total exceeds it, so
# that every call reads its KV from HBM rather than from L2
ROTATE_TOTAL_BYTES = 2 * L2_BYTES
METRIC = "paged decode attention: achieved HBM GB/s (% of peak) and KV tokens/s, 1×GB300"
FALLBACK_HBM_GBS = 6800.0


def kv_bytes_per_token_head(dtype: str, D: int) -> int:
    """Bytes of K+V (codes and scales) one token of one kv head occupies."""
    if dtype == "bf16":
        return 2 * D * 2
    if dtype == "int8":
        return 2 * (D + 2)
    if dtype == "fp8":
        return 2 * D
    return 2 * (D // 2 + D // 16)


def algorithmic_bytes(spec: dict, seq_lens) -> dict:
    lens = [int(x) for x in seq_lens]
    tokens = sum(lens)
    B, Q, Hq, Hkv, D = spec["B_eff"], spec["Q"], spec["Hq"], spec["Hkv"], spec["D"]
    kv = tokens * Hkv * kv_bytes_per_token_head(spec["dtype"], D)
    table = sum((L + 15) // 16 for L in lens) * 4
    q = B * Q * Hq * D * 2
    out = B * Q * Hq * D * 2
    return dict(total=kv + table + q + out, kv=kv, tokens=tokens)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def code_only(text: str) -> str:
    """C++ / CUDA source without its comments and with runs of white space
    collapsed: what the compiled kernel depends on."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(files=None) -> str:
    """sha256 prefix over the code (comments and white space aside) of the
    named files of csrc/ (default: all of them).  A profile summary records it;
    an edit to the code makes the summary stale, an edit to a comment does not."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_07_gb300", "csrc")
    for f in sorted(files or os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """dram bytes per launch of the attention kernel from the committed ncu
    summary for this workload, or None if absent or taken on other source."""
    lines = None
    # decode_<workload>.md, verify_<workload>.md; append workloads carry their kind in the name
    for fname in (f"decode_{workload}.md", f"verify_{workload}.md", f"{workload}.md"):
        try:
            lines = open(os.path.join(ROOT, "profiles", fname)).read().splitlines()
            break
        except OSError:
            continue
    if lines is None:
        return None
    vals = {}
    for ln in lines:
        if ":" in ln and ln.startswith("- "):
            k, v = ln[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    files = vals.get("kernel_sources", "").split() or None   # the files the kernel is built from
    if vals.get("kernel_source_hash") != kernel_source_hash(files):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ln in open(self.path).read().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl != "reference" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available() and args.impl != "reference":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- oracle

def oracle_sample(wl, bs, nthreads):
    """Times the fp64 oracle on sequences `bs` of the workload (compact host
    copy of their blocks).  Returns (seconds, seq_lens of the sample)."""
    import numpy as np
    import torch

    import oracle
    lens = wl.seq_lens.cpu()[bs]
    nblk = [(int(L) + 15) // 16 for L in lens.tolist()]
    tabs = wl.block_tables.cpu()
    ids = torch.cat([tabs[b, :n] for b, n in zip(bs, nblk)]).long().to(wl.k_cache.device)

    def take(t):
        if t is None:
            return None
        a = t[ids].contiguous().cpu()
        if a.dtype in (torch.bfloat16, torch.float16):
            return a.view(torch.int16).numpy().view(np.uint16)
        return a.numpy()

    tab = np.zeros((len(bs), max(nblk)), np.int32)
    pos = 0
    for r, n in enumerate(nblk):
        tab[r, :n] = np.arange(pos, pos + n)
        pos += n
    cache = oracle.HostCache(wl.dtype, take(wl.k_cache), take(wl.v_cache), take(wl.k_scale),
                             take(wl.v_scale), wl.k_global, wl.v_global)
    qb = wl.q[bs].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle.attend(cache, qb, tab, lens.numpy().astype(np.int32), wl.softmax_scale,
                  nthreads=nthreads)
    return time.perf_counter() - t0, lens.tolist()


def oracle_sparse_sample(wl, b, sb, top_k):
    """Times the oracle's block-sparse decode of sequence b (selection and the
    exact attention over the selected blocks; its mean keys are cache state,
    computed beforehand)."""
    import numpy as np
    import torch

    import oracle
    L = int(wl.seq_lens[b])
    n = (L + 15) // 16
    ids = wl.block_tables.cpu()[b, :n].long().to(wl.k_cache.device)

    def take(t):
        if t is None:
            return None
        a = t[ids].contiguous().cpu()
        if a.dtype in (torch.bfloat16, torch.float16):
            return a.view(torch.int16).numpy().view(np.uint16)
        return a.numpy()

    cache = oracle.HostCache(wl.dtype, take(wl.k_cache), take(wl.v_cache), take(wl.k_scale),
                             take(wl.v_scale), wl.k_global, wl.v_global)
    tab = np.arange(n, dtype=np.int32)[None]
    lens = np.array([L], np.int32)
    nsb = (L + sb - 1) // sb
    means = oracle.block_means(cache, tab, lens, sb, nsb)
    qb = wl.q[b:b + 1].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    _, sel = oracle.sparse_select(qb, wl.Hkv, means, np.array([nsb], np.int32), top_k)
    oracle.attend_sparse(cache, qb, tab, lens, sel, sb, wl.softmax_scale)
    return time.perf_counter() - t0


def pick_sample(seq_lens, budget_tokens):
    """Deterministic sample: sequences in index order until the token budget."""
    bs, tot = [], 0
    for b, L in enumerate(seq_lens):
        if L <= 0:
            continue
        bs.append(b)
        tot += int(L)
        if tot >= budget_tokens:
            break
    return bs


# ------------------------------------------------------------------ arms

def run_reference(args, world, rank):
    """The baseline arm: the fp64 CPU oracle, each step a bounded sample."""
    import torch

    from paged_kv_decode_07_gb300 import workloads as W
    if rank != 0:
        return
    spec = W.spec(args.workload)
    full_lens = W.make_seq_lens(spec["lens"], spec["B"], torch.Generator().manual_seed(1000 + spec["id"]))
    bs = pick_sample(full_lens.tolist(), args.ref_tokens)
    sample_lens = [int(full_lens[b]) for b in bs]
    wl = W.make_workload(args.workload, device="cpu", seq_lens=sample_lens)
    nthreads = os.cpu_count() or 1
    times = []
    for i in range(args.warmup + args.steps):
        dt, _ = oracle_sample(wl, list(range(len(bs))), nthreads)
        if i >= args.warmup:
            times.append(dt)
    sp = dict(spec, B_eff=len(bs))
    ab = algorithmic_bytes(sp, sample_lens)
    sec = sum(times) / len(times)
    value = ab["total"] / sec / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "sample_sequences": len(bs),
                   "sample_tokens": ab["tokens"]},
        "kv_tokens_per_s": ab["tokens"] / sec,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"{len(bs)} of {spec['B']} sequences ({ab['tokens']} keys) "
                                   f"of {args.workload}, fp64 two-pass softmax"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch

    from paged_kv_decode_07_gb300 import pa
    from paged_kv_decode_07_gb300 import workloads as W

    dev = torch.device("cuda", torch.cuda.current_device())
    spec = W.spec(args.workload)
    # weak scaling: every rank runs its own full batch (different seed)
    wl = W.make_workload(args.workload, device=dev, seed=1000 + spec["id"] + 7919 * rank,
                         B=args.batch or None)
    kv = pa.KvCache.from_workload(wl)
    lens = wl.seq_lens.cpu().tolist()
    sp = dict(spec, B_eff=wl.B)
    ab = algorithmic_bytes(sp, lens)
    fn = "pa_verify" if wl.Q > 1 else "pa_decode"
    out = torch.empty((wl.B, wl.Q, wl.Hq, wl.D), dtype=torch.bfloat16, device=dev)
    maxlen = wl.max_seq_len()
    ws_bytes = pa.workspace_bytes(kv, wl.B, wl.Q, wl.Hq, maxlen, kernel=args.kernel)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    call = pa.verify if wl.Q > 1 else pa.decode

    def step(events=None, q=None, tables=None, seq_lens=None):
        call(kv, wl.q if q is None else q, wl.block_tables if tables is None else tables,
             wl.seq_lens if seq_lens is None else seq_lens, wl.softmax_scale, out=out,
             max_seq_len=maxlen, workspace=ws, kernel=args.kernel, events=events)

    launches_per_step = 3          # planner, attention kernel, merge
    sparse = spec.get("top_k")
    if sparse:
        # block-sparse decode step: refresh the mean key of each sequence's last
        # sparse block, score + select, then the decode over the selection
        SB, K = spec["sparse_block"], spec["top_k"]
        M = (maxlen + SB - 1) // SB
        means = pa.block_means(kv, wl.block_tables, wl.seq_lens, SB, M)   # prefill-time state
        last = torch.tensor([max((L + SB - 1) // SB - 1, 0) for L in lens], dtype=torch.int32,
                            device=dev)
        ws = torch.empty(pa.sparse_workspace_bytes(kv, wl.B, wl.Hq, maxlen, means, SB, K,
                                                   kernel=args.kernel), dtype=torch.uint8,
                         device=dev)
        sel = torch.empty((wl.B, wl.Hkv, K), dtype=torch.int32, device=dev)

        def step(events=None, q=None, tables=None, seq_lens=None):
            t = wl.block_tables if tables is None else tables
            sl = wl.seq_lens if seq_lens is None else seq_lens
            pa.block_means(kv, t, sl, SB, M, first=last, count=1, means=means)
            pa.decode_sparse(kv, wl.q if q is None else q, t, sl, wl.softmax_scale, means, SB, K,
                             out=out, max_seq_len=maxlen, workspace=ws, kernel=args.kernel,
                             events=events)
        launches_per_step = 6      # means refresh, score, select, planner, attention, merge
        fn = "pa_decode_sparse"
        # algorithmic bytes: all mean keys scored, the refreshed blocks' keys
        # read and means written, the selected keys / values, tables, q, out
        step()
        torch.cuda.synchronize()
        _, _, selt, _ = pa.decode_sparse(kv, wl.q, wl.block_tables, wl.seq_lens,
                                         wl.softmax_scale, means, SB, K, return_lse=True,
                                         return_selected=True)
        selt = selt.cpu()
        toks = 0
        for b, L in enumerate(lens):
            for j in selt[b].flatten().tolist():
                if j >= 0:
                    toks += min((j + 1) * SB, L) - j * SB
        per_tok = kv_bytes_per_token_head(wl.dtype, wl.D)
        nsb_tot = sum((L + SB - 1) // SB for L in lens)
        refresh = sum(L - ((L + SB - 1) // SB - 1) * SB for L in lens if L > 0)
        total = (toks * per_tok                                   # selected K and V
                 + nsb_tot * wl.Hkv * wl.D * 4                    # mean keys scored
                 + refresh * wl.Hkv * per_tok // 2 + wl.B * wl.Hkv * wl.D * 4   # refresh
                 + (toks // 16) * 4 + wl.B * wl.Hq * wl.D * 4)    # tables, q, out
        # the attention kernel's own share: selected K / V, virtual tables, q, out
        ab = dict(total=total, kv=toks * per_tok, tokens=toks // wl.Hkv,
                  kernel=toks * per_tok + (toks // 16) * 4 + 2 * wl.B * wl.Hq * wl.D * 2,
                  pool=sum((L + 15) // 16 for L in lens) * 16 * wl.Hkv * per_tok)

    result = out                   # what the host reads back in the e2e loop
    wo_info = None
    if args.op == "wo":
        # attention + output projection y = o . W_O (random bf16 W_O, N(0, 1/K))
        K, N = wl.Hq * wl.D, args.wo_hidden
        gw = torch.Generator().manual_seed(77 + rank)
        wmat = (torch.randn(K, N, generator=gw) / math.sqrt(K)).to(torch.bfloat16).to(dev)
        y = torch.empty((wl.B * wl.Q, N), dtype=torch.bfloat16, device=dev)
        _, ws = pa.decode_wo(kv, wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale, wmat, y=y,
                             max_seq_len=maxlen, kernel=args.kernel)
        torch.cuda.synchronize()

        def step(events=None, q=None, tables=None, seq_lens=None):
            pa.decode_wo(kv, wl.q if q is None else q,
                         wl.block_tables if tables is None else tables,
                         wl.seq_lens if seq_lens is None else seq_lens, wl.softmax_scale, wmat,
                         y=y, max_seq_len=maxlen, workspace=ws, kernel=args.kernel,
                         events=events)
        launches_per_step = 5      # planner, attention, merge, W_O product, split reduce
        fn = fn + "_wo"
        result = y
        wo_bytes = K * N * 2 + wl.B * wl.Q * N * 2
        ab = dict(ab, total=ab["total"] + wo_bytes, kernel=ab["total"])   # the attention's own
        wo_info = {"hidden": N, "w_bytes": K * N * 2}

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    flags = pa.read_error(ws)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x}")

    # ---- device-timed region: inputs resident, steps back to back
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    # ---- the attention kernel alone: events recorded around it on its stream
    # (a separate pass, so that the events do not serialise the steps above)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in kev:          # torch creates the CUDA event on first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        step(events=kev[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    ms_step = max_over_ranks(total_ms / args.steps, world)
    kern_avg = max_over_ranks(sum(kern_ms) / len(kern_ms), world)
    launches = launches_per_step * args.steps

    # ---- end-to-end: pinned host inputs copied in, output copied out, every step
    e2e = None
    if not args.no_e2e:
        hq = wl.q.cpu().pin_memory()
        ht = wl.block_tables.cpu().pin_memory()
        hl = wl.seq_lens.cpu().pin_memory()
        dq, dt_, dl = torch.empty_like(wl.q), torch.empty_like(wl.block_tables), torch.empty_like(wl.seq_lens)
        hout = torch.empty(result.shape, dtype=result.dtype).pin_memory()
        h2d = hq.numel() * hq.element_size() + ht.numel() * 4 + hl.numel() * 4
        d2h = hout.numel() * hout.element_size()
        for _ in range(2):
            dq.copy_(hq, non_blocking=True)
            dt_.copy_(ht, non_blocking=True)
            dl.copy_(hl, non_blocking=True)
            step(q=dq, tables=dt_, seq_lens=dl)
            hout.copy_(result, non_blocking=True)
        torch.cuda.synchronize()
        barrier(world)
        s0 = time.perf_counter()
        for _ in range(args.steps):
            dq.copy_(hq, non_blocking=True)
            dt_.copy_(ht, non_blocking=True)
            dl.copy_(hl, non_blocking=True)
            step(q=dq, tables=dt_, seq_lens=dl)
            hout.copy_(result, non_blocking=True)
            torch.cuda.current_stream().synchronize()   # the host reads the result each step
        e2e_s = max_over_ranks((time.perf_counter() - s0) / args.steps, world)
        e2e = {"value": world * ab["total"] / e2e_s / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_s * 1e3,
               "resident": "KV pool (cache state, written by prefill/append)"}

    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    value = world * ab["total"] / (ms_step * 1e-3) / 1e9
    achieved = ab.get("kernel", ab["total"]) / (kern_avg * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload) if args.kernel in (0,) else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np  # noqa: F401
        nthreads = os.cpu_count() or 1
        if sparse:
            dt = oracle_sparse_sample(wl, 0, spec["sparse_block"], spec["top_k"])
            cpu = {"value": ab["total"] / wl.B / dt / 1e9, "unit": "GB/s", "cores": 1,
                   "kind": "oracle",
                   "sample": f"sequence 0 of {wl.B} of {args.workload}: selection + exact "
                             f"attention over the selected blocks (mean keys given), {dt:.1f} s"}
        else:
            bs = pick_sample(lens, args.cpu_tokens)
            dt, slens = oracle_sample(wl, bs, nthreads)
            cab = algorithmic_bytes(dict(spec, B_eff=len(bs)), slens)
            cpu = {"value": cab["total"] / dt / 1e9, "unit": "GB/s", "cores": nthreads,
                   "kind": "oracle",
                   "sample": f"{len(bs)} of {wl.B} sequences ({cab['tokens']} keys) of "
                             f"{args.workload}, fp64 two-pass softmax, {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype + "-kv/fp32-acc",
            "data": "synthetic",
            "config": {"workload": args.workload, "batch": wl.B, "q_len": wl.Q,
                       "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.D,
                       "kv_tokens": ab["tokens"], "algorithmic_bytes": ab["total"],
                       "l2": "inputs larger than L2 (KV pool %.2f GB > 129 MB)"
                             % (ab.get("pool", ab["kv"]) / 1e9),
                       "parallelism": f"replicas x{world}, no collective"},
            "kv_tokens_per_s": world * ab["tokens"] / (ms_step * 1e-3),
            "pct_of_peak": 100.0 * value / world / peak,
            "peak_gbs": peak, "peak_kind": peak_kind,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel_ms": kern_avg, "kernel": f"{fn} attention kernel",
                         "peak_kind": peak_kind},
            "gpu_launches": launches,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        if wo_info:
            line["wo"] = wo_info
        if args.batch:
            line["config"]["batch_override"] = args.batch
        if world == 1 and not args.no_per_config and args.op == "decode" and not sparse:
            del wl, kv, ws, out
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            line["per_config"] = [time_config(n, args, dev, peak, peak_kind)
                                  for n in PER_CONFIG if n != args.workload]
        print(json.dumps(line), flush=True)


# ------------------------------------------------------- other workloads

def _pool_bytes(kv) -> int:
    return sum(t.numel() * t.element_size()
               for t in (kv.k_cache, kv.v_cache, kv.k_scale, kv.v_scale) if t is not None)


def time_config(name, args, dev, peak, peak_kind):
    """Times one workload the way the headline is timed (steps back to back
    with CUDA events around all of them; the attention kernel alone with
    events recorded on its stream by the library) and returns its
    `per_config` entry.  Pools smaller than twice the L2 are rotated over
    copies, one per call, so that every call reads its KV from HBM; for them
    the device time per call is also taken from a CUDA graph of one call per
    copy, replayed (what a serving loop that captures its decode step pays)."""
    import torch

    from paged_kv_decode_07_gb300 import pa
    from paged_kv_decode_07_gb300 import workloads as W
    spec = W.spec(name)
    wl = W.make_workload(name, device=dev)
    kv0 = pa.KvCache.from_workload(wl)
    lens = wl.seq_lens.cpu().tolist()
    ab = algorithmic_bytes(dict(spec, B_eff=wl.B), lens)
    pool = _pool_bytes(kv0)
    ncopy = 1 if pool >= ROTATE_TOTAL_BYTES else -(-ROTATE_TOTAL_BYTES // pool)
    kvs = [kv0] + [pa.KvCache(kv0.dtype, kv0.k_cache.clone(), kv0.v_cache.clone(),
                              None if kv0.k_scale is None else kv0.k_scale.clone(),
                              None if kv0.v_scale is None else kv0.v_scale.clone(),
                              kv0.k_global, kv0.v_global) for _ in range(ncopy - 1)]
    call = pa.verify if wl.Q > 1 else pa.decode
    out = torch.empty((wl.B, wl.Q, wl.Hq, wl.D), dtype=torch.bfloat16, device=dev)
    maxlen = wl.max_seq_len()
    ws = torch.empty(pa.workspace_bytes(kvs[0], wl.B, wl.Q, wl.Hq, maxlen), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def step(i, events=None):
        call(kvs[i % ncopy], wl.q, wl.block_tables, wl.seq_lens, wl.softmax_scale, out=out,
             max_seq_len=maxlen, workspace=ws, events=events)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    flags = pa.read_error(ws)
    if flags:
        raise RuntimeError(f"{name}: device error flags {flags:#x}")
    steps = max(args.steps, ncopy) if ncopy > 1 else args.steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    ms_step = t0.elapsed_time(t1) / steps
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in kev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        step(i, events=kev[i])
    torch.cuda.synchronize()
    kern_ms = sum(a.elapsed_time(b) for a, b in kev) / steps
    entry = {
        "workload": name, "kv_dtype": wl.dtype, "batch": wl.B, "q_len": wl.Q,
        "kv_tokens": ab["tokens"], "algorithmic_bytes": ab["total"],
        "kernel_ms": kern_ms, "achieved_gbs": ab["total"] / (kern_ms * 1e-3) / 1e9,
        "frac": ab["total"] / (kern_ms * 1e-3) / 1e9 / peak, "peak_gbs": peak,
        "peak_kind": peak_kind,
        "step_ms": ms_step, "us_per_call": ms_step * 1e3,
        "step_gbs": ab["total"] / (ms_step * 1e-3) / 1e9,
        "kv_tokens_per_s": ab["tokens"] / (ms_step * 1e-3),
        "traffic": profiled_traffic(name),
        "l2": ("inputs larger than L2 (KV pool %.2f GB)" % (pool / 1e9)) if ncopy == 1 else
              ("%d pool copies of %.2f MB rotated, one per call (%.0f MB > L2)"
               % (ncopy, pool / 1e6, ncopy * pool / 1e6)),
    }
    if wl.Q > 1:
        flop = 0
        for L in lens:   # QK and PV over the keys each query row sees
            flop += sum(4 * wl.Hq * wl.D * (L - wl.Q + 1 + i) for i in range(wl.Q))
        entry["tflops"] = flop / (kern_ms * 1e-3) / 1e12
    if ncopy > 1:
        # one graph of one call per pool copy, replayed: device time per call
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(0)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(ncopy):
                step(i)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, args.steps // 4)
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        entry["us_per_call_graph"] = t0.elapsed_time(t1) * 1e3 / (reps * ncopy)
        entry["us_per_call"] = entry["us_per_call_graph"]
        entry["us_per_call_eager"] = ms_step * 1e3
        del g
    del kvs, kv0, wl, ws, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


# ------------------------------------------------------------- KV append

APPEND_METRIC = "paged KV append (quantise-on-write): achieved HBM GB/s and rows/s, 1×GB300"


def append_bytes(aw) -> int:
    """Algorithmic bytes of one append: bf16 K and V of every valid row in,
    their codes and scales out, and the slot mapping."""
    rows = aw.valid_rows * aw.Hkv
    return rows * (2 * aw.D * 2 + kv_bytes_per_token_head(aw.dtype, aw.D)) + aw.T * 8


def oracle_append_sample(aw, tokens: int):
    """Times the oracle's append of the first `tokens` tokens of the workload."""
    import oracle
    from paged_kv_decode_07_gb300 import workloads as W
    h = W.append_host_arrays(aw)
    cache = oracle.HostCache(aw.dtype, h["k_cache"], h["v_cache"], h["k_scale"], h["v_scale"],
                             aw.k_global, aw.v_global)
    n = min(tokens, aw.T)
    sm = h["slot_mapping"][:n]
    t0 = time.perf_counter()
    oracle.append(cache, h["k_new"][:n], h["v_new"][:n], sm)
    dt = time.perf_counter() - t0
    rows = int((sm >= 0).sum()) * aw.Hkv
    byts = rows * (2 * aw.D * 2 + kv_bytes_per_token_head(aw.dtype, aw.D)) + n * 8
    return dt, rows, byts, n


def run_append(args, world, rank):
    import torch

    from paged_kv_decode_07_gb300 import workloads as W
    name = args.workload if args.workload.startswith("append_") else "append_int8_t64k_d256"
    if args.impl == "reference":
        if rank != 0:
            return
        aw = W.make_append_workload(name, device="cpu")
        times = []
        for i in range(args.warmup + args.steps):
            dt, rows, byts, n = oracle_append_sample(aw, args.ref_tokens // 8)
            if i >= args.warmup:
                times.append(dt)
        sec = sum(times) / len(times)
        value = byts / sec / 1e9
        nthreads = 1
        print(json.dumps({
            "metric": APPEND_METRIC, "value": value, "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": name, "sample_tokens": n},
            "rows_per_s": rows / sec,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                             "sample": f"first {n} of {aw.T} tokens of {name}"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    from paged_kv_decode_07_gb300 import pa
    dev = torch.device("cuda", torch.cuda.current_device())
    spec = W.APPEND_WORKLOADS[name]
    aw = W.make_append_workload(name, device=dev, seed=1000 + spec["id"] + 7919 * rank,
                                T=args.append_tokens or None)
    kv = pa.KvCache(aw.dtype, aw.k_cache, aw.v_cache, aw.k_scale, aw.v_scale, aw.k_global,
                    aw.v_global)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    nbytes = append_bytes(aw)

    def step(k=None, v=None, sm=None, w=None):
        pa.append_kv(kv, aw.k_new if k is None else k, aw.v_new if v is None else v,
                     aw.slot_mapping if sm is None else sm, workspace=w)

    for _ in range(max(args.warmup, 3)):
        step(w=ws)
    torch.cuda.synchronize()
    flags = pa.read_error(ws)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x}")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step()                      # one kernel launch per step, no flag reset
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)

    e2e = None
    if not args.no_e2e:
        hk = aw.k_new.cpu().pin_memory()
        hv = aw.v_new.cpu().pin_memory()
        hs = aw.slot_mapping.cpu().pin_memory()
        dk, dv, ds = torch.empty_like(aw.k_new), torch.empty_like(aw.v_new), torch.empty_like(aw.slot_mapping)
        hflag = torch.empty(1, dtype=torch.int32).pin_memory()
        h2d = 2 * hk.numel() * 2 + hs.numel() * 8

        def e2e_step():
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            ds.copy_(hs, non_blocking=True)
            step(dk, dv, ds, ws)
            hflag.copy_(ws[:4].view(torch.int32), non_blocking=True)
            torch.cuda.current_stream().synchronize()   # the host reads the flags each step
        for _ in range(2):
            e2e_step()
        barrier(world)
        s0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        e2e_s = max_over_ranks((time.perf_counter() - s0) / args.steps, world)
        e2e = {"value": world * nbytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": 4, "ms_per_step": e2e_s * 1e3,
               "resident": "KV pool (written in place)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, rows, byts, n = oracle_append_sample(aw, args.ref_tokens // 8)
        cpu = {"value": byts / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n} of {aw.T} tokens of {name}, {dt:.1f} s"}
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = nbytes / (ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": APPEND_METRIC, "value": world * achieved, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16-in/" + aw.dtype + "-kv", "data": "synthetic",
            "config": {"workload": name, "tokens": aw.T, "valid_rows": aw.valid_rows * aw.Hkv,
                       "kv_heads": aw.Hkv, "head_dim": aw.D, "algorithmic_bytes": nbytes,
                       "l2": "inputs larger than L2 (new K/V %.2f GB > 129 MB)"
                             % (4 * aw.T * aw.Hkv * aw.D / 1e9),
                       "parallelism": f"replicas x{world}, no collective"},
            "rows_per_s": world * aw.valid_rows * aw.Hkv / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(name),
                         "kernel_ms": ms, "kernel": "pa_append_kv kernel (one launch per step)",
                         "peak_kind": peak_kind},
            "gpu_launches": args.steps, "clocks": clk, "e2e": e2e, "cpu_baseline": cpu}),
              flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tensor-core")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences of the headline workload (default: its recipe's; a smaller "
                         "batch of the same distribution is for profiling captures)")
    ap.add_argument("--ref-tokens", type=int, default=60000,
                    help="keys in the oracle's bounded sample")
    ap.add_argument("--cpu-tokens", type=int, default=1 << 40,
                    help="keys in the cpu_baseline sample (default: the whole workload)")
    ap.add_argument("--op", default="decode", choices=["decode", "append", "wo"],
                    help="decode: the attention step (default); append: the KV append; "
                         "wo: attention + output projection")
    ap.add_argument("--wo-hidden", type=int, default=5120,
                    help="columns of W_O for --op wo")
    ap.add_argument("--append-tokens", type=int, default=0,
                    help="tokens per append call (default: the workload's)")
    args = ap.parse_args()
    world, rank, local = dist_setup(args)
    if args.op == "append":
        run_append(args, world, rank)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
