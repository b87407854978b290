"""pa_decode / pa_verify can be captured in a CUDA graph: the split plan is
computed on the device from seq_lens, nothing is allocated and the host
reads no device data.  One capture is replayed with new query values and
shorter lengths written in place, and each replay matches the oracle."""
import pytest
import torch

from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import compare, oracle_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name,fn,lens", [
    ("int8_b32_l1k_32k_d256", "decode", [2000, 517, 33, 1200]),
    ("bf16_skewed_b256_l16_128k_d256", "decode", [2000, 517, 33, 1200]),
    ("nvfp4_verify_q8_b4_ctx64k_d256", "verify", [2000, 517, 33, 1200]),
    ("fp8_verify_q8_b4_ctx64k_d256", "verify", [2000, 517, 33, 1200]),
    ("bf16_b1_l1000_d128", "decode", [1000, 517, 33, 700])])   # single-launch decode
def test_capture_and_replay_with_new_inputs(name, fn, lens):
    wl = W.make_workload(name, device=DEV, seq_lens=lens)
    kv = pa.KvCache.from_workload(wl)
    call = pa.decode if fn == "decode" else pa.verify
    maxlen = max(lens)
    out = torch.empty((wl.B, wl.Q, wl.Hq, wl.D), dtype=torch.float32, device=DEV)
    ws = torch.empty(pa.workspace_bytes(kv, wl.B, wl.Q, wl.Hq, maxlen), dtype=torch.uint8,
                     device=DEV)
    q, tables, seq = wl.q.clone(), wl.block_tables.clone(), wl.seq_lens.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(kv, q, tables, seq, wl.softmax_scale, out=out, workspace=ws, max_seq_len=maxlen)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(kv, q, tables, seq, wl.softmax_scale, out=out, workspace=ws, max_seq_len=maxlen)
    for step in range(3):
        if step > 0:   # new inputs in the same buffers
            q.copy_(torch.randn(q.shape, device=DEV, generator=torch.Generator(DEV).manual_seed(step))
                    .to(torch.bfloat16))
            seq.copy_(torch.tensor([L - 7 * step for L in lens], dtype=torch.int32))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        cur = W.Workload(**{**wl.__dict__, "q": q, "seq_lens": seq})
        ref, _ = oracle_rows(cur)
        compare(out, ref, f"{name} replay {step}")
