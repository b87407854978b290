"""Failure detection on the GPU without a fault: a capped wait that runs out.

Every wait of the attention kernels on a copy or a peer is capped; when the
cap is reached the kernel records PA_ERRF_WAIT_TIMEOUT in the workspace
header, lets the copies it issued land, and returns, so the context stays
usable.  The test option PA_TEST_EXPIRE_WAIT makes the tensor-core decode
kernel withhold the copy of each warp's first block (nothing ever arrives on
that barrier) and cap the wait for it at about a thousand polls.  The call
must return, the host must read the flag, and the next ordinary call on the
same workspace must be correct and flag-free.
"""
import pytest
import torch

from paged_kv_decode_07_gb300 import pa
from paged_kv_decode_07_gb300 import workloads as W
from tests.gpu_helpers import compare, compare_lse, oracle_rows, run

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("kernel", [2, 5])   # planned split-K, single launch
@pytest.mark.parametrize("name", ["bf16_skewed_b256_l16_128k_d256", "int8_b32_l1k_32k_d256",
                                  "nvfp4_b4_l262k_d256", "fp8_b32_l1k_32k_d256"])
def test_expired_wait_is_reported_and_the_context_stays_usable(name, kernel):
    wl = W.make_workload(name, device=DEV, seq_lens=[3000, 17, 640, 1])
    out, ws = run(wl, kernel=kernel, test_flags=pa.PA_TEST_EXPIRE_WAIT)
    torch.cuda.synchronize()                      # returns: no hang, no fault
    flags = pa.read_error(ws)
    assert flags & pa.PA_ERRF_WAIT_TIMEOUT, f"flags {flags:#x}"
    assert flags & ~pa.PA_ERRF_WAIT_TIMEOUT == 0, f"flags {flags:#x}"
    # the same workspace, an ordinary call: correct and no flags
    o32, lse, _ = run(wl, out_fp32=True, return_lse=True, kernel=kernel, workspace=ws)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    ref_o, ref_l = oracle_rows(wl)
    compare(o32, ref_o, f"{name} after an expired wait")
    compare_lse(lse, ref_l, f"{name} after an expired wait")
