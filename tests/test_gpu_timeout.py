"""Failure path of the bounded device waits, without a GPU fault: with the wait
limit at 0 every wait for a bulk copy that has not landed gives up at once; the
call must report SPEC_DEV_TIMEOUT in the status word (the warps still let their
copies land before exiting), and the next call with the default limit must be
correct again (the context stays usable)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import compare, gpu_run, host_inputs, oracle_run

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_recoverable():
    import speculative_decoding_verification_69_gb300 as sv
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    sv.load_library()
    inp = workloads.make_inputs(1, rep=17, B=16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        sv.set_wait_limit(0)
        out, acc = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                             inp["temperature"], inp["seed"], dev_status=st)
        torch.cuda.synchronize()
    finally:
        sv.set_wait_limit(None)
    assert int(st.item()) & sv.DEV_TIMEOUT
    acc = acc.cpu().numpy()
    assert ((acc >= 0) & (acc <= 8)).all()          # undefined but in range
    idx = list(range(16))
    gpu = gpu_run(inp)
    assert gpu["status"] == 0
    h = host_inputs(inp)
    ng, ns, nu, nsamp, nflag = compare(gpu, oracle_run(h, idx), h, idx)
    assert ng == 0 and nu == 0
