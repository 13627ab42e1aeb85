"""spec_verify_noalloc: the entry point for callers that cannot allocate device
memory at the call site (no workspace argument; the library's static scratch
array is used instead).

The GPU test calls it through the C ABI twice in a row, on two different
batches, and checks each result against spec_verify with a caller-provided
workspace: tokens and accept lengths are integers, so they must be identical.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads


def _lib():
    import speculative_decoding_verification_69_gb300 as sv
    return sv, sv.load_library()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_rejects_oversize_on_host():
    """Sizes whose workspace exceeds the static scratch are refused before any
    CUDA call (safe without a GPU)."""
    sv, L = _lib()
    B, K, V = 4096, 32, 1 << 20
    assert L.spec_verify_workspace_bytes(B, K, V, sv.DTYPE_BF16) > sv.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    st = L.spec_verify_noalloc(fake, fake, sv.DTYPE_BF16, fake, None, fake, 1, B, K, V, fake, fake,
                               None, None)
    assert st == 4  # SPEC_ERR_WORKSPACE
    assert L.spec_verify_noalloc(fake, fake, sv.DTYPE_BF16, fake, None, fake, 1, 0, K, V, fake,
                                 fake, None, None) == 1


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_two_calls():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    sv, L = _lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for rep in range(2):  # two calls in a row on different inputs
        inp = workloads.make_inputs(1, rep=40 + rep)
        B, K1, V = inp["target"].shape
        K = K1 - 1
        assert L.spec_verify_workspace_bytes(B, K, V, sv.DTYPE_BF16) <= sv.NOALLOC_SCRATCH_BYTES
        out_n = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
        acc_n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        st_n = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = L.spec_verify_noalloc(_p(inp["target"]), _p(inp["draft"]), sv.DTYPE_BF16,
                                   _p(inp["tokens"]), _p(inp["verify_len"]),
                                   _p(inp["temperature"]), inp["seed"], B, K, V, _p(out_n),
                                   _p(acc_n), _p(st_n), stream)
        assert rc == 0, L.spec_status_str(rc)
        out_w, acc_w = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                                 inp["temperature"], inp["seed"])
        torch.cuda.synchronize()
        assert int(st_n.item()) == 0
        assert np.array_equal(out_n.cpu().numpy(), out_w.cpu().numpy())
        assert np.array_equal(acc_n.cpu().numpy(), acc_w.cpu().numpy())
        assert (acc_n.cpu().numpy() >= 0).all()


@pytest.mark.gpu
def test_noalloc_binding_matches_verify():
    """The same entry point through the Python binding (argument marshalling
    only), on the mixed greedy / sampled recipe of the B=512 workload shrunk to
    64 requests: identical tokens and accept lengths, no status bit."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    sv, L = _lib()
    inp = workloads.make_inputs(4, rep=41, B=64)
    B, K1, V = inp["target"].shape
    assert L.spec_verify_workspace_bytes(B, K1 - 1, V, sv.DTYPE_BF16) <= sv.NOALLOC_SCRATCH_BYTES
    args = (inp["target"], inp["draft"], inp["tokens"], inp["verify_len"], inp["temperature"],
            inp["seed"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, a1 = sv.verify_noalloc(*args, dev_status=st)
    o2, a2 = sv.verify(*args)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(a1, a2)
    t = inp["temperature"].cpu()
    assert (t == 0).any() and (t > 0).any()  # both paths exercised
