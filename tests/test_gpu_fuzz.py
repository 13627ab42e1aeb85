"""Seeded random shapes through the whole step, every request against the
oracle: B in [1, 80], K in [1, 32], V from 2 to 70,000 (row sizes a multiple
of 16 bytes or not), bf16 and fp32, temperatures mixed per request (greedy,
sampled, and the special values NaN, inf, 0 and a subnormal), ragged lengths
with some outside [0, K], and a few draft tokens outside [0, V).  The same
inputs also go through spec_verify_from_host and spec_verify_early_exit, whose
outputs must equal the single pass's bit for bit."""

import numpy as np
import pytest
import torch

from gpu_helpers import compare, gpu_run, host_inputs, oracle_run

pytestmark = pytest.mark.gpu

N_CASES = 160


def _case(i):
    rng = np.random.default_rng(91_000 + i)
    B = int(rng.integers(1, 81))
    K = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 32]))
    V = int(rng.choice([2, 7, 64, 1000, 1001, 4096, 4104, 8195, 32000, 70000]))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    sigma = float(rng.choice([0.5, 2.0, 6.0]))
    g = torch.Generator(device="cuda").manual_seed(5_000 + i)
    tgt = (torch.randn((B, K + 1, V), generator=g, device="cuda") * sigma).to(dtype)
    drf = (tgt[:, :K].float() + float(rng.choice([0.1, 0.5, 1.5])) *
           torch.randn((B, K, V), generator=g, device="cuda")).to(dtype)
    T = rng.choice([0.0, 0.3, 0.7, 1.0, 1.6], size=B).astype(np.float32)
    special = rng.random(B) < 0.08
    T[special] = rng.choice(np.array([np.nan, np.inf, -1.0, 1e-40], dtype=np.float32), size=int(special.sum()))
    L = rng.integers(0, K + 1, size=B).astype(np.int32)
    odd = rng.random(B) < 0.05
    L[odd] = rng.choice([-2, K + 3], size=int(odd.sum()))
    tok = np.empty((B, K), dtype=np.int32)
    probs = torch.softmax(drf.float() / 0.9, dim=-1).view(B * K, V)
    tok[:] = torch.multinomial(probs, 1, generator=g).view(B, K).to(torch.int32).cpu().numpy()
    bad = rng.random((B, K)) < 0.02
    tok[bad] = rng.choice([-1, V, V + 7], size=int(bad.sum()))
    return dict(target=tgt.contiguous(), draft=drf.contiguous(),
                tokens=torch.from_numpy(tok).cuda(), temperature=torch.from_numpy(T).cuda(),
                verify_len=torch.from_numpy(L).cuda(), seed=int(rng.integers(0, 2**63)))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i):
    import speculative_decoding_verification_69_gb300 as sv
    inp = _case(i)
    B, K1, V = inp["target"].shape
    K = K1 - 1
    gpu = gpu_run(inp)
    h = host_inputs(inp)
    idx = list(range(B))
    orc = oracle_run(h, idx)
    ng, ns, nu, nsamp, nflag = compare(gpu, orc, h, idx)
    assert ng == 0 and nu == 0, (i, ng, ns, nu, nsamp, nflag)
    assert ns <= max(1, nsamp // 100), (i, ns, nsamp)
    # host-memory inputs: the same bits
    hv = sv.HostVerifier()
    hin = {k: inp[k].cpu().pin_memory() for k in ("target", "draft", "tokens", "temperature",
                                                 "verify_len")}
    o_h, a_h = hv(hin["target"], hin["draft"], hin["tokens"], hin["verify_len"],
                  hin["temperature"], inp["seed"])
    torch.cuda.synchronize()
    assert np.array_equal(o_h.numpy(), gpu["out_tokens"]) and np.array_equal(a_h.numpy(), gpu["accept_len"])
    # two waves: the same bits
    if K >= 2:
        v = sv.Verifier()
        o_e, a_e = v(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                     inp["temperature"], inp["seed"], early_exit=max(1, K // 2))
        torch.cuda.synchronize()
        assert np.array_equal(o_e.cpu().numpy(), gpu["out_tokens"])
        assert np.array_equal(a_e.cpu().numpy(), gpu["accept_len"])
