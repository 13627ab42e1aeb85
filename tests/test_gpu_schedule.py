"""Confidence-scheduled verification on the GPU: the draft confidences
(spec_draft_confidence) against the oracle within 1e-5 relative, and the
load-aware schedule (spec_schedule_budget) bit-exact against the oracle's sort,
including ties, clamped and NaN probabilities and the edge budgets."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import speculative_decoding_verification_69_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("cfg,n", [(3, 24), (4, 24), (0, 1)])
def test_draft_confidence_against_oracle(sv, cfg, n):
    inp = workloads.make_inputs(cfg, rep=2)
    got = sv.draft_confidence(inp["draft"], inp["temperature"]).cpu().numpy()
    ref = oracle.draft_confidence(workloads.to_numpy_logits(inp["draft"][:n]),
                                  inp["temperature"][:n].cpu().numpy())
    assert np.allclose(got[:n], ref, rtol=1e-5, atol=0.0), np.abs(got[:n] / ref - 1).max()
    greedy = np.array([oracle.is_greedy(t) for t in inp["temperature"].cpu().numpy()])
    assert (got[greedy] == 1.0).all()
    assert ((got > 0) & (got <= 1.0 + 1e-6)).all()


def test_draft_confidence_shapes(sv):
    """Odd vocabularies (vector path with bounds), fp32, -inf entries."""
    g = torch.Generator(device="cuda").manual_seed(21)
    for B, K, V, dt in [(3, 2, 1001, torch.bfloat16), (2, 5, 999, torch.float32),
                        (4, 3, 16384 + 8, torch.bfloat16)]:
        d = (torch.randn((B, K, V), generator=g, device="cuda") * 3.0).to(dt)
        d[0, 0, ::2] = float("-inf")
        T = torch.tensor([0.7, 1.3, 0.2, 2.0][:B], device="cuda")
        got = sv.draft_confidence(d.contiguous(), T).cpu().numpy()
        ref = oracle.draft_confidence(workloads.to_numpy_logits(d), T.cpu().numpy())
        assert np.allclose(got, ref, rtol=1e-5, atol=0.0), (B, K, V)


def _budget_cases():
    rng = np.random.default_rng(3)
    for B, K in [(1, 1), (7, 5), (256, 16), (4096, 32), (20000, 3)]:
        mp = rng.uniform(0.0, 1.0, size=(B, K)).astype(np.float32)
        mp[rng.random((B, K)) < 0.1] = 1.0          # ties: survival stays put
        mp[rng.random((B, K)) < 0.02] = 0.0
        if B > 1:
            mp[0, 0] = np.nan                        # counts as 0
            mp[1, 0] = 1.5                           # clamped to 1
        n = B * K
        for budget in sorted({0, 1, n // 3, n // 2, n - 1, n, n + 5}):
            yield mp, budget


def test_schedule_budget_bitexact(sv):
    for mp, budget in _budget_cases():
        got = sv.schedule_budget(torch.from_numpy(mp).cuda(), budget).cpu().numpy()
        ref = oracle.schedule_budget(mp, budget)
        assert np.array_equal(got, ref), (mp.shape, budget)
        assert got.sum() == min(max(budget, 0), mp.size)


def test_schedule_budget_equals_threshold_schedule(sv):
    """Budget = positions whose survival reaches the threshold: the GPU's
    budgeted lengths equal the GPU's threshold schedule (c3's draft
    max-probabilities)."""
    inp = workloads.make_inputs(3, rep=1)
    mp = inp["draft_maxprob"]
    L = sv.schedule_len(mp, inp["threshold"])
    got = sv.schedule_budget(mp, int(L.sum().item()))
    assert torch.equal(got, L)


def test_confidence_budget_verify_chain(sv):
    """The whole chain on the device: confidences from the draft logits, a
    budget of 5 positions per request, verification; the lengths follow the
    oracle's schedule of the same confidences."""
    inp = workloads.make_inputs(3, rep=4, B=32)
    conf = sv.draft_confidence(inp["draft"], inp["temperature"])
    B = conf.shape[0]
    vl = sv.schedule_budget(conf, 5 * B)
    assert np.array_equal(vl.cpu().numpy(), oracle.schedule_budget(conf.cpu().numpy(), 5 * B))
    out, acc = sv.verify(inp["target"], inp["draft"], inp["tokens"], vl, inp["temperature"],
                         inp["seed"])
    torch.cuda.synchronize()
    assert (acc.cpu() <= vl.cpu()).all()
