"""Greedy verification of candidate trees (spec_verify_tree_greedy) against the
oracle, bit-exact: random trees over several sizes and vocabularies, chains
(which must equal the linear greedy verification), and invalid parents."""
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


def _random_trees(B, N, V, dtype, seed):
    """Trees whose tokens often follow the target's argmax (so paths go deep);
    the generator only draws numbers."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    tgt = (torch.randn((B, N, V), generator=g, device="cuda") * 2.0).to(dtype)
    rng = np.random.default_rng(seed)
    parent = np.full((B, N), -1, np.int32)
    tok = np.zeros((B, N), np.int32)
    am = tgt.float().argmax(dim=-1).cpu().numpy()
    for b in range(B):
        for n in range(1, N):
            p = int(rng.integers(0, n))
            parent[b, n] = p
            tok[b, n] = am[b, p] if rng.random() < 0.5 else int(rng.integers(0, V))
    return tgt.contiguous(), torch.from_numpy(parent).cuda(), torch.from_numpy(tok).cuda()


@pytest.mark.parametrize("B,N,V,dtype", [
    (64, 1, 1000, torch.bfloat16), (64, 2, 1000, torch.bfloat16), (32, 9, 3000, torch.float32),
    (16, 64, 4096 + 8, torch.bfloat16), (8, 33, 1001, torch.bfloat16), (4, 17, 151936, torch.bfloat16),
])
def test_random_trees_against_oracle(sv, B, N, V, dtype):
    tgt, parent, tok = _random_trees(B, N, V, dtype, seed=B * 100 + N)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nodes, acc = sv.verify_tree_greedy(tgt, parent, tok, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    h_t = workloads.to_numpy_logits(tgt)
    p, t = parent.cpu().numpy(), tok.cpu().numpy()
    out, nodes, acc = out.cpu().numpy(), nodes.cpu().numpy(), acc.cpu().numpy()
    deep = 0
    for b in range(B):
        ot, on, a = oracle.verify_tree_greedy(h_t[b], p[b], t[b])
        assert acc[b] == a and np.array_equal(out[b], ot) and np.array_equal(nodes[b], on), b
        deep = max(deep, a)
    assert N < 3 or deep >= 2  # some paths go past the first level


def test_chain_trees_equal_linear_greedy(sv):
    """A chain tree is the linear draft: same outputs as spec_verify at T = 0 on
    c4's shapes (the target rows of a K = 8 call are the chain's node rows)."""
    inp = workloads.make_inputs(4, rep=6, B=64, greedy=True)
    B, K1, V = inp["target"].shape
    out_l, acc_l = sv.verify(inp["target"], inp["draft"], inp["tokens"], inp["verify_len"],
                             inp["temperature"], inp["seed"])
    parent = torch.arange(-1, K1 - 1, dtype=torch.int32, device="cuda").expand(B, K1).contiguous()
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), inp["tokens"]], dim=1)
    out_t, nodes, acc_t = sv.verify_tree_greedy(inp["target"], parent, tok.contiguous())
    torch.cuda.synchronize()
    assert torch.equal(acc_t, acc_l) and torch.equal(out_t, out_l)


def test_invalid_parents_flagged(sv):
    tgt, parent, tok = _random_trees(4, 6, 500, torch.bfloat16, seed=3)
    parent[1, 3] = 5   # not an earlier node
    parent[2, 4] = -2
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nodes, acc = sv.verify_tree_greedy(tgt, parent.contiguous(), tok, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & sv.DEV_BAD_TREE
    h_t = workloads.to_numpy_logits(tgt)
    for b in range(4):
        ot, on, a = oracle.verify_tree_greedy(h_t[b], parent[b].cpu().numpy(), tok[b].cpu().numpy())
        assert acc[b].item() == a and np.array_equal(out[b].cpu().numpy(), ot)
