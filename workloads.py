"""Seeded synthetic inputs for the verification step (shared by tests, bench, smoke).

This module holds no arithmetic of the verification method: it only draws
logits, draft tokens, temperatures and draft confidences.  Both the CUDA path
and the CPU oracle consume exactly these tensors.

The pages measure on production sessions and public suites (MATH-500, HumanEval,
Spec-Bench) with trained models; none of that is available, so these synthetic
logits stand in for them, using the vocabulary sizes of the model families the
pages name (Qwen3 151936, Llama 3.x 128256, gpt-oss 201088).

Workloads (sigma is a standard deviation):
  c0  B=1,   K=4,  V=32000,  float32; target ~ N(0, 2); draft = target + N(0, 0.5);
      tokens drawn from the draft softmax at T=1; run sampled (T=1) and greedy (T=0).
  c1  B=32,  K=8,  V=151936, bf16; target ~ N(0, 2.5); draft = target + N(0, 0.7); T=1;
      verify_len = 8.
  c2  B=128, K=16, V=151936, bf16; target ~ N(0, 2.5); draft row k = target + N(0, 0.3+0.1k)
      (k 0-based, a suffix-decay stand-in); T=0.8; verify_len = 16.
  c3  B=256, K=16, V=128256, bf16; target ~ N(0, 2) plus one confidence spike per row
      (one uniformly drawn token raised by U(10, 20)); draft = target + N(0, 0.6); T=0.7;
      verify_len from the confidence schedule of the draft max-probabilities, threshold 0.3.
  c4  B=512, K=8,  V=201088, bf16; target ~ N(0, 3); draft = target + N(0, 0.5);
      exactly 128 requests (a seeded random choice) greedy (T=0), the others T ~ U(0, 1.2];
      verify_len = 8.
Draft tokens: multinomial draws from softmax(draft/T) of the (rounded) draft logits;
argmax of the draft for greedy requests.
"""
import math

import torch

BASE_SEED = 20261202

CONFIGS = {
    0: dict(B=1, K=4, V=32000, dtype=torch.float32, sigma=2.0, noise=0.5, T=1.0),
    1: dict(B=32, K=8, V=151936, dtype=torch.bfloat16, sigma=2.5, noise=0.7, T=1.0),
    2: dict(B=128, K=16, V=151936, dtype=torch.bfloat16, sigma=2.5, noise="decay", T=0.8),
    3: dict(B=256, K=16, V=128256, dtype=torch.bfloat16, sigma=2.0, noise=0.6, T=0.7,
            spike=(10.0, 20.0), threshold=0.3),
    4: dict(B=512, K=8, V=201088, dtype=torch.bfloat16, sigma=3.0, noise=0.5, T="mixed",
            n_greedy=128, t_max=1.2),
}

NAMES = {
    0: "c0: B=1 K=4 V=32000 fp32, sampled and greedy",
    1: "c1: B=32 K=8 V=151936 bf16, T=1, verify_len 8",
    2: "c2: B=128 K=16 V=151936 bf16, T=0.8, draft noise 0.3+0.1k",
    3: "c3: B=256 K=16 V=128256 bf16, T=0.7, confidence-scheduled verify_len (threshold 0.3)",
    4: "c4: B=512 K=8 V=201088 bf16, 25% greedy, T~U(0,1.2]",
}


def seed_for(cfg: int, rep: int = 0) -> int:
    return BASE_SEED + 1000 * cfg + rep


def make_inputs(cfg: int, rep: int = 0, device="cuda", B=None, V=None, K=None, greedy=None,
                T=None):
    """Inputs of workload `cfg` (optionally shrunk: B, V, K overrides).

    Returns dict(target [B,K+1,V], draft [B,K,V], tokens int32 [B,K], temperature float32 [B],
    verify_len int32 [B] or None, draft_maxprob float32 [B,K] (c3 only), threshold (c3 only),
    seed).  greedy=True forces T=0 everywhere (c0's second mode); T overrides the temperature."""
    c = dict(CONFIGS[cfg])
    B = B or c["B"]
    V = V or c["V"]
    K = K or c["K"]
    seed = seed_for(cfg, rep)
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    target = torch.randn((B, K + 1, V), generator=g, device=dev, dtype=torch.float32)
    target.mul_(c["sigma"])
    if "spike" in c:
        lo, hi = c["spike"]
        idx = torch.randint(0, V, (B, K + 1, 1), generator=g, device=dev)
        delta = lo + (hi - lo) * torch.rand((B, K + 1, 1), generator=g, device=dev)
        target.scatter_add_(2, idx, delta)
    noise = torch.randn((B, K, V), generator=g, device=dev, dtype=torch.float32)
    if c["noise"] == "decay":
        sig = 0.3 + 0.1 * torch.arange(K, device=dev, dtype=torch.float32)
        noise.mul_(sig.view(1, K, 1))
    else:
        noise.mul_(c["noise"])
    draft = noise.add_(target[:, :K])
    target = target.to(c["dtype"])
    draft = draft.to(c["dtype"])

    # temperatures
    if c["T"] == "mixed":
        temp = c["t_max"] * (1.0 - torch.rand((B,), generator=g, device=dev))  # (0, t_max]
        n_greedy = max(0, min(B, round(c["n_greedy"] * B / c["B"])))
        perm = torch.randperm(B, generator=g, device=dev)
        temp[perm[:n_greedy]] = 0.0
    else:
        temp = torch.full((B,), float(c["T"]), device=dev)
    if T is not None:
        temp.fill_(float(T))
    if greedy:
        temp.zero_()
    temp = temp.to(torch.float32).contiguous()

    # draft tokens from the draft softmax at each request's temperature
    tokens = torch.empty((B, K), dtype=torch.int64, device=dev)
    maxprob = torch.empty((B, K), dtype=torch.float32, device=dev)
    chunk = max(1, (1 << 26) // (K * V))
    for b0 in range(0, B, chunk):
        b1 = min(B, b0 + chunk)
        d = draft[b0:b1].float()
        tb = temp[b0:b1].view(-1, 1, 1)
        sampled = tb > 0
        probs = torch.softmax(d / torch.where(sampled, tb, torch.ones_like(tb)), dim=-1)
        maxprob[b0:b1] = probs.max(dim=-1).values
        draws = torch.multinomial(probs.view(-1, V), 1, generator=g).view(b1 - b0, K)
        amax = d.argmax(dim=-1)
        tokens[b0:b1] = torch.where(sampled.view(-1, 1), draws, amax)
    out = dict(target=target.contiguous(), draft=draft.contiguous(),
               tokens=tokens.to(torch.int32).contiguous(), temperature=temp,
               verify_len=None, seed=seed)
    if cfg != 3:
        out["verify_len"] = torch.full((B,), K, dtype=torch.int32, device=dev)
    if "threshold" in c:
        out["draft_maxprob"] = maxprob.contiguous()
        out["threshold"] = c["threshold"]
    return out


def make_tree_inputs(B, N, V, dtype=torch.bfloat16, seed=0, T=1.0, sigma=2.5, noise=0.7,
                     chain_prob=0.5, n_greedy=0, device="cuda", distinct=False):
    """Seeded candidate trees: target [B, N, V] ~ N(0, sigma); draft [B, N-1, V] =
    target rows + N(0, noise); node n >= 1 hangs under node n - 1 with
    probability chain_prob, else under a uniformly drawn earlier node; its
    token is a multinomial draw from softmax(draft row of its parent / T)
    (independently for siblings), the argmax of that row for greedy requests.
    distinct: siblings are drawn one after another without replacement (a
    node's draw excludes the tokens of its earlier siblings), the top-k style
    candidates.  The first n_greedy requests are greedy (T = 0).  Returns
    dict(target, draft, parent, tokens, temperature, seed)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(int(seed))
    target = (torch.randn((B, N, V), generator=g, device=dev) * sigma).to(dtype)
    draft = (target[:, :max(N - 1, 0)].float()
             + torch.randn((B, max(N - 1, 0), V), generator=g, device=dev) * noise).to(dtype)
    gc = torch.Generator().manual_seed(int(seed) + 1)
    parent = torch.full((B, N), -1, dtype=torch.int64)
    for n in range(1, N):
        chain = torch.rand((B,), generator=gc) < chain_prob
        anyp = torch.randint(0, n, (B,), generator=gc)
        parent[:, n] = torch.where(chain, torch.full((B,), n - 1), anyp)
    temp = torch.full((B,), float(T), dtype=torch.float32, device=dev)
    temp[:n_greedy] = 0.0
    tokens = torch.zeros((B, N), dtype=torch.int64, device=dev)
    if N > 1:
        par = parent[:, 1:].to(dev)
        chunk = max(1, (1 << 26) // ((N - 1) * V))
        for b0 in range(0, B, chunk):
            b1 = min(B, b0 + chunk)
            rows = torch.gather(draft[b0:b1], 1,
                                par[b0:b1].view(b1 - b0, N - 1, 1).expand(-1, -1, V)).float()
            tb = temp[b0:b1].view(-1, 1, 1)
            sampled = tb > 0
            probs = torch.softmax(rows / torch.where(sampled, tb, torch.ones_like(tb)), dim=-1)
            if distinct:  # node by node, without the earlier siblings' tokens
                par_c = parent[b0:b1, 1:]
                draws = torch.zeros((b1 - b0, N - 1), dtype=torch.int64, device=dev)
                for j in range(N - 1):
                    pj = probs[:, j].clone()
                    for i in range(j):
                        same = (par_c[:, i] == par_c[:, j]).to(dev)
                        pj[same, draws[same, i]] = 0.0
                    empty = pj.sum(dim=-1) <= 0
                    pj[empty] = 1.0  # no mass left (a tiny vocabulary): any token
                    draws[:, j] = torch.multinomial(pj, 1, generator=g).view(-1)
            else:
                draws = torch.multinomial(probs.view(-1, V), 1, generator=g).view(b1 - b0, N - 1)
            tokens[b0:b1, 1:] = torch.where(sampled.view(-1, 1), draws, rows.argmax(dim=-1))
    return dict(target=target.contiguous(), draft=draft.contiguous(),
                parent=parent.to(torch.int32).to(dev).contiguous(),
                tokens=tokens.to(torch.int32).contiguous(), temperature=temp, seed=int(seed) * 7 + 3)


def algorithmic_bytes(temperature, verify_len, V, esize):
    """Bytes the step must read, each needed row once: (2L+1) rows of V logits
    for a sampled request, (L+1) for a greedy one."""
    t = temperature.detach().float().cpu()
    L = verify_len.detach().cpu().long()
    sampled = (t > 0) & torch.isfinite(t) & (t >= torch.finfo(torch.float32).tiny)
    rows = torch.where(sampled, 2 * L + 1, L + 1)
    return int(rows.sum().item()) * V * esize


def verified_positions(verify_len):
    return int(verify_len.detach().cpu().long().sum().item())


def to_numpy_logits(t):
    """Host copy of logits in the oracle's layout (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()




# LM-head inputs: hidden sizes of the model families the vocabularies belong to
# (Qwen3-8B 4096, Llama-3.1-8B 4096, gpt-oss 2880).
LM_HIDDEN = {0: 256, 1: 4096, 2: 4096, 3: 4096, 4: 2880}


def make_lmhead_inputs(B, K, V, d, seed=0, T=1.0, sigma=2.5, noise=0.5, n_greedy=0, exact=False,
                       device="cuda"):
    """Seeded inputs of the LM-head path: hidden_target [B, K+1, d],
    hidden_draft [B, K, d], one shared weight w [V, d] (the drafter uses the
    target's head), all bf16, with logits of standard deviation ~sigma and
    draft logits ~ target + N(0, noise).  exact: small-integer hidden states
    and weights of +-2^-s, so every partial sum of a logit is exactly
    representable in float32 (the product's result does not depend on the
    summation order).  T: one temperature (the first n_greedy requests greedy)
    or a [B] tensor of them.  Draft tokens are drawn from the draft logits'
    softmax at each request's T (argmax for greedy requests).  Returns
    dict(hidden_target, hidden_draft, w, tokens, temperature, verify_len,
    seed)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(int(seed))
    if exact:
        s = max(0, round(math.log2(math.sqrt(4.0 * d / 3.0) / sigma)))
        ht = torch.randint(-2, 3, (B, K + 1, d), generator=g, device=dev).float()
        w = torch.randint(-1, 2, (V, d), generator=g, device=dev).float() * (2.0 ** -s)
        flip = torch.rand((B, K, d), generator=g, device=dev) < 0.1
        step = torch.randint(-1, 2, (B, K, d), generator=g, device=dev).float()
        hd = ht[:, :K] + torch.where(flip, step, torch.zeros_like(step))
    else:
        ht = torch.randn((B, K + 1, d), generator=g, device=dev)
        w = torch.randn((V, d), generator=g, device=dev) * (sigma / math.sqrt(d))
        hd = ht[:, :K] + torch.randn((B, K, d), generator=g, device=dev) * (noise / sigma)
    ht, hd, w = ht.to(torch.bfloat16), hd.to(torch.bfloat16), w.to(torch.bfloat16)
    if torch.is_tensor(T):  # per-request temperatures given
        temp = T.to(device=dev, dtype=torch.float32).clone()
    else:
        temp = torch.full((B,), float(T), dtype=torch.float32, device=dev)
        temp[:n_greedy] = 0.0
    tokens = torch.empty((B, K), dtype=torch.int64, device=dev)
    chunk = max(1, (1 << 26) // (K * V))
    wf = w.float()
    for b0 in range(0, B, chunk):
        b1 = min(B, b0 + chunk)
        z = hd[b0:b1].float() @ wf.t()
        tb = temp[b0:b1].view(-1, 1, 1)
        sampled = tb > 0
        probs = torch.softmax(z / torch.where(sampled, tb, torch.ones_like(tb)), dim=-1)
        draws = torch.multinomial(probs.view(-1, V), 1, generator=g).view(b1 - b0, K)
        tokens[b0:b1] = torch.where(sampled.view(-1, 1), draws, z.argmax(dim=-1))
    return dict(hidden_target=ht.contiguous(), hidden_draft=hd.contiguous(), w=w.contiguous(),
                tokens=tokens.to(torch.int32).contiguous(), temperature=temp,
                verify_len=torch.full((B,), K, dtype=torch.int32, device=dev), seed=int(seed) * 5 + 1)


def workload_temperatures(cfg, B, device="cuda"):
    """The per-request temperatures of workload cfg, drawn as make_inputs
    draws them (c4: a quarter greedy, the others U(0, t_max])."""
    c = CONFIGS[cfg]
    dev = torch.device(device)
    if c["T"] != "mixed":
        return torch.full((B,), float(c["T"]), dtype=torch.float32, device=dev)
    g = torch.Generator(device=dev).manual_seed(seed_for(cfg, 0) + 17)
    temp = c["t_max"] * (1.0 - torch.rand((B,), generator=g, device=dev))
    n_greedy = max(0, min(B, round(c["n_greedy"] * B / c["B"])))
    temp[torch.randperm(B, generator=g, device=dev)[:n_greedy]] = 0.0
    return temp.contiguous()


def bf16_bits(t):
    """Host copy of a bf16 tensor as its uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
