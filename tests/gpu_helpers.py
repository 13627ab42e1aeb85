"""Helpers shared by the GPU parity tests: run both paths on the same inputs
and compare them element by element."""
import numpy as np
import torch

import oracle
import workloads

# Near-tie window of the acceptance test and of the inverse CDF: a sampled
# request may differ from the oracle only when the oracle's uniform lies within
# this distance of a decision boundary (|u - p/q| or the normalised CDF).
NEAR_TIE = 1e-6
# Intermediates (row max, log-sum, p(x), q(x)): relative tolerance.
REL_TOL = 1e-5


def gpu_run(inp, debug=False, verify_len=None):
    import speculative_decoding_verification_69_gb300 as sv
    vl = inp["verify_len"] if verify_len is None else verify_len
    status = torch.zeros(1, dtype=torch.int32, device=inp["target"].device)
    if debug:
        o, a, rs, pr = sv.verify_debug(inp["target"], inp["draft"], inp["tokens"], vl,
                                       inp["temperature"], inp["seed"], dev_status=status)
    else:
        o, a = sv.verify(inp["target"], inp["draft"], inp["tokens"], vl, inp["temperature"],
                         inp["seed"], dev_status=status)
        rs = pr = None
    torch.cuda.synchronize()
    res = dict(out_tokens=o.cpu().numpy(), accept_len=a.cpu().numpy(),
               status=int(status.item()))
    if debug:
        res["row_stats"] = rs.cpu().numpy()
        res["probs"] = pr.cpu().numpy()
    return res


def host_inputs(inp, verify_len=None):
    vl = inp["verify_len"] if verify_len is None else verify_len
    return dict(target=workloads.to_numpy_logits(inp["target"]),
                draft=workloads.to_numpy_logits(inp["draft"]),
                tokens=inp["tokens"].cpu().numpy(),
                verify_len=None if vl is None else vl.cpu().numpy(),
                temperature=inp["temperature"].cpu().numpy(),
                seed=inp["seed"])


def oracle_run(h, idx, nthreads=None):
    """Oracle results for the requests in idx (sorted list of indices)."""
    nthreads = nthreads or oracle.cpu_count()
    out = dict(out_tokens={}, accept_len={}, accept_margin={}, cdf_margin={}, status={})
    # contiguous runs keep the global request index for Philox
    runs = []
    for b in idx:
        if runs and runs[-1][1] == b:
            runs[-1][1] = b + 1
        else:
            runs.append([b, b + 1])
    for b0, b1 in runs:
        r = oracle.verify(h["target"], h["draft"], h["tokens"], h["verify_len"], h["temperature"],
                          h["seed"], b0=b0, b1=b1, nthreads=min(nthreads, b1 - b0))
        for i, b in enumerate(range(b0, b1)):
            for key in out:
                out[key][b] = r[key][i]
    return out


def compare(gpu, orc, h, idx):
    """Returns (n_greedy_mismatch, n_sampled_mismatch, n_unflagged, n_sampled, n_flagged)."""
    ng = ns = nu = nsamp = nflag = 0
    for b in idx:
        greedy = oracle.is_greedy(h["temperature"][b])
        same = (gpu["accept_len"][b] == orc["accept_len"][b]
                and np.array_equal(gpu["out_tokens"][b], orc["out_tokens"][b]))
        flagged = (orc["accept_margin"][b] < NEAR_TIE) or (orc["cdf_margin"][b] < NEAR_TIE)
        if not greedy:
            nsamp += 1
            nflag += int(flagged)
        if same:
            continue
        if greedy:
            ng += 1
        else:
            ns += 1
            if not flagged:
                nu += 1
    return ng, ns, nu, nsamp, nflag


def check_intermediates(gpu, h, idx, max_rows=None):
    """Compare row max / log-sum / p(x) / q(x) of sampled requests with the
    oracle's; returns the worst relative error."""
    K = h["tokens"].shape[1]
    worst = 0.0
    n = 0
    for b in idx:
        T = float(h["temperature"][b])
        if oracle.is_greedy(T):
            continue
        L = int(gpu_len(h, b))
        for k in range(L + 1):
            rows = [(k, h["target"][b, k])]
            if k < L:
                rows.append((K + 1 + k, h["draft"][b, k]))
            for slot, row in rows:
                x = int(h["tokens"][b, k]) if k < L else -1
                m, ls, px = oracle.row_intermediates(row, T, x)
                gm, gls = gpu["row_stats"][b, slot]
                worst = max(worst, abs(gm - m) / max(abs(m), 1e-30))
                worst = max(worst, abs(gls - ls) / max(abs(ls), 1.0))
                if k < L:
                    gp = gpu["probs"][b, k, 0 if slot <= K else 1]
                    worst = max(worst, abs(gp - px) / max(abs(px), 1e-30))
                n += 1
                if max_rows and n >= max_rows:
                    return worst
    return worst


def gpu_len(h, b):
    K = h["tokens"].shape[1]
    L = K if h["verify_len"] is None else int(h["verify_len"][b])
    L = min(max(L, 0), K)
    V = h["target"].shape[2]
    for k in range(L):
        x = int(h["tokens"][b, k])
        if x < 0 or x >= V:
            return k
    return L
