"""Benchmark of the verification step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic inputs
already resident in HBM: spec_schedule_len (for the confidence-scheduled
workload c3) and spec_verify.  Default workload: c4 (B=512, K=8, V=201088,
bf16, a quarter of the requests greedy, the others T ~ U(0, 1.2]); --config
picks c1-c3.  L2: every workload reads more logits per step than L2 holds, and the
timed steps cycle round-robin through several device copies of the logits, so
that at least twice the L2 size is read between two uses of the same copy:
each step starts L2-cold without a flush write (whose dirty lines would be
written back during the next step).  Two timed loops run the same steps: the
first gives the step time (nothing recorded inside a step), the second brackets
the dominant kernel with CUDA events for the roofline figure (those events end
the programmatic launch overlap around it, so its steps are slower).

Printed JSON line (rank 0):
  value     verified draft positions per second (sum of verify lengths / time)
  e2e       the same metric through the public API with the step's inputs copied
            from pinned host memory and the outputs read back, every step
  roofline  achieved HBM GB/s of the dominant kernel (algorithmic bytes per
            launch / its CUDA-event duration) against the measured copy peak
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

Multi-GPU: replicas only.  Each rank verifies its own batch (seeded by rank);
value = all ranks' positions / the max over ranks of the timed region.
--impl reference times the CPU oracle (the only reference implementation: the
pages publish no code) on the host cores, on the same workload.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

HBM_NOMINAL_GBS = 8000.0
FALLBACK_PEAK_GBS = 6800.0
def early_exit_bytes(temperature, verify_len, accept_len, K, V, esize, W):
    """Logit bytes the two-wave path reads: per request, wave [0, W) lists
    target rows 0..min(L, W-1) (0..L when L <= W) and, when sampled, draft rows
    0..min(L, W)-1; a request still open after it (L > W, no rejection below W)
    reads the rest of its rows."""
    t = temperature.detach().float().cpu()
    L = verify_len.detach().cpu().long().clamp(0, K)
    a = accept_len.detach().cpu().long()
    sampled = (t > 0) & torch.isfinite(t) & (t >= torch.finfo(torch.float32).tiny)

    def rows(k0, k1):
        t1 = torch.where(L <= k1, L, torch.full_like(L, k1 - 1))
        nt = (t1 - k0 + 1).clamp(min=0)
        nd = torch.where(sampled, (torch.minimum(L, torch.full_like(L, k1)) - k0).clamp(min=0),
                         torch.zeros_like(L))
        return nt + nd

    if W >= K:
        n = rows(0, K)
    else:
        open_ = (L > W) & (a >= W)
        n = rows(0, W) + torch.where(open_, rows(W, K), torch.zeros_like(L))
    return int(n.sum().item()) * V * esize


def logit_copies(alg_bytes, l2_bytes):
    """Copies of the logits to cycle through so that >= 2x L2 is read between
    two uses of one copy."""
    n = 2
    while (n - 1) * alg_bytes < 2 * l2_bytes:
        n += 1
    return n


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_PEAK_GBS, "fallback"


def kernel_source_hash():
    """Hash of the sources the dominant kernel (sv_pass1) is built and launched
    from: the common device header, spec_verify.cu up to the decision kernel
    (parameters, the per-request kernel, the statistics pass) and the host
    launch sequence."""
    d = os.path.join(ROOT, "speculative_decoding_verification_69_gb300", "csrc")
    with open(os.path.join(d, "sv_common.cuh"), "rb") as f:
        common = f.read()
    with open(os.path.join(d, "spec_verify.cu"), "rb") as f:
        src = f.read()
    head = src[:src.index(b"// ------------------------------------------------------------------ 3. decide")]
    a = src.index(b"static void launch_all(")
    launch = src[a:src.index(b"\n}\n", a)]
    h = hashlib.sha256()
    for part in (common, head, launch):
        h.update(part)
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, only if it was taken on the current kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(workload)
        if e and e.get("source_hash") == kernel_source_hash():
            return e.get("dram_bytes_per_launch"), e
    except Exception:
        pass
    return None, None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None
        self.window = (0.0, float("inf"))

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.perf_counter()
        while not self.lines and time.perf_counter() - t0 < 3.0:  # wait for the first sample
            time.sleep(0.01)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.perf_counter(), ln.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self, timed=None, label=None):
        """Median SM clock, max clock and active throttle reasons over the
        marked window (the whole stretch of GPU work: warm-up, timed loops and
        the end-to-end loop, so that short timed regions still get samples);
        `timed` = (t0, t1) of the timed region, whose sample count is also
        given."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = self.window
        n_timed = 0
        for ts, ln in self.lines:
            if ts < lo or ts > hi:
                continue
            if timed and timed[0] <= ts <= timed[1]:
                n_timed += 1
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        res = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
               "samples": len(sm)}
        if label:
            res["window"] = label
        if timed:
            res["timed_region_samples"] = n_timed
        return res


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle

def host_arrays(inp):
    """Host copies of one workload's inputs in the oracle's layout (made once)."""
    return dict(t=workloads.to_numpy_logits(inp["target"]), d=workloads.to_numpy_logits(inp["draft"]),
                tok=inp["tokens"].cpu().numpy(),
                vl=inp["verify_len"].cpu().numpy() if inp["verify_len"] is not None else None,
                T=inp["temperature"].cpu().numpy())


def oracle_sample(inp, max_seconds=12.0, min_requests=2, host=None):
    """Time the CPU oracle on a bounded sample of the workload's requests (all
    host cores, rows-parallel over requests).  Returns (positions/s, cores,
    sample description, seconds)."""
    import oracle
    host = host or host_arrays(inp)
    h_t, h_d, tok, vl, T = host["t"], host["d"], host["tok"], host["vl"], host["T"]
    B, K = tok.shape
    cores = oracle.cpu_count()
    nthreads = min(cores, B)
    t0 = time.perf_counter()
    oracle.verify(h_t, h_d, tok, vl, T, inp["seed"], b0=0, b1=1, nthreads=1)
    t_one = max(time.perf_counter() - t0, 1e-6)
    n = B
    if t_one * B / nthreads > max_seconds:  # a prefix of the batch fits the budget
        n = int(min(B, max(nthreads, max_seconds * nthreads / t_one)))
        nthreads = min(nthreads, n)
    pos_per_pass = int(vl[:n].clip(0, K).sum()) if vl is not None else n * K
    # the sample, repeated until the time budget is spent (at least once)
    reps, dt, r = 0, 0.0, None
    while reps == 0 or dt < max_seconds:
        t0 = time.perf_counter()
        r = oracle.verify(h_t, h_d, tok, vl, T, inp["seed"], b0=0, b1=n, nthreads=nthreads)
        dt += time.perf_counter() - t0
        reps += 1
    pos = pos_per_pass * reps
    return (pos / dt, nthreads,
            "requests 0..%d of %d x %d passes (%d verified positions), %d threads"
            % (n - 1, B, reps, pos, nthreads), dt, r)


def oracle_single_thread(inp, host, max_seconds=4.0):
    """The oracle on one host thread: requests one at a time from the start of
    the batch until the time budget is spent (at least one)."""
    import oracle
    B, K = host["tok"].shape
    vl = host["vl"]
    pos, dt, b = 0, 0.0, 0
    while b == 0 or (dt < max_seconds and b < B):
        t0 = time.perf_counter()
        oracle.verify(host["t"], host["d"], host["tok"], vl, host["T"], inp["seed"], b0=b,
                      b1=b + 1, nthreads=1)
        dt += time.perf_counter() - t0
        pos += int(min(max(int(vl[b]), 0), K)) if vl is not None else K
        b += 1
    return pos / max(dt, 1e-9), "requests 0..%d, one at a time, 1 thread (%d positions, %.2f s)" % (
        b - 1, pos, dt)


def parity_counts(o_host, a_host, r, T, window=1e-6):
    """GPU outputs of the timed steps against the oracle on the requests the CPU
    baseline verified: exact agreement, and the oracle's near-tie flags (its
    uniform within `window` of an acceptance ratio or a normalised CDF
    boundary)."""
    import numpy as np
    import oracle
    n = len(r["accept_len"])
    same = (a_host[:n] == r["accept_len"]) & np.all(o_host[:n] == r["out_tokens"], axis=1)
    greedy = np.array([oracle.is_greedy(float(t)) for t in T[:n]])
    flagged = (r["accept_margin"] < window) | (r["cdf_margin"] < window)
    samp = ~greedy
    return {"requests": int(n), "greedy": int(greedy.sum()), "sampled": int(samp.sum()),
            "greedy_mismatch": int((~same & greedy).sum()),
            "sampled_mismatch": int((~same & samp).sum()),
            "unflagged_mismatch": int((~same & samp & ~flagged).sum()),
            "near_tie_flagged": int((flagged & samp).sum()), "window": window}


# ---------------------------------------------------------------- GPU arm

def prepare(cfg, rank, device, batch=None):
    inp = workloads.make_inputs(cfg, rep=rank, device=device, B=batch)
    if "draft_maxprob" in inp:
        import speculative_decoding_verification_69_gb300 as sv
        inp["verify_len"] = sv.schedule_len(inp["draft_maxprob"], inp["threshold"])
    return inp


def run_tree(args, world, rank, local):
    """Candidate-tree verification: B requests of N-node trees (N = --tree) at
    the workload's vocabulary.  Greedy: the node rows are the workload's
    target logits and half the nodes carry their parent's argmax, so paths go
    deep.  Sampled (--tree-sampled): seeded trees whose tokens are drawn from
    their parent's draft row, target and draft rows as in the workload, at its
    temperature (c4: a quarter of the requests greedy).  Positions =
    candidate nodes verified (N - 1 per request)."""
    import numpy as np
    import speculative_decoding_verification_69_gb300 as sv
    sv.load_library()
    dev = torch.device("cuda", local)
    N = args.tree
    c = workloads.CONFIGS[args.config]
    if args.tree_sampled:
        T = c["T"] if isinstance(c["T"], float) else 1.0
        noise = c["noise"] if isinstance(c["noise"], float) else 0.5
        inp = workloads.make_tree_inputs(c["B"], N, c["V"], c["dtype"],
                                         seed=workloads.seed_for(args.config, rank), T=T,
                                         sigma=c["sigma"], noise=noise,
                                         n_greedy=c.get("n_greedy", 0), device=dev,
                                         distinct=args.distinct)
        tgt, drf = inp["target"], inp["draft"]
        parent, tok, temp, seed = inp["parent"], inp["tokens"], inp["temperature"], inp["seed"]
        B, _, V = tgt.shape
        esz = tgt.element_size()
    else:
        inp = workloads.make_inputs(args.config, rep=rank, device=dev, K=N - 1)
        tgt = inp["target"]
        B, _, V = tgt.shape
        esz = tgt.element_size()
        rng = np.random.default_rng(workloads.seed_for(args.config, rank))
        am = tgt.float().argmax(dim=-1).cpu().numpy() if N > 1 else np.zeros((B, 1), np.int64)
        parent = np.full((B, N), -1, np.int32)
        tok = np.zeros((B, N), np.int32)
        for b in range(B):
            for n in range(1, N):
                p = int(rng.integers(0, n))
                parent[b, n] = p
                tok[b, n] = am[b, p] if rng.random() < 0.5 else int(rng.integers(0, V))
        parent = torch.from_numpy(parent).to(dev)
        tok = torch.from_numpy(tok).to(dev)
        drf = None
        temp, seed = None, 0  # greedy walk: no temperatures, no uniforms
    if drf is None:
        alg_bytes = B * N * V * esz
    else:  # every target row, and the draft rows of sampled requests, once
        n_samp = int((temp > 0).sum().item())
        alg_bytes = (B * N + n_samp * (N - 1)) * V * esz
    l2_bytes = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    ncopies = logit_copies(alg_bytes, l2_bytes)
    copies = [(tgt, drf)] + [(tgt.clone(), None if drf is None else drf.clone())
                             for _ in range(ncopies - 1)]
    ws = torch.empty(max(int(sv.load_library().spec_tree_workspace_bytes(B, N, V, sv._dtype_code(tgt))), 256),
                     dtype=torch.uint8, device=dev)

    def step(i):
        t, d = copies[i % ncopies]
        if d is None:
            sv.verify_tree_greedy(t, parent, tok)
        else:
            sv.verify_tree(t, d, parent, tok, temp, seed, workspace=ws, distinct=args.distinct)

    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    t_gpu0 = time.perf_counter()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    graphs = [] if args.no_graph else capture_steps(step, ncopies, stream)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    total_s, _, t0, t1 = timed_loop(args, world, stream, step, graphs, args.warmup)
    total_s_max = max_over_ranks(total_s, world)
    positions = sum_over_ranks(B * (N - 1) * args.steps, world)
    peak, peak_kind = measured_peak()
    step_s = total_s_max / args.steps
    res = {
        "metric": "verified draft positions/s", "value": positions / total_s_max,
        "unit": "positions/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if tgt.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded logits and trees; no datasets or trained weights)",
        "config": {"workload": workloads.NAMES[args.config] + (
                       " target rows as %d-node trees" % N if drf is None else
                       " shapes, %d-node sampled trees (tokens drawn from the parent's draft row%s)"
                       % (N, ", siblings without replacement" if args.distinct else "")),
                   "B": B, "N": N, "V": V,
                   "mode": "greedy tree verification" if drf is None else
                   "tree verification (sampled requests: multi-candidate residual walk%s)"
                   % (", distinct siblings" if args.distinct else ""),
                   "logit_bytes_per_step": alg_bytes,
                   "logits_GBps": alg_bytes / step_s / 1e9,
                   "l2": "inputs larger than L2: %d copies cycled; no flush" % ncopies,
                   "timing": ("%d steps, each a replay of the CUDA graph captured from its call, "
                              "one pair of CUDA events around them" % args.steps) if graphs else
                             ("%d plain calls, one pair of CUDA events around them" % args.steps)},
        "roofline": {"bound": "hbm", "kernel": "whole step", "achieved": alg_bytes / step_s / 1e9,
                     "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                     "frac": alg_bytes / step_s / 1e9 / peak, "traffic": None},
        "e2e": tree_e2e(args, world, sv, dev, tgt, drf, parent, tok, temp, seed, N, args.distinct),
        "gpu_launches": 3 * args.steps,
    }
    clocks.mark(t_gpu0, time.perf_counter() + 0.05)
    res["clocks"] = clocks.stop(timed=(t0, t1),
                                label="warm-up, the timed loop and the end-to-end loop")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pps, cores, sample, dt = tree_oracle_sample(tgt, drf, parent, tok, temp, seed,
                                                    args.cpu_seconds, args.distinct)
        res["cpu_baseline"] = {"value": pps, "unit": "positions/s", "cores": cores,
                               "kind": "oracle", "sample": sample, "seconds": dt}
    return res


def tree_e2e(args, world, sv, dev, tgt, drf, parent, tok, temp, seed, N, distinct=False):
    """The tree metric through the public API with the step's inputs copied
    from pinned host memory and the outputs read back, every step."""
    B = tgt.shape[0]
    host = {"t": tgt.cpu().pin_memory(), "p": parent.cpu().pin_memory(), "k": tok.cpu().pin_memory()}
    if drf is not None:
        host["d"] = drf.cpu().pin_memory()
        host["T"] = temp.cpu().pin_memory()
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    h_out = torch.empty((B, N), dtype=torch.int32).pin_memory()
    h_nodes = torch.empty((B, N), dtype=torch.int32).pin_memory()
    h_acc = torch.empty((B,), dtype=torch.int32).pin_memory()
    ws = torch.empty(max(int(sv.load_library().spec_tree_workspace_bytes(B, N, tgt.shape[2],
                                                                          sv._dtype_code(tgt))), 256),
                     dtype=torch.uint8, device=dev)

    def e2e_step():
        for k, v in host.items():
            dbuf[k].copy_(v, non_blocking=True)
        if drf is None:
            o, n, a = sv.verify_tree_greedy(dbuf["t"], dbuf["p"], dbuf["k"])
        else:
            o, n, a = sv.verify_tree(dbuf["t"], dbuf["d"], dbuf["p"], dbuf["k"], dbuf["T"], seed,
                                     workspace=ws, distinct=distinct)
        h_out.copy_(o, non_blocking=True)
        h_nodes.copy_(n, non_blocking=True)
        h_acc.copy_(a, non_blocking=True)

    steps = max(1, min(args.steps, 50))
    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(world)
    for i in range(steps):
        ev[i][0].record(stream)
        e2e_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / 1e3, world)
    positions = sum_over_ranks(B * (N - 1) * steps, world)
    return {"value": positions / e2e_s, "unit": "positions/s",
            "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
            "d2h_bytes_per_step": (h_out.numel() + h_nodes.numel() + h_acc.numel()) * 4,
            "steps": steps}


def tree_oracle_sample(tgt, drf, parent, tok, temp, seed, max_seconds, distinct=False):
    """Time the CPU oracle's tree verification on a bounded sample of the
    workload's requests, one host thread per core (the oracle's C code runs
    outside the interpreter lock), requests split across the threads."""
    import numpy as np
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    B, N, V = tgt.shape
    t = workloads.to_numpy_logits(tgt)
    par, tk = parent.cpu().numpy(), tok.cpu().numpy()
    if drf is not None:
        d = workloads.to_numpy_logits(drf)
        d = np.concatenate([d, np.zeros((B, 1, V), d.dtype)], axis=1)  # the last node has no children
        T = temp.cpu().numpy()

    def run(b0, b1):
        if drf is None:
            for b in range(b0, b1):
                oracle.verify_tree_greedy(t[b], par[b], tk[b])
        else:
            oracle.verify_tree(t[b0:b1], d[b0:b1], par[b0:b1], tk[b0:b1], T[b0:b1], seed, b0=b0,
                               distinct=distinct)

    cores = oracle.cpu_count()
    t0 = time.perf_counter()
    run(0, 1)
    t_one = max(time.perf_counter() - t0, 1e-6)
    nthreads = min(cores, B)
    n = B if t_one * B / nthreads <= max_seconds else int(min(B, max(nthreads, max_seconds * nthreads / t_one)))
    nthreads = min(nthreads, n)
    bounds = [(i * n // nthreads, (i + 1) * n // nthreads) for i in range(nthreads)]
    reps, dt = 0, 0.0
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        while reps == 0 or dt < max_seconds:
            t0 = time.perf_counter()
            list(ex.map(lambda r: run(*r), bounds))
            dt += time.perf_counter() - t0
            reps += 1
    pos = n * (N - 1) * reps
    return (pos / dt, nthreads, "requests 0..%d of %d x %d passes (%d candidate nodes), %d threads"
            % (n - 1, B, reps, pos, nthreads), dt)


def lm_oracle_sample(inp, max_seconds):
    """The oracle's LM-head step (float64 logits of each request's rows, then
    its verification) on requests taken in order until the time budget is
    spent (at least one): the rows of a request are split across host threads
    (the C loops run outside the interpreter lock)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    ht = workloads.bf16_bits(inp["hidden_target"])
    hd = workloads.bf16_bits(inp["hidden_draft"])
    w = workloads.bf16_bits(inp["w"])
    tok = inp["tokens"].cpu().numpy()
    T = inp["temperature"].cpu().numpy()
    B, K1, d = ht.shape
    K = K1 - 1
    rows = [(0, k) for k in range(K + 1)] + [(1, k) for k in range(K)]
    cores = oracle.cpu_count()
    nthreads = min(cores, len(rows))
    pos, dt, b = 0, 0.0, 0
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        while b == 0 or (dt < max_seconds and b < B):
            t0 = time.perf_counter()
            z = list(ex.map(lambda r: oracle.lm_logits((ht if r[0] == 0 else hd)[b, r[1]], w), rows))
            zt = np.stack(z[:K + 1])[None]
            zd = np.stack(z[K + 1:])[None]
            oracle.verify(zt, zd, tok, None, T, inp["seed"], b0=b, b1=b + 1, broadcast_rows=True)
            dt += time.perf_counter() - t0
            pos += K
            b += 1
    return pos / dt, nthreads, ("requests 0..%d, each one's %d logit rows split over %d threads "
                                "(%d positions, %.1f s)" % (b - 1, len(rows), nthreads, pos, dt)), dt


def run_lmhead(args, world, rank, local):
    """The verification step with the LM-head product fused: hidden states of
    the K+1 target and K draft positions and the head's weights in, tokens
    out; the logits live only in the GEMM's accumulators (and, for the rows
    the sampler draws from, a recompute).  Hidden size of the workload's model
    family; synthetic normal hidden states and weights."""
    import speculative_decoding_verification_69_gb300 as sv
    sv.load_library()
    dev = torch.device("cuda", local)
    cfg = args.config
    c = workloads.CONFIGS[cfg]
    B, K, V = c["B"], c["K"], c["V"]
    d = workloads.LM_HIDDEN[cfg]
    T = workloads.workload_temperatures(cfg, B, device=dev)
    noise = c["noise"] if isinstance(c["noise"], float) else 0.5
    inp = workloads.make_lmhead_inputs(B, K, V, d, seed=workloads.seed_for(cfg, rank), T=T,
                                       sigma=c["sigma"], noise=noise, device=dev)
    ws = torch.empty(sv.lmhead_workspace_bytes(B, K, V, d), dtype=torch.uint8, device=dev)
    out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    # hidden states cycled through copies (the weights are the model's, resident)
    ncopies = 2
    copies = [(inp["hidden_target"], inp["hidden_draft"])] + [
        (inp["hidden_target"].clone(), inp["hidden_draft"].clone()) for _ in range(ncopies - 1)]

    def step(i, ht=None, hd=None):
        if ht is None:
            ht, hd = copies[i % ncopies]
        sv.verify_lmhead(ht, hd, inp["w"], inp["w"], inp["tokens"], inp["verify_len"],
                         inp["temperature"], inp["seed"], out_tokens=out_tokens,
                         accept_len=accept_len, workspace=ws)

    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    t_gpu0 = time.perf_counter()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    graphs = [] if args.no_graph else capture_steps(step, ncopies, stream)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in kev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    total_s, _, t0, t1 = timed_loop(args, world, stream, step, graphs, args.warmup)
    for i in range(args.steps):  # the statistics GEMM bracketed by events (plain calls)
        sv.profile_events(*kev[i])
        step(args.warmup + args.steps + i)
    sv.profile_events(None, None)
    torch.cuda.synchronize()
    t2 = time.perf_counter()
    a_host = accept_len.cpu().numpy()
    o_host = out_tokens.cpu().numpy()
    total_s_max = max_over_ranks(total_s, world)
    positions = B * K
    gemm_s = sum(a.elapsed_time(b) for a, b in kev) / 1e3 / args.steps
    flop_stats = 2.0 * (B * (2 * K + 1)) * d * V
    # end to end: the step's hidden states, tokens and temperatures copied in
    # from pinned host memory, the outputs read back
    host = {k: inp[k].cpu().pin_memory() for k in ("hidden_target", "hidden_draft", "tokens",
                                                   "temperature")}
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    h_out = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    h_acc = torch.empty((B,), dtype=torch.int32).pin_memory()

    def e2e_step():
        for k, v in host.items():
            dbuf[k].copy_(v, non_blocking=True)
        o, a = sv.verify_lmhead(dbuf["hidden_target"], dbuf["hidden_draft"], inp["w"], inp["w"],
                                dbuf["tokens"], inp["verify_len"], dbuf["temperature"],
                                inp["seed"], out_tokens=out_tokens, accept_len=accept_len,
                                workspace=ws)
        h_out.copy_(o, non_blocking=True)
        h_acc.copy_(a, non_blocking=True)

    e2e_steps = max(1, min(args.steps, 100))
    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(e2e_steps)]
    barrier(world)
    for i in range(e2e_steps):
        e2e_ev[i][0].record(stream)
        e2e_step()
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev) / 1e3, world)
    clocks.mark(t_gpu0, time.perf_counter() + 0.05)
    clk = clocks.stop(timed=(t0, t2), label="warm-up, both timed loops and the end-to-end loop")
    n_samp = int((inp["temperature"] > 0).sum().item())
    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops_sustained"]), "measured, sustained"
    except Exception:
        peak, peak_kind = 1700.0, "fallback, sustained"
    achieved = flop_stats / gemm_s / 1e12
    res = {
        "metric": "verified draft positions/s", "value": sum_over_ranks(positions * args.steps, world) / total_s_max,
        "unit": "positions/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_s_max * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal hidden states and LM-head weights; no trained weights)",
        "config": {"workload": workloads.NAMES[cfg] + " shapes, LM head fused (d=%d)" % d,
                   "B": B, "K": K, "V": V, "d": d,
                   "mode": "LM-head product with the row statistics in its epilogue; the "
                           "sampled requests' draw rows recomputed after the decisions",
                   "flop_per_step": flop_stats + 2.0 * 2 * n_samp * d * V,
                   "tflops_step": (flop_stats + 4.0 * n_samp * d * V) * args.steps / total_s / 1e12,
                   "logit_bytes_never_written": B * (2 * K + 1) * V * 4,
                   "l2": "weights %d bytes (larger than L2) stream once per step; hidden states "
                         "cycled through %d copies" % (V * d * 2, ncopies),
                   "timing": ("%d steps, each a replay of the CUDA graph captured from its call, "
                              "one pair of CUDA events around them" % args.steps) if graphs else
                             ("%d plain calls, one pair of CUDA events around them" % args.steps)},
        "roofline": {"bound": "tensor", "kernel": "lm_gemm<LmStatsEpi> (target and draft rows)",
                     "achieved": achieved, "peak": peak, "peak_source": peak_kind,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "algorithmic_flop_per_launch_pair": flop_stats, "kernel_ms": gemm_s * 1e3},
        "e2e": {"value": sum_over_ranks(positions * e2e_steps, world) / e2e_s, "unit": "positions/s",
                "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
                "d2h_bytes_per_step": (h_out.numel() + h_acc.numel()) * 4, "steps": e2e_steps},
        "gpu_launches": 7 * args.steps, "clocks": clk,  # shared head: 7 kernels per call
        "accept_len_hist": [int(x) for x in np.bincount(a_host, minlength=K + 1)],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pps, cores, sample, dt = lm_oracle_sample(inp, args.cpu_seconds)
        res["cpu_baseline"] = {"value": pps, "unit": "positions/s", "cores": cores,
                               "kind": "oracle", "sample": sample, "seconds": dt}
    return res


def capture_steps(step, n, stream):
    """One CUDA graph per logit copy j (step j), captured on a side stream after
    the warm-up; replaying graph i % n is step i.  The library's calls allocate
    nothing and do not synchronise, so a step captures as it is enqueued."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graphs = []
    with torch.cuda.stream(side):
        for j in range(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step(j)
            graphs.append(g)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    return graphs


def timed_loop(args, world, stream, step, graphs, first):
    """Timed region: exactly args.steps steps (graph replays, or plain calls
    without graphs) bracketed by one pair of CUDA events on the launching
    stream, with a barrier and a synchronisation on both sides.  Returns
    (seconds on the device, wall seconds, wall start, wall end)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(args.steps):
        if graphs:
            graphs[(first + i) % len(graphs)].replay()
        else:
            step(first + i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.perf_counter()
    return e0.elapsed_time(e1) / 1e3, t1 - t0, t0, t1


def run_ours(args, world, rank, local):
    import speculative_decoding_verification_69_gb300 as sv
    sv.load_library()
    dev = torch.device("cuda", local)
    cfg = args.config
    inp = prepare(cfg, rank, dev, args.batch)
    B, K1, V = inp["target"].shape
    K = K1 - 1
    esz = inp["target"].element_size()
    scheduled = "draft_maxprob" in inp
    verifier = sv.Verifier()
    out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    vlen = torch.empty((B,), dtype=torch.int32, device=dev) if scheduled else inp["verify_len"]
    stream = torch.cuda.current_stream()
    if scheduled:
        sv.schedule_len(inp["draft_maxprob"], inp["threshold"], out=vlen)
    torch.cuda.synchronize()
    positions = workloads.verified_positions(vlen)
    alg_bytes = workloads.algorithmic_bytes(inp["temperature"], vlen, V, esz)
    l2_bytes = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    ncopies = logit_copies(alg_bytes, l2_bytes)
    copies = [(inp["target"], inp["draft"])] + [
        (inp["target"].clone(), inp["draft"].clone()) for _ in range(ncopies - 1)]

    ee = args.early_exit
    chain = args.chain
    conf = torch.empty((B, K), dtype=torch.float32, device=dev)
    fused = chain or (scheduled and not ee)  # one spec_verify_scheduled call per step
    if chain:
        # confidences from the draft rows (read once; their statistics serve the
        # step too), a budget of `chain` positions per request, verification
        vlen = torch.empty((B,), dtype=torch.int32, device=dev)
        sv.verify_scheduled(inp["target"], inp["draft"], inp["tokens"], inp["temperature"],
                            inp["seed"], budget=chain * B, maxprob_out=conf, verify_len_out=vlen,
                            out_tokens=out_tokens, accept_len=accept_len, verifier=verifier)
        torch.cuda.synchronize()
        positions = workloads.verified_positions(vlen)
        t_ = inp["temperature"].float().cpu()
        n_samp = int(((t_ > 0) & torch.isfinite(t_) & (t_ >= torch.finfo(torch.float32).tiny)).sum())
        alg_bytes = (n_samp * K + int((vlen.cpu().long() + 1).sum())) * V * esz

    def step(i):
        tgt, drf = copies[i % ncopies]
        if chain:
            sv.verify_scheduled(tgt, drf, inp["tokens"], inp["temperature"], inp["seed"],
                                budget=chain * B, maxprob_out=conf, verify_len_out=vlen,
                                out_tokens=out_tokens, accept_len=accept_len, verifier=verifier)
        elif fused:  # the threshold schedule formed inside the step's first kernel
            sv.verify_scheduled(tgt, drf, inp["tokens"], inp["temperature"], inp["seed"],
                                threshold=inp["threshold"], draft_maxprob=inp["draft_maxprob"],
                                verify_len_out=vlen, out_tokens=out_tokens, accept_len=accept_len,
                                verifier=verifier)
        else:
            if scheduled:
                sv.schedule_len(inp["draft_maxprob"], inp["threshold"], out=vlen)
            verifier(tgt, drf, inp["tokens"], vlen, inp["temperature"],
                     inp["seed"], out_tokens=out_tokens, accept_len=accept_len, early_exit=ee)

    clocks = ClockSampler(local)
    clocks.start()
    t_gpu0 = time.perf_counter()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    graphs = [] if args.no_graph else capture_steps(step, ncopies, stream)
    for g in graphs:  # the replays themselves warmed up once
        g.replay()
    torch.cuda.synchronize()
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in kev:  # torch creates the CUDA event on first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    # timed region 1: the steps back to back as a serving loop issues them
    # (value, ms_per_step)
    total_s, t_wall, t_wall0, t_wall1 = timed_loop(args, world, stream, step, graphs, args.warmup)
    # timed region 2: the same steps with CUDA events bracketing the dominant
    # kernel on its stream (roofline); the events end the programmatic launch
    # overlap on both sides of it, so these steps run slower.  (Early exit runs
    # the statistics pass once per wave: its roofline is taken over the step.)
    for i in range(args.steps):
        if not ee and not chain:
            sv.profile_events(*kev[i])
        ev_k[i][0].record(stream)
        step(args.warmup + args.steps + i)
        ev_k[i][1].record(stream)
    sv.profile_events(None, None)
    torch.cuda.synchronize()
    barrier(world)
    t_wall2 = time.perf_counter()
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    step_k_ms = [a.elapsed_time(b) for a, b in ev_k]
    total_s_max = max_over_ranks(total_s, world)
    all_pos = sum_over_ranks(positions * args.steps, world)
    value = all_pos / total_s_max
    kern_avg_s = sum(kern_ms) / len(kern_ms) / 1e3
    read_bytes = alg_bytes
    if ee:  # logit bytes the two waves actually read, from each request's outcome
        read_bytes = early_exit_bytes(inp["temperature"], vlen, accept_len, K, V, esz, ee)
        kern_avg_s = total_s / args.steps
    if chain:  # two statistics passes (draft rows, then target rows): the step's rate
        kern_avg_s = total_s / args.steps

    # outcome of the timed steps (each step verifies the same batch)
    o_host = out_tokens.cpu().numpy()
    a_host = accept_len.cpu().numpy()
    accept_hist = [int(x) for x in np.bincount(a_host, minlength=K + 1)]

    # end to end through the public API: pinned host inputs -> device -> verify -> host
    host = {k: inp[k].cpu().pin_memory() for k in ("target", "draft", "tokens", "temperature")}
    if scheduled:
        host["draft_maxprob"] = inp["draft_maxprob"].cpu().pin_memory()
    elif inp["verify_len"] is not None:
        host["verify_len"] = inp["verify_len"].cpu().pin_memory()
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    h_out = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    h_acc = torch.empty((B,), dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = h_out.numel() * 4 + h_acc.numel() * 4
    # spec_verify_from_host copies only the rows the step reads; with given
    # confidences the scheduled variant forms the lengths on the device and
    # reads them back first.  Computed confidences need every draft row, and
    # early exit decides per wave: those copy whole tensors.
    from_host = not (chain or ee)
    hv = sv.HostVerifier(dev) if from_host else None
    h_vl = torch.empty((B,), dtype=torch.int32).pin_memory()

    def e2e_step():
        if from_host and scheduled:
            hv.scheduled(host["target"], host["draft"], host["tokens"], host["temperature"],
                         inp["seed"], host["draft_maxprob"], threshold=inp["threshold"],
                         out_tokens=h_out, accept_len=h_acc, verify_len_out=h_vl)
            return
        if from_host:
            hv(host["target"], host["draft"], host["tokens"], host.get("verify_len"),
               host["temperature"], inp["seed"], out_tokens=h_out, accept_len=h_acc)
            return
        for k, v in host.items():
            dbuf[k].copy_(v, non_blocking=True)
        if chain:
            o, a, _, _ = sv.verify_scheduled(
                dbuf["target"], dbuf["draft"], dbuf["tokens"], dbuf["temperature"], inp["seed"],
                budget=chain * B, maxprob_out=conf, verify_len_out=vlen, out_tokens=out_tokens,
                accept_len=accept_len, verifier=verifier)
        elif scheduled:
            o, a, _, _ = sv.verify_scheduled(
                dbuf["target"], dbuf["draft"], dbuf["tokens"], dbuf["temperature"], inp["seed"],
                threshold=inp["threshold"], draft_maxprob=dbuf["draft_maxprob"],
                verify_len_out=vlen, out_tokens=out_tokens, accept_len=accept_len,
                verifier=verifier)
        else:
            o, a = verifier(dbuf["target"], dbuf["draft"], dbuf["tokens"], dbuf.get("verify_len"),
                            dbuf["temperature"], inp["seed"], out_tokens=out_tokens,
                            accept_len=accept_len)
        h_out.copy_(o, non_blocking=True)
        h_acc.copy_(a, non_blocking=True)

    e2e_steps = max(1, min(args.steps, 100))  # each copies the batch over the host link
    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    if from_host:
        h2d = hv.last_h2d_bytes  # the rows the step reads, plus tokens, lengths, temperatures
        if scheduled:
            d2h += B * 4  # the scheduled lengths, read back before the rows are copied
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(e2e_steps)]
    barrier(world)
    for i in range(e2e_steps):
        e2e_ev[i][0].record(stream)
        e2e_step()
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev) / 1e3, world)
    e2e_value = sum_over_ranks(positions * e2e_steps, world) / e2e_s
    t_gpu1 = time.perf_counter()
    clocks.mark(t_gpu0, t_gpu1 + 0.05)
    clk = clocks.stop(timed=(t_wall0, t_wall2),
                      label="warm-up, both timed loops and the end-to-end loop")

    peak, peak_kind = measured_peak()
    achieved = read_bytes / kern_avg_s / 1e9
    traffic, _ = recorded_traffic("c%d" % cfg) if not ee else (None, None)
    if chain:
        per_step = sv.kernels_per_scheduled(True, True)
    elif fused:
        per_step = sv.kernels_per_scheduled(False, False)
    elif ee:
        per_step = (8 if ee < K else 5) + (1 if scheduled else 0)
    else:
        per_step = sv.kernels_per_verify()
    launches = per_step * args.steps  # timed region 1

    result = {
        "metric": "verified draft positions/s",
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_s_max * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if inp["target"].dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded logits; no datasets or trained weights)",
        "config": {
            "workload": workloads.NAMES[cfg] + ("" if args.batch is None else
                                                " shapes with B=%d" % B),
            "B": B, "K": K, "V": V,
            "verified_positions_per_step": positions,
            "logit_bytes_per_step": alg_bytes,
            # logit bytes the step read (early exit reads fewer rows than the single pass)
            "logits_GBps": read_bytes * args.steps / total_s / 1e9,
            "logits_frac_of_8TBps": read_bytes * args.steps / total_s / 1e9 / HBM_NOMINAL_GBS,
            "l2": ("inputs larger than L2: %d device copies of the logits cycled round-robin, "
                   "%d logit bytes read per step, L2 %d bytes; no flush" %
                   (ncopies, alg_bytes, l2_bytes)),
            "timing": ("two timed loops of the same steps: value from the first (%s, one "
                       "pair of CUDA events around the %d steps), the dominant kernel's "
                       "CUDA-event duration from the second (plain calls, events bracket the "
                       "kernel, %.4f ms per step there)"
                       % ("each step replays the CUDA graph captured from that step's call"
                          if graphs else "plain calls", args.steps,
                          sum(step_k_ms) / len(step_k_ms))),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "mode": (("early exit, first wave %d positions (%d logit bytes read per step)"
                      % (ee, read_bytes)) if ee else "single pass") + (
                     ("; one call: confidences from the draft rows (read once, their "
                      "statistics reused by the step), a budget of %d positions per request, "
                      "verification" % chain) if chain else
                     ("; one call: threshold schedule formed in the step's first kernel"
                      if fused else "")),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "whole step (logit bytes read)" if (ee or chain) else "sv_pass1",
            "achieved": achieved,
            "peak": peak,
            "peak_source": peak_kind,
            "unit": "GB/s",
            "frac": achieved / peak,
            "frac_of_8TBps": achieved / HBM_NOMINAL_GBS,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": read_bytes,
            "kernel_ms": kern_avg_s * 1e3,
        },
        "e2e": {"value": e2e_value, "unit": "positions/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": (("spec_verify_scheduled_from_host: pinned host inputs, the threshold "
                          "schedule of the given confidences formed on the device and its "
                          "lengths read back, the logit rows they need copied, outputs copied "
                          "back") if from_host and scheduled else
                         "spec_verify_from_host: pinned host inputs, the logit rows the step "
                         "reads copied to the device, outputs copied back" if from_host else
                         "pinned host tensors copied whole to the device, the call, outputs "
                         "copied back")},
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s": t_wall,
        "accept_len_hist": accept_hist,
        "emitted_tokens_per_step": int(a_host.sum()) + B,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        oinp = dict(inp, verify_len=vlen)  # the lengths the GPU verified
        host_o = host_arrays(oinp)
        pps, cores, sample, dt, r = oracle_sample(oinp, max_seconds=args.cpu_seconds, host=host_o)
        pps1, sample1 = oracle_single_thread(oinp, host_o, max_seconds=min(4.0, args.cpu_seconds))
        result["cpu_baseline"] = {"value": pps, "unit": "positions/s", "cores": cores,
                                  "kind": "oracle", "sample": sample, "seconds": dt,
                                  "single_thread": {"value": pps1, "unit": "positions/s",
                                                    "sample": sample1}}
        result["parity_sample"] = parity_counts(o_host, a_host, r, host_o["T"])
    return result


def run_reference(args, world, rank, local):
    """The CPU oracle on the machine's host cores, same workload and metric."""
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    inp = workloads.make_inputs(args.config, rep=0, device=dev)
    if "draft_maxprob" in inp:
        import oracle
        vl = oracle.schedule_len(inp["draft_maxprob"].cpu().numpy(), inp["threshold"])
        inp["verify_len"] = torch.from_numpy(vl)
    budget = min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup))
    host = host_arrays(inp)
    for _ in range(args.warmup):
        oracle_sample(inp, max_seconds=budget, host=host)
    vals, secs = [], []
    for _ in range(args.steps):
        pps, cores, sample, dt, _ = oracle_sample(inp, max_seconds=budget, host=host)
        vals.append(pps)
        secs.append(dt)
    value = statistics.median(vals)
    B, K1, V = inp["target"].shape
    return {
        "impl": "reference",
        "metric": "verified draft positions/s",
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": statistics.median(secs) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded logits; no datasets or trained weights)",
        "config": {"workload": workloads.NAMES[args.config], "B": B, "K": K1 - 1, "V": V},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chain", type=int, default=0,
                    help="per step: draft confidences, a budget of N positions per request, "
                         "then verification (N = the value given)")
    ap.add_argument("--tree", type=int, default=0,
                    help="greedy verification of N-node candidate trees instead of chains")
    ap.add_argument("--tree-sampled", action="store_true",
                    help="with --tree: sampled trees (draft rows, the workload's temperature)")
    ap.add_argument("--distinct", action="store_true",
                    help="with --tree-sampled: siblings drawn without replacement (top-k style), "
                         "verified by spec_verify_tree_distinct")
    ap.add_argument("--no-graph", action="store_true",
                    help="time plain calls instead of replays of the CUDA graphs captured from "
                         "them")
    ap.add_argument("--batch", type=int, default=None,
                    help="requests per step instead of the workload's B (smaller cases of the same "
                         "shapes, for profiler captures); the bench line then names the batch")
    ap.add_argument("--lmhead", action="store_true",
                    help="hidden states and LM-head weights in: the product on the tensor cores "
                         "with the row statistics in its epilogue (spec_verify_lmhead)")
    ap.add_argument("--early-exit", type=int, default=0,
                    help="verify positions [0, W) first, then the rest for open requests")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it; other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            local = int(os.environ.get("LOCAL_RANK", "0"))
            if torch.cuda.is_available():
                torch.cuda.set_device(local)
            world = int(os.environ.get("WORLD_SIZE", "1"))
            print(json.dumps(run_reference(args, world, 0, local)), flush=True)
        return 0
    world, rank, local = dist_setup(args.gpus)
    if args.tree:
        res = run_tree(args, world, rank, local)
    elif args.lmhead:
        res = run_lmhead(args, world, rank, local)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
