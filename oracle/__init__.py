"""CPU oracle for the speculative-decoding verification step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  It wraps ``spec_oracle.c`` (IEEE double, its own
Philox4x32-10) with ctypes and numpy; it shares no code with the CUDA path.

Every function follows the verification rule of "Спекулятивный декодинг в проде"
(kiosknews.app), section "Немного теории" ("Правило проверки", "Утверждение 1",
"Утверждение 2"), the greedy and bonus-token remarks of "speculative decoding от
черновика до проверки" (braintools.ru), section "Как это работает" and "Почему
ответ не портится", and the confidence-scheduled verify length of the DSpark
summary (iitog.ru).  See spec_oracle.c for the readings where the pages are
silent.

Parity pins (tests/test_oracle_pins.py): Philox known-answer vectors, the
hand-worked 4-token rule, exact enumeration of the output law (lossless
invariant) by bisection over the uniforms, greedy == argmax decoding, a
chi-square test of the first-token marginal, the closed-form mean accept
length, and hand cases of the schedule.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, F64 = 0, 1, 2
BAD_TOKEN, BAD_LEN = 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        f32p = ctypes.POINTER(ctypes.c_float)
        vp = ctypes.c_void_p
        L.svo_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.svo_u_accept.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        L.svo_u_accept.restype = ctypes.c_double
        L.svo_u_sample.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        L.svo_u_sample.restype = ctypes.c_double
        L.svo_is_greedy.argtypes = [ctypes.c_float]
        L.svo_accept.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double]
        L.svo_inverse_cdf.argtypes = [f64p, ctypes.c_int, ctypes.c_double, f64p]
        L.svo_sample_residual.argtypes = [f64p, f64p, ctypes.c_int, ctypes.c_double, f64p, f64p]
        L.svo_row_argmax.argtypes = [vp, ctypes.c_int, ctypes.c_int]
        L.svo_row_softmax.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_double, f64p,
                                      f64p, f64p]
        L.svo_row_intermediates.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                            ctypes.c_int, f64p, f64p, f64p]
        L.svo_verify_request_u.argtypes = [vp, vp, ctypes.c_int, i32p, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_float, f64p,
                                           f64p, i32p, f64p, vp]
        L.svo_verify_batch.argtypes = [vp, ctypes.c_size_t, vp, ctypes.c_size_t, ctypes.c_int,
                                       i32p, ctypes.c_size_t, i32p, f32p, ctypes.c_uint64,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, i32p, i32p, f64p, f64p, u32p]
        L.svo_schedule_len.argtypes = [f32p, ctypes.c_float, ctypes.c_int, ctypes.c_int, i32p]
        L.svo_verify_tree_greedy.argtypes = [vp, ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int,
                                             i32p, i32p]
        L.svo_verify_tree_greedy.restype = ctypes.c_int
        L.svo_verify_tree_u.argtypes = [vp, vp, ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_int, f64p, f64p, i32p, i32p, f64p, vp]
        L.svo_verify_tree_u.restype = ctypes.c_int
        L.svo_verify_tree_sampled.argtypes = [vp, vp, ctypes.c_int, i32p, i32p, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, f32p,
                                              ctypes.c_uint64, ctypes.c_int,
                                              i32p, i32p, i32p, f64p, f64p]
        L.svo_schedule_budget.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_longlong, i32p]
        L.svo_draft_confidence.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, f32p, f64p]
        L.svo_lm_logits.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, f64p]
        L.svo_lm_logits.restype = None
        _lib = L
    return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def dtype_code(arr):
    """Map a logits array to the oracle's dtype code.  bf16 logits are passed
    as their raw uint16 bit patterns."""
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.float64:
        return F64
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError("logits must be float32, float64 or uint16 (bf16 bits), got %s" % arr.dtype)


# ------------------------------------------------------------------- Philox

def philox4x32_10(ctr, key):
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib().svo_philox4x32_10(c, k, o)
    return [int(x) for x in o]


def u_accept(seed, b, k):
    return lib().svo_u_accept(seed, b, k)


def u_sample(seed, b, pos):
    return lib().svo_u_sample(seed, b, pos)


# ------------------------------------------------------------------- rows

def is_greedy(T):
    return bool(lib().svo_is_greedy(float(T)))


def accept(p_x, q_x, u):
    return bool(lib().svo_accept(p_x, q_x, u))


def inverse_cdf(w, u):
    w = np.ascontiguousarray(w, dtype=np.float64)
    m = ctypes.c_double()
    t = lib().svo_inverse_cdf(_ptr(w, ctypes.c_double), w.size, float(u), ctypes.byref(m))
    return t, m.value


def sample_residual(p, q, u):
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    r = np.empty_like(p)
    m = ctypes.c_double()
    t = lib().svo_sample_residual(_ptr(p, ctypes.c_double), _ptr(q, ctypes.c_double), p.size,
                                  float(u), _ptr(r, ctypes.c_double), ctypes.byref(m))
    return t, m.value


def row_argmax(row):
    row = np.ascontiguousarray(row)
    return lib().svo_row_argmax(row.ctypes.data, dtype_code(row), row.size)


def row_softmax(row, T):
    row = np.ascontiguousarray(row)
    p = np.empty(row.size, dtype=np.float64)
    m, S = ctypes.c_double(), ctypes.c_double()
    lib().svo_row_softmax(row.ctypes.data, dtype_code(row), row.size, float(T),
                          _ptr(p, ctypes.c_double), ctypes.byref(m), ctypes.byref(S))
    return p, m.value, S.value


def row_intermediates(row, T, x=-1):
    """(max of z/T, log sum exp(z/T - max), p(x)) for one row."""
    row = np.ascontiguousarray(row)
    m, ls, px = ctypes.c_double(), ctypes.c_double(), ctypes.c_double(float("nan"))
    lib().svo_row_intermediates(row.ctypes.data, dtype_code(row), row.size, float(T), int(x),
                                ctypes.byref(m), ctypes.byref(ls), ctypes.byref(px))
    return m.value, ls.value, px.value


def verify_request_u(target, draft, tokens, L, T, u_acc, u_s):
    """One request with explicit uniforms.  target [K+1,V], draft [K,V] (any
    supported dtype; draft may be None when greedy), tokens [K], u_acc [K],
    u_s [K+1] or a scalar used at every position.  Returns (out[K+1], a)."""
    target = np.ascontiguousarray(target)
    K1, V = target.shape
    K = K1 - 1
    dc = dtype_code(target)
    if draft is not None:
        draft = np.ascontiguousarray(draft, dtype=target.dtype)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    u_acc = np.ascontiguousarray(np.broadcast_to(np.asarray(u_acc, dtype=np.float64), (K,)))
    u_s = np.ascontiguousarray(np.broadcast_to(np.asarray(u_s, dtype=np.float64), (K + 1,)))
    out = np.empty(K + 1, dtype=np.int32)
    work = np.empty(3 * V, dtype=np.float64)
    a = lib().svo_verify_request_u(target.ctypes.data, None if draft is None else draft.ctypes.data,
                                   dc, _ptr(tokens, ctypes.c_int32), K, V, int(L), float(T),
                                   _ptr(u_acc, ctypes.c_double), _ptr(u_s, ctypes.c_double),
                                   _ptr(out, ctypes.c_int32), _ptr(work, ctypes.c_double), None)
    return out, a


def verify(target, draft, tokens, verify_len, temperature, seed, b0=0, b1=None, nthreads=1,
           broadcast_rows=False):
    """Batch verification with the oracle's own Philox.

    target [B,K+1,V], draft [B,K,V] (float32, float64 or uint16 bf16 bits),
    tokens [B,K] int32, verify_len [B] int32 or None (=> K), temperature [B]
    float32.  Only requests [b0, b1) are computed (Philox counters use the
    global request index).  With broadcast_rows the logits hold a single
    request ([1,K+1,V], [1,K,V]) shared by every request.

    Returns dict(out_tokens [n,K+1], accept_len [n], accept_margin [n],
    cdf_margin [n], status [n]) for the n = b1 - b0 requests."""
    target = np.ascontiguousarray(target)
    dc = dtype_code(target)
    Bt, K1, V = target.shape
    K = K1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B = tokens.shape[0]
    if draft is not None:
        draft = np.ascontiguousarray(draft)
        assert draft.dtype == target.dtype and draft.shape[1:] == (K, V)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    assert temperature.shape == (B,)
    vl = None
    if verify_len is not None:
        vl = np.ascontiguousarray(verify_len, dtype=np.int32)
        assert vl.shape == (B,)
    if b1 is None:
        b1 = B
    assert 0 <= b0 <= b1 <= B
    n = b1 - b0
    out = np.empty((n, K + 1), dtype=np.int32)
    al = np.empty(n, dtype=np.int32)
    am = np.empty(n, dtype=np.float64)
    cm = np.empty(n, dtype=np.float64)
    st = np.empty(n, dtype=np.uint32)
    ts = 0 if broadcast_rows else (K + 1) * V
    ds = 0 if broadcast_rows else K * V
    rc = lib().svo_verify_batch(
        target.ctypes.data, ts, None if draft is None else draft.ctypes.data, ds, dc,
        _ptr(tokens, ctypes.c_int32), K, None if vl is None else _ptr(vl, ctypes.c_int32),
        _ptr(temperature, ctypes.c_float), int(seed) & 0xFFFFFFFFFFFFFFFF, K, V, b0, b1,
        int(nthreads), _ptr(out, ctypes.c_int32), _ptr(al, ctypes.c_int32),
        _ptr(am, ctypes.c_double), _ptr(cm, ctypes.c_double), _ptr(st, ctypes.c_uint32))
    if rc != 0:
        raise RuntimeError("oracle verify failed (%d)" % rc)
    return dict(out_tokens=out, accept_len=al, accept_margin=am, cdf_margin=cm, status=st)


def schedule_len(draft_maxprob, threshold):
    mp = np.ascontiguousarray(draft_maxprob, dtype=np.float32)
    B, K = mp.shape
    out = np.empty(B, dtype=np.int32)
    lib().svo_schedule_len(_ptr(mp, ctypes.c_float), float(np.float32(threshold)), B, K,
                           _ptr(out, ctypes.c_int32))
    return out


def verify_tree_greedy(target, parent, token):
    """Greedy verification of one candidate tree: target [N, V] (row n predicts
    the token after node n), parent [N] (parent[0] ignored), token [N].
    Returns (out_tokens [N], out_nodes [N], accepted)."""
    target = np.ascontiguousarray(target)
    N, V = target.shape
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    token = np.ascontiguousarray(token, dtype=np.int32)
    ot = np.empty(N, dtype=np.int32)
    on = np.empty(N, dtype=np.int32)
    a = lib().svo_verify_tree_greedy(target.ctypes.data, dtype_code(target), _ptr(parent, ctypes.c_int32),
                                     _ptr(token, ctypes.c_int32), N, V, _ptr(ot, ctypes.c_int32),
                                     _ptr(on, ctypes.c_int32))
    return ot, on, a


def verify_tree_u(target, draft, parent, token, T, u_acc, u_s, distinct=False):
    """Sampled verification of one candidate tree with explicit uniforms:
    target, draft [N, V] (row n: the target / draft distribution after node n),
    parent, token [N], u_acc [N] (entry c: the uniform of candidate node c;
    entry 0 unused) and u_s [N] (entry n: the sampling uniform when node n emits)
    or scalars.  distinct: the siblings were drawn without replacement from
    their parent's draft row (each child's draft law excludes the tokens of
    the siblings rejected before it).  Returns (out_tokens [N], out_nodes [N],
    accepted)."""
    target = np.ascontiguousarray(target)
    N, V = target.shape
    draft = np.ascontiguousarray(draft, dtype=target.dtype)
    assert draft.shape == (N, V)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    token = np.ascontiguousarray(token, dtype=np.int32)
    u_acc = np.ascontiguousarray(np.broadcast_to(np.asarray(u_acc, dtype=np.float64), (N,)))
    u_s = np.ascontiguousarray(np.broadcast_to(np.asarray(u_s, dtype=np.float64), (N,)))
    ot = np.empty(N, dtype=np.int32)
    on = np.empty(N, dtype=np.int32)
    work = np.empty(3 * V, dtype=np.float64)
    a = lib().svo_verify_tree_u(target.ctypes.data, draft.ctypes.data, dtype_code(target),
                                _ptr(parent, ctypes.c_int32), _ptr(token, ctypes.c_int32), N, V,
                                float(T), 1 if distinct else 0, _ptr(u_acc, ctypes.c_double),
                                _ptr(u_s, ctypes.c_double),
                                _ptr(ot, ctypes.c_int32), _ptr(on, ctypes.c_int32),
                                _ptr(work, ctypes.c_double), None)
    return ot, on, a


def verify_tree(target, draft, parent, token, temperature, seed, b0=0, distinct=False):
    """A batch of candidate trees with the oracle's own Philox (greedy rows take
    the greedy walk): target, draft [B, N, V]; parent, token [B, N];
    temperature [B]; row b is request b0 + b (its Philox index); distinct as
    verify_tree_u.  Returns dict(out_tokens, out_nodes [B, N], accept_len,
    accept_margin, cdf_margin [B])."""
    target = np.ascontiguousarray(target)
    B, N, V = target.shape
    draft = np.ascontiguousarray(draft)
    assert draft.dtype == target.dtype and draft.shape == (B, N, V)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    token = np.ascontiguousarray(token, dtype=np.int32)
    assert parent.shape == (B, N) and token.shape == (B, N)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    ot = np.empty((B, N), dtype=np.int32)
    on = np.empty((B, N), dtype=np.int32)
    al = np.empty(B, dtype=np.int32)
    am = np.empty(B, dtype=np.float64)
    cm = np.empty(B, dtype=np.float64)
    rc = lib().svo_verify_tree_sampled(
        target.ctypes.data, draft.ctypes.data, dtype_code(target), _ptr(parent, ctypes.c_int32),
        _ptr(token, ctypes.c_int32), int(b0), B, N, V, _ptr(temperature, ctypes.c_float),
        int(seed) & 0xFFFFFFFFFFFFFFFF, 1 if distinct else 0, _ptr(ot, ctypes.c_int32),
        _ptr(on, ctypes.c_int32),
        _ptr(al, ctypes.c_int32), _ptr(am, ctypes.c_double), _ptr(cm, ctypes.c_double))
    if rc != 0:
        raise RuntimeError("oracle tree verification failed (%d)" % rc)
    return dict(out_tokens=ot, out_nodes=on, accept_len=al, accept_margin=am, cdf_margin=cm)


def schedule_budget(draft_maxprob, budget):
    """Load-aware schedule: the `budget` positions with the largest prefix
    survival probabilities (ties to the lower request, then position)."""
    mp = np.ascontiguousarray(draft_maxprob, dtype=np.float32)
    B, K = mp.shape
    out = np.empty(B, dtype=np.int32)
    lib().svo_schedule_budget(_ptr(mp, ctypes.c_float), B, K, int(budget), _ptr(out, ctypes.c_int32))
    return out


def draft_confidence(draft, temperature):
    """max_v q_k(v) of every draft row [B, K, V] at the request's temperature
    (1 for greedy requests), in float64."""
    draft = np.ascontiguousarray(draft)
    B, K, V = draft.shape
    T = np.ascontiguousarray(temperature, dtype=np.float32)
    out = np.empty((B, K), dtype=np.float64)
    lib().svo_draft_confidence(draft.ctypes.data, dtype_code(draft), B, K, V,
                               _ptr(T, ctypes.c_float), _ptr(out, ctypes.c_double))
    return out


def lm_logits(hidden, weight):
    """LM-head logits in float64: hidden [..., d] and weight [V, d] as bf16 bit
    patterns (uint16); returns [..., V] float64, z = sum_j h_j w_vj in
    ascending j."""
    h = np.ascontiguousarray(hidden, dtype=np.uint16)
    w = np.ascontiguousarray(weight, dtype=np.uint16)
    d = h.shape[-1]
    V = w.shape[0]
    assert w.shape == (V, d)
    M = h.size // d
    z = np.empty((M, V), dtype=np.float64)
    lib().svo_lm_logits(h.ctypes.data, w.ctypes.data, M, V, d, _ptr(z, ctypes.c_double))
    return z.reshape(h.shape[:-1] + (V,))


def cpu_count():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
