"""GB300-native verification step of speculative decoding.

Thin Python binding (ctypes) over the C ABI of libspecverify.so
(include/spec_verify.h).  The binding only marshals arguments: tensors are
passed as raw device pointers with torch's current CUDA stream; every step of
the verification runs in the library's sm_103a kernels.  There is no CPU or
PyTorch fallback: if the library is missing or fails to load, every call
raises.

    out_tokens, accept_len = verify(target, draft, tokens, verify_len, temperature, seed)
    verify_len = schedule_len(draft_maxprob, threshold)
"""
import ctypes
import os

import torch

from . import _build

SPEC_OK = 0
DTYPE_F32, DTYPE_BF16 = 0, 1
DEV_BAD_TOKEN, DEV_BAD_LEN, DEV_TIMEOUT, DEV_BAD_TREE = 1, 2, 4, 8
MAX_K = 32

_lib = None


class SpecVerifyError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libspecverify.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if _build.stale():
        _build.build()
    if not os.path.exists(path):
        raise SpecVerifyError("libspecverify.so is not built: run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    vp, i32p, f32p, u32p, f64p = (ctypes.c_void_p,) * 5
    L.spec_verify_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.spec_verify_workspace_bytes.restype = ctypes.c_size_t
    common = [vp, vp, ctypes.c_int, i32p, i32p, f32p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
              ctypes.c_int, i32p, i32p, vp, ctypes.c_size_t, u32p]
    L.spec_verify.argtypes = common + [vp]
    L.spec_verify.restype = ctypes.c_int
    L.spec_verify_debug.argtypes = common + [f64p, f64p, vp]
    L.spec_verify_debug.restype = ctypes.c_int
    L.spec_schedule_len.argtypes = [f32p, ctypes.c_float, ctypes.c_int, ctypes.c_int, i32p, vp]
    L.spec_schedule_len.restype = ctypes.c_int
    L.spec_verify_early_exit.argtypes = common[:10] + [ctypes.c_int] + common[10:] + [vp]
    L.spec_verify_early_exit.restype = ctypes.c_int
    L.spec_draft_confidence.argtypes = [vp, ctypes.c_int, f32p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, f32p, vp, ctypes.c_size_t, vp]
    L.spec_draft_confidence.restype = ctypes.c_int
    L.spec_tree_workspace_bytes.argtypes = [ctypes.c_int] * 4
    L.spec_tree_workspace_bytes.restype = ctypes.c_size_t
    L.spec_verify_tree_greedy.argtypes = [vp, ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, i32p, i32p, i32p, vp, ctypes.c_size_t, u32p, vp]
    L.spec_verify_tree_greedy.restype = ctypes.c_int
    L.spec_verify_tree.argtypes = [vp, vp, ctypes.c_int, i32p, i32p, f32p, ctypes.c_uint64,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, i32p, i32p, vp,
                                   ctypes.c_size_t, u32p, vp]
    L.spec_verify_tree.restype = ctypes.c_int
    L.spec_verify_tree_distinct.argtypes = L.spec_verify_tree.argtypes
    L.spec_verify_tree_distinct.restype = ctypes.c_int
    L.spec_schedule_budget.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_longlong, i32p, vp]
    L.spec_schedule_budget.restype = ctypes.c_int
    L.spec_verify_scheduled.argtypes = [vp, vp, ctypes.c_int, i32p, f32p, ctypes.c_uint64,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, f32p, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_longlong, f32p, i32p, i32p, i32p,
                                        vp, ctypes.c_size_t, u32p, vp]
    L.spec_verify_scheduled.restype = ctypes.c_int
    L.spec_lmhead_workspace_bytes.argtypes = [ctypes.c_int] * 4
    L.spec_lmhead_workspace_bytes.restype = ctypes.c_size_t
    L.spec_verify_lmhead.argtypes = [vp, vp, vp, vp, ctypes.c_int, i32p, i32p, f32p, ctypes.c_uint64,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, i32p, vp,
                                     ctypes.c_size_t, u32p, f64p, f64p, vp]
    L.spec_verify_lmhead.restype = ctypes.c_int
    L.spec_verify_noalloc.argtypes = common[:12] + [u32p, vp]
    L.spec_verify_noalloc.restype = ctypes.c_int
    L.spec_verify_from_host.argtypes = (common[:10] + [vp, vp, i32p, i32p, f32p, i32p, i32p, i32p, i32p,
                                                       vp, ctypes.c_size_t, u32p, vp,
                                                       ctypes.POINTER(ctypes.c_size_t)])
    L.spec_verify_from_host.restype = ctypes.c_int
    L.spec_verify_scheduled_from_host.argtypes = (
        [vp, vp, ctypes.c_int, i32p, f32p, f32p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
         ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, vp, vp, i32p, f32p, f32p,
         i32p, i32p, i32p, i32p, i32p, i32p, vp, ctypes.c_size_t, u32p, vp,
         ctypes.POINTER(ctypes.c_size_t)])
    L.spec_verify_scheduled_from_host.restype = ctypes.c_int
    L.spec_profile_events.argtypes = [vp, vp]
    L.spec_profile_events.restype = None
    L.spec_verify_kernel_count.argtypes = []
    L.spec_verify_kernel_count.restype = ctypes.c_int
    L.spec_debug_force_wait_timeout.argtypes = [ctypes.c_int]
    L.spec_debug_force_wait_timeout.restype = ctypes.c_int
    L.spec_status_str.argtypes = [ctypes.c_int]
    L.spec_status_str.restype = ctypes.c_char_p
    _lib = L
    return L


def exported_symbols():
    return ["spec_verify_workspace_bytes", "spec_verify", "spec_verify_debug",
            "spec_verify_early_exit", "spec_tree_workspace_bytes", "spec_verify_tree_greedy",
            "spec_verify_tree", "spec_verify_tree_distinct",
            "spec_draft_confidence", "spec_schedule_budget", "spec_verify_scheduled",
            "spec_lmhead_workspace_bytes", "spec_verify_lmhead",
            "spec_schedule_len", "spec_verify_noalloc", "spec_verify_from_host",
            "spec_verify_scheduled_from_host",
            "spec_profile_events", "spec_debug_force_wait_timeout",
            "spec_verify_kernel_count", "spec_status_str"]


NOALLOC_SCRATCH_BYTES = 32 << 20


def verify_noalloc(target, draft, tokens, verify_len, temperature, seed, *, out_tokens=None,
                   accept_len=None, dev_status=None, stream=None):
    """verify() on the library's static scratch (no workspace): for callers that
    cannot allocate device memory at the call site.  Pass preallocated
    out_tokens / accept_len to allocate nothing at all.  Calls on one device
    share the scratch and must not overlap on the GPU."""
    L = load_library()
    B, K, V = _prepare(target, draft, tokens, verify_len, temperature)
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if accept_len is None:
        accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(L.spec_verify_noalloc(_ptr(target), _ptr(draft), _dtype_code(target), _ptr(tokens),
                                 _ptr(verify_len), _ptr(temperature),
                                 int(seed) & 0xFFFFFFFFFFFFFFFF, B, K, V, _ptr(out_tokens),
                                 _ptr(accept_len), _ptr(dev_status), _stream(stream)))
    return out_tokens, accept_len


def profile_events(start=None, end=None):
    """Record torch.cuda.Event pairs around the dominant kernel of later calls
    (None, None switches it off)."""
    L = load_library()
    if start is None or end is None:
        L.spec_profile_events(None, None)
    else:
        L.spec_profile_events(ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(end.cuda_event))


def force_wait_timeout(enable: bool):
    """Diagnostics: make the bounded waits of later calls run out (see the header)."""
    _check(load_library().spec_debug_force_wait_timeout(1 if enable else 0))


def kernels_per_verify() -> int:
    return int(load_library().spec_verify_kernel_count())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError("logits must be bfloat16 or float32, got %s" % t.dtype)


def _check(status: int):
    if status != SPEC_OK:
        msg = load_library().spec_status_str(status).decode()
        raise SpecVerifyError("spec_verify failed: %s (%d)" % (msg, status))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_bytes(B: int, K: int, V: int, dtype=torch.bfloat16) -> int:
    code = DTYPE_BF16 if dtype == torch.bfloat16 else DTYPE_F32
    return int(load_library().spec_verify_workspace_bytes(B, K, V, code))


def _prepare(target, draft, tokens, verify_len, temperature):
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    if draft.shape != (B, K, V) or draft.dtype != target.dtype:
        raise ValueError("draft must be [B, K, V] with the target's dtype")
    if tokens.shape != (B, K) or tokens.dtype != torch.int32:
        raise ValueError("tokens must be int32 [B, K]")
    if verify_len is not None and (verify_len.shape != (B,) or verify_len.dtype != torch.int32):
        raise ValueError("verify_len must be int32 [B] or None")
    if temperature.shape != (B,) or temperature.dtype != torch.float32:
        raise ValueError("temperature must be float32 [B]")
    for t in (target, draft, tokens, temperature) + ((verify_len,) if verify_len is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    return B, K, V


class Verifier:
    """Reusable verifier: owns the workspace so repeated calls allocate nothing."""

    def __init__(self):
        self._ws = None

    def workspace(self, B, K, V, dtype, device):
        n = workspace_bytes(B, K, V, dtype)
        if self._ws is None or self._ws.numel() < n or self._ws.device != device:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        return self._ws, n

    def __call__(self, target, draft, tokens, verify_len, temperature, seed, *, out_tokens=None,
                 accept_len=None, dev_status=None, stream=None, row_stats=None, probs=None,
                 early_exit=0):
        """early_exit = W >= 1 verifies positions [0, W) first and reads the
        remaining rows only for requests still open (spec_verify_early_exit);
        0 is the single-pass spec_verify."""
        L = load_library()
        B, K, V = _prepare(target, draft, tokens, verify_len, temperature)
        dev = target.device
        if out_tokens is None:
            out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        if accept_len is None:
            accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
        ws, n = self.workspace(B, K, V, target.dtype, dev)
        args = [_ptr(target), _ptr(draft), _dtype_code(target), _ptr(tokens), _ptr(verify_len),
                _ptr(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF, B, K, V, _ptr(out_tokens),
                _ptr(accept_len), _ptr(ws), ws.numel(), _ptr(dev_status)]
        if early_exit:
            if row_stats is not None or probs is not None:
                raise ValueError("early_exit has no debug outputs")
            st = L.spec_verify_early_exit(*args[:10], int(early_exit), *args[10:], _stream(stream))
        elif row_stats is not None or probs is not None:
            st = L.spec_verify_debug(*args, _ptr(row_stats), _ptr(probs), _stream(stream))
        else:
            st = L.spec_verify(*args, _stream(stream))
        _check(st)
        return out_tokens, accept_len


class HostVerifier:
    """spec_verify for inputs in host memory (spec_verify_from_host): owns the
    device buffers and the workspace for the last shape it saw, copies only
    the logit rows the step reads, and returns the outputs in host memory.
    Host tensors should be pinned so the copies run asynchronously; the call
    is asynchronous on `stream`, so synchronise before reading the outputs or
    changing the inputs."""

    def __init__(self, device=None):
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self._key = None
        self._d = None
        self.last_h2d_bytes = 0

    def _buffers(self, B, K, V, dtype):
        key = (B, K, V, dtype)
        if self._key != key:
            dev = self.device
            n = workspace_bytes(B, K, V, dtype)
            self._d = dict(
                target=torch.empty((B, K + 1, V), dtype=dtype, device=dev),
                draft=torch.empty((B, K, V), dtype=dtype, device=dev),
                tokens=torch.empty((B, K), dtype=torch.int32, device=dev),
                verify_len=torch.empty((B,), dtype=torch.int32, device=dev),
                temperature=torch.empty((B,), dtype=torch.float32, device=dev),
                maxprob=torch.empty((B, K), dtype=torch.float32, device=dev),
                out_tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                ws=torch.empty(max(n, 256), dtype=torch.uint8, device=dev))
            self._key = key
        return self._d

    def __call__(self, target, draft, tokens, verify_len, temperature, seed, *, out_tokens=None,
                 accept_len=None, dev_status=None, stream=None):
        L = load_library()
        if target.dim() != 3:
            raise ValueError("target must be [B, K+1, V]")
        B, K1, V = target.shape
        K = K1 - 1
        host = (target, draft, tokens, temperature) + ((verify_len,) if verify_len is not None else ())
        for t in host:
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("inputs must be contiguous host tensors")
        if draft.shape != (B, K, V) or draft.dtype != target.dtype:
            raise ValueError("draft must be [B, K, V] with the target's dtype")
        if tokens.shape != (B, K) or tokens.dtype != torch.int32:
            raise ValueError("tokens must be int32 [B, K]")
        if verify_len is not None and (verify_len.shape != (B,) or verify_len.dtype != torch.int32):
            raise ValueError("verify_len must be int32 [B] or None")
        if temperature.shape != (B,) or temperature.dtype != torch.float32:
            raise ValueError("temperature must be float32 [B]")
        d = self._buffers(B, K, V, target.dtype)
        if out_tokens is None:
            out_tokens = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
        if accept_len is None:
            accept_len = torch.empty((B,), dtype=torch.int32).pin_memory()
        nbytes = ctypes.c_size_t(0)
        with torch.cuda.device(self.device):
            _check(L.spec_verify_from_host(
                _ptr(target), _ptr(draft), _dtype_code(target), _ptr(tokens), _ptr(verify_len),
                _ptr(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF, B, K, V, _ptr(d["target"]),
                _ptr(d["draft"]), _ptr(d["tokens"]), _ptr(d["verify_len"]), _ptr(d["temperature"]),
                _ptr(d["out_tokens"]), _ptr(d["accept_len"]), _ptr(out_tokens), _ptr(accept_len),
                _ptr(d["ws"]), d["ws"].numel(), _ptr(dev_status), _stream(stream),
                ctypes.byref(nbytes)))
        self.last_h2d_bytes = int(nbytes.value)
        return out_tokens, accept_len

    def scheduled(self, target, draft, tokens, temperature, seed, draft_maxprob, *,
                  threshold=None, budget=None, out_tokens=None, accept_len=None,
                  verify_len_out=None, dev_status=None, stream=None):
        """spec_verify_scheduled_from_host: lengths from the threshold or budget
        schedule of the given host confidences, formed on the device and read
        back (the call waits for them), then only the rows they need copied.
        Returns (out_tokens, accept_len, verify_len) in host memory."""
        L = load_library()
        if (threshold is None) == (budget is None):
            raise ValueError("give exactly one of threshold, budget")
        B, K1, V = target.shape
        K = K1 - 1
        for t in (target, draft, tokens, temperature, draft_maxprob):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("inputs must be contiguous host tensors")
        if draft_maxprob.shape != (B, K) or draft_maxprob.dtype != torch.float32:
            raise ValueError("draft_maxprob must be float32 [B, K]")
        d = self._buffers(B, K, V, target.dtype)
        if out_tokens is None:
            out_tokens = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
        if accept_len is None:
            accept_len = torch.empty((B,), dtype=torch.int32).pin_memory()
        if verify_len_out is None:
            verify_len_out = torch.empty((B,), dtype=torch.int32).pin_memory()
        mode = 0 if threshold is not None else 1
        nbytes = ctypes.c_size_t(0)
        with torch.cuda.device(self.device):
            _check(L.spec_verify_scheduled_from_host(
                _ptr(target), _ptr(draft), _dtype_code(target), _ptr(tokens), _ptr(temperature),
                _ptr(draft_maxprob), int(seed) & 0xFFFFFFFFFFFFFFFF, B, K, V, mode,
                float(threshold or 0.0), int(budget or 0), _ptr(d["target"]), _ptr(d["draft"]),
                _ptr(d["tokens"]), _ptr(d["temperature"]), _ptr(d["maxprob"]),
                _ptr(d["verify_len"]), _ptr(d["out_tokens"]), _ptr(d["accept_len"]),
                _ptr(out_tokens), _ptr(accept_len), _ptr(verify_len_out), _ptr(d["ws"]),
                d["ws"].numel(), _ptr(dev_status), _stream(stream), ctypes.byref(nbytes)))
        self.last_h2d_bytes = int(nbytes.value)
        return out_tokens, accept_len, verify_len_out


def draft_confidence(draft, temperature, *, out=None, stream=None, verifier=None):
    """max_v q_k(v) of every draft row [B, K, V] at the request's temperature
    (1 for greedy requests): float32 [B, K] on the device."""
    L = load_library()
    if draft.dim() != 3 or not draft.is_cuda or not draft.is_contiguous():
        raise ValueError("draft must be a contiguous CUDA tensor [B, K, V]")
    B, K, V = draft.shape
    if temperature.shape != (B,) or temperature.dtype != torch.float32 or not temperature.is_cuda:
        raise ValueError("temperature must be float32 [B] on the device")
    if out is None:
        out = torch.empty((B, K), dtype=torch.float32, device=draft.device)
    v = verifier or _default_verifier()
    ws, n = v.workspace(B, K, V, draft.dtype, draft.device)
    _check(L.spec_draft_confidence(_ptr(draft), _dtype_code(draft), _ptr(temperature), B, K, V,
                                   _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def verify_tree_greedy(target, parent, node_tokens, *, dev_status=None, stream=None):
    """Greedy verification of candidate trees: target [B, N, V] (row n: logits
    after node n), parent / node_tokens int32 [B, N].  Returns (out_tokens
    [B, N], out_nodes [B, N], accept_len [B]) on the device."""
    L = load_library()
    if target.dim() != 3 or not target.is_cuda or not target.is_contiguous():
        raise ValueError("target must be a contiguous CUDA tensor [B, N, V]")
    B, N, V = target.shape
    for t in (parent, node_tokens):
        if t.shape != (B, N) or t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("parent and node_tokens must be contiguous int32 CUDA tensors [B, N]")
    dev = target.device
    out = torch.empty((B, N), dtype=torch.int32, device=dev)
    nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    n = int(L.spec_tree_workspace_bytes(B, N, V, _dtype_code(target)))
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    _check(L.spec_verify_tree_greedy(_ptr(target), _dtype_code(target), _ptr(parent),
                                     _ptr(node_tokens), B, N, V, _ptr(out), _ptr(nodes), _ptr(acc),
                                     _ptr(ws), ws.numel(), _ptr(dev_status), _stream(stream)))
    return out, nodes, acc


def verify_tree(target, draft, parent, node_tokens, temperature, seed, *, dev_status=None,
                workspace=None, stream=None, distinct=False):
    """Verification of candidate trees at each request's temperature (greedy
    requests take the greedy walk; sampled ones check siblings against
    successively updated residuals): target [B, N, V], draft [B, N-1, V] (row
    n: the draft's logits after node n; None when N = 1), parent / node_tokens
    int32 [B, N], temperature float32 [B].  distinct: the siblings are distinct
    tokens drawn without replacement from their parent's draft row
    (spec_verify_tree_distinct).  Returns (out_tokens [B, N], out_nodes [B, N],
    accept_len [B]) on the device."""
    L = load_library()
    if target.dim() != 3 or not target.is_cuda or not target.is_contiguous():
        raise ValueError("target must be a contiguous CUDA tensor [B, N, V]")
    B, N, V = target.shape
    if N > 1:
        if (draft is None or draft.shape != (B, N - 1, V) or draft.dtype != target.dtype
                or not draft.is_cuda or not draft.is_contiguous()):
            raise ValueError("draft must be a contiguous CUDA tensor [B, N-1, V] of target's dtype")
    for t in (parent, node_tokens):
        if t.shape != (B, N) or t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("parent and node_tokens must be contiguous int32 CUDA tensors [B, N]")
    if (temperature.shape != (B,) or temperature.dtype != torch.float32 or not temperature.is_cuda
            or not temperature.is_contiguous()):
        raise ValueError("temperature must be a contiguous float32 CUDA tensor [B]")
    dev = target.device
    out = torch.empty((B, N), dtype=torch.int32, device=dev)
    nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    n = int(L.spec_tree_workspace_bytes(B, N, V, _dtype_code(target)))
    if workspace is None or workspace.numel() < n:
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    fn = L.spec_verify_tree_distinct if distinct else L.spec_verify_tree
    _check(fn(_ptr(target), _ptr(draft) if N > 1 else None, _dtype_code(target),
                              _ptr(parent), _ptr(node_tokens), _ptr(temperature),
                              int(seed) & 0xFFFFFFFFFFFFFFFF, B, N, V, _ptr(out), _ptr(nodes),
                              _ptr(acc), _ptr(workspace), workspace.numel(), _ptr(dev_status),
                              _stream(stream)))
    return out, nodes, acc


def schedule_budget(draft_maxprob, budget, *, out=None, stream=None):
    """Verify lengths keeping the `budget` positions with the largest prefix
    survival probabilities: int32 [B] on the device."""
    L = load_library()
    B, K = draft_maxprob.shape
    if draft_maxprob.dtype != torch.float32 or not draft_maxprob.is_cuda or not draft_maxprob.is_contiguous():
        raise ValueError("draft_maxprob must be a contiguous float32 CUDA tensor [B, K]")
    if out is None:
        out = torch.empty((B,), dtype=torch.int32, device=draft_maxprob.device)
    _check(L.spec_schedule_budget(_ptr(draft_maxprob), B, K, int(budget), _ptr(out), _stream(stream)))
    return out


SCHED_THRESHOLD, SCHED_BUDGET = 0, 1


def verify_scheduled(target, draft, tokens, temperature, seed, *, threshold=None, budget=None,
                     draft_maxprob=None, maxprob_out=None, verify_len_out=None, out_tokens=None,
                     accept_len=None, dev_status=None, verifier=None, stream=None):
    """Confidence-scheduled verification in one call (spec_verify_scheduled):
    exactly one of threshold (survival product >= threshold) or budget (the
    `budget` positions of highest survival).  With draft_maxprob None the
    confidences are computed from the draft rows, whose statistics the step
    then reuses.  Returns (out_tokens [B, K+1], accept_len [B], verify_len [B],
    maxprob [B, K] or None) on the device."""
    L = load_library()
    if (threshold is None) == (budget is None):
        raise ValueError("give exactly one of threshold or budget")
    B, K, V = _prepare(target, draft, tokens, None, temperature)
    dev = target.device
    if draft_maxprob is not None and (draft_maxprob.shape != (B, K) or draft_maxprob.dtype != torch.float32
                                      or not draft_maxprob.is_cuda or not draft_maxprob.is_contiguous()):
        raise ValueError("draft_maxprob must be a contiguous float32 CUDA tensor [B, K]")
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if accept_len is None:
        accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if verify_len_out is None:
        verify_len_out = torch.empty((B,), dtype=torch.int32, device=dev)
    if draft_maxprob is None and maxprob_out is None:
        maxprob_out = torch.empty((B, K), dtype=torch.float32, device=dev)
    v = verifier or _default_verifier()
    ws, n = v.workspace(B, K, V, target.dtype, dev)
    mode = SCHED_THRESHOLD if threshold is not None else SCHED_BUDGET
    _check(L.spec_verify_scheduled(_ptr(target), _ptr(draft), _dtype_code(target), _ptr(tokens),
                                   _ptr(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF, B, K, V,
                                   _ptr(draft_maxprob), mode,
                                   float(threshold) if threshold is not None else 0.0,
                                   int(budget) if budget is not None else 0,
                                   _ptr(maxprob_out) if draft_maxprob is None else None,
                                   _ptr(verify_len_out), _ptr(out_tokens), _ptr(accept_len),
                                   _ptr(ws), ws.numel(), _ptr(dev_status), _stream(stream)))
    return out_tokens, accept_len, verify_len_out, (maxprob_out if draft_maxprob is None else None)


def lmhead_workspace_bytes(B, K, V, d) -> int:
    return int(load_library().spec_lmhead_workspace_bytes(B, K, V, d))


def verify_lmhead(hidden_target, hidden_draft, w_target, w_draft, tokens, verify_len, temperature,
                  seed, *, out_tokens=None, accept_len=None, dev_status=None, workspace=None,
                  debug=False, stream=None):
    """Verification with the LM-head product fused (spec_verify_lmhead):
    hidden_target [B, K+1, d], hidden_draft [B, K, d], w_target / w_draft [V, d],
    all bf16 CUDA tensors.  Returns (out_tokens, accept_len), plus (row_stats,
    probs) with debug."""
    L = load_library()
    if hidden_target.dim() != 3:
        raise ValueError("hidden_target must be [B, K+1, d]")
    B, K1, d = hidden_target.shape
    K = K1 - 1
    V = w_target.shape[0]
    for t, shape in ((hidden_target, (B, K + 1, d)), (hidden_draft, (B, K, d)),
                     (w_target, (V, d)), (w_draft, (V, d))):
        if (t.shape != shape or t.dtype != torch.bfloat16 or not t.is_cuda
                or not t.is_contiguous()):
            raise ValueError("hidden states and weights must be contiguous bf16 CUDA tensors "
                             "[B, K+1, d], [B, K, d], [V, d], [V, d]")
    if tokens.shape != (B, K) or tokens.dtype != torch.int32 or not tokens.is_cuda:
        raise ValueError("tokens must be int32 [B, K] on the device")
    if verify_len is not None and (verify_len.shape != (B,) or verify_len.dtype != torch.int32):
        raise ValueError("verify_len must be int32 [B] or None")
    if temperature.shape != (B,) or temperature.dtype != torch.float32 or not temperature.is_cuda:
        raise ValueError("temperature must be float32 [B] on the device")
    dev = hidden_target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if accept_len is None:
        accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    n = lmhead_workspace_bytes(B, K, V, d)
    if n == 0:
        raise SpecVerifyError("unsupported LM-head shape B=%d K=%d V=%d d=%d" % (B, K, V, d))
    if workspace is None or workspace.numel() < n:
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    rs = pr = None
    if debug:
        rs = torch.full((B, 2 * K + 1, 2), float("nan"), dtype=torch.float64, device=dev)
        pr = torch.full((B, K, 2), float("nan"), dtype=torch.float64, device=dev)
    _check(L.spec_verify_lmhead(_ptr(hidden_target), _ptr(hidden_draft), _ptr(w_target),
                                _ptr(w_draft), d, _ptr(tokens), _ptr(verify_len),
                                _ptr(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF, B, K, V,
                                _ptr(out_tokens), _ptr(accept_len), _ptr(workspace),
                                workspace.numel(), _ptr(dev_status), _ptr(rs), _ptr(pr),
                                _stream(stream)))
    if debug:
        return out_tokens, accept_len, rs, pr
    return out_tokens, accept_len


def kernels_per_scheduled(confidence: bool, budget: bool) -> int:
    """Kernels one spec_verify_scheduled call launches."""
    return kernels_per_verify() + (3 if confidence else 0) + (1 if budget else 0)


_default = None


def _default_verifier():
    global _default
    if _default is None:
        _default = Verifier()
    return _default


def verify(target, draft, tokens, verify_len, temperature, seed, **kw):
    """One verification step; see include/spec_verify.h for the semantics.
    Returns (out_tokens [B, K+1] int32, accept_len [B] int32) on the device."""
    global _default
    if _default is None:
        _default = Verifier()
    return _default(target, draft, tokens, verify_len, temperature, seed, **kw)


def verify_debug(target, draft, tokens, verify_len, temperature, seed, **kw):
    """verify() plus intermediates: returns (out_tokens, accept_len, row_stats
    [B, 2K+1, 2] float64, probs [B, K, 2] float64)."""
    B, K1, V = target.shape
    K = K1 - 1
    rs = torch.empty((B, 2 * K + 1, 2), dtype=torch.float64, device=target.device)
    pr = torch.empty((B, K, 2), dtype=torch.float64, device=target.device)
    o, a = verify(target, draft, tokens, verify_len, temperature, seed, row_stats=rs, probs=pr, **kw)
    return o, a, rs, pr


def schedule_len(draft_maxprob, threshold, out=None, stream=None):
    """Confidence-scheduled verify lengths (float32 running product >= threshold)."""
    L = load_library()
    if draft_maxprob.dim() != 2 or draft_maxprob.dtype != torch.float32 or not draft_maxprob.is_cuda:
        raise ValueError("draft_maxprob must be a float32 CUDA tensor [B, K]")
    draft_maxprob = draft_maxprob.contiguous()
    B, K = draft_maxprob.shape
    if out is None:
        out = torch.empty((B,), dtype=torch.int32, device=draft_maxprob.device)
    _check(L.spec_schedule_len(_ptr(draft_maxprob), float(threshold), B, K, _ptr(out), _stream(stream)))
    return out
