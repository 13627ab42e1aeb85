"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every function include/*.h declares; host-side argument validation
returns errors before anything is launched."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", src, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import speculative_decoding_verification_69_gb300 as sv
    return sv.load_library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("spec_verify", "spec_verify_debug", "spec_verify_workspace_bytes",
              "spec_schedule_len", "spec_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_workspace_bytes(lib):
    import speculative_decoding_verification_69_gb300 as sv
    assert lib.spec_verify_workspace_bytes(0, 4, 100, 0) == 0
    assert lib.spec_verify_workspace_bytes(1, 33, 100, 0) == 0
    assert lib.spec_verify_workspace_bytes(1, 4, 1, 0) == 0
    assert lib.spec_verify_workspace_bytes(1, 4, 100, 7) == 0
    n1 = lib.spec_verify_workspace_bytes(32, 8, 151936, sv.DTYPE_BF16)
    n2 = lib.spec_verify_workspace_bytes(64, 8, 151936, sv.DTYPE_BF16)
    assert 0 < n1 < n2 and n1 % 256 == 0
    # small compared with the logits themselves
    assert n1 < 0.05 * 32 * 17 * 151936 * 2


def test_host_validation_without_gpu(lib):
    """Invalid sizes, null pointers and bad workspaces are rejected on the host,
    before any CUDA call (safe on a machine without a GPU)."""
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    i32 = ctypes.c_void_p(0x10000)
    base = dict(t=fake, d=fake, dt=1, tok=i32, vl=None, T=fake, seed=1, B=2, K=4, V=100,
                o=i32, a=i32, ws=ctypes.c_void_p(0x10000), wsb=1 << 30, st=None)

    def call(**kw):
        a = dict(base, **kw)
        return lib.spec_verify(a["t"], a["d"], a["dt"], a["tok"], a["vl"], a["T"], a["seed"],
                               a["B"], a["K"], a["V"], a["o"], a["a"], a["ws"], a["wsb"],
                               a["st"], None)

    assert call(B=0) == 1
    assert call(K=0) == 1 and call(K=33) == 1
    assert call(V=1) == 1
    assert call(dt=5) == 2
    assert call(t=None) == 1 and call(d=None) == 1 and call(tok=None) == 1
    assert call(T=None) == 1 and call(o=None) == 1 and call(a=None) == 1
    assert call(t=ctypes.c_void_p(0x10008)) == 1          # logits not 16-byte aligned
    assert call(ws=None) == 4
    assert call(wsb=16) == 4
    assert call(ws=ctypes.c_void_p(0x10010)) == 4          # workspace not 256-byte aligned
    assert lib.spec_schedule_len(None, 0.3, 4, 4, i32, None) == 1
    assert lib.spec_schedule_len(fake, 0.3, 0, 4, i32, None) == 1
    assert lib.spec_schedule_len(fake, 0.3, 4, 40, i32, None) == 1
    assert lib.spec_status_str(0) == b"ok"
    assert b"workspace" in lib.spec_status_str(4)

    def call_ee(W, **kw):
        a = dict(base, **kw)
        return lib.spec_verify_early_exit(a["t"], a["d"], a["dt"], a["tok"], a["vl"], a["T"],
                                          a["seed"], a["B"], a["K"], a["V"], W, a["o"], a["a"],
                                          a["ws"], a["wsb"], a["st"], None)

    assert call_ee(0) == 1 and call_ee(-3) == 1              # first wave must be >= 1
    assert call_ee(2, B=0) == 1 and call_ee(2, t=None) == 1
    assert call_ee(2, ws=None) == 4


def test_from_host_validation_without_gpu(lib):
    """spec_verify_from_host checks every argument before its first copy."""
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    base = dict(th=fake, dh=fake, dt=1, tokh=fake, vlh=None, Th=fake, seed=1, B=2, K=4, V=100,
                td=fake, dd=fake, tokd=fake, vld=None, Td=fake, od=fake, ad=fake, oh=fake, ah=fake,
                ws=ctypes.c_void_p(0x10000), wsb=1 << 30, st=None, nb=None)

    def call(**kw):
        a = dict(base, **kw)
        return lib.spec_verify_from_host(
            a["th"], a["dh"], a["dt"], a["tokh"], a["vlh"], a["Th"], a["seed"], a["B"], a["K"],
            a["V"], a["td"], a["dd"], a["tokd"], a["vld"], a["Td"], a["od"], a["ad"], a["oh"],
            a["ah"], a["ws"], a["wsb"], a["st"], None, a["nb"])

    for k in ("th", "dh", "tokh", "Th", "td", "dd", "tokd", "Td", "od", "ad", "oh", "ah"):
        assert call(**{k: None}) == 1, k
    assert call(vlh=fake) == 1                            # host lengths without a device buffer
    assert call(B=0) == 1 and call(K=33) == 1 and call(V=1) == 1
    assert call(dt=5) == 2
    assert call(td=ctypes.c_void_p(0x10008)) == 1         # device logits not 16-byte aligned
    assert call(ws=None) == 4 and call(wsb=16) == 4


def test_scheduled_from_host_validation_without_gpu(lib):
    """spec_verify_scheduled_from_host checks every argument before its first copy."""
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    base = dict(th=fake, dh=fake, dt=1, tokh=fake, Th=fake, mph=fake, seed=1, B=2, K=4, V=100,
                mode=0, thr=0.3, budget=3, td=fake, dd=fake, tokd=fake, Td=fake, mpd=fake, vld=fake,
                od=fake, ad=fake, oh=fake, ah=fake, vlh=fake, ws=ctypes.c_void_p(0x10000),
                wsb=1 << 30, st=None, nb=None)

    def call(**kw):
        a = dict(base, **kw)
        return lib.spec_verify_scheduled_from_host(
            a["th"], a["dh"], a["dt"], a["tokh"], a["Th"], a["mph"], a["seed"], a["B"], a["K"],
            a["V"], a["mode"], a["thr"], a["budget"], a["td"], a["dd"], a["tokd"], a["Td"],
            a["mpd"], a["vld"], a["od"], a["ad"], a["oh"], a["ah"], a["vlh"], a["ws"], a["wsb"],
            a["st"], None, a["nb"])

    for k in ("th", "dh", "tokh", "Th", "mph", "td", "dd", "tokd", "Td", "mpd", "vld", "od", "ad",
              "oh", "ah", "vlh"):
        assert call(**{k: None}) == 1, k
    assert call(mode=2) == 1
    assert call(B=0) == 1 and call(K=33) == 1 and call(dt=5) == 2
    assert call(ws=None) == 4
    assert call(mode=1, B=200_000, K=32) == 2          # budget selection over more than 2^22 positions


def test_tree_host_validation_without_gpu(lib):
    """The tree entry points reject bad sizes, null pointers, misaligned logits
    and small workspaces on the host, before any CUDA call."""
    fake = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x10000)
    assert lib.spec_tree_workspace_bytes(2, 0, 100, 1) == 0
    assert lib.spec_tree_workspace_bytes(2, 65, 100, 1) == 0
    assert lib.spec_tree_workspace_bytes(2, 64, 100, 1) > 0
    base = dict(t=fake, d=fake, dt=1, par=fake, tok=fake, T=fake, seed=1, B=2, N=5, V=100,
                o=fake, n=fake, a=fake, ws=ws, wsb=1 << 30, st=None)

    def call(**kw):
        x = dict(base, **kw)
        return lib.spec_verify_tree(x["t"], x["d"], x["dt"], x["par"], x["tok"], x["T"], x["seed"],
                                    x["B"], x["N"], x["V"], x["o"], x["n"], x["a"], x["ws"],
                                    x["wsb"], x["st"], None)

    assert call(N=0) == 1 and call(N=65) == 1 and call(B=0) == 1 and call(V=1) == 1
    assert call(dt=7) == 2
    assert call(t=None) == 1 and call(d=None) == 1 and call(par=None) == 1
    assert call(tok=None) == 1 and call(T=None) == 1
    assert call(o=None) == 1 and call(n=None) == 1 and call(a=None) == 1
    assert call(d=ctypes.c_void_p(0x10008)) == 1          # draft logits not 16-byte aligned
    assert call(ws=None) == 4 and call(wsb=16) == 4
    greedy = lib.spec_verify_tree_greedy
    assert greedy(fake, 1, fake, fake, 2, 0, 100, fake, fake, fake, ws, 1 << 30, None, None) == 1
    assert greedy(None, 1, fake, fake, 2, 5, 100, fake, fake, fake, ws, 1 << 30, None, None) == 1
    assert greedy(fake, 1, fake, fake, 2, 5, 100, fake, fake, fake, None, 1 << 30, None, None) == 4


def test_scheduled_host_validation_without_gpu(lib):
    """spec_verify_scheduled rejects an unknown schedule mode, the step's bad
    sizes, null pointers and workspaces, and a budget over too many positions,
    on the host before any CUDA call."""
    fake = ctypes.c_void_p(0x10000)
    base = dict(t=fake, d=fake, dt=1, tok=fake, T=fake, seed=1, B=2, K=4, V=100, mp=None, mode=0,
                thr=0.3, budget=4, mpo=None, vlo=None, o=fake, a=fake, ws=fake, wsb=1 << 40,
                st=None)

    def call(**kw):
        x = dict(base, **kw)
        return lib.spec_verify_scheduled(x["t"], x["d"], x["dt"], x["tok"], x["T"], x["seed"],
                                         x["B"], x["K"], x["V"], x["mp"], x["mode"], x["thr"],
                                         x["budget"], x["mpo"], x["vlo"], x["o"], x["a"], x["ws"],
                                         x["wsb"], x["st"], None)

    assert call(mode=2) == 1 and call(mode=-1) == 1
    assert call(B=0) == 1 and call(K=33) == 1 and call(V=1) == 1
    assert call(dt=3) == 2
    assert call(t=None) == 1 and call(d=None) == 1 and call(tok=None) == 1 and call(T=None) == 1
    assert call(o=None) == 1 and call(a=None) == 1
    assert call(d=ctypes.c_void_p(0x10004)) == 1              # draft logits not 16-byte aligned
    assert call(ws=None) == 4 and call(wsb=64) == 4
    assert call(mode=1, B=1 << 20, K=8) == 2                  # budget over more than 2^22 positions
    # the workspace covers the schedule's own buffers: it grows with B * K
    n1 = lib.spec_verify_workspace_bytes(8, 4, 100, 1)
    n2 = lib.spec_verify_workspace_bytes(8, 8, 100, 1)
    assert n2 > n1


def test_lmhead_host_validation_without_gpu(lib):
    """spec_verify_lmhead rejects bad sizes (d not a multiple of 64, V not a
    multiple of 4), null pointers, misaligned buffers and small workspaces on
    the host, before any CUDA call; its workspace size follows B, V and d."""
    fake = ctypes.c_void_p(0x10000)
    assert lib.spec_lmhead_workspace_bytes(2, 4, 1000, 96) == 0      # d % 64
    assert lib.spec_lmhead_workspace_bytes(2, 4, 1001, 64) == 0      # V % 4
    assert lib.spec_lmhead_workspace_bytes(0, 4, 1000, 64) == 0
    assert lib.spec_lmhead_workspace_bytes(2, 33, 1000, 64) == 0
    n1 = lib.spec_lmhead_workspace_bytes(2, 4, 1000, 64)
    n2 = lib.spec_lmhead_workspace_bytes(4, 4, 1000, 64)
    n3 = lib.spec_lmhead_workspace_bytes(2, 4, 1000, 128)
    assert 0 < n1 < n2 and n1 < n3 and n1 % 256 == 0
    assert n1 >= 8 * 2 * 1000                                        # the recomputed rows
    base = dict(ht=fake, hd=fake, wt=fake, wd=fake, d=64, tok=fake, vl=None, T=fake, seed=1, B=2,
                K=4, V=1000, o=fake, a=fake, ws=fake, wsb=1 << 40, st=None, rs=None, pr=None)

    def call(**kw):
        x = dict(base, **kw)
        return lib.spec_verify_lmhead(x["ht"], x["hd"], x["wt"], x["wd"], x["d"], x["tok"], x["vl"],
                                      x["T"], x["seed"], x["B"], x["K"], x["V"], x["o"], x["a"],
                                      x["ws"], x["wsb"], x["st"], x["rs"], x["pr"], None)

    assert call(d=96) == 1 and call(d=0) == 1 and call(V=1001) == 1 and call(B=0) == 1
    assert call(K=0) == 1 and call(K=33) == 1
    for k in ("ht", "hd", "wt", "wd", "tok", "T", "o", "a"):
        assert call(**{k: None}) == 1, k
    for k in ("ht", "hd", "wt", "wd"):
        assert call(**{k: ctypes.c_void_p(0x10008)}) == 1, k        # not 16-byte aligned
    assert call(ws=None) == 4 and call(wsb=1024) == 4
    assert call(ws=ctypes.c_void_p(0x10080)) == 4                    # not 256-byte aligned
