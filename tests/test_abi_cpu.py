"""C-ABI checks that need no GPU.

The shared library must load, export every function include/spec_verify.h
declares, and reject bad arguments on the host before touching CUDA.  A call
whose arguments pass validation reaches the CUDA runtime, which fails without
a GPU (SPEC_E_CUDA) instead of enqueuing anything.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")
LIB = os.path.join(ROOT, "speculative_decoding_verify_07_gb300", "lib", "libspecverify.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from speculative_decoding_verify_07_gb300 import build
        build.build()
    L = ctypes.CDLL(LIB)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    L.spec_verify.argtypes = [vp, i32, vp, vp, vp, u64, ctypes.c_uint32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_verify.restype = i32
    L.spec_commit.argtypes = [vp, vp, vp, vp, vp, vp] + [i32] * 9 + [vp, vp]
    L.spec_commit.restype = i32
    L.spec_verify_workspace_size.argtypes = [i32, i32, i32]
    L.spec_verify_workspace_size.restype = sz
    L.spec_philox4x32_10.argtypes = [vp, u64, vp, ctypes.c_int64, vp]
    L.spec_philox4x32_10.restype = i32
    L.spec_status_string.restype = ctypes.c_char_p
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("spec_verify", "spec_commit", "spec_verify_workspace_size", "spec_status_string",
              "spec_version", "spec_philox4x32_10"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.spec_version() == 5
    for code in range(0, -8, -1):
        s = lib.spec_status_string(code).decode()
        assert s and s != "unknown status code"
    assert lib.spec_status_string(-99).decode() == "unknown status code"


def test_workspace_size(lib):
    assert lib.spec_verify_workspace_size(64, 2, 151936) >= 64 * 3 * 32
    assert lib.spec_verify_workspace_size(-1, 2, 10) == 0


P = 4096   # a fake, aligned, non-null address; validation fails before any dereference


def _verify(lib, **kw):
    a = dict(logits=P, dt=1, q=P, x=P, params=P, seed=0, row_base=0, B=4, k=2, V=1000, tok=P, acc=P,
             lp=P, alpha=P, flags=P, ws=P, wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.spec_verify(a["logits"], a["dt"], a["q"], a["x"], a["params"], a["seed"], a["row_base"],
                           a["B"], a["k"], a["V"], a["tok"], a["acc"], a["lp"], a["alpha"], a["flags"],
                           a["ws"], a["wsb"], a["stream"])


def test_verify_argument_errors(lib):
    assert _verify(lib, B=-1) == -2
    assert _verify(lib, k=17) == -2
    assert _verify(lib, V=0) == -2
    assert _verify(lib, V=524289) == -2
    assert _verify(lib, dt=7) == -3
    assert _verify(lib, B=0) == 0                       # empty batch: nothing to do
    assert _verify(lib, logits=None) == -1
    assert _verify(lib, q=None) == -1
    assert _verify(lib, q=None, x=None, alpha=None, k=0) != -1   # k == 0 needs no draft arrays
    assert _verify(lib, flags=None) == -1
    assert _verify(lib, logits=P + 1) == -4              # bf16 needs 2-byte alignment
    assert _verify(lib, dt=0, logits=P + 2) == -4        # f32 needs 4-byte alignment
    assert _verify(lib, ws=P + 8) == -4                  # workspace needs 16-byte alignment
    assert _verify(lib, wsb=16) == -5
    # valid arguments reach the CUDA runtime, which has no device here
    assert _verify(lib) in (-6, -7)
    assert _verify(lib, row_base=2 ** 32 - 1) in (-6, -7)


def _noalloc(lib, **kw):
    vp, i32, u32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
    lib.spec_verify_noalloc.argtypes = [vp, i32, vp, vp, vp, u64, u32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_noalloc.restype = i32
    a = dict(logits=P, dt=1, q=P, x=P, params=P, seed=0, row_base=0, B=4, k=2, V=1000, tok=P, acc=P,
             lp=P, alpha=P, flags=P, stream=None)
    a.update(kw)
    return lib.spec_verify_noalloc(a["logits"], a["dt"], a["q"], a["x"], a["params"], a["seed"],
                                   a["row_base"], a["B"], a["k"], a["V"], a["tok"], a["acc"], a["lp"],
                                   a["alpha"], a["flags"], a["stream"])


def test_noalloc_checks_arguments_before_touching_cuda(lib):
    # a refused call returns before any CUDA call (here: before the runtime
    # would report that there is no device), so it enqueues nothing
    assert _noalloc(lib, logits=None) == -1
    assert _noalloc(lib, flags=None) == -1
    assert _noalloc(lib, tok=P + 2) == -4
    assert _noalloc(lib, dt=9) == -3
    assert _noalloc(lib, k=17) == -2
    assert _noalloc(lib, B=4000, k=16, V=151936) == -5   # beyond the library's scratch
    assert _noalloc(lib, B=0) == 0
    assert _noalloc(lib) in (-6, -7)


def _commit(lib, **kw):
    a = dict(vr=P, vc=P, acc=P, slot=P, cr=P, cc=P, L=2, B=3, S=3, H=2, Dk=4, Dv=4, W=2, C=8,
             slots=3, flags=P, stream=None)
    a.update(kw)
    return lib.spec_commit(a["vr"], a["vc"], a["acc"], a["slot"], a["cr"], a["cc"], a["L"], a["B"],
                           a["S"], a["H"], a["Dk"], a["Dv"], a["W"], a["C"], a["slots"], a["flags"],
                           a["stream"])


def test_commit_argument_errors(lib):
    assert _commit(lib, S=0) == -2
    assert _commit(lib, H=0) == -2
    assert _commit(lib, L=0) == 0
    assert _commit(lib, acc=None) == -1
    assert _commit(lib, vr=None, vc=None) == -1
    assert _commit(lib, cr=None) == -1
    assert _commit(lib, slot=None, slots=2) == -2        # identity slots need slots >= B
    assert _commit(lib, acc=P + 2) == -4
    assert _commit(lib, vr=P + 2) == -4
    assert _commit(lib) in (-6, -7)


def test_philox_argument_errors(lib):
    assert lib.spec_philox4x32_10(P, 0, P, -1, None) == -2
    assert lib.spec_philox4x32_10(P, 0, P, 0, None) == 0
    assert lib.spec_philox4x32_10(None, 0, P, 4, None) == -1
    assert lib.spec_philox4x32_10(P + 4, 0, P, 4, None) == -4
    assert lib.spec_philox4x32_10(P, 0, P, 4, None) in (-6, -7)


def _fused(lib, **kw):
    vp, i32, u32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t
    lib.spec_verify_commit.argtypes = ([vp, i32, vp, vp, vp, u64, u32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz]
                                       + [vp] * 5 + [i32] * 7 + [vp])
    lib.spec_verify_commit.restype = i32
    a = dict(logits=P, dt=1, q=P, x=P, params=P, seed=0, row_base=0, B=4, k=2, V=1000, tok=P, acc=P,
             lp=P, alpha=P, flags=P, ws=P, wsb=1 << 20, vr=P, vc=P, slot=P, cr=P, cc=P, L=2, H=2, Dk=4,
             Dv=4, W=2, C=8, slots=4, stream=None)
    a.update(kw)
    return lib.spec_verify_commit(a["logits"], a["dt"], a["q"], a["x"], a["params"], a["seed"], a["row_base"],
                                  a["B"], a["k"], a["V"], a["tok"], a["acc"], a["lp"], a["alpha"], a["flags"],
                                  a["ws"], a["wsb"], a["vr"], a["vc"], a["slot"], a["cr"], a["cc"], a["L"],
                                  a["H"], a["Dk"], a["Dv"], a["W"], a["C"], a["slots"], a["stream"])


def test_fused_verify_commit_checks_every_argument_before_touching_cuda(lib):
    # the verify's checks
    assert _fused(lib, B=-1) == -2
    assert _fused(lib, k=17) == -2
    assert _fused(lib, V=0) == -2
    assert _fused(lib, dt=7) == -3
    assert _fused(lib, logits=None) == -1
    assert _fused(lib, flags=None) == -1
    assert _fused(lib, wsb=16) == -5
    assert _fused(lib, ws=None) == -1
    # the commit's checks
    assert _fused(lib, H=0) == -2
    assert _fused(lib, L=-1) == -2
    assert _fused(lib, cr=None) == -1
    assert _fused(lib, vr=None, vc=None) == -1
    assert _fused(lib, slot=None, slots=2) == -2      # identity slots need slots >= B
    assert _fused(lib, vr=P + 2) == -4
    assert _fused(lib, slot=P + 2) == -4
    # nothing to do, or nothing to commit: the verify alone
    assert _fused(lib, B=0) == 0
    assert _fused(lib, L=0) in (-6, -7)
    assert _fused(lib) in (-6, -7)


def _draft(lib, **kw):
    vp, i32, u32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t
    lib.spec_draft_sample.argtypes = [vp, i32, vp, u64, u32, u32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.spec_draft_sample.restype = i32
    lib.spec_draft_workspace_size.argtypes = [i32, i32]
    lib.spec_draft_workspace_size.restype = sz
    a = dict(logits=P, dt=1, params=P, seed=0, row_base=0, pos=0, B=4, V=1000, q=P, tok=P, lp=P, flags=P,
             ws=P, wsb=1 << 22, stream=None)
    a.update(kw)
    return lib.spec_draft_sample(a["logits"], a["dt"], a["params"], a["seed"], a["row_base"], a["pos"], a["B"],
                                 a["V"], a["q"], a["tok"], a["lp"], a["flags"], a["ws"], a["wsb"], a["stream"])


def test_draft_sample_checks_arguments_before_touching_cuda(lib):
    assert lib.spec_draft_workspace_size(4, 1000) >= lib.spec_verify_workspace_size(4, 0, 1000)
    assert lib.spec_draft_workspace_size(-1, 10) == 0
    assert _draft(lib, B=-1) == -2
    assert _draft(lib, V=0) == -2
    assert _draft(lib, V=524289) == -2
    assert _draft(lib, dt=5) == -3
    assert _draft(lib, B=0) == 0
    assert _draft(lib, logits=None) == -1
    assert _draft(lib, tok=None) == -1
    assert _draft(lib, lp=None) == -1
    assert _draft(lib, ws=None) == -1
    assert _draft(lib, q=P + 2) == -4
    assert _draft(lib, ws=P + 8) == -4
    assert _draft(lib, wsb=64) == -5
    assert _draft(lib, logits=P + 1) == -4
    # valid arguments reach the CUDA runtime (q may be NULL: tokens only)
    assert _draft(lib) in (-6, -7)
    assert _draft(lib, q=None) in (-6, -7)
