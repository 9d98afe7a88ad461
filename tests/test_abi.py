"""The C ABI library: it loads, exports every symbol include/cconv.h declares,
and validates arguments on the host. No compute call reaches a GPU here: the
checked calls are rejected before any launch, and the one valid call is made
only where no CUDA device exists, to show that it fails loudly instead of
falling back to anything."""
import ctypes
import os
import re

import pytest
import torch

from state_cached_causal_gb300 import build as cbuild
from state_cached_causal_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cconv.h")


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return ops.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    names = re.findall(r"^\s*(?:CCONV_API\s+)?(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", text,
                       flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for")))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("cconv_fwd_varlen", "cconv_update", "cca_qk_conv", "cconv_fwd_varlen_fused",
              "cconv_update_fused", "cconv_status_string", "cconv_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_library_exports_nothing_else():
    """Only the C ABI is visible: internal kernels and helpers stay hidden."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", cbuild.build()], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    assert ops.status_string(0) == "ok"
    for s in (-1, -2, -3, -4):
        assert ops.status_string(s) not in ("ok", "unknown status")
    assert ops.status_string(17) == "unknown status"
    assert ops.abi_version() == 6


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation

# Calls with fake pointers run only where no CUDA device exists, so that a
# validation bug can never launch a kernel on a fake address.
no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers: CPU-only")


def _pool(num_slots=4, C=16, cap=3, layout="DS", dtype=1, base=FAKE):
    if layout == "DS":
        return ops.Pool(ctypes.c_void_p(base), C * cap, cap, 1, num_slots, cap, dtype)
    return ops.Pool(ctypes.c_void_p(base), C * cap, 1, C, num_slots, cap, dtype)


def fwd(lib, **kw):
    a = dict(x=FAKE, xrs=16, w=FAKE, bias=None, pool=_pool(), sidx=FAKE, cu=FAKE, hi=None,
             B=2, T=8, C=16, W=4, D=1, act=1, dt=1, out=FAKE, ors=16)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    return lib.cconv_fwd_varlen(P(a["x"]), a["xrs"], P(a["w"]), P(a["bias"]), a["pool"],
                                P(a["sidx"]), P(a["cu"]), P(a["hi"]), a["B"], a["T"], a["C"],
                                a["W"], a["D"], a["act"], a["dt"], P(a["out"]), a["ors"], None,
                                None)


def upd(lib, **kw):
    a = dict(x=FAKE, xrs=16, pool=_pool(cap=6), w=FAKE, bias=None, sidx=FAKE, B=2, ns=3,
             na=FAKE, hi=None, C=16, W=4, D=1, act=1, dt=1, out=FAKE, ors=16)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    return lib.cconv_update(P(a["x"]), a["xrs"], a["pool"], P(a["w"]), P(a["bias"]),
                            P(a["sidx"]), a["B"], a["ns"], P(a["na"]), P(a["hi"]), a["C"],
                            a["W"], a["D"], a["act"], a["dt"], P(a["out"]), a["ors"], None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(x=None), -1), (dict(x=None, out=None, T=0), -3), (dict(w=None), -1), (dict(out=None), -1), (dict(sidx=None), -1),
    (dict(cu=None), -1), (dict(C=12), -1), (dict(C=0), -1), (dict(x=FAKE + 2), -1),
    (dict(out=FAKE + 8), -1), (dict(xrs=8), -1), (dict(ors=20), -1), (dict(dt=5), -1),
    (dict(act=7), -1), (dict(W=0), -1), (dict(W=1), -1), (dict(W=9), -1), (dict(D=9), -1),
    (dict(D=0), -1), (dict(W=8, D=8, pool=_pool(cap=56)), -3), (dict(W=5, D=2, pool=_pool(cap=8)), -3),
    (dict(pool=_pool(cap=2)), -1), (dict(B=-1), -1), (dict(T=-1), -1),
    (dict(pool=_pool(num_slots=0)), -1), (dict(pool=_pool(dtype=2)), -1),
    (dict(pool=_pool(dtype=0, base=FAKE + 2)), -1), (dict(pool=_pool(base=FAKE + 1)), -1)])
@no_gpu
def test_fwd_varlen_rejects_bad_arguments(lib, kw, want):
    assert fwd(lib, **kw) == want


@no_gpu
def test_fwd_varlen_empty_batch_is_a_noop(lib):
    assert fwd(lib, B=0) == 0


@pytest.mark.parametrize("kw,want", [
    (dict(na=None), -1), (dict(ns=8), -2), (dict(ns=-1), -1),
    (dict(pool=_pool(cap=5)), -1), (dict(C=4, dt=1), -1), (dict(x=None), -1),
    (dict(W=9), -1), (dict(D=9), -1), (dict(W=1), -1), (dict(W=8, D=8, pool=_pool(cap=59)), -3),
    (dict(W=8, D=8, pool=_pool(cap=58)), -1)])
@no_gpu
def test_update_rejects_bad_arguments(lib, kw, want):
    assert upd(lib, **kw) == want


@pytest.mark.parametrize("pool_dtype,dt", [(0, 1), (1, 0), (0, 0), (1, 1)])
@no_gpu
def test_state_dtype_may_differ_from_the_call(lib, pool_dtype, dt):
    # every (activation, pool) type pair passes validation (-3: no device);
    # a bf16 pool needs only 2-byte alignment on the element-wise path
    assert fwd(lib, dt=dt, pool=_pool(dtype=pool_dtype)) == -3
    assert upd(lib, dt=dt, pool=_pool(cap=6, dtype=pool_dtype)) == -3
    if pool_dtype == 1 and dt == 0:
        assert fwd(lib, dt=dt, pool=_pool(dtype=1, base=FAKE + 2)) == -3


@no_gpu
def test_valid_call_without_gpu_fails_loudly(lib):
    # A valid request on a machine with no CUDA device must report a launch
    # failure, never compute anything on the host.
    assert fwd(lib, C=16) == -3


def fwd_fused(lib, epi, **kw):
    a = dict(x=FAKE, xrs=16, w=FAKE, bias=None, pool=_pool(), sidx=FAKE, cu=FAKE, hi=None,
             B=2, T=8, C=16, W=4, D=1, act=1, dt=1)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    return lib.cconv_fwd_varlen_fused(P(a["x"]), a["xrs"], P(a["w"]), P(a["bias"]), a["pool"],
                                      P(a["sidx"]), P(a["cu"]), P(a["hi"]), a["B"], a["T"],
                                      a["C"], a["W"], a["D"], a["act"], a["dt"], epi, None,
                                      None)


def _epi(res=FAKE, rrs=16, outer=None, ors=0, idx=None, rows=8):
    P = lambda v: None if v is None else v
    return ops.Epilogue(P(res), rrs, P(outer), ors, P(idx), rows)


@pytest.mark.parametrize("epi,want", [
    (dict(res=None), -1), (dict(res=FAKE + 4), -1), (dict(rrs=8), -1),
    (dict(rows=0), -1), (dict(rows=7), -1), (dict(outer=FAKE + 2, ors=16), -1),
    (dict(outer=FAKE, ors=12), -1), (dict(rows=4, idx=FAKE), -3), (dict(), -3)])
@no_gpu
def test_fwd_fused_checks_its_epilogue(lib, epi, want):
    # -3: the epilogue passed every check and the launch failed (no device)
    assert fwd_fused(lib, _epi(**epi)) == want


@pytest.mark.parametrize("kw,want", [
    (dict(pool=_pool(cap=65)), -1), (dict(W=9), -1), (dict(D=9), -1), (dict(W=8, D=8), -1),
    (dict(W=8, D=8, pool=_pool(cap=56)), -3), (dict(num=0), 0), (dict(x=FAKE + 4), -1),
    (dict(rows=3, idx=None), -1), (dict(), -3), (dict(pool=_pool(cap=9, dtype=0)), -3),
    (dict(pool=_pool(cap=9, dtype=3)), -1)])
@no_gpu
def test_checkpoint_export_validation(lib, kw, want):
    a = dict(x=FAKE, pool=_pool(cap=9), num=2, rows=8, idx=FAKE, W=4, D=3)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    rc = lib.cconv_checkpoint_export(P(a["x"]), 16, a["pool"], P(FAKE), P(FAKE), P(FAKE),
                                     a["num"], P(FAKE), 2, 8, P(a["idx"]), a["rows"], 16,
                                     a["W"], a["D"], 1, None, None)
    assert rc == want


def cca(lib, fused=False, noalloc=False, **kw):
    # Zaya shapes: 16 q + 4 kv heads of 128 (20 groups), Dv = 256, history n = 2
    a = dict(qk=FAKE, qrs=2560, w_dw=FAKE, b_dw=None, w_gr=FAKE, b_gr=None, G=20, Hq=16, t0=2,
             t1=2, dl=FAKE, drs=256, dinit=FAKE, Dv=256, vc=FAKE, vcrs=256,
             pool=_pool(C=2560, cap=2), ds=FAKE, dsrs=256, sidx=FAKE, cu=FAKE, hi=None, B=2,
             T=8, C=2560, dt=1, out=FAKE, ors=2560 + 512, dp=FAKE, dprs=256)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)
    if fused:
        return lib.cca_qk_conv_fused(P(a["qk"]), a["qrs"], P(a["w_dw"]), P(a["b_dw"]),
                                     P(a["w_gr"]), P(a["b_gr"]), a["G"], a["Hq"], a["t0"],
                                     a["t1"], P(a["dl"]), a["drs"], P(a["dinit"]), a["Dv"],
                                     P(a["vc"]), a["vcrs"], a["pool"], P(a["ds"]), a["dsrs"],
                                     P(a["sidx"]), P(a["cu"]), P(a["hi"]), a["B"], a["T"],
                                     a["C"], a["dt"], P(a["out"]), a["ors"], None, None)
    fn = lib.cca_qk_conv_noalloc if noalloc else lib.cca_qk_conv
    return fn(P(a["qk"]), a["qrs"], P(a["w_dw"]), P(a["b_dw"]), P(a["w_gr"]),
                           P(a["b_gr"]), a["G"], a["t0"], a["t1"], P(a["dl"]), a["drs"],
                           P(a["dinit"]), a["Dv"], a["pool"], P(a["ds"]), a["dsrs"],
                           P(a["sidx"]), P(a["cu"]), P(a["hi"]), a["B"], a["T"], a["C"], a["dt"],
                           P(a["out"]), a.get("oqrs", 2560), P(a["dp"]), a["dprs"], None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(), -3), (dict(dt=0), -2), (dict(dt=5), -1), (dict(w_gr=None), -1),
    (dict(C=2570), -1), (dict(C=2500), -2), (dict(G=40), -2), (dict(t0=5), -2), (dict(t1=3), -2), (dict(t0=0), -1),
    (dict(pool=_pool(C=2560, cap=1)), -1), (dict(pool=_pool(C=2560, cap=2, dtype=4)), -1),
    (dict(pool=_pool(C=2560, cap=2, dtype=0)), -3), (dict(ds=FAKE + 8), -1),
    (dict(dsrs=100), -1), (dict(Dv=250), -1), (dict(qk=FAKE + 2), -1), (dict(qrs=2500), -1),
    (dict(B=0), 0), (dict(T=-1), -1)])
@no_gpu
def test_cca_validation(lib, kw, want):
    assert cca(lib, **kw) == want
    # the no-allocation form checks its arguments exactly as cca_qk_conv does
    assert cca(lib, noalloc=True, **kw) == want


@no_gpu
def test_cca_noalloc_rejects_more_work_than_its_scratch_counts(lib):
    # 2^30 tokens in tiles of 127 rows, times 600 groups: about 5.1e9
    # units, more than the 2^30 its fixed counters may count; cca_qk_conv
    # itself takes the call to the launch (-3: no device here)
    big = dict(T=2**30, G=600, C=600 * 128, qrs=600 * 128, oqrs=600 * 128,
               pool=_pool(C=600 * 128, cap=2))
    assert cca(lib, noalloc=True, **big) == ops.ERR_TOO_LARGE
    assert cca(lib, noalloc=False, **big) == -3


@pytest.mark.parametrize("kw,want", [
    (dict(), -3), (dict(Hq=15), -1), (dict(Hq=20), -1), (dict(Dv=128, dsrs=128, drs=128), -1),
    (dict(vc=None), -1), (dict(vc=FAKE + 4), -1), (dict(vcrs=200), -1), (dict(ors=2560), -1)])
@no_gpu
def test_cca_fused_validation(lib, kw, want):
    # the fused form also checks the head split (Hq q heads over groups - Hq kv
    # heads, Dv = kv heads * 64), v_current and the [query | key | value] rows
    assert cca(lib, fused=True, **kw) == want
