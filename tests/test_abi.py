"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, and rejects bad arguments on the host before touching
CUDA."""

import ctypes
import os
import re

import pytest

from piecewise_sparse_attention_gb300 import pisa as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pisa_[a-z_0-9]+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return P.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"pisa_block_stats", "pisa_route", "pisa_forward", "pisa_status_string"} <= names
    for name in names:
        assert hasattr(lib, name), name
    assert set(P.EXPORTED) == names


def test_status_strings_and_version(lib):
    assert P.status_string(0) == "ok"
    assert "invalid" in P.status_string(1)
    assert P.status_string(99) == "unknown status"
    assert lib.pisa_version() >= 100


NULL = None
FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x10008)


def fwd(lib, q=FAKE, out=FAKE, in_dt=1, heads=2, n=128, d=128, block=64, scale=0.1, ms=4,
        out_dt=1, idx=FAKE, cnt=FAKE):
    return lib.pisa_forward(q, FAKE, FAKE, in_dt, heads, n, d, block, ctypes.c_float(scale), idx,
                            cnt, ms, out, out_dt, NULL, NULL)


def test_forward_rejects_bad_arguments(lib):
    assert fwd(lib, q=NULL) == P.ERR_INVALID_ARG
    assert fwd(lib, q=MISALIGNED) == P.ERR_INVALID_ARG
    assert fwd(lib, out=MISALIGNED) == P.ERR_INVALID_ARG
    assert fwd(lib, idx=NULL) == P.ERR_INVALID_ARG
    assert fwd(lib, in_dt=7) == P.ERR_INVALID_ARG
    assert fwd(lib, out_dt=-1) == P.ERR_INVALID_ARG
    assert fwd(lib, heads=0) == P.ERR_INVALID_ARG
    assert fwd(lib, n=0) == P.ERR_INVALID_ARG
    assert fwd(lib, block=32) == P.ERR_INVALID_ARG
    assert fwd(lib, scale=0.0) == P.ERR_INVALID_ARG
    assert fwd(lib, scale=float("nan")) == P.ERR_INVALID_ARG
    assert fwd(lib, ms=0) == P.ERR_INVALID_ARG
    assert fwd(lib, d=96) == P.ERR_UNSUPPORTED
    assert fwd(lib, n=(1 << 20) + 1) == P.ERR_UNSUPPORTED


def test_stats_rejects_bad_arguments(lib):
    f = lambda **kw: lib.pisa_block_stats(
        kw.get("q", FAKE), FAKE, FAKE, kw.get("dt", 1), kw.get("heads", 1), kw.get("n", 64),
        kw.get("d", 128), 64, kw.get("qbar", FAKE), NULL, NULL, kw.get("h", NULL),
        kw.get("hdt", 0), NULL, NULL)
    assert f(q=NULL) == P.ERR_INVALID_ARG
    assert f(qbar=NULL) == P.ERR_INVALID_ARG  # no output requested at all
    assert f(qbar=MISALIGNED) == P.ERR_INVALID_ARG
    assert f(dt=3) == P.ERR_INVALID_ARG
    assert f(h=FAKE, hdt=5) == P.ERR_INVALID_ARG
    assert f(d=32) == P.ERR_UNSUPPORTED
    assert f(heads=70000) == P.ERR_INVALID_ARG


def test_route_rejects_bad_arguments(lib):
    f = lambda **kw: lib.pisa_route(
        kw.get("qbar", FAKE), FAKE, kw.get("heads", 1), kw.get("nb", 16), kw.get("d", 128),
        ctypes.c_float(kw.get("scale", 0.1)), kw.get("topk", 4), kw.get("band", 1), FAKE, FAKE,
        kw.get("ms", 7), NULL, NULL)
    assert f(qbar=NULL) == P.ERR_INVALID_ARG
    assert f(topk=-1) == P.ERR_INVALID_ARG
    assert f(band=-2) == P.ERR_INVALID_ARG
    assert f(ms=6) == P.ERR_INVALID_ARG          # needs min(nb, 4 + 2 + 1) = 7
    assert f(scale=-1.0) == P.ERR_INVALID_ARG
    assert f(nb=0) == P.ERR_INVALID_ARG
    assert f(d=256) == P.ERR_UNSUPPORTED
    assert f(nb=16385, ms=7) == P.ERR_UNSUPPORTED


def test_covariance_calls_reject_bad_arguments(lib):
    h = lambda **kw: lib.pisa_block_heterogeneity(
        kw.get("k", FAKE), FAKE, kw.get("dt", 1), 2, kw.get("n", 256), kw.get("d", 128), 64,
        kw.get("kbar", FAKE), kw.get("hbar", FAKE), kw.get("norm", 0), kw.get("m", FAKE), NULL, NULL)
    assert h(k=NULL) == P.ERR_INVALID_ARG
    assert h(hbar=NULL) == P.ERR_INVALID_ARG
    assert h(m=MISALIGNED) == P.ERR_INVALID_ARG
    assert h(norm=2) == P.ERR_INVALID_ARG
    assert h(dt=7) == P.ERR_INVALID_ARG
    assert h(d=96) == P.ERR_UNSUPPORTED
    r = lambda **kw: lib.pisa_route_covariance(
        FAKE, FAKE, kw.get("m", FAKE), ctypes.c_float(kw.get("eps", 1e-6)), 1, kw.get("nb", 16),
        128, ctypes.c_float(kw.get("scale", 0.1)), 4, 1, FAKE, FAKE, kw.get("ms", 7), NULL, NULL)
    assert r(m=NULL) == P.ERR_INVALID_ARG
    assert r(eps=0.0) == P.ERR_INVALID_ARG
    assert r(eps=float("inf")) == P.ERR_INVALID_ARG
    assert r(scale=0.0) == P.ERR_INVALID_ARG
    assert r(ms=6) == P.ERR_INVALID_ARG
    assert r(nb=16385) == P.ERR_UNSUPPORTED


def test_global_first_order_rejects_bad_arguments(lib):
    f = lambda **kw: lib.pisa_global_first_order(
        kw.get("k", FAKE), FAKE, kw.get("dt", 1), kw.get("heads", 2), kw.get("n", 256),
        kw.get("d", 128), kw.get("block", 64), kw.get("kbar", FAKE), FAKE, kw.get("hbar", FAKE),
        NULL, NULL)
    assert f(k=NULL) == P.ERR_INVALID_ARG
    assert f(kbar=NULL) == P.ERR_INVALID_ARG
    assert f(hbar=MISALIGNED) == P.ERR_INVALID_ARG
    assert f(dt=9) == P.ERR_INVALID_ARG
    assert f(block=16) == P.ERR_INVALID_ARG
    assert f(d=80) == P.ERR_UNSUPPORTED


def test_forward_hybrid_rejects_bad_arguments(lib):
    # bf16 hi + lo copies of kbar, Vhat (2 x 2 heads x 2 blocks x d) and Hbar
    # (2 x 2 heads x d x d), rounded up to 256 bytes, then the plan: 4 query
    # blocks per 256 rows and head, int32
    plan = 2 * 4 * 1 * 4
    need = lib.pisa_forward_hybrid_workspace_size(1, 2, 128, 128)
    assert need == -(-(2 * 2 * 2 * 2 * 128 + 2 * 2 * 128 * 128) * 2 // 256) * 256 + plan
    assert lib.pisa_forward_hybrid_workspace_size(0, 2, 128, 128) == 0
    assert lib.pisa_forward_hybrid_workspace_size(1, 2, 128, 64) == (
        -(-(2 * 2 * 2 * 2 * 64 + 2 * 2 * 64 * 64) * 2 // 256) * 256 + plan)
    # 3 heads x 1000 rows: 16 blocks of 64 (the last partial), 8 query tiles, 4 CTAs
    assert lib.pisa_forward_hybrid_workspace_size(1, 3, 1000, 64) == (
        -(-(2 * 2 * 3 * 16 * 64 + 2 * 3 * 64 * 64) * 2 // 256) * 256 + 3 * 4 * 4 * 4)
    assert lib.pisa_forward_hybrid_workspace_size(1, 2, 128, 96) == 0
    f = lambda **kw: lib.pisa_forward_hybrid(
        kw.get("q", FAKE), FAKE, FAKE, 1, 2, 128, kw.get("d", 128), 64, ctypes.c_float(0.1),
        kw.get("kbar", FAKE), FAKE, kw.get("hbar", FAKE), FAKE, FAKE, 4, FAKE, 1,
        kw.get("ws", FAKE), kw.get("wsb", need), NULL, NULL)
    assert f(q=NULL) == P.ERR_INVALID_ARG
    assert f(kbar=NULL) == P.ERR_INVALID_ARG
    assert f(hbar=MISALIGNED) == P.ERR_INVALID_ARG
    assert f(ws=NULL) == P.ERR_INVALID_ARG
    assert f(wsb=need - 1) == P.ERR_INVALID_ARG
    assert f(d=48) == P.ERR_UNSUPPORTED


def test_selftest_rejects_bad_arguments(lib):
    assert lib.pisa_selftest_tc(NULL, FAKE, FAKE, FAKE, 0, NULL, NULL) == P.ERR_INVALID_ARG
    assert lib.pisa_selftest_tc(FAKE, FAKE, FAKE, FAKE, 2, NULL, NULL) == P.ERR_INVALID_ARG
    assert lib.pisa_selftest_tc(MISALIGNED, FAKE, FAKE, FAKE, 0, NULL, NULL) == P.ERR_INVALID_ARG


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "piecewise_sparse_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("oracle/", ""), f


def host_call(lib, q=FAKE, out=FAKE, in_dt=1, heads=4, n=256, d=128, block=64, scale=0.1, topk=2,
              band=1, out_dt=1, groups=2, taper=1, ws=FAKE, ws_bytes=1 << 30):
    return lib.pisa_attention_host(q, FAKE, FAKE, in_dt, heads, n, d, block, ctypes.c_float(scale),
                                   topk, band, out, out_dt, groups, taper, ws, ws_bytes, NULL, NULL)


def test_attention_host_rejects_bad_arguments_before_any_cuda_call(lib):
    big = lib.pisa_attention_host_workspace_size(1, 1, 4, 256, 128, 2, 1, 2, 1)
    ws = ctypes.c_void_p(0x100000)  # 256-byte aligned, never dereferenced
    assert host_call(lib, q=NULL, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, out=NULL, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, in_dt=7, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, out_dt=7, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, block=32, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, groups=0, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, groups=65, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, scale=-1.0, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, topk=-1, ws=ws, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, d=96, ws=ws, ws_bytes=big) == P.ERR_UNSUPPORTED
    # workspace: missing, misaligned, one byte short
    assert host_call(lib, ws=NULL, ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, ws=ctypes.c_void_p(0x100010), ws_bytes=big) == P.ERR_INVALID_ARG
    assert host_call(lib, ws=ws, ws_bytes=big - 1) == P.ERR_INVALID_ARG
    assert "workspace" in P.last_error()


def test_attention_host_workspace_size(lib):
    f = lib.pisa_attention_host_workspace_size
    # two buffer sets of the widest group: more groups, smaller workspace
    one = f(1, 1, 40, 32760, 128, 64, 1, 1, 0)
    ten = f(1, 1, 40, 32760, 128, 64, 1, 10, 1)
    assert one > ten > 0
    # bf16 in and out: two groups of 40 heads hold 2 x 4 x 40 x 32760 x 128 x 2 bytes of tensors
    assert one >= 2 * 4 * 40 * 32760 * 128 * 2
    assert f(1, 0, 40, 32760, 128, 64, 1, 1, 0) > one  # float32 output
    assert f(1, 1, 0, 32760, 128, 64, 1, 1, 0) == 0
