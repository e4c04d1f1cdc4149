"""The C ABI without a GPU: the library builds, loads and exports every
function include/kmassign.h declares; argument errors come back as status
codes before anything touches CUDA."""

import ctypes
import os
import re

import pytest

import means_nearest_centroid_gb300 as km
from means_nearest_centroid_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b(kmassign\w*)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return km.library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["kmassign", "kmassign_norms", "kmassign_ex", "kmassign_plan", "kmassign_check",
              "kmassign_strerror", "kmassign_topk", "kmassign_topk_ex"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(km.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_strerror_covers_every_code(lib):
    for name, code in km.STATUS.items():
        text = km.kmassign_strerror(code)
        assert text and "unknown" not in text, name
    assert "unknown" in km.kmassign_strerror(12345)


P = ctypes.c_void_p
NULL = P(0)
A16 = P(0x10000)           # aligned fake addresses: never dereferenced, the
A16B = P(0x20000)          # checks below fail before any pointer is used
MIS = P(0x10008)           # 8-byte aligned only


def call(lib, X=A16, C=A16B, cn=NULL, N=10, K=5, D=64, idx=A16, ms=NULL):
    return lib.kmassign(X, C, cn, N, K, D, idx, ms, NULL)


def test_shape_errors(lib):
    S = km.STATUS
    assert call(lib, N=-1) == S["KMASSIGN_ERR_SHAPE"]
    assert call(lib, N=2**31) == S["KMASSIGN_ERR_SHAPE"]
    assert call(lib, K=0) == S["KMASSIGN_ERR_SHAPE"]
    assert call(lib, K=2**31) == S["KMASSIGN_ERR_SHAPE"]
    for D in (0, 8, 24, 272, 512, -16):
        assert call(lib, D=D) == S["KMASSIGN_ERR_UNSUPPORTED_D"], D


def test_empty_input_is_a_no_op(lib):
    assert call(lib, X=NULL, idx=NULL, N=0) == 0


def test_null_and_alignment_errors(lib):
    S = km.STATUS
    assert call(lib, X=NULL) == S["KMASSIGN_ERR_NULL"]
    assert call(lib, C=NULL) == S["KMASSIGN_ERR_NULL"]
    assert call(lib, idx=NULL) == S["KMASSIGN_ERR_NULL"]
    assert call(lib, X=MIS) == S["KMASSIGN_ERR_ALIGN"]
    assert call(lib, C=MIS) == S["KMASSIGN_ERR_ALIGN"]
    assert call(lib, cn=MIS) == S["KMASSIGN_ERR_ALIGN"]
    assert call(lib, idx=P(0x10002)) == S["KMASSIGN_ERR_ALIGN"]
    assert call(lib, ms=P(0x10001)) == S["KMASSIGN_ERR_ALIGN"]


def test_plan_value_errors(lib):
    S = km.STATUS
    ex = lib.kmassign_ex
    assert ex(A16, A16B, NULL, 10, 5, 64, A16, NULL, -1, 0, 0, 0, NULL) == S["KMASSIGN_ERR_ARG"]
    assert ex(A16, A16B, NULL, 10, 5, 64, A16, NULL, 0, 64, 0, 0, NULL) == S["KMASSIGN_ERR_ARG"]
    assert ex(A16, A16B, NULL, 10, 5, 64, A16, NULL, 0, 0, 96, 0, NULL) == S["KMASSIGN_ERR_ARG"]
    assert ex(A16, A16B, NULL, 10, 5, 64, A16, NULL, 0, 0, 0, 32, NULL) == S["KMASSIGN_ERR_ARG"]
    assert ex(A16, A16B, NULL, 10, 5, 64, A16, NULL, 0, 0, 0, 12, NULL) == S["KMASSIGN_ERR_ARG"]


def test_norms_argument_errors(lib):
    S = km.STATUS
    assert lib.kmassign_norms(A16, 0, 64, A16B, NULL) == S["KMASSIGN_ERR_SHAPE"]
    assert lib.kmassign_norms(A16, 4, 40, A16B, NULL) == S["KMASSIGN_ERR_UNSUPPORTED_D"]
    assert lib.kmassign_norms(NULL, 4, 64, A16B, NULL) == S["KMASSIGN_ERR_NULL"]
    assert lib.kmassign_norms(A16, 4, 64, NULL, NULL) == S["KMASSIGN_ERR_NULL"]
    assert lib.kmassign_norms(MIS, 4, 64, A16B, NULL) == S["KMASSIGN_ERR_ALIGN"]


def topk(lib, X=A16, C=A16B, cn=NULL, N=10, K=5, D=64, k=3, idx=A16, sc=NULL, dist=0, ksplit=None):
    if ksplit is None:
        return lib.kmassign_topk(X, C, cn, N, K, D, k, idx, sc, dist, NULL)
    return lib.kmassign_topk_ex(X, C, cn, N, K, D, k, idx, sc, dist, ksplit, NULL)


def test_topk_argument_errors(lib):
    S = km.STATUS
    for k in (0, -1, 6, 33):                       # k in [1, min(K, 32)]
        assert topk(lib, k=k, K=5) == S["KMASSIGN_ERR_ARG"], k
    assert topk(lib, k=33, K=100) == S["KMASSIGN_ERR_ARG"]
    assert topk(lib, dist=2) == S["KMASSIGN_ERR_ARG"]
    assert topk(lib, ksplit=-1) == S["KMASSIGN_ERR_ARG"]
    assert topk(lib, N=2**26, k=32, K=64) == S["KMASSIGN_ERR_SHAPE"]     # N * k >= 2^31
    assert topk(lib, D=40) == S["KMASSIGN_ERR_UNSUPPORTED_D"]
    assert topk(lib, N=0, X=NULL, idx=NULL) == 0
    assert topk(lib, X=NULL) == S["KMASSIGN_ERR_NULL"]
    assert topk(lib, idx=NULL) == S["KMASSIGN_ERR_NULL"]
    assert topk(lib, dist=1, sc=NULL) == S["KMASSIGN_ERR_NULL"]      # distances need an output
    assert topk(lib, X=MIS) == S["KMASSIGN_ERR_ALIGN"]
    assert topk(lib, sc=P(0x10002)) == S["KMASSIGN_ERR_ALIGN"]


def test_plan_rejects_null_output(lib):
    assert lib.kmassign_plan(10, 5, 64, NULL) == km.STATUS["KMASSIGN_ERR_NULL"]
    assert lib.kmassign_plan_ex(10, 5, 64, 0, 0, 0, 0, NULL) == km.STATUS["KMASSIGN_ERR_NULL"]


def test_plan_ex_rejects_forcing_arguments_no_kernel_has(lib):
    """Checked before the device is queried, as kmassign_ex checks them."""
    out = (ctypes.c_int32 * 9)()
    o = ctypes.cast(out, ctypes.c_void_p)
    for ks, rows, nt, cw in [(-1, 0, 0, 0), (0, 64, 0, 0), (0, 0, 512, 0), (0, 0, 0, 12)]:
        assert lib.kmassign_plan_ex(10, 5, 64, ks, rows, nt, cw, o) == km.STATUS["KMASSIGN_ERR_ARG"]
    assert lib.kmassign_plan_ex(10, 5, 40, 0, 0, 0, 0, o) == km.STATUS["KMASSIGN_ERR_UNSUPPORTED_D"]


def test_binding_fails_loudly_without_library(tmp_path):
    import means_nearest_centroid_gb300 as mod
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError, match="no CPU fallback"):
            mod.library(str(tmp_path / "missing.so"))
    finally:
        mod._lib = saved


def host_call(lib, X=A16, C=A16B, cn=NULL, N=10, K=5, D=64, idx=A16, ms=NULL, rows=0):
    return lib.kmassign_host_ex(X, C, cn, N, K, D, idx, ms, rows, NULL)


def test_host_path_argument_errors(lib):
    """kmassign_host checks its arguments before touching CUDA."""
    S = km.STATUS
    assert host_call(lib, N=-1) == S["KMASSIGN_ERR_SHAPE"]
    assert host_call(lib, K=0) == S["KMASSIGN_ERR_SHAPE"]
    for D in (0, 8, 24, 272):
        assert host_call(lib, D=D) == S["KMASSIGN_ERR_UNSUPPORTED_D"], D
    assert host_call(lib, rows=-1) == S["KMASSIGN_ERR_ARG"]
    assert host_call(lib, X=NULL, idx=NULL, N=0) == 0
    assert host_call(lib, X=NULL) == S["KMASSIGN_ERR_NULL"]
    assert host_call(lib, C=NULL) == S["KMASSIGN_ERR_NULL"]
    assert host_call(lib, idx=NULL) == S["KMASSIGN_ERR_NULL"]
    # no alignment is required of host buffers: a misaligned pointer passes
    # the checks and fails only for want of a GPU here
    assert lib.kmassign_host(MIS, A16B, NULL, 10, 5, 64, A16, NULL, NULL) != \
        S["KMASSIGN_ERR_ALIGN"]
