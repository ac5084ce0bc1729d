"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/sparse_attn.h declares, and rejects bad
arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparse_attn.h")


@pytest.fixture(scope="module")
def lib_path():
    from video_dit_sparse_gb300 import build
    return build.build()


@pytest.fixture(scope="module")
def lib(lib_path):
    return ctypes.CDLL(lib_path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sparse_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sparse_attn_build_index", "sparse_attn_forward", "sparse_attn_validate_index",
              "sparse_attn_build_index_workspace_size", "sparse_attn_status_string",
              "sparse_attn_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib_path, lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_library_targets_sm103a(lib_path):
    from video_dit_sparse_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Nq", ctypes.c_int32),
                ("Nk", ctypes.c_int32), ("d", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("scale", ctypes.c_float), ("out_dtype", ctypes.c_int32)]


class Select(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("topk", ctypes.c_int64),
                ("threshold", ctypes.c_double), ("mass", ctypes.c_double)]


def _sigs(lib):
    P, vp, i64 = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int64
    lib.sparse_attn_forward.argtypes = [P(Problem), vp, vp, vp, vp, vp, i64, vp, vp, vp, vp]
    lib.sparse_attn_forward.restype = ctypes.c_int
    lib.sparse_attn_build_index.argtypes = [P(Problem), P(Select), vp, vp, vp, vp, i64,
                                            P(ctypes.c_int64), vp, ctypes.c_size_t, vp]
    lib.sparse_attn_build_index.restype = ctypes.c_int
    lib.sparse_attn_build_index_workspace_size.argtypes = [P(Problem)]
    lib.sparse_attn_build_index_workspace_size.restype = ctypes.c_size_t
    lib.sparse_attn_validate_index.argtypes = [P(Problem), vp, vp, i64, vp, vp]
    lib.sparse_attn_validate_index.restype = ctypes.c_int
    lib.sparse_attn_status_string.argtypes = [ctypes.c_int]
    lib.sparse_attn_status_string.restype = ctypes.c_char_p


def test_status_strings_and_version(lib):
    _sigs(lib)
    names = [lib.sparse_attn_status_string(i).decode() for i in range(7)]
    assert names[0] == "ok" and len(set(names)) == 7
    assert lib.sparse_attn_version() >= 10000


def test_workspace_size(lib):
    _sigs(lib)
    p = Problem(1, 24, 16384, 16384, 128, 128, 128 ** -0.5)
    ws = lib.sparse_attn_build_index_workspace_size(ctypes.byref(p))
    rows = 24 * 128
    assert ws >= rows * 16384 * 4 + 2 * rows * 128 * 2
    assert ws % 256 == 0
    for bad in (Problem(0, 1, 8, 8, 128, 128, 1.0), Problem(1, 1, 8, 8, 96, 128, 1.0),
                Problem(1, 1, 8, 8, 128, 0, 1.0), Problem(1, 1, 8, 8, 128, 300, 1.0),
                Problem(1, 1, 8, 8, 128, 128, float("nan"))):
        assert lib.sparse_attn_build_index_workspace_size(ctypes.byref(bad)) == 0
    assert lib.sparse_attn_build_index_workspace_size(None) == 0


def test_host_argument_checks(lib):
    """Rejected before any CUDA call, so these run without a GPU."""
    _sigs(lib)
    ok = Problem(1, 1, 256, 256, 128, 128, 128 ** -0.5)
    a16 = ctypes.c_void_p(0x10000)
    mis = ctypes.c_void_p(0x10008)
    f = lib.sparse_attn_forward
    assert f(None, a16, a16, a16, a16, a16, 1, a16, None, None, None) == 1
    assert f(ctypes.byref(ok), None, a16, a16, a16, a16, 1, a16, None, None, None) == 1
    assert f(ctypes.byref(ok), mis, a16, a16, a16, a16, 1, a16, None, None, None) == 1
    assert f(ctypes.byref(ok), a16, a16, a16, a16, None, 5, a16, None, None, None) == 1
    assert f(ctypes.byref(ok), a16, a16, a16, a16, a16, -1, a16, None, None, None) == 1
    d96 = Problem(1, 1, 256, 256, 96, 128, 1.0)
    assert f(ctypes.byref(d96), a16, a16, a16, a16, a16, 1, a16, None, None, None) == 2
    m300 = Problem(1, 1, 256, 256, 128, 300, 1.0)
    assert f(ctypes.byref(m300), a16, a16, a16, a16, a16, 1, a16, None, None, None) == 2
    bad_out = Problem(1, 1, 256, 256, 128, 128, 1.0, 7)
    assert f(ctypes.byref(bad_out), a16, a16, a16, a16, a16, 1, a16, None, None, None) == 1
    b = lib.sparse_attn_build_index
    nnz = ctypes.c_int64(0)
    top = Select(0, 16, 0.0, 0.0)
    assert b(ctypes.byref(ok), None, a16, a16, a16, a16, 1 << 20, None, a16, 1 << 30, None) == 1
    assert b(ctypes.byref(ok), ctypes.byref(Select(0, 0, 0.0, 0.0)), a16, a16, a16, a16, 1 << 20,
             None, a16, 1 << 30, None) == 1
    assert b(ctypes.byref(ok), ctypes.byref(Select(2, 0, 0.0, 1.5)), a16, a16, a16, a16, 1 << 20,
             None, a16, 1 << 30, None) == 1
    assert b(ctypes.byref(ok), ctypes.byref(Select(1, 0, -0.1, 0.0)), a16, a16, a16, a16, 1 << 20,
             None, a16, 1 << 30, None) == 1
    assert b(ctypes.byref(ok), ctypes.byref(Select(7, 1, 0.0, 0.0)), a16, a16, a16, a16, 1 << 20,
             None, a16, 1 << 30, None) == 1
    # workspace too small
    assert b(ctypes.byref(ok), ctypes.byref(top), a16, a16, a16, a16, 1 << 20, None, a16, 64, None) == 1
    # TOPK capacity is known up front: 2 groups x 16 keys do not fit in 31
    assert b(ctypes.byref(ok), ctypes.byref(top), a16, a16, a16, a16, 31, ctypes.byref(nnz), a16,
             1 << 30, None) == 3
    assert nnz.value == 32
    # MASS without a host nnz needs worst-case capacity
    mass = Select(2, 0, 0.0, 0.99)
    assert b(ctypes.byref(ok), ctypes.byref(mass), a16, a16, a16, a16, 100, None, a16, 1 << 30, None) == 1
    v = lib.sparse_attn_validate_index
    assert v(ctypes.byref(ok), a16, a16, 4, None, None) == 1
