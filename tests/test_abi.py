"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/tsv.h declares; host-side argument checks need no device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(tsv_[a-z_0-9]+)\s*\(", text, re.M)
    return sorted(set(names))


def _build_module():
    import importlib.util
    path = os.path.join(ROOT, "tree_speculative_verification_attention_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("tsv_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(_build_module().build())


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tsv_tree_prepare", "tsv_tree_attention", "tsv_tree_verify_greedy",
              "tsv_tree_verify_stochastic", "tsv_create", "tsv_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _build_module().LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (tsv_[a-z_0-9]+)$", out, re.M))
    assert set(declared_functions()) <= exported


def test_binding_mirrors_the_header(lib):
    import tree_speculative_verification_attention_gb300 as tsv
    assert set(tsv.EXPORTED) == set(declared_functions())
    for name in tsv.EXPORTED:
        if name != "tsv_status_string":
            assert callable(getattr(tsv, name))


def header_constants():
    """Every numeric #define and enum value of the header (name -> value)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    found = {m.group(1): int(m.group(2)) for m in re.finditer(r"^#define\s+(TSV_[A-Z0-9_]+)\s+(\d+)u?\s*$", text, re.M)}
    for body in re.findall(r"typedef\s+enum\s*\{(.*?)\}", text, re.S):
        found.update({m.group(1): int(m.group(2)) for m in re.finditer(r"(TSV_[A-Z0-9_]+)\s*=\s*(\d+)", body)})
    return found


def test_binding_constants_match_the_header(lib):
    import tree_speculative_verification_attention_gb300 as tsv
    consts = header_constants()
    for name in ("TSV_OK", "TSV_ERR_TIMEOUT", "TSV_BF16", "TSV_MAX_NODES", "TSV_ANC_WORDS", "TSV_ATTN_SIMT",
                 "TSV_OVERLAP_GREEDY", "TSV_OVERLAP_STOCHASTIC", "TSV_OVERLAP_STOCHASTIC_FULL"):
        assert name in consts, name
    for name, value in consts.items():
        assert getattr(tsv, name) == value, name


def test_status_strings(lib):
    lib.tsv_status_string.restype = ctypes.c_char_p
    assert lib.tsv_status_string(0) == b"ok"
    assert b"tree" in lib.tsv_status_string(2)
    assert lib.tsv_status_string(99) == b"unknown status"
    assert lib.tsv_version() == 100


def test_null_handle_and_bad_arguments_are_rejected_on_the_host(lib):
    assert lib.tsv_destroy(None) == 1
    assert lib.tsv_tree_prepare(None, None, None, 1, None, None, None, None) == 1
    size = ctypes.c_size_t()
    assert lib.tsv_tree_verify_greedy_workspace_size(None, 1, 1, ctypes.c_int64(10), ctypes.byref(size)) == 1
    h = ctypes.c_void_p()
    assert lib.tsv_create(None, 0) == 1
    lib.tsv_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]
    assert lib.tsv_selftest_bounded_wait(None, 1, None, None, None) == 1


def test_every_entry_point_rejects_a_null_handle_on_the_host():
    """No call touches a device, or any pointer, before checking its handle."""
    import tree_speculative_verification_attention_gb300 as tsv
    L = tsv._lib
    size = ctypes.c_size_t()
    calls = {
        "tsv_tree_attention_workspace_size": (None, 1, 1, None, None, 1, 1, 64, 0, 0, ctypes.byref(size)),
        "tsv_tree_attention": (None, 1, None, None, None, 0, 0, 0, None, None, None, None, None, None, None,
                               1, 1, 1, 64, 0.0, None, 0, None, 0, None),
        "tsv_tree_verify_greedy_workspace_size": (None, 1, 1, 10, ctypes.byref(size)),
        "tsv_tree_verify_greedy": (None, None, 10, None, None, None, 1, 1, None, None, None, None, 0, None, None),
        "tsv_tree_verify_greedy_noalloc": (None, None, 10, None, None, None, 1, 1, None, None, None, None, None),
        "tsv_tree_verify_stochastic_workspace_size": (None, 1, 1, 10, ctypes.byref(size)),
        "tsv_tree_verify_stochastic": (None, None, None, 10, None, None, None, None, None, 1.0, 1, 1, None, None,
                                       None, None, None, 0, None, None),
        "tsv_tree_verify_stochastic_warped": (None, None, None, 10, None, None, None, None, None, 1.0, 5, 0.9, 1,
                                              1, None, None, None, None, None, 0, None, None),
        "tsv_tree_expand": (None, None, 10, 1, 1, None, None),
        "tsv_tree_merge": (None, None, None, None, None, 1, None, None, None, None, None, None),
        "tsv_kv_commit": (None, 1, None, None, 0, 0, 0, 1, 1, 64, None, None, None, None, None, None, None),
        "tsv_tree_prepare": (None, None, None, 1, None, None, None, None),
        "tsv_selftest_bounded_wait": (None, 1, None, None, None),
        "tsv_set_verify_overlap": (None, 1),
    }
    for name, args in calls.items():
        assert getattr(L, name)(*args) == tsv.TSV_ERR_INVALID_ARG, name
    # The other exports make or free a handle (checked above) or take none.
    assert set(calls) | {"tsv_create", "tsv_destroy", "tsv_status_string", "tsv_version"} == set(tsv.EXPORTED)


def test_create_without_a_device_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    h = ctypes.c_void_p()
    assert lib.tsv_create(ctypes.byref(h), 0) == 4
    assert not h.value


def test_plain_c_caller(lib, tmp_path):
    """include/tsv.h compiles as strict C99 and the library links into a C
    program that makes host-side calls (tests/c/abi_check.c)."""
    libdir = os.path.dirname(_build_module().LIB)
    exe = tmp_path / "abi_check"
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                         "-I" + os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_check.c"),
                         "-L" + libdir, "-ltsv", "-Wl,-rpath," + libdir, "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.startswith("bad tree")

