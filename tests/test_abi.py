"""The C ABI library without a GPU: it loads, exports every declared entry
point, and rejects bad arguments on the host before touching the device."""
import ctypes
import glob
import os
import re

import pytest

import allreduce_reduction_emulated_gb300 as ar
from allreduce_reduction_emulated_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ar.library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ar_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ar_init", "ar_allreduce", "ar_destroy", "ar_get_status", "ar_get_error_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libar.so does not export {name}"


def test_library_is_built_for_sm_103a():
    text = open(_build.__file__).read()
    assert "arch=compute_103a,code=sm_103a" in text


def test_error_strings(lib):
    for st in range(6):
        assert ar.ar_get_error_string(st)
    assert ar.ar_get_error_string(99) == "unknown status"


def test_host_argument_checks_without_device(lib):
    vp = ctypes.c_void_p
    h = vp()
    assert lib.ar_init(0, ctypes.byref(h)) == ar.AR_ERR_INVALID_ARG
    assert lib.ar_init(ar.AR_MAX_RANKS + 1, ctypes.byref(h)) == ar.AR_ERR_INVALID_ARG
    assert lib.ar_init(4, None) == ar.AR_ERR_INVALID_ARG
    arr = (vp * 1)(None)
    assert lib.ar_allreduce(None, arr, arr, 4, 0, 0, 1, 1.0, None) == ar.AR_ERR_INVALID_ARG
    assert lib.ar_destroy(None) == ar.AR_SUCCESS
    assert lib.ar_get_status(None) == ar.AR_ERR_INVALID_ARG
    assert lib.ar_set_option(None, 0, 1) == ar.AR_ERR_INVALID_ARG
    out = ctypes.c_int()
    assert lib.ar_select_algo(None, 4, 0, 0, ctypes.byref(out)) == ar.AR_ERR_INVALID_ARG


def test_no_gpu_means_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert lib.ar_init(8, ctypes.byref(h)) == ar.AR_ERR_CUDA
    assert h.value is None


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "allreduce_reduction_emulated_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            text = open(path).read()
            assert "oracle" not in text.lower(), f"{path} mentions the oracle"
