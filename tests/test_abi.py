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


def test_binding_rejects_tensors_the_library_cannot_check():
    """The C ABI sees only pointers: the binding refuses tensors that are not
    contiguous, not in CUDA memory, too short or of the wrong element size
    before any call reaches the library (so these run without a GPU)."""
    import torch

    x = torch.zeros(64)
    cases = [
        (lambda: ar.ar_allreduce(1, [x[::2]], [x[::2]], 8, ar.AR_FLOAT32), "not contiguous"),
        (lambda: ar.ar_allreduce(1, [x], [x], 8, ar.AR_FLOAT32), "not in CUDA memory"),
        (lambda: ar.ar_reduce_scatter(1, [x, x], [x, x], 40, ar.AR_FLOAT32), "not in CUDA memory"),
        (lambda: ar.ar_all_gather(1, [x], [x[:3].clone()], 8, ar.AR_FLOAT32), "not in CUDA memory"),
    ]
    for call, reason in cases:
        with pytest.raises(ar.ArError) as e:
            call()
        assert e.value.status == ar.AR_ERR_INVALID_ARG and reason in str(e.value)


class CudaLike:
    """Stands in for a CUDA tensor on device `index` (a CPU tensor's memory)."""

    def __init__(self, t, index: int = 0):
        import torch

        self.t = t
        self.is_cuda = True
        self.device = torch.device("cuda", index)
        self.dtype = t.dtype

    def is_contiguous(self):
        return self.t.is_contiguous()

    def element_size(self):
        return self.t.element_size()

    def numel(self):
        return self.t.numel()

    def data_ptr(self):
        return self.t.data_ptr()


def test_binding_checks_length_and_element_size(monkeypatch):
    """Length and element size, with the CUDA check satisfied by a stand-in."""
    import torch

    monkeypatch.setattr(ar, "_current_device", lambda: 0)

    short = CudaLike(torch.zeros(7))
    wide = CudaLike(torch.zeros(16, dtype=torch.float64))
    with pytest.raises(ar.ArError) as e:
        ar._ptrs([short], 8, ar.AR_FLOAT32, "x")
    assert "7 elements, 8 needed" in str(e.value)
    with pytest.raises(ar.ArError) as e:
        ar._ptrs([wide], 8, ar.AR_FLOAT32, "x")
    assert "8-byte elements" in str(e.value)
    ok = CudaLike(torch.zeros(8, dtype=torch.int16))
    assert ar._ptrs([ok], 8, ar.AR_BFLOAT16, "x")[0] == ok.data_ptr()
    # reduce-scatter inputs need P * recvcount elements, all-gather outputs too
    with pytest.raises(ar.ArError) as e:
        ar._ptrs([CudaLike(torch.zeros(15))], 2 * 8, ar.AR_FLOAT32, "x")
    assert "15 elements, 16 needed" in str(e.value)


def test_convenience_call_rejects_bad_names_and_empty_input():
    import torch

    x = torch.zeros(8)
    for kw, reason in ((dict(op="avg"), "op must be one of"), (dict(algo="nvls"), "algo one of")):
        with pytest.raises(ar.ArError) as e:
            ar.allreduce([x, x], **kw)
        assert e.value.status == ar.AR_ERR_INVALID_ARG and reason in str(e.value)
    with pytest.raises(ar.ArError) as e:
        ar.allreduce([])
    assert "no tensors" in str(e.value)
    with pytest.raises(ar.ArError) as e:
        ar.allreduce([x, x])                       # CPU tensors: refused before the library
    assert "contiguous CUDA tensors" in str(e.value)


def test_binding_refuses_a_tensor_on_another_gpu(monkeypatch):
    """The kernels launch on the current device; a buffer on another GPU is
    refused with AR_ERR_INVALID_ARG before the library is called."""
    import torch

    monkeypatch.setattr(ar, "_current_device", lambda: 0)

    def fail(*a, **k):
        raise AssertionError("the library must not be called")

    monkeypatch.setattr(ar, "library", lambda: type("L", (), {"__getattr__": lambda self, n: fail,
                                                             "ar_get_error_string": lambda self, s: b"x"})())
    here = [CudaLike(torch.zeros(16)) for _ in range(2)]
    there = CudaLike(torch.zeros(16), index=1)
    calls = (
        lambda: ar.ar_allreduce(1, [here[0], there], here, 16, ar.AR_FLOAT32),
        lambda: ar.ar_allreduce(1, here, [here[0], there], 16, ar.AR_FLOAT32),
        lambda: ar.ar_reduce_scatter(1, [CudaLike(torch.zeros(32)), CudaLike(torch.zeros(32), 1)],
                                     here, 16, ar.AR_FLOAT32),
        lambda: ar.ar_all_gather(1, here, [CudaLike(torch.zeros(32), 1), CudaLike(torch.zeros(32))],
                                 16, ar.AR_FLOAT32),
        lambda: ar.ar_allreduce_ll_noalloc([there, here[1]], here, 16, ar.AR_FLOAT32),
    )
    for call in calls:
        with pytest.raises(ar.ArError) as e:
            call()
        assert e.value.status == ar.AR_ERR_INVALID_ARG and "cuda:1" in str(e.value)
    # the convenience call: every tensor on the first tensor's device
    with pytest.raises(ar.ArError) as e:
        ar.allreduce([here[0], there])
    assert e.value.status == ar.AR_ERR_INVALID_ARG and "one GPU" in str(e.value)
