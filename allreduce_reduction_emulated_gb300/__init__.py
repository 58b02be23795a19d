"""Python binding of libar.so: an all-reduce over P ranks emulated as P buffers
in one GPU's memory (the C ABI is declared in include/ar.h).

Argument marshalling only: tensors become device pointers, torch streams
become cudaStream_t handles, status codes become exceptions.  Every step of
the all-reduce runs in the library's CUDA kernels; there is no fallback --
if libar.so is missing or cannot be loaded, every call raises.

    comm = ar_init(P)
    ar_allreduce(comm, sends, recvs, count, AR_FLOAT32, AR_SUM, AR_ALGO_RING, scale, stream)
    ar_destroy(comm)

``allreduce(sends, recvs, op="sum", algo="auto", scale=1.0)`` is the same
call with dtype / count taken from the tensors and a cached communicator.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libar.so")

# ar_status_t
AR_SUCCESS, AR_ERR_INVALID_ARG, AR_ERR_CUDA, AR_ERR_UNSUPPORTED, AR_ERR_TIMEOUT, AR_ERR_OOM = range(6)
# ar_dtype_t, ar_op_t, ar_algo_t, ar_option_t
AR_FLOAT32, AR_BFLOAT16, AR_INT32 = 0, 1, 2
AR_SUM, AR_MIN, AR_MAX = 0, 1, 2
AR_ALGO_AUTO, AR_ALGO_RING, AR_ALGO_TREE, AR_ALGO_LL, AR_ALGO_HIER, AR_ALGO_LL128 = range(6)
(AR_OPT_LL_MAX_BYTES, AR_OPT_LL_SPIN_LIMIT, AR_OPT_DEBUG, AR_OPT_LL_SKIP_PRODUCER, AR_OPT_HIER_GROUP,
 AR_OPT_MAX_BLOCKS, AR_OPT_LL128_MAX_BYTES, AR_OPT_AUTO_TUNED) = range(8)
AR_OPT_LL_EPOCH = 8
AR_OPT_CAPPED_KERNEL = 9
AR_CAPPED_WIDE, AR_CAPPED_TMA = 0, 1
AR_TUNE_BUCKETS = 22
AR_MAX_RANKS = 256
AR_NOALLOC_MAX_RANKS, AR_NOALLOC_MAX_BYTES = 8, 65536

OPS = {"sum": AR_SUM, "min": AR_MIN, "max": AR_MAX}
ALGOS = {"auto": AR_ALGO_AUTO, "ring": AR_ALGO_RING, "tree": AR_ALGO_TREE, "ll": AR_ALGO_LL,
         "hier": AR_ALGO_HIER, "ll128": AR_ALGO_LL128}


class ArError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ar_get_error_string(status)} (status {status})")


_lib = None
_lib_lock = threading.Lock()


def library() -> ctypes.CDLL:
    """The loaded libar.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                                       "(python -c 'import __graft_entry__ as g; g.build()')")
                L = ctypes.CDLL(LIB_PATH)
                vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
                L.ar_init.argtypes = [i, ctypes.POINTER(vp)]
                L.ar_init.restype = i
                L.ar_allreduce.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i, i, i,
                                           ctypes.c_float, vp]
                L.ar_allreduce.restype = i
                L.ar_get_status.argtypes = [vp]
                L.ar_get_status.restype = i
                L.ar_get_error_string.argtypes = [i]
                L.ar_get_error_string.restype = ctypes.c_char_p
                L.ar_destroy.argtypes = [vp]
                L.ar_destroy.restype = i
                L.ar_select_algo.argtypes = [vp, sz, i, i, ctypes.POINTER(i)]
                L.ar_select_algo.restype = i
                L.ar_set_option.argtypes = [vp, i, ctypes.c_longlong]
                L.ar_set_option.restype = i
                L.ar_tune.argtypes = [vp, ctypes.POINTER(i), i]
                L.ar_tune.restype = i
                L.ar_reduce_scatter.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i, i,
                                                 ctypes.c_float, vp]
                L.ar_reduce_scatter.restype = i
                L.ar_all_gather.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i, vp]
                L.ar_all_gather.restype = i
                L.ar_allreduce_ll_noalloc.argtypes = [i, ctypes.POINTER(vp), ctypes.POINTER(vp), sz,
                                                      i, i, ctypes.c_float, vp, ctypes.POINTER(i)]
                L.ar_allreduce_ll_noalloc.restype = i
                _lib = L
    return _lib


_ESIZE = {AR_FLOAT32: 4, AR_BFLOAT16: 2, AR_INT32: 4}


def _current_device() -> int:
    import torch

    return torch.cuda.current_device()


def _ptr(x, elems: int, dtype: int, what: str, device: int | None = None) -> int:
    """Device address of a buffer: a raw pointer (int) is passed through; a
    tensor must be contiguous CUDA memory on the current device (`device`)
    holding at least `elems` elements of the data type's size, else
    ArError(AR_ERR_INVALID_ARG) -- the library only sees a pointer and launches
    on the current device, so these are the checks it cannot make.  A tensor
    on another GPU is refused before anything is launched: the kernels would
    otherwise read or write that GPU's memory."""
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ArError(AR_ERR_INVALID_ARG, f"{what}: tensor is not contiguous")
    if not x.is_cuda:
        raise ArError(AR_ERR_INVALID_ARG, f"{what}: tensor is not in CUDA memory")
    if device is None:
        device = _current_device()
    if x.device.index != device:
        raise ArError(AR_ERR_INVALID_ARG, f"{what}: tensor is on cuda:{x.device.index}, "
                                          f"the current device is cuda:{device}")
    if x.element_size() != _ESIZE.get(int(dtype), 0):
        raise ArError(AR_ERR_INVALID_ARG, f"{what}: {x.element_size()}-byte elements for this data type")
    if x.numel() < elems:
        raise ArError(AR_ERR_INVALID_ARG, f"{what}: {x.numel()} elements, {elems} needed")
    return x.data_ptr()


def _ptrs(bufs, elems: int, dtype: int, what: str):
    device = _current_device() if any(getattr(b, "is_cuda", False) for b in bufs) else None
    return (ctypes.c_void_p * len(bufs))(*[_ptr(b, elems, dtype, f"{what}[{i}]", device)
                                           for i, b in enumerate(bufs)])


def _stream_handle(stream) -> int:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def ar_get_error_string(status: int) -> str:
    return library().ar_get_error_string(int(status)).decode()


def ar_init(nranks: int) -> int:
    """Creates a communicator for nranks emulated ranks on the current device."""
    h = ctypes.c_void_p()
    st = library().ar_init(int(nranks), ctypes.byref(h))
    if st != AR_SUCCESS:
        raise ArError(st, "ar_init")
    return h.value


def ar_destroy(comm: int) -> None:
    st = library().ar_destroy(comm)
    if st != AR_SUCCESS:
        raise ArError(st, "ar_destroy")


def ar_allreduce(comm: int, sendbufs, recvbufs, count: int, dtype: int, op: int = AR_SUM,
                 algo: int = AR_ALGO_AUTO, scale: float = 1.0, stream=None) -> None:
    """sendbufs / recvbufs: P device tensors or raw device pointers."""
    P = len(sendbufs)
    if len(recvbufs) != P:
        raise ArError(AR_ERR_INVALID_ARG, "ar_allreduce: sendbufs and recvbufs differ in length")
    sp = _ptrs(sendbufs, int(count), dtype, "ar_allreduce sendbufs")
    rp = _ptrs(recvbufs, int(count), dtype, "ar_allreduce recvbufs")
    st = library().ar_allreduce(comm, sp, rp, int(count), int(dtype), int(op), int(algo),
                                float(scale), _stream_handle(stream))
    if st != AR_SUCCESS:
        raise ArError(st, "ar_allreduce")


def ar_reduce_scatter(comm: int, sendbufs, recvbufs, recvcount: int, dtype: int, op: int = AR_SUM,
                      scale: float = 1.0, stream=None) -> None:
    """sendbufs: P buffers of P * recvcount elements; recvbufs[s] gets shard s."""
    P = len(sendbufs)
    if len(recvbufs) != P:
        raise ArError(AR_ERR_INVALID_ARG, "ar_reduce_scatter: sendbufs and recvbufs differ in length")
    sp = _ptrs(sendbufs, P * int(recvcount), dtype, "ar_reduce_scatter sendbufs")
    rp = _ptrs(recvbufs, int(recvcount), dtype, "ar_reduce_scatter recvbufs")
    st = library().ar_reduce_scatter(comm, sp, rp, int(recvcount), int(dtype), int(op), float(scale),
                                     _stream_handle(stream))
    if st != AR_SUCCESS:
        raise ArError(st, "ar_reduce_scatter")


def ar_all_gather(comm: int, sendbufs, recvbufs, sendcount: int, dtype: int, stream=None) -> None:
    """sendbufs: P buffers of sendcount elements; every recvbufs[r] gets all P of them."""
    P = len(sendbufs)
    if len(recvbufs) != P:
        raise ArError(AR_ERR_INVALID_ARG, "ar_all_gather: sendbufs and recvbufs differ in length")
    sp = _ptrs(sendbufs, int(sendcount), dtype, "ar_all_gather sendbufs")
    rp = _ptrs(recvbufs, P * int(sendcount), dtype, "ar_all_gather recvbufs")
    st = library().ar_all_gather(comm, sp, rp, int(sendcount), int(dtype), _stream_handle(stream))
    if st != AR_SUCCESS:
        raise ArError(st, "ar_all_gather")


def ar_get_status(comm: int) -> int:
    """Device-side status since the last query (call after synchronizing)."""
    return int(library().ar_get_status(comm))


def ar_select_algo(comm: int, count: int, dtype: int, algo: int = AR_ALGO_AUTO) -> int:
    out = ctypes.c_int()
    st = library().ar_select_algo(comm, int(count), int(dtype), int(algo), ctypes.byref(out))
    if st != AR_SUCCESS:
        raise ArError(st, "ar_select_algo")
    return out.value


def ar_tune(comm: int) -> list:
    """Times ring / tree / LL / LL128 per size on this device and makes AUTO use
    the fastest; returns the chosen algorithm for 8 B, 16 B, ... 16 MiB per rank."""
    table = (ctypes.c_int * AR_TUNE_BUCKETS)()
    st = library().ar_tune(comm, table, AR_TUNE_BUCKETS)
    if st != AR_SUCCESS:
        raise ArError(st, "ar_tune")
    return list(table)


def ar_set_option(comm: int, option: int, value: int) -> None:
    st = library().ar_set_option(comm, int(option), int(value))
    if st != AR_SUCCESS:
        raise ArError(st, "ar_set_option")


def ar_allreduce_ll_noalloc(sendbufs, recvbufs, count: int, dtype: int, op: int = AR_SUM,
                            scale: float = 1.0, stream=None, wait_status: bool = False):
    """LL all-reduce that allocates no device memory (for callers that cannot).

    Limited to AR_NOALLOC_MAX_RANKS ranks and AR_NOALLOC_MAX_BYTES bytes per
    rank.  With wait_status=True the call waits for the stream and returns the
    device status (AR_SUCCESS or AR_ERR_TIMEOUT); otherwise it returns None.
    """
    P = len(sendbufs)
    if len(recvbufs) != P:
        raise ArError(AR_ERR_INVALID_ARG, "ar_allreduce_ll_noalloc: sendbufs and recvbufs differ in length")
    sp = _ptrs(sendbufs, int(count), dtype, "ar_allreduce_ll_noalloc sendbufs")
    rp = _ptrs(recvbufs, int(count), dtype, "ar_allreduce_ll_noalloc recvbufs")
    status = ctypes.c_int(-1)
    st = library().ar_allreduce_ll_noalloc(P, sp, rp, int(count), int(dtype), int(op), float(scale),
                                           _stream_handle(stream),
                                           ctypes.byref(status) if wait_status else None)
    if st != AR_SUCCESS:
        raise ArError(st, "ar_allreduce_ll_noalloc")
    return status.value if wait_status else None


# ------------------------------------------------------------- convenience

_comms: dict = {}
_comms_lock = threading.Lock()


def dtype_of(t) -> int:
    import torch

    table = {torch.float32: AR_FLOAT32, torch.bfloat16: AR_BFLOAT16, torch.int32: AR_INT32}
    if t.dtype not in table:
        raise ArError(AR_ERR_UNSUPPORTED, f"dtype {t.dtype}")
    return table[t.dtype]


def allreduce(sends, recvs=None, op: str = "sum", algo: str = "auto", scale: float = 1.0,
              stream=None):
    """All-reduce of P same-shaped contiguous CUDA tensors; returns recvs.

    recvs=None reduces in place.  A communicator per (P, device) is created on
    first use and kept for the life of the process; calls that share it must
    not overlap on the GPU (one stream, or streams ordered by events), as for
    any communicator.
    """
    import torch

    if op not in OPS or algo not in ALGOS:
        raise ArError(AR_ERR_INVALID_ARG, f"allreduce: op must be one of {sorted(OPS)}, "
                                          f"algo one of {sorted(ALGOS)}")
    if len(sends) == 0:
        raise ArError(AR_ERR_INVALID_ARG, "allreduce: no tensors")
    recvs = list(sends) if recvs is None else list(recvs)
    t0 = sends[0]
    for t in list(sends) + recvs:
        if not t.is_cuda or not t.is_contiguous() or t.dtype != t0.dtype or t.numel() != t0.numel():
            raise ArError(AR_ERR_INVALID_ARG, "allreduce: tensors must be contiguous CUDA tensors "
                                              "of one dtype and size")
        if t.device != t0.device:
            raise ArError(AR_ERR_INVALID_ARG, f"allreduce: tensors on {t0.device} and {t.device}; "
                                              "all must be on one GPU")
    key = (len(sends), t0.device.index if t0.device.index is not None else torch.cuda.current_device())
    with _comms_lock:
        if key not in _comms:
            with torch.cuda.device(key[1]):
                _comms[key] = ar_init(len(sends))
    with torch.cuda.device(key[1]):
        ar_allreduce(_comms[key], sends, recvs, t0.numel(), dtype_of(t0), OPS[op], ALGOS[algo],
                     scale, stream)
    return recvs
