"""Thin ctypes binding of libhisa (include/hisa.h): the same names, argument
marshalling only. Tensors are torch CUDA tensors; the call is enqueued on the
current torch stream unless a stream is given. Every computation runs in the
library's CUDA kernels; there is no Python or CPU fallback: if libhisa.so is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhisa.so")

HISA_OK, HISA_EINVAL, HISA_EDTYPE, HISA_EWORKSPACE, HISA_ECUDA, HISA_EDEVICE = 0, -1, -2, -3, -4, -5
HISA_F32, HISA_BF16 = 0, 1
FLAG_CHAINED = 0x1
DEV_BAD_OFFSETS, DEV_GATE, DEV_BAD_ID, DEV_NONFINITE, DEV_BAD_BLOCK, DEV_TIMEOUT = \
    0x1, 0x2, 0x4, 0x8, 0x10, 0x20
FLAT_NOALLOC_MAX_SCORES = 1 << 22
OP_COMPRESS = 6
OP_INDEX_SCORES, OP_BLOCK_MEANS, OP_BLOCK_FILTER, OP_SELECT_TOPK, OP_FLAT_TOPK, OP_SPARSE_ATTEND = \
    range(6)


class HisaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class IndexDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("L", ctypes.c_int32), ("H_i", ctypes.c_int32),
                ("D_i", ctypes.c_int32), ("r", ctypes.c_int32), ("index_topk", ctypes.c_int32),
                ("index_block", ctypes.c_int32), ("index_keep", ctypes.c_int32),
                ("Np_max", ctypes.c_int64), ("keys_rows", ctypes.c_int64),
                ("means_rows", ctypes.c_int64),
                ("q_dtype", ctypes.c_int32), ("k_dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("L", ctypes.c_int32), ("H", ctypes.c_int32),
                ("Dh", ctypes.c_int32), ("window", ctypes.c_int32), ("W_max", ctypes.c_int32),
                ("r", ctypes.c_int32), ("k", ctypes.c_int32), ("Np_max", ctypes.c_int64),
                ("kv_rows", ctypes.c_int64), ("scale", ctypes.c_float), ("q_dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("flags", ctypes.c_int32), ("out_dtype", ctypes.c_int32)]


class CompressDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("D_i", ctypes.c_int32), ("r", ctypes.c_int32),
                ("overlap", ctypes.c_int32), ("rope_dims", ctypes.c_int32),
                ("index_block", ctypes.c_int32), ("n_new_max", ctypes.c_int32),
                ("k_dtype", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("eps", ctypes.c_float),
                ("tok_rows", ctypes.c_int64), ("keys_rows", ctypes.c_int64),
                ("means_rows", ctypes.c_int64), ("flags", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_SIG = {
    "hisa_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32, _P]),
    "hisa_workspace_init": (ctypes.c_int32, [_P, ctypes.c_size_t, _P]),
    "hisa_device_status": (ctypes.c_int32, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "hisa_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "hisa_index_scores": (ctypes.c_int32, [_P] * 7 + [ctypes.c_int64, _P, ctypes.c_size_t, _P]),
    "hisa_block_means": (ctypes.c_int32, [_P] * 7 + [ctypes.c_size_t, _P]),
    "hisa_block_filter": (ctypes.c_int32, [_P] * 9 + [ctypes.c_int64, _P, ctypes.c_size_t, _P]),
    "hisa_select_topk": (ctypes.c_int32, [_P] * 10 + [ctypes.c_size_t, _P]),
    "hisa_flat_topk": (ctypes.c_int32, [_P] * 8 + [ctypes.c_size_t, _P]),
    "hisa_block_filter_append": (ctypes.c_int32, [_P] * 11 + [ctypes.c_int64, _P, ctypes.c_size_t, _P]),
    "hisa_flat_topk_noalloc": (ctypes.c_int32, [_P] * 9),
    "hisa_sparse_attend": (ctypes.c_int32, [_P] * 12 + [ctypes.c_size_t, _P]),
    "hisa_compress_append": (ctypes.c_int32, [_P] * 13 + [ctypes.c_size_t, _P]),
}


def lib() -> ctypes.CDLL:
    """The loaded libhisa.so (raises if it was never built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ "
                        f"as g; g.build()\"` (the CUDA library is required; there is no fallback)")
                L = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIG.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().hisa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != HISA_OK:
        raise HisaError(status, where)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return HISA_F32
    if t.dtype == torch.bfloat16:
        return HISA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------------------
# workspace / status
# ----------------------------------------------------------------------------
def workspace_bytes(op: int, desc) -> int:
    return int(lib().hisa_workspace_bytes(op, ctypes.byref(desc)))


def workspace_init(ws, stream=None) -> None:
    _check(lib().hisa_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "hisa_workspace_init")


def alloc_workspace(nbytes: int, device="cuda", stream=None):
    """A uint8 device buffer (torch's allocator aligns to >= 256 B) with a cleared status."""
    import torch
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    workspace_init(ws, stream)
    return ws


def device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns the device status bits (0 = clean)."""
    flags = ctypes.c_uint32(0)
    st = lib().hisa_device_status(_ptr(ws), _stream(stream), ctypes.byref(flags))
    if st not in (HISA_OK, HISA_EDEVICE):
        _check(st, "hisa_device_status")
    return int(flags.value)


# ----------------------------------------------------------------------------
# the step
# ----------------------------------------------------------------------------
def index_scores(desc, q, w, keys, key_off, t0, scores, ld_scores, ws, stream=None):
    _check(lib().hisa_index_scores(ctypes.byref(desc), _ptr(q), _ptr(w), _ptr(keys), _ptr(key_off),
                                   _ptr(t0), _ptr(scores), int(ld_scores), _ptr(ws),
                                   ws.numel(), _stream(stream)), "hisa_index_scores")


def block_means(desc, keys, key_off, means_off, first_block, means, ws, stream=None):
    _check(lib().hisa_block_means(ctypes.byref(desc), _ptr(keys), _ptr(key_off), _ptr(means_off),
                                  _ptr(first_block), _ptr(means), _ptr(ws), ws.numel(),
                                  _stream(stream)), "hisa_block_means")


def block_filter(desc, q, w, means, means_off, key_off, t0, top_blk, ws, cscores=None,
                 ld_cscores=0, stream=None):
    _check(lib().hisa_block_filter(ctypes.byref(desc), _ptr(q), _ptr(w), _ptr(means),
                                   _ptr(means_off), _ptr(key_off), _ptr(t0), _ptr(top_blk),
                                   _ptr(cscores), int(ld_cscores), _ptr(ws), ws.numel(),
                                   _stream(stream)), "hisa_block_filter")


def select_topk(desc, q, w, keys, key_off, t0, top_blk, I, ws, fscores=None, stream=None):
    _check(lib().hisa_select_topk(ctypes.byref(desc), _ptr(q), _ptr(w), _ptr(keys), _ptr(key_off),
                                  _ptr(t0), _ptr(top_blk), _ptr(I), _ptr(fscores), _ptr(ws),
                                  ws.numel(), _stream(stream)), "hisa_select_topk")


def flat_topk(desc, q, w, keys, key_off, t0, I, ws, stream=None):
    _check(lib().hisa_flat_topk(ctypes.byref(desc), _ptr(q), _ptr(w), _ptr(keys), _ptr(key_off),
                                _ptr(t0), _ptr(I), _ptr(ws), ws.numel(), _stream(stream)),
           "hisa_flat_topk")


def block_filter_append(desc, q, w, keys, key_off, means, means_off, first_block, t0, top_blk, ws,
                        cscores=None, ld_cscores=0, stream=None):
    _check(lib().hisa_block_filter_append(ctypes.byref(desc), _ptr(q), _ptr(w), _ptr(keys),
                                          _ptr(key_off), _ptr(means), _ptr(means_off),
                                          _ptr(first_block), _ptr(t0), _ptr(top_blk), _ptr(cscores),
                                          ld_cscores, _ptr(ws), ws.numel(), _stream(stream)),
           "hisa_block_filter_append")


def flat_topk_noalloc(desc, q, w, keys, key_off, t0, I, dev_status=None, stream=None):
    """hisa_flat_topk without a workspace: the library's own fixed device array holds the
    scores (B * L * Np_max <= FLAT_NOALLOC_MAX_SCORES). dev_status: optional int32 device
    tensor of one element that receives the call's HISA_DEV_* bits."""
    _check(lib().hisa_flat_topk_noalloc(ctypes.byref(desc), _ptr(q), _ptr(w), _ptr(keys),
                                        _ptr(key_off), _ptr(t0), _ptr(I), _ptr(dev_status),
                                        _stream(stream)), "hisa_flat_topk_noalloc")


def sparse_attend(desc, q, local_kv, local_len, local_pos0, pooled_kv, kv_off, I, sinks, t0, out,
                  ws, stream=None):
    _check(lib().hisa_sparse_attend(ctypes.byref(desc), _ptr(q), _ptr(local_kv), _ptr(local_len),
                                    _ptr(local_pos0), _ptr(pooled_kv), _ptr(kv_off), _ptr(I),
                                    _ptr(sinks), _ptr(t0), _ptr(out), _ptr(ws), ws.numel(),
                                    _stream(stream)), "hisa_sparse_attend")


def compress_append(desc, kv, gate, tok_off, p_first, n_new, ape, norm_w, keys, key_off, means,
                    means_off, ws, stream=None):
    _check(lib().hisa_compress_append(ctypes.byref(desc), _ptr(kv), _ptr(gate), _ptr(tok_off),
                                      _ptr(p_first), _ptr(n_new), _ptr(ape), _ptr(norm_w),
                                      _ptr(keys), _ptr(key_off), _ptr(means), _ptr(means_off),
                                      _ptr(ws), ws.numel(), _stream(stream)),
           "hisa_compress_append")


# ----------------------------------------------------------------------------
# page-locked host memory as a device-accessible output
# ----------------------------------------------------------------------------
_cudart = None


def _runtime():
    """The CUDA runtime library (the one torch loads, else the toolkit's)."""
    global _cudart
    if _cudart is None:
        import glob
        import torch
        base = os.path.dirname(os.path.dirname(torch.__file__))
        cands = glob.glob(os.path.join(base, "nvidia", "cu*", "lib", "libcudart.so*")) + \
            glob.glob("/usr/local/cuda/lib64/libcudart.so*")
        for c in cands:
            try:
                _cudart = ctypes.CDLL(c)
                break
            except OSError:
                continue
        if _cudart is None:
            raise RuntimeError("no CUDA runtime library found")
    return _cudart


def device_pointer_of_pinned(t) -> int:
    """The device address of a page-locked host tensor (torch's pin_memory), for a call that
    should read or write host memory directly (on GB300 over NVLink-C2C). Under unified
    addressing it is the host address itself; raises if the runtime does not map it."""
    dptr = ctypes.c_void_p()
    rc = _runtime().cudaHostGetDevicePointer(ctypes.byref(dptr), ctypes.c_void_p(t.data_ptr()),
                                             ctypes.c_uint(0))
    if rc != 0 or not dptr.value:
        raise RuntimeError(f"cudaHostGetDevicePointer failed ({rc})")
    return int(dptr.value)


class DevicePointer:
    """A raw device address passed where a tensor is expected (data_ptr() only)."""

    def __init__(self, addr: int, numel: int = 0):
        self.addr = int(addr)
        self._numel = numel

    def data_ptr(self) -> int:
        return self.addr

    def numel(self) -> int:
        return self._numel


# ----------------------------------------------------------------------------
# host arrays -> device tensors (uint16 arrays are bf16 bit patterns)
# ----------------------------------------------------------------------------
def to_device(a, device="cuda"):
    import torch
    if isinstance(a, torch.Tensor):
        return a.to(device).contiguous()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)
