"""Python binding of libqmv.so, the sm_103a group-quantized mat-vec (affine and mxfp4).

Argument marshalling only: every step of the computation runs in the CUDA
library. The names match the C ABI of ``include/qmv.h``. Device buffers may be
given as torch tensors (their ``data_ptr()`` is passed) or as integer device
addresses; streams as ``torch.cuda.Stream``, an integer handle, or ``None``
(torch's current stream on the current device).

Raises ``QmvError`` for any non-OK status, and ``RuntimeError`` when the
library has not been built -- there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libqmv.so")

QMV_TILE_M = 16
QMV_MAX_M = 256
F32_OUT = 0x1
FORCE_M1_PER_COLUMN = 0x2
PDL = 0x4
SB_INTERLEAVED = 0x8

STATUS = {
    0: "QMV_OK", 1: "QMV_ERR_NULL", 2: "QMV_ERR_BITS", 3: "QMV_ERR_GROUP", 4: "QMV_ERR_SHAPE",
    5: "QMV_ERR_M_RANGE", 6: "QMV_ERR_ALIGN", 7: "QMV_ERR_CUDA", 8: "QMV_ERR_WORKSPACE",
    9: "QMV_ERR_VALUE", 10: "QMV_ERR_FLAGS",
}

EXPORTED = ("qmv_packed_words", "qmv_pack", "qmv_unpack", "qmv_pack_sb", "qmv_split_count", "qmv_workspace_size",
            "qmv_run", "qmv_run_ex", "qmv_run_noalloc", "qmv_mxfp4_run", "qmv_workspace_init", "qmv_device_error", "qmv_last_cuda_error",
            "qmv_status_string")


class QmvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {qmv_status_string(code)}"
        if code == 7:
            msg += f" [{qmv_last_cuda_error()}]"
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libqmv.so (built by ``python -m group_quantized_mat_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built: run `python -m group_quantized_mat_gb300.build`")
        lib = ctypes.CDLL(p)
        P, I, I64, SZ, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint
        lib.qmv_packed_words.restype = SZ
        lib.qmv_packed_words.argtypes = [I64, I64, I]
        lib.qmv_pack.restype = I
        lib.qmv_pack.argtypes = [P, P, I64, I64, I]
        lib.qmv_unpack.restype = I
        lib.qmv_unpack.argtypes = [P, P, I64, I64, I]
        lib.qmv_pack_sb.restype = I
        lib.qmv_pack_sb.argtypes = [P, P, P, I64, I64]
        lib.qmv_split_count.restype = I
        lib.qmv_split_count.argtypes = [I, I, I, I]
        lib.qmv_workspace_size.restype = SZ
        lib.qmv_workspace_size.argtypes = [I, I, I, I, I]
        lib.qmv_run.restype = I
        lib.qmv_run.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
        lib.qmv_run_ex.restype = I
        lib.qmv_run_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, P, SZ, U, P]
        lib.qmv_run_noalloc.restype = I
        lib.qmv_run_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
        lib.qmv_mxfp4_run.restype = I
        lib.qmv_mxfp4_run.argtypes = [P, P, P, P, I, I, I, U, P]
        lib.qmv_workspace_init.restype = I
        lib.qmv_workspace_init.argtypes = [P, SZ, P]
        lib.qmv_device_error.restype = I
        lib.qmv_device_error.argtypes = [ctypes.POINTER(U)]
        lib.qmv_last_cuda_error.restype = ctypes.c_char_p
        lib.qmv_last_cuda_error.argtypes = []
        lib.qmv_status_string.restype = ctypes.c_char_p
        lib.qmv_status_string.argtypes = [I]
        if path is None:
            _lib = lib
        return lib


def _ptr(a) -> int | None:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return int(a.data_ptr())  # torch.Tensor


def _stream(s) -> int | None:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(code: int, where: str) -> None:
    if code != 0:
        raise QmvError(code, where)


def qmv_status_string(code: int) -> str:
    try:
        return load().qmv_status_string(int(code)).decode()
    except RuntimeError:
        return STATUS.get(int(code), f"status {code}")


# ----------------------------------------------------------------- codec --
def qmv_packed_words(N: int, K: int, bits: int) -> int:
    return int(load().qmv_packed_words(N, K, bits))


def qmv_pack(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack host q[N, K] (uint8, values < 2**bits) into uint32 [N, K*bits/32]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    if (K * bits) % 32:
        raise QmvError(4, "qmv_pack")
    out = np.empty((N, K * bits // 32), dtype=np.uint32)
    _check(load().qmv_pack(q.ctypes.data, out.ctypes.data, N, K, bits), "qmv_pack")
    return out


def qmv_unpack(w_q: np.ndarray, K: int, bits: int) -> np.ndarray:
    w_q = np.ascontiguousarray(w_q, dtype=np.uint32)
    N = w_q.shape[0]
    out = np.empty((N, K), dtype=np.uint8)
    _check(load().qmv_unpack(w_q.ctypes.data, out.ctypes.data, N, K, bits), "qmv_unpack")
    return out


def qmv_pack_sb(scales: np.ndarray, biases: np.ndarray) -> np.ndarray:
    """Interleave host bf16 bit patterns scales, biases [N, G] (uint16) into
    uint32 [N, G]: scale in the low half of each word, bias in the high half."""
    s = np.ascontiguousarray(scales, dtype=np.uint16)
    b = np.ascontiguousarray(biases, dtype=np.uint16)
    if s.shape != b.shape or s.ndim != 2:
        raise QmvError(4, "qmv_pack_sb")
    out = np.empty(s.shape, dtype=np.uint32)
    _check(load().qmv_pack_sb(s.ctypes.data, b.ctypes.data, out.ctypes.data, s.shape[0], s.shape[1]), "qmv_pack_sb")
    return out


# ------------------------------------------------------------------ plan --
def qmv_split_count(N: int, K: int, bits: int, group_size: int) -> int:
    return int(load().qmv_split_count(N, K, bits, group_size))


def qmv_workspace_size(M: int, N: int, K: int, bits: int, group_size: int) -> int:
    return int(load().qmv_workspace_size(M, N, K, bits, group_size))


# ------------------------------------------------------------------- run --
def qmv_run(w_q, scales, biases, x, y, M: int, N: int, K: int, bits: int, group_size: int, stream=None) -> None:
    """y[M, N] (bf16) = W x, enqueued on ``stream``; see include/qmv.h."""
    code = load().qmv_run(_ptr(w_q), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K, bits, group_size,
                          _stream(stream))
    _check(code, "qmv_run")


def qmv_run_ex(w_q, scales, biases, x, y, M: int, N: int, K: int, bits: int, group_size: int,
               workspace=None, workspace_bytes: int = 0, flags: int = 0, stream=None) -> None:
    code = load().qmv_run_ex(_ptr(w_q), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K, bits, group_size,
                             _ptr(workspace), int(workspace_bytes), int(flags), _stream(stream))
    _check(code, "qmv_run_ex")


NOALLOC_SCRATCH_BYTES = 8 << 20


def qmv_run_noalloc(w_q, scales, biases, x, y, M: int, N: int, K: int, bits: int, group_size: int,
                    stream=None) -> None:
    """qmv_run without any device allocation (fixed scratch array in the library)."""
    code = load().qmv_run_noalloc(_ptr(w_q), _ptr(scales), _ptr(biases), _ptr(x), _ptr(y), M, N, K, bits,
                                  group_size, _stream(stream))
    _check(code, "qmv_run_noalloc")


def qmv_mxfp4_run(w_q, scales, x, y, M: int, N: int, K: int, flags: int = 0, stream=None) -> None:
    """y[M, N] = W x in the mxfp4 mode (E2M1 codes packed by ``qmv_pack(q, 4)``,
    uint8 E8M0 scales [N, K/32]); see include/qmv.h."""
    code = load().qmv_mxfp4_run(_ptr(w_q), _ptr(scales), _ptr(x), _ptr(y), M, N, K, int(flags), _stream(stream))
    _check(code, "qmv_mxfp4_run")


def qmv_workspace_init(workspace, nbytes: int, stream=None) -> None:
    _check(load().qmv_workspace_init(_ptr(workspace), int(nbytes), _stream(stream)), "qmv_workspace_init")


def qmv_last_cuda_error() -> str:
    return load().qmv_last_cuda_error().decode()


def qmv_device_error() -> int:
    w = ctypes.c_uint(0)
    _check(load().qmv_device_error(ctypes.byref(w)), "qmv_device_error")
    return int(w.value)
