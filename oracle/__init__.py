"""CPU oracle for the group-quantized mat-vec (qmv; affine and mxfp4) -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. The product path never does.

The arithmetic lives in ``qmv_oracle.c`` (plain C, built here with gcc,
``-ffp-contract=off``); this module compiles it and marshals numpy arrays.
Nothing here is shared with the CUDA library.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(mutant: int = 0) -> str:
    name = "libqmv_oracle.so" if mutant == 0 else f"libqmv_oracle_mut{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally with planted mistake ``mutant``)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           f"-DORACLE_MUTANT={int(mutant)}", "-o", tmp, _SRC, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant in _libs:
            return _libs[mutant]
        lib = ctypes.CDLL(build(mutant))
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16_array.restype = None
        lib.oracle_f32_to_bf16_array.argtypes = [_P, _P, _I64]
        lib.oracle_field.restype = ctypes.c_uint32
        lib.oracle_field.argtypes = [_P, _I64, _I]
        lib.oracle_pack.restype = None
        lib.oracle_pack.argtypes = [_P, _P, _I64, _I64, _I]
        lib.oracle_byte_fields.restype = None
        lib.oracle_byte_fields.argtypes = [ctypes.c_uint8, _I, _P]
        lib.oracle_byte_fields_floatfloor.restype = None
        lib.oracle_byte_fields_floatfloor.argtypes = [ctypes.c_uint8, _I, _P]
        for fn in ("oracle_qmv_f64_dequant", "oracle_qmv_f64_factored", "oracle_qmv_abs_terms"):
            f = getattr(lib, fn)
            f.restype = None
            f.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I]
        lib.oracle_qmv_f32_factored.restype = _I
        lib.oracle_qmv_f32_factored.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I]
        lib.oracle_e2m1_to_f64.restype = ctypes.c_double
        lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_to_f64.restype = ctypes.c_double
        lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        for fn in ("oracle_mxfp4_qmv_f64", "oracle_mxfp4_abs_terms"):
            f = getattr(lib, fn)
            f.restype = None
            f.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64]
        lib.oracle_mutant.restype = _I
        _libs[mutant] = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """numpy-facing wrapper; ``mutant`` selects a build with a planted mistake."""

    def __init__(self, mutant: int = 0):
        self.lib = _load(mutant)
        self.mutant = mutant

    # -- bf16 --------------------------------------------------------------
    def bf16_to_f64(self, h: np.ndarray) -> np.ndarray:
        return np.array([self.lib.oracle_bf16_to_f64(int(v)) for v in np.ravel(h)],
                        dtype=np.float64).reshape(np.shape(h))

    def f32_to_bf16(self, f: np.ndarray) -> np.ndarray:
        f = np.ascontiguousarray(f, dtype=np.float32)
        out = np.empty(f.shape, dtype=np.uint16)
        self.lib.oracle_f32_to_bf16_array(_ptr(f), _ptr(out), f.size)
        return out

    # -- fields ------------------------------------------------------------
    def pack(self, q: np.ndarray, bits: int) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.uint8)
        N, K = q.shape
        w = np.empty((N, K * bits // 32), dtype=np.uint32)
        self.lib.oracle_pack(_ptr(q), _ptr(w), N, K, bits)
        return w

    def field(self, row_words: np.ndarray, i: int, bits: int) -> int:
        row_words = np.ascontiguousarray(row_words, dtype=np.uint32)
        return int(self.lib.oracle_field(_ptr(row_words), int(i), int(bits)))

    def byte_fields(self, byte: int, bits: int) -> list[int]:
        out = np.zeros(8, dtype=np.int32)
        self.lib.oracle_byte_fields(ctypes.c_uint8(byte), bits, _ptr(out))
        return out[: 8 // bits].tolist()

    def byte_fields_floatfloor(self, byte: int, bits: int) -> list[int]:
        out = np.zeros(8, dtype=np.int32)
        self.lib.oracle_byte_fields_floatfloor(ctypes.c_uint8(byte), bits, _ptr(out))
        return out[: 8 // bits].tolist()

    # -- qmv ---------------------------------------------------------------
    @staticmethod
    def _args(wq, s, b, x, bits, gs):
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        s = np.ascontiguousarray(s, dtype=np.uint16)
        b = np.ascontiguousarray(b, dtype=np.uint16)
        x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.uint16)
        N = wq.shape[0]
        M, K = x.shape
        assert wq.shape[1] == K * bits // 32 and s.shape == (N, K // gs) and b.shape == s.shape
        return wq, s, b, x, M, N, K

    def _f64(self, fn, wq, s, b, x, bits, gs):
        wq, s, b, x, M, N, K = self._args(wq, s, b, x, bits, gs)
        y = np.empty((M, N), dtype=np.float64)
        getattr(self.lib, fn)(_ptr(wq), _ptr(s), _ptr(b), _ptr(x), _ptr(y), M, N, K, bits, gs)
        return y

    def qmv_f64_dequant(self, wq, s, b, x, bits, gs):
        return self._f64("oracle_qmv_f64_dequant", wq, s, b, x, bits, gs)

    def qmv_f64_factored(self, wq, s, b, x, bits, gs):
        return self._f64("oracle_qmv_f64_factored", wq, s, b, x, bits, gs)

    def abs_terms(self, wq, s, b, x, bits, gs):
        return self._f64("oracle_qmv_abs_terms", wq, s, b, x, bits, gs)

    def qmv_f32_factored(self, wq, s, b, x, bits, gs, nthreads: int = 1, want_f32: bool = False):
        """Returns (y_bf16_bits[M,N], y_f32[M,N] or None, threads_used)."""
        wq, s, b, x, M, N, K = self._args(wq, s, b, x, bits, gs)
        y = np.empty((M, N), dtype=np.uint16)
        y32 = np.empty((M, N), dtype=np.float32) if want_f32 else None
        used = self.lib.oracle_qmv_f32_factored(_ptr(wq), _ptr(s), _ptr(b), _ptr(x), _ptr(y),
                                                _ptr(y32), M, N, K, bits, gs, int(nthreads))
        return y, y32, used

    # -- mxfp4 (E2M1 elements, one E8M0 scale per 32 along K) --------------
    def e2m1_to_f64(self, codes) -> np.ndarray:
        return np.array([self.lib.oracle_e2m1_to_f64(int(c)) for c in np.ravel(codes)],
                        dtype=np.float64).reshape(np.shape(codes))

    def e8m0_to_f64(self, codes) -> np.ndarray:
        return np.array([self.lib.oracle_e8m0_to_f64(int(c)) for c in np.ravel(codes)],
                        dtype=np.float64).reshape(np.shape(codes))

    def _mx(self, fn, wq, scales, x):
        wq = np.ascontiguousarray(wq, dtype=np.uint32)
        scales = np.ascontiguousarray(scales, dtype=np.uint8)
        x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.uint16)
        N = wq.shape[0]
        M, K = x.shape
        assert K % 32 == 0 and wq.shape[1] == K // 8 and scales.shape == (N, K // 32)
        y = np.empty((M, N), dtype=np.float64)
        getattr(self.lib, fn)(_ptr(wq), _ptr(scales), _ptr(x), _ptr(y), M, N, K)
        return y

    def mxfp4_qmv_f64(self, wq, scales, x):
        """y[M, N] = sum_i scale * e2m1(q) * x, fp64 (wq from ``pack(codes, 4)``)."""
        return self._mx("oracle_mxfp4_qmv_f64", wq, scales, x)

    def mxfp4_abs_terms(self, wq, scales, x):
        return self._mx("oracle_mxfp4_abs_terms", wq, scales, x)


def tolerance_ok(y_test: np.ndarray, y_ref: np.ndarray, abs_terms: np.ndarray,
                 rel: float = 8e-3, atol: float = 1e-5):
    """Acceptance bound |y_test - y_ref| <= rel * sum_i|w_i x_i| + atol, per element.

    Returns (all_ok, worst_ratio) where worst_ratio = max |err| / bound.
    """
    err = np.abs(y_test.astype(np.float64) - y_ref)
    bound = rel * abs_terms + atol
    ratio = err / bound
    return bool(np.all(ratio <= 1.0)), float(ratio.max()) if ratio.size else 0.0
