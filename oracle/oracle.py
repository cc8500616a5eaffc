"""ctypes front end of the CPU oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's CPU-baseline leg may use
this module; the product path (the CUDA library and its binding) never does. Every function cites the
passage it follows in ``oracle.cpp``'s header: block-scaled FP8 contraction with per-128-K-block
scaling and higher-precision accumulation, as the DeepGEMM pages describe it.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]


def _digest() -> str:
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(_FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``_build/liboracle.so`` (plain g++, portable flags); rebuilt whenever the
    source digest differs from the one recorded beside the library."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stamp = _LIB + ".sha256"
    digest = _digest()
    fresh = os.path.exists(_LIB) and os.path.exists(stamp) and open(stamp).read().strip() == digest
    if force or not fresh:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["g++", *_FLAGS, _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB)
        with open(stamp + f".tmp{os.getpid()}", "w") as f:
            f.write(digest + "\n")
        os.replace(stamp + f".tmp{os.getpid()}", stamp)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            L.oracle_e4m3_value.restype = D
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.oracle_bf16_bits.restype = ctypes.c_uint16
            L.oracle_bf16_bits.argtypes = [D]
            L.oracle_hardware_threads.restype = I32
            L.oracle_gemm_fp8_nt.restype = I32
            L.oracle_gemm_fp8_nt.argtypes = [P, P, P, P, P, I64, I64, I64, P, I64, I32]
            L.oracle_m_grouped_contiguous.restype = I32
            L.oracle_m_grouped_contiguous.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, P, I64, I32]
            L.oracle_m_grouped_masked.restype = I32
            L.oracle_m_grouped_masked.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, P, I64, I32]
            L.oracle_k_grouped_wgrad.restype = I32
            L.oracle_k_grouped_wgrad.argtypes = [P, P, P, P, P, P, I64, I64, I64, P, I64, I32]
            _lib = L
    return _lib


def _np(x, dtype):
    """Contiguous numpy view of a CPU tensor or array with the given dtype."""
    if hasattr(x, "numpy"):
        x = x.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != dtype:
        a = a.astype(dtype)
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, len(r)


def e4m3_value(code: int) -> float:
    """Value of one e4m3 code (OCP FP8 E4M3, 'fn' variant: no infinities, S.1111.111 = NaN)."""
    return lib().oracle_e4m3_value(code)


def bf16_bits(x: float) -> int:
    """BF16 bit pattern of ``x`` rounded once, to nearest even, from FP64."""
    return lib().oracle_bf16_bits(float(x))


def hardware_threads() -> int:
    return lib().oracle_hardware_threads()


def gemm_fp8_nt(A, sfa, B, sfb, rows=None, threads: int = 0) -> np.ndarray:
    """BF16 bits (uint16 [len(rows) or M, N]) of D = A . B^T with 1x128 / 128x128 block scales."""
    A = _np(A, np.uint8); B = _np(B, np.uint8)
    sfa = _np(sfa, np.float32); sfb = _np(sfb, np.float32)
    M, K = A.shape
    N = B.shape[0]
    r, nr = _rows(rows)
    D = np.zeros((nr if r is not None else M, N), dtype=np.uint16)
    rc = lib().oracle_gemm_fp8_nt(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(D), M, N, K, _ptr(r), nr, threads)
    assert rc == 0
    return D


def m_grouped_contiguous(A, sfa, B, sfb, m_indices, D_init=None, rows=None, threads: int = 0) -> np.ndarray:
    """BF16 bits of the contiguous-layout grouped GEMM; rows with group -1 keep ``D_init``."""
    A = _np(A, np.uint8); B = _np(B, np.uint8)
    sfa = _np(sfa, np.float32); sfb = _np(sfb, np.float32)
    mi = _np(m_indices, np.int32)
    Mt, K = A.shape
    G, N, _ = B.shape
    r, nr = _rows(rows)
    n_out = nr if r is not None else Mt
    D = np.zeros((n_out, N), dtype=np.uint16) if D_init is None else _np(D_init, np.uint16).copy()
    rc = lib().oracle_m_grouped_contiguous(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(mi), _ptr(D),
                                          Mt, N, K, G, _ptr(r), nr, threads)
    assert rc == 0
    return D


def m_grouped_masked(A, sfa, B, sfb, masked_m, D_init=None, rows=None, threads: int = 0) -> np.ndarray:
    """BF16 bits of the masked-layout grouped GEMM, [G*max_m (or len(rows)), N]; rows past
    ``masked_m[g]`` keep ``D_init``."""
    A = _np(A, np.uint8); B = _np(B, np.uint8)
    sfa = _np(sfa, np.float32); sfb = _np(sfb, np.float32)
    mm = _np(masked_m, np.int32)
    G, max_m, K = A.shape
    N = B.shape[1]
    r, nr = _rows(rows)
    n_out = nr if r is not None else G * max_m
    D = np.zeros((n_out, N), dtype=np.uint16) if D_init is None else _np(D_init, np.uint16).reshape(n_out, N).copy()
    rc = lib().oracle_m_grouped_masked(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(mm), _ptr(D),
                                      G, max_m, N, K, _ptr(r), nr, threads)
    assert rc == 0
    return D


def k_grouped_wgrad(A, sfa, B, sfb, ks, D_in, rows=None, threads: int = 0) -> np.ndarray:
    """FP32 [G, len(rows) or M, N]: ``D_in + X_g^T . dY_g`` per expert g (1x128 scales on both)."""
    A = _np(A, np.uint8); B = _np(B, np.uint8)
    sfa = _np(sfa, np.float32); sfb = _np(sfb, np.float32)
    ks_a = np.ascontiguousarray(np.asarray(ks, dtype=np.int64))
    M = A.shape[0]
    N = B.shape[0]
    G = len(ks_a)
    r, nr = _rows(rows)
    D_in = _np(D_in, np.float32)
    D = (D_in[:, r, :] if r is not None else D_in).copy()
    rc = lib().oracle_k_grouped_wgrad(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(ks_a), _ptr(D),
                                     G, M, N, _ptr(r), nr, threads)
    assert rc == 0
    return D


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
