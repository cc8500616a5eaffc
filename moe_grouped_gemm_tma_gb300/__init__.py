"""Block-scaled FP8 GEMM and MoE grouped GEMM for GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/dg.h`` (``libdg.so``, built in-tree by
``build.py``). The functions carry the C names and only marshal arguments: torch tensors provide
device memory and the current CUDA stream; every step of the computation runs in the library's CUDA
kernels. There is no fallback: when the library or a supported GPU is missing, calls raise.

Operation (DeepGEMM pages, "DeepSeek DeepGEMM" usage example and feature list):
``D[m,n] = sum_kb sfa[m,kb] * sfb[n//128,kb] * sum_{k in block kb} A[m,k] B[n,k]`` with e4m3 A/B,
FP32 1x128 (A) and 128x128 (B) block scales, BF16 output; plus the m-grouped contiguous and masked
layouts and the k-grouped FP32 weight gradient.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

__all__ = [
    "DGError", "load", "dg_gemm_fp8_nt", "dg_gemm_fp8", "dg_gemm_fp8_nt_ue8m0", "dg_gemm_fp8_nt_ue8m0_packed",
    "dg_m_grouped_contiguous", "dg_m_grouped_masked",
    "dg_k_grouped_wgrad", "dg_wgrad_fp8_nt", "dg_device_status", "dg_status_string", "scale_shapes", "library_path",
    "TUNE_KNOBS", "dg_tuning_set", "dg_tuning_get", "dg_tuning_reset", "tuning", "dg_testing_arm_wait_timeout",
]

_lock = threading.Lock()
_lib = None

DG_OK = 0
STATUS_NAMES = {0: "DG_OK", 1: "DG_INVALID_ARG", 2: "DG_UNSUPPORTED_SHAPE", 3: "DG_MISALIGNED",
                4: "DG_CUDA_ERROR", 5: "DG_NO_DEVICE_SUPPORT", 6: "DG_DEVICE_TIMEOUT", 7: "DG_SCALE_NOT_UE8M0"}


class DGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


def library_path() -> str:
    from . import build as _build
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load ``libdg.so`` (building it with nvcc first when absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            from . import build as _build
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libdg.so not found at {path}; run moe_grouped_gemm_tma_gb300/build.py")
            L = ctypes.CDLL(path)
            P, I = ctypes.c_void_p, ctypes.c_int
            L.dg_gemm_fp8_nt.argtypes = [P, P, P, P, P, I, I, I, P]
            L.dg_gemm_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
            L.dg_gemm_fp8_nt_ue8m0.argtypes = [P, P, P, P, P, I, I, I, P]
            L.dg_gemm_fp8_nt_ue8m0_packed.argtypes = [P, P, P, P, P, I, I, I, P]
            L.dg_m_grouped_contiguous.argtypes = [P, P, P, P, P, P, I, I, I, I, P]
            L.dg_m_grouped_masked.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P]
            L.dg_k_grouped_wgrad.argtypes = [P, P, P, P, P, P, I, I, I, P]
            L.dg_wgrad_fp8_nt.argtypes = [P, P, P, P, P, I, I, I, I, P]
            L.dg_device_status.argtypes = [P]
            L.dg_tuning_set.argtypes = [I, I]
            L.dg_tuning_set.restype = I
            L.dg_tuning_get.argtypes = [I]
            L.dg_tuning_get.restype = I
            L.dg_tuning_reset.argtypes = []
            L.dg_tuning_reset.restype = None
            L.dg_testing_arm_wait_timeout.argtypes = [ctypes.c_uint64]
            L.dg_testing_arm_wait_timeout.restype = I
            L.dg_status_string.argtypes = [I]
            L.dg_status_string.restype = ctypes.c_char_p
            for f in ("dg_gemm_fp8_nt", "dg_gemm_fp8", "dg_gemm_fp8_nt_ue8m0", "dg_gemm_fp8_nt_ue8m0_packed",
                      "dg_m_grouped_contiguous", "dg_m_grouped_masked",
                      "dg_k_grouped_wgrad", "dg_wgrad_fp8_nt", "dg_device_status"):
                getattr(L, f).restype = I
            _lib = L
    return _lib


def _torch():
    import torch
    return torch


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _codes(t, name):
    torch = _torch()
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must hold e4m3 codes (torch.float8_e4m3fn or uint8), got {t.dtype}")
    return _dense(t, name)


def _dense(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _f32(t, name):
    torch = _torch()
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    return _dense(t, name)


def _check(status: int, where: str):
    if status != DG_OK:
        raise DGError(status, where)


def scale_shapes(M: int, N: int, K: int):
    """Shapes of (sfa, sfb) for a normal GEMM: ([M, K/128], [ceil(N/128), K/128])."""
    return (M, K // 128), ((N + 127) // 128, K // 128)


def dg_gemm_fp8_nt(A, sfa, B, sfb, D, stream=None):
    """D[M,N] (bf16) = A[M,K] . B[N,K]^T with sfa [M,K/128] and sfb [ceil(N/128),K/128] scales."""
    torch = _torch()
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb = _f32(sfa, "sfa"), _f32(sfb, "sfb")
    D = _dense(D, "D")
    if D.dtype != torch.bfloat16:
        raise TypeError("D must be bfloat16")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)} B {tuple(B.shape)} D {tuple(D.shape)}")
    if (tuple(sfa.shape), tuple(sfb.shape)) != scale_shapes(M, N, K):
        raise ValueError(f"scale shapes {tuple(sfa.shape)}, {tuple(sfb.shape)} != {scale_shapes(M, N, K)}")
    st = load().dg_gemm_fp8_nt(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(D), M, N, K, _stream(stream))
    _check(st, "dg_gemm_fp8_nt")
    return D


def dg_gemm_fp8(A, sfa, B, sfb, D, a_mn_major=False, b_mn_major=False, stream=None):
    """The normal GEMM for any operand layout: A stored [M,K] or (a_mn_major) [K,M]; B stored [N,K] or
    (b_mn_major) [K,N]; same scales and output as dg_gemm_fp8_nt."""
    torch = _torch()
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb = _f32(sfa, "sfa"), _f32(sfb, "sfb")
    D = _dense(D, "D")
    if D.dtype != torch.bfloat16:
        raise TypeError("D must be bfloat16")
    K, M = A.shape if a_mn_major else A.shape[::-1]
    KB, N = B.shape if b_mn_major else B.shape[::-1]
    if KB != K or tuple(D.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)} B {tuple(B.shape)} D {tuple(D.shape)}")
    if (tuple(sfa.shape), tuple(sfb.shape)) != scale_shapes(M, N, K):
        raise ValueError(f"scale shapes {tuple(sfa.shape)}, {tuple(sfb.shape)} != {scale_shapes(M, N, K)}")
    st = load().dg_gemm_fp8(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(D), M, N, K,
                            1 if a_mn_major else 0, 1 if b_mn_major else 0, _stream(stream))
    _check(st, "dg_gemm_fp8")
    return D


def dg_gemm_fp8_nt_ue8m0(A, sfa, B, sfb, D, stream=None):
    """dg_gemm_fp8_nt for power-of-two scales on the block-scaled (UE8M0) tensor-core path."""
    torch = _torch()
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb = _f32(sfa, "sfa"), _f32(sfb, "sfb")
    D = _dense(D, "D")
    if D.dtype != torch.bfloat16:
        raise TypeError("D must be bfloat16")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)} B {tuple(B.shape)} D {tuple(D.shape)}")
    if (tuple(sfa.shape), tuple(sfb.shape)) != scale_shapes(M, N, K):
        raise ValueError(f"scale shapes {tuple(sfa.shape)}, {tuple(sfb.shape)} != {scale_shapes(M, N, K)}")
    st = load().dg_gemm_fp8_nt_ue8m0(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(D), M, N, K, _stream(stream))
    _check(st, "dg_gemm_fp8_nt_ue8m0")
    return D


def dg_gemm_fp8_nt_ue8m0_packed(A, sfa, B, sfb, D, stream=None):
    """The block-scaled GEMM with packed UE8M0 scales: sfa int32 [M, ceil(K/512)], sfb int32
    [ceil(N/128), ceil(K/512)], byte j of word w = biased exponent of K block 4w + j."""
    torch = _torch()
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb, D = _dense(sfa, "sfa"), _dense(sfb, "sfb"), _dense(D, "D")
    if sfa.dtype != torch.int32 or sfb.dtype != torch.int32:
        raise TypeError("packed scales must be int32")
    if D.dtype != torch.bfloat16:
        raise TypeError("D must be bfloat16")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)} B {tuple(B.shape)} D {tuple(D.shape)}")
    words = (K // 128 + 3) // 4
    if tuple(sfa.shape) != (M, words) or tuple(sfb.shape) != ((N + 127) // 128, words):
        raise ValueError(f"packed scale shapes {tuple(sfa.shape)}, {tuple(sfb.shape)} != {(M, words)}, {((N + 127) // 128, words)}")
    st = load().dg_gemm_fp8_nt_ue8m0_packed(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(D), M, N, K, _stream(stream))
    _check(st, "dg_gemm_fp8_nt_ue8m0_packed")
    return D


def dg_m_grouped_contiguous(A, sfa, B, sfb, m_indices, D, stream=None):
    """Contiguous-layout grouped GEMM: D[r] = A[r] . B[m_indices[r]]^T (bf16); A [Mt,K], B [G,N,K]."""
    torch = _torch()
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb = _f32(sfa, "sfa"), _f32(sfb, "sfb")
    m_indices, D = _dense(m_indices, "m_indices"), _dense(D, "D")
    if m_indices.dtype != torch.int32 or D.dtype != torch.bfloat16:
        raise TypeError("m_indices must be int32 and D bfloat16")
    Mt, K = A.shape
    G, N, K2 = B.shape
    if K2 != K or tuple(D.shape) != (Mt, N) or m_indices.numel() != Mt:
        raise ValueError("shape mismatch")
    if tuple(sfa.shape) != (Mt, K // 128) or tuple(sfb.shape) != (G, (N + 127) // 128, K // 128):
        raise ValueError("scale shape mismatch")
    st = load().dg_m_grouped_contiguous(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(m_indices), _ptr(D),
                                        Mt, N, K, G, _stream(stream))
    _check(st, "dg_m_grouped_contiguous")
    return D


def dg_m_grouped_masked(A, sfa, B, sfb, masked_m, D, expected_m: int = 0, stream=None):
    """Masked-layout grouped GEMM: D[g,r] = A[g,r] . B[g]^T for r < masked_m[g]; other rows untouched."""
    torch = _torch()
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb = _f32(sfa, "sfa"), _f32(sfb, "sfb")
    masked_m, D = _dense(masked_m, "masked_m"), _dense(D, "D")
    if masked_m.dtype != torch.int32 or D.dtype != torch.bfloat16:
        raise TypeError("masked_m must be int32 and D bfloat16")
    G, max_m, K = A.shape
    G2, N, K2 = B.shape
    if G2 != G or K2 != K or tuple(D.shape) != (G, max_m, N) or masked_m.numel() != G:
        raise ValueError("shape mismatch")
    if tuple(sfa.shape) != (G, max_m, K // 128) or tuple(sfb.shape) != (G, (N + 127) // 128, K // 128):
        raise ValueError("scale shape mismatch")
    st = load().dg_m_grouped_masked(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(masked_m), _ptr(D),
                                    G, max_m, N, K, int(expected_m), _stream(stream))
    _check(st, "dg_m_grouped_masked")
    return D


def dg_k_grouped_wgrad(A, sfa, B, sfb, ks, D, stream=None):
    """k-grouped FP32 weight gradient: D[g] += A[:, win_g] . B[:, win_g]^T, windows of widths ``ks``."""
    torch = _torch()
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb = _f32(sfa, "sfa"), _f32(sfb, "sfb")
    D = _f32(D, "D")
    ks_list = [int(k) for k in (ks.tolist() if hasattr(ks, "tolist") else ks)]
    G = len(ks_list)
    M, sumK = A.shape
    N = B.shape[0]
    if B.shape[1] != sumK or sum(ks_list) != sumK or tuple(D.shape) != (G, M, N):
        raise ValueError("shape mismatch")
    if tuple(sfa.shape) != (M, sumK // 128) or tuple(sfb.shape) != (N, sumK // 128):
        raise ValueError("scale shape mismatch")
    ks_arr = (ctypes.c_int32 * max(G, 1))(*ks_list)
    st = load().dg_k_grouped_wgrad(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), ks_arr, _ptr(D), G, M, N,
                                   _stream(stream))
    _check(st, "dg_k_grouped_wgrad")
    return D


def dg_wgrad_fp8_nt(A, sfa, B, sfb, D, accumulate=True, stream=None):
    """Dense FP32 weight gradient: D += A . B^T (accumulate) or D = A . B^T, 1x128 scales on both."""
    A, B = _codes(A, "A"), _codes(B, "B")
    sfa, sfb = _f32(sfa, "sfa"), _f32(sfb, "sfb")
    D = _f32(D, "D")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError("shape mismatch")
    if tuple(sfa.shape) != (M, K // 128) or tuple(sfb.shape) != (N, K // 128):
        raise ValueError("scale shape mismatch")
    st = load().dg_wgrad_fp8_nt(_ptr(A), _ptr(sfa), _ptr(B), _ptr(sfb), _ptr(D), M, N, K,
                                1 if accumulate else 0, _stream(stream))
    _check(st, "dg_wgrad_fp8_nt")
    return D


def dg_device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) any device-side timeout status."""
    return load().dg_device_status(_stream(stream))


def dg_status_string(status: int) -> str:
    return load().dg_status_string(int(status)).decode()


# Tuning knobs (include/dg_tuning.h): overrides of the automatic tile-shape choice, for sweeps and for
# tests that must reach one kernel specialisation. -1 (or None) is the automatic choice.
TUNE_KNOBS = {"bn": 0, "pair": 1, "split": 2, "swap": 3, "group_m": 4, "pdl": 5}


def dg_tuning_set(knob, value) -> None:
    k = TUNE_KNOBS[knob] if isinstance(knob, str) else int(knob)
    _check(load().dg_tuning_set(k, -1 if value is None else int(value)), "dg_tuning_set")


def dg_tuning_get(knob) -> int:
    return load().dg_tuning_get(TUNE_KNOBS[knob] if isinstance(knob, str) else int(knob))


def dg_tuning_reset() -> None:
    load().dg_tuning_reset()


@contextlib.contextmanager
def tuning(**knobs):
    """Set tuning knobs (bn=, pair=, split=, swap=, group_m=, pdl=) for the duration of a ``with`` block;
    every knob returns to the automatic choice afterwards."""
    try:
        for k, v in knobs.items():
            dg_tuning_set(k, v)
        yield
    finally:
        dg_tuning_reset()


def dg_testing_arm_wait_timeout(wait_limit_ns: int) -> None:
    """Test hook: the next launch of the main kernel bounds its waits by ``wait_limit_ns`` and leaves its
    first pipeline stage unfilled, so that a wait runs out and the kernel reports DG_DEVICE_TIMEOUT."""
    _check(load().dg_testing_arm_wait_timeout(int(wait_limit_ns)), "dg_testing_arm_wait_timeout")
