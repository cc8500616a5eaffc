"""Seeded synthetic inputs for the block-scaled FP8 GEMM and its MoE grouped variants.

This module is the only code shared by the CUDA path's tests/bench and the CPU oracle. It draws
random numbers and casts them to the storage formats the GEMM consumes; it holds none of the GEMM's
own arithmetic (no decode, no contraction, no scaling of products, no output rounding).

Random numbers come from a counter-based generator defined here in full, so every machine produces
the same bytes for the same seed:

* ``splitmix64``: the i-th 64-bit word of stream ``seed`` is ``mix(seed + (i+1)*0x9E3779B97F4A7C15)``
  with Steele/Lea/Flood's splitmix64 finaliser (shift 30/27/31, multipliers 0xBF58476D1CE4E5B9 and
  0x94D049BB133111EB), computed modulo 2**64.
* uniforms: ``u = ((w >> 11) + 1) * 2**-53`` in (0, 1].
* normals: Box-Muller on consecutive word pairs (2j, 2j+1): ``sqrt(-2 ln u1) * (cos, sin)(2 pi u2)``.

Block quantisation follows the workload description of the DeepGEMM pages (fine-grained scaling: one
FP32 scale per 1x128 row block of the LHS and per 128x128 block of the RHS, "DeepSeek DeepGEMM" usage
example): ``scale = max(amax, 1e-4) / 448`` and ``q = e4m3(clamp(x / scale, -448, 448))``. The e4m3
cast itself is torch's ``float8_e4m3fn`` conversion (round to nearest even), a library routine.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21
_THREADS = max(1, min(16, os.cpu_count() or 1))

E4M3_MAX = 448.0
SCALE_FLOOR = 1e-4
BLOCK = 128

# Sub-stream identifiers, added to the seed as stream * 2**40 so tensors never share words.
STREAM_A, STREAM_B, STREAM_SIZES, STREAM_DIN = 1, 2, 3, 4


def _stream_seed(seed: int, stream: int) -> np.uint64:
    return np.uint64((int(seed) + (int(stream) << 40)) & 0xFFFFFFFFFFFFFFFF)


def splitmix64_words(seed: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of the splitmix64 stream ``seed`` (uint64)."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniforms(seed: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` float64 uniforms in (0, 1] from words ``start ..`` of stream ``seed``."""
    w = splitmix64_words(seed, start, count)
    return ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normals(seed: int, count: int) -> np.ndarray:
    """``count`` standard normals (float32), Box-Muller over word pairs, generated in chunks (chunks
    run on a thread pool; numpy releases the GIL, and each chunk's words depend only on its index)."""
    out = np.empty(count, dtype=np.float32)
    pairs = (count + 1) // 2

    def chunk(p0):
        npair = min(_CHUNK, pairs - p0)
        u = uniforms(seed, 2 * npair, start=2 * p0).reshape(npair, 2)
        r = np.sqrt(-2.0 * np.log(u[:, 0]))
        th = (2.0 * math.pi) * u[:, 1]
        z = np.stack([r * np.cos(th), r * np.sin(th)], axis=1).reshape(-1)
        lo = 2 * p0
        n = min(2 * npair, count - lo)
        out[lo:lo + n] = z[:n]

    starts = list(range(0, pairs, _CHUNK))
    if len(starts) <= 1:
        for p0 in starts:
            chunk(p0)
    else:
        with ThreadPoolExecutor(max_workers=min(len(starts), _THREADS)) as ex:
            list(ex.map(chunk, starts))
    return out


def _t_shr(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns (torch's >> is arithmetic)."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def _u64_as_i64(v: int) -> int:
    v &= 0xFFFFFFFFFFFFFFFF
    return v - (1 << 64) if v >= (1 << 63) else v


def normals_torch(seed: int, count: int, device) -> torch.Tensor:
    """The same ``count`` normals as :func:`normals`, computed with torch ops on ``device`` (int64
    arithmetic wraps modulo 2**64 exactly like the uint64 definition; shifts are made logical)."""
    out = torch.empty(count, dtype=torch.float32, device=device)
    pairs = (count + 1) // 2
    g, m1, m2 = _u64_as_i64(0x9E3779B97F4A7C15), _u64_as_i64(0xBF58476D1CE4E5B9), _u64_as_i64(0x94D049BB133111EB)
    sd = _u64_as_i64(int(seed))
    step = 1 << 24
    for p0 in range(0, pairs, step):
        npair = min(step, pairs - p0)
        idx = torch.arange(2 * p0 + 1, 2 * p0 + 2 * npair + 1, dtype=torch.int64, device=device)
        z = sd + idx * g
        z = (z ^ _t_shr(z, 30)) * m1
        z = (z ^ _t_shr(z, 27)) * m2
        z = z ^ _t_shr(z, 31)
        u = (_t_shr(z, 11).to(torch.float64) + 1.0) * (2.0 ** -53)
        u = u.reshape(npair, 2)
        r = torch.sqrt(-2.0 * torch.log(u[:, 0]))
        th = (2.0 * math.pi) * u[:, 1]
        zz = torch.stack([r * torch.cos(th), r * torch.sin(th)], dim=1).reshape(-1)
        lo = 2 * p0
        n = min(2 * npair, count - lo)
        out[lo:lo + n] = zz[:n].to(torch.float32)
    return out


def _to_e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    x = x.clamp(-E4M3_MAX, E4M3_MAX)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _pow2_at_least(v: torch.Tensor) -> torch.Tensor:
    """The power of two 2^e with v <= 2^e (frexp: v = m * 2^e, 0.5 <= m < 1)."""
    _, e = torch.frexp(v)
    return torch.ldexp(torch.ones_like(v), e)


def quantize_1x128(x: torch.Tensor, pow2: bool = False) -> tuple[torch.Tensor, torch.Tensor]:
    """Per 1x128 row-block cast of ``x`` [R, K] (K % 128 == 0) -> (uint8 [R, K], fp32 [R, K/128]).
    With ``pow2`` the scale is rounded up to a power of two (UE8M0-representable scales)."""
    R, K = x.shape
    assert K % BLOCK == 0
    xb = x.reshape(R, K // BLOCK, BLOCK)
    amax = xb.abs().amax(dim=2).clamp_min(SCALE_FLOOR)
    s = (amax / E4M3_MAX).to(torch.float32)
    if pow2:
        s = _pow2_at_least(s)
    q = _to_e4m3_bytes(xb / s.unsqueeze(2)).reshape(R, K)
    return q.contiguous(), s.contiguous()


def quantize_128x128(x: torch.Tensor, pow2: bool = False) -> tuple[torch.Tensor, torch.Tensor]:
    """Per 128x128 block cast of ``x`` [N, K] -> (uint8 [N, K], fp32 [ceil(N/128), K/128]); ``pow2`` as
    for quantize_1x128."""
    N, K = x.shape
    assert K % BLOCK == 0
    nb = (N + BLOCK - 1) // BLOCK
    pad = nb * BLOCK - N
    xp = torch.nn.functional.pad(x, (0, 0, 0, pad)) if pad else x
    xb = xp.reshape(nb, BLOCK, K // BLOCK, BLOCK)
    amax = xb.abs().amax(dim=(1, 3)).clamp_min(SCALE_FLOOR)
    s = (amax / E4M3_MAX).to(torch.float32)
    if pow2:
        s = _pow2_at_least(s)
    q = _to_e4m3_bytes(xb / s[:, None, :, None]).reshape(nb * BLOCK, K)[:N]
    return q.contiguous(), s.contiguous()


# Where the matrices are drawn: "cpu" (numpy, the definition) or a torch device (same values).
_GEN_DEVICE = "cpu"


def set_generation_device(device) -> None:
    """Draw subsequent inputs on ``device`` (e.g. "cuda") with :func:`normals_torch`; "cpu" restores
    the numpy path. The values are the same either way."""
    global _GEN_DEVICE
    _GEN_DEVICE = str(device)


def _normal_matrix(seed: int, stream: int, rows: int, cols: int) -> torch.Tensor:
    if _GEN_DEVICE != "cpu":
        return normals_torch(_stream_seed(seed, stream), rows * cols, _GEN_DEVICE).reshape(rows, cols)
    return torch.from_numpy(normals(_stream_seed(seed, stream), rows * cols)).reshape(rows, cols)


def seed_for(config_index: int, sub_index: int = 0) -> int:
    """Seed of sub-case ``sub_index`` of workload ``config_index``: 0xD6E0 + 1000*config + sub."""
    return 0xD6E0 + 1000 * config_index + sub_index


@dataclass
class NormalCase:
    """Inputs of ``D[M,N] = A[M,K] . B[N,K]^T`` with 1x128 / 128x128 scales."""
    M: int
    N: int
    K: int
    A: torch.Tensor      # uint8 [M, K] e4m3 codes
    sfa: torch.Tensor    # fp32 [M, K/128]
    B: torch.Tensor      # uint8 [N, K]
    sfb: torch.Tensor    # fp32 [ceil(N/128), K/128]


def make_normal(seed: int, M: int, N: int, K: int, pow2: bool = False) -> NormalCase:
    A, sfa = quantize_1x128(_normal_matrix(seed, STREAM_A, M, K), pow2)
    B, sfb = quantize_128x128(_normal_matrix(seed, STREAM_B, N, K), pow2)
    return NormalCase(M, N, K, A, sfa, B, sfb)


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclass
class ContiguousCase:
    """m-grouped contiguous layout: expert segments of A stacked along M, each padded to 128 rows."""
    G: int
    N: int
    K: int
    group_m: list            # real rows per group
    Mt: int                  # total (padded) rows
    A: torch.Tensor          # uint8 [Mt, K]
    sfa: torch.Tensor        # fp32 [Mt, K/128]
    B: torch.Tensor          # uint8 [G, N, K]
    sfb: torch.Tensor        # fp32 [G, ceil(N/128), K/128]
    m_indices: torch.Tensor  # int32 [Mt], group of each row, -1 on padding rows


def contiguous_group_sizes(seed: int, G: int, base_m: int, lo: float = 0.7, hi: float = 1.3) -> list:
    u = uniforms(_stream_seed(seed, STREAM_SIZES), G)
    return [int(base_m * (lo + (hi - lo) * float(x))) for x in u]


def make_contiguous(seed: int, G: int, N: int, K: int, group_m: list) -> ContiguousCase:
    seg = [_round_up(m, BLOCK) for m in group_m]
    Mt = sum(seg)
    A, sfa = quantize_1x128(_normal_matrix(seed, STREAM_A, Mt, K)) if Mt else (
        torch.zeros(0, K, dtype=torch.uint8), torch.zeros(0, K // BLOCK, dtype=torch.float32))
    m_idx = torch.full((Mt,), -1, dtype=torch.int32, device=A.device)
    r = 0
    for g, (m, s) in enumerate(zip(group_m, seg)):
        m_idx[r:r + m] = g
        r += s
    Bs, sfbs = [], []
    for g in range(G):
        b, sb = quantize_128x128(_normal_matrix(seed + 7919 * (g + 1), STREAM_B, N, K))
        Bs.append(b)
        sfbs.append(sb)
    return ContiguousCase(G, N, K, list(group_m), Mt, A, sfa, torch.stack(Bs), torch.stack(sfbs), m_idx)


@dataclass
class MaskedCase:
    """m-grouped masked layout: per-expert buffers [G, max_m, K]; only rows < masked_m[g] count."""
    G: int
    max_m: int
    N: int
    K: int
    expected_m: int
    A: torch.Tensor          # uint8 [G, max_m, K]
    sfa: torch.Tensor        # fp32 [G, max_m, K/128]
    B: torch.Tensor          # uint8 [G, N, K]
    sfb: torch.Tensor        # fp32 [G, ceil(N/128), K/128]
    masked_m: torch.Tensor   # int32 [G]


def masked_sizes(seed: int, G: int, expected_m: int, max_m: int, lo: float = 0.7, hi: float = 1.0) -> list:
    u = uniforms(_stream_seed(seed, STREAM_SIZES), G)
    return [min(max_m, int(expected_m * (lo + (hi - lo) * float(x)))) for x in u]


def make_masked(seed: int, G: int, max_m: int, N: int, K: int, masked_m: list, expected_m: int = 0) -> MaskedCase:
    A, sfa = quantize_1x128(_normal_matrix(seed, STREAM_A, G * max_m, K))
    Bs, sfbs = [], []
    for g in range(G):
        b, sb = quantize_128x128(_normal_matrix(seed + 7919 * (g + 1), STREAM_B, N, K))
        Bs.append(b)
        sfbs.append(sb)
    return MaskedCase(G, max_m, N, K, expected_m, A.reshape(G, max_m, K), sfa.reshape(G, max_m, K // BLOCK),
                      torch.stack(Bs), torch.stack(sfbs), torch.tensor(masked_m, dtype=torch.int32, device=A.device))


@dataclass
class KGroupedCase:
    """k-grouped weight gradient: per expert g, ``D[g] += A[:, Kg] . B[:, Kg]^T`` (fp32 out).

    ``A`` is X^T [M, sumK] and ``B`` is dY^T [N, sumK]; each expert's tokens occupy a contiguous
    column window of width ks[g] (a multiple of 128). Both operands carry 1x128 scales along K.
    """
    G: int
    M: int
    N: int
    ks: list
    A: torch.Tensor      # uint8 [M, sumK]
    sfa: torch.Tensor    # fp32 [M, sumK/128]
    B: torch.Tensor      # uint8 [N, sumK]
    sfb: torch.Tensor    # fp32 [N, sumK/128]
    D_in: torch.Tensor   # fp32 [G, M, N], the buffer accumulated into


def kgrouped_sizes(seed: int, G: int, base_k: int, lo: float = 0.5, hi: float = 1.5) -> list:
    u = uniforms(_stream_seed(seed, STREAM_SIZES), G)
    return [_round_up(int(base_k * (lo + (hi - lo) * float(x))), BLOCK) for x in u]


def make_kgrouped(seed: int, G: int, M: int, N: int, ks: list, din_scale: float = 1.0) -> KGroupedCase:
    sumK = sum(ks)
    A, sfa = quantize_1x128(_normal_matrix(seed, STREAM_A, M, sumK))
    B, sfb = quantize_1x128(_normal_matrix(seed, STREAM_B, N, sumK))
    D_in = (_normal_matrix(seed, STREAM_DIN, G * M, N) * din_scale).reshape(G, M, N).contiguous()
    return KGroupedCase(G, M, N, list(ks), A, sfa, B, sfb, D_in)


BF16_SENTINEL = 0xFFFF  # a BF16 NaN bit pattern used to pre-fill outputs whose rows must stay unwritten
