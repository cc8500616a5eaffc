"""Helpers shared by the GPU parity tests: device copies, sentinels and the tolerance checks.

Tolerances (stated for this workload): BF16 outputs must satisfy, element by element,
|gpu - oracle| <= 1e-2 |oracle| + 1e-2 rms(oracle), and globally
1 - 2<x,y> / (|x|^2 + |y|^2) < 1e-5; FP32 weight gradients must satisfy |gpu - oracle| <= 1e-4 rms(oracle).
The GPU differs from the oracle only in where it rounds: the tensor cores' accumulation inside a
128-K block, the FP32 promotion sum and the single final rounding.
"""
import numpy as np
import torch

from moe_grouped_gemm_tma_gb300 import inputs as I

SENTINEL = I.BF16_SENTINEL


def dev(t):
    return t.contiguous().cuda()


def sentinel_bf16(*shape):
    return torch.full(shape, SENTINEL - 65536, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def bf16_bits(t):
    """uint16 numpy bits of a bf16 tensor (any device)."""
    return t.detach().view(torch.int16).cpu().numpy().astype(np.uint16)


def bits_to_f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_bf16(got_bits, want_bits, what=""):
    got_bits = np.asarray(got_bits)
    want_bits = np.asarray(want_bits)
    assert got_bits.shape == want_bits.shape, (got_bits.shape, want_bits.shape)
    g, w = bits_to_f64(got_bits), bits_to_f64(want_bits)
    assert np.isfinite(w).all(), f"{what}: oracle produced non-finite values"
    bad_nan = ~np.isfinite(g)
    assert not bad_nan.any(), f"{what}: {bad_nan.sum()} non-finite GPU outputs, first at {np.argwhere(bad_nan)[:5]}"
    rms = float(np.sqrt(np.mean(w * w))) if w.size else 0.0
    err = np.abs(g - w)
    bound = 1e-2 * np.abs(w) + 1e-2 * rms
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; worst at "
                           f"{np.unravel_index(np.argmax(err - bound), err.shape)} got "
                           f"{g.flat[np.argmax(err - bound)]} want {w.flat[np.argmax(err - bound)]} (rms {rms})")
    den = float((g * g).sum() + (w * w).sum())
    if den > 0:
        diff = 1.0 - 2.0 * float((g * w).sum()) / den
        assert diff < 1e-5, f"{what}: global similarity defect {diff}"


def check_f32(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape
    assert np.isfinite(got).all(), f"{what}: non-finite GPU outputs"
    rms = float(np.sqrt(np.mean(want * want)))
    err = np.abs(got - want)
    assert (err <= 1e-4 * rms).all(), f"{what}: max err {err.max()} > {1e-4 * rms} (rms {rms})"


def sample_rows(total, count, seed, must=()):
    """Sorted row sample: the given rows, tile-boundary rows and a seeded random subset."""
    rng = np.random.default_rng(seed)
    rows = {r for r in must if 0 <= r < total}
    for r in (0, 1, 127, 128, 255, 256, total - 1, total - 2):
        if 0 <= r < total:
            rows.add(r)
    extra = max(0, min(count, total) - len(rows))
    if extra:
        rows.update(int(x) for x in rng.choice(total, size=min(extra, total), replace=False))
    return np.array(sorted(rows), dtype=np.int64)


def pack_ue8m0(sf):
    """FP32 power-of-two scales [rows, kbs] -> packed UE8M0 int32 [rows, ceil(kbs/4)] (byte j of word w =
    biased exponent of block 4w + j); unused trailing bytes are 0xEE, which the kernel must ignore."""
    sf = sf.contiguous().numpy()
    rows, kbs = sf.shape
    words = (kbs + 3) // 4
    e = np.full((rows, words * 4), 0xEE, dtype=np.uint8)
    bits = sf.view(np.uint32)
    assert ((bits & 0x807FFFFF) == 0).all()
    e[:, :kbs] = (bits >> 23).astype(np.uint8)
    return torch.from_numpy(e.view(np.int32).reshape(rows, words).copy())
