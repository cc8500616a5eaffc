"""The packed UE8M0 scale format that dg_gemm_fp8_nt_ue8m0_packed takes (four biased exponents per
int32, least significant byte first, scale = 2^(e - 127)), pinned on the CPU: the test helper that
packs FP32 power-of-two scales for the GPU tests against words worked out by hand, and against the
decoding the header states."""
import numpy as np
import pytest
import torch

from tests.gpu_util import pack_ue8m0

FILL = 0xEE  # the helper's value for bytes past the last K block


def _word(b0, b1, b2, b3):
    """int32 whose bytes, least significant first, are b0..b3."""
    u = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24)
    return u - (1 << 32) if u >= (1 << 31) else u


def test_hand_packed_words():
    sf = torch.tensor([[1.0, 0.5, 1024.0, 2.0 ** -20, 4.0],
                       [2.0 ** -126, 2.0 ** 127, 1.0, 1.0, 0.25]], dtype=torch.float32)
    got = pack_ue8m0(sf)
    assert got.dtype == torch.int32 and tuple(got.shape) == (2, 2)
    # exponents: 1 -> 127, 1/2 -> 126, 1024 -> 137, 2^-20 -> 107, 4 -> 129, 2^-126 -> 1, 2^127 -> 254
    want = [[_word(127, 126, 137, 107), _word(129, FILL, FILL, FILL)],
            [_word(1, 254, 127, 127), _word(125, FILL, FILL, FILL)]]
    assert got.tolist() == want
    assert want[0][0] == 1804172927 and want[0][1] == -286331263


@pytest.mark.parametrize("kbs", [1, 3, 4, 5, 8, 56, 57])
def test_decoding_as_the_header_states_recovers_the_scales(kbs):
    rng = np.random.default_rng(kbs)
    e = rng.integers(1, 255, size=(7, kbs))
    sf = torch.from_numpy(np.ldexp(1.0, e - 127).astype(np.float32))
    words = pack_ue8m0(sf).numpy().astype(np.int64) & 0xFFFFFFFF
    assert words.shape == (7, (kbs + 3) // 4)
    for kb in range(kbs):
        byte = (words[:, kb // 4] >> (8 * (kb % 4))) & 0xFF
        np.testing.assert_array_equal(byte, e[:, kb])
        np.testing.assert_array_equal(np.ldexp(1.0, byte - 127), sf[:, kb].numpy().astype(np.float64))


def test_scales_that_are_not_powers_of_two_are_refused():
    with pytest.raises(AssertionError):
        pack_ue8m0(torch.tensor([[1.5]], dtype=torch.float32))
    with pytest.raises(AssertionError):
        pack_ue8m0(torch.tensor([[-2.0]], dtype=torch.float32))
