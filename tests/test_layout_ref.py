"""The two numpy statements of the repacked layout agree (CPU): the vectorized
one used by the GPU tests and a byte-by-byte transcription of the header text."""
import numpy as np
import pytest

from layout_ref import repack_ref, repack_loops


@pytest.mark.parametrize("N,nb", [(16, 4), (37, 3), (33, 9), (1, 1), (64, 16)])
def test_layout_statements_agree(N, nb):
    rng = np.random.default_rng(N * 100 + nb)
    q4 = rng.integers(0, 256, size=(N, nb, 18), dtype=np.uint8)
    assert np.array_equal(repack_ref(q4), repack_loops(q4))


@pytest.mark.parametrize("N,K", [(16, 32), (37, 96), (1, 64), (33, 160)])
def test_f16_layout_statements_agree(N, K):
    from layout_ref import repack_f16_ref, repack_f16_loops
    rng = np.random.default_rng(N * 1000 + K)
    w16 = rng.integers(0, 1 << 16, size=(N, K), dtype=np.uint16)
    assert np.array_equal(repack_f16_ref(w16), repack_f16_loops(w16))


@pytest.mark.parametrize("N,nb", [(16, 4), (37, 3), (33, 9), (1, 1)])
def test_q8_0_layout_statements_agree(N, nb):
    from layout_ref import repack_q8_0_ref, repack_q8_0_loops
    rng = np.random.default_rng(N * 10 + nb)
    q8 = rng.integers(0, 256, size=(N, nb, 34), dtype=np.uint8)
    assert np.array_equal(repack_q8_0_ref(q8), repack_q8_0_loops(q8))


def test_q5_0_high_word_gives_the_codes():
    """The stored fifth-bit word, shifted and masked as the kernel does for word w of a block,
    puts the fifth bit of each element at bit 4 of that element's byte."""
    from layout_ref import _q5_high_word
    rng = np.random.default_rng(3)
    for qh in [0, 0xFFFFFFFF, 0x0000FFFF, 0xFFFF0000] + [int(v) for v in rng.integers(0, 1 << 32, 20)]:
        h = _q5_high_word(qh)
        for w in range(4):
            lo = (h >> (3 - w)) & 0x10101010
            hi = (h << (1 + w)) & 0x10101010 & 0xFFFFFFFF
            for b in range(4):
                assert ((lo >> (8 * b + 4)) & 1) == (qh >> (4 * w + b)) & 1
                assert ((hi >> (8 * b + 4)) & 1) == (qh >> (16 + 4 * w + b)) & 1


@pytest.mark.parametrize("N,nb", [(16, 4), (37, 3), (33, 9), (1, 1)])
def test_q4_1_layout_statements_agree(N, nb):
    from layout_ref import repack_q4_1_ref, repack_q4_1_loops
    rng = np.random.default_rng(N * 7 + nb)
    q41 = rng.integers(0, 256, size=(N, nb, 20), dtype=np.uint8)
    assert np.array_equal(repack_q4_1_ref(q41), repack_q4_1_loops(q41))
