"""Exact check of the activation quantizer inside each product path (GPU only).

The weights are probes: row 32*b + j of src0 has d = 1 in every block, every
code 8 (weight 0) except element j of block b, whose code is 9 (weight 1).  The
product then has a single nonzero term per output,

    dst[m][32*b + j] = d8[m][b] * q8[m][b][j],

which the f32 arithmetic of the GEMV path reproduces exactly, so every Q8_0
code and scale that the fused (or separate) INIT stage produced can be read
back and compared with the oracle's quantizer bit for bit.  On the
tensor-core path the activation enters the MMA as the fp16 value of
q8 * d8, and the output is that value.

The activations are built to sit on and beside the rounding ties of x / d
(the Q8_0 code rounds ties away from zero), with blocks whose scale is a power
of two, blocks with an arbitrary scale, all-zero blocks and blocks whose
scale is subnormal.
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from oracle_pins import decode_q8_0

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert gq.gq_last_error() == gq.GQ_OK


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def probe_q4_0(K: int) -> np.ndarray:
    """Canonical Q4_0 bytes [K][K/32][18] of the probe rows described above."""
    nb = K // 32
    q4 = np.zeros((K, nb, 18), np.uint8)
    q4[:, :, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    q4[:, :, 2:] = 0x88
    r = np.arange(K)
    b, j = r // 32, r % 32
    lo = j < 16
    q4[r[lo], b[lo], 2 + j[lo]] = 0x89            # low nibble: element j
    q4[r[~lo], b[~lo], 2 + j[~lo] - 16] = 0x98    # high nibble: element j + 16 of byte j
    return q4


def tie_activations(seed: int, M: int, K: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    blocks = x.reshape(M, K // 32, 32)
    for m in range(M):
        for b in range(K // 32):
            kind = rng.integers(0, 6)
            k = rng.integers(-127, 127, 32).astype(np.float64)
            lead = rng.integers(0, 32)
            if kind == 0:      # power-of-two scale: x / d lands exactly on k + 1/2
                c = np.float32(2.0 ** rng.integers(-12, 5))
                v = ((k + 0.5) * c).astype(np.float32)
                v[lead] = np.float32(127 * c) * rng.choice([-1, 1])
            elif kind == 1:    # arbitrary scale: near the ties of the f32 quotient, a few ulps either side
                amax = np.float32(rng.uniform(0.01, 30.0))
                d = np.float32(amax / np.float32(127.0))
                v = ((k + 0.5) * np.float64(d)).astype(np.float32)
                steps = rng.integers(-3, 4, 32)
                v = np.array([np.float32(t) if s == 0 else
                              np.nextafter(np.float32(t), np.float32(np.inf if s > 0 else -np.inf), dtype=np.float32)
                              for t, s in zip(v, steps)], np.float32)
                v[lead] = amax * rng.choice([-1, 1])
            elif kind == 2:    # all zero
                v = np.zeros(32, np.float32)
            elif kind == 3:    # subnormal scale: 1/d overflows
                v = (rng.uniform(-1, 1, 32) * 1e-38).astype(np.float32)
            else:
                continue
            blocks[m, b] = v
    return x


def expected_gemv(oracle, x):
    codes, d8 = decode_q8_0(oracle.quantize_q8_0(x))
    return (d8.astype(np.float32)[..., None] * codes.astype(np.float32)).reshape(x.shape)


@pytest.mark.parametrize("M,K", [(1, 512), (5, 512), (16, 512), (1, 4096), (1, 11008), (2, 11008), (16, 4096)])
def test_gemv_q8_codes_exact(oracle, M, K):
    x = tie_activations(1000 + M + K, M, K)
    rep = gq.repack_q4_0(dev(probe_q4_0(K)), K, K)
    dst = host(gq.mul_mat_q4_0_f32(rep, dev(x), K, path=gq.GQ_PATH_GEMV))
    want = expected_gemv(oracle, x)
    bad = ~(dst == want)              # == : a zero scale times a negative code may come out as either zero
    assert not bad.any(), f"{bad.sum()} codes differ; first at {tuple(np.argwhere(bad)[0])}"


@pytest.mark.parametrize("M,K", [(32, 512), (64, 4096)])
def test_tc_q8_codes_exact(oracle, M, K):
    x = tie_activations(2000 + M + K, M, K)
    rep = gq.repack_q4_0(dev(probe_q4_0(K)), K, K)
    dst = host(gq.mul_mat_q4_0_f32(rep, dev(x), K, path=gq.GQ_PATH_TC))
    want = expected_gemv(oracle, x).astype(np.float16).astype(np.float32)
    bad = ~(dst == want)
    assert not bad.any(), f"{bad.sum()} values differ; first at {tuple(np.argwhere(bad)[0])}"


def test_quantize_rows_q8_0_ties(oracle):
    x = tie_activations(3000, 7, 4096)
    q8 = gq.quantize_rows_q8_0(dev(x))
    assert np.array_equal(host(q8), oracle.quantize_q8_0(x))
