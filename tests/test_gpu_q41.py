"""Q4_1 weights (gq_quantize_q4_1, gq_repack_q4_1, gq_mul_mat_q4_1_f32) against the CPU oracle,
through the C ABI (GPU only).

The weights are quantized with the Q4_1 quantizer (bit-exact against the
oracle), repacked (bit-exact against the numpy statement of the layout), and
multiplied: every output within 2e-3 of T and within the bound that f32
accumulation of the exact int32 block sums allows.
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth
from layout_ref import repack_q4_1_ref
from oracle_pins import decode_q4_1, decode_q8_0
from test_gpu_parity import assert_within, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert gq.gq_last_error() == gq.GQ_OK


def q41_weights(w):
    N, K = w.shape
    q41 = gq.quantize_q4_1(dev(w))
    return q41, gq.repack_q4_1(q41, N, K)


def exact_bound(o, qw, x):
    """(2 nb + 16) * 2^-23 * sum_b (|d dx sumi| + |m dx sx|): f32 accumulation of the exact
    integer block sums, two terms per block."""
    qx = o.quantize_q8_0(x)
    sums = o.block_sums_q4_1(qw, qx).astype(np.float64)
    _, d, m = decode_q4_1(qw)
    _, dx = decode_q8_0(qx)
    t = np.einsum("nb,mb,mnb->mn", np.abs(d), np.abs(dx), np.abs(sums[..., 0])) + \
        np.einsum("nb,mb,mnb->mn", np.abs(m), np.abs(dx), np.abs(sums[..., 1]))
    return (2 * qw.shape[1] + 16) * 2.0 ** -23 * t


@pytest.mark.parametrize("N,K", [(16, 128), (37, 96), (300, 1024), (533, 544)])
def test_quantize_and_repack(oracle, N, K):
    w = synth.weights(N + K, N, K)
    q41, rep = q41_weights(w)
    want = oracle.quantize_q4_1(w)
    assert np.array_equal(host(q41), want)
    assert np.array_equal(host(rep), repack_q4_1_ref(want))


CASES = [
    (1, 256, 512, 0), (2, 200, 96, 1), (3, 1000, 1024, 2), (7, 64, 32, 3), (8, 515, 544, 4),
    (9, 300, 4096, 5), (16, 4096, 4096, 6), (13, 2000, 512, 7), (1, 4096, 11008, 8), (5, 11008, 128, 9),
    (24, 100, 256, 10), (40, 77, 352, 11), (1, 300, 96, 12), (1, 37, 544, 14),
]


@pytest.mark.parametrize("M,N,K,seed", CASES)
def test_mul_mat_q4_1(oracle, M, N, K, seed):
    w, x = synth.problem(seed, M, N, K, outliers=(seed % 2 == 1))
    _, rep = q41_weights(w)
    dst = host(gq.mul_mat_q4_1_f32(rep, dev(x), N))
    qw = oracle.quantize_q4_1(w)
    ref, T = oracle.mul_mat_q4_1_f32(qw, x)
    assert_within(dst, ref, T, what="q4_1 gemv")
    assert np.all(np.abs(dst.astype(np.float64) - ref) <= exact_bound(oracle, qw, x)), "beyond the exact bound"


def test_edge_inputs(oracle):
    for M, K in ((11, 640), (1, 640), (1, 11008)):
        N = 97
        w = synth.edge_weights(40, N, K)
        x = synth.edge_activations(41 + M, M, K)
        _, rep = q41_weights(w)
        dst = host(gq.mul_mat_q4_1_f32(rep, dev(x), N))
        qw = oracle.quantize_q4_1(w)
        ref, T = oracle.mul_mat_q4_1_f32(qw, x)
        assert_within(dst, ref, T, what="edge q4_1")
        assert np.all(dst[T == 0] == 0)


def test_row_independence():
    """Row m of an M-row product is bit-identical to the product of row m alone (dp4a and
    MMA shapes add the same exact block dots in the same order)."""
    M, N, K = 9, 700, 1536
    w, x = synth.problem(40, M, N, K)
    _, rep = q41_weights(w)
    full = host(gq.mul_mat_q4_1_f32(rep, dev(x), N))
    for m in range(M):
        one = host(gq.mul_mat_q4_1_f32(rep, dev(x[m:m + 1]), N))
        assert np.array_equal(full[m], one[0]), f"row {m}"


def test_sentinels():
    M, N, K = 5, 131, 256
    w, x = synth.problem(50, M, N, K)
    _, rep = q41_weights(w)
    pad = 1024
    buf = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
    gq.gq_mul_mat_q4_1_f32(rep, dev(x), buf[pad:pad + M * N], M, N, K)
    b = host(buf)
    assert np.isnan(b[:pad]).all() and np.isnan(b[-pad:]).all() and np.isfinite(b[pad:-pad]).all()


@pytest.mark.parametrize("M,N,K", [(M, N, K) for (N, K) in synth.DECODE_SHAPES for M in (1, 8, 16)])
def test_full_size_sampled(oracle, M, N, K):
    """The 7B-shaped decode matrices: quantized bytes exact, 2048 sampled outputs."""
    w, x = synth.problem(100 + M, M, N, K)
    q41, rep = q41_weights(w)
    dst = host(gq.mul_mat_q4_1_f32(rep, dev(x), N))
    qw = oracle.quantize_q4_1(w)
    assert np.array_equal(host(q41), qw)
    rng = np.random.default_rng(M * 7 + N)
    ms = rng.integers(0, M, 2048)
    ns = rng.integers(0, N, 2048)
    ref, T = oracle.mul_mat_q4_1_q8_0_at(qw, oracle.quantize_q8_0(x), ms, ns)
    assert_within(dst[ms, ns], ref, T, what="q4_1 full size")
