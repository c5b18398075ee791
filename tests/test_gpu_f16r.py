"""F16 weights in the 16 x 32 tile layout (gq_repack_f16, gq_mul_mat_f16r_f32)
against the CPU oracle, through the C ABI (GPU only).

The repack is a byte permutation: bit-exact against the numpy statement of the
layout.  The product rounds the activations to fp16 and accumulates fp16
products in f32: every output within 2e-3 of T = sum_k |w_nk x_mk|.
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth
from layout_ref import repack_f16_ref
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


def f16_dev(w):
    return dev(synth.f16_bits(w).view(np.int16))


@pytest.mark.parametrize("N,K", [(16, 32), (37, 96), (1, 64), (300, 4096), (4111, 544)])
def test_repack_layout(N, K):
    w = synth.weights(N + K, N, K)
    got = host(gq.repack_f16(f16_dev(w)))
    assert np.array_equal(got, repack_f16_ref(synth.f16_bits(w)))


CASES = [
    (1, 256, 512, 0), (2, 200, 96, 1), (3, 1000, 1024, 2), (7, 64, 32, 3), (8, 515, 544, 4),
    (9, 300, 4096, 5), (16, 4096, 4096, 6), (13, 2000, 512, 7), (1, 4096, 11008, 8), (5, 11008, 128, 9),
    (24, 100, 256, 10), (40, 77, 352, 11), (16, 96, 11008, 12), (1, 17, 32, 13),
]


@pytest.mark.parametrize("M,N,K,seed", CASES)
def test_mul_mat_f16r(oracle, M, N, K, seed):
    w, x = synth.problem(seed, M, N, K, outliers=(seed % 2 == 1))
    rep = gq.repack_f16(f16_dev(w))
    dst = host(gq.mul_mat_f16r_f32(rep, dev(x), N))
    ref, T = oracle.mul_mat_f16_f32(synth.f16_bits(w), x)
    assert_within(dst, ref, T, what="f16r gemv")


def test_edge_inputs(oracle):
    M, N, K = 11, 97, 640
    w = synth.edge_weights(30, N, K).astype(np.float16).astype(np.float32)
    x = synth.edge_activations(31, M, K)
    rep = gq.repack_f16(f16_dev(w))
    dst = host(gq.mul_mat_f16r_f32(rep, dev(x), N))
    ref, T = oracle.mul_mat_f16_f32(synth.f16_bits(w), x)
    assert_within(dst, ref, T, what="edge f16r")
    assert np.all(dst[T == 0] == 0)


def test_row_independence():
    """Row m of an M-row product is bit-identical to the product of row m alone."""
    M, N, K = 9, 700, 1536
    w, x = synth.problem(40, M, N, K)
    rep = gq.repack_f16(f16_dev(w))
    full = host(gq.mul_mat_f16r_f32(rep, dev(x), N))
    for m in range(M):
        one = host(gq.mul_mat_f16r_f32(rep, dev(x[m:m + 1]), N))
        assert np.array_equal(full[m], one[0]), f"row {m}"


def test_repeatable_and_sentinels():
    M, N, K = 5, 131, 256
    w, x = synth.problem(50, M, N, K)
    rep = gq.repack_f16(f16_dev(w))
    pad = 1024
    buf = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
    dst = buf[pad:pad + M * N]
    gq.gq_mul_mat_f16r_f32(rep, dev(x), dst, M, N, K)
    b = host(buf)
    assert np.isnan(b[:pad]).all() and np.isnan(b[-pad:]).all()
    assert np.isfinite(b[pad:-pad]).all()
    again = host(gq.mul_mat_f16r_f32(rep, dev(x), N))
    assert np.array_equal(again.reshape(-1), b[pad:-pad])


@pytest.mark.parametrize("M,N,K", [(M, N, K) for (N, K) in synth.DECODE_SHAPES for M in (1, 8, 16)])
def test_full_size_sampled(oracle, M, N, K):
    """The 7B-shaped decode matrices: 2048 sampled outputs against the oracle."""
    w, x = synth.problem(100 + M, M, N, K)
    rep = gq.repack_f16(f16_dev(w))
    dst = host(gq.mul_mat_f16r_f32(rep, dev(x), N))
    rng = np.random.default_rng(M * 7 + N)
    ms = rng.integers(0, M, 2048)
    ns = rng.integers(0, N, 2048)
    ref, T = oracle.mul_mat_f16_f32_at(synth.f16_bits(w), x, ms, ns)
    assert_within(dst[ms, ns], ref, T, what="f16r full size")
