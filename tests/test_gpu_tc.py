"""The tcgen05 tensor-core path (M >= 32) against the CPU oracle (GPU).

The tile kernels round each de-quantized operand once to fp16 and accumulate in
f32, so every output must be within 2e-3 of T = sum_k |term_k|.  Shapes cover
ragged N (row tiles of 128), ragged M (activation tiles of 32/64/128/256), K not a
multiple of the 128-column stage, and the full-size prefill matrices (sampled).
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3


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


def assert_within(gpu, ref, T, what):
    err = np.abs(np.asarray(gpu, np.float64) - ref)
    bad = err > REL_TOL * T
    assert not bad.any(), f"{what}: {bad.sum()} outputs beyond {REL_TOL} T, worst {float((err / np.maximum(T, 1e-30)).max()):.3g}"


SMALL = [(32, 256, 512, 0), (33, 300, 96, 1), (64, 130, 256, 2), (100, 1000, 1024, 3), (128, 512, 4096, 4),
         (17, 128, 128, 5), (160, 257, 384, 6)]


@pytest.mark.parametrize("M,N,K,seed", SMALL)
def test_tc_q4_0(oracle, M, N, K, seed):
    w, x = synth.problem(200 + seed, M, N, K, outliers=(seed % 2 == 0))
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    dst = host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=gq.GQ_PATH_TC))
    ref, T = oracle.mul_mat_q4_0_f32(oracle.quantize_q4_0(w), x)
    assert_within(dst, ref, T, "q4_0 tc")


@pytest.mark.parametrize("M,N,K,seed", SMALL)
def test_tc_f16(oracle, M, N, K, seed):
    w, x = synth.problem(300 + seed, M, N, K, outliers=(seed % 2 == 1))
    wb = synth.f16_bits(w)
    dst = host(gq.mul_mat_f16_f32(dev(wb.view(np.int16)), dev(x), path=gq.GQ_PATH_TC))
    ref, T = oracle.mul_mat_f16_f32(wb, x)
    assert_within(dst, ref, T, "f16 tc")


@pytest.mark.parametrize("M,N,K", [(64, 11008, 4096), (128, 11008, 4096), (512, 4096, 4096), (128, 4096, 11008),
                                   (256, 11008, 4096), (64, 4096, 4096), (128, 4096, 4096), (512, 11008, 4096)])
def test_tc_full_size_sampled(oracle, M, N, K):
    """The prefill shapes, outliers included, in the configuration the benchmark times (auto dispatch);
    M = 256 on 11008 rows takes the 256-wide activation tile."""
    w, x = synth.problem(400 + M, M, N, K, outliers=True)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    dst = host(gq.mul_mat_q4_0_f32(rep, dev(x), N))
    q4 = oracle.quantize_q4_0(w)
    rng = np.random.default_rng(M + N)
    ms, ns = rng.integers(0, M, 2048), rng.integers(0, N, 2048)
    ref, T = oracle.mul_mat_q4_0_q8_0_at(q4, oracle.quantize_q8_0(x), ms, ns)
    assert_within(dst[ms, ns], ref, T, "q4_0 tc full size")
    wb = synth.f16_bits(w)
    dst16 = host(gq.mul_mat_f16_f32(dev(wb.view(np.int16)), dev(x)))
    ref16, T16 = oracle.mul_mat_f16_f32_at(wb, x, ms, ns)
    assert_within(dst16[ms, ns], ref16, T16, "f16 tc full size")


def test_dispatch_threshold():
    """M <= threshold runs the GEMV family (bit-exact row independence), above it the tiles."""
    assert gq.gq_get_m_threshold() == 16
    M, N, K = 20, 256, 512
    w, x = synth.problem(9, M, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    auto = host(gq.mul_mat_q4_0_f32(rep, dev(x), N))
    tc = host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=gq.GQ_PATH_TC))
    assert np.array_equal(auto, tc)
    try:
        gq.gq_set_m_threshold(32)
        auto = host(gq.mul_mat_q4_0_f32(rep, dev(x), N))
        gemv = host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=gq.GQ_PATH_GEMV))
        assert np.array_equal(auto, gemv)
    finally:
        gq.gq_set_m_threshold(16)


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("M,N,K", [(40, 300, 4096), (32, 131, 3200), (100, 520, 2048), (128, 256, 4096)])
def test_tc_split_k(oracle, monkeypatch, split, M, N, K):
    """Split-K over a cluster of 2, 4 or 8 CTAs (forced with GQ_TC_SPLIT): ragged M and N, K
    ranges of unequal length; within the tolerance of the oracle and within f32 reordering of
    the unsplit tiles' result."""
    w, x = synth.problem(600 + split + M, M, N, K, outliers=True)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    monkeypatch.setenv("GQ_TC_SPLIT", "1")
    whole = host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=gq.GQ_PATH_TC))
    monkeypatch.setenv("GQ_TC_SPLIT", str(split))
    dst = host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=gq.GQ_PATH_TC))
    again = host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=gq.GQ_PATH_TC))
    assert np.array_equal(dst, again), "split-K result is not deterministic"
    ref, T = oracle.mul_mat_q4_0_f32(oracle.quantize_q4_0(w), x)
    assert_within(dst, ref, T, f"q4_0 tc split {split}")
    assert np.all(np.abs(dst.astype(np.float64) - whole) <= 1e-5 * T + 1e-30), "split and unsplit tiles disagree"
    wb = synth.f16_bits(w)
    d16 = host(gq.mul_mat_f16_f32(dev(wb.view(np.int16)), dev(x), path=gq.GQ_PATH_TC))
    ref16, T16 = oracle.mul_mat_f16_f32(wb, x)
    assert_within(d16, ref16, T16, f"f16 tc split {split}")
