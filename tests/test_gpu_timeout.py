"""The failure path of the bounded in-kernel waits (GPU only).

A probe kernel (gq_debug_wait_timeout) waits, with a short poll limit, on an
mbarrier that nothing completes and that no copy signals; the wait gives up, the
kernel records the timeout in the device status word and returns.  No GPU fault
is involved: the kernel ends by itself.  The test checks that the timeout is
reported once by gq_last_error(), and that the products that follow (both kernel
families, with their workspace counters reset by that report) still match the
oracle.
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth
from test_gpu_parity import assert_within, dev, exact_dot_bound, host, run_q4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert gq.gq_last_error() == gq.GQ_OK


def test_probe_rejects_bad_limits():
    for limit in (0, (1 << 22) + 1):
        with pytest.raises(gq.GQError) as e:
            gq.gq_debug_wait_timeout(limit)
        assert e.value.status == gq.GQ_ERR_INVALID_ARG


@pytest.mark.parametrize("limit", [1, 1000])
def test_timeout_is_reported_and_the_next_products_are_right(oracle, limit):
    assert gq.gq_last_error() == gq.GQ_OK
    gq.gq_debug_wait_timeout(limit)
    assert gq.gq_last_error() == gq.GQ_ERR_TIMEOUT
    assert gq.gq_last_error() == gq.GQ_OK            # reading it cleared it
    for M, N, K, seed in ((1, 4096, 4096, 1), (4, 300, 4096, 2), (13, 2000, 512, 3), (64, 512, 1024, 4)):
        w, x = synth.problem(seed, M, N, K)
        path = gq.GQ_PATH_GEMV if M <= 16 else gq.GQ_PATH_TC
        q4, dst = run_q4(w, x, path)
        q4_ref = oracle.quantize_q4_0(w)
        assert np.array_equal(host(q4), q4_ref)
        ref, T = oracle.mul_mat_q4_0_f32(q4_ref, x)
        assert_within(dst, ref, T, what=f"after a timeout, M={M} N={N} K={K}")
        if M <= 16:
            err = np.abs(dst.astype(np.float64) - ref)
            assert np.all(err <= exact_dot_bound(oracle, q4_ref, x))
    assert gq.gq_last_error() == gq.GQ_OK
