"""The allocation-free Q4_0 product (GPU).

gq_mul_mat_q4_0_f32_noalloc serves callers that cannot allocate device memory
(work recorded into a CUDA graph during capture, applications whose pooling
allocator owns all device memory).  It keeps its scratch in a static device
array of the library, so its results must match the default entry point, which
takes its scratch from a cudaMalloc'ed per-stream workspace, call after call.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# one case per scratch use: row-group ranges only (M = 1), the INIT images
# (M = 9), and the K-split with partial sums and counters (M = 16, K = 11008)
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (9, 2000, 4096), (16, 4096, 11008)])
def test_noalloc_matches_default_entry_point(oracle, M, N, K):
    w, x = synth.problem(70 + M, M, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    q4_ref = oracle.quantize_q4_0(w)
    _, T = oracle.mul_mat_q4_0_f32(q4_ref, x)
    xd = dev(x)
    ref = torch.empty((M, N), device="cuda")
    gq.gq_mul_mat_q4_0_f32(rep, xd, ref, M, N, K)
    for call in range(2):                      # the array keeps the previous call's contents
        out = torch.full((M, N), float("nan"), device="cuda")
        gq.gq_mul_mat_q4_0_f32_noalloc(rep, xd, out, M, N, K)
        torch.cuda.synchronize()
        a = out.cpu().numpy().astype(np.float64)
        b = ref.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(a - b) <= 2e-3 * T), f"call {call}: differs from gq_mul_mat_q4_0_f32"
    assert gq.gq_last_error() == gq.GQ_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0_f32_noalloc(0x10000, 0x10000, 0x10000, 1, 65536, 65536)
    assert e.value.status == gq.GQ_ERR_INVALID_ARG and "scratch" in str(e.value)
