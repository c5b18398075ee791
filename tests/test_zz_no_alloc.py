"""The allocation-free Q4_0 product (GPU).

gq_mul_mat_q4_0_f32_noalloc serves callers that cannot let a library allocate
device memory (a serving process whose pooling allocator reserved the memory up
front, a plug-in whose host runtime forbids allocation, a loop in which
cudaMalloc may not run).  It keeps its scratch in a static device array of the
library and runs the GEMV family, so its results must equal those of the default
entry point's GEMV, which takes its scratch from a cudaMalloc'ed per-stream
workspace, bit for bit and call after call, and lie within the exact-block-dot
bound of the oracle.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth
from oracle_pins import decode_q4_0, decode_q8_0

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def exact_dot_bound(o, q4, x):
    """(nb + 16) * 2^-23 * sum_b |d4 d8 sumi|: f32 accumulation of exact block dots."""
    q8 = o.quantize_q8_0(x)
    sumi = o.block_dots(q4, q8).astype(np.float64)
    _, d4 = decode_q4_0(q4)
    _, d8 = decode_q8_0(q8)
    return (q4.shape[1] + 16) * 2.0 ** -23 * np.einsum("nb,mb,mnb->mn", np.abs(d4), np.abs(d8), np.abs(sumi))


# one case per scratch use: no scratch (M = 1), the INIT images (M = 9), the K-split with
# partial sums and counters (M = 16, K = 11008), and 16-row chunks that reuse the same
# counters one after the other (M = 40)
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (9, 2000, 4096), (16, 4096, 11008), (40, 300, 4096)])
def test_noalloc_matches_default_entry_point(oracle, M, N, K):
    w, x = synth.problem(70 + M, M, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    q4_ref = oracle.quantize_q4_0(w)
    ref, _ = oracle.mul_mat_q4_0_f32(q4_ref, x)
    bound = exact_dot_bound(oracle, q4_ref, x)
    xd = dev(x)
    want = torch.empty((M, N), device="cuda")
    gq.gq_mul_mat_q4_0_f32_path(rep, xd, want, M, N, K, gq.GQ_PATH_GEMV)
    torch.cuda.synchronize()
    want = want.cpu().numpy()
    for call in range(2):                      # the array keeps the previous call's contents
        out = torch.full((M, N), float("nan"), device="cuda")
        gq.gq_mul_mat_q4_0_f32_noalloc(rep, xd, out, M, N, K)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got, want), f"call {call}: differs from the default entry point's GEMV"
        assert np.all(np.abs(got.astype(np.float64) - ref) <= bound), f"call {call}: beyond the exact-block-dot bound"
    assert gq.gq_last_error() == gq.GQ_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0_f32_noalloc(0x10000, 0x10000, 0x10000, 1, 65536, 65536)
    assert e.value.status == gq.GQ_ERR_INVALID_ARG and "scratch" in str(e.value)
