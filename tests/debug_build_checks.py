"""Run with GQ_LIBRARY naming the GQ_DEBUG build (tests/test_gpu_debug_build.py does): every
kernel family on a few shapes, results against the oracle, and no device-side check failed."""
import math
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import quantized_skinny_matmul_gb300 as gq  # noqa: E402
from quantized_skinny_matmul_gb300 import synth  # noqa: E402


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def main() -> None:
    assert gq.LIB_PATH == os.environ["GQ_LIBRARY"], gq.LIB_PATH
    o = oracle.get()
    torch.cuda.set_device(0)
    rng = np.random.default_rng(5)
    # products: both GEMV kernels (one row; several rows, one and two K slices) and the tiles
    for M, N, K, path in ((1, 4096, 4096, gq.GQ_PATH_AUTO), (1, 300, 11008, gq.GQ_PATH_AUTO),
                          (4, 1000, 4096, gq.GQ_PATH_GEMV), (16, 700, 11008, gq.GQ_PATH_GEMV),
                          (64, 4096, 4096, gq.GQ_PATH_TC), (40, 300, 3200, gq.GQ_PATH_TC)):
        w, x = synth.problem(M + N, M, N, K)
        rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
        dst = gq.mul_mat_q4_0_f32(rep, dev(x), N, path=path).cpu().numpy().astype(np.float64)
        ms, ns = rng.integers(0, M, 256), rng.integers(0, N, 256)
        ref, T = o.mul_mat_q4_0_q8_0_at(o.quantize_q4_0(w), o.quantize_q8_0(x), ms, ns)
        assert np.all(np.abs(dst[ms, ns] - ref) <= 2e-3 * T), (M, N, K, path)
    # the INT8 KV cache: both attention kernels, every group size of the tensor-core one
    for B, Hq, Hkv, Tcap, D, lens in ((2, 8, 8, 300, 128, [300, 77]), (2, 16, 4, 700, 128, [700, 1]),
                                      (1, 16, 2, 5000, 128, [4999]), (3, 8, 2, 513, 64, [513, 0, 1])):
        qf, kf, vf = synth.kv_problem(B + Tcap, B, Hq, Hkv, Tcap, D)
        lens = np.array(lens, np.int32)
        k, ks = gq.kv_quantize_i8(dev(kf))
        v, vs = gq.kv_quantize_i8(dev(vf))
        c = 1.0 / math.sqrt(D)
        out = gq.attn_decode_i8(dev(qf), k, ks, v, vs, dev(lens), c).cpu().numpy()
        ok, oks = o.kv_quantize_i8(kf)
        ov, ovs = o.kv_quantize_i8(vf)
        ref, E, S = o.attn_decode_i8(qf, ok, oks, ov, ovs, lens, c)
        T = int(lens.max())
        tol = 2.0 * (70.0 * S[..., None] + T / 2.0 + 64.0) * 2.0 ** -24 * E + 1e-30
        assert np.all(np.abs(out - ref) <= tol), (B, Hq, Hkv, Tcap, D)
    torch.cuda.synchronize()
    status = gq.gq_last_error()
    assert status == gq.GQ_OK, f"gq_last_error() = {status}: {gq.lib().gq_last_error_message().decode()}"
    print("debug build clean")


if __name__ == "__main__":
    main()
