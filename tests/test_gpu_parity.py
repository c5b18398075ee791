"""CUDA path vs the CPU oracle, through the C ABI (GPU only).

Bit-exact: Q4_0 and Q8_0 bytes, the repacked layout, the int32 block dots.
Floating point: every output within 2e-3 of T = sum_k |term_k| (the terms of the
de-quantized operands), and on the GEMV path also within the much tighter bound
that f32 accumulation of exact block dots allows, which an off-by-one Q8_0 code
in the fused quantizer would exceed.
"""
import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth
from layout_ref import repack_ref
from oracle_pins import decode_q4_0, decode_q8_0

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


def assert_within(gpu, ref, T, rel=REL_TOL, what=""):
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - ref)
    bad = err > rel * T
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs beyond {rel} * T; first {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]!r} ref={ref[tuple(i)]!r} T={T[tuple(i)]!r}")


def exact_dot_bound(o, q4, x):
    """(nb + 16) * 2^-23 * sum_b |d4 d8 sumi|: f32 accumulation of exact block dots."""
    q8 = o.quantize_q8_0(x)
    sumi = o.block_dots(q4, q8).astype(np.float64)
    _, d4 = decode_q4_0(q4)
    _, d8 = decode_q8_0(q8)
    Tb = np.einsum("nb,mb,mnb->mn", np.abs(d4), np.abs(d8), np.abs(sumi))
    return (q4.shape[1] + 16) * 2.0 ** -23 * Tb


# --------------------------------------------------------------------------- bytes
@pytest.mark.parametrize("N,K,kind,seed", [
    (256, 512, "normal", 0), (37, 96, "edge", 1), (130, 2048, "edge", 2), (4096, 4096, "normal", 3)])
def test_quantize_q4_0_bytes(oracle, N, K, kind, seed):
    w = synth.weights(seed, N, K) if kind == "normal" else synth.edge_weights(seed, N, K)
    q4 = gq.quantize_q4_0(dev(w))
    assert np.array_equal(host(q4), oracle.quantize_q4_0(w))


@pytest.mark.parametrize("M,K,kind,seed", [
    (1, 512, "normal", 0), (24, 512, "edge", 4), (16, 4096, "normal", 5), (3, 11008, "outliers", 6)])
def test_quantize_rows_q8_0_bytes(oracle, M, K, kind, seed):
    if kind == "edge":
        x = synth.edge_activations(seed, M, K)
    else:
        x = synth.activations(seed, M, K, outliers=(kind == "outliers"))
    q8 = gq.quantize_rows_q8_0(dev(x))
    assert np.array_equal(host(q8), oracle.quantize_q8_0(x))


@pytest.mark.parametrize("N,K", [(256, 512), (37, 96), (33, 4096), (16, 32)])
def test_repack_layout(oracle, N, K):
    q4 = oracle.quantize_q4_0(synth.edge_weights(7, N, K))
    rep = gq.repack_q4_0(dev(q4), N, K)
    assert np.array_equal(host(rep), repack_ref(q4))


@pytest.mark.parametrize("M,N,K", [(1, 16, 32), (11, 40, 160), (8, 256, 512), (3, 33, 4096)])
def test_block_dots_exact(oracle, M, N, K):
    q4 = oracle.quantize_q4_0(synth.edge_weights(8, N, K))
    q8 = oracle.quantize_q8_0(synth.edge_activations(9, M, K))
    rep = gq.repack_q4_0(dev(q4), N, K)
    sumi = torch.full((M, N, K // 32), -(2 ** 31), dtype=torch.int32, device="cuda")
    gq.gq_debug_block_dots_q4_0(rep, dev(q8), sumi, M, N, K)
    assert np.array_equal(host(sumi), oracle.block_dots(q4, q8))


# --------------------------------------------------------------------------- products
GEMV_CASES = [
    (1, 256, 512, 0), (2, 200, 96, 1), (3, 1000, 1024, 2), (7, 64, 32, 3), (8, 515, 544, 4),
    (9, 300, 4096, 5), (16, 4096, 4096, 6), (13, 2000, 512, 7), (1, 4096, 11008, 8), (5, 11008, 128, 9),
    (24, 100, 256, 10), (40, 77, 352, 11), (1, 300, 96, 12), (1, 100, 20000, 13), (1, 37, 544, 14),
]


def run_q4(w, x, path):
    N, K = w.shape
    q4 = gq.quantize_q4_0(dev(w))
    rep = gq.repack_q4_0(q4, N, K)
    return q4, host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=path))


@pytest.mark.parametrize("M,N,K,seed", GEMV_CASES)
def test_mul_mat_q4_0_gemv(oracle, M, N, K, seed):
    w, x = synth.problem(seed, M, N, K, outliers=(seed % 2 == 1))
    q4, dst = run_q4(w, x, gq.GQ_PATH_GEMV)
    q4_ref = oracle.quantize_q4_0(w)
    assert np.array_equal(host(q4), q4_ref)
    ref, T = oracle.mul_mat_q4_0_f32(q4_ref, x)
    assert_within(dst, ref, T, what="q4_0 gemv")
    err = np.abs(dst.astype(np.float64) - ref)
    assert np.all(err <= exact_dot_bound(oracle, q4_ref, x)), "beyond the exact-block-dot bound"


@pytest.mark.parametrize("M,N,K,seed", GEMV_CASES)
def test_mul_mat_f16_gemv(oracle, M, N, K, seed):
    w, x = synth.problem(seed, M, N, K, outliers=(seed % 2 == 1))
    wb = synth.f16_bits(w)
    dst = host(gq.mul_mat_f16_f32(dev(wb.view(np.int16)), dev(x), path=gq.GQ_PATH_GEMV))
    ref, T = oracle.mul_mat_f16_f32(wb, x)
    assert_within(dst, ref, T, what="f16 gemv")


def test_edge_inputs_q4_0(oracle):
    M, N, K = 11, 97, 640
    w = synth.edge_weights(30, N, K)
    x = synth.edge_activations(31, M, K)
    q4, dst = run_q4(w, x, gq.GQ_PATH_GEMV)
    q4_ref = oracle.quantize_q4_0(w)
    ref, T = oracle.mul_mat_q4_0_f32(q4_ref, x)
    assert_within(dst, ref, T, what="edge q4_0")
    assert np.all(dst[T == 0] == 0)


@pytest.mark.parametrize("M,K", [(1, 640), (1, 11008), (2, 640)])
def test_edge_inputs_q4_0_few_rows(oracle, M, K):
    """Zero blocks, exact Q8_0 ties and wide ranges with one or two activation rows (the
    one-row product quantizes its activations per warp, chunk by chunk)."""
    N = 97
    w = synth.edge_weights(32, N, K)
    x = synth.edge_activations(33 + M, M, K)
    q4, dst = run_q4(w, x, gq.GQ_PATH_GEMV)
    q4_ref = oracle.quantize_q4_0(w)
    ref, T = oracle.mul_mat_q4_0_f32(q4_ref, x)
    assert_within(dst, ref, T, what="edge q4_0")
    err = np.abs(dst.astype(np.float64) - ref)
    assert np.all(err <= exact_dot_bound(oracle, q4_ref, x)), "beyond the exact-block-dot bound"


@pytest.mark.parametrize("kind", ["q4_0", "f16"])
def test_row_independence_gemv(oracle, kind):
    """Rows do not interact.  Q4_0: row m of a 9-row product is bit-identical to row m of
    the same rows taken in two products of 5 and 4 rows (the tensor-core and the dp4a
    block dots); the one-row product of row m splits row groups between CTAs, so its f32
    additions come in another order, and it agrees within the exact-block-dot bound.
    F16: bit-identical for every M."""
    M, N, K = 9, 700, 1536
    w, x = synth.problem(40, M, N, K)
    if kind == "q4_0":
        rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
        full = host(gq.mul_mat_q4_0_f32(rep, dev(x), N, path=gq.GQ_PATH_GEMV))
        split = np.concatenate([host(gq.mul_mat_q4_0_f32(rep, dev(x[:5]), N, path=gq.GQ_PATH_GEMV)),
                                host(gq.mul_mat_q4_0_f32(rep, dev(x[5:]), N, path=gq.GQ_PATH_GEMV))])
        assert np.array_equal(full, split)
        ones = np.concatenate([host(gq.mul_mat_q4_0_f32(rep, dev(x[m:m + 1]), N, path=gq.GQ_PATH_GEMV))
                               for m in range(M)])
        q4_ref = oracle.quantize_q4_0(w)
        bound = exact_dot_bound(oracle, q4_ref, x)
        assert np.all(np.abs(full.astype(np.float64) - ones) <= 2 * bound)
        ref, _ = oracle.mul_mat_q4_0_f32(q4_ref, x)
        assert np.all(np.abs(ones.astype(np.float64) - ref) <= bound)
    else:
        wd = dev(synth.f16_bits(w).view(np.int16))
        full = host(gq.mul_mat_f16_f32(wd, dev(x), path=gq.GQ_PATH_GEMV))
        ones = [host(gq.mul_mat_f16_f32(wd, dev(x[m:m + 1]), path=gq.GQ_PATH_GEMV)) for m in range(M)]
        for m in range(M):
            assert np.array_equal(full[m], ones[m][0]), f"row {m}"


@pytest.mark.parametrize("path", [gq.GQ_PATH_GEMV, gq.GQ_PATH_TC])
def test_sentinels_untouched(path):
    """Outputs are written inside [M][N] only: the padding around dst keeps its sentinel."""
    M, N, K = 5, 131, 256
    w, x = synth.problem(50, M, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    pad = 1024
    buf = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
    dst = buf[pad:pad + M * N]
    gq.gq_mul_mat_q4_0_f32_path(rep, dev(x), dst, M, N, K, path)
    wd = dev(synth.f16_bits(w).view(np.int16))
    buf2 = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
    dst2 = buf2[pad:pad + M * N]
    gq.gq_mul_mat_f16_f32_path(wd, dev(x), dst2, M, N, K, path)
    for b in (host(buf), host(buf2)):
        assert np.isnan(b[:pad]).all() and np.isnan(b[-pad:]).all()
        assert np.isfinite(b[pad:-pad]).all()


# --------------------------------------------------------------------------- full size
FULL_CASES = ([(M, N, K) for (N, K) in synth.DECODE_SHAPES for M in (1, 8, 16)]
              + [(M, N, K) for (N, K) in synth.DECODE_SHAPES[1:] for M in (2, 4, 32)])


@pytest.mark.parametrize("M,N,K", FULL_CASES)
def test_full_size_sampled(oracle, M, N, K):
    """The 7B-shaped decode matrices and the small-batch sweep (M = 2, 4, 32 on the two FFN
    shapes), in the launch configuration the benchmark times (automatic dispatch): all quantized
    bytes exact, 2048 sampled outputs against the oracle."""
    w, x = synth.problem(100 + M, M, N, K)
    q4, dst = run_q4(w, x, gq.GQ_PATH_AUTO)
    q4_ref = oracle.quantize_q4_0(w)
    assert np.array_equal(host(q4), q4_ref)
    rng = np.random.default_rng(M * 7 + N)
    ms = rng.integers(0, M, 2048)
    ns = rng.integers(0, N, 2048)
    ref, T = oracle.mul_mat_q4_0_q8_0_at(q4_ref, oracle.quantize_q8_0(x), ms, ns)
    assert_within(dst[ms, ns], ref, T, what="q4_0 full size")
    wb = synth.f16_bits(w)
    dst16 = host(gq.mul_mat_f16_f32(dev(wb.view(np.int16)), dev(x)))
    ref16, T16 = oracle.mul_mat_f16_f32_at(wb, x, ms, ns)
    assert_within(dst16[ms, ns], ref16, T16, what="f16 full size")


@pytest.mark.parametrize("M,N,K,pinned", [(1, 4096, 4096, True), (5, 300, 1024, False), (40, 77, 352, True),
                                         (16, 500, 11008, True), (1, 11008, 4096, False)])
def test_host_pointer_entry_equals_device_entry(M, N, K, pinned):
    """gq_mul_mat_q4_0_f32_host (src1 and dst in host memory) gives the device entry's
    result bit for bit, with page-locked and with pageable host buffers."""
    w, x = synth.problem(70 + M, M, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    want = host(gq.mul_mat_q4_0_f32(rep, dev(x), N))
    hx = torch.from_numpy(np.ascontiguousarray(x))
    hd = torch.full((M, N), float("nan"))
    if pinned:
        hx, hd = hx.pin_memory(), hd.pin_memory()
    s = torch.cuda.current_stream()
    gq.gq_mul_mat_q4_0_f32_host(rep, hx, hd, M, N, K, s)
    s.synchronize()
    assert np.array_equal(hd.numpy(), want)


def test_host_entry_back_to_back_calls():
    """Three host-entry calls in a row on one stream, with one synchronization at the end: the
    staging of each call's src1 waits for the product before it, and each dst is its own."""
    N, K = 4096, 4096
    w = synth.weights(80, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    xs = [synth.activations(81 + i, 1, K) for i in range(3)]
    wants = [host(gq.mul_mat_q4_0_f32(rep, dev(x), N)) for x in xs]
    hxs = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in xs]
    hds = [torch.full((1, N), float("nan")).pin_memory() for _ in xs]
    s = torch.cuda.current_stream()
    for hx, hd in zip(hxs, hds):
        gq.gq_mul_mat_q4_0_f32_host(rep, hx, hd, 1, N, K, s)
    s.synchronize()
    for hd, want in zip(hds, wants):
        assert np.array_equal(hd.numpy(), want)


def test_concatenated_rows_equal_separate_products(oracle):
    """Q/K/V-like matrices sharing an input: one product over the concatenated
    repacked buffers equals the separate products, bit for bit for several
    activation rows; for one row (whose kernel balances tile ranges over the whole
    product, so the split of row groups between CTAs depends on N) both agree
    with the oracle within the exact-block-dot bound."""
    K = 768
    Ns = (64, 48, 112)
    ws = [synth.weights(60 + i, N, K) for i, N in enumerate(Ns)]
    reps = [gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K) for w, N in zip(ws, Ns)]
    both = gq.concat_rows_q4_0(reps, Ns, K)
    q4_ref = np.concatenate([oracle.quantize_q4_0(w) for w in ws])
    for M in (1, 3, 8, 16, 40):
        xh = synth.activations(70 + M, M, K)
        x = dev(xh)
        whole = host(gq.mul_mat_q4_0_f32(both, x, sum(Ns)))
        parts = np.concatenate([host(gq.mul_mat_q4_0_f32(r, x, N)) for r, N in zip(reps, Ns)], axis=1)
        if M > 1:
            assert np.array_equal(whole, parts), f"M={M}"
        ref, T = oracle.mul_mat_q4_0_f32(q4_ref, xh)
        bound = exact_dot_bound(oracle, q4_ref, xh)
        for got in (whole, parts):
            assert_within(got, ref, T, what=f"concatenated M={M}")
            if M <= gq.gq_get_m_threshold():   # the GEMV: f32 sums of exact block dots
                assert np.all(np.abs(got.astype(np.float64) - ref) <= bound), f"M={M}"


def test_tuned_dispatch_profile(oracle):
    """tune_dispatch benches both families on the device; GQ_PATH_AUTO then follows the
    faster one at every benched M, and its products stay within the tolerance."""
    N, K = 512, 1024
    w, _ = synth.problem(80, 1, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    try:
        prof = gq.tune_dispatch(rep, N, K, Ms=(1, 16, 32, 64), reps=5)
        for M, tg, tt in zip(prof["M"], prof["gemv_us"], prof["tc_us"]):
            assert tg > 0 and tt > 0
            want = gq.GQ_PATH_TC if tt < tg else gq.GQ_PATH_GEMV
            assert gq.gq_choose_path(gq.GQ_KIND_Q4_0, N, K, M) == want
        q4_ref = oracle.quantize_q4_0(w)
        for M in (24, 48):
            _, x = synth.problem(81 + M, M, N, K)
            dst = host(gq.mul_mat_q4_0_f32(rep, dev(x), N))
            ref, T = oracle.mul_mat_q4_0_f32(q4_ref, x)
            assert_within(dst, ref, T, what=f"auto M={M}")
    finally:
        gq.gq_clear_dispatch_profiles()


def test_failed_workspace_growth_keeps_the_current_buffer(oracle):
    """A growth of the stream's workspace whose cudaMalloc fails returns GQ_ERR_NO_MEMORY and
    leaves the current workspace in place: products that fit it still run correctly on it."""
    s = torch.cuda.Stream()
    M, N, K = 9, 300, 4096
    w, x = synth.problem(90, M, N, K)
    rep = gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K)
    gq.gq_reserve_workspace(M, N, K, stream=s)
    with pytest.raises(gq.GQError) as e:
        gq.gq_reserve_workspace(1 << 30, 16, 1024, stream=s)   # 2 TiB of tile-path activations
    assert e.value.status == gq.GQ_ERR_NO_MEMORY
    xd = dev(x)
    out = torch.full((M, N), float("nan"), device="cuda")
    with torch.cuda.stream(s):
        gq.gq_mul_mat_q4_0_f32_path(rep, xd, out, M, N, K, gq.GQ_PATH_GEMV, stream=s)
    s.synchronize()
    q4_ref = oracle.quantize_q4_0(w)
    ref, T = oracle.mul_mat_q4_0_f32(q4_ref, x)
    got = out.cpu().numpy()
    assert_within(got, ref, T, what="after a failed growth")
    assert np.all(np.abs(got.astype(np.float64) - ref) <= exact_dot_bound(oracle, q4_ref, x))


@pytest.mark.parametrize("M", [1, 8])
def test_concatenated_decode_products_full_size(oracle, M):
    """The fused decode products of the 32-layer stack: Q|K|V (three 4096 x 4096 matrices,
    12,288 rows) and gate|up (two 11008 x 4096 matrices, 22,016 rows) as one product over the
    concatenated repacked buffers, 2048 sampled outputs each against the oracle."""
    K = 4096
    for Ns, seed in (((4096, 4096, 4096), 700), ((11008, 11008), 710)):
        ws = [synth.weights(seed + i, N, K) for i, N in enumerate(Ns)]
        reps = [gq.repack_q4_0(gq.quantize_q4_0(dev(w)), N, K) for w, N in zip(ws, Ns)]
        both = gq.concat_rows_q4_0(reps, Ns, K)
        del reps
        Nt = sum(Ns)
        x = synth.activations(seed + 9 + M, M, K)
        dst = host(gq.mul_mat_q4_0_f32(both, dev(x), Nt))
        q4 = np.concatenate([oracle.quantize_q4_0(w) for w in ws])
        rng = np.random.default_rng(seed + M)
        ms, ns = rng.integers(0, M, 2048), rng.integers(0, Nt, 2048)
        ref, T = oracle.mul_mat_q4_0_q8_0_at(q4, oracle.quantize_q8_0(x), ms, ns)
        assert_within(dst[ms, ns], ref, T, what=f"concatenated {Nt} x {K}, M = {M}")
