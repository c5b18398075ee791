"""The INT8 KV cache and the decode attention over it (gq_kv_quantize_i8,
gq_kv_append_i8, gq_attn_decode_i8) against the CPU oracle, through the C ABI
(GPU only).

xFasterTransformer, "2.2 Effective KV cache Optimization": INT8 codes with one
f32 scale per token and head; decode attention widens them to f32.

* Codes and scales are integer or exact decisions taken in f32 on both sides:
  they must be bit-identical.
* The attention output is f32 arithmetic against the oracle's f64.  Bound per
  output element j, with u = 2^-24, S the largest |score| bound of the row
  (oracle's S) and E_j = sum_t p_t |vs_t v_tj| (oracle's E):
    - a score is a dot of D terms: on the FP32 path split over lanes (at most 8
      products and a sum per f32 pair, a tree over the lanes of a token); on the
      tensor cores (D = 128) 8 MMA steps of 16 exact fp16 products each, with the
      query carried as two fp16 terms to within 4u of each element, accumulated in
      f32 (counted at 2u per step, in case the accumulation truncates); then the key
      scale and the softmax scale in base 2: at most 15 roundings of terms bounded by
      S on either path, and 2 more for the subtraction of the maximum;
    - exp2f is within 2 ulp (4u relative);
    - so every exponential, and hence the numerator and the denominator, is off by
      at most (34 S + 4) u relative, and p_t by twice that;
    - the denominator is a sum in f32 of at most T / 128 + 9 sequential roundings;
      the output sums T / 4 tokens per warp at most (each tensor-core step adds 16
      exact products of the two-term weights, again counted at 2u), then the warps,
      the division and, for split ranges, the merge (a few more roundings and one
      exp2f per part).
  Taken together and doubled: |out_j - oracle_j| <= 2 (70 S + T / 2 + 64) u E_j.
"""
import math

import numpy as np
import pytest
import torch

import quantized_skinny_matmul_gb300 as gq
from quantized_skinny_matmul_gb300 import synth
from test_gpu_parity import dev, host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert gq.gq_last_error() == gq.GQ_OK


def edge_rows(seed, rows, D):
    """Rows with a zero row, exact .5 ties (amax 127, so s = 1), tiny and huge magnitudes."""
    gen = np.random.default_rng(seed)
    x = gen.standard_normal((rows, D)).astype(np.float32)
    for r in range(rows):
        kind = r % 5
        if kind == 0:
            x[r] = 0.0
        elif kind == 1:
            c = gen.integers(-126, 126, size=D).astype(np.float32) + np.float32(0.5)
            c[gen.integers(D)] = 127.0
            x[r] = c
        elif kind == 2:
            x[r] *= np.float32(1e-30)
        elif kind == 3:
            x[r] *= np.float32(1e30)
    return x


def attn_tolerance(E, S, T):
    return 2.0 * (70.0 * S[..., None] + T / 2.0 + 64.0) * U * E + 1e-30


def assert_attention(got, want, E, S, T, what=""):
    tol = attn_tolerance(E, S, T)
    err = np.abs(got.astype(np.float64) - want)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} outputs outside the bound; first {bad[:3].tolist()}: "
                           f"got {got[tuple(bad[0])]}, want {want[tuple(bad[0])]}, tol {tol[tuple(bad[0])]}")
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("rows,D", [(1, 64), (7, 128), (130, 64), (1000, 128)])
def test_kv_quantize_is_bit_exact(oracle, rows, D):
    x = edge_rows(rows + D, rows, D)
    q, s = gq.kv_quantize_i8(dev(x))
    want_q, want_s = oracle.kv_quantize_i8(x)
    assert np.array_equal(host(q), want_q)
    assert np.array_equal(host(s).view(np.uint32), want_s.view(np.uint32))


def test_kv_append_writes_one_position_per_sequence(oracle):
    B, Hkv, Tcap, D = 5, 3, 40, 128
    x = edge_rows(3, B * Hkv, D).reshape(B, Hkv, D)
    q = torch.full((B, Hkv, Tcap, D), 7, dtype=torch.int8, device="cuda")
    s = torch.full((B, Hkv, Tcap), 2.5, dtype=torch.float32, device="cuda")
    pos = np.array([0, 39, 17, 40, 5], np.int32)          # 40 == Tcap: out of range
    gq.gq_kv_append_i8(dev(x), q, s, dev(pos), B, Hkv, Tcap, D)
    assert gq.gq_last_error() == gq.GQ_ERR_INVALID_ARG
    assert gq.gq_last_error() == gq.GQ_OK                  # reading it cleared it
    want_q, want_s = oracle.kv_quantize_i8(x)
    hq, hs = host(q), host(s)
    for b in range(B):
        rest = np.ones(Tcap, bool)
        if b != 3:
            assert np.array_equal(hq[b, :, pos[b]], want_q[b])
            assert np.array_equal(hs[b, :, pos[b]], want_s[b])
            rest[pos[b]] = False
        assert np.all(hq[b][:, rest] == 7) and np.all(hs[b][:, rest] == 2.5)


# (B, Hq, Hkv, Tcap, D, lens): ragged and empty sequences, every group size (1 .. 8 for D = 128),
# both head sizes, lengths across several 8 KB slots with a ragged last one, and few (sequence,
# head) pairs with long caches (split over CTAs and merged)
CASES = [
    (2, 8, 8, 300, 128, [300, 77]),
    (3, 8, 2, 513, 64, [513, 0, 1]),
    (1, 32, 4, 5000, 128, [4999]),
    (4, 16, 2, 2048, 128, "mix"),
    (2, 8, 1, 700, 64, [700, 129]),
    (1, 4, 4, 64, 128, [64]),
    (6, 4, 2, 1031, 128, "mix"),
    (1, 8, 8, 40000, 128, [40000]),
    (2, 2, 1, 9000, 64, [1, 9000]),
    (3, 12, 4, 600, 128, [600, 333, 17]),      # G = 3
    (2, 28, 4, 2100, 128, [2100, 1500]),       # G = 7 (28 query heads on 4 KV heads)
    (2, 10, 2, 800, 128, "mix"),               # G = 5
    (1, 24, 4, 3000, 128, [2999]),             # G = 6
]


@pytest.mark.parametrize("B,Hq,Hkv,Tcap,D,lens", CASES)
def test_attention_parity(oracle, B, Hq, Hkv, Tcap, D, lens):
    seed = B * 1000 + Hq * 10 + Hkv + Tcap
    qf, kf, vf = synth.kv_problem(seed, B, Hq, Hkv, Tcap, D)
    lens = synth.kv_lengths(seed, B, Tcap, "mix") if lens == "mix" else np.array(lens, np.int32)
    c = 1.0 / math.sqrt(D)
    k, ks = gq.kv_quantize_i8(dev(kf))
    v, vs = gq.kv_quantize_i8(dev(vf))
    ok, oks = oracle.kv_quantize_i8(kf)
    ov, ovs = oracle.kv_quantize_i8(vf)
    assert np.array_equal(host(k), ok) and np.array_equal(host(ks), oks)
    assert np.array_equal(host(v), ov) and np.array_equal(host(vs), ovs)
    out = gq.attn_decode_i8(dev(qf), k, ks, v, vs, dev(lens), c)
    want, E, S = oracle.attn_decode_i8(qf, ok, oks, ov, ovs, lens, c)
    got = host(out)
    assert_attention(got, want, E, S, int(lens.max()), f"B={B} Hq={Hq} Hkv={Hkv} T={Tcap} D={D}")
    for b in np.nonzero(lens == 0)[0]:
        assert np.all(got[b] == 0)
    again = host(gq.attn_decode_i8(dev(qf), k, ks, v, vs, dev(lens), c))
    assert np.array_equal(again.view(np.uint32), got.view(np.uint32)), "not deterministic"


@pytest.mark.parametrize("B,Hq,Hkv,Tcap,D,lens", [CASES[0], CASES[2], CASES[3], CASES[6]])
def test_attention_parity_fp32_kernel(oracle, monkeypatch, B, Hq, Hkv, Tcap, D, lens):
    """The FP32 kernel, which serves D = 64, forced for D = 128 (GQ_ATTN_FP32), on the same cases."""
    monkeypatch.setenv("GQ_ATTN_FP32", "1")
    test_attention_parity(oracle, B, Hq, Hkv, Tcap, D, lens)


def test_attention_dominant_score_and_zero_scale(oracle):
    """A score far beyond exp's range makes p one-hot (no overflow); a zero softmax scale
    gives the mean of the values."""
    B, Hq, Hkv, Tcap, D = 2, 4, 2, 200, 128
    gen = np.random.default_rng(77)
    k = gen.integers(-127, 128, size=(B, Hkv, Tcap, D)).astype(np.int8)
    v = gen.integers(-127, 128, size=(B, Hkv, Tcap, D)).astype(np.int8)
    ks = np.full((B, Hkv, Tcap), 1.0, np.float32)
    vs = (gen.random((B, Hkv, Tcap)) + 0.5).astype(np.float32) / 127
    k[0] = 0
    k[0, :, 123] = 127
    q = gen.standard_normal((B, Hq, D)).astype(np.float32)
    q[0] = np.abs(q[0]) + 1.0
    lens = np.array([Tcap, Tcap], np.int32)
    for c in (1.0 / math.sqrt(D), 0.0):
        out = host(gq.attn_decode_i8(dev(q), dev(k), dev(ks), dev(v), dev(vs), dev(lens), c))
        want, E, S = oracle.attn_decode_i8(q, k, ks, v, vs, lens, c)
        assert_attention(out, want, E, S, Tcap, f"c={c}")
    out = host(gq.attn_decode_i8(dev(q), dev(k), dev(ks), dev(v), dev(vs), dev(lens), 1.0 / math.sqrt(D)))
    for h in range(Hq):
        assert np.allclose(out[0, h], v[0, h // 2, 123].astype(np.float64) * vs[0, h // 2, 123], rtol=1e-6, atol=0)


def test_attention_length_out_of_range_is_reported(oracle):
    B, Hq, Hkv, Tcap, D = 3, 4, 4, 100, 64
    qf, kf, vf = synth.kv_problem(5, B, Hq, Hkv, Tcap, D)
    k, ks = gq.kv_quantize_i8(dev(kf))
    v, vs = gq.kv_quantize_i8(dev(vf))
    lens = np.array([100, 101, -1], np.int32)
    out = host(gq.attn_decode_i8(dev(qf), k, ks, v, vs, dev(lens), 0.125))
    assert gq.gq_last_error() == gq.GQ_ERR_INVALID_ARG
    assert np.all(out[1:] == 0)
    want, E, S = oracle.attn_decode_i8(qf, host(k), host(ks), host(v), host(vs), np.array([100, 0, 0], np.int32),
                                       0.125)
    assert_attention(out, want, E, S, Tcap)
    assert gq.gq_last_error() == gq.GQ_OK


def sampled_rows(oracle, q, k, ks, v, vs, lens, G, c, picks):
    """Oracle outputs for chosen (b, h) rows of a cache that lives on the device: each pick
    becomes a one-sequence, one-KV-head problem built from slices copied to the host."""
    got, want, E, S, T = [], [], [], [], []
    for b, h in picks:
        hk = h // G
        L = int(lens[b])
        kk = host(k[b, hk, :max(L, 1)])[None, None]
        vv = host(v[b, hk, :max(L, 1)])[None, None]
        kks = host(ks[b, hk, :max(L, 1)])[None, None]
        vvs = host(vs[b, hk, :max(L, 1)])[None, None]
        qq = host(q[b, hk * G:(hk + 1) * G])[None]
        o, e, s = oracle.attn_decode_i8(qq, kk, kks, vv, vvs, np.array([L], np.int32), c)
        want.append(o[0, h - hk * G])
        E.append(e[0, h - hk * G])
        S.append(s[0, h - hk * G])
        T.append(L)
    return np.array(want), np.array(E), np.array(S), max(T)


@pytest.mark.parametrize("lens_mode", ["full", "mix"])
def test_attention_full_size_sampled(oracle, lens_mode):
    """The Llama2-7B decode layer of the KV-cache page (batch 256, 32 heads of 128,
    1024 + 1024 tokens), in the launch configuration the benchmark times: sampled rows
    against the oracle, and bitwise repeatability."""
    cfg = synth.KV_LLAMA2_7B
    B, Hq, Hkv, Tcap, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["Tcap"], cfg["D"]
    k, ks, v, vs = synth.kv_codes_device(11, B, Hkv, Tcap, D, "cuda")
    gen = np.random.default_rng(12)
    q = dev(gen.standard_normal((B, Hq, D)).astype(np.float32))
    lens = synth.kv_lengths(13, B, Tcap, lens_mode)
    c = 1.0 / math.sqrt(D)
    out = gq.attn_decode_i8(q, k, ks, v, vs, dev(lens), c)
    again = gq.attn_decode_i8(q, k, ks, v, vs, dev(lens), c)
    assert torch.equal(out.view(torch.int32), again.view(torch.int32))
    picks = [(0, 0), (B - 1, Hq - 1), (17, 5), (128, 31)] + [
        (int(gen.integers(B)), int(gen.integers(Hq))) for _ in range(20)]
    want, E, S, T = sampled_rows(oracle, q, k, ks, v, vs, lens, Hq // Hkv, c, picks)
    got = np.stack([host(out[b, h]) for b, h in picks])
    assert_attention(got, want, E, S, T, f"full size, lens {lens_mode}")


def test_attention_shares_the_stream_workspace(oracle):
    """A split sequence keeps its parts in the stream's workspace, which the products use
    too: attention launches interleaved with Q4_0 products on one stream, and replays of a
    captured attention launch, give the same bits every time."""
    B, Hq, Hkv, Tcap, D = 8, 32, 8, 3000, 128
    qf, kf, vf = synth.kv_problem(21, B, Hq, Hkv, Tcap, D)
    lens = synth.kv_lengths(21, B, Tcap, "mix")
    c = 1.0 / math.sqrt(D)
    gen = np.random.default_rng(22)
    N, K, M = 4096, 11008, 2
    w = dev(gen.standard_normal((N, K)).astype(np.float32))
    x = dev(gen.standard_normal((M, K)).astype(np.float32))
    rp = gq.repack_q4_0(gq.quantize_q4_0(w), N, K)
    y_ref = gq.mul_mat_q4_0_f32(rp, x, N)   # on the default stream: its own workspace
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q, L = dev(qf), dev(lens)
        k, ks = gq.kv_quantize_i8(dev(kf))
        v, vs = gq.kv_quantize_i8(dev(vf))
        ref = gq.attn_decode_i8(q, k, ks, v, vs, L, c)
        for _ in range(3):
            y = gq.mul_mat_q4_0_f32(rp, x, N)
            got = gq.attn_decode_i8(q, k, ks, v, vs, L, c)
            assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
            assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
        out = torch.zeros_like(ref)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            gq.attn_decode_i8(q, k, ks, v, vs, L, c, out=out)
        for _ in range(3):
            out.zero_()
            g.replay()
            assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    s.synchronize()
    want, E, S = oracle.attn_decode_i8(qf, host(k), host(ks), host(v), host(vs), lens, c)
    assert_attention(host(ref), want, E, S, int(lens.max()))
