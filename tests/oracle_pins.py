"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Every function takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  ``test_oracle_pins.py`` runs them on the oracle as built; the
mutation test runs them on copies of the oracle with a mistake planted in the
C source and requires that at least one of them fails for every mistake.

What pins what:
  * binary16 conversion        -> numpy's IEEE float16 conversion (library routine)
  * the block byte layouts      -> the hand-derived worked examples in golden/
  * the quantizer's arithmetic  -> exact round trips of representable blocks, the
                                   range and de-quantization error bounds
  * the integer block dots      -> brute force over every (q4, q8) pair per lane, and
                                   every Q8_0 weight code against a spread of codes
  * the f64 products            -> float64 dense matmul of the de-quantized
                                   operands (textbook special case), structured
                                   weights with closed-form results, and the
                                   row independence of the batched product
  * the INT8 KV quantizer       -> worked examples in golden/, exact round trips of
                                   representable rows, the de-quantization bound
  * the decode attention        -> textbook attention on the de-quantized cache (numpy
                                   matmul and scipy's softmax), and special cases with
                                   closed forms: one token, equal keys, a zero softmax
                                   scale, an empty sequence, a dominant score far beyond
                                   exp's range, tokens past the length, a permutation
"""
from __future__ import annotations

import os

import numpy as np

from quantized_skinny_matmul_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "worked_examples.txt")


# ---------------------------------------------------------------------------
# helpers that decode the documented byte layout independently of the oracle
# ---------------------------------------------------------------------------
def decode_q4_0(q4: np.ndarray):
    """(codes uint8 [..., 32], fp16 scale as f64 [...]) from canonical Q4_0 bytes."""
    d = q4[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qs = q4[..., 2:18]
    codes = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)
    return codes, d


def decode_q4_1(q41: np.ndarray):
    """(codes uint8 [..., 32], fp16 d as f64 [...], fp16 m as f64 [...]) from Q4_1 bytes."""
    d = q41[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    m = q41[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    qs = q41[..., 4:20]
    return np.concatenate([qs & 0x0F, qs >> 4], axis=-1), d, m


def decode_q5_0(q5: np.ndarray):
    """(codes uint8 [..., 32] in 0..31, fp16 scale as f64 [...]) from Q5_0 bytes."""
    d = q5[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qh = q5[..., 2:6].copy().view(np.uint32)[..., 0]
    qs = q5[..., 6:22]
    lo = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)
    hi = (qh[..., None] >> np.arange(32, dtype=np.uint32)) & 1
    return (lo | (hi << 4)).astype(np.uint8), d


def decode_q8_0(q8: np.ndarray):
    d = q8[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    codes = q8[..., 2:34].view(np.int8)
    return codes, d


def round_half_away(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, np.float64)
    return np.trunc(v + np.copysign(0.5, v))


def parse_golden(path: str = GOLDEN):
    cases = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, expr, hexbytes = (s.strip() for s in line.split("|"))
            name, kind = head.split()
            j = np.arange(32)
            env = {"j": j}
            if expr.startswith("["):
                x = np.array(eval(expr, {}, env), dtype=np.float64)  # closed-form list
            else:
                x = np.broadcast_to(np.asarray(eval(expr, {}, env), np.float64), (32,))
            cases.append((name, kind, x.astype(np.float32),
                          bytes.fromhex(hexbytes.replace(" ", ""))))
    return cases


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------
def pin_f16_conversion(o) -> None:
    rng = np.random.default_rng(11)
    vals = [rng.standard_normal(4000).astype(np.float32) * np.float32(s)
            for s in (1e-8, 1e-6, 3e-5, 1e-3, 1.0, 1e3, 6e4)]
    # exact binary16 values, the half-way points between neighbours, and one
    # f32 ulp either side of those half-way points
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    f = h.view(np.float16).astype(np.float64)
    mids = ((f[:-1] + f[1:]) / 2).astype(np.float32)
    vals += [f.astype(np.float32), mids, np.nextafter(mids, np.float32(np.inf)),
             np.nextafter(mids, np.float32(0))]
    vals += [np.array([0.0, 65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -24,
                       1.5 * 2.0 ** -25, 2.0 ** -26, 1e-30], np.float32)]
    x = np.concatenate(vals)
    x = np.concatenate([x, -x])
    got = o.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"f32->f16 mismatch at {x[bad[:5]]}: {got[bad[:5]]} vs {want[bad[:5]]}"
    # every non-NaN binary16 pattern back to f32
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite_or_inf = (allh & 0x7C00) != 0x7C00
    finite_or_inf |= (allh & 0x03FF) == 0
    allh = allh[finite_or_inf]
    back = o.f16_bits_to_f32(allh)
    want_back = allh.view(np.float16).astype(np.float32)
    assert np.array_equal(back.view(np.uint32), want_back.view(np.uint32)), "f16->f32 mismatch"


def pin_worked_examples(o) -> None:
    for name, kind, x, want in parse_golden():
        if kind == "q4_0":
            got = o.quantize_q4_0(x.reshape(1, 32)).tobytes()
        elif kind == "q5_0":
            got = o.quantize_q5_0(x.reshape(1, 32)).tobytes()
        elif kind == "q4_1":
            got = o.quantize_q4_1(x.reshape(1, 32)).tobytes()
        elif kind == "kv_i8":
            codes, scale = o.kv_quantize_i8(x.reshape(1, 32))
            got = scale.astype("<f4").tobytes() + codes.tobytes()
        else:
            got = o.quantize_q8_0(x.reshape(1, 32)).tobytes()
        assert got == want, f"{name}: {got.hex(' ')} != {want.hex(' ')}"
    # the worked example W1 de-quantizes back to its input exactly
    x = ((np.arange(32) % 16) - 8).astype(np.float32).reshape(1, 32)
    assert np.array_equal(o.dequantize_q4_0(o.quantize_q4_0(x)), x.astype(np.float64))


def pin_roundtrip_q4_0(o) -> None:
    """Blocks whose values are codes times a power of two with a -8 code present
    quantize to exactly those codes and that scale."""
    rng = np.random.default_rng(5)
    N, nb = 64, 8
    c = rng.integers(-8, 8, size=(N, nb, 32))
    c[:, :, 0] = -8                                   # the signed max: d = scale
    e = rng.integers(-12, 4, size=(N, nb, 1))
    x = (c * np.exp2(e)).astype(np.float32).reshape(N, nb * 32)
    codes, d = decode_q4_0(o.quantize_q4_0(x))
    assert np.array_equal(codes.astype(np.int64) - 8, c)
    assert np.array_equal(d, np.exp2(e[..., 0]).astype(np.float64))
    # a positive signed max flips the sign of d and every code
    codes, d = decode_q4_0(o.quantize_q4_0(-x))
    assert np.array_equal(d, -np.exp2(e[..., 0]).astype(np.float64))
    assert np.array_equal(codes.astype(np.int64) - 8, c)


def pin_roundtrip_q8_0(o) -> None:
    rng = np.random.default_rng(6)
    M, nb = 16, 8
    c = rng.integers(-127, 128, size=(M, nb, 32))
    c[:, :, 3] = 127 * np.where(rng.random((M, nb)) < 0.5, 1, -1)
    e = rng.integers(-12, 4, size=(M, nb, 1))
    x = (c * np.exp2(e)).astype(np.float32).reshape(M, nb * 32)
    codes, d = decode_q8_0(o.quantize_q8_0(x))
    assert np.array_equal(codes.astype(np.int64), c)
    assert np.array_equal(d, np.exp2(e[..., 0]).astype(np.float64))


def pin_ranges_and_error_bounds(o) -> None:
    w = synth.edge_weights(21, 48, 512)
    x = synth.edge_activations(22, 24, 512)
    codes4, d4 = decode_q4_0(o.quantize_q4_0(w))
    codes8, d8 = decode_q8_0(o.quantize_q8_0(x))
    assert codes4.min() >= 0 and codes4.max() <= 15
    assert codes8.min() >= -127 and codes8.max() <= 127
    wb = w.reshape(codes4.shape).astype(np.float64)
    xb = x.reshape(codes8.shape).astype(np.float64)
    # the f32 scales the quantizers divide by, recomputed from the inputs
    am4 = np.abs(wb).max(-1)
    first = np.argmax(np.abs(wb) == am4[..., None], axis=-1)
    vmax = np.take_along_axis(wb, first[..., None], -1)[..., 0]
    dq4 = (vmax.astype(np.float32) / np.float32(-8.0)).astype(np.float64)
    dq8 = np.abs(xb).max(-1).astype(np.float32) / np.float32(127.0)
    dq8 = dq8.astype(np.float64)
    assert np.array_equal(d4, dq4.astype(np.float16).astype(np.float64))
    assert np.array_equal(d8, dq8.astype(np.float16).astype(np.float64))
    slack = 1.0 + 1e-6
    err4 = np.abs(wb - (codes4.astype(np.float64) - 8) * d4[..., None])
    with np.errstate(divide="ignore", invalid="ignore"):
        clamp = np.abs(wb / dq4[..., None]) > 7.5
    bound4 = np.where(clamp, np.abs(dq4)[..., None], np.abs(dq4)[..., None] / 2) * slack \
        + 8 * np.abs(dq4 - d4)[..., None]
    assert np.all(err4 <= bound4 + 1e-30), "Q4_0 de-quantization error above its bound"
    err8 = np.abs(xb - codes8.astype(np.float64) * d8[..., None])
    bound8 = np.abs(dq8)[..., None] / 2 * slack + 127 * np.abs(dq8 - d8)[..., None]
    assert np.all(err8 <= bound8 + 1e-30), "Q8_0 de-quantization error above its bound"
    # zero blocks are zero scales with neutral codes
    z4 = np.all(wb == 0, axis=-1)
    assert np.all(d4[z4] == 0) and np.all(codes4[z4] == 8)
    z8 = np.all(xb == 0, axis=-1)
    assert np.all(d8[z8] == 0) and np.all(codes8[z8] == 0)


def _q4_block(codes, d16_bits=0x3C00) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    out = np.empty(18, np.uint8)
    out[0], out[1] = d16_bits & 0xFF, d16_bits >> 8
    out[2:] = codes[:16] | (codes[16:] << 4)
    return out


def _q8_block(codes, d16_bits=0x3C00) -> np.ndarray:
    out = np.empty(34, np.uint8)
    out[0], out[1] = d16_bits & 0xFF, d16_bits >> 8
    out[2:] = np.asarray(codes, np.int8).view(np.uint8)
    return out


def pin_block_dot_bruteforce(o) -> None:
    """One lane at a time: sumi = (q4 - 8) * q8 for every q4 in 0..15 and q8 in -127..127."""
    q4v = np.arange(16)
    q8v = np.arange(-127, 128)
    for lane in (0, 5, 15, 16, 22, 31):
        blocks4 = []
        for a in q4v:
            c = np.full(32, 8)
            c[lane] = a
            blocks4.append(_q4_block(c))
        blocks8 = []
        for b in q8v:
            c = np.zeros(32, np.int64)
            c[lane] = b
            blocks8.append(_q8_block(c))
        q4 = np.stack(blocks4)[:, None, :]
        q8 = np.stack(blocks8)[:, None, :]
        got = o.block_dots(q4, q8)[:, :, 0]                 # [q8 index, q4 index]
        want = np.outer(q8v, q4v - 8)
        assert np.array_equal(got, want), f"block dot wrong at lane {lane}"
    # the extreme block: every q4 = 0 and every q8 = -127 gives 32 * 8 * 127
    got = o.block_dots(_q4_block(np.zeros(32))[None, None], _q8_block(np.full(32, -127))[None, None])
    assert int(got[0, 0, 0]) == 32512


def pin_block_dot_random(o) -> None:
    rng = np.random.default_rng(7)
    N, M, nb = 24, 5, 6
    c4 = rng.integers(0, 16, size=(N, nb, 32))
    c8 = rng.integers(-127, 128, size=(M, nb, 32))
    q4 = np.stack([np.stack([_q4_block(c4[n, b]) for b in range(nb)]) for n in range(N)])
    q8 = np.stack([np.stack([_q8_block(c8[m, b]) for b in range(nb)]) for m in range(M)])
    got = o.block_dots(q4, q8)
    want = np.einsum("nbj,mbj->mnb", c4.astype(np.int64) - 8, c8.astype(np.int64))
    assert np.array_equal(got, want)


def pin_matmul_vs_dense(o) -> None:
    """The f64 product equals float64 dequant(src0) @ dequant(wdata)^T to 1e-12 of T."""
    for (M, N, K, seed, outl) in ((3, 40, 96, 1, False), (7, 33, 256, 2, True), (1, 17, 32, 3, False)):
        w, x = synth.problem(seed, M, N, K, outliers=outl)
        q4 = o.quantize_q4_0(w)
        q8 = o.quantize_q8_0(x)
        c4, d4 = decode_q4_0(q4)
        c8, d8 = decode_q8_0(q8)
        A = ((c4.astype(np.float64) - 8) * d4[..., None]).reshape(N, K)
        B = (c8.astype(np.float64) * d8[..., None]).reshape(M, K)
        want = B @ A.T
        T_want = np.abs(B) @ np.abs(A).T
        dst, T = o.mul_mat_q4_0_f32(q4, x)
        assert np.all(np.abs(dst - want) <= 1e-12 * T_want + 1e-300), "Q4_0 product mismatch"
        assert np.allclose(T, T_want, rtol=1e-12, atol=0)
        ms = np.array([0, M - 1, M // 2])
        ns = np.array([N - 1, 0, N // 2])
        at, T_at = o.mul_mat_q4_0_q8_0_at(q4, q8, ms, ns)
        assert np.array_equal(at, dst[ms, ns]) and np.array_equal(T_at, T[ms, ns])


def pin_row_independence(o) -> None:
    """Row m of an M-row product equals the product of row m alone (bit for bit)."""
    M, N, K = 6, 20, 160
    w, x = synth.problem(9, M, N, K)
    q4 = o.quantize_q4_0(w)
    dst, _ = o.mul_mat_q4_0_f32(q4, x)
    for m in range(M):
        one, _ = o.mul_mat_q4_0_f32(q4, x[m:m + 1])
        assert np.array_equal(one[0], dst[m])
    dst2, _ = o.mul_mat_f16_f32(synth.f16_bits(w), x)
    for m in range(M):
        one, _ = o.mul_mat_f16_f32(synth.f16_bits(w), x[m:m + 1])
        assert np.array_equal(one[0], dst2[m])


def pin_f16_matmul(o) -> None:
    """F16 kind: selection weights give columns of src1 exactly; dense agreement."""
    rng = np.random.default_rng(13)
    M, N, K = 5, 37, 64
    x = rng.standard_normal((M, K)).astype(np.float32)
    perm = rng.integers(0, K, size=N)
    sel = np.zeros((N, K), np.float32)
    sel[np.arange(N), perm] = 1.0
    sel[::3, :] *= 2.0                      # powers of two stay exact
    dst, T = o.mul_mat_f16_f32(synth.f16_bits(sel), x)
    want = x[:, perm].astype(np.float64) * np.where(np.arange(N) % 3 == 0, 2.0, 1.0)
    assert np.array_equal(dst, want)
    w, x = synth.problem(14, 4, 29, 96)
    wb = synth.f16_bits(w)
    dst, T = o.mul_mat_f16_f32(wb, x)
    W = wb.view(np.float16).astype(np.float64)
    X = x.astype(np.float64)
    assert np.all(np.abs(dst - X @ W.T) <= 1e-12 * (np.abs(X) @ np.abs(W).T))
    assert np.allclose(T, np.abs(X) @ np.abs(W).T, rtol=1e-12, atol=0)
    ms, ns = np.array([3, 0, 2]), np.array([0, 28, 11])
    at, _ = o.mul_mat_f16_f32_at(wb, x, ms, ns)
    assert np.array_equal(at, dst[ms, ns])


def _q5_block(codes, d16_bits=0x3C00) -> np.ndarray:
    codes = np.asarray(codes, np.int64)
    out = np.empty(22, np.uint8)
    out[0], out[1] = d16_bits & 0xFF, d16_bits >> 8
    qh = int(sum(((int(c) >> 4) & 1) << j for j, c in enumerate(codes)))
    out[2:6] = np.frombuffer(qh.to_bytes(4, "little"), np.uint8)
    out[6:] = ((codes[:16] & 0x0F) | ((codes[16:] & 0x0F) << 4)).astype(np.uint8)
    return out


def pin_q5_0_quantizer(o) -> None:
    """Q5_0: exact round trips of codes times a power of two (a -16 code present) and of their
    negation; codes in 0..31; de-quantization error within |d|/2 (|d| where clamped);
    zero blocks are a zero scale with code 16."""
    rng = np.random.default_rng(25)
    N, nb = 48, 8
    c = rng.integers(-16, 16, size=(N, nb, 32))
    c[:, :, 3] = -16
    e = rng.integers(-12, 4, size=(N, nb, 1))
    x = (c * np.exp2(e)).astype(np.float32).reshape(N, nb * 32)
    codes, d = decode_q5_0(o.quantize_q5_0(x))
    assert np.array_equal(codes.astype(np.int64) - 16, c)
    assert np.array_equal(d, np.exp2(e[..., 0]).astype(np.float64))
    codes, d = decode_q5_0(o.quantize_q5_0(-x))
    assert np.array_equal(d, -np.exp2(e[..., 0]).astype(np.float64))
    assert np.array_equal(codes.astype(np.int64) - 16, c)
    assert np.array_equal(o.dequantize_q5_0(o.quantize_q5_0(x)), x.astype(np.float64))
    w = synth.edge_weights(26, 40, 512)
    codes, d5 = decode_q5_0(o.quantize_q5_0(w))
    assert codes.min() >= 0 and codes.max() <= 31
    wb = w.reshape(codes.shape).astype(np.float64)
    am = np.abs(wb).max(-1)
    first = np.argmax(np.abs(wb) == am[..., None], axis=-1)
    vmax = np.take_along_axis(wb, first[..., None], -1)[..., 0]
    dq = (vmax.astype(np.float32) / np.float32(-16.0)).astype(np.float64)
    assert np.array_equal(d5, dq.astype(np.float16).astype(np.float64))
    err = np.abs(wb - (codes.astype(np.float64) - 16) * d5[..., None])
    with np.errstate(divide="ignore", invalid="ignore"):
        clamp = np.abs(wb / dq[..., None]) > 15.5
    bound = np.where(clamp, np.abs(dq)[..., None], np.abs(dq)[..., None] / 2) * (1 + 1e-6) \
        + 16 * np.abs(dq - d5)[..., None]
    assert np.all(err <= bound + 1e-30), "Q5_0 de-quantization error above its bound"
    z = np.all(wb == 0, axis=-1)
    assert np.all(d5[z] == 0) and np.all(codes[z] == 16)


def pin_q5_0_block_dot_and_product(o) -> None:
    """Q5_0: block dots by brute force for every code against every Q8_0 code in a few lanes;
    the product against the float64 dense matmul of the de-quantized operands; row independence."""
    q5v = np.arange(32)
    q8v = np.arange(-127, 128)
    for lane in (0, 4, 15, 16, 20, 31):
        b5 = []
        for a in q5v:
            c = np.full(32, 16)
            c[lane] = a
            b5.append(_q5_block(c))
        b8 = []
        for b in q8v:
            c = np.zeros(32, np.int64)
            c[lane] = b
            b8.append(_q8_block(c))
        got = o.block_dots_q5_0(np.stack(b5)[:, None, :], np.stack(b8)[:, None, :])[:, :, 0]
        assert np.array_equal(got, np.outer(q8v, q5v - 16)), f"Q5_0 block dot wrong at lane {lane}"
    got = o.block_dots_q5_0(_q5_block(np.zeros(32))[None, None], _q8_block(np.full(32, -127))[None, None])
    assert int(got[0, 0, 0]) == 65024
    for (M, N, K, seed, outl) in ((3, 40, 96, 31, False), (5, 33, 256, 32, True), (1, 17, 32, 33, False)):
        w, x = synth.problem(seed, M, N, K, outliers=outl)
        q5 = o.quantize_q5_0(w)
        q8 = o.quantize_q8_0(x)
        A = o.dequantize_q5_0(q5)
        B = o.dequantize_q8_0(q8)
        c5, d5 = decode_q5_0(q5)
        assert np.array_equal(A, ((c5.astype(np.float64) - 16) * d5[..., None]).reshape(N, K))
        want, T_want = B @ A.T, np.abs(B) @ np.abs(A).T
        dst, T = o.mul_mat_q5_0_f32(q5, x)
        assert np.all(np.abs(dst - want) <= 1e-12 * T_want + 1e-300), "Q5_0 product mismatch"
        assert np.allclose(T, T_want, rtol=1e-12, atol=0)
        ms, ns = np.array([0, M - 1, M // 2]), np.array([N - 1, 0, N // 2])
        at, T_at = o.mul_mat_q5_0_q8_0_at(q5, q8, ms, ns)
        assert np.array_equal(at, dst[ms, ns]) and np.array_equal(T_at, T[ms, ns])
        for m in range(M):
            one, _ = o.mul_mat_q5_0_f32(q5, x[m:m + 1])
            assert np.array_equal(one[0], dst[m])


def _q41_block(codes, d16_bits=0x3C00, m16_bits=0x0000) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    out = np.empty(20, np.uint8)
    out[0], out[1] = d16_bits & 0xFF, d16_bits >> 8
    out[2], out[3] = m16_bits & 0xFF, m16_bits >> 8
    out[4:] = codes[:16] | (codes[16:] << 4)
    return out


def pin_q4_1_quantizer(o) -> None:
    """Q4_1: exact round trips of lo + code * 2^e with codes 0 and 15 present; codes in 0..15;
    the scale and minimum are fp16 of (max - min) / 15 and of min; de-quantization error within
    d/2 plus the fp16 roundings; constant blocks are code 0 with m = the value."""
    rng = np.random.default_rng(27)
    N, nb = 48, 8
    c = rng.integers(0, 16, size=(N, nb, 32))
    c[:, :, 5], c[:, :, 9] = 0, 15
    e = rng.integers(-10, 2, size=(N, nb, 1))
    lo = rng.integers(-40, 40, size=(N, nb, 1))
    x = ((lo + c) * np.exp2(e)).astype(np.float32).reshape(N, nb * 32)
    codes, d, m = decode_q4_1(o.quantize_q4_1(x))
    assert np.array_equal(codes.astype(np.int64), c)
    assert np.array_equal(d, np.exp2(e[..., 0]).astype(np.float64))
    assert np.array_equal(m, (lo * np.exp2(e))[..., 0].astype(np.float64))
    assert np.array_equal(o.dequantize_q4_1(o.quantize_q4_1(x)), x.astype(np.float64))
    w = synth.edge_weights(28, 40, 512)
    codes, d, m = decode_q4_1(o.quantize_q4_1(w))
    assert codes.min() >= 0 and codes.max() <= 15
    wb = w.reshape(codes.shape).astype(np.float64)
    lo32, hi32 = wb.min(-1).astype(np.float32), wb.max(-1).astype(np.float32)
    d32 = ((hi32 - lo32) / np.float32(15.0)).astype(np.float64)
    assert np.array_equal(d, d32.astype(np.float16).astype(np.float64))
    assert np.array_equal(m, lo32.astype(np.float16).astype(np.float64))
    err = np.abs(wb - (codes.astype(np.float64) * d[..., None] + m[..., None]))
    bound = (d32 / 2 * (1 + 1e-6) + 15 * np.abs(d32 - d) + np.abs(lo32.astype(np.float64) - m))[..., None] \
        + 1e-6 * np.abs(wb)
    assert np.all(err <= bound + 1e-30), "Q4_1 de-quantization error above its bound"
    const = np.all(wb == wb[..., :1], axis=-1)
    assert np.all(codes[const] == 0) and np.all(d[const] == 0)


def pin_q4_1_block_sums_and_product(o) -> None:
    """Q4_1: (sum q q8, sum q8) by brute force for every code against every Q8_0 code in a few
    lanes; the product against the float64 dense matmul of the de-quantized operands; rows."""
    qv = np.arange(16)
    q8v = np.arange(-127, 128)
    for lane in (0, 7, 16, 31):
        b41 = []
        for a in qv:
            cc = np.zeros(32, np.int64)
            cc[lane] = a
            b41.append(_q41_block(cc))
        b8 = []
        for b in q8v:
            cc = np.zeros(32, np.int64)
            cc[lane] = b
            b8.append(_q8_block(cc))
        got = o.block_sums_q4_1(np.stack(b41)[:, None, :], np.stack(b8)[:, None, :])[:, :, 0, :]
        assert np.array_equal(got[..., 0], np.outer(q8v, qv)), f"Q4_1 block dot wrong at lane {lane}"
        assert np.array_equal(got[..., 1], np.repeat(q8v[:, None], 16, axis=1))
    for (M, N, K, seed, outl) in ((3, 40, 96, 35, False), (5, 33, 256, 36, True), (1, 17, 32, 37, False)):
        w, x = synth.problem(seed, M, N, K, outliers=outl)
        q41 = o.quantize_q4_1(w)
        q8 = o.quantize_q8_0(x)
        A = o.dequantize_q4_1(q41)
        c, d, m = decode_q4_1(q41)
        assert np.array_equal(A, (c.astype(np.float64) * d[..., None] + m[..., None]).reshape(N, K))
        B = o.dequantize_q8_0(q8)
        want, T_want = B @ A.T, np.abs(B) @ np.abs(A).T
        dst, T = o.mul_mat_q4_1_f32(q41, x)
        assert np.all(np.abs(dst - want) <= 1e-12 * T_want + 1e-300), "Q4_1 product mismatch"
        assert np.allclose(T, T_want, rtol=1e-12, atol=0)
        ms, ns = np.array([0, M - 1, M // 2]), np.array([N - 1, 0, N // 2])
        at, T_at = o.mul_mat_q4_1_q8_0_at(q41, q8, ms, ns)
        assert np.array_equal(at, dst[ms, ns]) and np.array_equal(T_at, T[ms, ns])
        for mm in range(M):
            one, _ = o.mul_mat_q4_1_f32(q41, x[mm:mm + 1])
            assert np.array_equal(one[0], dst[mm])


def pin_q8_0_block_dot_bruteforce(o) -> None:
    """Q8_0 weights, one lane at a time: sumi = qw * qx for every qw in -127..127 against a
    spread of qx; the extreme block (all 127 against all -127) gives -32 * 127 * 127."""
    qwv = np.arange(-127, 128)
    qxv = np.array([-127, -64, -3, -1, 0, 1, 2, 77, 127])
    for lane in (0, 9, 16, 31):
        bw = []
        for a in qwv:
            c = np.zeros(32, np.int64)
            c[lane] = a
            bw.append(_q8_block(c))
        bx = []
        for b in qxv:
            c = np.zeros(32, np.int64)
            c[lane] = b
            bx.append(_q8_block(c))
        got = o.block_dots_q8_0(np.stack(bw)[:, None, :], np.stack(bx)[:, None, :])[:, :, 0]
        assert np.array_equal(got, np.outer(qxv, qwv)), f"Q8_0 block dot wrong at lane {lane}"
    got = o.block_dots_q8_0(_q8_block(np.full(32, 127))[None, None], _q8_block(np.full(32, -127))[None, None])
    assert int(got[0, 0, 0]) == -516128


def pin_q8_0_matmul_vs_dense(o) -> None:
    """Q8_0 weights: the f64 product equals float64 dequant(src0) @ dequant(wdata)^T to 1e-12
    of T; random integer blocks give the integer block dots exactly; rows are independent."""
    rng = np.random.default_rng(17)
    N, M, nb = 11, 4, 5
    cw = rng.integers(-127, 128, size=(N, nb, 32))
    cx = rng.integers(-127, 128, size=(M, nb, 32))
    qw = np.stack([np.stack([_q8_block(cw[n, b]) for b in range(nb)]) for n in range(N)])
    qx = np.stack([np.stack([_q8_block(cx[m, b]) for b in range(nb)]) for m in range(M)])
    assert np.array_equal(o.block_dots_q8_0(qw, qx),
                          np.einsum("nbj,mbj->mnb", cw.astype(np.int64), cx.astype(np.int64)))
    for (M, N, K, seed, outl) in ((3, 40, 96, 21, False), (6, 33, 256, 22, True), (1, 17, 32, 23, False)):
        w, x = synth.problem(seed, M, N, K, outliers=outl)
        qw = o.quantize_q8_0(w)                       # the weights in the Q8_0 block format
        qx = o.quantize_q8_0(x)
        cw_, dw = decode_q8_0(qw)
        cx_, dx = decode_q8_0(qx)
        A = (cw_.astype(np.float64) * dw[..., None]).reshape(N, K)
        B = (cx_.astype(np.float64) * dx[..., None]).reshape(M, K)
        want, T_want = B @ A.T, np.abs(B) @ np.abs(A).T
        dst, T = o.mul_mat_q8_0_f32(qw, x)
        assert np.all(np.abs(dst - want) <= 1e-12 * T_want + 1e-300), "Q8_0 product mismatch"
        assert np.allclose(T, T_want, rtol=1e-12, atol=0)
        ms, ns = np.array([0, M - 1, M // 2]), np.array([N - 1, 0, N // 2])
        at, T_at = o.mul_mat_q8_0_q8_0_at(qw, qx, ms, ns)
        assert np.array_equal(at, dst[ms, ns]) and np.array_equal(T_at, T[ms, ns])
        for m in range(M):
            one, _ = o.mul_mat_q8_0_f32(qw, x[m:m + 1])
            assert np.array_equal(one[0], dst[m])


# ---------------------------------------------------------------------------
# INT8 KV cache (xFasterTransformer, "2.2 Effective KV cache Optimization")
# ---------------------------------------------------------------------------
def pin_kv_quantizer(o) -> None:
    rng = np.random.default_rng(31)
    # rows c * 2^e with a +-127 code present quantize to exactly c with scale 2^e
    R, D = 96, 128
    c = rng.integers(-127, 128, size=(R, D))
    c[np.arange(R), rng.integers(D, size=R)] = 127 * np.where(rng.random(R) < 0.5, 1, -1)
    e = rng.integers(-20, 6, size=(R, 1))
    x = (c * np.exp2(e)).astype(np.float32)
    codes, scale = o.kv_quantize_i8(x)
    assert np.array_equal(codes.astype(np.int64), c)
    assert np.array_equal(scale.astype(np.float64), np.exp2(e[:, 0]).astype(np.float64))
    # Gaussian rows with a wide spread of magnitudes: range, the f32 scale recomputed
    # from its definition, and the round-to-nearest error bound
    x = rng.standard_normal((R, D)).astype(np.float32) * np.exp2(rng.integers(-30, 30, size=(R, 1))).astype(np.float32)
    x[0] = 0.0
    codes, scale = o.kv_quantize_i8(x)
    assert codes.min() >= -127 and codes.max() <= 127
    want_s = np.abs(x).max(-1) / np.float32(127.0)
    assert np.array_equal(scale, want_s)
    xd = x.astype(np.float64)
    err = np.abs(xd - codes.astype(np.float64) * scale[:, None].astype(np.float64))
    assert np.all(err <= scale[:, None].astype(np.float64) * (0.5 + 1e-6)), "INT8 KV bound"
    amax_at = np.argmax(np.abs(x), axis=-1)
    assert np.all(np.abs(codes[np.arange(1, R), amax_at[1:]]) == 127)
    assert scale[0] == 0 and np.all(codes[0] == 0)
    deq = o.kv_dequantize_i8(codes, scale)
    assert np.array_equal(deq, codes.astype(np.float64) * scale[:, None].astype(np.float64))


def _kv_case(rng, B, Hkv, Tcap, D, key_scale=1.0):
    k = rng.integers(-127, 128, size=(B, Hkv, Tcap, D)).astype(np.int8)
    v = rng.integers(-127, 128, size=(B, Hkv, Tcap, D)).astype(np.int8)
    ks = (np.exp(rng.standard_normal((B, Hkv, Tcap)) * 0.3) * key_scale / 127).astype(np.float32)
    vs = (np.exp(rng.standard_normal((B, Hkv, Tcap)) * 0.3) / 127).astype(np.float32)
    return k, ks, v, vs


def _textbook_attention(q, k, ks, v, vs, lens, c):
    """Scaled dot-product attention of each query row over the de-quantized cache."""
    from scipy.special import softmax
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    Kd = k.astype(np.float64) * ks[..., None].astype(np.float64)
    Vd = v.astype(np.float64) * vs[..., None].astype(np.float64)
    out = np.zeros((B, Hq, D))
    E = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for h in range(Hq):
            kv = h // G
            p = softmax(c * (Kd[b, kv, :L] @ q[b, h].astype(np.float64)))
            out[b, h] = p @ Vd[b, kv, :L]
            E[b, h] = p @ np.abs(Vd[b, kv, :L])
    return out, E


def pin_attn_vs_textbook(o) -> None:
    rng = np.random.default_rng(32)
    for (B, Hq, Hkv, Tcap, D, lens) in ((3, 4, 2, 37, 64, [37, 1, 20]),
                                        (2, 8, 8, 50, 128, [50, 33]),
                                        (1, 6, 1, 9, 32, [9])):
        k, ks, v, vs = _kv_case(rng, B, Hkv, Tcap, D, key_scale=2.0)
        q = rng.standard_normal((B, Hq, D)).astype(np.float32)
        lens = np.array(lens, np.int32)
        c = 1.0 / np.sqrt(D)
        out, E, S = o.attn_decode_i8(q, k, ks, v, vs, lens, c)
        want, E_want = _textbook_attention(q, k, ks, v, vs, lens, c)
        assert np.all(np.abs(out - want) <= 1e-12 * E_want + 1e-300), "attention vs textbook"
        assert np.allclose(E, E_want, rtol=1e-12, atol=0)
        # S: the largest absolute score magnitude bound over the tokens
        G = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                L = int(lens[b])
                terms = np.abs(q[b, h].astype(np.float64) * k[b, h // G, :L].astype(np.float64))
                want_s = (c * ks[b, h // G, :L].astype(np.float64) * terms.sum(-1)).max(initial=0.0)
                assert np.isclose(S[b, h], want_s, rtol=1e-12, atol=0)


def pin_attn_special_cases(o) -> None:
    rng = np.random.default_rng(33)
    B, Hq, Hkv, Tcap, D = 5, 4, 2, 24, 64
    k, ks, v, vs = _kv_case(rng, B, Hkv, Tcap, D)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    c = 1.0 / np.sqrt(D)
    Vd = v.astype(np.float64) * vs[..., None].astype(np.float64)
    # sequence 0: one token, p = 1 exactly
    # sequence 1: every token has the same key codes and scale, so p is uniform
    k[1] = k[1, :, :1]
    ks[1] = ks[1, :, :1]
    # sequence 2: empty; sequence 3: full; sequence 4: one score far beyond exp's range
    k[4], ks[4] = 0, np.float32(1.0)
    k[4, :, 7] = 127
    lens = np.array([1, Tcap, 0, Tcap, Tcap], np.int32)
    q[4] = np.abs(q[4]) + np.float32(1.0)           # score of token 7 >= 127 * 64 * c, others 0
    out, E, S = o.attn_decode_i8(q, k, ks, v, vs, lens, c)
    G = Hq // Hkv
    for h in range(Hq):
        assert np.array_equal(out[0, h], Vd[0, h // G, 0])
        assert np.allclose(out[1, h], Vd[1, h // G].mean(0), rtol=1e-12, atol=1e-15)
        assert np.array_equal(out[4, h], Vd[4, h // G, 7])
    assert np.all(out[2] == 0) and np.all(E[2] == 0)
    # a zero softmax scale gives the plain mean of the values
    out0, _, _ = o.attn_decode_i8(q, k, ks, v, vs, lens, 0.0)
    for h in range(Hq):
        assert np.allclose(out0[3, h], Vd[3, h // G].mean(0), rtol=1e-12, atol=1e-15)
    # tokens past the length take no part, whatever they hold
    lens2 = lens.copy()
    lens2[3] = 10
    k2, v2 = k.copy(), v.copy()
    k2[3, :, 10:] = 127
    v2[3, :, 10:] = -127
    a, _, _ = o.attn_decode_i8(q, k, ks, v, vs, lens2, c)
    b, _, _ = o.attn_decode_i8(q, k2, ks, v2, vs, lens2, c)
    assert np.array_equal(a[3], b[3])
    # permuting the tokens (with their scales) leaves the output unchanged up to rounding
    perm = rng.permutation(Tcap)
    kp, ksp, vp, vsp = k[:, :, perm], ks[:, :, perm], v[:, :, perm], vs[:, :, perm]
    outp, _, _ = o.attn_decode_i8(q, kp, ksp, vp, vsp, lens, c)
    assert np.all(np.abs(outp[3] - out[3]) <= 1e-12 * E[3] + 1e-300)


ALL_PINS = [
    pin_f16_conversion,
    pin_worked_examples,
    pin_roundtrip_q4_0,
    pin_roundtrip_q8_0,
    pin_ranges_and_error_bounds,
    pin_block_dot_bruteforce,
    pin_block_dot_random,
    pin_matmul_vs_dense,
    pin_row_independence,
    pin_f16_matmul,
    pin_q8_0_block_dot_bruteforce,
    pin_q8_0_matmul_vs_dense,
    pin_q5_0_quantizer,
    pin_q5_0_block_dot_and_product,
    pin_q4_1_quantizer,
    pin_q4_1_block_sums_and_product,
    pin_kv_quantizer,
    pin_attn_vs_textbook,
    pin_attn_special_cases,
]
