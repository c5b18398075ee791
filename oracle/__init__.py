"""The CPU oracle for the quantized skinny MUL_MAT and the INT8 KV-cache decode
attention -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library (``quantized_skinny_matmul_gb300``)
never imports it, and the two share no code: the oracle is the plain scalar C in
``gq_oracle.c`` (see its header for what it computes and which page passage each
step follows), wrapped here with ctypes and numpy for argument marshalling only.

``build()`` compiles ``gq_oracle.c`` with the host C compiler into
``oracle/_build/`` (no fast-math, no FP contraction), so the oracle runs the same
on the x86 development host and the aarch64 GPU host.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgq_oracle.so")

QK = 32
Q4_0_BYTES = 18
Q8_0_BYTES = 34
Q5_0_BYTES = 22
Q4_1_BYTES = 20

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def _for_this_cpu(path: str) -> bool:
    """Whether the shared library at path is an ELF object for this host's CPU."""
    machines = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}
    want = machines.get(platform.machine().lower())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    return (len(head) == 20 and head[:4] == b"\x7fELF"
            and (want is None or int.from_bytes(head[18:20], "little") == want))


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the oracle C source into a shared library (skipped when up to date and built
    for this CPU)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src) and _for_this_cpu(out)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cc = os.environ.get("CC", "gcc")
    subprocess.run([cc, *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    I = ctypes.c_int64
    sig = {
        "oracle_quantize_q4_0": ([P, P, I, I], None),
        "oracle_quantize_q8_0": ([P, P, I, I], None),
        "oracle_dequantize_q4_0": ([P, P, I, I], None),
        "oracle_dequantize_q8_0": ([P, P, I, I], None),
        "oracle_block_dots": ([P, P, P, I, I, I], None),
        "oracle_mul_mat_q4_0_f32": ([P, P, P, P, I, I, I, I, I], ctypes.c_int),
        "oracle_mul_mat_q4_0_q8_0_at": ([P, P, P, P, I, I, P, P], None),
        "oracle_block_dots_q8_0": ([P, P, P, I, I, I], None),
        "oracle_quantize_q5_0": ([P, P, I, I], None),
        "oracle_quantize_q4_1": ([P, P, I, I], None),
        "oracle_dequantize_q4_1": ([P, P, I, I], None),
        "oracle_block_sums_q4_1": ([P, P, P, I, I, I], None),
        "oracle_mul_mat_q4_1_f32": ([P, P, P, P, I, I, I, I, I], ctypes.c_int),
        "oracle_mul_mat_q4_1_q8_0_at": ([P, P, P, P, I, I, P, P], None),
        "oracle_dequantize_q5_0": ([P, P, I, I], None),
        "oracle_block_dots_q5_0": ([P, P, P, I, I, I], None),
        "oracle_mul_mat_q5_0_f32": ([P, P, P, P, I, I, I, I, I], ctypes.c_int),
        "oracle_mul_mat_q5_0_q8_0_at": ([P, P, P, P, I, I, P, P], None),
        "oracle_mul_mat_q8_0_f32": ([P, P, P, P, I, I, I, I, I], ctypes.c_int),
        "oracle_mul_mat_q8_0_q8_0_at": ([P, P, P, P, I, I, P, P], None),
        "oracle_mul_mat_f16_f32": ([P, P, P, P, I, I, I, I, I], None),
        "oracle_mul_mat_f16_f32_at": ([P, P, P, P, I, I, P, P], None),
        "oracle_f32_to_f16_array": ([P, P, I], None),
        "oracle_f16_to_f32_array": ([P, P, I], None),
        "oracle_kv_quantize_i8": ([P, P, P, I, I], None),
        "oracle_kv_dequantize_i8": ([P, P, P, I, I], None),
        "oracle_attn_decode_i8": ([P, P, P, P, P, P, ctypes.c_double, P, P, P, I, I, I, I, I],
                                  ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """Thin numpy front end over one build of the oracle library."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    # -- binary16 ---------------------------------------------------------
    def f32_to_f16_bits(self, x) -> np.ndarray:
        x = _c(x, np.float32).ravel()
        out = np.empty(x.size, np.uint16)
        self.lib.oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
        return out

    def f16_bits_to_f32(self, h) -> np.ndarray:
        h = _c(h, np.uint16).ravel()
        out = np.empty(h.size, np.float32)
        self.lib.oracle_f16_to_f32_array(_ptr(h), _ptr(out), h.size)
        return out

    # -- quantizers -------------------------------------------------------
    def quantize_q4_0(self, w) -> np.ndarray:
        """f32 [N, K] -> canonical Q4_0 bytes, uint8 [N, K/32, 18]."""
        w = _c(w, np.float32)
        N, K = w.shape
        assert K % QK == 0
        out = np.empty((N, K // QK, Q4_0_BYTES), np.uint8)
        self.lib.oracle_quantize_q4_0(_ptr(w), _ptr(out), N, K)
        return out

    def quantize_q8_0(self, x) -> np.ndarray:
        """f32 [M, K] -> Q8_0 bytes, uint8 [M, K/32, 34]."""
        x = _c(x, np.float32)
        M, K = x.shape
        assert K % QK == 0
        out = np.empty((M, K // QK, Q8_0_BYTES), np.uint8)
        self.lib.oracle_quantize_q8_0(_ptr(x), _ptr(out), M, K)
        return out

    def dequantize_q4_0(self, q4) -> np.ndarray:
        q4 = _c(q4, np.uint8)
        N, nb = q4.shape[0], q4.shape[1]
        out = np.empty((N, nb * QK), np.float64)
        self.lib.oracle_dequantize_q4_0(_ptr(q4), _ptr(out), N, nb * QK)
        return out

    def dequantize_q8_0(self, q8) -> np.ndarray:
        q8 = _c(q8, np.uint8)
        M, nb = q8.shape[0], q8.shape[1]
        out = np.empty((M, nb * QK), np.float64)
        self.lib.oracle_dequantize_q8_0(_ptr(q8), _ptr(out), M, nb * QK)
        return out

    # -- products ---------------------------------------------------------
    def block_dots(self, q4, q8) -> np.ndarray:
        """int32 [M, N, K/32]: sum_j (q4_j - 8) * q8_j for every block pair."""
        q4 = _c(q4, np.uint8)
        q8 = _c(q8, np.uint8)
        N, nb = q4.shape[0], q4.shape[1]
        M = q8.shape[0]
        assert q8.shape[1] == nb
        out = np.empty((M, N, nb), np.int32)
        self.lib.oracle_block_dots(_ptr(q4), _ptr(q8), _ptr(out), M, N, nb * QK)
        return out

    def mul_mat_q4_0_f32(self, q4, src1, n_range=None):
        """(dst, T), both f64 [M, N]; src1 is quantized to Q8_0 inside (INIT)."""
        q4 = _c(q4, np.uint8)
        src1 = _c(src1, np.float32)
        N, nb = q4.shape[0], q4.shape[1]
        M, K = src1.shape
        assert K == nb * QK
        dst = np.zeros((M, N), np.float64)
        T = np.zeros((M, N), np.float64)
        b, e = (0, N) if n_range is None else n_range
        rc = self.lib.oracle_mul_mat_q4_0_f32(_ptr(q4), _ptr(src1), _ptr(dst), _ptr(T),
                                              M, N, K, b, e)
        if rc != 0:
            raise MemoryError("oracle_mul_mat_q4_0_f32: allocation failed")
        return dst, T

    def mul_mat_q4_0_q8_0_at(self, q4, q8, ms, ns):
        """Selected outputs (ms[i], ns[i]) from quantized operands: (dst, T) f64 [count]."""
        q4 = _c(q4, np.uint8)
        q8 = _c(q8, np.uint8)
        ms = _c(ms, np.int64)
        ns = _c(ns, np.int64)
        K = q4.shape[1] * QK
        out = np.empty(ms.size, np.float64)
        T = np.empty(ms.size, np.float64)
        self.lib.oracle_mul_mat_q4_0_q8_0_at(_ptr(q4), _ptr(q8), _ptr(ms), _ptr(ns), ms.size,
                                             K, _ptr(out), _ptr(T))
        return out, T

    def quantize_q4_1(self, w) -> np.ndarray:
        """f32 [N, K] -> Q4_1 bytes, uint8 [N, K/32, 20]."""
        w = _c(w, np.float32)
        N, K = w.shape
        assert K % QK == 0
        out = np.empty((N, K // QK, Q4_1_BYTES), np.uint8)
        self.lib.oracle_quantize_q4_1(_ptr(w), _ptr(out), N, K)
        return out

    def dequantize_q4_1(self, q41) -> np.ndarray:
        q41 = _c(q41, np.uint8)
        N, nb = q41.shape[0], q41.shape[1]
        out = np.empty((N, nb * QK), np.float64)
        self.lib.oracle_dequantize_q4_1(_ptr(q41), _ptr(out), N, nb * QK)
        return out

    def block_sums_q4_1(self, q41, q8) -> np.ndarray:
        """int32 [M, N, K/32, 2]: (sum_j q_j * q8_j, sum_j q8_j) for every block pair."""
        q41 = _c(q41, np.uint8)
        q8 = _c(q8, np.uint8)
        N, nb = q41.shape[0], q41.shape[1]
        M = q8.shape[0]
        assert q8.shape[1] == nb
        out = np.empty((M, N, nb, 2), np.int32)
        self.lib.oracle_block_sums_q4_1(_ptr(q41), _ptr(q8), _ptr(out), M, N, nb * QK)
        return out

    def mul_mat_q4_1_f32(self, q41, src1, n_range=None):
        """(dst, T), both f64 [M, N], for Q4_1 weights; src1 is quantized to Q8_0 inside."""
        q41 = _c(q41, np.uint8)
        src1 = _c(src1, np.float32)
        N, nb = q41.shape[0], q41.shape[1]
        M, K = src1.shape
        assert K == nb * QK
        dst = np.zeros((M, N), np.float64)
        T = np.zeros((M, N), np.float64)
        b, e = (0, N) if n_range is None else n_range
        rc = self.lib.oracle_mul_mat_q4_1_f32(_ptr(q41), _ptr(src1), _ptr(dst), _ptr(T), M, N, K, b, e)
        if rc != 0:
            raise MemoryError("oracle_mul_mat_q4_1_f32: allocation failed")
        return dst, T

    def mul_mat_q4_1_q8_0_at(self, q41, q8, ms, ns):
        q41 = _c(q41, np.uint8)
        q8 = _c(q8, np.uint8)
        ms = _c(ms, np.int64)
        ns = _c(ns, np.int64)
        K = q41.shape[1] * QK
        out = np.empty(ms.size, np.float64)
        T = np.empty(ms.size, np.float64)
        self.lib.oracle_mul_mat_q4_1_q8_0_at(_ptr(q41), _ptr(q8), _ptr(ms), _ptr(ns), ms.size,
                                             K, _ptr(out), _ptr(T))
        return out, T

    def quantize_q5_0(self, w) -> np.ndarray:
        """f32 [N, K] -> Q5_0 bytes, uint8 [N, K/32, 22]."""
        w = _c(w, np.float32)
        N, K = w.shape
        assert K % QK == 0
        out = np.empty((N, K // QK, Q5_0_BYTES), np.uint8)
        self.lib.oracle_quantize_q5_0(_ptr(w), _ptr(out), N, K)
        return out

    def dequantize_q5_0(self, q5) -> np.ndarray:
        q5 = _c(q5, np.uint8)
        N, nb = q5.shape[0], q5.shape[1]
        out = np.empty((N, nb * QK), np.float64)
        self.lib.oracle_dequantize_q5_0(_ptr(q5), _ptr(out), N, nb * QK)
        return out

    def block_dots_q5_0(self, q5, q8) -> np.ndarray:
        """int32 [M, N, K/32]: sum_j (q5_j - 16) * q8_j."""
        q5 = _c(q5, np.uint8)
        q8 = _c(q8, np.uint8)
        N, nb = q5.shape[0], q5.shape[1]
        M = q8.shape[0]
        assert q8.shape[1] == nb
        out = np.empty((M, N, nb), np.int32)
        self.lib.oracle_block_dots_q5_0(_ptr(q5), _ptr(q8), _ptr(out), M, N, nb * QK)
        return out

    def mul_mat_q5_0_f32(self, q5, src1, n_range=None):
        """(dst, T), both f64 [M, N], for Q5_0 weights; src1 is quantized to Q8_0 inside."""
        q5 = _c(q5, np.uint8)
        src1 = _c(src1, np.float32)
        N, nb = q5.shape[0], q5.shape[1]
        M, K = src1.shape
        assert K == nb * QK
        dst = np.zeros((M, N), np.float64)
        T = np.zeros((M, N), np.float64)
        b, e = (0, N) if n_range is None else n_range
        rc = self.lib.oracle_mul_mat_q5_0_f32(_ptr(q5), _ptr(src1), _ptr(dst), _ptr(T), M, N, K, b, e)
        if rc != 0:
            raise MemoryError("oracle_mul_mat_q5_0_f32: allocation failed")
        return dst, T

    def mul_mat_q5_0_q8_0_at(self, q5, q8, ms, ns):
        q5 = _c(q5, np.uint8)
        q8 = _c(q8, np.uint8)
        ms = _c(ms, np.int64)
        ns = _c(ns, np.int64)
        K = q5.shape[1] * QK
        out = np.empty(ms.size, np.float64)
        T = np.empty(ms.size, np.float64)
        self.lib.oracle_mul_mat_q5_0_q8_0_at(_ptr(q5), _ptr(q8), _ptr(ms), _ptr(ns), ms.size,
                                             K, _ptr(out), _ptr(T))
        return out, T

    def block_dots_q8_0(self, qw, qx) -> np.ndarray:
        """int32 [M, N, K/32]: sum_j qw_j * qx_j for every pair of Q8_0 blocks."""
        qw = _c(qw, np.uint8)
        qx = _c(qx, np.uint8)
        N, nb = qw.shape[0], qw.shape[1]
        M = qx.shape[0]
        assert qx.shape[1] == nb
        out = np.empty((M, N, nb), np.int32)
        self.lib.oracle_block_dots_q8_0(_ptr(qw), _ptr(qx), _ptr(out), M, N, nb * QK)
        return out

    def mul_mat_q8_0_f32(self, qw, src1, n_range=None):
        """(dst, T), both f64 [M, N], for Q8_0 weights; src1 is quantized to Q8_0 inside."""
        qw = _c(qw, np.uint8)
        src1 = _c(src1, np.float32)
        N, nb = qw.shape[0], qw.shape[1]
        M, K = src1.shape
        assert K == nb * QK
        dst = np.zeros((M, N), np.float64)
        T = np.zeros((M, N), np.float64)
        b, e = (0, N) if n_range is None else n_range
        rc = self.lib.oracle_mul_mat_q8_0_f32(_ptr(qw), _ptr(src1), _ptr(dst), _ptr(T), M, N, K, b, e)
        if rc != 0:
            raise MemoryError("oracle_mul_mat_q8_0_f32: allocation failed")
        return dst, T

    def mul_mat_q8_0_q8_0_at(self, qw, qx, ms, ns):
        qw = _c(qw, np.uint8)
        qx = _c(qx, np.uint8)
        ms = _c(ms, np.int64)
        ns = _c(ns, np.int64)
        K = qw.shape[1] * QK
        out = np.empty(ms.size, np.float64)
        T = np.empty(ms.size, np.float64)
        self.lib.oracle_mul_mat_q8_0_q8_0_at(_ptr(qw), _ptr(qx), _ptr(ms), _ptr(ns), ms.size,
                                             K, _ptr(out), _ptr(T))
        return out, T

    def mul_mat_f16_f32(self, w16_bits, src1, n_range=None):
        """(dst, T) f64 [M, N] for F16 weights given as uint16 bit patterns [N, K]."""
        w = _c(w16_bits, np.uint16)
        src1 = _c(src1, np.float32)
        N, K = w.shape
        M = src1.shape[0]
        assert src1.shape[1] == K
        dst = np.zeros((M, N), np.float64)
        T = np.zeros((M, N), np.float64)
        b, e = (0, N) if n_range is None else n_range
        self.lib.oracle_mul_mat_f16_f32(_ptr(w), _ptr(src1), _ptr(dst), _ptr(T), M, N, K, b, e)
        return dst, T

    def mul_mat_f16_f32_at(self, w16_bits, src1, ms, ns):
        w = _c(w16_bits, np.uint16)
        src1 = _c(src1, np.float32)
        ms = _c(ms, np.int64)
        ns = _c(ns, np.int64)
        out = np.empty(ms.size, np.float64)
        T = np.empty(ms.size, np.float64)
        self.lib.oracle_mul_mat_f16_f32_at(_ptr(w), _ptr(src1), _ptr(ms), _ptr(ns), ms.size,
                                           w.shape[1], _ptr(out), _ptr(T))
        return out, T

    # -- INT8 KV cache ----------------------------------------------------
    def kv_quantize_i8(self, x):
        """f32 [..., D] -> (int8 codes [..., D], f32 scales [...]): one scale per row of D."""
        x = _c(x, np.float32)
        D = x.shape[-1]
        rows = x.size // D if D else 0
        q = np.empty(x.shape, np.int8)
        s = np.empty(x.shape[:-1], np.float32)
        self.lib.oracle_kv_quantize_i8(_ptr(x), _ptr(q), _ptr(s), rows, D)
        return q, s

    def kv_dequantize_i8(self, q, s) -> np.ndarray:
        """f64 [..., D]: codes times their row's scale."""
        q = _c(q, np.int8)
        s = _c(s, np.float32)
        D = q.shape[-1]
        assert s.shape == q.shape[:-1]
        out = np.empty(q.shape, np.float64)
        self.lib.oracle_kv_dequantize_i8(_ptr(q), _ptr(s), _ptr(out), q.size // D if D else 0, D)
        return out

    def attn_decode_i8(self, q, k, ks, v, vs, lens, c):
        """Decode attention over an INT8 cache: (out, E) f64 [B, Hq, D] and S f64 [B, Hq].

        q f32 [B, Hq, D]; k, v int8 [B, Hkv, Tcap, D]; ks, vs f32 [B, Hkv, Tcap];
        lens int32 [B]; c the softmax scale.
        """
        q = _c(q, np.float32)
        k, v = _c(k, np.int8), _c(v, np.int8)
        ks, vs = _c(ks, np.float32), _c(vs, np.float32)
        lens = _c(lens, np.int32)
        B, Hq, D = q.shape
        _, Hkv, Tcap, _ = k.shape
        assert k.shape == v.shape == (B, Hkv, Tcap, D)
        assert ks.shape == vs.shape == (B, Hkv, Tcap) and lens.shape == (B,)
        out = np.zeros((B, Hq, D), np.float64)
        E = np.zeros((B, Hq, D), np.float64)
        S = np.zeros((B, Hq), np.float64)
        rc = self.lib.oracle_attn_decode_i8(_ptr(q), _ptr(k), _ptr(ks), _ptr(v), _ptr(vs),
                                            _ptr(lens), float(c), _ptr(out), _ptr(E), _ptr(S),
                                            B, Hq, Hkv, Tcap, D)
        if rc == -2:
            raise MemoryError("oracle_attn_decode_i8: allocation failed")
        if rc != 0:
            raise ValueError("oracle_attn_decode_i8: Hq must be a multiple of Hkv and "
                             "0 <= lens[b] <= Tcap")
        return out, E, S


_default: Oracle | None = None


def get() -> Oracle:
    """The process-wide oracle over the default build."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
