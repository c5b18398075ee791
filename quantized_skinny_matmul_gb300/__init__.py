"""Python binding of libgq, the GB300 quantized skinny MUL_MAT library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_lib/libgq.so`` (built by ``_build.py``); PyTorch supplies device
memory and streams.  There is no CPU fallback: when the library is missing or
the device is not a GB300, the calls raise.

The functions below carry the names of the C entry points in ``include/gq.h``
and take the same arguments, with torch CUDA tensors (or raw device addresses
as ints) in place of pointers and an optional stream (default: torch's current
stream).  They raise ``GQError`` when the C call returns a non-zero status.
The lower-case helpers at the end allocate the outputs with torch and call them.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# GQ_LIBRARY may name another build of the same ABI (the GQ_DEBUG build, _lib/libgq_debug.so)
LIB_PATH = os.environ.get("GQ_LIBRARY") or os.path.join(_PKG, "_lib", "libgq.so")

GQ_OK = 0
GQ_ERR_INVALID_ARG = 1
GQ_ERR_MISALIGNED = 2
GQ_ERR_UNSUPPORTED_DEVICE = 3
GQ_ERR_CUDA = 4
GQ_ERR_TIMEOUT = 5
GQ_ERR_NO_MEMORY = 6
GQ_ERR_DEVICE_CHECK = 7

GQ_PATH_AUTO = 0
GQ_PATH_GEMV = 1
GQ_PATH_TC = 2

_lock = threading.Lock()
_lib = None


class GQError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: status {status}: {message}")


_P = ctypes.c_void_p
_I = ctypes.c_int64
_S = ctypes.c_int

# name -> (argtypes, restype); the signatures of include/gq.h
SIGNATURES = {
    "gq_debug_wait_timeout": ([ctypes.c_uint32, _P], _S),
    "gq_debug_dp4a_probe": ([_I, _P, _I, _P], _S),
    "gq_kv_quantize_i8": ([_P, _P, _P, _I, _I, _P], _S),
    "gq_kv_append_i8": ([_P, _P, _P, _P, _I, _I, _I, _I, _P], _S),
    "gq_attn_decode_i8": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P], _S),
    "gq_abi_version": ([], ctypes.c_int),
    "gq_status_string": ([_S], ctypes.c_char_p),
    "gq_last_error_message": ([], ctypes.c_char_p),
    "gq_last_error": ([], _S),
    "gq_q4_0_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_q8_0_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_q4_0_repacked_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_quantize_q4_0": ([_P, _P, _I, _I, _P], _S),
    "gq_quantize_rows_q8_0": ([_P, _P, _I, _I, _P], _S),
    "gq_repack_q4_0": ([_P, _P, _I, _I, _P], _S),
    "gq_mul_mat_q4_0_f32": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_mul_mat_f16_f32": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_mul_mat_q4_0_f32_path": ([_P, _P, _P, _I, _I, _I, _S, _P], _S),
    "gq_mul_mat_f16_f32_path": ([_P, _P, _P, _I, _I, _I, _S, _P], _S),
    "gq_reserve_workspace": ([_I, _I, _I, _P], _S),
    "gq_set_m_threshold": ([_I], _S),
    "gq_set_static_weights": ([ctypes.c_int], _S),
    "gq_get_static_weights": ([], ctypes.c_int),
    "gq_get_m_threshold": ([], _I),
    "gq_debug_block_dots_q4_0": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_mul_mat_q4_0_f32_noalloc": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_mul_mat_q4_0_f32_host": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_set_dispatch_profile": ([ctypes.c_int, _I, _I, _P, _P, _P, _I], _S),
    "gq_clear_dispatch_profiles": ([], _S),
    "gq_choose_path": ([ctypes.c_int, _I, _I, _I], ctypes.c_int),
    "gq_q4_1_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_q4_1_repacked_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_quantize_q4_1": ([_P, _P, _I, _I, _P], _S),
    "gq_repack_q4_1": ([_P, _P, _I, _I, _P], _S),
    "gq_mul_mat_q4_1_f32": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_q5_0_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_q5_0_repacked_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_quantize_q5_0": ([_P, _P, _I, _I, _P], _S),
    "gq_repack_q5_0": ([_P, _P, _I, _I, _P], _S),
    "gq_mul_mat_q5_0_f32": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_q8_0_repacked_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_repack_q8_0": ([_P, _P, _I, _I, _P], _S),
    "gq_mul_mat_q8_0_f32": ([_P, _P, _P, _I, _I, _I, _P], _S),
    "gq_f16_repacked_bytes": ([_I, _I], ctypes.c_size_t),
    "gq_repack_f16": ([_P, _P, _I, _I, _P], _S),
    "gq_mul_mat_f16r_f32": ([_P, _P, _P, _I, _I, _I, _P], _S),
}


def lib() -> ctypes.CDLL:
    """The loaded libgq.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m quantized_skinny_matmul_gb300._build` (nvcc, sm_103a)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (args, res) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.argtypes = args
                    fn.restype = res
                _lib = handle
    return _lib


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != GQ_OK:
        msg = lib().gq_last_error_message().decode(errors="replace")
        raise GQError(status, where, msg or lib().gq_status_string(status).decode())


# ---------------------------------------------------------------------------
# the entry points of include/gq.h
# ---------------------------------------------------------------------------
def gq_abi_version() -> int:
    return lib().gq_abi_version()


def gq_last_error() -> int:
    """Status of the device-side sticky word (synchronizes the device)."""
    return lib().gq_last_error()


def gq_q4_0_bytes(N: int, K: int) -> int:
    return lib().gq_q4_0_bytes(N, K)


def gq_q8_0_bytes(M: int, K: int) -> int:
    return lib().gq_q8_0_bytes(M, K)


def gq_q4_0_repacked_bytes(N: int, K: int) -> int:
    return lib().gq_q4_0_repacked_bytes(N, K)


def gq_quantize_q4_0(w, q4_blocks, N: int, K: int, stream=None) -> None:
    _check(lib().gq_quantize_q4_0(_ptr(w), _ptr(q4_blocks), N, K, _stream(stream)), "gq_quantize_q4_0")


def gq_quantize_rows_q8_0(x, q8_blocks, M: int, K: int, stream=None) -> None:
    _check(lib().gq_quantize_rows_q8_0(_ptr(x), _ptr(q8_blocks), M, K, _stream(stream)),
           "gq_quantize_rows_q8_0")


def gq_repack_q4_0(q4_blocks, q4_repacked, N: int, K: int, stream=None) -> None:
    _check(lib().gq_repack_q4_0(_ptr(q4_blocks), _ptr(q4_repacked), N, K, _stream(stream)),
           "gq_repack_q4_0")


def gq_mul_mat_q4_0_f32(q4_repacked, src1, dst, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_mul_mat_q4_0_f32(_ptr(q4_repacked), _ptr(src1), _ptr(dst), M, N, K, _stream(stream)),
           "gq_mul_mat_q4_0_f32")


def gq_mul_mat_f16_f32(src0_f16, src1, dst, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_mul_mat_f16_f32(_ptr(src0_f16), _ptr(src1), _ptr(dst), M, N, K, _stream(stream)),
           "gq_mul_mat_f16_f32")


def gq_mul_mat_q4_0_f32_path(q4_repacked, src1, dst, M: int, N: int, K: int, path: int,
                             stream=None) -> None:
    _check(lib().gq_mul_mat_q4_0_f32_path(_ptr(q4_repacked), _ptr(src1), _ptr(dst), M, N, K, path,
                                          _stream(stream)), "gq_mul_mat_q4_0_f32_path")


def gq_mul_mat_f16_f32_path(src0_f16, src1, dst, M: int, N: int, K: int, path: int,
                            stream=None) -> None:
    _check(lib().gq_mul_mat_f16_f32_path(_ptr(src0_f16), _ptr(src1), _ptr(dst), M, N, K, path,
                                         _stream(stream)), "gq_mul_mat_f16_f32_path")


def gq_reserve_workspace(M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_reserve_workspace(M, N, K, _stream(stream)), "gq_reserve_workspace")


def gq_set_m_threshold(t: int) -> None:
    _check(lib().gq_set_m_threshold(t), "gq_set_m_threshold")


def gq_get_m_threshold() -> int:
    return lib().gq_get_m_threshold()


def gq_set_static_weights(enable: bool) -> None:
    _check(lib().gq_set_static_weights(1 if enable else 0), "gq_set_static_weights")


def gq_get_static_weights() -> bool:
    return bool(lib().gq_get_static_weights())


def gq_mul_mat_q4_0_f32_noalloc(q4_repacked, src1, dst, M: int, N: int, K: int, stream=None) -> None:
    """The Q4_0 product with no device allocation (static scratch in the library)."""
    _check(lib().gq_mul_mat_q4_0_f32_noalloc(_ptr(q4_repacked), _ptr(src1), _ptr(dst), M, N, K,
                                             _stream(stream)), "gq_mul_mat_q4_0_f32_noalloc")


def _host_ptr(a) -> int:
    if isinstance(a, int):
        return a
    if getattr(a, "is_cuda", False):
        raise ValueError("expected a host (CPU) tensor")
    if not a.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return a.data_ptr()


def gq_mul_mat_q4_0_f32_host(q4_repacked, src1_host, dst_host, M: int, N: int, K: int, stream=None) -> None:
    """The Q4_0 product from host src1 into host dst (copies enqueued on the stream)."""
    _check(lib().gq_mul_mat_q4_0_f32_host(_ptr(q4_repacked), _host_ptr(src1_host), _host_ptr(dst_host), M, N, K,
                                          _stream(stream)), "gq_mul_mat_q4_0_f32_host")


GQ_KIND_Q4_0 = 0
GQ_KIND_F16 = 1


def gq_set_dispatch_profile(kind: int, N: int, K: int, Ms, t_gemv, t_tc) -> None:
    """Install the benched times of both kernel families at the given M for one shape."""
    n = len(Ms)
    if len(t_gemv) != n or len(t_tc) != n:
        raise ValueError("one time per M and family")
    m_arr = (ctypes.c_int64 * n)(*[int(m) for m in Ms])
    g_arr = (ctypes.c_double * n)(*[float(t) for t in t_gemv])
    t_arr = (ctypes.c_double * n)(*[float(t) for t in t_tc])
    _check(lib().gq_set_dispatch_profile(kind, N, K, ctypes.addressof(m_arr), ctypes.addressof(g_arr),
                                         ctypes.addressof(t_arr), n), "gq_set_dispatch_profile")


def gq_clear_dispatch_profiles() -> None:
    _check(lib().gq_clear_dispatch_profiles(), "gq_clear_dispatch_profiles")


def gq_choose_path(kind: int, N: int, K: int, M: int) -> int:
    return lib().gq_choose_path(kind, N, K, M)


def gq_q4_1_bytes(N: int, K: int) -> int:
    return lib().gq_q4_1_bytes(N, K)


def gq_q4_1_repacked_bytes(N: int, K: int) -> int:
    return lib().gq_q4_1_repacked_bytes(N, K)


def gq_quantize_q4_1(w, q41_blocks, N: int, K: int, stream=None) -> None:
    _check(lib().gq_quantize_q4_1(_ptr(w), _ptr(q41_blocks), N, K, _stream(stream)), "gq_quantize_q4_1")


def gq_repack_q4_1(q41_blocks, q41_repacked, N: int, K: int, stream=None) -> None:
    _check(lib().gq_repack_q4_1(_ptr(q41_blocks), _ptr(q41_repacked), N, K, _stream(stream)), "gq_repack_q4_1")


def gq_mul_mat_q4_1_f32(q41_repacked, src1, dst, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_mul_mat_q4_1_f32(_ptr(q41_repacked), _ptr(src1), _ptr(dst), M, N, K, _stream(stream)),
           "gq_mul_mat_q4_1_f32")


def gq_q5_0_bytes(N: int, K: int) -> int:
    return lib().gq_q5_0_bytes(N, K)


def gq_q5_0_repacked_bytes(N: int, K: int) -> int:
    return lib().gq_q5_0_repacked_bytes(N, K)


def gq_quantize_q5_0(w, q5_blocks, N: int, K: int, stream=None) -> None:
    _check(lib().gq_quantize_q5_0(_ptr(w), _ptr(q5_blocks), N, K, _stream(stream)), "gq_quantize_q5_0")


def gq_repack_q5_0(q5_blocks, q5_repacked, N: int, K: int, stream=None) -> None:
    _check(lib().gq_repack_q5_0(_ptr(q5_blocks), _ptr(q5_repacked), N, K, _stream(stream)), "gq_repack_q5_0")


def gq_mul_mat_q5_0_f32(q5_repacked, src1, dst, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_mul_mat_q5_0_f32(_ptr(q5_repacked), _ptr(src1), _ptr(dst), M, N, K, _stream(stream)),
           "gq_mul_mat_q5_0_f32")


def gq_q8_0_repacked_bytes(N: int, K: int) -> int:
    return lib().gq_q8_0_repacked_bytes(N, K)


def gq_repack_q8_0(q8_blocks, q8_repacked, N: int, K: int, stream=None) -> None:
    _check(lib().gq_repack_q8_0(_ptr(q8_blocks), _ptr(q8_repacked), N, K, _stream(stream)), "gq_repack_q8_0")


def gq_mul_mat_q8_0_f32(q8_repacked, src1, dst, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_mul_mat_q8_0_f32(_ptr(q8_repacked), _ptr(src1), _ptr(dst), M, N, K, _stream(stream)),
           "gq_mul_mat_q8_0_f32")


def gq_f16_repacked_bytes(N: int, K: int) -> int:
    return lib().gq_f16_repacked_bytes(N, K)


def gq_repack_f16(src0_f16, f16_repacked, N: int, K: int, stream=None) -> None:
    _check(lib().gq_repack_f16(_ptr(src0_f16), _ptr(f16_repacked), N, K, _stream(stream)), "gq_repack_f16")


def gq_mul_mat_f16r_f32(f16_repacked, src1, dst, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_mul_mat_f16r_f32(_ptr(f16_repacked), _ptr(src1), _ptr(dst), M, N, K, _stream(stream)),
           "gq_mul_mat_f16r_f32")


def gq_debug_block_dots_q4_0(q4_repacked, q8_blocks, sumi, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().gq_debug_block_dots_q4_0(_ptr(q4_repacked), _ptr(q8_blocks), _ptr(sumi), M, N, K,
                                          _stream(stream)), "gq_debug_block_dots_q4_0")


def gq_debug_wait_timeout(limit: int, stream=None) -> None:
    _check(lib().gq_debug_wait_timeout(limit, _stream(stream)), "gq_debug_wait_timeout")


def gq_debug_dp4a_probe(iters: int, sink, blocks: int, stream=None) -> None:
    _check(lib().gq_debug_dp4a_probe(iters, _ptr(sink), blocks, _stream(stream)), "gq_debug_dp4a_probe")


def gq_kv_quantize_i8(x, q, scale, rows: int, D: int, stream=None) -> None:
    _check(lib().gq_kv_quantize_i8(_ptr(x), _ptr(q), _ptr(scale), rows, D, _stream(stream)), "gq_kv_quantize_i8")


def gq_kv_append_i8(x, q, scale, pos, B: int, Hkv: int, Tcap: int, D: int, stream=None) -> None:
    _check(lib().gq_kv_append_i8(_ptr(x), _ptr(q), _ptr(scale), _ptr(pos), B, Hkv, Tcap, D, _stream(stream)),
           "gq_kv_append_i8")


def gq_attn_decode_i8(q, k, k_scale, v, v_scale, lens, out, B: int, Hq: int, Hkv: int, Tcap: int, D: int,
                      softmax_scale: float, stream=None) -> None:
    _check(lib().gq_attn_decode_i8(_ptr(q), _ptr(k), _ptr(k_scale), _ptr(v), _ptr(v_scale), _ptr(lens), _ptr(out),
                                   B, Hq, Hkv, Tcap, D, float(softmax_scale), _stream(stream)),
           "gq_attn_decode_i8")


# ---------------------------------------------------------------------------
# allocating helpers (torch tensors in, torch tensors out)
# ---------------------------------------------------------------------------
def quantize_q4_0(w):
    """f32 CUDA tensor [N, K] -> canonical Q4_0 bytes, uint8 [N, K/32, 18]."""
    import torch
    N, K = w.shape
    out = torch.empty((N, K // 32, 18), dtype=torch.uint8, device=w.device)
    gq_quantize_q4_0(w, out, N, K)
    return out


def quantize_rows_q8_0(x):
    import torch
    M, K = x.shape
    out = torch.empty((M, K // 32, 34), dtype=torch.uint8, device=x.device)
    gq_quantize_rows_q8_0(x, out, M, K)
    return out


def repack_q4_0(q4, N: int, K: int):
    import torch
    out = torch.empty(gq_q4_0_repacked_bytes(N, K), dtype=torch.uint8, device=q4.device)
    gq_repack_q4_0(q4, out, N, K)
    return out


def concat_rows_q4_0(repacked, Ns, K: int):
    """Several repacked weight matrices with the same K as one matrix of sum(Ns) rows.

    The repacked layout stores whole 16-row groups one after the other, so when
    every N is a multiple of 16 the concatenated buffers are the repacked layout
    of the stacked matrix: one product then computes [x W1^T | x W2^T | ...]
    (for example Q, K and V, or gate and up, which share their input) with one
    weight stream and one quantized copy of the activations.
    """
    import torch
    if len(repacked) != len(Ns):
        raise ValueError("one N per matrix")
    for r, n in zip(repacked, Ns):
        if n % 16:
            raise ValueError(f"N={n} is not a multiple of 16: row groups would be padded")
        if r.numel() != gq_q4_0_repacked_bytes(n, K):
            raise ValueError(f"a buffer of {r.numel()} bytes is not the repacked layout of N={n}, K={K}")
    return torch.cat([r.reshape(-1) for r in repacked])


def mul_mat_q4_0_f32(q4_repacked, src1, N: int, path: int = GQ_PATH_AUTO, out=None):
    import torch
    M, K = src1.shape
    dst = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=src1.device)
    gq_mul_mat_q4_0_f32_path(q4_repacked, src1, dst, M, N, K, path)
    return dst


def mul_mat_f16_f32(src0_f16, src1, path: int = GQ_PATH_AUTO, out=None):
    import torch
    N, K = src0_f16.shape
    M = src1.shape[0]
    dst = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=src1.device)
    gq_mul_mat_f16_f32_path(src0_f16, src1, dst, M, N, K, path)
    return dst


def repack_f16(src0_f16):
    """F16 CUDA tensor [N, K] -> the 16 x 32 tile layout of gq_repack_f16 (uint8)."""
    import torch
    N, K = src0_f16.shape
    out = torch.empty(gq_f16_repacked_bytes(N, K), dtype=torch.uint8, device=src0_f16.device)
    gq_repack_f16(src0_f16, out, N, K)
    return out


def mul_mat_f16r_f32(f16_repacked, src1, N: int, out=None):
    import torch
    M, K = src1.shape
    dst = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=src1.device)
    gq_mul_mat_f16r_f32(f16_repacked, src1, dst, M, N, K)
    return dst


def repack_q8_0(q8, N: int, K: int):
    """Q8_0 weight blocks (uint8 [N, K/32, 34], e.g. from quantize_rows_q8_0) -> the tile layout."""
    import torch
    out = torch.empty(gq_q8_0_repacked_bytes(N, K), dtype=torch.uint8, device=q8.device)
    gq_repack_q8_0(q8, out, N, K)
    return out


def mul_mat_q8_0_f32(q8_repacked, src1, N: int, out=None):
    import torch
    M, K = src1.shape
    dst = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=src1.device)
    gq_mul_mat_q8_0_f32(q8_repacked, src1, dst, M, N, K)
    return dst


def quantize_q5_0(w):
    """f32 CUDA tensor [N, K] -> Q5_0 bytes, uint8 [N, K/32, 22]."""
    import torch
    N, K = w.shape
    out = torch.empty((N, K // 32, 22), dtype=torch.uint8, device=w.device)
    gq_quantize_q5_0(w, out, N, K)
    return out


def repack_q5_0(q5, N: int, K: int):
    import torch
    out = torch.empty(gq_q5_0_repacked_bytes(N, K), dtype=torch.uint8, device=q5.device)
    gq_repack_q5_0(q5, out, N, K)
    return out


def mul_mat_q5_0_f32(q5_repacked, src1, N: int, out=None):
    import torch
    M, K = src1.shape
    dst = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=src1.device)
    gq_mul_mat_q5_0_f32(q5_repacked, src1, dst, M, N, K)
    return dst


def quantize_q4_1(w):
    """f32 CUDA tensor [N, K] -> Q4_1 bytes, uint8 [N, K/32, 20]."""
    import torch
    N, K = w.shape
    out = torch.empty((N, K // 32, 20), dtype=torch.uint8, device=w.device)
    gq_quantize_q4_1(w, out, N, K)
    return out


def repack_q4_1(q41, N: int, K: int):
    import torch
    out = torch.empty(gq_q4_1_repacked_bytes(N, K), dtype=torch.uint8, device=q41.device)
    gq_repack_q4_1(q41, out, N, K)
    return out


def mul_mat_q4_1_f32(q41_repacked, src1, N: int, out=None):
    import torch
    M, K = src1.shape
    dst = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=src1.device)
    gq_mul_mat_q4_1_f32(q41_repacked, src1, dst, M, N, K)
    return dst


def tune_dispatch(weights, N: int, K: int, kind: int = GQ_KIND_Q4_0,
                  Ms=(1, 2, 4, 8, 16, 32, 64, 128, 256, 512), reps: int = 20, install: bool = True):
    """Bench both kernel families on the current device for one shape and install the profile.

    ``weights`` are the product's weights on the device (Q4_0 repacked, or row-major F16).
    Each M is timed with CUDA events over ``reps`` back-to-back products after a warm-up.
    Returns {"M": [...], "gemv_us": [...], "tc_us": [...]}.
    """
    import torch
    fn = gq_mul_mat_q4_0_f32_path if kind == GQ_KIND_Q4_0 else gq_mul_mat_f16_f32_path
    out = {"M": [], "gemv_us": [], "tc_us": []}
    gen = torch.Generator(device=weights.device).manual_seed(1234)
    for M in Ms:
        x = torch.randn((M, K), generator=gen, device=weights.device, dtype=torch.float32)
        dst = torch.empty((M, N), device=weights.device, dtype=torch.float32)
        times = []
        for path in (GQ_PATH_GEMV, GQ_PATH_TC):
            for _ in range(3):
                fn(weights, x, dst, M, N, K, path)
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record()
            for _ in range(reps):
                fn(weights, x, dst, M, N, K, path)
            end.record()
            end.synchronize()
            times.append(start.elapsed_time(end) * 1e3 / reps)
        out["M"].append(int(M))
        out["gemv_us"].append(times[0])
        out["tc_us"].append(times[1])
    if install:
        gq_set_dispatch_profile(kind, N, K, out["M"], out["gemv_us"], out["tc_us"])
    return out


def kv_quantize_i8(x):
    """f32 CUDA tensor [..., D] -> (int8 codes [..., D], f32 scales [...]), one scale per row of D."""
    import torch
    x = x.contiguous()
    D = x.shape[-1]
    q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    s = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    gq_kv_quantize_i8(x, q, s, x.numel() // D, D)
    return q, s


def attn_decode_i8(q, k, k_scale, v, v_scale, lens, softmax_scale=None, out=None):
    """Decode attention over an INT8 cache: q f32 [B, Hq, D]; k, v int8 [B, Hkv, Tcap, D];
    scales f32 [B, Hkv, Tcap]; lens int32 [B].  Returns f32 [B, Hq, D]."""
    import torch
    B, Hq, D = q.shape
    Hkv, Tcap = k.shape[1], k.shape[2]
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    gq_attn_decode_i8(q, k, k_scale, v, v_scale, lens, out, B, Hq, Hkv, Tcap, D, softmax_scale)
    return out
