"""The C ABI without a GPU: the library loads, exports every entry point that
include/gq.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

import quantized_skinny_matmul_gb300 as gq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__  # noqa: F401  (build() is what the driver runs)
    from quantized_skinny_matmul_gb300 import _build
    _build.build()
    return gq.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("gq_quantize_q4_0", "gq_quantize_rows_q8_0", "gq_repack_q4_0",
                     "gq_mul_mat_q4_0_f32", "gq_mul_mat_f16_f32", "gq_last_error",
                     "gq_debug_block_dots_q4_0"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(gq.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert set(declared_functions()) <= set(gq.SIGNATURES)


def test_version_and_strings(lib):
    assert gq.gq_abi_version() == 1
    for s in range(8):
        assert lib.gq_status_string(s)
    assert lib.gq_status_string(99) == b"unknown status"


def test_sizes(lib):
    assert gq.gq_q4_0_bytes(4096, 4096) == 4096 * 128 * 18
    assert gq.gq_q8_0_bytes(3, 64) == 3 * 2 * 34
    assert gq.gq_q4_0_repacked_bytes(4096, 4096) == 256 * 32 * 1152 == 4096 * 128 * 18
    assert gq.gq_q4_0_repacked_bytes(11008, 4096) == 11008 * 128 * 18
    assert gq.gq_q4_0_repacked_bytes(4096, 11008) == 4096 * 344 * 18
    assert gq.gq_q4_0_repacked_bytes(17, 96) == 2 * 1 * 1152
    assert gq.gq_q4_0_bytes(4, 33) == 0 and gq.gq_q4_0_repacked_bytes(0, 32) == 0
    assert gq.gq_f16_repacked_bytes(4096, 4096) == 4096 * 4096 * 2
    assert gq.gq_f16_repacked_bytes(17, 96) == 2 * 3 * 1024
    assert gq.gq_f16_repacked_bytes(16, 48) == 0
    assert gq.gq_q8_0_repacked_bytes(4096, 4096) == 4096 * 128 * 34
    assert gq.gq_q5_0_bytes(4096, 4096) == 4096 * 128 * 22 == gq.gq_q5_0_repacked_bytes(4096, 4096)
    assert gq.gq_q5_0_repacked_bytes(17, 96) == 2 * 1 * 1408 and gq.gq_q5_0_bytes(4, 33) == 0
    assert gq.gq_q4_1_bytes(4096, 4096) == 4096 * 128 * 20 == gq.gq_q4_1_repacked_bytes(4096, 4096)
    assert gq.gq_q4_1_repacked_bytes(17, 96) == 2 * 1 * 1280
    assert gq.gq_q8_0_repacked_bytes(17, 96) == 2 * 1 * 2176 and gq.gq_q8_0_repacked_bytes(16, 48) == 0


FAKE = 0x10000            # 16-byte aligned, never dereferenced: checks fail first
ODD = 0x10008


@pytest.mark.parametrize("args, status", [
    ((FAKE, FAKE, FAKE, 1, 64, 48), gq.GQ_ERR_INVALID_ARG),     # K % 32
    ((FAKE, FAKE, FAKE, 0, 64, 64), gq.GQ_ERR_INVALID_ARG),     # M == 0
    ((FAKE, FAKE, FAKE, 1, -1, 64), gq.GQ_ERR_INVALID_ARG),     # N < 0
    ((0, FAKE, FAKE, 1, 64, 64), gq.GQ_ERR_INVALID_ARG),        # null weights
    ((FAKE, 0, FAKE, 1, 64, 64), gq.GQ_ERR_INVALID_ARG),        # null src1
    ((FAKE, FAKE, 0, 1, 64, 64), gq.GQ_ERR_INVALID_ARG),        # null dst
    ((ODD, FAKE, FAKE, 1, 64, 64), gq.GQ_ERR_MISALIGNED),
    ((FAKE, ODD, FAKE, 1, 64, 64), gq.GQ_ERR_MISALIGNED),
    ((FAKE, FAKE, ODD, 1, 64, 64), gq.GQ_ERR_MISALIGNED),
])
def test_argument_checks_mul_mat(lib, args, status):
    for fn in (lib.gq_mul_mat_q4_0_f32, lib.gq_mul_mat_f16_f32):
        assert fn(*args, None) == status
        assert lib.gq_last_error_message()


def test_argument_checks_other_entries(lib):
    assert lib.gq_quantize_q4_0(FAKE, FAKE, 4, 40, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_quantize_q4_0(ODD, FAKE, 4, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_quantize_rows_q8_0(FAKE, 0, 4, 64, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_repack_q4_0(FAKE, FAKE, 4, 64, None) == gq.GQ_ERR_INVALID_ARG   # overlap
    assert lib.gq_repack_f16(FAKE, FAKE + 256, 4, 64, None) == gq.GQ_ERR_INVALID_ARG   # overlap
    assert lib.gq_repack_f16(FAKE, FAKE, 4, 48, None) == gq.GQ_ERR_INVALID_ARG   # K % 32
    assert lib.gq_mul_mat_f16r_f32(FAKE, FAKE, ODD, 1, 64, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_mul_mat_f16r_f32(0, FAKE, FAKE, 1, 64, 64, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_repack_q8_0(FAKE, FAKE + 64, 4, 64, None) == gq.GQ_ERR_INVALID_ARG   # overlap
    assert lib.gq_repack_q5_0(FAKE, FAKE + 32, 4, 64, None) == gq.GQ_ERR_INVALID_ARG   # overlap
    assert lib.gq_repack_q4_1(FAKE, FAKE + 32, 4, 64, None) == gq.GQ_ERR_INVALID_ARG   # overlap
    assert lib.gq_quantize_q4_1(ODD, FAKE, 4, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_mul_mat_q4_1_f32(FAKE, FAKE, FAKE, 0, 64, 64, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_quantize_q5_0(FAKE, FAKE, 4, 40, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_mul_mat_q5_0_f32(FAKE, ODD, FAKE, 1, 64, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_mul_mat_q8_0_f32(FAKE, FAKE, ODD, 1, 64, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_mul_mat_q8_0_f32(FAKE, FAKE, FAKE, 1, 64, 48, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_mul_mat_q4_0_f32_host(FAKE, 0, FAKE, 1, 64, 64, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_mul_mat_q4_0_f32_host(FAKE, FAKE, 0, 1, 64, 64, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_mul_mat_q4_0_f32_host(ODD, FAKE, FAKE, 1, 64, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_mul_mat_q4_0_f32_host(FAKE, FAKE, FAKE, 1, 64, 40, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_debug_block_dots_q4_0(FAKE, FAKE, ODD, 1, 16, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_mul_mat_q4_0_f32_path(FAKE, FAKE, FAKE, 1, 64, 64, 7, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_set_m_threshold(-1) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_debug_wait_timeout(0, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_debug_wait_timeout((1 << 22) + 1, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_set_m_threshold(16) == gq.GQ_OK and lib.gq_get_m_threshold() == 16


def test_binding_raises(lib):
    with pytest.raises(gq.GQError) as e:
        gq.gq_mul_mat_q4_0_f32(FAKE, FAKE, FAKE, 1, 64, 48, stream=0)
    assert e.value.status == gq.GQ_ERR_INVALID_ARG and "multiple of 32" in str(e.value)


def test_dispatch_profiles(lib):
    """A benched profile decides GQ_PATH_AUTO by linear interpolation in M (no GPU involved)."""
    gq.gq_clear_dispatch_profiles()
    # GEMV 10, 20, 40 and tiles 25, 22, 30 at M = 16, 32, 64
    gq.gq_set_dispatch_profile(gq.GQ_KIND_Q4_0, 64, 128, [16, 32, 64], [10, 20, 40], [25, 22, 30])
    cases = {8: gq.GQ_PATH_GEMV,      # extrapolated: 5 vs 26.5
             16: gq.GQ_PATH_GEMV, 24: gq.GQ_PATH_GEMV, 32: gq.GQ_PATH_GEMV,   # 20 vs 22 at 32
             48: gq.GQ_PATH_TC,       # 30 vs 26
             64: gq.GQ_PATH_TC, 128: gq.GQ_PATH_TC}   # extrapolated: 80 vs 46
    for M, want in cases.items():
        assert gq.gq_choose_path(gq.GQ_KIND_Q4_0, 64, 128, M) == want, M
    # another kind or shape falls back to the M threshold
    assert gq.gq_choose_path(gq.GQ_KIND_F16, 64, 128, 48) == gq.GQ_PATH_TC
    assert gq.gq_choose_path(gq.GQ_KIND_Q4_0, 64, 256, 8) == gq.GQ_PATH_GEMV
    assert gq.gq_choose_path(gq.GQ_KIND_Q4_0, 64, 256, 48) == gq.GQ_PATH_TC
    # a new profile replaces the old one; one point is a constant curve
    gq.gq_set_dispatch_profile(gq.GQ_KIND_Q4_0, 64, 128, [32], [1.0], [2.0])
    assert gq.gq_choose_path(gq.GQ_KIND_Q4_0, 64, 128, 512) == gq.GQ_PATH_GEMV
    with pytest.raises(gq.GQError):
        gq.gq_set_dispatch_profile(gq.GQ_KIND_Q4_0, 64, 128, [32, 16], [1, 2], [1, 2])   # M not increasing
    with pytest.raises(gq.GQError):
        gq.gq_set_dispatch_profile(gq.GQ_KIND_Q4_0, 64, 100, [16], [1], [2])             # K % 32
    with pytest.raises(gq.GQError):
        gq.gq_set_dispatch_profile(7, 64, 128, [16], [1], [2])                           # kind
    with pytest.raises(gq.GQError):
        gq.gq_set_dispatch_profile(gq.GQ_KIND_Q4_0, 64, 128, [16], [float("nan")], [2])
    gq.gq_clear_dispatch_profiles()
    assert gq.gq_choose_path(gq.GQ_KIND_Q4_0, 64, 128, 48) == gq.GQ_PATH_TC


@pytest.mark.parametrize("value,expected", [("24", 24), ("0", 0), ("-3", 16), ("abc", 16), ("12x", 16), (None, 16)])
def test_threshold_from_environment(value, expected):
    """GQ_M_THRESHOLD replaces the default M threshold when the library loads (a fresh
    process per case); values that are not non-negative integers leave the default."""
    import subprocess
    import sys
    env = dict(os.environ)
    env.pop("GQ_M_THRESHOLD", None)
    if value is not None:
        env["GQ_M_THRESHOLD"] = value
    code = "import quantized_skinny_matmul_gb300 as gq; print(gq.gq_get_m_threshold())"
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120,
                         cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert out.returncode == 0, out.stderr
    assert int(out.stdout.strip().splitlines()[-1]) == expected


def test_build_rejects_a_library_for_another_cpu(tmp_path):
    """An in-tree libgq.so built on another machine (the GPU machine is aarch64, this one may be
    x86-64) is not taken as up to date."""
    import platform
    from quantized_skinny_matmul_gb300 import _build
    this = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine().lower())
    if this is None:
        pytest.skip("unknown host CPU")
    other = 183 if this == 62 else 62
    for machine, want in ((this, True), (other, False)):
        f = tmp_path / f"lib{machine}.so"
        f.write_bytes(b"\x7fELF" + bytes(14) + machine.to_bytes(2, "little") + bytes(44))
        assert _build.built_for_this_machine(str(f)) is want
    assert _build.built_for_this_machine(str(tmp_path / "missing.so")) is False


def test_dispatch_takes_the_tiles_when_the_gemv_needs_several_slices(lib):
    """Without a profile, Q4_0 products of up to 16 rows take the GEMV unless its activation
    image needs several K slices for them (one launch per slice), as at K = 11008 with 9 or more
    rows; one row always takes the GEMV (no GPU involved)."""
    gq.gq_clear_dispatch_profiles()
    Q = gq.GQ_KIND_Q4_0
    for M in (1, 2, 8):
        assert gq.gq_choose_path(Q, 4096, 11008, M) == gq.GQ_PATH_GEMV, M
    for M in (9, 12, 16, 17, 64):
        assert gq.gq_choose_path(Q, 4096, 11008, M) == gq.GQ_PATH_TC, M
    for N, K in ((4096, 4096), (11008, 4096)):
        for M in (1, 8, 16):
            assert gq.gq_choose_path(Q, N, K, M) == gq.GQ_PATH_GEMV, (N, K, M)
        assert gq.gq_choose_path(Q, N, K, 17) == gq.GQ_PATH_TC
    assert gq.gq_choose_path(Q, 64, 100000, 1) == gq.GQ_PATH_GEMV


def test_dispatch_f16_takes_the_tiles_for_large_grids_or_images(lib):
    """Without a profile, F16 products take the GEMV only for fewer than 64 weight rows per SM
    and at most 64 KiB of fp16 activations (no GPU involved: the SM count then defaults to 148)."""
    gq.gq_clear_dispatch_profiles()
    F = gq.GQ_KIND_F16
    for M in (1, 4, 16):
        assert gq.gq_choose_path(F, 11008, 4096, M) == gq.GQ_PATH_TC, M
    for M in (1, 2):
        assert gq.gq_choose_path(F, 4096, 11008, M) == gq.GQ_PATH_GEMV, M
    for M in (3, 8, 16):
        assert gq.gq_choose_path(F, 4096, 11008, M) == gq.GQ_PATH_TC, M
    for M in (1, 8):
        assert gq.gq_choose_path(F, 4096, 4096, M) == gq.GQ_PATH_GEMV, M
    for M in (9, 16, 17):
        assert gq.gq_choose_path(F, 4096, 4096, M) == gq.GQ_PATH_TC, M
    assert gq.gq_choose_path(F, 4096, 40000, 1) == gq.GQ_PATH_TC


def test_argument_checks_kv_cache(lib):
    """The INT8 KV-cache entry points reject bad sizes, head counts and pointers before
    touching the GPU."""
    a = lib.gq_attn_decode_i8
    ok_args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 4, 64, 128, 0.1, None)
    for i, bad in ((9, 6), (9, 12), (9, 40), (10, 0), (8, 3), (8, 36)):   # Hq not G * Hkv, G in 1 .. 8
        args = list(ok_args)
        args[i] = bad
        assert a(*args) == gq.GQ_ERR_INVALID_ARG, (i, bad)
    for Hq, D in ((12, 64), (20, 64), (24, 64)):   # G = 3, 5, 6: the tensor-core kernel only (D = 128)
        args = list(ok_args)
        args[8], args[11] = Hq, D
        assert a(*args) == gq.GQ_ERR_INVALID_ARG, (Hq, D)
    for D in (32, 96, 256):
        args = list(ok_args)
        args[11] = D
        assert a(*args) == gq.GQ_ERR_INVALID_ARG
    for j in range(7):
        args = list(ok_args)
        args[j] = 0
        assert a(*args) == gq.GQ_ERR_INVALID_ARG
        args[j] = ODD
        assert a(*args) == gq.GQ_ERR_MISALIGNED
    args = list(ok_args)
    args[12] = float("inf")
    assert a(*args) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_kv_quantize_i8(FAKE, FAKE, FAKE, 0, 128, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_kv_quantize_i8(FAKE, FAKE, FAKE, 4, 48, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_kv_quantize_i8(FAKE, FAKE, ODD, 4, 64, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_kv_append_i8(FAKE, FAKE, FAKE, 0, 2, 4, 64, 128, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_kv_append_i8(FAKE, FAKE, FAKE, FAKE, 2, 4, 0, 128, None) == gq.GQ_ERR_INVALID_ARG
    assert lib.gq_kv_append_i8(FAKE, ODD, FAKE, FAKE, 2, 4, 64, 128, None) == gq.GQ_ERR_MISALIGNED
    assert lib.gq_last_error_message()


def test_debug_build_and_library_override(tmp_path):
    """The GQ_DEBUG build compiles (nvcc here, no GPU) into its own library, and the binding
    loads the library GQ_LIBRARY names."""
    from quantized_skinny_matmul_gb300 import _build
    path = _build.build(debug=True)
    assert path.endswith("libgq_debug.so") and os.path.exists(path) and path != _build.LIB_PATH
    code = ("import quantized_skinny_matmul_gb300 as gq; print(gq.LIB_PATH); "
            "print(gq.gq_abi_version()); print(gq.lib().gq_status_string(gq.GQ_ERR_DEVICE_CHECK).decode())")
    res = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, GQ_LIBRARY=path), cwd=ROOT,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    lines = res.stdout.split("\n")
    assert lines[0] == path and lines[1] == "1" and "bounds check" in lines[2]
