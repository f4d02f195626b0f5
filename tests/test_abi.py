"""Host-side checks of libtern's C ABI (no GPU needed).

The library must load, export every function include/tern.h declares, and
reject bad arguments with the documented status before touching the GPU.
"""
import ctypes
import os
import re
import subprocess

import pytest

import oracle
from conftest import ROOT

tbw = pytest.importorskip("ternary_bit_weight_gb300")
from ternary_bit_weight_gb300 import binding  # noqa: E402

HEADER = os.path.join(ROOT, "include", "tern.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tern_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(binding.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name


def test_status_strings_and_version():
    for code, name in binding.STATUS_NAMES.items():
        assert binding.status_string(code).startswith(name)
    assert binding.status_string(99) == "TERN_ERR_UNKNOWN"
    assert binding.tern_version() == 10100


@pytest.mark.parametrize("N,K", [(1, 128), (16, 128), (17, 256), (5120, 5120), (55296, 5120),
                                 (5120, 27648)])
def test_tiled_bytes_matches_layout(N, K):
    assert binding.tern_tiled_bytes(N, K) == oracle.tiled_bytes(N, K)


def test_tiled_bytes_rejects_bad_shapes():
    for N, K in [(-1, 128), (16, 0), (16, 100), (16, -128)]:
        assert binding.tern_tiled_bytes(N, K) == 0


def _raw(func, *args):
    return getattr(binding.library(), func)(*args)


FAKE = 1 << 40       # a 256-byte-aligned address that is never dereferenced


def test_pack_unpack_argument_errors():
    assert _raw("tern_pack", FAKE, 4, 6, FAKE, None, None) == 2      # K % 4
    assert _raw("tern_pack", FAKE, -1, 8, FAKE, None, None) == 2
    assert _raw("tern_pack", None, 4, 8, FAKE, None, None) == 1
    assert _raw("tern_pack", FAKE, 0, 8, None, None, None) == 0       # empty: no-op
    assert _raw("tern_pack", FAKE, 4, 8, FAKE, FAKE + 1, None) == 3   # misaligned counter
    assert _raw("tern_unpack", FAKE, 4, 6, FAKE, None, None) == 2
    assert _raw("tern_unpack", FAKE, 4, 8, None, None, None) == 1


def test_repack_argument_errors():
    need = binding.tern_tiled_bytes(32, 256)
    assert _raw("tern_repack", FAKE, FAKE, 32, 200, FAKE, need, None, None) == 2
    assert _raw("tern_repack", None, FAKE, 32, 256, FAKE, need, None, None) == 1
    assert _raw("tern_repack", FAKE, FAKE, 32, 256, FAKE + 8, need, None, None) == 3
    assert _raw("tern_repack", FAKE + 2, FAKE, 32, 256, FAKE, need, None, None) == 3
    assert _raw("tern_repack", FAKE, FAKE, 32, 256, FAKE, need - 1, None, None) == 4
    assert _raw("tern_repack", FAKE, FAKE, 0, 256, FAKE, 0, None, None) == 0
    assert _raw("tern_unrepack", FAKE, 32, 100, FAKE, FAKE, None, None) == 2
    assert _raw("tern_unrepack", FAKE, 32, 256, None, FAKE, None, None) == 1


def test_linear_argument_errors():
    f = "tern_linear"
    # shape: K not a multiple of 128, negative M, ldx < K, ldy < N
    assert _raw(f, FAKE, 256, FAKE, 1, 64, 200, FAKE, 64, None, 0, None) == 2
    assert _raw(f, FAKE, 256, FAKE, -1, 64, 256, FAKE, 64, None, 0, None) == 2
    assert _raw(f, FAKE, 128, FAKE, 1, 64, 256, FAKE, 64, None, 0, None) == 2
    assert _raw(f, FAKE, 256, FAKE, 1, 64, 256, FAKE, 63, None, 0, None) == 2
    # empty problems are no-ops
    assert _raw(f, None, 256, None, 0, 64, 256, None, 64, None, 0, None) == 0
    assert _raw(f, None, 256, None, 4, 0, 256, None, 0, None, 0, None) == 0
    # null pointers
    assert _raw(f, None, 256, FAKE, 1, 64, 256, FAKE, 64, None, 0, None) == 1
    assert _raw(f, FAKE, 256, None, 1, 64, 256, FAKE, 64, None, 0, None) == 1
    assert _raw(f, FAKE, 256, FAKE, 1, 64, 256, None, 64, None, 0, None) == 1
    # alignment: X 16 B, ldx % 8, tiled 16 B, Y 4 B
    assert _raw(f, FAKE + 2, 256, FAKE, 1, 64, 256, FAKE, 64, None, 0, None) == 3
    assert _raw(f, FAKE, 260, FAKE, 1, 64, 256, FAKE, 64, None, 0, None) == 3
    assert _raw(f, FAKE, 256, FAKE + 4, 1, 64, 256, FAKE, 64, None, 0, None) == 3
    assert _raw(f, FAKE, 256, FAKE, 1, 64, 256, FAKE + 2, 64, None, 0, None) == 3


def test_linear_multi_argument_errors():
    lib = binding.library()
    i64 = ctypes.c_int64
    sizes = (i64 * 2)(64, 64)
    ptrs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    lds = (i64 * 2)(64, 64)
    f = lib.tern_linear_multi
    assert f(FAKE, 256, FAKE, 1, 256, 0, sizes, ptrs, lds, None, 0, None) == 2   # n_out
    assert f(FAKE, 256, FAKE, 1, 256, 5, sizes, ptrs, lds, None, 0, None) == 2
    assert f(FAKE, 256, FAKE, 1, 256, 2, None, ptrs, lds, None, 0, None) == 1
    bad = (i64 * 2)(64, -1)
    assert f(FAKE, 256, FAKE, 1, 256, 2, bad, ptrs, lds, None, 0, None) == 2
    small_ld = (i64 * 2)(64, 32)
    assert f(FAKE, 256, FAKE, 1, 256, 2, sizes, ptrs, small_ld, None, 0, None) == 2
    nullp = (ctypes.c_void_p * 2)(FAKE, None)
    assert f(FAKE, 256, FAKE, 1, 256, 2, sizes, nullp, lds, None, 0, None) == 1
    assert f(FAKE, 256, FAKE, 1, 200, 2, sizes, ptrs, lds, None, 0, None) == 2   # K % 128


def test_workspace_bytes_is_zero_for_empty_or_invalid():
    assert binding.tern_workspace_bytes(0, 64, 256) == 0
    assert binding.tern_workspace_bytes(4, 0, 256) == 0
    assert binding.tern_workspace_bytes(4, 64, 100) == 0


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "ternary_bit_weight_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.replace("oracle_", ""), fn


def test_linear_ex_and_swiglu_argument_errors():
    lib = binding.library()
    i64 = ctypes.c_int64
    sizes = (i64 * 1)(64)
    ptrs = (ctypes.c_void_p * 1)(FAKE)
    lds = (i64 * 1)(64)
    f = lib.tern_linear_ex
    assert f(FAKE, 2, 256, FAKE, 1, 256, 1, sizes, ptrs, lds, 0, None, 0, None) == 2    # x_type
    assert f(FAKE, 0, 256, FAKE, 1, 256, 1, sizes, ptrs, lds, 3, None, 0, None) == 2    # out_type
    odd = (ctypes.c_void_p * 1)(FAKE + 2)
    assert f(FAKE, 0, 256, FAKE, 1, 256, 1, sizes, odd, lds, 0, None, 0, None) == 3     # fp32 needs 4 B
    assert f(FAKE, 1, 256, FAKE, 1, 256, 1, sizes, ptrs, lds, 3, None, 0, None) == 2
    g = lib.tern_linear_swiglu
    assert g(FAKE, 0, 256, FAKE, 1, 64, 256, FAKE, 63, 1, None, 0, None) == 2           # ldh < I
    assert g(FAKE, 0, 256, FAKE, 1, 64, 200, FAKE, 64, 1, None, 0, None) == 2           # K % 128
    assert g(FAKE, 0, 256, FAKE, 1, 64, 256, None, 64, 1, None, 0, None) == 1
    assert g(FAKE, 0, 256, FAKE, 1, 64, 256, FAKE + 1, 64, 1, None, 0, None) == 3
    assert g(FAKE, 0, 256, FAKE, 1, 64, 256, FAKE + 2, 64, 0, None, 0, None) == 3       # fp32 H
    assert g(None, 0, 256, None, 0, 64, 256, None, 64, 1, None, 0, None) == 0           # M == 0


def test_glu_sizes_follow_the_layout():
    for I, K in [(1, 128), (16, 256), (20, 256), (27648, 5120), (3072, 1024)]:
        rows = oracle.glu_rows(I)
        assert binding.tern_tiled_glu_bytes(I, K) == oracle.tiled_bytes(rows, K)
        assert binding.tern_swiglu_workspace_bytes(4, I, K) == binding.tern_workspace_bytes(4, rows, K)
    need = binding.tern_tiled_glu_bytes(20, 256)
    r = binding.library().tern_repack_glu
    assert r(FAKE, FAKE, FAKE, FAKE, 20, 200, FAKE, need, None, None) == 2
    assert r(FAKE, FAKE, None, FAKE, 20, 256, FAKE, need, None, None) == 1
    assert r(FAKE, FAKE, FAKE + 2, FAKE, 20, 256, FAKE, need, None, None) == 3
    assert r(FAKE, FAKE, FAKE, FAKE, 20, 256, FAKE, need - 1, None, None) == 4


def test_workspace_maintenance_argument_errors():
    lib = binding.library()
    out = ctypes.c_int32(0)
    assert lib.tern_workspace_error(None, ctypes.addressof(out), None) == 1
    assert lib.tern_workspace_error(FAKE, None, None) == 1
    assert lib.tern_workspace_error(FAKE + 16, ctypes.addressof(out), None) == 3
    assert lib.tern_workspace_reset(None, 256, None) == 1
    assert lib.tern_workspace_reset(FAKE + 16, 256, None) == 3
    assert lib.tern_workspace_reset(FAKE, 0, None) == 0


def test_i8_argument_errors():
    lib = binding.library()
    assert binding.tern_xq_bytes(3, 256) == 768 and binding.tern_xq_bytes(3, 100) == 0
    q = lib.tern_quantize_x
    assert q(FAKE, 2, 256, 1, 256, FAKE, FAKE, None) == 2          # x_type
    assert q(FAKE, 0, 128, 1, 256, FAKE, FAKE, None) == 2          # ldx < K
    assert q(FAKE, 0, 256, 1, 256, None, FAKE, None) == 1
    assert q(FAKE, 0, 256, 1, 256, FAKE + 8, FAKE, None) == 3      # xq 16 B
    assert q(None, 0, 256, 0, 256, None, None, None) == 0          # M == 0
    f = lib.tern_linear_i8
    assert f(FAKE, FAKE, FAKE, 1, 64, 200, FAKE, 64, 0, FAKE, 1 << 20, None) == 2
    assert f(FAKE, FAKE, FAKE, 1, 64, 256, FAKE, 64, 7, FAKE, 1 << 20, None) == 2
    assert f(FAKE, None, FAKE, 1, 64, 256, FAKE, 64, 0, FAKE, 1 << 20, None) == 1
    assert f(FAKE, FAKE, FAKE, 1, 64, 256, FAKE + 2, 64, 0, FAKE, 1 << 20, None) == 3
    assert f(FAKE, FAKE, FAKE, 1, 64, 256, FAKE, 63, 0, FAKE, 1 << 20, None) == 2
    assert binding.tern_i8_workspace_bytes(1, 64, 256) >= 256


def test_s8_sizes_and_argument_errors():
    for N, K in [(1, 128), (130, 256), (55296, 5120)]:
        R, G = (N + 127) // 128, K // 128
        assert binding.tern_tiled_s8_bytes(N, K) == oracle.tiled_s8_bytes(N, K) == R * G * 4224 + R * 512
    lib = binding.library()
    need = binding.tern_tiled_s8_bytes(32, 256)
    assert lib.tern_repack_s8(FAKE, FAKE, FAKE, 32, 200, FAKE, need, None, None) == 2
    assert lib.tern_repack_s8(FAKE, None, FAKE, 32, 256, FAKE, need, None, None) == 1
    assert lib.tern_repack_s8(FAKE, FAKE, FAKE, 32, 256, FAKE, need - 1, None, None) == 4
    assert lib.tern_quantize_scales(FAKE, 32, 256, FAKE, FAKE + 2, None) == 3
    assert lib.tern_quantize_scales(FAKE, 32, 100, FAKE, FAKE, None) == 2


def test_grouped_sizes_and_argument_errors():
    lib = binding.library()
    i64 = ctypes.c_int64
    vp = ctypes.c_void_p

    def arr(t, vals):
        return (t * len(vals))(*vals)

    Ns, Ks = arr(i64, [256, 512]), arr(i64, [256, 1024])
    ws_fn = lib.tern_grouped_workspace_bytes
    assert ws_fn(1, 2, Ns, Ks) > 0
    assert ws_fn(1, 2, Ns, Ks) >= binding.tern_workspace_bytes(1, 512, 1024)
    # M > 16: one GEMM launch for the group, so the workspace holds every
    # problem's fp16 activations (40 x K x 2 bytes each) at once (its K
    # splits are planned for the group, not per problem)
    assert ws_fn(40, 2, Ns, Ks) >= 256 + 40 * 256 * 2 + 40 * 1024 * 2
    assert ws_fn(1, 0, Ns, Ks) == 0
    assert ws_fn(1, binding.MAX_GROUP + 1, Ns, Ks) == 0
    assert ws_fn(1, 1, arr(i64, [256]), arr(i64, [200])) == 0     # K % 128
    assert ws_fn(0, 2, Ns, Ks) == 0
    f = lib.tern_linear_grouped
    X, W, Y = arr(vp, [FAKE, FAKE]), arr(vp, [FAKE, FAKE]), arr(vp, [FAKE, FAKE])
    ld = arr(i64, [1024, 1024])
    assert f(2, 1, 2, X, ld, W, Ns, Ks, Y, ld, 0, None, 0, None) == 2            # x_type
    assert f(0, 1, 2, X, ld, W, Ns, Ks, Y, ld, 3, None, 0, None) == 2            # out_type
    assert f(0, 1, 0, X, ld, W, Ns, Ks, Y, ld, 0, None, 0, None) == 2            # count
    assert f(0, 1, binding.MAX_GROUP + 1, X, ld, W, Ns, Ks, Y, ld, 0, None, 0, None) == 2
    assert f(0, 1, 2, None, ld, W, Ns, Ks, Y, ld, 0, None, 0, None) == 1         # host arrays
    assert f(0, 1, 2, X, ld, W, Ns, arr(i64, [256, 100]), Y, ld, 0, None, 0, None) == 2
    assert f(0, 1, 2, X, arr(i64, [255, 1024]), W, Ns, Ks, Y, ld, 0, None, 0, None) == 2   # ldx < K
    assert f(0, 1, 2, arr(vp, [FAKE + 2, FAKE]), ld, W, Ns, Ks, Y, ld, 0, None, 0, None) == 3
    assert f(0, 1, 2, X, ld, W, Ns, Ks, arr(vp, [FAKE, None]), ld, 0, None, 0, None) == 1
    assert f(0, 1, 2, X, ld, W, Ns, Ks, Y, arr(i64, [1024, 511]), 0, None, 0, None) == 2  # ldy < N
    assert f(0, 1, 2, X, ld, W, Ns, Ks, arr(vp, [FAKE + 2, FAKE]), ld, 0, None, 0, None) == 3   # fp32 Y
    assert f(0, 0, 2, X, ld, W, Ns, Ks, Y, ld, 0, None, 0, None) == 0            # M == 0
    assert f(0, 1, 1, X, ld, W, arr(i64, [0]), Ks, Y, ld, 0, None, 0, None) == 0  # N == 0 only


def test_repack_grouped_argument_errors():
    lib = binding.library()
    i64, vp, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t

    def arr(t, vals):
        return (t * len(vals))(*vals)

    P, S, T = arr(vp, [FAKE, FAKE]), arr(vp, [FAKE, FAKE]), arr(vp, [FAKE, FAKE])
    Ns, Ks = arr(i64, [256, 100]), arr(i64, [256, 512])
    big = arr(sz, [1 << 30, 1 << 30])
    f = lib.tern_repack_grouped
    assert f(0, P, S, Ns, Ks, T, big, None, None) == 2                       # count
    assert f(binding.MAX_GROUP + 1, P, S, Ns, Ks, T, big, None, None) == 2
    assert f(2, None, S, Ns, Ks, T, big, None, None) == 1                    # host arrays
    assert f(2, P, S, Ns, arr(i64, [256, 200]), T, big, None, None) == 2      # K % 128
    assert f(2, P, S, Ns, Ks, T, arr(sz, [1 << 30, 16]), None, None) == 4    # tiled too small
    assert f(2, arr(vp, [FAKE, FAKE + 2]), S, Ns, Ks, T, big, None, None) == 3   # packed 4-byte aligned
    assert f(2, P, S, Ns, Ks, arr(vp, [FAKE, FAKE + 8]), big, None, None) == 3   # tiled 16-byte aligned
    assert f(2, P, arr(vp, [FAKE, None]), Ns, Ks, T, big, None, None) == 1
    assert f(1, P, S, arr(i64, [0]), Ks, T, big, None, None) == 0            # N == 0: nothing to do
