"""CPU oracle for the ternary-weight linear layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never
does and has no fallback to it.

The arithmetic lives in ``oracle.c`` (plain C, fp64), written from the
pages' packing rule and the plain definition of the layer; this module only
compiles it with gcc and marshals numpy arrays.  Its pins (the checks that
tie it to the pages and to mathematics rather than to itself) are in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP)."""
    src = os.path.join(_HERE, "oracle.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps x*w and the fp64 sums as separately rounded ops
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                           "-std=c11", "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, vp, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.orc_fp16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_fp16_to_double.restype = dbl
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = dbl
            lib.orc_code_to_ternary.argtypes = [ctypes.c_uint]
            lib.orc_code_to_ternary.restype = ctypes.c_int
            lib.orc_pack.argtypes = [vp, i64, i64, vp]
            lib.orc_pack.restype = i64
            lib.orc_unpack.argtypes = [vp, i64, i64, vp]
            lib.orc_unpack.restype = i64
            lib.orc_tiled_bytes.argtypes = [i64, i64]
            lib.orc_tiled_bytes.restype = i64
            lib.orc_repack.argtypes = [vp, vp, i64, i64, vp]
            lib.orc_repack.restype = i64
            lib.orc_unrepack.argtypes = [vp, i64, i64, vp, vp]
            lib.orc_unrepack.restype = i64
            lib.orc_linear.argtypes = [vp, i64, vp, vp, i64, i64, i64, vp, vp]
            lib.orc_linear.restype = None
            lib.orc_linear_cols.argtypes = [vp, i64, vp, vp, i64, i64, i64, vp, i64, vp, vp]
            lib.orc_linear_cols.restype = None
            lib.orc_linear_x.argtypes = [vp, ctypes.c_int, i64, vp, vp, i64, i64, i64, vp, vp]
            lib.orc_linear_x.restype = None
            lib.orc_linear_cols_x.argtypes = [vp, ctypes.c_int, i64, vp, vp, i64, i64, i64, vp, i64, vp, vp]
            lib.orc_linear_cols_x.restype = None
            lib.orc_quantize_scales.argtypes = [vp, i64, i64, vp, vp]
            lib.orc_quantize_scales.restype = None
            lib.orc_linear_s8.argtypes = [vp, i64, vp, vp, vp, i64, i64, i64, vp, vp]
            lib.orc_linear_s8.restype = None
            lib.orc_quantize_x.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, vp]
            lib.orc_quantize_x.restype = None
            lib.orc_linear_i8.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp]
            lib.orc_linear_i8.restype = None
            lib.orc_swiglu.argtypes = [vp, vp, i64, vp]
            lib.orc_swiglu.restype = None
            lib.orc_num_threads.argtypes = []
            lib.orc_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def fp16_to_double(bits: int) -> float:
    return float(_load().orc_fp16_to_double(bits))


def bf16_to_double(bits: int) -> float:
    return float(_load().orc_bf16_to_double(bits))


def code_to_ternary(code: int) -> int:
    return int(_load().orc_code_to_ternary(code))


def pack(t: np.ndarray):
    """t int8 [N, K] -> (packed uint8 [N, K/4], number of invalid entries)."""
    t = _c(t, np.int8)
    N, K = t.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    out = np.empty((N, K // 4), dtype=np.uint8)
    bad = _load().orc_pack(t.ctypes.data, N, K, out.ctypes.data)
    return out, int(bad)


def unpack(packed: np.ndarray, K: int):
    """packed uint8 [N, K/4] -> (t int8 [N, K], number of reserved code-11 entries)."""
    packed = _c(packed, np.uint8)
    N = packed.shape[0]
    out = np.empty((N, K), dtype=np.int8)
    bad = _load().orc_unpack(packed.ctypes.data, N, K, out.ctypes.data)
    return out, int(bad)


def tiled_bytes(N: int, K: int) -> int:
    return int(_load().orc_tiled_bytes(N, K))


def repack(packed: np.ndarray, scales: np.ndarray, K: int):
    """(packed [N,K/4], fp16 bits [N,K/128]) -> (tiled uint8 bytes, reserved count)."""
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint16)
    N = packed.shape[0]
    out = np.empty(tiled_bytes(N, K), dtype=np.uint8)
    bad = _load().orc_repack(packed.ctypes.data, scales.ctypes.data, N, K, out.ctypes.data)
    return out, int(bad)


def unrepack(tiled: np.ndarray, N: int, K: int):
    """tiled bytes -> (packed [N,K/4], fp16 bits [N,K/128], invalid count)."""
    tiled = _c(tiled, np.uint8)
    packed = np.empty((N, K // 4), dtype=np.uint8)
    scales = np.empty((N, K // 128), dtype=np.uint16)
    bad = _load().orc_unrepack(tiled.ctypes.data, N, K, packed.ctypes.data, scales.ctypes.data)
    return packed, scales, int(bad)


def linear(x_bits: np.ndarray, packed: np.ndarray, scales: np.ndarray, K: int, x_f16: bool = False):
    """Y[M, N] = X . (s (.) T)^T in fp64, and the per-output bound sum_k |x w|.
    X holds bf16 bits, or fp16 bits with ``x_f16``."""
    x = _c(x_bits, np.uint16)
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint16)
    M, N = x.shape[0], packed.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64)
    _load().orc_linear_x(x.ctypes.data, int(x_f16), K, packed.ctypes.data, scales.ctypes.data,
                         M, N, K, y.ctypes.data, b.ctypes.data)
    return y, b


def linear_cols(x_bits: np.ndarray, packed: np.ndarray, scales: np.ndarray, K: int, cols,
                x_f16: bool = False):
    """Like ``linear`` for the output columns ``cols`` only: returns [M, len(cols)]."""
    x = _c(x_bits, np.uint16)
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint16)
    cols = _c(np.asarray(cols), np.int64)
    M, N = x.shape[0], packed.shape[0]
    y = np.empty((M, cols.size), dtype=np.float64)
    b = np.empty((M, cols.size), dtype=np.float64)
    _load().orc_linear_cols_x(x.ctypes.data, int(x_f16), K, packed.ctypes.data, scales.ctypes.data,
                              M, N, K, cols.ctypes.data, cols.size, y.ctypes.data, b.ctypes.data)
    return y, b


def quantize_scales(scales: np.ndarray, K: int):
    """FP16 scale bits [N, K/128] -> (q8 int8 [N, K/128], f fp32 [N])."""
    scales = _c(scales, np.uint16)
    N = scales.shape[0]
    q8 = np.empty((N, K // 128), dtype=np.int8)
    f = np.empty(N, dtype=np.float32)
    _load().orc_quantize_scales(scales.ctypes.data, N, K, q8.ctypes.data, f.ctypes.data)
    return q8, f


def tiled_s8_bytes(N: int, K: int) -> int:
    R, G = (N + 127) // 128, K // 128
    return R * G * (4096 + 128) + R * 128 * 4


def repack_s8(packed: np.ndarray, q8: np.ndarray, f: np.ndarray, K: int) -> np.ndarray:
    """INT8-scale tile layout: the tiled layout's code units, then per unit
    (b, g) the bytes q8[128b + r][g], then per row tile the fp32 f[128b + r]
    (padding rows 0)."""
    packed = _c(packed, np.uint8)
    N = packed.shape[0]
    R, G = (N + 127) // 128, K // 128
    zero_scales = np.zeros((N, G), dtype=np.uint16)
    tiled, _ = repack(packed, zero_scales, K)
    codes = tiled[:R * G * 4096]
    q = np.zeros((R * 128, G), dtype=np.int8)
    q[:N] = q8
    units = np.empty((R, G, 128), dtype=np.int8)
    for b in range(R):
        for g in range(G):
            units[b, g] = q[128 * b:128 * b + 128, g]
    fac = np.zeros(R * 128, dtype=np.float32)
    fac[:N] = f
    return np.concatenate([codes, units.reshape(-1).view(np.uint8), fac.view(np.uint8)])


def linear_s8(x_bits: np.ndarray, packed: np.ndarray, q8: np.ndarray, f: np.ndarray, K: int):
    """Y = X . (q8 * f (.) T)^T in fp64 and its bound."""
    x = _c(x_bits, np.uint16)
    packed = _c(packed, np.uint8)
    q8 = _c(q8, np.int8)
    f = _c(f, np.float32)
    M, N = x.shape[0], packed.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64)
    _load().orc_linear_s8(x.ctypes.data, K, packed.ctypes.data, q8.ctypes.data, f.ctypes.data, M, N, K,
                          y.ctypes.data, b.ctypes.data)
    return y, b


def quantize_x(x_bits: np.ndarray, x_f16: bool = False):
    """Per-token absmax int8: (q int8 [M, K] in k order, a fp32 [M])."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.int8)
    a = np.empty(M, dtype=np.float32)
    _load().orc_quantize_x(x.ctypes.data, int(x_f16), K, M, K, q.ctypes.data, a.ctypes.data)
    return q, a


def linear_i8(q: np.ndarray, a: np.ndarray, packed: np.ndarray, scales: np.ndarray, K: int):
    """Y = a * sum_g s * (exact integer group sums of t q), and its bound."""
    q = _c(q, np.int8)
    a = _c(a, np.float32)
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint16)
    M, N = q.shape[0], packed.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64)
    _load().orc_linear_i8(q.ctypes.data, a.ctypes.data, packed.ctypes.data, scales.ctypes.data, M, N, K,
                          y.ctypes.data, b.ctypes.data)
    return y, b


def zero_units(packed: np.ndarray, K: int) -> np.ndarray:
    """Per unit (128 rows x 128 weights, rows padded to a multiple of 128
    with zeros, index b*G + g): 1 if every weight is 0 (codes 00 or 11)."""
    t, _ = unpack(packed, K)
    N = t.shape[0]
    R, G = (N + 127) // 128, K // 128
    pad = np.zeros((R * 128, K), dtype=np.int8)
    pad[:N] = t
    blocks = pad.reshape(R, 128, G, 128)
    return (~blocks.any(axis=(1, 3))).astype(np.uint8).reshape(-1)


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g) * u elementwise in fp64 (silu(g) = g / (1 + e^-g))."""
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    h = np.empty_like(g)
    _load().orc_swiglu(g.ctypes.data, u.ctypes.data, g.size, h.ctypes.data)
    return h


def glu_rows(I: int) -> int:
    """Rows of the GLU tile layout: 2 * ceil(I/16) * 16."""
    return 2 * ((I + 15) // 16) * 16


def glu_source(n: int):
    """Source of GLU row n: ('gate' or 'up', row index), from the layout's
    definition (blocks of 16 rows alternating between gate and up)."""
    block, j = divmod(n, 32)
    return ("gate" if j < 16 else "up"), 16 * block + (j % 16)


def repack_glu(packed_gate, scales_gate, packed_up, scales_up, K: int):
    """(gate, up) on-disk pairs of I rows -> GLU tile layout bytes: the
    interleaved weight assembled row by row, then ``repack``."""
    packed_gate = _c(packed_gate, np.uint8)
    packed_up = _c(packed_up, np.uint8)
    I = packed_gate.shape[0]
    rows = glu_rows(I)
    packed = np.zeros((rows, K // 4), dtype=np.uint8)
    scales = np.zeros((rows, K // 128), dtype=np.uint16)
    for n in range(rows):
        which, i = glu_source(n)
        if i < I:
            packed[n] = (packed_gate if which == "gate" else packed_up)[i]
            scales[n] = (scales_gate if which == "gate" else scales_up)[i]
    return repack(packed, scales, K)


def num_threads() -> int:
    return int(_load().orc_num_threads())
