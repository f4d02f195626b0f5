"""Seeded synthetic inputs shared by the CUDA path's tests/benchmarks and the oracle.

Holds no arithmetic of the ternary method itself: it draws ternary values
t in {-1,0,+1}, FP16 group scales and BF16 activations from a counter-based
SplitMix64 stream (see ``synth.c``) and describes the workload shapes.

Workloads (shapes from the pages: the 0.6B embedding model of "Ternary
embedding model in vLLM" (2kiu.com/news/5082861) and the 48-layer,
8-KV-head Ternary-Bonsai-2-27B of "Ternary-Bonsai-2-27B TQ1_0 GGUF via
llama.cpp" (bhfrc.com/news/45317) §4.3):

* ``single``     one linear K=N=1024, P(0)=1/3, scales U[0.005,0.05]
* ``embed06b``   28 layers: qkv 1024->2048+1024+1024, o 2048->1024,
                 gate_up 1024->2x3072, down 3072->1024; P(0)=0.4, U[0.005,0.05]
* ``dec27b``     one layer: qkv 5120->5120+1024+1024, o 5120->5120,
                 gate_up 5120->2x27648, down 27648->5120; P(0)=0.35,
                 scales exp(N(-4, 0.5^2))
* ``stack27b``   dec27b repeated for 48 distinct layers
* ``prefill27b`` dec27b shapes at prefill batch sizes

Every tensor has its own stream, named ``"<workload>/<layer>/<linear>/<tensor>"``
and hashed with FNV-1a; the seed is 0 throughout.  Activations are drawn
row-major [M, K], so the first rows of a larger draw equal a smaller draw.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` with gcc + OpenMP."""
    src = os.path.join(_HERE, "synth.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.synth_ternary.argtypes = [u64, u64, dbl, vp, i64, i64]
            lib.synth_scales_uniform.argtypes = [u64, u64, dbl, dbl, vp, i64, i64]
            lib.synth_scales_lognormal.argtypes = [u64, u64, dbl, dbl, vp, i64, i64]
            lib.synth_normal_bf16.argtypes = [u64, u64, vp, i64, i64]
            lib.synth_uniform.argtypes = [u64, u64, vp, i64]
            lib.synth_raw.argtypes = [u64, u64, vp, i64]
            lib.synth_sequential_splitmix.argtypes = [u64, vp, i64]
            lib.synth_stream_key.argtypes = [u64, u64]
            lib.synth_stream_key.restype = u64
            lib.synth_round_fp16.argtypes = [dbl]
            lib.synth_round_fp16.restype = ctypes.c_uint16
            lib.synth_round_bf16.argtypes = [dbl]
            lib.synth_round_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def stream_id(name: str) -> int:
    """FNV-1a 64-bit hash of a stream name."""
    h = 0xCBF29CE484222325
    for b in name.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ----------------------------------------------------------------- raw draws

def ternary(stream: str, n: int, p_zero: float, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int8)
    _load().synth_ternary(seed, stream_id(stream), p_zero, _ptr(out), 0, n)
    return out


def scales_uniform(stream: str, n: int, lo: float, hi: float, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _load().synth_scales_uniform(seed, stream_id(stream), lo, hi, _ptr(out), 0, n)
    return out


def scales_lognormal(stream: str, n: int, mu: float, sigma: float, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _load().synth_scales_lognormal(seed, stream_id(stream), mu, sigma, _ptr(out), 0, n)
    return out


def normal_bf16(stream: str, n: int, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _load().synth_normal_bf16(seed, stream_id(stream), _ptr(out), 0, n)
    return out


def uniform(stream: str, n: int, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform(seed, stream_id(stream), _ptr(out), n)
    return out


def raw(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_raw(seed, stream, _ptr(out), n)
    return out


def sequential_splitmix(state: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_sequential_splitmix(state, _ptr(out), n)
    return out


def stream_key(seed: int, stream: int) -> int:
    return int(_load().synth_stream_key(seed, stream))


def round_fp16(x: float) -> int:
    return int(_load().synth_round_fp16(float(x)))


def round_bf16(x: float) -> int:
    return int(_load().synth_round_bf16(float(x)))


# ----------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Linear:
    """One linear layer Y[M, N] = X[M, K] . W^T, W = s (.) T with N = sum(splits)."""
    name: str
    K: int
    splits: tuple  # output widths; len > 1 means a fused multi-output linear

    @property
    def N(self) -> int:
        return int(sum(self.splits))


@dataclass(frozen=True)
class Workload:
    name: str
    linears: tuple
    layers: int
    p_zero: float
    scale_kind: str          # "uniform" or "lognormal"
    scale_args: tuple
    batch_sizes: tuple


_EMBED = (Linear("qkv", 1024, (2048, 1024, 1024)), Linear("o", 2048, (1024,)),
          Linear("gate_up", 1024, (3072, 3072)), Linear("down", 3072, (1024,)))
_DEC27 = (Linear("qkv", 5120, (5120, 1024, 1024)), Linear("o", 5120, (5120,)),
          Linear("gate_up", 5120, (27648, 27648)), Linear("down", 27648, (5120,)))

WORKLOADS = {
    "single": Workload("single", (Linear("linear", 1024, (1024,)),), 1, 1.0 / 3.0,
                       "uniform", (0.005, 0.05), (1, 8)),
    "embed06b": Workload("embed06b", _EMBED, 28, 0.4, "uniform", (0.005, 0.05), (1, 32, 512)),
    "dec27b": Workload("dec27b", _DEC27, 1, 0.35, "lognormal", (-4.0, 0.5), (1, 2, 4, 8, 16)),
    "stack27b": Workload("stack27b", _DEC27, 48, 0.35, "lognormal", (-4.0, 0.5),
                         (1, 32, 64, 128, 256)),
    "prefill27b": Workload("prefill27b", _DEC27, 48, 0.35, "lognormal", (-4.0, 0.5),
                           (1024, 2048, 4096)),
}

GROUP = 128  # weights along K that share one FP16 scale


def weights(wl: Workload, layer: int, lin: Linear, rows: slice | None = None):
    """Ternary values t int8 [N, K] and FP16 scale bits uint16 [N, K/128].

    ``rows`` draws only a contiguous row range (same values as the full draw).
    """
    N, K = lin.N, lin.K
    r0, r1 = (0, N) if rows is None else (rows.start or 0, rows.stop if rows.stop is not None else N)
    base = f"{wl.name}/{layer}/{lin.name}"
    lib = _load()
    t = np.empty((r1 - r0, K), dtype=np.int8)
    # draw the row range directly: element i of the stream is row i // K
    _draw_range(lib.synth_ternary, (0, stream_id(base + "/codes"), wl.p_zero), t, r0 * K)
    G = K // GROUP
    s = np.empty((r1 - r0, G), dtype=np.uint16)
    if wl.scale_kind == "uniform":
        _draw_range(lib.synth_scales_uniform, (0, stream_id(base + "/scales")) + wl.scale_args, s, r0 * G)
    else:
        _draw_range(lib.synth_scales_lognormal, (0, stream_id(base + "/scales")) + wl.scale_args, s, r0 * G)
    return t, s


def _draw_range(fn, args, out: np.ndarray, start: int):
    """Fill ``out`` with stream elements [start, start + out.size)."""
    fn(*args, _ptr(out), start, out.size)


def activations(wl: Workload, layer: int, lin: Linear, M: int) -> np.ndarray:
    """BF16 activation bits uint16 [M, K] ~ N(0,1)."""
    x = np.empty((M, lin.K), dtype=np.uint16)
    _load().synth_normal_bf16(0, stream_id(f"{wl.name}/{layer}/{lin.name}/x"), _ptr(x), 0, x.size)
    return x


def fp16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
