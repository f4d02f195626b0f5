"""ctypes binding of libtern's C ABI (include/tern.h).

Argument marshalling only: every step of the layer runs in libtern's CUDA
kernels.  Functions carry the C names; tensor arguments may be torch
tensors (their ``data_ptr()`` is passed) or raw integer addresses, and
``stream`` may be a ``torch.cuda.Stream``, a raw ``cudaStream_t`` integer or
None (the current torch stream).  A non-zero status raises ``TernError``.
If the library has not been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

TERN_OK = 0
TERN_X_BF16, TERN_X_F16 = 0, 1
TERN_OUT_F32, TERN_OUT_BF16, TERN_OUT_F16 = 0, 1, 2
STATUS_NAMES = {0: "TERN_OK", 1: "TERN_ERR_NULL", 2: "TERN_ERR_SHAPE", 3: "TERN_ERR_ALIGN",
                4: "TERN_ERR_SIZE", 5: "TERN_ERR_UNSUPPORTED", 6: "TERN_ERR_CUDA"}

# Every symbol include/tern.h declares.
EXPORTED = ("tern_status_string", "tern_version", "tern_pack", "tern_unpack", "tern_tiled_bytes",
            "tern_repack", "tern_unrepack", "tern_workspace_bytes", "tern_linear",
            "tern_linear_multi", "tern_linear_noalloc", "tern_linear_ex", "tern_tiled_glu_bytes",
            "tern_repack_glu", "tern_swiglu_workspace_bytes", "tern_linear_swiglu",
            "tern_workspace_error", "tern_workspace_reset", "tern_xq_bytes", "tern_quantize_x",
            "tern_i8_workspace_bytes", "tern_linear_i8", "tern_tiled_s8_bytes", "tern_quantize_scales",
            "tern_repack_s8", "tern_linear_s8", "tern_unit_count", "tern_zero_units", "tern_linear_sparse",
            "tern_grouped_workspace_bytes", "tern_linear_grouped", "tern_repack_grouped")

MAX_GROUP = 8


class TernError(RuntimeError):
    def __init__(self, status: int, func: str):
        self.status = status
        super().__init__(f"{func}: {status_string(status)}")


def _load():
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libtern.so is not built ({_build.LIB}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_build.LIB)
    i64, vp, sz, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.tern_status_string.argtypes = [i32]
    lib.tern_status_string.restype = ctypes.c_char_p
    lib.tern_version.argtypes = []
    lib.tern_version.restype = i32
    lib.tern_pack.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.tern_pack.restype = i32
    lib.tern_unpack.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.tern_unpack.restype = i32
    lib.tern_tiled_bytes.argtypes = [i64, i64]
    lib.tern_tiled_bytes.restype = sz
    lib.tern_repack.argtypes = [vp, vp, i64, i64, vp, sz, vp, vp]
    lib.tern_repack.restype = i32
    lib.tern_unrepack.argtypes = [vp, i64, i64, vp, vp, vp, vp]
    lib.tern_unrepack.restype = i32
    lib.tern_workspace_bytes.argtypes = [i64, i64, i64]
    lib.tern_workspace_bytes.restype = sz
    lib.tern_linear.argtypes = [vp, i64, vp, i64, i64, i64, vp, i64, vp, sz, vp]
    lib.tern_linear.restype = i32
    lib.tern_linear_multi.argtypes = [vp, i64, vp, i64, i64, i32, ctypes.POINTER(i64),
                                      ctypes.POINTER(vp), ctypes.POINTER(i64), vp, sz, vp]
    lib.tern_linear_multi.restype = i32
    lib.tern_linear_noalloc.argtypes = [vp, i64, vp, i64, i64, i64, vp, i64, vp]
    lib.tern_linear_noalloc.restype = i32
    lib.tern_linear_ex.argtypes = [vp, i32, i64, vp, i64, i64, i32, ctypes.POINTER(i64),
                                   ctypes.POINTER(vp), ctypes.POINTER(i64), i32, vp, sz, vp]
    lib.tern_linear_ex.restype = i32
    lib.tern_grouped_workspace_bytes.argtypes = [i64, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.tern_grouped_workspace_bytes.restype = sz
    lib.tern_linear_grouped.argtypes = [i32, i64, i32, ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(vp),
                                        ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(vp),
                                        ctypes.POINTER(i64), i32, vp, sz, vp]
    lib.tern_linear_grouped.restype = i32
    lib.tern_repack_grouped.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64),
                                        ctypes.POINTER(i64), ctypes.POINTER(vp), ctypes.POINTER(sz), vp, vp]
    lib.tern_repack_grouped.restype = i32
    lib.tern_tiled_glu_bytes.argtypes = [i64, i64]
    lib.tern_tiled_glu_bytes.restype = sz
    lib.tern_repack_glu.argtypes = [vp, vp, vp, vp, i64, i64, vp, sz, vp, vp]
    lib.tern_repack_glu.restype = i32
    lib.tern_swiglu_workspace_bytes.argtypes = [i64, i64, i64]
    lib.tern_swiglu_workspace_bytes.restype = sz
    lib.tern_linear_swiglu.argtypes = [vp, i32, i64, vp, i64, i64, i64, vp, i64, i32, vp, sz, vp]
    lib.tern_linear_swiglu.restype = i32
    lib.tern_workspace_error.argtypes = [vp, vp, vp]
    lib.tern_workspace_error.restype = i32
    lib.tern_workspace_reset.argtypes = [vp, sz, vp]
    lib.tern_workspace_reset.restype = i32
    lib.tern_xq_bytes.argtypes = [i64, i64]
    lib.tern_xq_bytes.restype = sz
    lib.tern_quantize_x.argtypes = [vp, i32, i64, i64, i64, vp, vp, vp]
    lib.tern_quantize_x.restype = i32
    lib.tern_i8_workspace_bytes.argtypes = [i64, i64, i64]
    lib.tern_i8_workspace_bytes.restype = sz
    lib.tern_linear_i8.argtypes = [vp, vp, vp, i64, i64, i64, vp, i64, i32, vp, sz, vp]
    lib.tern_linear_i8.restype = i32
    lib.tern_tiled_s8_bytes.argtypes = [i64, i64]
    lib.tern_tiled_s8_bytes.restype = sz
    lib.tern_quantize_scales.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.tern_quantize_scales.restype = i32
    lib.tern_repack_s8.argtypes = [vp, vp, vp, i64, i64, vp, sz, vp, vp]
    lib.tern_repack_s8.restype = i32
    lib.tern_linear_s8.argtypes = list(lib.tern_linear_ex.argtypes)
    lib.tern_linear_s8.restype = i32
    lib.tern_unit_count.argtypes = [i64, i64]
    lib.tern_unit_count.restype = sz
    lib.tern_zero_units.argtypes = [vp, i64, i64, vp, vp]
    lib.tern_zero_units.restype = i32
    lib.tern_linear_sparse.argtypes = [vp, i32, i64, vp, vp, i64, i64, i32, ctypes.POINTER(i64),
                                       ctypes.POINTER(vp), ctypes.POINTER(i64), i32, vp, sz, vp]
    lib.tern_linear_sparse.restype = i32
    return lib


_lib = _load()


def library():
    """The loaded ctypes library object."""
    return _lib


def library_path() -> str:
    return _build.LIB


def _p(x):
    """Device/host address of a tensor or an int (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, func: str):
    if status != TERN_OK:
        raise TernError(status, func)


def status_string(status: int) -> str:
    return _lib.tern_status_string(status).decode()


def tern_status_string(status: int) -> str:
    return status_string(status)


def tern_version() -> int:
    return int(_lib.tern_version())


def tern_pack(t, N: int, K: int, packed, err=None, stream=None):
    _check(_lib.tern_pack(_p(t), N, K, _p(packed), _p(err), _s(stream)), "tern_pack")


def tern_unpack(packed, N: int, K: int, t, err=None, stream=None):
    _check(_lib.tern_unpack(_p(packed), N, K, _p(t), _p(err), _s(stream)), "tern_unpack")


def tern_tiled_bytes(N: int, K: int) -> int:
    return int(_lib.tern_tiled_bytes(N, K))


def tern_repack(packed, scales, N: int, K: int, tiled, tiled_bytes: int | None = None, err=None,
                stream=None):
    if tiled_bytes is None:
        tiled_bytes = tiled.numel() * tiled.element_size()
    _check(_lib.tern_repack(_p(packed), _p(scales), N, K, _p(tiled), tiled_bytes, _p(err), _s(stream)),
           "tern_repack")


def tern_unrepack(tiled, N: int, K: int, packed, scales, err=None, stream=None):
    _check(_lib.tern_unrepack(_p(tiled), N, K, _p(packed), _p(scales), _p(err), _s(stream)),
           "tern_unrepack")


def tern_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_lib.tern_workspace_bytes(M, N, K))


def tern_linear(X, ldx: int, tiled, M: int, N: int, K: int, Y, ldy: int, ws=None,
                ws_bytes: int | None = None, stream=None):
    if ws_bytes is None:
        ws_bytes = 0 if ws is None or isinstance(ws, int) else ws.numel() * ws.element_size()
    _check(_lib.tern_linear(_p(X), ldx, _p(tiled), M, N, K, _p(Y), ldy, _p(ws), ws_bytes, _s(stream)),
           "tern_linear")


def tern_linear_multi(X, ldx: int, tiled, M: int, K: int, n_sizes, Ys, ldys, ws=None,
                      ws_bytes: int | None = None, stream=None):
    n_out = len(n_sizes)
    sizes = (ctypes.c_int64 * n_out)(*[int(v) for v in n_sizes])
    ptrs = (ctypes.c_void_p * n_out)(*[_p(y) for y in Ys])
    lds = (ctypes.c_int64 * n_out)(*[int(v) for v in ldys])
    if ws_bytes is None:
        ws_bytes = 0 if ws is None or isinstance(ws, int) else ws.numel() * ws.element_size()
    _check(_lib.tern_linear_multi(_p(X), ldx, _p(tiled), M, K, n_out, sizes, ptrs, lds, _p(ws),
                                  ws_bytes, _s(stream)), "tern_linear_multi")


def tern_linear_noalloc(X, ldx: int, tiled, M: int, N: int, K: int, Y, ldy: int, stream=None):
    """tern_linear with the library's built-in scratch instead of a workspace."""
    _check(_lib.tern_linear_noalloc(_p(X), ldx, _p(tiled), M, N, K, _p(Y), ldy, _s(stream)),
           "tern_linear_noalloc")


def _nbytes(t):
    return 0 if t is None or isinstance(t, int) else t.numel() * t.element_size()


def tern_linear_ex(X, x_type: int, ldx: int, tiled, M: int, K: int, n_sizes, Ys, ldys, out_type: int,
                   ws=None, ws_bytes: int | None = None, stream=None):
    """Multi-output linear with the activation and output element types chosen."""
    n_out = len(n_sizes)
    sizes = (ctypes.c_int64 * n_out)(*[int(v) for v in n_sizes])
    ptrs = (ctypes.c_void_p * n_out)(*[_p(y) for y in Ys])
    lds = (ctypes.c_int64 * n_out)(*[int(v) for v in ldys])
    if ws_bytes is None:
        ws_bytes = _nbytes(ws)
    _check(_lib.tern_linear_ex(_p(X), x_type, ldx, _p(tiled), M, K, n_out, sizes, ptrs, lds, out_type,
                               _p(ws), ws_bytes, _s(stream)), "tern_linear_ex")


def _i64s(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def _ptrs(vals):
    return (ctypes.c_void_p * len(vals))(*[_p(v) for v in vals])


def tern_grouped_workspace_bytes(M: int, Ns, Ks) -> int:
    return int(_lib.tern_grouped_workspace_bytes(M, len(Ns), _i64s(Ns), _i64s(Ks)))


def tern_linear_grouped(x_type: int, M: int, Xs, ldxs, tiled, Ns, Ks, Ys, ldys, out_type: int, ws=None,
                        ws_bytes: int | None = None, stream=None):
    """Independent linears (one output each, the same M) in one launch: the
    streaming kernel for M <= 16, the tensor-core GEMM above."""
    count = len(Ns)
    if ws_bytes is None:
        ws_bytes = _nbytes(ws)
    _check(_lib.tern_linear_grouped(x_type, M, count, _ptrs(Xs), _i64s(ldxs), _ptrs(tiled), _i64s(Ns), _i64s(Ks),
                                    _ptrs(Ys), _i64s(ldys), out_type, _p(ws), ws_bytes, _s(stream)),
           "tern_linear_grouped")


def tern_repack_grouped(packed, scales, Ns, Ks, tiled, tiled_bytes=None, err=None, stream=None):
    """Several disk -> tiled repacks in one launch."""
    count = len(Ns)
    if tiled_bytes is None:
        tiled_bytes = [_nbytes(t) for t in tiled]
    sizes = (ctypes.c_size_t * count)(*[int(v) for v in tiled_bytes])
    _check(_lib.tern_repack_grouped(count, _ptrs(packed), _ptrs(scales), _i64s(Ns), _i64s(Ks), _ptrs(tiled), sizes,
                                    _p(err), _s(stream)), "tern_repack_grouped")


def tern_tiled_glu_bytes(I: int, K: int) -> int:
    return int(_lib.tern_tiled_glu_bytes(I, K))


def tern_repack_glu(packed_gate, scales_gate, packed_up, scales_up, I: int, K: int, tiled,
                    tiled_bytes: int | None = None, err=None, stream=None):
    if tiled_bytes is None:
        tiled_bytes = _nbytes(tiled)
    _check(_lib.tern_repack_glu(_p(packed_gate), _p(scales_gate), _p(packed_up), _p(scales_up), I, K,
                                _p(tiled), tiled_bytes, _p(err), _s(stream)), "tern_repack_glu")


def tern_swiglu_workspace_bytes(M: int, I: int, K: int) -> int:
    return int(_lib.tern_swiglu_workspace_bytes(M, I, K))


def tern_linear_swiglu(X, x_type: int, ldx: int, tiled_glu, M: int, I: int, K: int, H, ldh: int,
                       out_type: int, ws=None, ws_bytes: int | None = None, stream=None):
    if ws_bytes is None:
        ws_bytes = _nbytes(ws)
    _check(_lib.tern_linear_swiglu(_p(X), x_type, ldx, _p(tiled_glu), M, I, K, _p(H), ldh, out_type,
                                   _p(ws), ws_bytes, _s(stream)), "tern_linear_swiglu")


def tern_workspace_error(ws, stream=None) -> int:
    """The workspace's error word (waits for ``stream`` to reach this point)."""
    out = ctypes.c_int32(0)
    _check(_lib.tern_workspace_error(_p(ws), ctypes.addressof(out), _s(stream)), "tern_workspace_error")
    return int(out.value)


def tern_workspace_reset(ws, ws_bytes: int | None = None, stream=None):
    if ws_bytes is None:
        ws_bytes = _nbytes(ws)
    _check(_lib.tern_workspace_reset(_p(ws), ws_bytes, _s(stream)), "tern_workspace_reset")


def tern_xq_bytes(M: int, K: int) -> int:
    return int(_lib.tern_xq_bytes(M, K))


def tern_quantize_x(X, x_type: int, ldx: int, M: int, K: int, xq, a, stream=None):
    _check(_lib.tern_quantize_x(_p(X), x_type, ldx, M, K, _p(xq), _p(a), _s(stream)), "tern_quantize_x")


def tern_i8_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_lib.tern_i8_workspace_bytes(M, N, K))


def tern_linear_i8(xq, a, tiled, M: int, N: int, K: int, Y, ldy: int, out_type: int = 0, ws=None,
                   ws_bytes: int | None = None, stream=None):
    if ws_bytes is None:
        ws_bytes = _nbytes(ws)
    _check(_lib.tern_linear_i8(_p(xq), _p(a), _p(tiled), M, N, K, _p(Y), ldy, out_type, _p(ws), ws_bytes,
                               _s(stream)), "tern_linear_i8")


def tern_tiled_s8_bytes(N: int, K: int) -> int:
    return int(_lib.tern_tiled_s8_bytes(N, K))


def tern_quantize_scales(scales, N: int, K: int, q8, f, stream=None):
    _check(_lib.tern_quantize_scales(_p(scales), N, K, _p(q8), _p(f), _s(stream)), "tern_quantize_scales")


def tern_repack_s8(packed, q8, f, N: int, K: int, tiled, tiled_bytes: int | None = None, err=None, stream=None):
    if tiled_bytes is None:
        tiled_bytes = _nbytes(tiled)
    _check(_lib.tern_repack_s8(_p(packed), _p(q8), _p(f), N, K, _p(tiled), tiled_bytes, _p(err), _s(stream)),
           "tern_repack_s8")


def tern_linear_s8(X, x_type: int, ldx: int, tiled_s8, M: int, K: int, n_sizes, Ys, ldys, out_type: int,
                   ws=None, ws_bytes: int | None = None, stream=None):
    n_out = len(n_sizes)
    sizes = (ctypes.c_int64 * n_out)(*[int(v) for v in n_sizes])
    ptrs = (ctypes.c_void_p * n_out)(*[_p(y) for y in Ys])
    lds = (ctypes.c_int64 * n_out)(*[int(v) for v in ldys])
    if ws_bytes is None:
        ws_bytes = _nbytes(ws)
    _check(_lib.tern_linear_s8(_p(X), x_type, ldx, _p(tiled_s8), M, K, n_out, sizes, ptrs, lds, out_type,
                               _p(ws), ws_bytes, _s(stream)), "tern_linear_s8")


def tern_unit_count(N: int, K: int) -> int:
    return int(_lib.tern_unit_count(N, K))


def tern_zero_units(tiled, N: int, K: int, flags, stream=None):
    _check(_lib.tern_zero_units(_p(tiled), N, K, _p(flags), _s(stream)), "tern_zero_units")


def tern_linear_sparse(X, x_type: int, ldx: int, tiled, flags, M: int, K: int, n_sizes, Ys, ldys, out_type: int,
                       ws=None, ws_bytes: int | None = None, stream=None):
    n_out = len(n_sizes)
    sizes = (ctypes.c_int64 * n_out)(*[int(v) for v in n_sizes])
    ptrs = (ctypes.c_void_p * n_out)(*[_p(y) for y in Ys])
    lds = (ctypes.c_int64 * n_out)(*[int(v) for v in ldys])
    if ws_bytes is None:
        ws_bytes = _nbytes(ws)
    _check(_lib.tern_linear_sparse(_p(X), x_type, ldx, _p(tiled), _p(flags), M, K, n_out, sizes, ptrs, lds,
                                   out_type, _p(ws), ws_bytes, _s(stream)), "tern_linear_sparse")
