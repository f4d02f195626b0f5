"""Helpers for the GPU parity tests: move seeded inputs to the device and
run libtern through its C ABI."""
import numpy as np
import torch

from ternary_bit_weight_gb300 import binding as tb

DEV = "cuda:0"
TOL = 1e-4   # |y - y_ref| <= TOL * sum_k |x w| per output


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def gpu_pack(t_np: np.ndarray) -> torch.Tensor:
    N, K = t_np.shape
    t = dev(t_np)
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=DEV)
    tb.tern_pack(t, N, K, packed)
    return packed


def gpu_repack(packed: torch.Tensor, scales_np: np.ndarray, N: int, K: int) -> torch.Tensor:
    scales = dev(scales_np.view(np.int16)) if scales_np.dtype == np.uint16 else dev(scales_np)
    tiled = torch.empty(tb.tern_tiled_bytes(N, K), dtype=torch.uint8, device=DEV)
    tb.tern_repack(packed, scales, N, K, tiled)
    return tiled


def tiled_from_ternary(t_np: np.ndarray, scales_np: np.ndarray) -> torch.Tensor:
    N, K = t_np.shape
    return gpu_repack(gpu_pack(t_np), scales_np, N, K)


def workspace(M: int, N: int, K: int) -> torch.Tensor | None:
    nbytes = tb.tern_workspace_bytes(M, N, K)
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=DEV)


def gpu_linear(x_np: np.ndarray, tiled: torch.Tensor, N: int, K: int, ws=None) -> torch.Tensor:
    M = x_np.shape[0]
    X = dev(x_np.view(np.int16))
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    if ws is None:
        ws = workspace(M, N, K)
    tb.tern_linear(X, K, tiled, M, N, K, Y, N, ws)
    return Y


def assert_within_bound(y_gpu: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    lim = TOL * bound
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs outside "
                             f"1e-4*sum|xw|; first {idx.tolist()}: gpu {y_gpu[tuple(idx[0])]} "
                             f"ref {y_ref[tuple(idx[0])]} bound {bound[tuple(idx[0])]}")
