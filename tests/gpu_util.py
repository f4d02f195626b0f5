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


def gpu_linear(x_np: np.ndarray, tiled: torch.Tensor, N: int, K: int, ws=None, ldx: int | None = None) -> torch.Tensor:
    """tern_linear on host activations; with ldx > K the rows of X are laid
    out with that stride (the extra columns hold NaN, which must never be read)."""
    M = x_np.shape[0]
    if ldx is None or ldx == K:
        X = dev(x_np.view(np.int16))
        ldx = K
    else:
        X = torch.full((M, ldx), 0x7FC0, dtype=torch.int16, device=DEV)   # bf16 NaN
        X[:, :K] = dev(x_np.view(np.int16))
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    if ws is None:
        ws = workspace(M, N, K)
    tb.tern_linear(X, ldx, tiled, M, N, K, Y, N, ws)
    return Y


def gpu_linear_multi(x_np: np.ndarray, tiled: torch.Tensor, splits, K: int, pad: int = 3):
    """tern_linear_multi with one fp32 output per split (row stride n + pad,
    padding columns NaN); returns the outputs as host arrays [M, n + pad]."""
    M = x_np.shape[0]
    N = int(sum(splits))
    Ys = [torch.full((M, n + pad), float("nan"), device=DEV) for n in splits]
    tb.tern_linear_multi(dev(x_np.view(np.int16)), K, tiled, M, K, list(splits), Ys,
                         [n + pad for n in splits], workspace(M, N, K))
    return [host(Y) for Y in Ys]


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
