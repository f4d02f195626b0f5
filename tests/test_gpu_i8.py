"""GPU-vs-oracle parity of the int8-activation variant (the page's
integer-accumulation route): the per-token quantiser bit-exactly (both
sides round in fp32, ties to even), and the layer within
|y - y_ref| <= 1e-4 * sum_k |a q w| per output."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_util import DEV, assert_within_bound, dev, host, tiled_from_ternary  # noqa: E402
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu


def rand_x(rng, M, K, x_f16):
    v = rng.standard_normal((M, K)) * rng.uniform(0.1, 10, (M, 1))
    if x_f16:
        return v.astype(np.float16).view(np.uint16)
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def tile_order(K):
    """Position of weight k in a quantised row: per 16, even k then odd k."""
    k = np.arange(K)
    return (k & ~15) + (k & 1) * 8 + ((k & 15) >> 1)


def gpu_quantize(x, x_f16):
    M, K = x.shape
    xq = torch.zeros(tb.tern_xq_bytes(M, K), dtype=torch.int8, device=DEV)
    a = torch.zeros(M, dtype=torch.float32, device=DEV)
    tb.tern_quantize_x(dev(x.view(np.int16)), tb.TERN_X_F16 if x_f16 else tb.TERN_X_BF16, K, M, K, xq, a)
    return xq, a


@pytest.mark.parametrize("M,K", [(1, 128), (5, 1024), (37, 5120)])
@pytest.mark.parametrize("x_f16", [False, True])
def test_quantize_x_bit_exact(M, K, x_f16):
    rng = np.random.default_rng(M + K + x_f16)
    x = rand_x(rng, M, K, x_f16)
    x[0, :5] = x[0, 5]          # repeated values, including the maximum's neighbours
    xq, a = gpu_quantize(x, x_f16)
    q_ref, a_ref = oracle.quantize_x(x, x_f16)
    q = host(xq)[:M * K].reshape(M, K)[:, tile_order(K)]
    assert np.array_equal(q, q_ref)
    assert np.array_equal(host(a), a_ref)


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (1, 1000, 5120), (1, 300, 27648), (3, 1000, 512),
                                   (16, 300, 5120), (17, 1000, 1024), (40, 130, 256)])
def test_linear_i8(M, N, K):
    rng = np.random.default_rng(M * 11 + N + K)
    u = rng.random((N, K))
    t = np.where(u < 0.33, -1, np.where(u < 0.66, 0, 1)).astype(np.int8)
    s = rng.uniform(0.005, 0.05, (N, K // 128)).astype(np.float16).view(np.uint16)
    x = rand_x(rng, M, K, False)
    tiled = tiled_from_ternary(t, s)
    xq, a = gpu_quantize(x, False)
    Y = torch.full((M, N + 2), float("nan"), device=DEV)
    ws = torch.zeros(max(tb.tern_i8_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device=DEV)
    tb.tern_linear_i8(xq, a, tiled, M, N, K, Y, N + 2, tb.TERN_OUT_F32, ws)
    y = host(Y)
    assert np.all(np.isnan(y[:, N:]))
    q_ref, a_ref = oracle.quantize_x(x)
    y_ref, bound = oracle.linear_i8(q_ref, a_ref, oracle.pack(t)[0], s, K)
    assert_within_bound(y[:, :N], y_ref, bound, f"i8 M={M} N={N} K={K}")
    assert tb.tern_workspace_error(ws) == 0


@pytest.mark.parametrize("M", [1, 4])
def test_linear_i8_27b_down_sampled(M):
    # full-size 27B-class down projection (K = 27648 -> N = 5120): the
    # single-token kernel (M = 1) and the batched one
    wl = synth.WORKLOADS["dec27b"]
    lin = next(l for l in wl.linears if l.name == "down")
    t, s = synth.weights(wl, 0, lin)
    tiled = tiled_from_ternary(t, s)
    x = synth.activations(wl, 0, lin, M)
    xq, a = gpu_quantize(x, False)
    Y = torch.empty((M, lin.N), device=DEV)
    ws = torch.zeros(max(tb.tern_i8_workspace_bytes(M, lin.N, lin.K), 256), dtype=torch.uint8, device=DEV)
    tb.tern_linear_i8(xq, a, tiled, M, lin.N, lin.K, Y, lin.N, tb.TERN_OUT_F32, ws)
    rows = np.array([0, 1, 127, 128, 2560, 5119])
    q_ref, a_ref = oracle.quantize_x(x)
    y_ref, bound = oracle.linear_i8(q_ref, a_ref, oracle.pack(t[rows])[0], s[rows], lin.K)
    assert_within_bound(host(Y)[:, rows], y_ref, bound, "i8 27B down")
