"""GPU-vs-oracle parity of INT8 group scales: the scale quantiser and the
INT8-scale repack bit-exactly, and the layer (both kernels: M <= 16 and the
tensor-core GEMM) within |y - y_ref| <= 1e-4 * sum_k |x t q8 f|."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from gpu_util import DEV, assert_within_bound, dev, gpu_pack, host  # noqa: E402
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu


def weights(rng, N, K):
    u = rng.random((N, K))
    t = np.where(u < 0.33, -1, np.where(u < 0.66, 0, 1)).astype(np.int8)
    s = np.exp(rng.normal(-4, 0.5, (N, K // 128))).astype(np.float16).view(np.uint16)
    return t, s


def gpu_s8(t, s):
    N, K = t.shape
    q8 = torch.empty((N, K // 128), dtype=torch.int8, device=DEV)
    f = torch.empty(N, dtype=torch.float32, device=DEV)
    tb.tern_quantize_scales(dev(s.view(np.int16)), N, K, q8, f)
    tiled = torch.empty(tb.tern_tiled_s8_bytes(N, K), dtype=torch.uint8, device=DEV)
    tb.tern_repack_s8(gpu_pack(t), q8, f, N, K, tiled)
    return q8, f, tiled


@pytest.mark.parametrize("N,K", [(1, 128), (130, 256), (1000, 5120)])
def test_quantize_and_repack_s8_bit_exact(N, K):
    rng = np.random.default_rng(N + K)
    t, s = weights(rng, N, K)
    s[0, 0] = 0                                   # a zero scale
    q8, f, tiled = gpu_s8(t, s)
    q_ref, f_ref = oracle.quantize_scales(s, K)
    assert np.array_equal(host(q8), q_ref)
    assert np.array_equal(host(f), f_ref)
    assert np.array_equal(host(tiled), oracle.repack_s8(oracle.pack(t)[0], q_ref, f_ref, K))


@pytest.mark.parametrize("M,N,K", [(1, 1000, 512), (4, 300, 5120), (16, 1000, 1024), (24, 300, 512), (33, 520, 512),
                                   (300, 1000, 512)])
def test_linear_s8(M, N, K):
    rng = np.random.default_rng(M + 3 * N + K)
    t, s = weights(rng, N, K)
    q8, f, tiled = gpu_s8(t, s)
    x = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Y = torch.full((M, N + 1), float("nan"), device=DEV)
    ws = torch.zeros(tb.tern_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    tb.tern_linear_s8(dev(x.view(np.int16)), tb.TERN_X_BF16, K, tiled, M, K, [N], [Y], [N + 1],
                      tb.TERN_OUT_F32, ws)
    y = host(Y)
    assert np.all(np.isnan(y[:, N:]))
    q_ref, f_ref = oracle.quantize_scales(s, K)
    y_ref, bound = oracle.linear_s8(x, oracle.pack(t)[0], q_ref, f_ref, K)
    assert_within_bound(y[:, :N], y_ref, bound, f"s8 M={M} N={N} K={K}")
    assert tb.tern_workspace_error(ws) == 0
