"""Zero-block skipping: tern_zero_units against the oracle's flags (from
the unpacked weights, not from the tile layout), and tern_linear_sparse
against the plain oracle layer -- skipping a zero unit must not change any
output -- on weights with structured zero blocks, through both kernels."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from gpu_util import DEV, assert_within_bound, dev, host, tiled_from_ternary  # noqa: E402
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu


def sparse_weights(rng, N, K, pattern):
    u = rng.random((N, K))
    t = np.where(u < 0.33, -1, np.where(u < 0.66, 0, 1)).astype(np.int8)
    R, G = (N + 127) // 128, K // 128
    if pattern == "half":
        keep = rng.random((R, G)) < 0.5
    elif pattern == "leading":           # the first groups of every tile are zero
        keep = np.ones((R, G), dtype=bool)
        keep[:, :G // 2] = False
    elif pattern == "tile":              # row tile 1 entirely zero
        keep = np.ones((R, G), dtype=bool)
        keep[min(1, R - 1), :] = False
    else:                                # everything zero
        keep = np.zeros((R, G), dtype=bool)
    for b in range(R):
        for g in range(G):
            if not keep[b, g]:
                t[128 * b:128 * b + 128, 128 * g:128 * g + 128] = 0
    s = rng.uniform(0.005, 0.05, (N, G)).astype(np.float16).view(np.uint16)
    return t, s


@pytest.mark.parametrize("pattern", ["half", "leading", "tile", "all"])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 1024), (5, 300, 512), (16, 1000, 512), (32, 520, 512), (40, 520, 1024),
                                   (300, 1000, 512)])
def test_linear_sparse(M, N, K, pattern):
    rng = np.random.default_rng(M + N + K + len(pattern))
    t, s = sparse_weights(rng, N, K, pattern)
    tiled = tiled_from_ternary(t, s)
    flags = torch.zeros(tb.tern_unit_count(N, K), dtype=torch.uint8, device=DEV)
    tb.tern_zero_units(tiled, N, K, flags)
    packed, _ = oracle.pack(t)
    assert np.array_equal(host(flags), oracle.zero_units(packed, K))
    x = (rng.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    splits = [N // 2, N - N // 2]
    Ys = [torch.full((M, n), float("nan"), device=DEV) for n in splits]
    ws = torch.zeros(tb.tern_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    tb.tern_linear_sparse(dev(x.view(np.int16)), tb.TERN_X_BF16, K, tiled, flags, M, K, splits, Ys, splits,
                          tb.TERN_OUT_F32, ws)
    y = np.concatenate([host(Y) for Y in Ys], axis=1)
    y_ref, bound = oracle.linear(x, packed, s, K)
    assert_within_bound(y, y_ref, bound, f"sparse {pattern} M={M}")
    if pattern == "all":
        assert not y.any()
    assert tb.tern_workspace_error(ws) == 0
