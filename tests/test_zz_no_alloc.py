"""tern_linear_noalloc: the layer for callers that cannot allocate.

Such callers (code running under CUDA graph capture, plug-ins whose device
memory belongs to a host framework's allocator) get the split-K scratch from
an array built into the library.  This file runs last so that, if it fails,
a run that stops at the first failure has already run every other test; it
passes both alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_util import DEV, assert_within_bound, dev, host, tiled_from_ternary, workspace  # noqa: E402
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 16 << 20   # the size include/tern.h states for the built-in scratch


def _case(name, M):
    wl = synth.WORKLOADS["dec27b"]
    lin = next(l for l in wl.linears if l.name == name)
    t, s = synth.weights(wl, 0, lin)
    x = synth.activations(wl, 0, lin, M)
    return lin.N, lin.K, t, s, x


@pytest.mark.parametrize("name,M", [("o", 1), ("down", 1), ("o", 16), ("qkv", 8)])
def test_noalloc_matches_workspace_entry_point_twice(name, M):
    N, K, t, s, x = _case(name, M)
    need = tb.tern_workspace_bytes(M, N, K)
    assert need <= SCRATCH_LIMIT
    tiled = tiled_from_ternary(t, s)
    X = dev(x.view(np.int16))
    # the existing entry point with a caller-owned workspace
    Y_ws = torch.full((M, N), float("nan"), device=DEV)
    tb.tern_linear(X, K, tiled, M, N, K, Y_ws, N, workspace(M, N, K))
    # both are held to the tests' tolerance against the fp64 oracle:
    # |y - y_ref| <= 1e-4 * sum_k |x w| per output
    packed, _ = oracle.pack(t)
    y_ref, bound = oracle.linear(x, packed, s, K)
    assert_within_bound(host(Y_ws), y_ref, bound, f"tern_linear {name} M={M}")
    for call in range(2):   # two calls in a row share the same scratch
        Y = torch.full((M, N), float("nan"), device=DEV)
        tb.tern_linear_noalloc(X, K, tiled, M, N, K, Y, N)
        torch.cuda.synchronize()
        y = host(Y).astype(np.float64)
        assert np.all(np.isfinite(y)), call
        assert_within_bound(y, y_ref, bound, f"noalloc {name} M={M} call {call}")
        # and it agrees with the workspace entry point within the same tolerance
        assert_within_bound(y, host(Y_ws).astype(np.float64), bound, f"noalloc vs tern_linear call {call}")


def test_noalloc_rejects_problems_beyond_the_scratch():
    M, N, K = 4096, 4 << 20, 128 * 256    # a workspace far above the built-in scratch
    need = tb.tern_workspace_bytes(M, N, K)
    assert need > SCRATCH_LIMIT
    X = torch.zeros(16, dtype=torch.int16, device=DEV)
    Y = torch.zeros(16, dtype=torch.float32, device=DEV)
    tiled = torch.zeros(16, dtype=torch.uint8, device=DEV)
    status = tb.library().tern_linear_noalloc(X.data_ptr(), K, tiled.data_ptr(), M, N, K,
                                              Y.data_ptr(), N, None)
    assert status == 4   # TERN_ERR_SIZE, returned before anything is enqueued
