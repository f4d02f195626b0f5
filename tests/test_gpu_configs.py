"""GPU-vs-oracle parity at the workloads' full sizes, in the call forms the
benchmark times.

Each case runs libtern on the workload's full shapes (all rows, all
tokens) and compares sampled outputs with the fp64 oracle element by
element: |y_gpu - y_ref| <= 1e-4 * sum_k |x[m,k] * W[n,k]|.  Samples cover
the first and last rows and tokens, tile edges and the borders between the
outputs of the fused (multi-output) projections.  Byte formats are compared
in full.
"""
import hashlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_util import (DEV, assert_within_bound, dev, gpu_linear, gpu_linear_multi, host,  # noqa: E402
                      tiled_from_ternary, workspace)
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu


def sample_rows(lin, per=16):
    """Rows at the start and end of every output slice and one in the middle."""
    rows, off = set(), 0
    for n in lin.splits:
        for s in (off, off + n // 2, off + n - per):
            rows.update(range(max(off, s), min(off + n, s + per)))
        off += n
    return np.array(sorted(rows))


def sample_tokens(M):
    cand = {0, 1, 15, 16, 17, 127, 128, M // 2, M - 129, M - 128, M - 2, M - 1}
    return np.array(sorted(m for m in cand if 0 <= m < M))


_CACHE = {}


def layer(wl_name, lin_name, layer_idx=0):
    """(lin, tiled on the GPU, t, s) of one linear, generated once per module."""
    key = (wl_name, lin_name, layer_idx)
    if key not in _CACHE:
        wl = synth.WORKLOADS[wl_name]
        lin = next(l for l in wl.linears if l.name == lin_name)
        t, s = synth.weights(wl, layer_idx, lin)
        _CACHE[key] = (lin, tiled_from_ternary(t, s), t, s)
    return _CACHE[key]


def run_call_form(lin, tiled, x):
    """The call the benchmark makes: tern_linear_multi for fused projections,
    tern_linear otherwise.  Returns the concatenated output [M, N]."""
    if len(lin.splits) == 1:
        return host(gpu_linear(x, tiled, lin.N, lin.K))
    parts = gpu_linear_multi(x, tiled, lin.splits, lin.K)
    for p, n in zip(parts, lin.splits):
        assert np.all(np.isnan(p[:, n:])), "padding columns written"
    return np.concatenate([p[:, :n] for p, n in zip(parts, lin.splits)], axis=1)


def check_sampled(wl_name, lin_name, M, layer_idx=0):
    wl = synth.WORKLOADS[wl_name]
    lin, tiled, t, s = layer(wl_name, lin_name, layer_idx)
    x = synth.activations(wl, layer_idx, lin, M)
    y = run_call_form(lin, tiled, x)
    assert y.shape == (M, lin.N)
    assert np.all(np.isfinite(y))
    rows, toks = sample_rows(lin), sample_tokens(M)
    packed_rows, _ = oracle.pack(t[rows])
    y_ref, bound = oracle.linear(x[toks], packed_rows, s[rows], lin.K)
    assert_within_bound(y[np.ix_(toks, rows)], y_ref, bound, f"{wl_name} {lin_name} M={M}")


# ----------------------------------------------- 0.6B embedding-model layers

@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
@pytest.mark.parametrize("M", [1, 32, 512])
def test_embedding_model_layer(name, M):
    check_sampled("embed06b", name, M, layer_idx=5)


# --------------------------------------- 27B-class stack, batched decode

@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
@pytest.mark.parametrize("M", [32, 64, 128, 256])
def test_stack27b_batched_decode(name, M):
    check_sampled("stack27b", name, M, layer_idx=17)


# ------------------------------------------------------ 27B-class prefill

@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
@pytest.mark.parametrize("M", [1024, 2048, 4096])
def test_prefill27b(name, M):
    check_sampled("prefill27b", name, M)


# ------------------------------------------------------- full-size repack

@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
def test_repack_full_27b_layer_bit_exact(name):
    """All four linears of a 27B-class layer, disk -> tiled, byte for byte."""
    wl = synth.WORKLOADS["stack27b"]
    lin = next(l for l in wl.linears if l.name == name)
    t, s = synth.weights(wl, 31, lin)
    packed, _ = oracle.pack(t)
    del t
    ref, reserved = oracle.repack(packed, s, lin.K)
    assert reserved == 0
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tiled = torch.full((tb.tern_tiled_bytes(lin.N, lin.K),), 0xEE, dtype=torch.uint8, device=DEV)
    tb.tern_repack(dev(packed), dev(s.view(np.int16)), lin.N, lin.K, tiled, err=err)
    got = host(tiled)
    assert hashlib.sha256(got.tobytes()).hexdigest() == hashlib.sha256(ref.tobytes()).hexdigest()
    assert int(err.item()) == 0
    # and back: unrepack restores the disk bytes
    p2 = torch.empty((lin.N, lin.K // 4), dtype=torch.uint8, device=DEV)
    s2 = torch.empty((lin.N, lin.K // 128), dtype=torch.int16, device=DEV)
    tb.tern_unrepack(tiled, lin.N, lin.K, p2, s2)
    assert np.array_equal(host(p2), packed)
    assert np.array_equal(host(s2).view(np.uint16), s)


# -------------------------------------------------- strides and ordering

@pytest.mark.parametrize("M", [1, 5, 16, 40, 300])
def test_strided_activations(M):
    """ldx > K: the kernels read only the first K columns of each X row."""
    wl = synth.WORKLOADS["dec27b"]
    lin, tiled, t, s = layer("dec27b", "o")
    x = synth.activations(wl, 0, lin, M)
    y = host(gpu_linear(x, tiled, lin.N, lin.K, ldx=lin.K + 72))
    rows, toks = sample_rows(lin), sample_tokens(M)
    packed_rows, _ = oracle.pack(t[rows])
    y_ref, bound = oracle.linear(x[toks], packed_rows, s[rows], lin.K)
    assert_within_bound(y[np.ix_(toks, rows)], y_ref, bound, f"strided X M={M}")


@pytest.mark.parametrize("M", [1, 4, 64])
def test_repack_directly_followed_by_linear(M):
    """tern_repack then tern_linear on one stream with nothing in between:
    the linear kernel may start streaming weights before the repack kernel
    has completed, so the repack must have made its writes visible."""
    wl = synth.WORKLOADS["dec27b"]
    lin = next(l for l in wl.linears if l.name == "gate_up")
    t, s = synth.weights(wl, 0, lin)
    N, K = lin.N, lin.K
    x = synth.activations(wl, 0, lin, M)
    packed_dev = dev(oracle.pack(t)[0])
    scales_dev = dev(s.view(np.int16))
    X = dev(x.view(np.int16))
    Y = torch.full((M, N), float("nan"), device=DEV)
    ws = workspace(M, N, K)
    # stale contents: stored value 3 everywhere (decodes to a wrong weight)
    tiled = torch.full((tb.tern_tiled_bytes(N, K),), 0xFF, dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    tb.tern_repack(packed_dev, scales_dev, N, K, tiled, stream=stream)
    tb.tern_linear(X, K, tiled, M, N, K, Y, N, ws, stream=stream)
    y = host(Y)
    rows = sample_rows(lin)
    rows = np.unique(np.concatenate([rows, np.arange(0, N, 997)]))
    toks = sample_tokens(M)
    packed_rows, _ = oracle.pack(t[rows])
    y_ref, bound = oracle.linear(x[toks], packed_rows, s[rows], K)
    assert_within_bound(y[np.ix_(toks, rows)], y_ref, bound, f"repack->linear M={M}")
