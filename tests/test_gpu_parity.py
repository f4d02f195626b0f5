"""GPU-vs-oracle parity through libtern's C ABI.

Byte formats (pack, unpack, repack, unrepack) must match the oracle
bit-exactly.  The linear layer must satisfy, per output,
|y_gpu - y_ref| <= 1e-4 * sum_k |x[m,k] * W[n,k]|, with y_ref and the bound
from the fp64 oracle on the same seeded inputs.  Small shapes are compared
in full (several tiles plus ragged tails); the full-size 27B-class shapes
are compared on sampled rows and columns, in the same launch configuration
the benchmark uses.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_util import (DEV, assert_within_bound, dev, gpu_linear, gpu_pack, gpu_repack,  # noqa: E402
                      host, tiled_from_ternary, workspace)
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu


def rand_ternary(rng, N, K, p_zero=1 / 3):
    u = rng.random((N, K))
    pm = (1 - p_zero) / 2
    return np.where(u < pm, -1, np.where(u < pm + p_zero, 0, 1)).astype(np.int8)


def rand_scales(rng, N, K):
    return np.array([synth.round_fp16(v) for v in rng.uniform(0.005, 0.05, N * (K // 128))],
                    dtype=np.uint16).reshape(N, K // 128)


def rand_x(rng, M, K):
    return np.array([synth.round_bf16(v) for v in rng.standard_normal(M * K)],
                    dtype=np.uint16).reshape(M, K)


# ------------------------------------------------------------ byte formats

@pytest.mark.parametrize("N,K", [(1, 4), (3, 20), (5, 36), (64, 1024), (1000, 4096)])
def test_pack_bit_exact(N, K):
    rng = np.random.default_rng(N + K)
    t = rand_ternary(rng, N, K)
    ref, bad = oracle.pack(t)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=DEV)
    tb.tern_pack(dev(t), N, K, packed, err)
    assert np.array_equal(host(packed), ref)
    assert int(err.item()) == bad == 0


def test_pack_unaligned_and_invalid_values():
    rng = np.random.default_rng(9)
    N, K = 7, 52
    t = rand_ternary(rng, N, K)
    t[0, 3] = 2
    t[4, 50] = -7
    t[6, 0] = 127
    ref, bad = oracle.pack(t)
    buf = torch.zeros(N * K + 1, dtype=torch.int8, device=DEV)
    buf[1:] = dev(t).reshape(-1)              # odd address: byte path
    out = torch.zeros(N * K // 4 + 1, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tb.tern_pack(buf.data_ptr() + 1, N, K, out.data_ptr() + 1, err)
    assert np.array_equal(host(out[1:]).reshape(N, K // 4), ref)
    assert int(err.item()) == bad == 3


@pytest.mark.parametrize("N,K", [(1, 4), (3, 20), (64, 1024), (300, 2048)])
def test_unpack_bit_exact_with_reserved_codes(N, K):
    rng = np.random.default_rng(N * K)
    raw = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    ref, reserved = oracle.unpack(raw, K)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    t = torch.empty((N, K), dtype=torch.int8, device=DEV)
    tb.tern_unpack(dev(raw), N, K, t, err)
    assert np.array_equal(host(t), ref)
    assert int(err.item()) == reserved


@pytest.mark.parametrize("N,K", [(1, 128), (16, 128), (17, 256), (100, 384), (1024, 1024),
                                 (7168, 512)])
def test_repack_bit_exact(N, K):
    rng = np.random.default_rng(N * 7 + K)
    raw = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)   # includes code 11
    scales = rng.integers(0, 1 << 16, size=(N, K // 128), dtype=np.uint16)
    ref, reserved = oracle.repack(raw, scales, K)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tiled = torch.full((tb.tern_tiled_bytes(N, K),), 0xEE, dtype=torch.uint8, device=DEV)
    tb.tern_repack(dev(raw), dev(scales.view(np.int16)), N, K, tiled, err=err)
    assert np.array_equal(host(tiled), ref)
    assert int(err.item()) == reserved


@pytest.mark.parametrize("N,K", [(1, 128), (17, 256), (1024, 1024)])
def test_unrepack_bit_exact(N, K):
    rng = np.random.default_rng(N + 3 * K)
    raw = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    scales = rng.integers(0, 1 << 16, size=(N, K // 128), dtype=np.uint16)
    tiled_ref, _ = oracle.repack(raw, scales, K)
    tiled_ref[0] |= 0x03      # plant one stored value 3 (invalid) at weight (0, 0)
    p_ref, s_ref, invalid = oracle.unrepack(tiled_ref, N, K)
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=DEV)
    sc = torch.empty((N, K // 128), dtype=torch.int16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tb.tern_unrepack(dev(tiled_ref), N, K, packed, sc, err)
    assert np.array_equal(host(packed), p_ref)
    assert np.array_equal(host(sc).view(np.uint16), s_ref)
    assert int(err.item()) == invalid == 1


# ------------------------------------------------------------ linear layer

def _check_linear(t, scales, x, what):
    N, K = t.shape
    packed_ref, _ = oracle.pack(t)
    y_ref, bound = oracle.linear(x, packed_ref, scales, K)
    tiled = tiled_from_ternary(t, scales)
    y = host(gpu_linear(x, tiled, N, K))
    assert_within_bound(y, y_ref, bound, what)
    return y


@pytest.mark.parametrize("M", [1, 8])
def test_linear_single_layer_workload(M):
    wl = synth.WORKLOADS["single"]
    lin = wl.linears[0]
    t, s = synth.weights(wl, 0, lin)
    x = synth.activations(wl, 0, lin, M)
    _check_linear(t, s, x, f"single M={M}")


@pytest.mark.parametrize("N,K", [(1, 128), (15, 384), (17, 128), (200, 1280), (1000, 256)])
@pytest.mark.parametrize("M", [1, 2, 3, 7, 8, 9, 15, 16, 17, 24, 32, 33])
def test_linear_ragged_shapes(N, K, M):
    rng = np.random.default_rng(N * 131 + K * 7 + M)
    t = rand_ternary(rng, N, K)
    s = rand_scales(rng, N, K)
    x = rand_x(rng, M, K)
    _check_linear(t, s, x, f"N={N} K={K} M={M}")


def test_linear_special_cases():
    K, N = 256, 40
    rng = np.random.default_rng(4)
    x = rand_x(rng, 3, K)
    one = np.full((N, K // 128), 0x3C00, np.uint16)
    # all-zero weights: exactly zero output
    y = host(gpu_linear(x, tiled_from_ternary(np.zeros((N, K), np.int8), one), N, K))
    assert np.all(y == 0.0)
    # all +1 with unit scale: row sums of X, and all -1: their negation
    xs = synth.bf16_bits_to_float(x).sum(axis=1)
    yp = host(gpu_linear(x, tiled_from_ternary(np.ones((N, K), np.int8), one), N, K))
    yn = host(gpu_linear(x, tiled_from_ternary(-np.ones((N, K), np.int8), one), N, K))
    for m in range(3):
        assert np.allclose(yp[m], xs[m], rtol=0, atol=1e-4 * np.abs(synth.bf16_bits_to_float(x[m])).sum())
        assert np.array_equal(yn[m], -yp[m])
    # one-hot X picks one weight times its own group's scale, exactly
    t = rand_ternary(rng, N, K)
    s = np.array([[synth.round_fp16(2.0 ** -(n % 7 + 3 * g)) for g in range(K // 128)]
                  for n in range(N)], np.uint16)
    tiled = tiled_from_ternary(t, s)
    for k in (0, 5, 127, 128, 200, 255):
        xo = np.zeros((1, K), np.uint16)
        xo[0, k] = 0x3F80
        yo = host(gpu_linear(xo, tiled, N, K))[0]
        want = np.array([t[n, k] * 2.0 ** -(n % 7 + 3 * (k // 128)) for n in range(N)])
        assert np.array_equal(yo.astype(np.float64), want), k


def test_linear_multi_output_embedding_qkv_and_gate_up():
    wl = synth.WORKLOADS["embed06b"]
    for lin in (wl.linears[0], wl.linears[2]):
        N, K = lin.N, lin.K
        t, s = synth.weights(wl, 3, lin)
        packed_ref, _ = oracle.pack(t)
        tiled = tiled_from_ternary(t, s)
        for M in (1, 8, 32):
            x = synth.activations(wl, 3, lin, M)
            y_ref, bound = oracle.linear(x, packed_ref, s, K)
            Ys = [torch.full((M, n + 3), float("nan"), device=DEV) for n in lin.splits]
            ws = workspace(M, N, K)
            tb.tern_linear_multi(dev(x.view(np.int16)), K, tiled, M, K, list(lin.splits), Ys,
                                 [n + 3 for n in lin.splits], ws)
            off = 0
            for Y, n in zip(Ys, lin.splits):
                yh = host(Y)
                assert_within_bound(yh[:, :n], y_ref[:, off:off + n], bound[:, off:off + n],
                                    f"{lin.name} M={M} part@{off}")
                assert np.all(np.isnan(yh[:, n:]))   # padding columns untouched
                off += n


def test_linear_is_deterministic_and_leaves_workspace_zeroed():
    rng = np.random.default_rng(12)
    N, K, M = 5120, 5120, 1
    t = rand_ternary(rng, N, K, 0.35)
    s = rand_scales(rng, N, K)
    x = rand_x(rng, M, K)
    tiled = tiled_from_ternary(t, s)
    ws = workspace(M, N, K)
    y1 = gpu_linear(x, tiled, N, K, ws)
    y2 = gpu_linear(x, tiled, N, K, ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    # workspace: error word, then one arrival counter per (token tile, row
    # tile, row quarter); all back to zero after the calls
    R = -(-N // 128)
    head = ws[: 256 + 16 * R].view(torch.int32)
    assert int(head.count_nonzero().item()) == 0


def test_linear_empty_problems_are_noops():
    Y = torch.full((2, 8), 7.0, device=DEV)
    tiled = torch.zeros(tb.tern_tiled_bytes(8, 128), dtype=torch.uint8, device=DEV)
    X = torch.zeros((2, 128), dtype=torch.int16, device=DEV)
    tb.tern_linear(X, 128, tiled, 0, 8, 128, Y, 8)
    tb.tern_linear(X, 128, tiled, 2, 0, 128, Y, 8)
    assert torch.all(Y == 7.0)


# ------------------------------------------- full-size 27B-class layers

SAMPLE_ROWS = 16


def _sample_rows(N):
    starts = sorted({0, N // 3, N // 2, N - SAMPLE_ROWS})
    return np.concatenate([np.arange(s, s + SAMPLE_ROWS) for s in starts])


_LAYER_CACHE = {}


def _layer_27b(name):
    """Tiled weights of one dec27b linear on the GPU plus the oracle's packed
    copy of the sampled rows (generated once per module)."""
    if name not in _LAYER_CACHE:
        wl = synth.WORKLOADS["dec27b"]
        lin = next(l for l in wl.linears if l.name == name)
        t, s = synth.weights(wl, 0, lin)
        rows = _sample_rows(lin.N)
        packed_rows, _ = oracle.pack(t[rows])
        _LAYER_CACHE[name] = (lin, tiled_from_ternary(t, s), rows, packed_rows, s[rows].copy())
    return _LAYER_CACHE[name]


@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_linear_27b_layer_sampled(name, M):
    lin, tiled, rows, packed_rows, s_rows = _layer_27b(name)
    N, K = lin.N, lin.K
    x = synth.activations(synth.WORKLOADS["dec27b"], 0, lin, M)
    y = host(gpu_linear(x, tiled, N, K))
    y_ref, bound = oracle.linear(x, packed_rows, s_rows, K)
    assert_within_bound(y[:, rows], y_ref, bound, f"27b {name} M={M}")
    assert np.all(np.isfinite(y))


def test_linear_prefill_shape_sampled():
    wl = synth.WORKLOADS["prefill27b"]
    lin = next(l for l in wl.linears if l.name == "o")
    N, K, M = lin.N, lin.K, 1024
    t, s = synth.weights(wl, 0, lin)
    x = synth.activations(wl, 0, lin, M)
    tiled = tiled_from_ternary(t, s)
    y = host(gpu_linear(x, tiled, N, K))
    rows = _sample_rows(N)
    mrows = np.array([0, 1, 15, 16, 17, 511, 512, 1000, 1023])
    packed_rows, _ = oracle.pack(t[rows])
    y_ref, bound = oracle.linear(x[mrows], packed_rows, s[rows], K)
    assert_within_bound(y[np.ix_(mrows, rows)], y_ref, bound, "prefill o M=1024")
