"""GPU-vs-oracle parity of tern_linear_grouped: independent linears of
different shapes in one streaming launch (M <= 16) or one GEMM launch with
the items of all problems (M > 16).

Tolerance: every output within 1e-4 * sum_k |x w| of the oracle's fp64
value (the layer's bound), plus half an ulp of the result for bf16 / fp16
outputs (2^-8 |y|, 2^-11 |y| + 2^-24).  Outputs are written with a row
stride larger than N; the padding must stay untouched (NaN)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_util import DEV, dev, host, tiled_from_ternary  # noqa: E402
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-4
ROUND = {tb.TERN_OUT_F32: 0.0, tb.TERN_OUT_BF16: 2.0 ** -8, tb.TERN_OUT_F16: 2.0 ** -11}
FLOOR = {tb.TERN_OUT_F32: 0.0, tb.TERN_OUT_BF16: 0.0, tb.TERN_OUT_F16: 2.0 ** -24}
TORCH_OUT = {tb.TERN_OUT_F32: torch.float32, tb.TERN_OUT_BF16: torch.bfloat16, tb.TERN_OUT_F16: torch.float16}
PAD = 5


def rand_ternary(rng, N, K, p_zero=0.35):
    u = rng.random((N, K))
    pm = (1 - p_zero) / 2
    return np.where(u < pm, -1, np.where(u < pm + p_zero, 0, 1)).astype(np.int8)


def rand_scales(rng, N, K):
    return rng.uniform(0.005, 0.05, (N, K // 128)).astype(np.float16).view(np.uint16)


def rand_x(rng, M, K, x_f16):
    v = rng.standard_normal((M, K))
    if x_f16:
        return v.astype(np.float16).view(np.uint16)
    return np.array([synth.round_bf16(a) for a in v.ravel()], dtype=np.uint16).reshape(M, K)


def check(y_gpu, y_ref, bound, out_type, what):
    y = np.asarray(y_gpu, dtype=np.float64)
    lim = TOL * bound + ROUND[out_type] * (np.abs(y_ref) + TOL * bound) + FLOOR[out_type]
    bad = ~(np.abs(y - y_ref) <= lim)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside; first {i}: gpu {y[i]} "
                             f"ref {y_ref[i]} lim {lim[i]}")


def make_problems(rng, shapes, M, x_f16):
    probs = []
    for N, K in shapes:
        t, s = rand_ternary(rng, N, K), rand_scales(rng, N, K)
        x = rand_x(rng, M, K, x_f16)
        probs.append((N, K, t, s, x, tiled_from_ternary(t, s) if N > 0 else torch.zeros(16, dtype=torch.uint8,
                                                                                        device=DEV)))
    return probs


def run_grouped(probs, M, x_f16, out_type, ws=None):
    Ns = [p[0] for p in probs]
    Ks = [p[1] for p in probs]
    Xs = [dev(p[4].view(np.int16)) for p in probs]
    Ys = [torch.full((M, max(N, 1) + PAD), float("nan"), dtype=TORCH_OUT[out_type], device=DEV) for N in Ns]
    if ws is None:
        ws = torch.zeros(tb.tern_grouped_workspace_bytes(M, Ns, Ks), dtype=torch.uint8, device=DEV)
    tb.tern_linear_grouped(tb.TERN_X_F16 if x_f16 else tb.TERN_X_BF16, M, Xs, Ks, [p[5] for p in probs], Ns, Ks, Ys,
                           [max(N, 1) + PAD for N in Ns], out_type, ws)
    return [host(Y.float()) for Y in Ys], ws


def check_all(probs, ys, out_type, x_f16, what):
    for i, ((N, K, t, s, x, _), y) in enumerate(zip(probs, ys)):
        assert np.all(np.isnan(y[:, N:])), f"{what}: problem {i} padding written"
        if N == 0:
            continue
        y_ref, bound = oracle.linear(x, oracle.pack(t)[0], s, K, x_f16=x_f16)
        check(y[:, :N], y_ref, bound, out_type, f"{what} problem {i} ({N}x{K})")


SHAPES = [(1000, 512), (300, 1024), (129, 256), (64, 128), (0, 256), (517, 640)]


@pytest.mark.parametrize("M", [1, 2, 16, 32, 40, 130, 300])
@pytest.mark.parametrize("out_type", [tb.TERN_OUT_F32, tb.TERN_OUT_BF16])
def test_grouped_matches_oracle(M, out_type):
    rng = np.random.default_rng(7 * M + out_type)
    probs = make_problems(rng, SHAPES, M, False)
    ys, _ = run_grouped(probs, M, False, out_type)
    check_all(probs, ys, out_type, False, f"M={M}")


@pytest.mark.parametrize("M", [1, 5, 64])
def test_grouped_fp16_activations_eight_problems(M):
    # the largest group, with problems of one tile and of several hundred units
    rng = np.random.default_rng(40 + M)
    shapes = [(7, 128), (2000, 256), (128, 1024), (255, 384), (1, 128), (640, 512), (33, 2048), (900, 128)]
    probs = make_problems(rng, shapes, M, True)
    ys, _ = run_grouped(probs, M, True, tb.TERN_OUT_F16)
    check_all(probs, ys, tb.TERN_OUT_F16, True, f"M={M}")


@pytest.mark.parametrize("M", [1, 40])
def test_grouped_workspace_serves_again_and_is_deterministic(M):
    rng = np.random.default_rng(3 + M)
    probs = make_problems(rng, [(1500, 512), (700, 1024), (90, 128)], M, False)
    ys1, ws = run_grouped(probs, M, False, tb.TERN_OUT_F32)
    ys2, _ = run_grouped(probs, M, False, tb.TERN_OUT_F32, ws=ws)
    for a, b in zip(ys1, ys2):
        assert np.array_equal(np.nan_to_num(a, nan=7.0), np.nan_to_num(b, nan=7.0))
    check_all(probs, ys2, tb.TERN_OUT_F32, False, "second call")


@pytest.mark.parametrize("M", [1, 32])
def test_grouped_27b_layer_sampled(M):
    # the four linears of a 27B-class layer in one launch (synthetic weights
    # of the workload's recipe); 64 sampled rows per problem against the oracle
    wl = synth.WORKLOADS["stack27b"]
    probs, Xs, tiled, Ns, Ks, Ys = [], [], [], [], [], []
    for lin in wl.linears:
        t, s = synth.weights(wl, 0, lin)
        x = synth.activations(wl, 0, lin, M)
        Ns.append(lin.N)
        Ks.append(lin.K)
        Xs.append(dev(x.view(np.int16)))
        tiled.append(tiled_from_ternary(t, s))
        Ys.append(torch.full((M, lin.N), float("nan"), dtype=torch.float32, device=DEV))
        rows = np.random.default_rng(lin.N).choice(lin.N, 64, replace=False)
        probs.append((rows, oracle.pack(t[rows])[0], s[rows], x, lin.K))
        del t
    ws = torch.zeros(tb.tern_grouped_workspace_bytes(M, Ns, Ks), dtype=torch.uint8, device=DEV)
    tb.tern_linear_grouped(tb.TERN_X_BF16, M, Xs, Ks, tiled, Ns, Ks, Ys, Ns, tb.TERN_OUT_F32, ws)
    for (rows, packed, s, x, K), Y, N in zip(probs, Ys, Ns):
        y = host(Y)
        assert not np.isnan(y).any()
        y_ref, bound = oracle.linear(x, packed, s, K)
        check(y[:, rows], y_ref, bound, tb.TERN_OUT_F32, f"27B layer N={N}")


def test_grouped_argument_errors():
    X = torch.zeros(128, dtype=torch.int16, device=DEV)
    W = torch.zeros(tb.tern_tiled_bytes(128, 128), dtype=torch.uint8, device=DEV)
    Y = torch.zeros(128, dtype=torch.float32, device=DEV)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(tb.TernError, match="SHAPE"):   # K not a multiple of 128
        tb.tern_linear_grouped(tb.TERN_X_BF16, 1, [X], [100], [W], [128], [100], [Y], [128], tb.TERN_OUT_F32, ws)
    with pytest.raises(tb.TernError, match="SHAPE"):   # ldy < N
        tb.tern_linear_grouped(tb.TERN_X_BF16, 1, [X], [128], [W], [128], [128], [Y], [64], tb.TERN_OUT_F32, ws)
    with pytest.raises(tb.TernError, match="SIZE"):    # workspace too small
        tb.tern_linear_grouped(tb.TERN_X_BF16, 1, [X], [128], [W], [128], [128], [Y], [128], tb.TERN_OUT_F32, ws,
                               ws_bytes=256)
    with pytest.raises(tb.TernError, match="ALIGN"):   # X not 16-byte aligned
        tb.tern_linear_grouped(tb.TERN_X_BF16, 1, [X.data_ptr() + 2], [128], [W], [128], [128], [Y], [128],
                               tb.TERN_OUT_F32, ws)
