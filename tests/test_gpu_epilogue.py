"""GPU-vs-oracle parity of the output forms: bf16 and fp16 outputs, fp16
activations, the fused gate+up SwiGLU epilogue over the GLU tile layout,
the row-wise repack (aligned and unaligned sources) and the workspace
maintenance calls.

Tolerances (written out per test, derived from the arithmetic):
  * fp32 results: |y - y_ref| <= 1e-4 * B, B = sum_k |x w| (the layer's bound);
  * an output rounded to bf16 / fp16 adds half an ulp of the result:
    2^-8 |y| (8 significant bits) / 2^-11 |y| (11 bits, plus the fp16
    subnormal spacing 2^-24 as a floor);
  * h = silu(g) * u from fp32 g, u within eg = 1e-4 B_g and eu = 1e-4 B_u:
    silu is 1.1-Lipschitz, so |h - h_ref| <= 1.1 |u| eg + |silu(g)| eu +
    1.1 eg eu, plus a few fp32 roundings (16 * 2^-24 |h|), plus the output
    rounding.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_util import DEV, dev, gpu_pack, gpu_repack, host, tiled_from_ternary  # noqa: E402
from ternary_bit_weight_gb300 import binding as tb  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-4
ROUND = {tb.TERN_OUT_F32: 0.0, tb.TERN_OUT_BF16: 2.0 ** -8, tb.TERN_OUT_F16: 2.0 ** -11}
FLOOR = {tb.TERN_OUT_F32: 0.0, tb.TERN_OUT_BF16: 0.0, tb.TERN_OUT_F16: 2.0 ** -24}
TORCH_OUT = {tb.TERN_OUT_F32: torch.float32, tb.TERN_OUT_BF16: torch.bfloat16, tb.TERN_OUT_F16: torch.float16}


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


def out_tensor(M, n, out_type, pad=3):
    return torch.full((M, n + pad), float("nan"), dtype=TORCH_OUT[out_type], device=DEV)


def check(y_gpu, y_ref, bound, out_type, what):
    y = np.asarray(y_gpu, dtype=np.float64)
    lim = TOL * bound + ROUND[out_type] * (np.abs(y_ref) + TOL * bound) + FLOOR[out_type]
    bad = ~(np.abs(y - y_ref) <= lim)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside; first {i}: gpu {y[i]} "
                             f"ref {y_ref[i]} lim {lim[i]}")


# ------------------------------------------------------------------ repack

@pytest.mark.parametrize("N,K", [(1, 128), (300, 256), (1000, 1024)])
def test_repack_unaligned_source_bit_exact(N, K):
    # a packed source that is 4- but not 16-byte aligned takes the scalar-load path
    rng = np.random.default_rng(N)
    t = rand_ternary(rng, N, K)
    s = rand_scales(rng, N, K)
    packed = gpu_pack(t)
    buf = torch.zeros(packed.numel() + 16, dtype=torch.uint8, device=DEV)
    buf[4:4 + packed.numel()] = packed.reshape(-1)
    tiled = torch.empty(tb.tern_tiled_bytes(N, K), dtype=torch.uint8, device=DEV)
    tb.tern_repack(buf.data_ptr() + 4, dev(s.view(np.int16)), N, K, tiled, tiled.numel())
    ref, _ = oracle.repack(oracle.pack(t)[0], s, K)
    assert np.array_equal(host(tiled), ref)


def test_repack_grouped_bit_exact():
    # one launch over weights of several shapes (ragged N, K from 128), one
    # of them from a source that is 4- but not 16-byte aligned
    rng = np.random.default_rng(11)
    shapes = [(1000, 512), (1, 128), (300, 1024), (129, 256), (0, 256), (517, 640)]
    packed, scales, tiled, refs = [], [], [], []
    for i, (N, K) in enumerate(shapes):
        t, s = rand_ternary(rng, max(N, 1), K)[:N], rand_scales(rng, max(N, 1), K)[:N]
        if N == 0:
            packed.append(torch.zeros(16, dtype=torch.uint8, device=DEV))
            scales.append(torch.zeros(16, dtype=torch.int16, device=DEV))
            tiled.append(torch.zeros(16, dtype=torch.uint8, device=DEV))
            refs.append(None)
            continue
        p = gpu_pack(t)
        if i == 3:
            buf = torch.zeros(p.numel() + 16, dtype=torch.uint8, device=DEV)
            buf[4:4 + p.numel()] = p.reshape(-1)
            packed.append(buf.data_ptr() + 4)
            tiled_keep = buf
        else:
            packed.append(p)
        scales.append(dev(s.view(np.int16)))
        tiled.append(torch.full((tb.tern_tiled_bytes(N, K),), 0xAB, dtype=torch.uint8, device=DEV))
        refs.append(oracle.repack(oracle.pack(t)[0], s, K)[0])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tb.tern_repack_grouped(packed, scales, [n for n, _ in shapes], [k for _, k in shapes], tiled,
                           [t.numel() for t in tiled], err=err)
    torch.cuda.synchronize()
    del tiled_keep
    for (N, K), t, ref in zip(shapes, tiled, refs):
        if ref is not None:
            assert np.array_equal(host(t), ref), f"{N}x{K}"
    assert int(err.item()) == 0


@pytest.mark.parametrize("I,K", [(1, 128), (20, 256), (200, 512), (1000, 1024)])
def test_repack_glu_bit_exact(I, K):
    rng = np.random.default_rng(I + K)
    tg, tu = rand_ternary(rng, I, K), rand_ternary(rng, I, K)
    sg, su = rand_scales(rng, I, K), rand_scales(rng, I, K)
    # one fused [2I, K/4] tensor cut by offsets, as the pages store gate+up
    packed = gpu_pack(np.concatenate([tg, tu]))
    scales = dev(np.concatenate([sg, su]).view(np.int16))
    tiled = torch.empty(tb.tern_tiled_glu_bytes(I, K), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tb.tern_repack_glu(packed, scales, packed.data_ptr() + I * (K // 4), scales.data_ptr() + I * (K // 128) * 2,
                       I, K, tiled, err=err)
    ref, _ = oracle.repack_glu(oracle.pack(tg)[0], sg, oracle.pack(tu)[0], su, K)
    assert np.array_equal(host(tiled), ref)
    assert int(err.item()) == 0


# ------------------------------------------------------------ output forms

CASES = [(1, 1000), (5, 1000), (16, 300), (32, 1000), (40, 1000), (200, 520)]


@pytest.mark.parametrize("M,N", CASES)
@pytest.mark.parametrize("out_type", [tb.TERN_OUT_BF16, tb.TERN_OUT_F16])
def test_linear_ex_half_outputs(M, N, out_type):
    K = 512
    rng = np.random.default_rng(M * 7 + N + out_type)
    t, s = rand_ternary(rng, N, K), rand_scales(rng, N, K)
    x = rand_x(rng, M, K, False)
    tiled = tiled_from_ternary(t, s)
    splits = [N // 3, N - N // 3]
    Ys = [out_tensor(M, n, out_type) for n in splits]
    ws = torch.zeros(tb.tern_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    tb.tern_linear_ex(dev(x.view(np.int16)), tb.TERN_X_BF16, K, tiled, M, K, splits, Ys,
                      [n + 3 for n in splits], out_type, ws)
    y_ref, bound = oracle.linear(x, oracle.pack(t)[0], s, K)
    off = 0
    for Y, n in zip(Ys, splits):
        y = host(Y.float())
        assert np.all(np.isnan(y[:, n:])), "padding written"
        check(y[:, :n], y_ref[:, off:off + n], bound[:, off:off + n], out_type, f"M={M} split {n}")
        off += n


@pytest.mark.parametrize("M", [1, 3, 16, 20, 40, 300])
def test_linear_ex_fp16_activations(M):
    N, K = 700, 1024
    rng = np.random.default_rng(100 + M)
    t, s = rand_ternary(rng, N, K), rand_scales(rng, N, K)
    x = rand_x(rng, M, K, True)
    tiled = tiled_from_ternary(t, s)
    Y = out_tensor(M, N, tb.TERN_OUT_F32, pad=0)
    ws = torch.zeros(tb.tern_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    tb.tern_linear_ex(dev(x.view(np.int16)), tb.TERN_X_F16, K, tiled, M, K, [N], [Y], [N],
                      tb.TERN_OUT_F32, ws)
    y_ref, bound = oracle.linear(x, oracle.pack(t)[0], s, K, x_f16=True)
    check(host(Y), y_ref, bound, tb.TERN_OUT_F32, f"fp16 X M={M}")


# ------------------------------------------------------------------ SwiGLU

def swiglu_limit(g, u, bg, bu, h, out_type):
    eg, eu = TOL * bg, TOL * bu
    silu = g / (1 + np.exp(-g))
    base = 1.1 * np.abs(u) * eg + np.abs(silu) * eu + 1.1 * eg * eu + 16 * 2.0 ** -24 * np.abs(h)
    return base + ROUND[out_type] * (np.abs(h) + base) + FLOOR[out_type]


def run_swiglu(x, x_f16, tg, tu, sg, su, out_type):
    M, K = x.shape
    I = tg.shape[0]
    packed = gpu_pack(np.concatenate([tg, tu]))
    scales = dev(np.concatenate([sg, su]).view(np.int16))
    tiled = torch.empty(tb.tern_tiled_glu_bytes(I, K), dtype=torch.uint8, device=DEV)
    tb.tern_repack_glu(packed, scales, packed.data_ptr() + I * (K // 4), scales.data_ptr() + I * (K // 128) * 2,
                       I, K, tiled)
    H = out_tensor(M, I, out_type)
    ws = torch.zeros(tb.tern_swiglu_workspace_bytes(M, I, K), dtype=torch.uint8, device=DEV)
    tb.tern_linear_swiglu(dev(x.view(np.int16)), tb.TERN_X_F16 if x_f16 else tb.TERN_X_BF16, K, tiled, M, I, K,
                          H, I + 3, out_type, ws)
    assert tb.tern_workspace_error(ws) == 0
    return host(H.float())


@pytest.mark.parametrize("M,I", [(1, 200), (1, 1000), (7, 200), (16, 1000), (32, 1000), (33, 200), (300, 520)])
@pytest.mark.parametrize("out_type", [tb.TERN_OUT_F32, tb.TERN_OUT_BF16])
def test_linear_swiglu(M, I, out_type):
    K = 512
    rng = np.random.default_rng(M * 31 + I + out_type)
    tg, tu = rand_ternary(rng, I, K), rand_ternary(rng, I, K)
    sg, su = rand_scales(rng, I, K), rand_scales(rng, I, K)
    x = rand_x(rng, M, K, False)
    h = run_swiglu(x, False, tg, tu, sg, su, out_type)
    assert np.all(np.isnan(h[:, I:])), "padding written"
    g, bg = oracle.linear(x, oracle.pack(tg)[0], sg, K)
    u, bu = oracle.linear(x, oracle.pack(tu)[0], su, K)
    h_ref = oracle.swiglu(g, u)
    lim = swiglu_limit(g, u, bg, bu, h_ref, out_type)
    bad = ~(np.abs(h[:, :I] - h_ref) <= lim)
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3].tolist())


def test_linear_swiglu_fp16_in_fp16_out():
    M, I, K = 9, 333, 256
    rng = np.random.default_rng(9)
    tg, tu = rand_ternary(rng, I, K), rand_ternary(rng, I, K)
    sg, su = rand_scales(rng, I, K), rand_scales(rng, I, K)
    x = rand_x(rng, M, K, True)
    h = run_swiglu(x, True, tg, tu, sg, su, tb.TERN_OUT_F16)
    g, bg = oracle.linear(x, oracle.pack(tg)[0], sg, K, x_f16=True)
    u, bu = oracle.linear(x, oracle.pack(tu)[0], su, K, x_f16=True)
    h_ref = oracle.swiglu(g, u)
    lim = swiglu_limit(g, u, bg, bu, h_ref, tb.TERN_OUT_F16)
    assert np.all(np.abs(h[:, :I] - h_ref) <= lim)


@pytest.mark.parametrize("M", [1, 64])
def test_linear_swiglu_27b_gate_up_sampled(M):
    # full-size 27B-class gate+up (I = 27648, K = 5120), sampled outputs
    wl = synth.WORKLOADS["dec27b"]
    lin = next(l for l in wl.linears if l.name == "gate_up")
    I, K = lin.splits[0], lin.K
    t, s = synth.weights(wl, 0, lin)
    packed = gpu_pack(t)
    scales = dev(s.view(np.int16))
    tiled = torch.empty(tb.tern_tiled_glu_bytes(I, K), dtype=torch.uint8, device=DEV)
    tb.tern_repack_glu(packed, scales, packed.data_ptr() + I * (K // 4), scales.data_ptr() + I * (K // 128) * 2,
                       I, K, tiled)
    x = synth.activations(wl, 0, lin, M)
    H = torch.full((M, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(tb.tern_swiglu_workspace_bytes(M, I, K), dtype=torch.uint8, device=DEV)
    tb.tern_linear_swiglu(dev(x.view(np.int16)), tb.TERN_X_BF16, K, tiled, M, I, K, H, I, tb.TERN_OUT_BF16, ws)
    h = host(H.float())
    assert np.all(np.isfinite(h))
    cols = np.array(sorted({0, 1, 15, 16, 17, 31, 32, 4095, 13824, I - 17, I - 16, I - 1}))
    toks = np.array(sorted({0, M // 2, M - 1}))
    pk, _ = oracle.pack(t[np.concatenate([cols, I + cols])])
    sc = s[np.concatenate([cols, I + cols])]
    y, b = oracle.linear(x[toks], pk, sc, K)
    g, u = y[:, :cols.size], y[:, cols.size:]
    bg, bu = b[:, :cols.size], b[:, cols.size:]
    h_ref = oracle.swiglu(g, u)
    lim = swiglu_limit(g, u, bg, bu, h_ref, tb.TERN_OUT_BF16)
    assert np.all(np.abs(h[np.ix_(toks, cols)] - h_ref) <= lim)


# ------------------------------------------------------ workspace upkeep

def test_workspace_error_word_and_reset():
    N, K, M = 256, 256, 4
    rng = np.random.default_rng(3)
    t, s = rand_ternary(rng, N, K), rand_scales(rng, N, K)
    tiled = tiled_from_ternary(t, s)
    ws = torch.zeros(tb.tern_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    Y = torch.empty((M, N), device=DEV)
    tb.tern_linear(dev(rand_x(rng, M, K, False).view(np.int16)), K, tiled, M, N, K, Y, N, ws)
    assert tb.tern_workspace_error(ws) == 0
    ws.fill_(7)
    assert tb.tern_workspace_error(ws) == 0x07070707
    tb.tern_workspace_reset(ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0


@pytest.mark.parametrize("M", [17, 200, 300])
@pytest.mark.parametrize("out_type", [tb.TERN_OUT_F32, tb.TERN_OUT_BF16, tb.TERN_OUT_F16])
def test_linear_ex_tile_aligned_outputs(M, out_type):
    # outputs cut at multiples of 128 rows (the fused-QKV shape class), the
    # last one ragged, with padded row strides: the GEMM writes these by TMA
    K = 512
    splits = [256, 128, 300]
    N = sum(splits)
    rng = np.random.default_rng(M + out_type)
    t, s = rand_ternary(rng, N, K), rand_scales(rng, N, K)
    x = rand_x(rng, M, K, False)
    tiled = tiled_from_ternary(t, s)
    pad = 8 if out_type == tb.TERN_OUT_F32 else 16     # rows stay 16-byte aligned
    Ys = [out_tensor(M, n, out_type, pad=pad) for n in splits]
    ws = torch.zeros(tb.tern_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    tb.tern_linear_ex(dev(x.view(np.int16)), tb.TERN_X_BF16, K, tiled, M, K, splits, Ys, [n + pad for n in splits],
                      out_type, ws)
    y_ref, bound = oracle.linear(x, oracle.pack(t)[0], s, K)
    off = 0
    for Y, n in zip(Ys, splits):
        y = host(Y.float())
        assert np.all(np.isnan(y[:, n:])), "padding written"
        check(y[:, :n], y_ref[:, off:off + n], bound[:, off:off + n], out_type, f"M={M} split {n}")
        off += n
