"""Pins for the CPU oracle: checks that tie it to the pages and to mathematics.

Every oracle function is checked here against something other than itself:
hand-worked bytes from the packing rule ("Ternary embedding model in vLLM",
2kiu.com/news/5082861, §3.1), exhaustive comparison with independent
implementations (numpy's IEEE half, a vectorised restatement of the page's
unpack routine), closed forms, brute force against a dense fp64 matmul, and
special cases chosen so that a dropped term, a wrong sign, a wrong group
index or a transposed operand fails at least one test.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from conftest import golden_lines


# ------------------------------------------------------------ scalar formats

def test_fp16_decode_matches_numpy_exhaustively():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decode_matches_float32_top_half_exhaustively():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# ------------------------------------------------------------- packing rule

def test_code_mapping_from_the_rule():
    # 00 -> 0, 01 -> +1, 10 -> -1, 11 -> reserved, read as 0
    assert [oracle.code_to_ternary(c) for c in range(4)] == [0, 1, -1, 0]


def test_unpack_hand_worked_bytes():
    n = 0
    for parts in golden_lines("packing_rule.txt"):
        if parts[0] != "unpack":
            continue
        byte = int(parts[1], 16)
        want = [int(v) for v in parts[2:6]]
        t, reserved = oracle.unpack(np.array([[byte]], dtype=np.uint8), 4)
        assert t[0].tolist() == want, (hex(byte), t[0].tolist(), want)
        codes = [(byte >> (2 * j)) & 3 for j in range(4)]
        assert reserved == codes.count(3)
        n += 1
    assert n >= 15


def test_pack_hand_worked_bytes():
    n = 0
    for parts in golden_lines("packing_rule.txt"):
        if parts[0] != "pack":
            continue
        t = np.array([[int(v) for v in parts[1:5]]], dtype=np.int8)
        packed, bad = oracle.pack(t)
        assert bad == 0
        assert packed[0, 0] == int(parts[5], 16), (parts, hex(packed[0, 0]))
        n += 1
    assert n >= 5


def _page_unpack(packed):
    """The page's unpack routine ([EMB] §3.1) restated with numpy: stack the
    four 2-bit windows at shifts 0,2,4,6 on the last axis, then map
    1 -> +1, 2 -> -1, everything else -> 0."""
    p = packed.astype(np.uint8)
    codes = np.stack([(p >> s) & 3 for s in (0, 2, 4, 6)], axis=-1)
    vals = np.where(codes == 1, 1, np.where(codes == 2, -1, 0))
    return vals.reshape(p.shape[0], -1).astype(np.int8)


def test_unpack_all_256_bytes_matches_page_routine():
    allbytes = np.arange(256, dtype=np.uint8).reshape(4, 64)
    t, reserved = oracle.unpack(allbytes, 256)
    assert np.array_equal(t, _page_unpack(allbytes))
    # each of the 4 positions holds code 11 in exactly 64 of the 256 bytes
    assert reserved == 4 * 64


def test_pack_unpack_round_trips():
    rng = np.random.default_rng(1)
    t = rng.integers(-1, 2, size=(37, 64), dtype=np.int8)
    packed, bad = oracle.pack(t)
    assert bad == 0
    back, reserved = oracle.unpack(packed, 64)
    assert reserved == 0 and np.array_equal(back, t)
    # pack(unpack(bytes)) canonicalises the reserved code 11 to 00
    raw = rng.integers(0, 256, size=(5, 16), dtype=np.uint8)
    tt, _ = oracle.unpack(raw, 64)
    again, bad = oracle.pack(tt)
    canon = raw.copy()
    for s in (0, 2, 4, 6):
        is11 = ((raw >> s) & 3) == 3
        canon[is11] &= np.uint8(~(3 << s) & 0xFF)
    assert bad == 0 and np.array_equal(again, canon)


def test_pack_counts_values_outside_ternary():
    t = np.array([[1, 2, -1, -3, 0, 0, 0, 5]], dtype=np.int8)
    packed, bad = oracle.pack(t)
    assert bad == 3
    back, _ = oracle.unpack(packed, 8)
    assert back.tolist() == [[1, 0, -1, 0, 0, 0, 0, 0]]


def test_pack_layout_is_row_major_bytes():
    # row n holds byte k/4 of its own K codes ([EMB] §2.2: packed [N, K/4])
    t = np.zeros((3, 8), dtype=np.int8)
    t[2, 5] = -1   # row 2, byte 1, position 1 -> 10 << 2
    packed, _ = oracle.pack(t)
    want = np.zeros((3, 2), dtype=np.uint8)
    want[2, 1] = 0x08
    assert np.array_equal(packed, want)


# ----------------------------------------------------------------- tiled

def _one_weight(N, K, n, k, t):
    tt = np.zeros((N, K), dtype=np.int8)
    tt[n, k] = t
    packed, _ = oracle.pack(tt)
    scales = np.zeros((N, K // 128), dtype=np.uint16)
    return packed, scales


def test_tiled_hand_worked_code_positions():
    n_checked = 0
    for parts in golden_lines("tiled_layout.txt"):
        if parts[0] != "code":
            continue
        N, K, n, k, t, off, val = [int(v) for v in parts[1:6]] + [int(parts[6]), int(parts[7], 16)]
        packed, scales = _one_weight(N, K, n, k, t)
        tiled, _ = oracle.repack(packed, scales, K)
        R, G = (N + 127) // 128, K // 128
        codes = tiled[: R * G * 4096]
        assert codes[off] == val, (parts, hex(codes[off]))
        others = np.delete(codes, off)
        assert np.all(others == 0x55), parts
        n_checked += 1
    assert n_checked >= 10


def test_tiled_hand_worked_scale_positions():
    for parts in golden_lines("tiled_layout.txt"):
        if parts[0] != "scale":
            continue
        N, K, n, g, off = [int(v) for v in parts[1:6]]
        packed = np.zeros((N, K // 4), dtype=np.uint8)
        scales = np.zeros((N, K // 128), dtype=np.uint16)
        scales[n, g] = 0xABCD
        tiled, _ = oracle.repack(packed, scales, K)
        R, G = (N + 127) // 128, K // 128
        sc = tiled[R * G * 4096:]
        assert tiled[off] == 0xCD and tiled[off + 1] == 0xAB, parts
        assert int(np.count_nonzero(sc)) == 2, parts


@pytest.mark.parametrize("N,K", [(16, 128), (20, 256), (1, 128), (33, 384), (130, 1024), (256, 256)])
def test_repack_round_trip(N, K):
    rng = np.random.default_rng(N * 1000 + K)
    raw = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    scales = rng.integers(0, 1 << 16, size=(N, K // 128), dtype=np.uint16)
    tiled, reserved = oracle.repack(raw, scales, K)
    assert tiled.size == oracle.tiled_bytes(N, K) == ((N + 127) // 128) * (K // 128) * 4352
    codes = np.stack([(raw >> s) & 3 for s in (0, 2, 4, 6)])
    assert reserved == int((codes == 3).sum())
    packed2, scales2, invalid = oracle.unrepack(tiled, N, K)
    assert invalid == 0
    t_raw, _ = oracle.unpack(raw, K)
    t_back, r2 = oracle.unpack(packed2, K)
    assert r2 == 0
    assert np.array_equal(t_back, t_raw)   # same weights, code 11 canonicalised to 00
    assert np.array_equal(scales2, scales)
    # padding rows of the last tile hold weight 0 (v = 1) and scale 0
    R, G = (N + 127) // 128, K // 128
    if N % 128:
        tt = np.zeros(((N + 127) // 128 * 128, K), dtype=np.int8)
        tt[:N] = t_raw
        p_full, _ = oracle.pack(tt)
        s_full = np.zeros((tt.shape[0], G), dtype=np.uint16)
        s_full[:N] = scales
        tiled_full, _ = oracle.repack(p_full, s_full, K)
        assert np.array_equal(tiled_full, tiled)


def test_unrepack_counts_invalid_biased_code():
    N, K = 16, 128
    tiled, _ = oracle.repack(np.zeros((N, K // 4), np.uint8), np.zeros((N, 1), np.uint16), K)
    tiled[0] |= 0x03     # v = 3 at weight (0, 0)
    _, _, invalid = oracle.unrepack(tiled, N, K)
    assert invalid == 1


# ------------------------------------------------------------------ linear

def _dequant_dense(packed, scales, K):
    """Dense fp64 W[N, K] = t * s, built from the pinned unpack and numpy."""
    t, _ = oracle.unpack(packed, K)
    s = np.asarray(scales, np.uint16).view(np.float16).astype(np.float64)
    return t.astype(np.float64) * np.repeat(s, 128, axis=1)


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (3, 8, 256), (2, 5, 128), (3, 7, 384)])
def test_linear_brute_force_against_dense_matmul(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    packed, _ = oracle.pack(t)
    scales = np.array([[synth.round_fp16(v) for v in row]
                       for row in rng.uniform(0.005, 0.05, size=(N, K // 128))], dtype=np.uint16)
    x = np.array([[synth.round_bf16(v) for v in row] for row in rng.standard_normal((M, K))],
                 dtype=np.uint16)
    y, bound = oracle.linear(x, packed, scales, K)
    xf = synth.bf16_bits_to_float(x)
    W = _dequant_dense(packed, scales, K)
    ref = xf @ W.T                      # [M, N]: X times W transposed
    assert y.shape == (M, N)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(bound, np.abs(xf) @ np.abs(W).T, rtol=1e-12, atol=1e-14)
    assert np.all(np.abs(y) <= bound + 1e-15)


def test_linear_all_zero_codes_gives_exact_zero():
    K, N, M = 256, 4, 2
    packed = np.zeros((N, K // 4), np.uint8)
    packed[1] = 0xFF          # reserved code everywhere: still zero weight
    scales = np.full((N, K // 128), 0x3C00, np.uint16)   # 1.0
    x = np.full((M, K), 0x3F80, np.uint16)                # 1.0
    y, bound = oracle.linear(x, packed, scales, K)
    assert np.all(y == 0.0) and np.all(bound == 0.0)


def test_linear_all_plus_one_unit_scale_gives_row_sums():
    K, N, M = 256, 3, 2
    rng = np.random.default_rng(7)
    packed = np.full((N, K // 4), 0x55, np.uint8)         # every weight +1
    scales = np.full((N, K // 128), 0x3C00, np.uint16)    # s = 1.0
    x = np.array([[synth.round_bf16(v) for v in row] for row in rng.standard_normal((M, K))],
                 dtype=np.uint16)
    y, _ = oracle.linear(x, packed, scales, K)
    xf = synth.bf16_bits_to_float(x)
    for m in range(M):
        assert np.all(y[m] == math.fsum(xf[m]))
    # all -1: the negation
    y2, _ = oracle.linear(x, np.full((N, K // 4), 0xAA, np.uint8), scales, K)
    assert np.array_equal(y2, -y)


def test_linear_one_hot_x_selects_a_weight_and_its_group_scale():
    K, N = 384, 6
    rng = np.random.default_rng(3)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    packed, _ = oracle.pack(t)
    # group g of row n gets scale 2^-(n+3g): any wrong group index changes y
    scales = np.array([[synth.round_fp16(2.0 ** -(n + 3 * g)) for g in range(K // 128)]
                       for n in range(N)], dtype=np.uint16)
    for k in (0, 1, 127, 128, 129, 255, 256, 383):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y, _ = oracle.linear(x, packed, scales, K)
        want = [t[n, k] * 2.0 ** -(n + 3 * (k // 128)) for n in range(N)]
        assert y[0].tolist() == want, k


def test_linear_power_of_two_scaling_is_exact():
    K, N, M = 256, 5, 3
    rng = np.random.default_rng(11)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    packed, _ = oracle.pack(t)
    s1 = np.array([[synth.round_fp16(v) for v in row] for row in rng.uniform(0.01, 0.04, (N, 2))],
                  np.uint16)
    s2 = np.array([[synth.round_fp16(2 * oracle.fp16_to_double(int(v))) for v in row] for row in s1],
                  np.uint16)
    x = np.array([[synth.round_bf16(v) for v in row] for row in rng.standard_normal((M, K))],
                 np.uint16)
    y1, _ = oracle.linear(x, packed, s1, K)
    y2, _ = oracle.linear(x, packed, s2, K)
    assert np.array_equal(y2, 2 * y1)     # linear in s
    x2 = np.array([[synth.round_bf16(-0.5 * synth.bf16_bits_to_float(np.array([v]))[0]) for v in row]
                   for row in x], np.uint16)
    y3, _ = oracle.linear(x2, packed, s1, K)
    assert np.array_equal(y3, -0.5 * y1)  # linear in x


def test_linear_cols_matches_full_linear():
    K, N, M = 256, 9, 2
    rng = np.random.default_rng(5)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    packed, _ = oracle.pack(t)
    scales = rng.integers(0x2000, 0x2C00, size=(N, 2), dtype=np.uint16)
    x = rng.integers(0x3E00, 0x4000, size=(M, K), dtype=np.uint16)
    y, b = oracle.linear(x, packed, scales, K)
    cols = [8, 0, 3]
    yc, bc = oracle.linear_cols(x, packed, scales, K, cols)
    assert np.array_equal(yc, y[:, cols]) and np.array_equal(bc, b[:, cols])


# --------------------------------------------------------------- generator

def test_splitmix_known_answers_and_counter_form():
    # published SplitMix64 outputs for state 0
    seq = synth.sequential_splitmix(0, 3)
    assert [int(v) for v in seq] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # the counter form equals the sequential generator started at the stream key
    key = synth.stream_key(0, synth.stream_id("a/b"))
    assert np.array_equal(synth.raw(0, synth.stream_id("a/b"), 50), synth.sequential_splitmix(key, 50))


def test_generator_distributions():
    t = synth.ternary("dist/t", 300000, 0.35)
    p = np.bincount(t.astype(np.int64) + 1, minlength=3) / t.size
    assert abs(p[1] - 0.35) < 0.005 and abs(p[0] - 0.325) < 0.005 and abs(p[2] - 0.325) < 0.005
    s = synth.fp16_bits_to_float(synth.scales_uniform("dist/s", 100000, 0.005, 0.05))
    assert s.min() >= 0.005 - 1e-5 and s.max() <= 0.05 + 1e-4 and abs(s.mean() - 0.0275) < 3e-4
    ln = np.log(synth.fp16_bits_to_float(synth.scales_lognormal("dist/l", 100000, -4.0, 0.5)))
    assert abs(ln.mean() + 4.0) < 0.01 and abs(ln.std() - 0.5) < 0.01
    x = synth.bf16_bits_to_float(synth.normal_bf16("dist/x", 100000))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_rounding_is_nearest_even():
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 4, 2000),
                           [1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 2 ** -24, 3 * 2 ** -25, 65519.0]])
    for v in vals:   # fp16: numpy rounds double -> half correctly (RNE)
        assert synth.round_fp16(v) == int(np.array([v]).astype(np.float16).view(np.uint16)[0]), v
    for v in list(rng.standard_normal(2000)) + [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8)]:
        b = synth.round_bf16(v)
        got = synth.bf16_bits_to_float(np.array([b]))[0]
        # nearest: no other bf16 is closer; ties go to the even pattern
        nb = [synth.bf16_bits_to_float(np.array([(b + d) & 0xFFFF]))[0] for d in (-1, 1)]
        for o in nb:
            assert abs(v - got) < abs(v - o) or (abs(v - got) == abs(v - o) and b % 2 == 0), v


def test_prefix_and_row_range_consistency():
    wl = synth.WORKLOADS["single"]
    lin = wl.linears[0]
    x8 = synth.activations(wl, 0, lin, 8)
    x1 = synth.activations(wl, 0, lin, 1)
    assert np.array_equal(x8[:1], x1)
    t, s = synth.weights(wl, 0, lin)
    t2, s2 = synth.weights(wl, 0, lin, rows=slice(500, 530))
    assert np.array_equal(t[500:530], t2) and np.array_equal(s[500:530], s2)


# ------------------------------------------------------ fp16 activations

def test_linear_fp16_activations_match_dense_matmul():
    # x given as IEEE half bits ("Ternary embedding model in vLLM" §4.2: the
    # page's kernel reads half activations); brute force against numpy's half
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 256
    t = rng.integers(-1, 2, (N, K)).astype(np.int8)
    packed, _ = oracle.pack(t)
    s = rng.uniform(0.01, 0.04, (N, K // 128)).astype(np.float16)
    x = rng.standard_normal((M, K)).astype(np.float16)
    y, b = oracle.linear(x.view(np.uint16), packed, s.view(np.uint16), K, x_f16=True)
    w = t.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)
    ref = x.astype(np.float64) @ w.T
    assert np.allclose(y, ref, rtol=0, atol=1e-12)
    assert np.allclose(b, np.abs(x.astype(np.float64)) @ np.abs(w).T, rtol=1e-12)
    # the same bits read as bf16 give a different answer: the flag is used
    y2, _ = oracle.linear(x.view(np.uint16), packed, s.view(np.uint16), K, x_f16=False)
    assert not np.allclose(y, y2)


# ------------------------------------------------------------------ SwiGLU

def test_swiglu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 2.5, -30.0, 30.0])
    u = np.array([3.0, 1.0, 2.0, -0.5, 1.0, 1.0])
    h = oracle.swiglu(g, u)
    sig = [1 / (1 + math.exp(-v)) for v in g]
    want = [gv * sv * uv for gv, sv, uv in zip(g, sig, u)]
    assert np.allclose(h, want, rtol=1e-15, atol=0)
    assert h[0] == 0.0                                  # silu(0) = 0
    assert abs(h[4]) < 1e-11 and abs(h[5] - 30.0) < 1e-11   # tails: 0 and identity
    # gate and up are not interchangeable
    assert not np.allclose(oracle.swiglu(u, g), h)


def test_glu_layout_rows_from_its_definition():
    # blocks of 16 rows alternate between gate and up; I = 20 -> 64 rows
    assert oracle.glu_rows(20) == 64 and oracle.glu_rows(16) == 32 and oracle.glu_rows(1) == 32
    want = {0: ("gate", 0), 15: ("gate", 15), 16: ("up", 0), 31: ("up", 15),
            32: ("gate", 16), 47: ("gate", 31), 48: ("up", 16), 63: ("up", 31)}
    for n, src in want.items():
        assert oracle.glu_source(n) == src


def test_repack_glu_rows_unrepack_to_their_sources():
    rng = np.random.default_rng(5)
    I, K = 20, 256
    tg = rng.integers(-1, 2, (I, K)).astype(np.int8)
    tu = rng.integers(-1, 2, (I, K)).astype(np.int8)
    pg, _ = oracle.pack(tg)
    pu, _ = oracle.pack(tu)
    sg = rng.integers(0x2000, 0x2C00, (I, K // 128)).astype(np.uint16)
    su = rng.integers(0x2000, 0x2C00, (I, K // 128)).astype(np.uint16)
    tiled, bad = oracle.repack_glu(pg, sg, pu, su, K)
    assert bad == 0
    rows = oracle.glu_rows(I)
    packed, scales, _ = oracle.unrepack(tiled, rows, K)
    t_all, _ = oracle.unpack(packed, K)
    # row 16 of the GLU weight is up row 0, row 33 gate row 17, rows of i >= 20 zero
    assert np.array_equal(t_all[16], tu[0]) and np.array_equal(scales[16], su[0])
    assert np.array_equal(t_all[33], tg[17]) and np.array_equal(scales[33], sg[17])
    assert np.array_equal(t_all[0], tg[0]) and np.array_equal(t_all[50], tu[18])
    assert not t_all[36].any() and not scales[36].any()      # gate row 20: padding
    assert not t_all[52].any() and not t_all[63].any()       # up rows 20, 31: padding


def test_swiglu_of_the_layer_by_hand():
    # one-hot x at k0: gate = x * t_g * s_g, up = x * t_u * s_u
    K = 128
    x = np.zeros((1, K), dtype=np.float32)
    x[0, 7] = 1.5
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    tg = np.zeros((1, K), dtype=np.int8); tg[0, 7] = 1
    tu = np.zeros((1, K), dtype=np.int8); tu[0, 7] = -1
    s = np.array([[0x3800]], dtype=np.uint16)           # 0.5
    g, _ = oracle.linear(xb, oracle.pack(tg)[0], s, K)
    u, _ = oracle.linear(xb, oracle.pack(tu)[0], s, K)
    h = oracle.swiglu(g, u)
    gv, uv = 0.75, -0.75
    assert g[0, 0] == gv and u[0, 0] == uv
    assert abs(h[0, 0] - gv / (1 + math.exp(-gv)) * uv) < 1e-15


# ------------------------------------------------------- int8 activations

def _bf16(vals):
    x = np.array(vals, dtype=np.float32).reshape(1, -1)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def test_quantize_x_hand_worked():
    # absmax 2 -> 127/2 = 63.5 per unit; 1.0 -> 63.5 -> 64 (tie to even),
    # -2 -> -127, 0.5 -> 31.75 -> 32, 0.25 -> 15.875 -> 16; a = 2/127
    q, a = oracle.quantize_x(_bf16([1.0, -2.0, 0.5, 0.25] + [0.0] * 124))
    assert q[0, :4].tolist() == [64, -127, 32, 16] and not q[0, 4:].any()
    assert a[0] == np.float32(2.0) / np.float32(127.0)
    # absmax 127: the scale is exactly 1 and ties go to even
    q, a = oracle.quantize_x(_bf16([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 126.0, -127.0] + [0.0] * 120))
    assert q[0, :8].tolist() == [127, 0, 2, 2, 0, -2, 126, -127] and a[0] == 1.0
    # a row of zeros: a = 0, q = 0
    q, a = oracle.quantize_x(np.zeros((1, 128), dtype=np.uint16))
    assert a[0] == 0.0 and not q.any()
    # fp16 bits are read as fp16
    xh = np.array([[3.0, -1.5] + [0.0] * 126], dtype=np.float16)
    q, a = oracle.quantize_x(xh.view(np.uint16), x_f16=True)
    assert q[0, :2].tolist() == [127, -64] and a[0] == np.float32(3.0) / np.float32(127.0)


def test_linear_i8_matches_integer_matmul():
    rng = np.random.default_rng(8)
    M, N, K = 3, 7, 384
    t = rng.integers(-1, 2, (N, K)).astype(np.int8)
    q = rng.integers(-127, 128, (M, K)).astype(np.int8)
    a = rng.uniform(0.001, 0.1, M).astype(np.float32)
    s = rng.uniform(0.005, 0.05, (N, K // 128)).astype(np.float16)
    packed, _ = oracle.pack(t)
    y, b = oracle.linear_i8(q, a, packed, s.view(np.uint16), K)
    G = K // 128
    # integer group sums from numpy's int64 matmul, then the scales
    isum = np.stack([q[:, 128 * g:128 * g + 128].astype(np.int64) @ t[:, 128 * g:128 * g + 128].T.astype(np.int64)
                     for g in range(G)], axis=-1)                      # [M, N, G]
    ref = a.astype(np.float64)[:, None] * np.einsum("mng,ng->mn", isum.astype(np.float64), s.astype(np.float64))
    assert np.allclose(y, ref, rtol=1e-13, atol=0)
    w = t.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)
    mag = a.astype(np.float64)[:, None] * (np.abs(q.astype(np.float64)) @ np.abs(w).T)
    assert np.allclose(b, mag, rtol=1e-13)


# ------------------------------------------------------ INT8 group scales

def test_quantize_scales_hand_worked():
    # row max 0.05 -> f = 0.05/127; 0.025 -> 63.5 -> 64 (tie to even)
    s = np.array([[0.05, 0.025, 0.0125, -0.05]], dtype=np.float16)
    q8, f = oracle.quantize_scales(s.view(np.uint16), 512)
    m = np.float32(np.float16(0.05))
    assert f[0] == m / np.float32(127.0)
    inv = np.float32(127.0) / m
    want = [int(np.rint(np.float32(np.float16(v)) * inv)) for v in (0.05, 0.025, 0.0125, -0.05)]
    assert q8[0].tolist() == want and want[0] == 127 and want[3] == -127
    # exactly representable case: scales 1, 0.5, 0.25 with max 1 -> f = 1/127
    s = np.array([[1.0, 0.5, 0.25, -1.0]], dtype=np.float16)
    q8, f = oracle.quantize_scales(s.view(np.uint16), 512)
    assert q8[0].tolist() == [127, 64, 32, -127]          # 63.5 -> 64, 31.75 -> 32
    q8, f = oracle.quantize_scales(np.zeros((1, 2), dtype=np.uint16), 256)
    assert f[0] == 0.0 and not q8.any()


def test_repack_s8_layout_by_hand():
    rng = np.random.default_rng(2)
    N, K = 130, 256                                      # two row tiles, the second ragged
    t = rng.integers(-1, 2, (N, K)).astype(np.int8)
    packed, _ = oracle.pack(t)
    q8 = rng.integers(-127, 128, (N, K // 128)).astype(np.int8)
    f = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    tiled = oracle.repack_s8(packed, q8, f, K)
    R, G = 2, 2
    assert tiled.size == oracle.tiled_s8_bytes(N, K) == R * G * 4224 + R * 512
    base = R * G * 4096
    # unit (b=1, g=0) starts at base + (1*2 + 0)*128; its row 1 is weight row 129
    assert tiled.view(np.int8)[base + 2 * 128 + 1] == q8[129, 0]
    assert tiled.view(np.int8)[base + 1 * 128 + 5] == q8[5, 1]
    assert not tiled[base + 2 * 128 + 2:base + 3 * 128].any()    # rows 130..255: padding
    fac = tiled[base + R * G * 128:].view(np.float32)
    assert fac[129] == f[129] and fac[0] == f[0] and not fac[130:].any()
    # the code units are those of the plain tiled layout
    plain, _ = oracle.repack(packed, np.zeros((N, 2), dtype=np.uint16), K)
    assert np.array_equal(tiled[:base], plain[:base])


def test_linear_s8_matches_dense_matmul():
    rng = np.random.default_rng(12)
    M, N, K = 2, 5, 256
    t = rng.integers(-1, 2, (N, K)).astype(np.int8)
    q8 = rng.integers(-127, 128, (N, K // 128)).astype(np.int8)
    f = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    y, _ = oracle.linear_s8(xb, oracle.pack(t)[0], q8, f, K)
    w = t.astype(np.float64) * np.repeat(q8.astype(np.float64), 128, axis=1) * f.astype(np.float64)[:, None]
    xd = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(y, xd @ w.T, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------- zero units

def test_zero_units_by_hand():
    K = 256
    t = np.zeros((130, K), dtype=np.int8)          # 2 row tiles x 2 groups, second tile ragged
    t[5, 200] = -1                                  # unit (0, 1)
    t[129, 3] = 1                                   # unit (1, 0)
    packed, _ = oracle.pack(t)
    assert oracle.zero_units(packed, K).tolist() == [1, 0, 0, 1]
    # a reserved code 11 reads as 0, so it leaves a unit zero
    packed[0, 0] = 0b11
    assert oracle.zero_units(packed, K).tolist() == [1, 0, 0, 1]
    assert oracle.zero_units(oracle.pack(np.ones((1, 128), dtype=np.int8))[0], 128).tolist() == [0]
