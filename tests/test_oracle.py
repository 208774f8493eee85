"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what it pins and where the fact comes from: numpy's independent binary16
conversion, exact rational or integer arithmetic, closed forms and invariants of the method, and
the worked example printed on the source pages.  A plausible slip in the oracle (a dropped term,
a wrong sign or index, a transposed operand, the wrong rounding) fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from weight_quantized_linear_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------------------------
# binary16 conversion: pinned against numpy's own float16 implementation
# ------------------------------------------------------------------------------------------------

def test_half_to_float_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_float(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_matches_numpy_including_ties_and_subnormals():
    rng = np.random.default_rng(1)
    vals = [rng.standard_normal(200000).astype(np.float32) * s for s in (1e-6, 1e-3, 1.0, 100.0, 3e4)]
    # exact midpoints between adjacent fp16 values (ties), normal and subnormal, both signs
    h = np.arange(0, 0x7bff, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    special = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, np.inf, -np.inf, 2.0 ** -25,
                        2.0 ** -24, 1.5 * 2.0 ** -24, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -26], np.float32)
    x = np.concatenate(vals + [mid, -mid, special])
    ours = oracle.float_to_half(x).view(np.uint16)
    with np.errstate(over="ignore"):  # +-1e9 and +-inf overflow to +-inf on purpose
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------------------------------------
# AWQ int4 quantisation and packing
# ------------------------------------------------------------------------------------------------

def _exact_grid_weight(K, N, G, seed=3):
    """Weights that are exactly (c - z) * 2^-6 with codes c covering 0 and 15 in every group."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(K, N))
    for g in range(K // G):
        codes[g * G, :] = 0
        codes[g * G + 1, :] = 15
    zs = rng.integers(1, 15, size=(K // G, N))
    z_full = np.repeat(zs, G, axis=0)
    W = ((codes - z_full) * 2.0 ** -6).astype(np.float32)
    return W, codes, zs


@pytest.mark.parametrize("G", [32, 64, 128])
def test_awq_recovers_exactly_representable_weights(G):
    # Closed form: if every group holds (c - z) * s for an fp16 scale s with both code 0 and code 15
    # present, min/max quantisation returns exactly s, z and c, and dequantisation is exact.
    K, N = 2 * G, 40
    W, codes, zs = _exact_grid_weight(K, N, G)
    qw, s, qz = oracle.awq_quantize(W, G)
    q, z = oracle.awq_unpack(qw, qz, K, N, G)
    assert np.array_equal(q, codes)
    assert np.array_equal(z, zs)
    assert np.all(s.astype(np.float32) == np.float32(2.0 ** -6))
    assert np.array_equal(oracle.awq_dequant(qw, s, qz, K, N, G), W)


def test_awq_nibble_layout_is_column_n_at_bits_4_n_mod_8():
    # Layout pin by construction: a single nonzero code per word at a known column.
    G, K, N = 32, 32, 32
    W, codes, zs = _exact_grid_weight(K, N, G, seed=11)
    qw, s, qz = oracle.awq_quantize(W, G)
    for k in range(K):
        for n in range(N):
            assert (int(qw[k, n // 8]) >> (4 * (n % 8))) & 15 == codes[k, n]
    for n in range(N):
        assert (int(qz[0, n // 8]) >> (4 * (n % 8))) & 15 == zs[0, n]


def test_awq_unpack_roundtrip_exhaustive_over_positions_and_values():
    # Every value 0..15 at every nibble position of a word survives pack -> unpack.
    G, K, N = 32, 32, 128
    codes = np.zeros((K, N), np.int64)
    for n in range(N):
        codes[:, n] = (np.arange(K) + n) % 16
    codes[0, :] = 0
    codes[1, :] = 15
    z = 7
    W = ((codes - z) * 2.0 ** -5).astype(np.float32)
    qw, s, qz = oracle.awq_quantize(W, G)
    q, zz = oracle.awq_unpack(qw, qz, K, N, G)
    assert np.array_equal(q, codes)
    assert np.all(zz == z)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_awq_error_bound_and_code_range(G):
    # For groups whose range contains zero: |w - (q - z) s| <= s/2 + 15 |s16 - s32| (+ fp32 slack),
    # the group minimum maps to code 0 and the maximum to code 14 or 15.
    K, N = 512, 256
    W = inputs.weight(K, N, seed=5, outliers=True)
    qw, s, qz = oracle.awq_quantize(W, G)
    q, z = oracle.awq_unpack(qw, qz, K, N, G)
    deq = oracle.awq_dequant(qw, s, qz, K, N, G).astype(np.float64)
    Wg = W.reshape(K // G, G, N).astype(np.float64)
    mn, mx = Wg.min(axis=1), Wg.max(axis=1)
    s16 = s.astype(np.float64)
    s_exact = (mx - mn) / 15.0
    bound = s16 / 2 + 15 * np.abs(s16 - s_exact) + 1e-7 * np.abs(Wg).max(axis=1)
    err = np.abs(deq.reshape(K // G, G, N) - Wg).max(axis=1)
    straddle = (mn <= 0) & (mx >= 0)
    assert straddle.mean() > 0.99
    assert np.all(err[straddle] <= bound[straddle])
    qg = q.reshape(K // G, G, N).astype(np.int64)
    assert np.all(qg.min(axis=1)[straddle] == 0)
    assert np.all(np.isin(qg.max(axis=1)[straddle], [14, 15]))
    # the scale spreads the range over 15 steps, up to one fp16 rounding
    assert np.all(np.abs(s16 * 15 - (mx - mn)) <= (mx - mn) * 2.0 ** -10 + 1e-12)


def test_awq_degenerate_group_gets_scale_one():
    G, K, N = 32, 64, 32
    W = np.zeros((K, N), np.float32)
    W[G:, :] = np.random.default_rng(0).normal(0, 0.02, (K - G, N)).astype(np.float32)
    qw, s, qz = oracle.awq_quantize(W, G)
    assert np.all(s[0].astype(np.float32) == 1.0)
    assert np.all(oracle.awq_dequant(qw, s, qz, K, N, G)[:G] == 0.0)


def test_w4a16_linear_matches_exact_rational_brute_force():
    # Brute force with exact rationals (fp16 / fp32 values are dyadic) on a tiny shape.
    M, K, N, G = 2, 64, 16, 32
    W = inputs.weight(K, N, seed=7, outliers=True)
    X = inputs.activations(M, K, seed=7)
    qw, s, qz = oracle.awq_quantize(W, G)
    q, z = oracle.awq_unpack(qw, qz, K, N, G)
    Y = oracle.w4a16_linear(X, qw, s, qz, G)
    Xf = X.astype(np.float64)
    sf = s.astype(np.float64)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(float(Xf[m, k])) * (int(q[k, n]) - int(z[k // G, n])) * Fraction(float(sf[k // G, n]))
            exact = float(acc)
            assert abs(Y[m, n] - exact) <= 1e-13 * max(1.0, abs(exact))


def test_w4a16_linear_one_hot_rows_and_special_cases():
    M, K, N, G = 5, 128, 64, 64
    W = inputs.weight(K, N, seed=9, outliers=True)
    qw, s, qz = oracle.awq_quantize(W, G)
    deq = oracle.awq_dequant(qw, s, qz, K, N, G)
    # one-hot activations select one row of the dequantised weight (pins the k index and layout)
    X = np.zeros((M, K), np.float16)
    ks = [0, 1, 63, 64, 127]
    for m, k in enumerate(ks):
        X[m, k] = 1.0
    Y = oracle.w4a16_linear(X, qw, s, qz, G)
    for m, k in enumerate(ks):
        assert np.array_equal(Y[m], deq[k].astype(np.float64))
    # zero activations give zero output
    assert np.all(oracle.w4a16_linear(np.zeros((2, K), np.float16), qw, s, qz, G) == 0.0)
    # rows selection returns the same rows as the full product
    Xr = inputs.activations(6, K, seed=2)
    full = oracle.w4a16_linear(Xr, qw, s, qz, G)
    part = oracle.w4a16_linear(Xr, qw, s, qz, G, rows=np.array([4, 1]))
    assert np.array_equal(part, full[[4, 1]])


def test_w4a16_linear_single_group_equals_numpy_float64_product():
    # G == K: one group; compare with numpy's float64 matmul of the dequantised weight.
    M, K, N, G = 3, 128, 32, 128
    W = inputs.weight(K, N, seed=4)
    X = inputs.activations(M, K, seed=4)
    qw, s, qz = oracle.awq_quantize(W, G)
    deq = oracle.awq_dequant(qw, s, qz, K, N, G).astype(np.float64)
    ref = X.astype(np.float64) @ deq
    assert np.allclose(oracle.w4a16_linear(X, qw, s, qz, G), ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------------
# QRMSNorm + per-token int8
# ------------------------------------------------------------------------------------------------

def _rmsnorm64(X, g, eps):
    Xf = X.astype(np.float64)
    r = 1.0 / np.sqrt((Xf * Xf).mean(axis=1, keepdims=True) + eps)
    return Xf * r * g.astype(np.float64)[None, :]


def test_sumsq_close_to_exact_sum():
    X = inputs.activations(4, 4096, seed=1, outlier_channels=True)
    for row in X:
        exact = math.fsum(float(v) * float(v) for v in row.astype(np.float64))
        assert abs(oracle.sumsq(row) - exact) <= 1e-6 * exact


def _round_f32(v: Fraction) -> Fraction:
    """v rounded to the nearest binary32 value, ties to even (normal range), in exact rationals."""
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return (n * ulp) if v > 0 else -(n * ulp)


def _sumsq_in_lanes(sq, lane_of):
    """Sum of the squares in 256 lanes (each in increasing k), then the pairwise fold (t, t+128),
    (t, t+64), ..., (t, t+1), rounding to fp32 after every addition."""
    lanes = [Fraction(0)] * 256
    for k, v in enumerate(sq):
        t = lane_of(k)
        lanes[t] = _round_f32(lanes[t] + v)
    stride = 128
    while stride >= 1:
        for t in range(stride):
            lanes[t] = _round_f32(lanes[t] + lanes[t + stride])
        stride //= 2
    return lanes[0]


def test_sumsq_follows_the_documented_lane_order():
    """The fixed reduction order that the bit-exact QRMSNorm comparison depends on (element k in
    lane (k / 8) mod 256, lanes in increasing k, then the pairwise fold), re-evaluated in exact
    rationals with an explicit round-to-fp32 after each addition.  The row is built so that the
    sequential order and the (k mod 256) lane order give other fp32 sums: large squares (2^20)
    share lanes with mid-size ones under one order and not under the other."""
    K = 4096
    x = np.zeros(K, np.float16)
    j = np.arange(16)
    x[8 * j] = 1024.0
    x[8 * j + 1] = (0.8 + 0.0137 * j).astype(np.float16)
    rest = np.setdiff1d(np.arange(K), np.concatenate([8 * j, 8 * j + 1]))
    x[rest] = (np.random.default_rng(3).standard_normal(rest.size) * 0.05).astype(np.float16)
    sq = [Fraction(float(v)) ** 2 for v in x]  # each square is exact in fp32 (11-bit significands)
    documented = _sumsq_in_lanes(sq, lambda k: (k // 8) % 256)
    mod256 = _sumsq_in_lanes(sq, lambda k: k % 256)
    sequential = Fraction(0)
    for v in sq:
        sequential = _round_f32(sequential + v)
    assert len({documented, mod256, sequential}) == 3  # the three orders are told apart
    assert Fraction(oracle.sumsq(x)) == documented


def test_qrmsnorm_against_float64_definition():
    # Independent fp64 evaluation of RMSNorm + absmax/127 + round-half-even: codes may differ only
    # where the fp64 quotient sits within 1e-4 of a .5 boundary; scales agree to fp32 precision.
    M, K = 16, 4096
    X = inputs.activations(M, K, seed=2, outlier_channels=True)
    g = inputs.gamma(K, seed=2)
    q, xs = oracle.qrmsnorm_quant_i8(X, g, inputs.EPS)
    y64 = _rmsnorm64(X, g, inputs.EPS)
    xs64 = np.abs(y64).max(axis=1) / 127.0
    assert np.allclose(xs, xs64, rtol=1e-5)
    t = y64 / xs64[:, None]
    q64 = np.clip(np.rint(t), -128, 127)
    near_tie = np.abs(np.abs(t - np.floor(t)) - 0.5) < 1e-4
    assert np.all((q == q64) | near_tie)
    assert (q != q64).mean() < 1e-3
    # the row maximum lands on +-127 and the dequantisation error is at most half a step
    assert np.all(np.abs(q.astype(np.int64)).max(axis=1) == 127)
    y32 = oracle.rmsnorm(X, g, inputs.EPS).astype(np.float64)
    assert np.all(np.abs(q * xs[:, None].astype(np.float64) - y32) <= xs[:, None] * (0.5 + 1e-5))


def test_qrmsnorm_closed_forms():
    K = 512
    g1 = np.ones(K, np.float16)
    # constant row: every code is +-127 (or 0 for a zero row, whose scale is 1)
    X = np.stack([np.full(K, 0.75, np.float16), np.full(K, -3.0, np.float16), np.zeros(K, np.float16)])
    q, xs = oracle.qrmsnorm_quant_i8(X, g1, 1e-6)
    assert np.all(q[0] == 127) and np.all(q[1] == -127) and np.all(q[2] == 0)
    assert xs[2] == 1.0
    # with eps = 0, scaling a row by a power of two leaves every code unchanged
    Xr = inputs.activations(3, K, seed=8, outlier_channels=True)
    g = inputs.gamma(K, seed=8)
    qa, xa = oracle.qrmsnorm_quant_i8(Xr, g, 0.0)
    qb, xb = oracle.qrmsnorm_quant_i8((Xr.astype(np.float32) * 0.25).astype(np.float16), g, 0.0)
    assert np.array_equal(qa, qb) and np.array_equal(xa, xb)


def test_add_qrmsnorm_residual_sum_and_special_cases():
    # [W8A8] residual fusion: h = fp16(x + r) from an fp32 sum, then the unfused QRMSNorm of h
    M, K = 6, 1024
    X = inputs.activations(M, K, seed=11, outlier_channels=True)
    R = inputs.activations(M, K, seed=12)
    g = inputs.gamma(K, seed=11)
    h, q, xs = oracle.add_qrmsnorm_quant_i8(X, R, g, inputs.EPS)
    # the residual sum against numpy's own fp32 addition and round-to-nearest-even fp16 cast
    assert np.array_equal(h.view(np.uint16), (X.astype(np.float32) + R.astype(np.float32)).astype(np.float16).view(np.uint16))
    q2, xs2 = oracle.qrmsnorm_quant_i8(h, g, inputs.EPS)
    assert np.array_equal(q, q2) and np.array_equal(xs, xs2)
    # r = 0: the fused op is the plain QRMSNorm of x, bit for bit
    h0, q0, xs0 = oracle.add_qrmsnorm_quant_i8(X, np.zeros_like(X), g, inputs.EPS)
    qx, xsx = oracle.qrmsnorm_quant_i8(X, g, inputs.EPS)
    assert np.array_equal(h0.view(np.uint16), X.view(np.uint16)) and np.array_equal(q0, qx) and np.array_equal(xs0, xsx)
    # r = -x: every row cancels to zero, all codes 0 with scale 1
    hz, qz, xsz = oracle.add_qrmsnorm_quant_i8(X, -X, g, inputs.EPS)
    assert np.all(hz == 0) and np.all(qz == 0) and np.all(xsz == 1.0)


def test_act_absmax_matches_float64_rmsnorm():
    M, K = 32, 1024
    X = inputs.activations(M, K, seed=3, outlier_channels=True)
    g = inputs.gamma(K, seed=3)
    a = oracle.act_absmax(X, g, inputs.EPS)
    a64 = np.abs(_rmsnorm64(X, g, inputs.EPS)).max(axis=0)
    assert np.allclose(a, a64, rtol=1e-5)


# ------------------------------------------------------------------------------------------------
# SmoothQuant smoothing and per-channel weight quantisation
# ------------------------------------------------------------------------------------------------

def test_smoothing_invariance_and_balance():
    M, K, N = 64, 512, 256
    X = inputs.activations(M, K, seed=4, outlier_channels=True)
    g = inputs.gamma(K, seed=4)
    W = inputs.weight(K, N, seed=4)
    a = oracle.act_absmax(X, g, inputs.EPS)
    s, g2, W2 = oracle.smooth(a, g, W)
    s64 = s.astype(np.float64)
    # X W = (X diag(s)^-1)(diag(s) W) in exact arithmetic; the oracle's W' is diag(s) W to fp32 rounding
    assert np.allclose(W2.astype(np.float64), W.astype(np.float64) * s64[:, None], rtol=2 ** -23, atol=0)
    Xn = _rmsnorm64(X, g, inputs.EPS)
    lhs = (Xn / s64[None, :]) @ (W.astype(np.float64) * s64[:, None])
    assert np.allclose(lhs, Xn @ W.astype(np.float64), rtol=1e-12, atol=1e-12)
    # the stored model (fp16 gamma', fp32 W') reproduces the original layer to fp16 precision
    Xn2 = _rmsnorm64(X, g2, inputs.EPS)
    y_new, y_old = Xn2 @ W2.astype(np.float64), Xn @ W.astype(np.float64)
    rel = np.linalg.norm(y_new - y_old, axis=1) / np.linalg.norm(y_old, axis=1)
    assert rel.max() < 2e-3
    # alpha = 0.5 balances the per-channel ranges: max|act'_j| == max|W'_j| == sqrt(a_j w_j)
    w_j = np.abs(W.astype(np.float64)).max(axis=1)
    assert np.allclose(np.abs(W2.astype(np.float64)).max(axis=1), np.sqrt(a * w_j), rtol=1e-6)
    assert np.allclose(a / s64, np.sqrt(a * w_j), rtol=1e-6)


def test_per_channel_quant_bounds():
    K, N = 256, 96
    W = inputs.weight(K, N, seed=6, outliers=True)
    W[:, 5] = 0.0
    qW, ws = oracle.per_channel_quant_i8(W)
    assert qW.shape == (N, K)
    deq = qW.astype(np.float64).T * ws.astype(np.float64)[None, :]
    assert np.all(np.abs(deq - W) <= ws[None, :] * (0.5 + 1e-6))
    nz = np.abs(W).max(axis=0) > 0
    assert np.all(np.abs(qW.astype(np.int64)).max(axis=1)[nz] == 127)
    assert ws[5] == 1.0 and np.all(qW[5] == 0)
    assert np.allclose(ws[nz], np.abs(W).max(axis=0)[nz] / 127.0, rtol=1e-6)


# ------------------------------------------------------------------------------------------------
# int8 GEMM and its dequantising epilogue
# ------------------------------------------------------------------------------------------------

def test_w8a8_acc_matches_python_integers_and_numpy_int64():
    rng = np.random.default_rng(0)
    M, K, N = 3, 48, 8
    q = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    qW = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    acc = oracle.w8a8_acc(q, qW)
    for m in range(M):
        for n in range(N):
            assert acc[m, n] == sum(int(q[m, k]) * int(qW[n, k]) for k in range(K))
    q2 = rng.integers(-128, 128, size=(17, 4096), dtype=np.int8)
    W2 = rng.integers(-127, 128, size=(40, 4096), dtype=np.int8)
    assert np.array_equal(oracle.w8a8_acc(q2, W2), q2.astype(np.int64) @ W2.astype(np.int64).T)
    # the adversarial extreme exceeds 2^24 but not 2^31
    q3 = np.full((1, 4096), -128, np.int8)
    W3 = np.full((2, 4096), -127, np.int8)
    assert np.all(oracle.w8a8_acc(q3, W3) == 4096 * 128 * 127)


def test_w8a8_epilogue_against_float64():
    rng = np.random.default_rng(1)
    acc = rng.integers(-2 ** 20, 2 ** 20, size=(5, 64), dtype=np.int32)
    xs = rng.uniform(0.001, 0.1, 5).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, 64).astype(np.float32)
    y = oracle.w8a8_epilogue(acc, xs, ws).astype(np.float64)
    y64 = acc.astype(np.float64) * xs[:, None].astype(np.float64) * ws[None, :].astype(np.float64)
    assert np.array_equal(oracle.w8a8_epilogue_f64(acc, xs, ws), y64)
    assert np.all(np.abs(y - y64) <= np.abs(y64) * (2.0 ** -11 + 2.0 ** -22) + 2.0 ** -25)


def test_w8a8_fused_epilogue_bias_residual():
    rng = np.random.default_rng(4)
    R, N = 7, 96
    acc = rng.integers(-2 ** 20, 2 ** 20, size=(R, N), dtype=np.int32)
    xs = rng.uniform(0.001, 0.1, R).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    bias = rng.normal(0, 2, N).astype(np.float16)
    res = rng.normal(0, 4, (R, N)).astype(np.float16)
    # without the optional terms it is the plain epilogue, bit for bit
    assert np.array_equal(oracle.w8a8_epilogue_fused(acc, xs, ws).view(np.uint16),
                          oracle.w8a8_epilogue(acc, xs, ws).view(np.uint16))
    # against the exact value: fp32 steps of relative size 2^-24 each, one fp16 rounding at the end
    y = oracle.w8a8_epilogue_fused(acc, xs, ws, bias, res).astype(np.float64)
    t64 = acc.astype(np.float64) * xs[:, None].astype(np.float64) * ws[None, :].astype(np.float64)
    y64 = t64 + bias.astype(np.float64)[None, :] + res.astype(np.float64)
    slack = (np.abs(t64) + np.abs(bias.astype(np.float64))[None, :] + np.abs(res.astype(np.float64))) * 2.0 ** -22
    assert np.all(np.abs(y - y64) <= np.abs(y64) * 2.0 ** -11 + slack + 2.0 ** -24)
    # closed forms with acc = 0: the result is the residual itself, bias + residual, or +0 when they cancel
    z = np.zeros((R, N), np.int32)
    assert np.array_equal(oracle.w8a8_epilogue_fused(z, xs, ws, residual=res).view(np.uint16), res.view(np.uint16))
    assert np.array_equal(oracle.w8a8_epilogue_fused(z, xs, ws, bias=bias).view(np.uint16),
                          np.broadcast_to(bias, (R, N)).view(np.uint16))
    cancel = oracle.w8a8_epilogue_fused(z, xs, ws, bias=bias, residual=np.broadcast_to(-bias, (R, N)))
    assert np.all(cancel.view(np.uint16) == 0)


# ------------------------------------------------------------------------------------------------
# The worked example printed on the pages (off-path symmetric per-tensor int4)
# ------------------------------------------------------------------------------------------------

def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_printed_symmetric_int4_example():
    gv = _golden("p1_symmetric_int4.txt")
    w = np.array([gv["max_abs"], -0.05, 0.0166, -gv["max_abs"], 0.02], np.float32)
    scale, q = oracle.sym_int4_per_tensor(w)
    assert abs(scale - gv["scale"]) <= gv["scale_abs_tol"]
    assert q.min() >= gv["code_min"] and q.max() <= gv["code_max"]
    assert q[0] == gv["code_max"] and q[3] == gv["code_min"]


# ------------------------------------------------------------------------------------------------
# fp8 (float8_e4m3fn) variant of the W8A8 path
# ------------------------------------------------------------------------------------------------

def _torch_e4m3_values():
    """The 256 e4m3 codes decoded by torch's own float8_e4m3fn type (a library independent of the
    oracle), as float64."""
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _nearest_e4m3_brute(x):
    """Nearest finite e4m3 code of each float64 x by exhaustive search over the 254 finite codes
    (decoded by torch): smallest |v - x|, ties to the even code (the one whose lowest fraction bit
    is 0), magnitudes of 448 and more saturated.  Exact for 2^-12 <= |x| < 2^10, where every
    difference fits in a double."""
    vals = _torch_e4m3_values()
    pos = np.arange(0, 0x7f)  # finite non-negative codes 0x00..0x7e
    a = np.abs(x)
    d = np.abs(vals[pos][None, :] - a[:, None])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & (pos[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    code = pos[pick].astype(np.uint8)
    code[a >= 448.0] = 0x7e
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def test_e4m3_decode_all_codes_match_torch_and_qmax_is_448():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float(codes).astype(np.float64)
    ref = _torch_e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2  # only S.1111.111
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))  # -0.0 is code 0x80
    # Q_MAX as torch.finfo reports it, and the smallest subnormal / normal of the format
    assert float(torch.finfo(torch.float8_e4m3fn).max) == 448.0 == np.nanmax(ours)
    assert ours[1] == 2.0 ** -9 and ours[8] == 2.0 ** -6


def test_float_to_e4m3_matches_brute_force_nearest_with_ties_and_saturation():
    rng = np.random.default_rng(41)
    vals = _torch_e4m3_values()
    fin = np.sort(np.unique(vals[:0x7f]))
    mids = (fin[:-1] + fin[1:]) / 2  # every exact tie between neighbouring non-negative values
    rand = np.concatenate([rng.standard_normal(20000) * s for s in (3e-3, 0.1, 1.0, 30.0, 200.0)])
    x = np.concatenate([rand, mids, -mids, fin, -fin, [448.0, 449.0, 463.9, 464.0, 480.0, 1000.0, -600.0]])
    x = x.astype(np.float32)
    keep = (np.abs(x.astype(np.float64)) >= 2.0 ** -12) & (np.abs(x) < 2.0 ** 10)
    ours = oracle.float_to_e4m3(x[keep])
    assert np.array_equal(ours, _nearest_e4m3_brute(x[keep].astype(np.float64)))
    # tiny magnitudes go to a signed zero; large ones and infinities saturate; NaN stays NaN
    tiny = np.array([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11), 2.0 ** -30], np.float32)
    assert list(oracle.float_to_e4m3(tiny)) == [0x00, 0x80, 0x00, 0x80, 0x00]
    big = np.array([1e9, -1e9, np.inf, -np.inf], np.float32)
    assert list(oracle.float_to_e4m3(big)) == [0x7e, 0xfe, 0x7e, 0xfe]
    assert (oracle.float_to_e4m3(np.array([np.nan], np.float32))[0] & 0x7f) == 0x7f


def test_float_to_e4m3_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    # every finite fp16 value below 448 in magnitude, as fp32
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float32)
    h = h[np.isfinite(h) & (np.abs(h) < 448.0)]
    ours = oracle.float_to_e4m3(h)
    ref = torch.from_numpy(h).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def _e4m3_error_ok(codes, target, scale):
    """|decode(code) * scale - target| within half a unit of e4m3 at the code's magnitude: 2^-4 of
    the value for normals, 2^-10 * scale below the smallest normal (units of 2^-9 * scale)."""
    v = oracle.e4m3_to_float(codes).astype(np.float64) * np.asarray(scale, np.float64)
    err = np.abs(v - target.astype(np.float64))
    bound = np.maximum(np.abs(target) * 2.0 ** -4, 2.0 ** -10 * np.asarray(scale, np.float64)) * (1 + 1e-6)
    return bool(np.all(err <= bound))


def test_qrmsnorm_fp8_against_definition_and_brute_force():
    M, K = 9, 640
    X = inputs.activations(M, K, seed=42, outlier_channels=True)
    X[3] = 0  # an all-zero row
    g = inputs.gamma(K, seed=42)
    q, xs = oracle.qrmsnorm_quant_fp8(X, g, inputs.EPS)
    y = oracle.rmsnorm(X, g, inputs.EPS)
    amax = np.abs(y).max(axis=1)
    want_xs = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(xs.view(np.uint32), want_xs.view(np.uint32))
    t = (y / xs[:, None]).astype(np.float32).astype(np.float64)
    nz = np.abs(t) >= 2.0 ** -12
    assert np.array_equal(q[nz], _nearest_e4m3_brute(t[nz]))
    assert np.all((q[~nz] & 0x7f) == 0)
    dec = oracle.e4m3_to_float(q)
    for m in range(M):
        if m == 3:
            assert xs[m] == 1.0 and np.all((q[m] & 0x7f) == 0)
        else:
            assert np.abs(dec[m]).max() == 448.0  # the row's absmax lands exactly on Q_MAX
    assert _e4m3_error_ok(q, y, xs[:, None])


def test_per_token_quant_i8_recovers_exactly_representable_rows():
    # each row is c * 2^-e with integer codes c in [-127, 127] and |c| = 127 present: the scale is
    # 127 * 2^-e / 127 = 2^-e exactly, so the codes come back as c
    rng = np.random.default_rng(70)
    M, K = 7, 1000
    c = rng.integers(-127, 128, size=(M, K))
    c[np.arange(M), (np.arange(M) * 37) % K] = np.where(np.arange(M) % 2 == 0, 127, -127)
    e = np.arange(M) - 3  # 2^3 .. 2^-3
    x = (c * (2.0 ** -e)[:, None]).astype(np.float16)
    q, xs = oracle.per_token_quant_i8(x)
    assert np.array_equal(xs, (2.0 ** -e).astype(np.float32))
    assert np.array_equal(q.astype(np.int64), c)


def test_per_token_quant_i8_definition_bounds_and_zero_row():
    X = inputs.activations(11, 4096, seed=71, outlier_channels=True)
    X[4] = 0  # an all-zero row
    X[6] *= np.float16(1e-3)
    q, xs = oracle.per_token_quant_i8(X)
    xf = X.astype(np.float32)
    amax = np.abs(xf).max(axis=1)
    want = np.where(amax == 0, np.float32(1.0), amax / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(xs.view(np.uint32), want.view(np.uint32))  # absmax / Q_MAX in fp32
    assert xs[4] == 1.0 and np.all(q[4] == 0)
    nz = amax > 0
    assert np.all(np.abs(q[nz].astype(np.int64)).max(axis=1) == 127)  # the row's absmax lands on 127
    err = np.abs(q.astype(np.float64) * xs[:, None].astype(np.float64) - xf)
    assert np.all(err <= xs[:, None].astype(np.float64) * (0.5 + 1e-5))  # nearest code: half a step
    # an independent fp64 evaluation: codes may differ only within 1e-4 of a .5 tie
    t = xf.astype(np.float64) / xs[:, None].astype(np.float64)
    ref = np.clip(np.round(t), -128, 127)  # numpy rounds half to even
    diff = q.astype(np.float64) != ref
    assert np.all(np.abs(np.abs(t[diff] - np.floor(t[diff])) - 0.5) < 1e-4)


def test_per_token_quant_i8_half_integer_ties_go_to_even():
    # a row whose scale is exactly 1 (absmax 127) holds every half-integer tie in [-126.5, 126.5]
    ties = np.arange(-126.5, 127.0, 1.0)
    x = np.concatenate([[127.0], ties, [0.0] * 2]).astype(np.float16)[None, :]
    q, xs = oracle.per_token_quant_i8(x)
    assert xs[0] == 1.0
    assert np.array_equal(q[0, 1:1 + ties.size].astype(np.float64), np.round(ties))  # to even


def test_per_token_quant_fp8_against_definition_and_brute_force():
    M, K = 9, 640
    X = inputs.activations(M, K, seed=72, outlier_channels=True)
    X[3] = 0  # an all-zero row
    q, xs = oracle.per_token_quant_fp8(X)
    xf = X.astype(np.float32)
    amax = np.abs(xf).max(axis=1)
    want_xs = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(xs.view(np.uint32), want_xs.view(np.uint32))
    t = (xf / xs[:, None]).astype(np.float32).astype(np.float64)
    nz = np.abs(t) >= 2.0 ** -12
    assert np.array_equal(q[nz], _nearest_e4m3_brute(t[nz]))
    assert np.all((q[~nz] & 0x7f) == 0)
    dec = oracle.e4m3_to_float(q)
    for m in range(M):
        if m == 3:
            assert xs[m] == 1.0 and np.all((q[m] & 0x7f) == 0)
        else:
            assert np.abs(dec[m]).max() == 448.0  # the row's absmax lands exactly on Q_MAX
    assert _e4m3_error_ok(q, xf, xs[:, None])


def test_add_qrmsnorm_fp8_residual_sum():
    M, K = 5, 256
    X = inputs.activations(M, K, seed=43)
    R = inputs.activations(M, K, seed=44, outlier_channels=True)
    g = inputs.gamma(K, seed=43)
    h, q, xs = oracle.add_qrmsnorm_quant_fp8(X, R, g, inputs.EPS)
    # fp16(x + r): the exact sum of two fp16 values rounded once (numpy's binary16 rounding)
    want_h = (X.astype(np.float64) + R.astype(np.float64)).astype(np.float32).astype(np.float16)
    assert np.array_equal(h.view(np.uint16), want_h.view(np.uint16))
    q2, xs2 = oracle.qrmsnorm_quant_fp8(want_h, g, inputs.EPS)
    assert np.array_equal(q, q2) and np.array_equal(xs, xs2)
    # r = -x: every row cancels to zero
    h0, q0, xs0 = oracle.add_qrmsnorm_quant_fp8(X, -X, g, inputs.EPS)
    assert np.all(h0 == 0) and np.all((q0 & 0x7f) == 0) and np.all(xs0 == 1.0)


def test_per_channel_quant_fp8_bounds_and_layout():
    K, N = 192, 48
    rng = np.random.default_rng(45)
    W = (rng.standard_normal((K, N)) * rng.uniform(0.01, 3.0, N)).astype(np.float32)
    W[:, 7] = 0
    W[5, 9] = 1e-7  # tiny values land among the subnormals
    qW, ws = oracle.per_channel_quant_fp8(W)
    assert qW.shape == (N, K) and ws.shape == (N,)
    amax = np.abs(W).max(axis=0)
    want = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(ws.view(np.uint32), want.view(np.uint32))
    dec = oracle.e4m3_to_float(qW)
    assert np.all(np.abs(dec[np.arange(N) != 7]).max(axis=1) == 448.0)
    assert np.all((qW[7] & 0x7f) == 0) and ws[7] == 1.0
    assert _e4m3_error_ok(qW, W.T, ws[:, None])
    t = (W.T / ws[:, None]).astype(np.float32).astype(np.float64)
    nz = np.abs(t) >= 2.0 ** -12
    assert np.array_equal(qW[nz], _nearest_e4m3_brute(t[nz]))


def test_fp8_acc_exact_against_rationals_and_numpy():
    rng = np.random.default_rng(46)
    finite = np.array([c for c in range(256) if (c & 0x7f) != 0x7f], np.uint8)
    vals = _torch_e4m3_values()
    # tiny: exact rational sums
    q = rng.choice(finite, size=(3, 24)).astype(np.uint8)
    qW = rng.choice(finite, size=(5, 24)).astype(np.uint8)
    acc, absacc = oracle.fp8_acc(q, qW)
    for i in range(3):
        for n in range(5):
            s = sum(Fraction(float(vals[a])) * Fraction(float(vals[b])) for a, b in zip(q[i], qW[n]))
            assert Fraction(acc[i, n]) == s
            assert absacc[i, n] == float(sum(abs(Fraction(float(vals[a])) * Fraction(float(vals[b])))
                                             for a, b in zip(q[i], qW[n])))
    # larger, with extremes (+-448 everywhere): numpy's float64 matmul is exact here too
    K = 4096
    q = rng.choice(finite, size=(4, K)).astype(np.uint8)
    qW = rng.choice(finite, size=(6, K)).astype(np.uint8)
    q[0] = 0x7e
    qW[0] = 0x7e
    qW[1] = 0xfe
    rows = np.array([3, 0, 2], np.int64)
    acc, absacc = oracle.fp8_acc(q, qW, rows=rows)
    ref = vals[q[rows]] @ vals[qW].T
    assert np.array_equal(acc, ref)
    assert acc[1, 0] == 448.0 * 448.0 * K and acc[1, 1] == -448.0 * 448.0 * K
    assert np.all(absacc >= np.abs(acc))
    with pytest.raises(ValueError):
        bad = q.copy()
        bad[0, 0] = 0x7f
        oracle.fp8_acc(bad, qW)


def test_fp8_epilogue_terms():
    rng = np.random.default_rng(47)
    acc = rng.standard_normal((3, 8)) * 1e4
    xs = rng.uniform(1e-3, 1e-2, 3).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, 8).astype(np.float32)
    bias = rng.standard_normal(8).astype(np.float16)
    res = rng.standard_normal((3, 8)).astype(np.float16)
    base = oracle.fp8_epilogue_f64(acc, xs, ws)
    assert np.allclose(base, acc * xs[:, None].astype(np.float64) * ws[None, :].astype(np.float64), rtol=1e-15)
    both = oracle.fp8_epilogue_f64(acc, xs, ws, bias, res)
    assert np.allclose(both - base, bias.astype(np.float64)[None, :] + res.astype(np.float64), rtol=0, atol=1e-9)
    only_b = oracle.fp8_epilogue_f64(acc, xs, ws, bias=bias)
    assert np.allclose(only_b - base, np.broadcast_to(bias.astype(np.float64), (3, 8)), rtol=0, atol=1e-9)


# ------------------------------------------------------------------------------------------------
# KV-cache int8, groups of 128 channels
# ------------------------------------------------------------------------------------------------

def test_kv_quant_recovers_exactly_representable_groups():
    # every group is c * 2^-7 with integer codes c in [-127, 127] and |c| = 127 present: the scale is
    # 127 * 2^-7 / 127 = 2^-7 exactly, so the codes come back as c and the cache entry as x itself
    rng = np.random.default_rng(50)
    rows, D = 6, 512
    c = rng.integers(-127, 128, size=(rows, D))
    for g in range(D // 128):
        c[:, 128 * g + (g * 7) % 128] = np.where(np.arange(rows) % 2 == 0, 127, -127)
    x = (c * 2.0 ** -7).astype(np.float16)
    q, s = oracle.kv_quant_i8(x)
    assert np.all(s == np.float32(2.0 ** -7))
    assert np.array_equal(q.astype(np.int64), c)
    assert np.array_equal(oracle.kv_dequant_i8(q, s).view(np.uint16), x.view(np.uint16))


def test_kv_quant_groups_bounds_and_zero_group():
    rng = np.random.default_rng(51)
    rows, D = 40, 1024
    x = (rng.standard_normal((rows, D)) * rng.uniform(0.01, 50, size=(rows, 1))).astype(np.float16)
    x[3, 256:384] = 0  # one all-zero group
    x[7, 128:256] *= np.float16(0.001)  # a small group next to large ones
    q, s = oracle.kv_quant_i8(x)
    assert q.shape == (rows, D) and s.shape == (rows, D // 128)
    xf = x.astype(np.float32)
    for g in range(D // 128):
        amax = np.abs(xf[:, 128 * g:128 * (g + 1)]).max(axis=1)
        want = np.where(amax == 0, np.float32(1.0), amax / np.float32(127.0)).astype(np.float32)
        assert np.array_equal(s[:, g].view(np.uint32), want.view(np.uint32)), g  # each group's own absmax
        qg = q[:, 128 * g:128 * (g + 1)].astype(np.int64)
        nz = amax > 0
        assert np.all(np.abs(qg[nz]).max(axis=1) == 127)  # the group's absmax lands on 127
        err = np.abs(qg * s[:, g:g + 1].astype(np.float64) - xf[:, 128 * g:128 * (g + 1)])
        assert np.all(err <= s[:, g:g + 1] * (0.5 + 1e-5))  # round to nearest: half a step
    assert s[3, 2] == 1.0 and np.all(q[3, 256:384] == 0)


def test_kv_dequant_is_one_fp16_rounding_of_the_fp32_product():
    rng = np.random.default_rng(52)
    q = rng.integers(-128, 128, size=(9, 384)).astype(np.int8)
    s = rng.uniform(1e-6, 10, size=(9, 3)).astype(np.float32)
    s[0, 0] = 1e-9  # products in the fp16 subnormal range
    out = oracle.kv_dequant_i8(q, s)
    prod = q.astype(np.float32) * np.repeat(s, 128, axis=1)  # the fp32 product, rounded once (IEEE)
    assert np.array_equal(out.view(np.uint16), prod.astype(np.float16).view(np.uint16))  # numpy's rounding


# ------------------------------------------------------------------------------------------------
# fused gate/up activation: SiLU(gate) * up on interleaved channels
# ------------------------------------------------------------------------------------------------

def test_silu_mul_against_scipy_and_closed_forms():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(60)
    y = rng.standard_normal((5, 64)) * 6
    y[0, 0], y[0, 2], y[0, 4] = 0.0, 800.0, -800.0  # silu(0) = 0; silu(x) -> x and -> 0 far out
    out = oracle.silu_mul_f64(y)
    g, u = y[:, 0::2], y[:, 1::2]
    ref = g * special.expit(g) * u  # silu(g) = g * sigmoid(g), scipy's logistic
    assert np.allclose(out, ref, rtol=1e-14, atol=0)
    assert out[0, 0] == 0.0
    assert out[0, 1] == pytest.approx(800.0 * y[0, 3], rel=1e-15)
    assert abs(out[0, 2]) < 1e-300
    # the pairing: gate j is column 2j, up j is column 2j + 1 (swapping them changes the result)
    sw = y.copy()
    sw[:, 0::2], sw[:, 1::2] = y[:, 1::2], y[:, 0::2]
    assert not np.allclose(oracle.silu_mul_f64(sw), out)
    # silu(-x) = silu(x) - x
    x = rng.standard_normal(32) * 3
    pos = oracle.silu_mul_f64(np.stack([x, np.ones_like(x)], axis=1).reshape(1, -1))[0]
    neg = oracle.silu_mul_f64(np.stack([-x, np.ones_like(x)], axis=1).reshape(1, -1))[0]
    assert np.allclose(neg, pos - x, rtol=0, atol=1e-12)
