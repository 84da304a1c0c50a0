"""Pins of the oracle's chains: brute force on tiny inputs, special cases and invariants.

The chains are checked against explicit Python loops written from the
definitions (not against numpy's matmul), against special weights whose
result is known in closed form (identity and delta kernels, shifted taps,
1x1-equivalent convolutions), and against the row independence that the
sampled full-size parity checks rely on.
"""

import itertools

import numpy as np
import pytest

from oracle import activations, bf16, chains


def _bf16_ints(rng, shape, lo=-3, hi=4):
    return rng.integers(lo, hi, size=shape).astype(np.float64)


def _loop_matmul(A, B):
    m, k = A.shape
    k2, n = B.shape
    assert k == k2
    out = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for t in range(k):
                acc += A[i, t] * B[t, j]
            out[i, j] = acc
    return out


def test_mlp_gelu_brute_force():
    rng = np.random.default_rng(3)
    X = _bf16_ints(rng, (3, 5)) / 4
    W1 = _bf16_ints(rng, (5, 4)) / 8
    W2 = _bf16_ints(rng, (4, 2))
    H, Y = chains.mlp_gelu(X, W1, W2)
    Z = _loop_matmul(X, W1)                       # integer/8 sums: exact
    Hb = np.zeros_like(Z)
    for i, j in itertools.product(range(3), range(4)):
        Hb[i, j] = bf16.canonicalize_zero(bf16.round_to_bf16(activations.gelu_tanh(Z[i, j])))
    np.testing.assert_array_equal(H, Hb)
    np.testing.assert_allclose(Y, _loop_matmul(Hb, W2), rtol=1e-15, atol=1e-15)
    assert H.shape == (3, 4) and Y.shape == (3, 2)


def test_mlp_gelu_identity_weights():
    rng = np.random.default_rng(4)
    X = bf16.round_to_bf16(rng.standard_normal((6, 8)))
    I = np.eye(8)
    H, Y = chains.mlp_gelu(X, I, I)
    np.testing.assert_array_equal(H, bf16.canonicalize_zero(bf16.round_to_bf16(activations.gelu_tanh(X))))
    np.testing.assert_array_equal(Y, H)
    assert not np.any(np.signbit(H) & (H == 0))   # no -0 in the intermediate


def test_mlp_gelu_column_sum_weights():
    rng = np.random.default_rng(5)
    X = bf16.round_to_bf16(rng.standard_normal((4, 6)))
    W1 = bf16.round_to_bf16(rng.standard_normal((6, 5)) * 0.5)
    H, Y = chains.mlp_gelu(X, W1, np.ones((5, 1)))
    np.testing.assert_allclose(Y[:, 0], H.sum(axis=1), rtol=1e-15)


def test_mlp_rows_independent():
    rng = np.random.default_rng(6)
    X = rng.standard_normal((9, 16))
    W1 = rng.standard_normal((16, 12)) * 0.1
    W2 = rng.standard_normal((12, 7)) * 0.1
    H, Y = chains.mlp_gelu(X, W1, W2)
    rows = [0, 4, 8]
    Hr, Yr = chains.mlp_gelu_rows(X, W1, W2, rows)
    np.testing.assert_array_equal(Hr, H[rows])
    np.testing.assert_allclose(Yr, Y[rows], rtol=1e-14, atol=1e-14)


def test_swiglu_brute_force():
    rng = np.random.default_rng(7)
    X = _bf16_ints(rng, (2, 3)) / 2
    Wg = _bf16_ints(rng, (3, 4)) / 4
    Wu = _bf16_ints(rng, (3, 4)) / 4
    Wd = _bf16_ints(rng, (4, 3))
    H, Y = chains.mlp_swiglu(X, Wg, Wu, Wd)
    G, U = _loop_matmul(X, Wg), _loop_matmul(X, Wu)
    Hb = np.zeros_like(G)
    for i, j in itertools.product(range(2), range(4)):
        g = G[i, j]
        Hb[i, j] = bf16.canonicalize_zero(bf16.round_to_bf16(g / (1 + np.exp(-g)) * U[i, j]))
    np.testing.assert_array_equal(H, Hb)
    np.testing.assert_allclose(Y, _loop_matmul(Hb, Wd), rtol=1e-15, atol=1e-15)


def _loop_conv(x, w, pad=1):
    n, h, wd, c = x.shape
    k, r_, s_, _ = w.shape
    y = np.zeros((n, h, wd, k))
    for b, p, q, o in itertools.product(range(n), range(h), range(wd), range(k)):
        acc = 0.0
        for r, s, ci in itertools.product(range(r_), range(s_), range(c)):
            hh, ww = p + r - pad, q + s - pad
            if 0 <= hh < h and 0 <= ww < wd:
                acc += x[b, hh, ww, ci] * w[o, r, s, ci]
        y[b, p, q, o] = acc
    return y


def test_conv_brute_force_with_padding():
    rng = np.random.default_rng(8)
    x = _bf16_ints(rng, (2, 4, 3, 2))
    w = _bf16_ints(rng, (3, 3, 3, 2))
    np.testing.assert_array_equal(chains.conv2d_nhwc(x, w), _loop_conv(x, w))


def test_conv_delta_kernel_is_identity():
    rng = np.random.default_rng(9)
    x = bf16.round_to_bf16(rng.standard_normal((2, 5, 5, 4)))
    w = np.zeros((4, 3, 3, 4))
    for c in range(4):
        w[c, 1, 1, c] = 1.0
    np.testing.assert_array_equal(chains.conv2d_nhwc(x, w), x)
    H, Y = chains.conv_relu_chain(x, w, w)
    np.testing.assert_array_equal(H, np.maximum(x, 0.0))
    np.testing.assert_array_equal(Y, H)


def test_conv_shifted_tap_orientation():
    # Only tap (r=0, s=1) is non-zero: y[n,p,q] = x[n,p-1,q], zero in the first row.
    rng = np.random.default_rng(10)
    x = bf16.round_to_bf16(rng.standard_normal((1, 4, 4, 2)))
    w = np.zeros((2, 3, 3, 2))
    w[0, 0, 1, 0] = 1.0
    w[1, 0, 1, 1] = 1.0
    y = chains.conv2d_nhwc(x, w)
    np.testing.assert_array_equal(y[:, 1:], x[:, :-1])
    np.testing.assert_array_equal(y[:, 0], 0.0)
    # tap (r=1, s=2): y[n,p,q] = x[n,p,q+1], zero in the last column
    w = np.zeros((2, 3, 3, 2))
    w[0, 1, 2, 0] = 1.0
    w[1, 1, 2, 1] = 1.0
    y = chains.conv2d_nhwc(x, w)
    np.testing.assert_array_equal(y[:, :, :-1], x[:, :, 1:])
    np.testing.assert_array_equal(y[:, :, -1], 0.0)


def test_conv_centre_tap_is_pixelwise_gemm():
    rng = np.random.default_rng(11)
    x = bf16.round_to_bf16(rng.standard_normal((2, 3, 5, 6)))
    wc = bf16.round_to_bf16(rng.standard_normal((4, 6)))
    w = np.zeros((4, 3, 3, 6))
    w[:, 1, 1, :] = wc
    y = chains.conv2d_nhwc(x, w)
    ref = _loop_matmul(x.reshape(-1, 6), wc.T).reshape(2, 3, 5, 4)
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-14)


def test_conv_chain_relu_and_rounding():
    rng = np.random.default_rng(12)
    x = _bf16_ints(rng, (1, 3, 3, 2))
    w1 = _bf16_ints(rng, (2, 3, 3, 2)) / 16
    w2 = _bf16_ints(rng, (2, 3, 3, 2))
    H, Y = chains.conv_relu_chain(x, w1, w2)
    y1 = _loop_conv(x, w1)
    Hb = bf16.canonicalize_zero(bf16.round_to_bf16(np.maximum(y1, 0.0)))
    np.testing.assert_array_equal(H, Hb)
    np.testing.assert_allclose(Y, _loop_conv(Hb, w2), rtol=1e-15, atol=1e-15)


# ----------------------------------------------------------------- convolution stack

def _delta(c, r=1, s=1, scale=1.0):
    w = np.zeros((c, 3, 3, c))
    for i in range(c):
        w[i, r, s, i] = scale
    return w


def test_conv_stack_brute_force_three_stages():
    """Every stage by explicit loops: conv, ReLU and bf16 rounding after the first two,
    nothing after the last."""
    rng = np.random.default_rng(13)
    x = _bf16_ints(rng, (1, 4, 3, 2))
    ws = [_bf16_ints(rng, (2, 3, 3, 2)) / 8 for _ in range(3)]
    hs, y = chains.conv_stack(x, ws)
    h = x
    for s in range(2):
        h = bf16.canonicalize_zero(bf16.round_to_bf16(np.maximum(_loop_conv(h, ws[s]), 0.0)))
        np.testing.assert_array_equal(hs[s], h)
    np.testing.assert_allclose(y, _loop_conv(h, ws[2]), rtol=1e-15, atol=1e-15)
    assert len(hs) == 2


def test_conv_stack_of_two_is_the_pair():
    rng = np.random.default_rng(14)
    x = bf16.round_to_bf16(rng.standard_normal((2, 5, 4, 3)))
    w1 = bf16.round_to_bf16(rng.standard_normal((3, 3, 3, 3)) * 0.2)
    w2 = bf16.round_to_bf16(rng.standard_normal((3, 3, 3, 3)) * 0.2)
    hs, y = chains.conv_stack(x, [w1, w2])
    H, Y = chains.conv_relu_chain(x, w1, w2)
    np.testing.assert_array_equal(hs[0], H)
    np.testing.assert_array_equal(y, Y)


def test_conv_stack_identity_kernels():
    """Centre-delta kernels: every convolution is the identity, so every intermediate and
    the output are relu(x)."""
    rng = np.random.default_rng(15)
    x = bf16.round_to_bf16(rng.standard_normal((2, 4, 4, 3)))
    hs, y = chains.conv_stack(x, [_delta(3)] * 5)
    for h in hs:
        np.testing.assert_array_equal(h, np.maximum(x, 0.0))
    np.testing.assert_array_equal(y, np.maximum(x, 0.0))


def test_conv_stack_shifts_accumulate():
    """Tap (r=1, s=2) moves the image one column left with a zero column entering on the
    right; on a non-negative image N stages move it N columns."""
    rng = np.random.default_rng(16)
    x = np.abs(bf16.round_to_bf16(rng.standard_normal((1, 3, 7, 2))))
    for n in (2, 3, 4):
        _, y = chains.conv_stack(x, [_delta(2, r=1, s=2)] * n)
        np.testing.assert_array_equal(y[:, :, :7 - n], x[:, :, n:])
        np.testing.assert_array_equal(y[:, :, 7 - n:], 0.0)


def test_conv_stack_scales_multiply():
    """Centre taps of 2 (exact in bf16): N stages multiply a non-negative image by 2^N."""
    rng = np.random.default_rng(17)
    x = np.abs(bf16.round_to_bf16(rng.standard_normal((1, 3, 3, 4))))
    hs, y = chains.conv_stack(x, [_delta(4, scale=2.0)] * 4)
    np.testing.assert_array_equal(y, 16.0 * x)
    np.testing.assert_array_equal(hs[1], 4.0 * x)


# ----------------------------------------------------------------- self-attention block

def bf16_vals(a):
    """Round an fp64 array to bf16 values with the oracle's (separately pinned) rounding."""
    return bf16.round_to_bf16(np.asarray(a, dtype=np.float64))

def test_attention_brute_force_small():
    """Python loops over every element on a 2-token, 2-head example."""
    import math
    rng = np.random.default_rng(21)
    M, K, N1, N2, head = 2, 3, 4, 5, 2
    X = bf16_vals(rng.standard_normal((M, K)))
    W = bf16_vals(0.5 * rng.standard_normal((K, 3 * N1)))
    W2 = bf16_vals(rng.standard_normal((N1, N2)))
    xqkv, xdot, y = chains.attention(X, W, W2, head=head)
    for r in range(M):
        row = [sum(X[r, k] * W[k, j] for k in range(K)) for j in range(3 * N1)]
        row = [float(chains.bf16_intermediate(np.array([v]))[0]) for v in row]
        assert np.allclose(xqkv[r], row, rtol=0, atol=0)
        for h in range(N1 // head):
            cols = range(h * head, (h + 1) * head)
            s = [row[j] * row[N1 + j] for j in cols]
            mx = max(s)
            e = [math.exp(v - mx) for v in s]
            for t, j in enumerate(cols):
                want = float(chains.bf16_intermediate(np.array([e[t] / sum(e) * row[2 * N1 + j]]))[0])
                assert xdot[r, j] == want
        for o in range(N2):
            assert y[r, o] == pytest.approx(sum(xdot[r, j] * W2[j, o] for j in range(N1)), rel=1e-12, abs=1e-12)


def test_attention_uniform_softmax_when_q_is_zero():
    """XQ = 0 makes every product 0, so each head's softmax is uniform: XDot = XK / head."""
    rng = np.random.default_rng(22)
    M, K, N1, head = 3, 8, 256, 128
    X = bf16_vals(rng.standard_normal((M, K)))
    W = bf16_vals(0.1 * rng.standard_normal((K, 3 * N1)))
    W[:, :N1] = 0.0
    xqkv, xdot, _ = chains.attention(X, W, np.eye(N1), head=head)
    assert np.array_equal(xdot, chains.bf16_intermediate(xqkv[:, 2 * N1:] / head))


def test_softmax_heads_sums_and_shift():
    rng = np.random.default_rng(23)
    s = rng.standard_normal((4, 512)) * 3
    p = chains.softmax_heads(s, 128)
    assert np.allclose(p.reshape(4, 4, 128).sum(axis=2), 1.0, rtol=0, atol=1e-12)
    shift = np.repeat(rng.standard_normal((4, 4)), 128, axis=1)
    assert np.allclose(chains.softmax_heads(s + shift, 128), p, rtol=0, atol=1e-12)
