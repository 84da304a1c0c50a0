"""The dependent chains, written as their plain definitions (oracle; test infrastructure).

Tile-level synchronisation ([cuSync] §IV, "Fine-Grained Synchronization
using cuSync") changes when a consumer thread block may start on a tile; it
never changes what any tile computes.  So the oracle of every chain is its
mathematical definition, evaluated in fp64 from the same bf16-valued inputs
the GPU receives:

* MLP ([cuSync] §II-B, Fig. ``fig:gpt-3:mlp``):
      XW1  = GeLU(X x W1)          X [M,K], W1 [K,N1]
      XW12 = XW1 x W2              W2 [N1,N2]
  The intermediate XW1 (called H here) is stored in bf16 by the producer
  kernel and read back by the consumer, so the oracle rounds it to bf16
  (round-to-nearest-even) and canonicalises -0 to +0 ([CUDA-FGS] §4.6.4.3,
  Canonicalization) before the second product.  Y is returned in fp64.

* SwiGLU MLP: H = bf16(silu(X x Wgate) * (X x Wup)), Y = H x Wdown.

* Conv pair ([cuSync] §II-B "ResNet", Table ``tab:resnet-sizes``; §IV-E
  "Conv2DTileSync"): y1 = conv(x, w1), H = bf16(relu(y1)), y2 = conv(H, w2),
  with NHWC activations, KRSC weights and zero padding:
      conv(x, w)[n,p,q,o] = sum_{r,s,c} x[n, p*stride + r - pad,
                                           q*stride + s - pad, c] * w[o,r,s,c]
  No bias, no activation after the second convolution, no residual add.

* Convolution stack ([cuSync] §II-B "ResNet", Table ``tab:resnet-sizes``: each layer of
  ResNet-38 is a pair of 3x3 convolutions with the same kernel size and channels, and a
  group of layers repeats that pair): N convolutions in a row,
      h_0 = x,  h_s = bf16(relu(conv(h_{s-1}, w_s)))  for s = 1 .. N-1,
      y = conv(h_{N-1}, w_N)
  so a stack of two is the conv pair above.  Same reading as the pair: ReLU after every
  convolution but the last, no bias, no residual add.

* Self-attention block ([cuSync] §II-B, Fig. ``fig:gpt-3:attention``):
      XQKV = X x QKV               QKV [K, 3*N1]; stored in bf16
      XQ, XV, XK = the column blocks [0,N1), [N1,2N1), [2N1,3N1) of XQKV
                                   (in the figure's order: the second block is XV)
      XDot = Dropout(Softmax(XQ . XV)) . XK, stored in bf16
      Y    = XDot x W2             W2 [N1, N2]
  Reading: "." is the element-wise product (the figure's fused dot-product
  kernel), and the softmax runs over the columns of one head (``head``
  columns), because the pages' tile dependencies have a column tile of XDot
  read only the same column tiles of XQ, XV and XK; dropout is the identity
  (inference).

All inputs are fp64 arrays whose values are exactly representable in bf16.
"""

import numpy as np

from .activations import gelu_tanh, relu, silu
from .bf16 import canonicalize_zero, round_to_bf16


def _as64(a):
    return np.asarray(a, dtype=np.float64)


def bf16_intermediate(v):
    """The value the producer stores: bf16 round-to-nearest-even, then -0 -> +0."""
    return canonicalize_zero(round_to_bf16(v))


def mlp_gelu(X, W1, W2):
    """Return (H, Y) for Y = bf16(GeLU_tanh(X @ W1)) @ W2.  H is bf16-exact fp64, Y is fp64."""
    X, W1, W2 = _as64(X), _as64(W1), _as64(W2)
    Z = X @ W1
    H = bf16_intermediate(gelu_tanh(Z))
    Y = H @ W2
    return H, Y


def mlp_swiglu(X, Wgate, Wup, Wdown):
    """Return (H, Y) for H = bf16(silu(X @ Wgate) * (X @ Wup)), Y = H @ Wdown."""
    X, Wg, Wu, Wd = _as64(X), _as64(Wgate), _as64(Wup), _as64(Wdown)
    G = X @ Wg
    U = X @ Wu
    H = bf16_intermediate(silu(G) * U)
    Y = H @ Wd
    return H, Y


def conv2d_nhwc(x, w, stride=1, pad=1):
    """Direct convolution, NHWC input [N,H,W,C], KRSC weights [K,R,S,C], zero padding.

    Output [N,P,Q,K] with P = (H + 2*pad - R)//stride + 1 (same for Q).
    Each filter tap (r, s) contributes the shifted input window times that
    tap's [K,C] weight slice; the sum over taps and channels is the
    definition above.
    """
    x, w = _as64(x), _as64(w)
    n, h, wd, c = x.shape
    k, r_, s_, c2 = w.shape
    if c != c2:
        raise ValueError("channel mismatch")
    p = (h + 2 * pad - r_) // stride + 1
    q = (wd + 2 * pad - s_) // stride + 1
    xp = np.zeros((n, h + 2 * pad, wd + 2 * pad, c), dtype=np.float64)
    xp[:, pad:pad + h, pad:pad + wd, :] = x
    y = np.zeros((n, p, q, k), dtype=np.float64)
    for r in range(r_):
        for s in range(s_):
            window = xp[:, r:r + stride * (p - 1) + 1:stride, s:s + stride * (q - 1) + 1:stride, :]
            y += window @ w[:, r, s, :].T
    return y


def conv_relu_chain(x, w1, w2, stride=1, pad=1):
    """Return (H, Y) for H = bf16(relu(conv(x, w1))), Y = conv(H, w2) (fp64)."""
    y1 = conv2d_nhwc(x, w1, stride, pad)
    H = bf16_intermediate(relu(y1))
    Y = conv2d_nhwc(H, w2, stride, pad)
    return H, Y


def conv_stack(x, ws, stride=1, pad=1):
    """Return (hs, y) of the convolution stack: hs[s] is the bf16 intermediate written by
    stage s (s = 0 .. N-2), y = the last convolution in fp64.  ws is a sequence of KRSC
    weight tensors, one per stage."""
    if len(ws) < 1:
        raise ValueError("a stack needs at least one convolution")
    h = _as64(x)
    hs = []
    for w in ws[:-1]:
        h = bf16_intermediate(relu(conv2d_nhwc(h, w, stride, pad)))
        hs.append(h)
    return hs, conv2d_nhwc(h, ws[-1], stride, pad)


def mlp_gelu_rows(X, W1, W2, rows):
    """(H[rows], Y[rows]) of ``mlp_gelu`` for a subset of token rows.

    Every output row of the chain depends only on the same input row, so a
    sampled check at full size evaluates just those rows.
    """
    X = _as64(X)[np.asarray(rows)]
    return mlp_gelu(X, W1, W2)


def mlp_swiglu_rows(X, Wgate, Wup, Wdown, rows):
    """(H[rows], Y[rows]) of ``mlp_swiglu`` for a subset of token rows."""
    X = _as64(X)[np.asarray(rows)]
    return mlp_swiglu(X, Wgate, Wup, Wdown)


def softmax_heads(s, head):
    """Softmax of each row of s [M, N] over consecutive groups of ``head`` columns."""
    M, N = s.shape
    g = s.reshape(M, N // head, head)
    e = np.exp(g - g.max(axis=2, keepdims=True))
    return (e / e.sum(axis=2, keepdims=True)).reshape(M, N)


def attention(X, Wqkv, W2, head=128):
    """(XQKV, XDot, Y) of the self-attention block; XQKV and XDot as stored (bf16 values)."""
    X, Wqkv, W2 = _as64(X), _as64(Wqkv), _as64(W2)
    n1 = Wqkv.shape[1] // 3
    xqkv = bf16_intermediate(X @ Wqkv)
    xq, xv, xk = xqkv[:, :n1], xqkv[:, n1:2 * n1], xqkv[:, 2 * n1:]
    xdot = bf16_intermediate(softmax_heads(xq * xv, head) * xk)
    return xqkv, xdot, xdot @ W2


def attention_rows(X, Wqkv, W2, rows, head=128):
    """(XQKV, XDot, Y) of ``attention`` for a subset of token rows (each output row
    depends only on the same input row)."""
    X = _as64(X)[np.asarray(rows)]
    return attention(X, Wqkv, W2, head)
