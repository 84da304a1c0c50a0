"""Epilogue activations of the producer GEMM (oracle; test infrastructure).

[cuSync] §II-B (GPT Models) and Fig. ``fig:gpt-3:mlp`` fuse a GeLU into the
first GeMM of the MLP; the page does not say which GeLU.  The tanh form is
used here (the reading recorded in the design notes):

    gelu(z) = 0.5 * z * (1 + tanh( sqrt(2/pi) * (z + 0.044715 * z**3) ))

The SwiGLU chain's epilogue is silu(g) * u with silu(g) = g * sigmoid(g),
and the conv chain's is ReLU ([cuSync] §II-B, ResNet; Table
``tab:resnet-sizes`` lists pairs of 3x3 convolutions).
"""

import numpy as np

_SQRT_2_OVER_PI = np.sqrt(2.0 / np.pi)
_GELU_CUBIC = 0.044715


def gelu_tanh(z):
    """tanh-approximated GeLU, fp64."""
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(_SQRT_2_OVER_PI * (z + _GELU_CUBIC * z ** 3)))


def silu(g):
    """g * sigmoid(g), fp64, written so that large |g| neither overflows nor loses sign."""
    g = np.asarray(g, dtype=np.float64)
    # sigmoid(g) = 1 / (1 + exp(-g)) for g >= 0 and exp(g) / (1 + exp(g)) for g < 0.
    e = np.exp(-np.abs(g))
    sig = np.where(g >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    return g * sig


def relu(y):
    """max(y, 0), fp64."""
    y = np.asarray(y, dtype=np.float64)
    return np.maximum(y, 0.0)
