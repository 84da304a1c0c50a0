"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and rounds them to bf16 with PyTorch's
conversion; it holds none of the chains' arithmetic.  The oracle never
imports it: callers pass the same bf16 tensors to the oracle (as fp64) and
to the CUDA library.

Recipe (one ``numpy.random.default_rng(seed)`` per workload, draws in the
order listed, each array rounded to bf16 with round-to-nearest-even):

* GeLU MLP:   X [M,K] ~ N(0,1); W1 [K,N1] ~ N(0,0.02); W2 [N1,N2] ~ N(0,0.02)
* SwiGLU MLP: X [M,K] ~ N(0,1); Wgate, Wup [K,N1] ~ N(0,0.02); Wdown [N1,N2] ~ N(0,0.02)
* conv pair:  x [N,H,W,C] ~ N(0,1) (NHWC); w1, w2 [K,3,3,C] ~ N(0,0.03) (KRSC)
* attention:  X [M,K] ~ N(0,1); QKV [K,3*N1] ~ N(0,0.02); W2 [N1,N2] ~ N(0,0.02)
* conv stack: x [N,H,W,C] ~ N(0,1); w [S,C,3,3,C] ~ N(0, 2/(9C)) (S stages' KRSC weights)

N(mu, sigma) takes sigma as the standard deviation.  Shapes follow the
GPT-3 145B MLP shard of [cuSync] §II-B / §III-A (H = 12288, one of 8
tensor-parallel shards: X [B,12288], W1 [12288,6144], W2 [6144,12288]) and
the 14x14x256 ResNet-38 layer of Table ``tab:resnet-sizes``; the self-attention
block of Fig. ``fig:gpt-3:attention`` takes the same shard (QKV [12288, 3*1536],
W2 [1536, 12288]); the convolution stacks are the four layer groups of that table
(56x56x64: 3 layers of two convolutions, 28x28x128: 4, 14x14x256: 6, 7x7x512: 3) at a
batch of 32 images, the batch of the convolution pair; no dataset or trained weights
are involved.
"""

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                  # "mlp_gelu" | "mlp_swiglu" | "conv_relu" | "attention" | "conv_stack"
    dims: dict = field(default_factory=dict)

    def gemm_flops(self):
        d = self.dims
        if self.kind == "mlp_gelu":
            return 2 * d["M"] * d["K"] * d["N1"] + 2 * d["M"] * d["N1"] * d["N2"]
        if self.kind == "mlp_swiglu":
            return 2 * d["M"] * d["K"] * (2 * d["N1"]) + 2 * d["M"] * d["N1"] * d["N2"]
        if self.kind == "conv_relu":
            pix = d["N"] * d["H"] * d["W"]
            return 2 * pix * d["K"] * 9 * d["C"] + 2 * pix * d["K"] * 9 * d["K"]
        if self.kind == "attention":   # the two GEMMs; the pointwise stage has no tensor work
            return 2 * d["M"] * d["K"] * (3 * d["N1"]) + 2 * d["M"] * d["N1"] * d["N2"]
        if self.kind == "conv_stack":
            return d["S"] * 2 * d["N"] * d["H"] * d["W"] * d["C"] * 9 * d["C"]
        raise ValueError(self.kind)


def _mlp(name, M, K, N1, N2):
    return Workload(name, "mlp_gelu", dict(M=M, K=K, N1=N1, N2=N2))


WORKLOADS = {
    w.name: w
    for w in [
        _mlp("mlp_tiny_m64", 64, 256, 1024, 256),
        _mlp("gpt3_mlp_m256", 256, 12288, 6144, 12288),
        _mlp("gpt3_mlp_m512", 512, 12288, 6144, 12288),
        _mlp("gpt3_mlp_m1024", 1024, 12288, 6144, 12288),
        _mlp("gpt3_mlp_m2048", 2048, 12288, 6144, 12288),
        _mlp("gpt3_mlp_m4096", 4096, 12288, 6144, 12288),
        Workload("swiglu_m256", "mlp_swiglu", dict(M=256, K=8192, N1=3584, N2=8192)),
        Workload("swiglu_m1024", "mlp_swiglu", dict(M=1024, K=8192, N1=3584, N2=8192)),
        Workload("conv_resnet14_n32", "conv_relu", dict(N=32, H=14, W=14, C=256, K=256)),
        Workload("gpt3_attn_m256", "attention", dict(M=256, K=12288, N1=1536, N2=12288)),
        Workload("gpt3_attn_m1024", "attention", dict(M=1024, K=12288, N1=1536, N2=12288)),
        Workload("resnet38_56x56x64_n32", "conv_stack", dict(N=32, H=56, W=56, C=64, S=6)),
        Workload("resnet38_28x28x128_n32", "conv_stack", dict(N=32, H=28, W=28, C=128, S=8)),
        Workload("resnet38_14x14x256_n32", "conv_stack", dict(N=32, H=14, W=14, C=256, S=12)),
        Workload("resnet38_7x7x512_n32", "conv_stack", dict(N=32, H=7, W=7, C=512, S=6)),
    ]
}


def to_bf16(a):
    """numpy float array -> CPU bf16 tensor (round to nearest even via float32)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng, shape, std):
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)


def mlp_gelu_inputs(M, K, N1, N2, seed=0):
    """(X [M,K], W1 [K,N1], W2 [N1,N2]) as CPU bf16 tensors."""
    rng = np.random.default_rng(seed)
    X = to_bf16(_normal(rng, (M, K), 1.0))
    W1 = to_bf16(_normal(rng, (K, N1), 0.02))
    W2 = to_bf16(_normal(rng, (N1, N2), 0.02))
    return X, W1, W2


def mlp_swiglu_inputs(M, K, N1, N2, seed=0):
    """(X [M,K], Wgate [K,N1], Wup [K,N1], Wdown [N1,N2]) as CPU bf16 tensors."""
    rng = np.random.default_rng(seed)
    X = to_bf16(_normal(rng, (M, K), 1.0))
    Wg = to_bf16(_normal(rng, (K, N1), 0.02))
    Wu = to_bf16(_normal(rng, (K, N1), 0.02))
    Wd = to_bf16(_normal(rng, (N1, N2), 0.02))
    return X, Wg, Wu, Wd


def conv_inputs(N, H, W, C, K, seed=0):
    """(x [N,H,W,C] NHWC, w1 [K,3,3,C], w2 [K,3,3,K] KRSC) as CPU bf16 tensors."""
    rng = np.random.default_rng(seed)
    x = to_bf16(_normal(rng, (N, H, W, C), 1.0))
    w1 = to_bf16(_normal(rng, (K, 3, 3, C), 0.03))
    w2 = to_bf16(_normal(rng, (K, 3, 3, K), 0.03))
    return x, w1, w2


def conv_stack_inputs(N, H, W, C, stages, seed=0):
    """(x [N,H,W,C] NHWC, w [stages,C,3,3,C]: each stage's KRSC weights) as CPU bf16 tensors.

    Weights ~ N(0, 2 / (9 C)) (He initialisation for a 3x3 convolution followed by ReLU),
    so the activations keep their scale through a deep stack; for the 14x14x256 layer
    group this is the 0.03 of the convolution pair."""
    rng = np.random.default_rng(seed)
    x = to_bf16(_normal(rng, (N, H, W, C), 1.0))
    w = to_bf16(_normal(rng, (stages, C, 3, 3, C), float(np.sqrt(2.0 / (9 * C)))))
    return x, w


def attention_inputs(M, K, N1, N2, seed=0):
    """(X [M,K], QKV [K,3*N1] -- the XQ, XV, XK column blocks --, W2 [N1,N2]) as CPU bf16
    tensors."""
    rng = np.random.default_rng(seed)
    X = to_bf16(_normal(rng, (M, K), 1.0))
    Wqkv = to_bf16(_normal(rng, (K, 3 * N1), 0.02))
    W2 = to_bf16(_normal(rng, (N1, N2), 0.02))
    return X, Wqkv, W2


def workload_inputs(w: Workload, seed=0):
    d = w.dims
    if w.kind == "mlp_gelu":
        return mlp_gelu_inputs(d["M"], d["K"], d["N1"], d["N2"], seed)
    if w.kind == "mlp_swiglu":
        return mlp_swiglu_inputs(d["M"], d["K"], d["N1"], d["N2"], seed)
    if w.kind == "conv_relu":
        return conv_inputs(d["N"], d["H"], d["W"], d["C"], d["K"], seed)
    if w.kind == "attention":
        return attention_inputs(d["M"], d["K"], d["N1"], d["N2"], seed)
    if w.kind == "conv_stack":
        return conv_stack_inputs(d["N"], d["H"], d["W"], d["C"], d["S"], seed)
    raise ValueError(w.kind)


def f64(t):
    """CPU bf16 tensor -> fp64 numpy array (exact)."""
    return t.to(torch.float64).numpy()
