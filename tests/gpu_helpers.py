"""Shared helpers of the GPU tests: run a chain through the C ABI and compare with the oracle."""

import numpy as np
import torch

import tile_level_sync_gb300 as cs
from tile_level_sync_gb300 import synth

RTOL_ABS = 2e-2   # |gpu - ref| <= 2e-2 * max(1, |ref|)


def within_tol(gpu, ref, scale=1.0):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = scale * RTOL_ABS * np.maximum(1.0, np.abs(ref))
    bad = err > bound
    return (not np.any(bad)), float(np.max(err / bound)) if err.size else 0.0


def assert_within_tol(gpu, ref, what, scale=1.0):
    ok, worst = within_tol(gpu, ref, scale)
    assert ok, f"{what}: worst error / bound = {worst:.3f}"


def device_mlp_operands(X, W1, W2, Wup=None):
    """CPU bf16 [K,N] weights -> device tensors in the library's [N,K] layout."""
    dev = "cuda"
    Xd = X.to(dev)
    if Wup is None:
        W1t = W1.t().contiguous().to(dev)
    else:
        W1t = torch.cat([W1.t(), Wup.t()], dim=0).contiguous().to(dev)
    W2t = W2.t().contiguous().to(dev)
    return Xd, W1t, W2t


def run_mlp(desc, Xd, W1t, W2t, runs=1, check=True):
    M, N1, N2 = desc.M, desc.N1, desc.N2
    H = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    ch = cs.Chain(desc)
    try:
        for _ in range(runs):
            ch.run(Xd, W1t, W2t, H, Y)
        st, code, detail = ch.check()
        if check:
            assert st == cs.OK, f"chain status {cs.status_string(st)} code=0x{code:08x} detail=0x{detail:x}"
        torch.cuda.synchronize()
        return H.cpu(), Y.cpu(), st
    finally:
        ch.close()


def run_conv(desc, x, w1, w2, runs=1, check=True):
    n, h, w, k = desc.n, desc.h, desc.w, desc.k_out
    y1 = torch.empty((n, h, w, k), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((n, h, w, k), dtype=torch.bfloat16, device="cuda")
    ch = cs.Chain(desc)
    try:
        for _ in range(runs):
            ch.run(x.cuda(), w1.cuda(), w2.cuda(), y1, y2)
        st, code, detail = ch.check()
        if check:
            assert st == cs.OK, f"chain status {cs.status_string(st)} code=0x{code:08x} detail=0x{detail:x}"
        torch.cuda.synchronize()
        return y1.cpu(), y2.cpu(), st
    finally:
        ch.close()


def f64(t):
    return synth.f64(t)


def bits(t):
    return t.view(torch.int16).numpy()
