"""GPU parity of the self-attention chain (QKV GEMM -> per-head softmax(XQ * XV) * XK ->
output GEMM): every policy and launch mode against the oracle, byte-identical to one
another and to the three stream-ordered kernels, with and without a K split of the QKV
GEMM, and replayed from a CUDA graph."""

import numpy as np
import pytest
import torch

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth

from gpu_helpers import assert_within_tol, bits, f64

pytestmark = pytest.mark.gpu

POLICIES = ["STREAM", "ROW", "TILE", "STRIDED"]
LAUNCHES = [cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL]


def _operands(M, K, N1, N2, seed):
    X, Wqkv, W2 = synth.attention_inputs(M, K, N1, N2, seed)
    ref = chains.attention(f64(X), f64(Wqkv), f64(W2))
    dev = (X.cuda(), Wqkv.t().contiguous().cuda(), W2.t().contiguous().cuda())
    return dev, ref


def _run(d, ops, M, N1, N2, runs=2):
    xqkv = torch.empty((M, 3 * N1), dtype=torch.bfloat16, device="cuda")
    xdot = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    ch = cs.Chain(d)
    try:
        for _ in range(runs):
            ch.run(ops[0], ops[1], ops[2], xqkv, y, h2=xdot)
        st, code, detail = ch.check()
        assert st == cs.OK, f"{cs.status_string(st)} 0x{code:08x} 0x{detail:x}"
        torch.cuda.synchronize()
        return xqkv.cpu(), xdot.cpu(), y.cpu()
    finally:
        ch.close()


@pytest.mark.parametrize("M,K,N1,N2,tile_n,ksplit", [
    (200, 512, 512, 384, 256, 1),     # ragged token count, 4 heads
    (256, 256, 768, 256, 128, 1),     # 18 QKV column tiles, 6 heads
    (130, 2048, 512, 264, 256, 3),    # K split of the QKV GEMM, ragged N2
])
@pytest.mark.parametrize("pair", [1, 2])
def test_attention_all_policies(M, K, N1, N2, tile_n, ksplit, pair):
    ops, (xqkv_ref, xdot_ref, y_ref) = _operands(M, K, N1, N2, seed=31)
    ref = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_ATTENTION, pol, launch, M=M, K=K, N1=N1, N2=N2, tile_n=tile_n,
                             cta_pair=pair, ksplit=ksplit)
            xqkv, xdot, y = _run(d, ops, M, N1, N2)
            assert_within_tol(f64(xqkv), xqkv_ref, f"XQKV {pol} {launch}")
            assert_within_tol(f64(xdot), xdot_ref, f"XDot {pol} {launch}")
            assert_within_tol(f64(y), y_ref, f"Y {pol} {launch}")
            b = (bits(xqkv), bits(xdot), bits(y))
            if ref is None:
                ref = b
            else:
                assert all(np.array_equal(u, v) for u, v in zip(b, ref)), (pol, launch)


def test_attention_graph_replay():
    M, K, N1, N2 = 256, 512, 512, 256
    ops, (_, _, y_ref) = _operands(M, K, N1, N2, seed=32)
    d = cs.make_desc(cs.CHAIN_ATTENTION, "STRIDED", M=M, K=K, N1=N1, N2=N2, cta_pair=1)
    ch = cs.Chain(d)
    xqkv = torch.empty((M, 3 * N1), dtype=torch.bfloat16, device="cuda")
    xdot = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    try:
        ch.run(ops[0], ops[1], ops[2], xqkv, y, h2=xdot)
        assert ch.check()[0] == cs.OK
        direct = bits(y.cpu())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ch.run(ops[0], ops[1], ops[2], xqkv, y, h2=xdot)
        for _ in range(3):
            y.zero_()
            g.replay()
            assert ch.check()[0] == cs.OK
            assert np.array_equal(bits(y.cpu()), direct)
        assert_within_tol(f64(y.cpu()), y_ref, "Y graph")
        del g
    finally:
        ch.close()
