"""CUDA-graph capture of chain runs: a captured run replays as a new run each time (the
run count the semaphores are compared against lives in device memory), for every
policy and launch mode, with results identical to direct calls and to the oracle."""

import numpy as np
import pytest
import torch

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth

from gpu_helpers import assert_within_tol, bits, device_mlp_operands, f64

pytestmark = pytest.mark.gpu

CASES = [("STREAM", cs.LAUNCH_PERSISTENT), ("ROW", cs.LAUNCH_PERSISTENT), ("ROW", cs.LAUNCH_PDL),
         ("TILE", cs.LAUNCH_PERSISTENT), ("TILE", cs.LAUNCH_PDL), ("STRIDED", cs.LAUNCH_PERSISTENT),
         ("SENTINEL", cs.LAUNCH_PERSISTENT), ("SENTINEL", cs.LAUNCH_PDL)]


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("pol,launch", CASES)
def test_mlp_graph_replay_matches_direct_runs(pol, launch, pair):
    M, K, N1, N2 = 520, 512, 1024, 512
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=11)
    H_ref, Y_ref = chains.mlp_gelu(f64(X), f64(W1), f64(W2))
    ops = device_mlp_operands(X, W1, W2)
    d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2, cta_pair=pair)
    ch = cs.Chain(d)
    H = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    try:
        ch.run(*ops, H, Y)                       # direct run (also the run count 1)
        st, code, _ = ch.check()
        assert st == cs.OK, hex(code)
        direct = (bits(H.cpu()), bits(Y.cpu()))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ch.run(*ops, H, Y)
            ch.run(*ops, H, Y)
        for _ in range(3):
            H.zero_()
            Y.zero_()
            g.replay()
            st, code, _ = ch.check()
            assert st == cs.OK, hex(code)
            assert np.array_equal(bits(H.cpu()), direct[0]) and np.array_equal(bits(Y.cpu()), direct[1])
        assert_within_tol(f64(Y.cpu()), Y_ref, f"Y {pol}")
        assert_within_tol(f64(H.cpu()), H_ref, f"H {pol}")
        # direct calls after the replays still see the right run count
        Y.zero_()
        ch.run(*ops, H, Y)
        st, _, _ = ch.check()
        assert st == cs.OK and np.array_equal(bits(Y.cpu()), direct[1])
        del g
    finally:
        ch.close()


def test_conv_graph_replay_matches_direct_runs():
    n, h, w, c, k = 2, 14, 14, 128, 128
    x, w1, w2 = synth.conv_inputs(n, h, w, c, k, seed=12)
    xd, w1d, w2d = x.cuda(), w1.cuda(), w2.cuda()
    for pol in ("ROW", "TILE", "SENTINEL"):
        d = cs.make_desc(cs.CHAIN_CONV_RELU, pol, n=n, h=h, w=w, c=c, k_out=k, tile_n=128)
        ch = cs.Chain(d)
        y1 = torch.empty((n, h, w, k), dtype=torch.bfloat16, device="cuda")
        y2 = torch.empty_like(y1)
        try:
            ch.run(xd, w1d, w2d, y1, y2)
            assert ch.check()[0] == cs.OK
            direct = bits(y2.cpu())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                ch.run(xd, w1d, w2d, y1, y2)
            for _ in range(3):
                y2.zero_()
                g.replay()
                assert ch.check()[0] == cs.OK
                assert np.array_equal(bits(y2.cpu()), direct), pol
            del g
        finally:
            ch.close()
