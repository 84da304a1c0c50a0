"""GPU tests of the row-band trigger that lets a tensor-parallel shard reduce its output
while later bands are still being computed (cusync_run_mlp_bands, cusync_band_wait).

On one GPU the reduction is stood in for by a copy: after each band wait, a side stream
copies the band's rows of Y, which holds NaN before the run.  A band released early would
copy NaN or a partly written band, so the copies equal the final Y only if every wait
ended after its band was complete.  The chain's output is byte-identical to a run without
bands.  Two shards run one after the other give the layer's output summed."""

import numpy as np
import pytest
import torch

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth, tp

from gpu_helpers import RTOL_ABS, assert_within_tol, bits, device_mlp_operands, f64, run_mlp

pytestmark = pytest.mark.gpu


def _banded_runs(desc, ops, runs=2):
    M, N1, N2 = desc.M, desc.N1, desc.N2
    H = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    Z = torch.empty_like(Y)
    ch = cs.Chain(desc)
    side = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    try:
        for _ in range(runs):
            Y.fill_(float("nan"))
            Z.fill_(float("nan"))
            side.wait_stream(cur)
            cs.cusync_run_mlp_bands(ch.handle, *ops, H, Y, side, cur)
            with torch.cuda.stream(side):
                for b, (r0, n) in enumerate(tp.band_slices(desc)):
                    cs.cusync_band_wait(ch.handle, b, side)
                    Z[r0:r0 + n].copy_(Y[r0:r0 + n])
            cur.wait_stream(side)
            torch.cuda.synchronize()
            st, code, detail = ch.check()
            assert st == cs.OK, (cs.status_string(st), hex(code), hex(detail))
            assert torch.equal(Z.view(torch.int16), Y.view(torch.int16)), "a band was reduced before it was complete"
        return H.cpu(), Y.cpu()
    finally:
        ch.close()


@pytest.mark.parametrize("pol,launch", [("ROW", cs.LAUNCH_PERSISTENT), ("TILE", cs.LAUNCH_PDL),
                                        ("STREAM", cs.LAUNCH_PERSISTENT), ("SENTINEL", cs.LAUNCH_PERSISTENT)])
@pytest.mark.parametrize("M,pair,bands,ks", [(1024, 2, 4, 0), (1000, 2, 3, 0), (640, 1, 5, 2)])
def test_band_waits_end_after_their_band(pol, launch, M, pair, bands, ks):
    K, N1, N2 = 512, 1024, 512
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=21)
    H_ref, Y_ref = chains.mlp_gelu(f64(X), f64(W1), f64(W2))
    ops = device_mlp_operands(X, W1, W2)
    d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2, cta_pair=pair, bands=bands,
                     ksplit_consumer=ks)
    H, Y = _banded_runs(d, ops)
    assert_within_tol(f64(H), H_ref, "H")
    assert_within_tol(f64(Y), Y_ref, "Y")
    d0 = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2, cta_pair=pair, ksplit_consumer=ks)
    H0, Y0, _ = run_mlp(d0, *ops)
    assert np.array_equal(bits(H), bits(H0)) and np.array_equal(bits(Y), bits(Y0))


def test_two_shards_sum_to_the_layer_output():
    """Tensor parallelism of two shards on one GPU, one after the other: each shard's chain
    with its band reductions (here: copies of each band as it completes), then the sum."""
    M, K, N1, N2, world = 1024, 512, 2048, 512, 2
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=22)
    _, Y_ref = chains.mlp_gelu(f64(X), f64(W1), f64(W2))
    Xd, W1t, W2t = device_mlp_operands(X, W1, W2)
    total = torch.zeros((M, N2), dtype=torch.float64)
    bound = torch.zeros((M, N2), dtype=torch.float64)
    for r in range(world):
        w1s, w2s = tp.shard_mlp_weights(W1t, W2t, r, world)
        d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, K=K, N1=N1 // world, N2=N2, bands=4)
        shard = tp.TensorParallelMLP(d)
        H = torch.empty((M, N1 // world), dtype=torch.bfloat16, device="cuda")
        Y = torch.full((M, N2), float("nan"), dtype=torch.bfloat16, device="cuda")
        got = []
        try:
            shard.run(Xd, w1s, w2s, H, Y, reduce=lambda t: got.append(t.clone()))
            torch.cuda.synchronize()
            st, code, _ = shard.check()
            assert st == cs.OK, hex(code)
        finally:
            shard.close()
        Yc = torch.cat(got, 0)
        assert torch.equal(Yc.view(torch.int16), Y.view(torch.int16))
        lo, hi = tp.shard_range(N1, r, world)
        _, Yr_ref = chains.mlp_gelu(f64(X), f64(W1[:, lo:hi]), f64(W2[lo:hi]))
        assert_within_tol(f64(Yc.cpu()), Yr_ref, f"shard {r}")
        total += Yc.cpu().double()
        bound += RTOL_ABS * torch.clamp(torch.from_numpy(np.abs(Yr_ref)), min=1.0)
    # each shard is within its own bound; the sum is within the sum of the shards' bounds
    assert bool(torch.all(torch.abs(total - torch.from_numpy(Y_ref)) <= bound))


def test_band_waits_end_when_a_tile_gives_up():
    """A producer tile that never posts makes consumer waits expire (a reported timeout);
    the band waits still end (the tiles post their bands, and the release after the run
    raises every band semaphore to its target), so nothing on the side stream hangs."""
    M, K, N1, N2 = 512, 256, 1024, 256
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=23)
    ops = device_mlp_operands(X, W1, W2)
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "TILE", M=M, K=K, N1=N1, N2=N2, bands=2, flags=cs.DEBUG_SKIP_POST,
                     timeout_ns=20_000_000)
    ch = cs.Chain(d)
    side = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    H = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    Z = torch.empty_like(Y)
    try:
        cs.cusync_run_mlp_bands(ch.handle, *ops, H, Y, side, cur)
        with torch.cuda.stream(side):
            for b, (r0, n) in enumerate(tp.band_slices(d)):
                cs.cusync_band_wait(ch.handle, b, side)
                Z[r0:r0 + n].copy_(Y[r0:r0 + n])
        cur.wait_stream(side)
        torch.cuda.synchronize()
        st, code, _ = ch.check()
        assert st == cs.ERR_TIMEOUT
        # after the reset that check performs, band waits need a new banded run
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_band_wait(ch.handle, 0, side)
        assert e.value.status == cs.ERR_INVALID_ARG
    finally:
        ch.close()


def test_band_calls_refused_in_capture_and_without_bands():
    M, K, N1, N2 = 512, 256, 1024, 256
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=24)
    ops = device_mlp_operands(X, W1, W2)
    H = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    plain = cs.Chain(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, K=K, N1=N1, N2=N2))
    banded = cs.Chain(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, K=K, N1=N1, N2=N2, bands=2))
    side = torch.cuda.Stream()
    try:
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_run_mlp_bands(plain.handle, *ops, H, Y, side)
        assert e.value.status == cs.ERR_INVALID_ARG
        with pytest.raises(cs.CusyncError) as e:     # no banded run yet
            cs.cusync_band_wait(banded.handle, 0, side)
        assert e.value.status == cs.ERR_INVALID_ARG
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            with pytest.raises(cs.CusyncError) as e:
                cs.cusync_run_mlp_bands(banded.handle, *ops, H, Y, side)
        assert e.value.status == cs.ERR_UNSUPPORTED
        torch.cuda.synchronize()
    finally:
        plain.close()
        banded.close()
