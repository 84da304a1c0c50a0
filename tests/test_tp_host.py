"""CPU tests of the tensor-parallel MLP shard (tile_level_sync_gb300.tp): the sum of the
shards' oracle outputs is the unsharded layer's output; the row bands tile Y; and two gloo
ranks running the band-by-band reduction on their shards' oracle outputs obtain the
unsharded output, each band reduced only after its wait."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth, tp


def _shards(kind, M, K, N1, N2, world, seed=3):
    """(unsharded (H, Y), per-rank oracle (H_r, Y_r)) from the same inputs."""
    if kind == "gelu":
        X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed)
        W1t = W1.t().contiguous()
        full = chains.mlp_gelu(synth.f64(X), synth.f64(W1), synth.f64(W2))
    else:
        X, Wg, Wu, W2 = synth.mlp_swiglu_inputs(M, K, N1, N2, seed)
        W1t = torch.cat([Wg.t(), Wu.t()], 0).contiguous()
        full = chains.mlp_swiglu(synth.f64(X), synth.f64(Wg), synth.f64(Wu), synth.f64(W2))
    W2t = W2.t().contiguous()
    parts = []
    for r in range(world):
        w1s, w2s = tp.shard_mlp_weights(W1t, W2t, r, world, swiglu=(kind != "gelu"))
        n = w2s.shape[1]
        if kind == "gelu":
            parts.append(chains.mlp_gelu(synth.f64(X), synth.f64(w1s.t()), synth.f64(w2s.t())))
        else:
            parts.append(chains.mlp_swiglu(synth.f64(X), synth.f64(w1s[:n].t()), synth.f64(w1s[n:].t()),
                                           synth.f64(w2s.t())))
    return full, parts


@pytest.mark.parametrize("kind", ["gelu", "swiglu"])
@pytest.mark.parametrize("world", [2, 4])
def test_shard_outputs_sum_to_the_layer_output(kind, world):
    """H's columns are independent (the activation acts element-wise), so each shard's H is
    the layer's H restricted to its columns, and sum_r H_r W2_r = H W2."""
    M, K, N1, N2 = 24, 64, 128, 48
    (H, Y), parts = _shards(kind, M, K, N1, N2, world)
    for r, (Hr, _) in enumerate(parts):
        lo, hi = tp.shard_range(N1, r, world)
        assert np.array_equal(Hr, H[:, lo:hi])
    Ysum = sum(Yr for _, Yr in parts)
    np.testing.assert_allclose(Ysum, Y, rtol=1e-12, atol=1e-12)


def test_shard_weights_layout():
    W1t = torch.arange(8 * 3, dtype=torch.float32).reshape(8, 3)        # [N1=8, K=3]
    W2t = torch.arange(5 * 8, dtype=torch.float32).reshape(5, 8)        # [N2=5, N1=8]
    w1, w2 = tp.shard_mlp_weights(W1t, W2t, 1, 2)
    assert torch.equal(w1, W1t[4:8]) and torch.equal(w2, W2t[:, 4:8])
    G = torch.cat([W1t, W1t + 100], 0)                                  # SwiGLU [2*N1, K]
    w1, w2 = tp.shard_mlp_weights(G, W2t, 0, 4, swiglu=True)
    assert torch.equal(w1, torch.cat([G[0:2], G[8:10]], 0)) and torch.equal(w2, W2t[:, 0:2])
    with pytest.raises(ValueError):
        tp.shard_range(10, 0, 4)


@pytest.mark.parametrize("M,pair,bands", [(1024, 2, 4), (1000, 2, 3), (640, 1, 5), (256, 2, 1), (4096, 2, 16)])
def test_bands_tile_the_output(M, pair, bands):
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, K=512, N1=1024, N2=512, cta_pair=pair, num_sms=148,
                     bands=bands)
    sl = tp.band_slices(d)
    assert len(sl) == bands
    tm = 128 * pair
    assert sl[0][0] == 0 and sum(n for _, n in sl) == M
    for (a, n), (b, _) in zip(sl, sl[1:]):
        assert a + n == b and a % tm == 0 and n > 0


def test_band_refusals():
    base = dict(M=1024, K=512, N1=1024, N2=512, num_sms=148)
    for kw, want in ((dict(bands=17), cs.ERR_UNSUPPORTED), (dict(bands=5), cs.ERR_UNSUPPORTED),  # 4 row tiles
                     (dict(bands=2, raster_rows=2), cs.ERR_UNSUPPORTED), (dict(bands=-1), cs.ERR_INVALID_ARG)):
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", **base, **kw))
        assert e.value.status == want, kw
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", n=2, h=14, w=14, c=64, k_out=64, bands=1))
    assert e.value.status == cs.ERR_UNSUPPORTED
    with pytest.raises(cs.CusyncError) as e:   # a chain without bands has none to describe
        cs.cusync_band_rows(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", **base), 0)
    assert e.value.status == cs.ERR_INVALID_ARG


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from tile_level_sync_gb300 import tp as tpm
        import tile_level_sync_gb300 as csm
        M, K, N1, N2 = 640, 64, 256, 96
        (H, Y), parts = _shards("gelu", M, K, N1, N2, world, seed=11)
        Yr = torch.from_numpy(parts[rank][1].copy())
        d = csm.make_desc(csm.CHAIN_MLP_GELU, "ROW", M=M, K=K, N1=N1 // world, N2=N2, cta_pair=1, num_sms=148,
                          bands=5)
        events = []
        tpm.reduce_bands(Yr, tpm.band_slices(d), lambda b: events.append(("wait", b)),
                         lambda t: (events.append(("reduce", int(t.data_ptr()))), dist.all_reduce(t)))
        q.put((rank, float(np.max(np.abs(Yr.numpy() - Y))), events, [int(Yr[r0:r0 + n].data_ptr())
                                                                      for r0, n in tpm.band_slices(d)]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_band_by_band_to_the_layer_output():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    for _ in range(world):
        rank, err, events, ptrs = q.get(timeout=10)
        assert err < 1e-9, (rank, err)
        # each band's reduction follows its wait, bands in order, each band's rows once
        assert [e[0] for e in events] == ["wait", "reduce"] * 5
        assert [e[1] for e in events[0::2]] == list(range(5))
        assert [e[1] for e in events[1::2]] == ptrs
