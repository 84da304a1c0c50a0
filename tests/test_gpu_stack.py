"""GPU parity of the convolution stack (N dependent 3x3 convolutions in one chain) against
the oracle, for every policy and launch mode; byte-identical across them.

Tolerance.  Each stage is held to the chains' bound, 2e-2 * max(1, |ref|), against the
oracle applied to the GPU's own bf16 input of that stage (the sentinel runs keep every
intermediate).  End to end, the output is compared with the fp64 oracle of the whole
stack under that bound times sqrt(N - 1): the GPU accumulates in fp32 and the oracle in
fp64, so where the two land on opposite sides of a bf16 rounding boundary an
intermediate element differs by one bf16 ulp; each of the N - 1 rounded intermediates
adds such differences independently of the others, and the He-scaled weights carry
them to the next stage with unit gain, so they grow like a random walk over the
roundings (a stack of two is the pair's bound)."""

import numpy as np
import pytest
import torch

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth

from gpu_helpers import assert_within_tol, bits, f64

pytestmark = pytest.mark.gpu

POLICIES = ["STREAM", "ROW", "TILE", "SENTINEL"]
LAUNCHES = [cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL]


def run_stack(desc, x, w, runs=1, check=True):
    info = cs.cusync_plan_info(desc)
    work = torch.empty(info.work_bytes // 2, dtype=torch.bfloat16, device="cuda")
    y = torch.empty((desc.n, desc.h, desc.w, desc.c), dtype=torch.bfloat16, device="cuda")
    ch = cs.Chain(desc)
    try:
        xd, wd = x.cuda(), w.cuda()
        for _ in range(runs):
            ch.run(xd, wd, None, work, y)
        st, code, detail = ch.check()
        if check:
            assert st == cs.OK, f"chain status {cs.status_string(st)} code=0x{code:08x} detail=0x{detail:x}"
        torch.cuda.synchronize()
        return work.cpu(), y.cpu(), info
    finally:
        ch.close()


def _buffers(work, info, shape):
    return work.view(info.work_buffers, *shape)


def sentinel_sets(work, info, shape, stages, runs):
    """(the set of intermediates the last of `runs` runs used, the other set): run r of a
    chain uses set r % 2, and fills the other one with the sentinel."""
    bufs = _buffers(work, info, shape)
    used = runs & 1
    return bufs[used * (stages - 1):(used + 1) * (stages - 1)], bufs[(1 - used) * (stages - 1):(2 - used) * (stages - 1)]


def assert_all_sentinel(bufs, what):
    b = bufs.contiguous().view(torch.int16).numpy().astype(np.uint16)
    assert np.all(b == 0x8000), f"{what}: {int((b != 0x8000).sum())} elements are not the sentinel"


def depth_scale(stages):
    return float(np.sqrt(stages - 1))


def check_stagewise(x, wt, bufs, y, stages, what):
    """Every stage against the oracle applied to the GPU's input of that stage."""
    inp = f64(x)
    for s in range(stages):
        out = chains.conv2d_nhwc(inp, f64(wt[s]))
        if s < stages - 1:
            want = chains.bf16_intermediate(np.maximum(out, 0.0))
            assert_within_tol(f64(bufs[s]), want, f"{what} stage {s}")
            inp = f64(bufs[s])
        else:
            assert_within_tol(f64(y), out, f"{what} last stage")


@pytest.mark.parametrize("n,h,w,c,stages,tile_n", [
    (2, 8, 8, 64, 3, 128),      # ragged column tile (64 of 128 channels)
    (1, 14, 14, 128, 4, 128),   # two row tiles per image, halo across them
    (2, 6, 20, 64, 5, 256),     # several row tiles, deep stack
    (1, 7, 7, 128, 2, 128),     # a stack of two is the convolution pair
])
def test_stack_all_policies(n, h, w, c, stages, tile_n):
    x, wt = synth.conv_stack_inputs(n, h, w, c, stages, seed=21)
    hs_ref, y_ref = chains.conv_stack(f64(x), [f64(wt[s]) for s in range(stages)])
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_CONV_STACK, pol, launch, n=n, h=h, w=w, c=c, stages=stages, tile_n=tile_n)
            work, y, info = run_stack(d, x, wt, runs=2)
            assert_within_tol(f64(y), y_ref, f"y {pol} {launch}", depth_scale(stages))
            bufs = _buffers(work, info, (n, h, w, c))
            if pol == "SENTINEL":
                # one buffer per intermediate in each of two sets: each stage of the last run
                # checked on its own input; its tail filled the other set with the sentinel
                assert info.work_buffers == 2 * (stages - 1)
                used, other = sentinel_sets(work, info, (n, h, w, c), stages, runs=2)
                check_stagewise(x, wt, used, y, stages, f"{pol} {launch}")
                assert_all_sentinel(other, f"{pol} {launch} next set")
            else:
                # two buffers in turn: the last two intermediates remain
                assert info.work_buffers == min(2, stages - 1)
                for s in range(max(0, stages - 3), stages - 1):
                    assert_within_tol(f64(bufs[s % info.work_buffers]), hs_ref[s], f"h{s} {pol} {launch}",
                                      depth_scale(s + 2))
            b = bits(y)
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b, ref_bits), (pol, launch)


@pytest.mark.parametrize("n,h,w,c,stages", [(2, 56, 56, 64, 6), (2, 28, 28, 128, 8),
                                            (2, 14, 14, 256, 12), (2, 7, 7, 512, 6)])
def test_stack_resnet38_layer_groups(n, h, w, c, stages):
    """The four layer groups of ResNet-38 ([cuSync] Table tab:resnet-sizes: 3, 4, 6 and 3
    layers of two convolutions) at a small batch, in one persistent launch; the sentinel
    run keeps every intermediate, so each stage is also checked on its own input."""
    x, wt = synth.conv_stack_inputs(n, h, w, c, stages, seed=22)
    _, y_ref = chains.conv_stack(f64(x), [f64(wt[s]) for s in range(stages)])
    ref_bits = None
    for pol in ("ROW", "TILE", "SENTINEL"):
        d = cs.make_desc(cs.CHAIN_CONV_STACK, pol, n=n, h=h, w=w, c=c, stages=stages)
        work, y, info = run_stack(d, x, wt)
        assert_within_tol(f64(y), y_ref, f"y {pol}", depth_scale(stages))
        if pol == "SENTINEL":
            used, other = sentinel_sets(work, info, (n, h, w, c), stages, runs=1)
            check_stagewise(x, wt, used, y, stages, pol)
            assert_all_sentinel(other, "next set")
        if ref_bits is None:
            ref_bits = bits(y)
        else:
            assert np.array_equal(bits(y), ref_bits), pol


@pytest.mark.parametrize("policy", ["TILE", "SENTINEL"])
def test_stack_repeated_runs_and_graph_replay(policy):
    """Runs count up the semaphores across runs (and, under the sentinel policy, alternate
    between the two sets of intermediates, each run filling the next one's): several runs
    in a row, and runs replayed from a CUDA graph, all give the same bytes."""
    n, h, w, c, stages = 1, 14, 14, 128, 5
    x, wt = synth.conv_stack_inputs(n, h, w, c, stages, seed=23)
    d = cs.make_desc(cs.CHAIN_CONV_STACK, policy, n=n, h=h, w=w, c=c, stages=stages)
    _, y1, info = run_stack(d, x, wt, runs=1)
    work = torch.empty(info.work_bytes // 2, dtype=torch.bfloat16, device="cuda")
    y = torch.empty((n, h, w, c), dtype=torch.bfloat16, device="cuda")
    xd, wd = x.cuda(), wt.cuda()
    ch = cs.Chain(d)
    try:
        ch.run(xd, wd, None, work, y)            # direct run
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ch.run(xd, wd, None, work, y)
            ch.run(xd, wd, None, work, y)
        for _ in range(3):
            y.zero_()
            g.replay()
            st, code, _ = ch.check()
            assert st == cs.OK, f"0x{code:08x}"
            assert np.array_equal(bits(y.cpu()), bits(y1))
        y.zero_()
        ch.run(xd, wd, None, work, y)            # direct again after the replays
        st, _, _ = ch.check()
        assert st == cs.OK and np.array_equal(bits(y.cpu()), bits(y1))
        del g
    finally:
        ch.close()
