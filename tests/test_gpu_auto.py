"""GPU check of the policy-choice model against measurement ("A Framework for Fine-Grained
Synchronization of Dependent GPU Kernels", §VI-B: no one policy is best for every shape).

On the ResNet-38 layer groups run as convolution stacks (Table tab:resnet-sizes), the
latency model's ranking of the stream-serialised chain against its best tile-synchronised
policy must agree with measurement wherever the measured difference is clear: the
56x56x64 group, whose 896 nine-k-block tiles per convolution pay a consult of the
semaphores each and leave little wave tail to fill, runs faster in stream order, and
CUSYNC_POLICY_AUTO must choose stream order there; the 28x28x128 group gains from
fusing."""

import statistics

import pytest
import torch

import tile_level_sync_gb300 as cs
from tile_level_sync_gb300 import synth

pytestmark = pytest.mark.gpu

NAMES = ["STREAM", "ROW", "TILE", "STRIDED", "SENTINEL"]
STACKS = [("56x56x64", dict(n=32, h=56, w=56, c=64, stages=6, tile_n=128), "STREAM"),
          ("28x28x128", dict(n=32, h=28, w=28, c=128, stages=8, tile_n=128), "SYNC")]


def _time_us(desc, ops, runs=20, rounds=5):
    ch = cs.Chain(desc)
    x, w, work, y = ops
    try:
        for _ in range(3):
            ch.run(x, w, None, work, y)
        st, code, _ = ch.check()
        assert st == cs.OK, hex(code)
        s = torch.cuda.current_stream()
        out = []
        for _ in range(rounds):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(s)
            for _ in range(runs):
                ch.run(x, w, None, work, y)
            e1.record(s)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) * 1e3 / runs)
        st, code, _ = ch.check()
        assert st == cs.OK, hex(code)
        return statistics.median(out)
    finally:
        ch.close()


@pytest.mark.parametrize("name,dims,winner", STACKS)
def test_model_ranks_stream_against_fused_as_measured(name, dims, winner):
    n, h, w, c, S = dims["n"], dims["h"], dims["w"], dims["c"], dims["stages"]
    x, wt = synth.conv_stack_inputs(n, h, w, c, S, seed=0)
    ops = (x.cuda(), wt.contiguous().cuda(),
           torch.empty((2 * (S - 1) * n * h * w * c,), dtype=torch.bfloat16, device="cuda"),
           torch.empty((n, h, w, c), dtype=torch.bfloat16, device="cuda"))
    base = dict(kind=cs.CHAIN_CONV_STACK, **dims)
    pred = cs.cusync_predict_policies(cs.make_desc(policy="ROW", **base))
    sync = NAMES[pred.best_sync]
    t_stream = _time_us(cs.make_desc(policy="STREAM", **base), ops)
    t_sync = _time_us(cs.make_desc(policy=sync, **base), ops)
    ratio = t_stream / t_sync
    # the measured difference is clear for these groups, and the model ranks them the same
    assert abs(ratio - 1.0) > 0.05, (name, t_stream, t_sync)
    assert (pred.us[0] < pred.us[pred.best_sync]) == (t_stream < t_sync), (name, list(pred.us), t_stream, t_sync)
    assert (winner == "STREAM") == (t_stream < t_sync), (name, t_stream, t_sync)
    auto = cs.cusync_plan_info(cs.make_desc(policy="AUTO", **base)).policy
    assert (auto == cs.POLICY_STREAM) == (winner == "STREAM"), (name, auto)
