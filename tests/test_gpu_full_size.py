"""GPU parity at the full sizes of every benchmarked configuration, with the planner's
default tiling (CTA pairs, K split, L2 prefetch as it chooses them); the self-attention
shard and the four ResNet-38 convolution stacks are at the end of the file:

* the GPT-3-shaped MLP slice X[M,12288] . W1[12288,6144] -> GeLU -> . W2[6144,12288]
  for M in {256, 512, 1024, 2048, 4096} ("A Framework for Fine-Grained Synchronization
  of Dependent GPU Kernels", §II-B and Table tab:waves:mlp, which measures every batch
  size);
* the SwiGLU MLP X[M,8192] . [Wgate|Wup][8192,2x3584] -> silu(g)*u -> . Wdown[3584,8192]
  for M in {256, 1024};
* the ResNet-style convolution pair on 32 NHWC images of 14x14x256 (Table
  tab:resnet-sizes), conv3x3 -> ReLU -> conv3x3.

Every policy under both launch forms (one persistent kernel, programmatic dependent
launch) and the stream-serialised chain must give byte-identical H and Y over the whole
tensors, and those bytes must match the oracle within |err| <= 2e-2 max(1, |ref|) on
sampled rows: the first and last token row of every 256-row tile (convolutions: the
first, a middle and the last image).  Each chain object runs twice, so the second run
waits on semaphores that count on from the first.
"""

import numpy as np
import pytest
import torch

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth

from gpu_helpers import assert_within_tol, f64

pytestmark = pytest.mark.gpu

VARIANTS = [("STREAM", cs.LAUNCH_PERSISTENT)] + [
    (pol, launch) for pol in ("ROW", "TILE", "STRIDED", "SENTINEL") for launch in (cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL)]

FULL_SIZE = ["gpt3_mlp_m256", "gpt3_mlp_m512", "gpt3_mlp_m1024", "gpt3_mlp_m2048", "gpt3_mlp_m4096",
             "swiglu_m256", "swiglu_m1024", "conv_resnet14_n32"]


def _operands(wl, inputs):
    """Device operands in the library's layout, the chain base descriptor, and the shapes of
    H and Y."""
    d = wl.dims
    if wl.kind == "conv_relu":
        x, w1, w2 = inputs
        base = dict(kind=cs.CHAIN_CONV_RELU, n=d["N"], h=d["H"], w=d["W"], c=d["C"], k_out=d["K"])
        shape = (d["N"], d["H"], d["W"], d["K"])
        return (x.cuda(), w1.contiguous().cuda(), w2.contiguous().cuda()), base, shape, shape
    if wl.kind == "mlp_gelu":
        X, W1, W2 = inputs
        W1t = W1.t().contiguous()
        kind = cs.CHAIN_MLP_GELU
    else:
        X, Wg, Wu, W2 = inputs
        W1t = torch.cat([Wg.t(), Wu.t()], 0).contiguous()
        kind = cs.CHAIN_MLP_SWIGLU
    base = dict(kind=kind, M=d["M"], K=d["K"], N1=d["N1"], N2=d["N2"])
    return (X.cuda(), W1t.cuda(), W2.t().contiguous().cuda()), base, (d["M"], d["N1"]), (d["M"], d["N2"])


def _sample_rows(M):
    rows = set()
    for t0 in range(0, M, 256):
        rows.add(t0)
        rows.add(min(t0 + 255, M - 1))
    return sorted(rows)


def _oracle_check(wl, inputs, H, Y):
    d = wl.dims
    if wl.kind == "conv_relu":
        x, w1, w2 = inputs
        imgs = [0, d["N"] // 2, d["N"] - 1]
        H_ref, Y_ref = chains.conv_relu_chain(f64(x[imgs]), f64(w1), f64(w2))
        assert_within_tol(f64(H[imgs].cpu()), H_ref, f"{wl.name} y1 images {imgs}")
        assert_within_tol(f64(Y[imgs].cpu()), Y_ref, f"{wl.name} y2 images {imgs}")
        return
    rows = _sample_rows(d["M"])
    idx = torch.tensor(rows)
    if wl.kind == "mlp_gelu":
        X, W1, W2 = inputs
        H_ref, Y_ref = chains.mlp_gelu(f64(X[idx]), f64(W1), f64(W2))
    else:
        X, Wg, Wu, Wd = inputs
        H_ref, Y_ref = chains.mlp_swiglu(f64(X[idx]), f64(Wg), f64(Wu), f64(Wd))
    assert_within_tol(f64(H[idx.cuda()].cpu()), H_ref, f"{wl.name} H rows {len(rows)}")
    assert_within_tol(f64(Y[idx.cuda()].cpu()), Y_ref, f"{wl.name} Y rows {len(rows)}")


@pytest.mark.parametrize("name", FULL_SIZE)
def test_full_size_every_policy_bit_identical_and_within_oracle(name):
    wl = synth.WORKLOADS[name]
    inputs = synth.workload_inputs(wl, seed=0)
    ops, base, h_shape, y_shape = _operands(wl, inputs)
    H = torch.empty(h_shape, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(y_shape, dtype=torch.bfloat16, device="cuda")
    ref = None
    ran = []
    for pol, launch in VARIANTS:
        desc = cs.make_desc(policy=pol, launch=launch, **base)
        try:
            cs.cusync_plan_info(desc)
        except cs.CusyncError as e:   # StridedSync needs a column-tile count divisible by G
            assert pol == "STRIDED" and e.status == cs.ERR_UNSUPPORTED, (pol, e)
            continue
        H.fill_(float("nan"))
        Y.fill_(float("nan"))
        ch = cs.Chain(desc)
        try:
            for _ in range(2):
                ch.run(*ops, H, Y)
            st, code, detail = ch.check()
        finally:
            ch.close()
        what = f"{name} {pol} {'pdl' if launch == cs.LAUNCH_PDL else 'persistent'}"
        assert st == cs.OK, f"{what}: {cs.status_string(st)} code=0x{code:08x} detail=0x{detail:x}"
        hb, yb = H.view(torch.int16), Y.view(torch.int16)
        if ref is None:
            ref = (hb.clone(), yb.clone())
        else:
            assert torch.equal(hb, ref[0]), f"{what}: H differs from {ran[0]}"
            assert torch.equal(yb, ref[1]), f"{what}: Y differs from {ran[0]}"
        ran.append(what)
    assert len(ran) >= 7, ran
    _oracle_check(wl, inputs, ref[0].view(torch.bfloat16), ref[1].view(torch.bfloat16))


ATTN_VARIANTS = [("STREAM", cs.LAUNCH_PERSISTENT)] + [
    (pol, launch) for pol in ("ROW", "TILE", "STRIDED") for launch in (cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL)]


@pytest.mark.parametrize("name", ["gpt3_attn_m256", "gpt3_attn_m1024"])
def test_full_size_attention_every_policy_bit_identical_and_within_oracle(name):
    """The GPT-3 self-attention shard at its benchmarked sizes (X[M,12288] . QKV[12288,
    3x1536] -> per-head softmax(XQ * XV) * XK -> . W2[1536,12288]; "A Framework for
    Fine-Grained Synchronization of Dependent GPU Kernels", Fig. fig:gpt-3:attention)
    with the planner's defaults (CTA pairs, the graded K split of the QKV GEMM at M=256):
    every policy and launch form and the three stream-ordered kernels give byte-identical
    XQKV, XDot and Y, and the oracle matches them on sampled token rows."""
    wl = synth.WORKLOADS[name]
    d = wl.dims
    M, N1, N2 = d["M"], d["N1"], d["N2"]
    X, Wqkv, W2 = synth.workload_inputs(wl, seed=0)
    ops = (X.cuda(), Wqkv.t().contiguous().cuda(), W2.t().contiguous().cuda())
    xqkv = torch.empty((M, 3 * N1), dtype=torch.bfloat16, device="cuda")
    xdot = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    ref = None
    for pol, launch in ATTN_VARIANTS:
        ch = cs.Chain(cs.make_desc(cs.CHAIN_ATTENTION, pol, launch, M=M, K=d["K"], N1=N1, N2=N2))
        try:
            for _ in range(2):
                xqkv.fill_(float("nan"))
                xdot.fill_(float("nan"))
                y.fill_(float("nan"))
                ch.run(ops[0], ops[1], ops[2], xqkv, y, h2=xdot)
            st, code, detail = ch.check()
            assert st == cs.OK, f"{name} {pol} {launch}: {cs.status_string(st)} 0x{code:08x} 0x{detail:x}"
        finally:
            ch.close()
        got = (xqkv.view(torch.int16).clone(), xdot.view(torch.int16).clone(), y.view(torch.int16).clone())
        if ref is None:
            ref = got
        else:
            assert all(torch.equal(u, v) for u, v in zip(got, ref)), f"{name} {pol} {launch} differs"
    rows = _sample_rows(M)
    q_ref, d_ref, y_ref = chains.attention_rows(f64(X), f64(Wqkv), f64(W2), rows)
    idx = torch.tensor(rows, device="cuda")
    assert_within_tol(f64(xqkv[idx].cpu()), q_ref, f"{name} XQKV rows {len(rows)}")
    assert_within_tol(f64(xdot[idx].cpu()), d_ref, f"{name} XDot rows {len(rows)}")
    assert_within_tol(f64(y[idx].cpu()), y_ref, f"{name} Y rows {len(rows)}")


STACKS = ["resnet38_56x56x64_n32", "resnet38_28x28x128_n32", "resnet38_14x14x256_n32", "resnet38_7x7x512_n32"]


@pytest.mark.parametrize("name", STACKS)
def test_full_size_stack_every_policy_bit_identical_and_within_oracle(name):
    """The four ResNet-38 layer groups at the benchmarked batch of 32 images ("A Framework
    for Fine-Grained Synchronization of Dependent GPU Kernels", Table tab:resnet-sizes),
    each a stack of dependent 3x3 convolutions in one chain: every policy and launch form
    and the stream-ordered stages give a byte-identical output, and the oracle matches it
    on the first, a middle and the last image (with the stack's depth-scaled bound)."""
    from test_gpu_stack import depth_scale
    wl = synth.WORKLOADS[name]
    d = wl.dims
    n, h, w, c, S = d["N"], d["H"], d["W"], d["C"], d["S"]
    x, wt = synth.workload_inputs(wl, seed=0)
    xd, wd = x.cuda(), wt.contiguous().cuda()
    y = torch.empty((n, h, w, c), dtype=torch.bfloat16, device="cuda")
    ref = None
    for pol, launch in [("STREAM", cs.LAUNCH_PERSISTENT)] + [
            (p, l) for p in ("ROW", "TILE", "SENTINEL") for l in (cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL)]:
        desc = cs.make_desc(cs.CHAIN_CONV_STACK, pol, launch, n=n, h=h, w=w, c=c, stages=S)
        info = cs.cusync_plan_info(desc)
        work = torch.empty(info.work_bytes // 2, dtype=torch.bfloat16, device="cuda")
        ch = cs.Chain(desc)
        try:
            for _ in range(2):
                y.fill_(float("nan"))
                ch.run(xd, wd, None, work, y)
            st, code, detail = ch.check()
            assert st == cs.OK, f"{name} {pol} {launch}: {cs.status_string(st)} 0x{code:08x} 0x{detail:x}"
        finally:
            ch.close()
        got = y.view(torch.int16).clone()
        if ref is None:
            ref = got
        else:
            assert torch.equal(got, ref), f"{name} {pol} {launch} differs"
        del work
    imgs = [0, n // 2, n - 1]
    _, y_ref = chains.conv_stack(f64(x[imgs]), [f64(wt[s]) for s in range(S)])
    assert_within_tol(f64(y[imgs].cpu()), y_ref, f"{name} images {imgs}", depth_scale(S))
