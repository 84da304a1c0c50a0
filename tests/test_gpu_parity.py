"""GPU parity: every chain, policy and launch mode against the oracle, element by element,
on seeded inputs; byte identity of H and Y across policies and the stream-serialised
baseline; device waits that expire report a status instead of hanging."""

import numpy as np
import pytest
import torch

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth

from gpu_helpers import assert_within_tol, bits, device_mlp_operands, f64, run_conv, run_mlp

pytestmark = pytest.mark.gpu

POLICIES = ["STREAM", "ROW", "TILE", "STRIDED", "SENTINEL"]
LAUNCHES = [cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL]


def _mlp_case(M, K, N1, N2, seed=0):
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed)
    H_ref, Y_ref = chains.mlp_gelu(f64(X), f64(W1), f64(W2))
    return (X, W1, W2), (H_ref, Y_ref)


@pytest.mark.parametrize("tile_n", [256, 128])
@pytest.mark.parametrize("pair", [1, 2])
def test_tiny_mlp_all_policies_bit_identical(tile_n, pair):
    """64x256 . 256x1024 . 1024x256 (the tiny MLP configuration)."""
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(64, 256, 1024, 256)
    ops = device_mlp_operands(X, W1, W2)
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=64, K=256, N1=1024, N2=256, tile_n=tile_n,
                             cta_pair=pair)
            H, Y, _ = run_mlp(d, *ops, runs=2)
            assert_within_tol(f64(H), H_ref, f"H {pol} {launch}")
            assert_within_tol(f64(Y), Y_ref, f"Y {pol} {launch}")
            b = (bits(H), bits(Y))
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), (pol, launch)


@pytest.mark.parametrize("M,K,N1,N2,tile_n", [
    (200, 384, 640, 264, 256),     # ragged M, N1 (H columns) and N2
    (384, 1024, 2048, 1024, 128),  # several row and column tiles, longer K
    (1, 64, 512, 128, 256),        # a single token
    (520, 512, 1536, 512, 256),    # more tiles than a persistent CTA's ring holds
    (264, 200, 512, 256, 256),     # K not a whole number of k-blocks: 2-D copies inside two-k-block stages
    (136, 320, 768, 200, 128),     # an odd k-block count: a pair's last stage holds one k-block of its box
])
@pytest.mark.parametrize("pair", [1, 2])
def test_mlp_shapes_all_policies(M, K, N1, N2, tile_n, pair):
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(M, K, N1, N2, seed=1)
    ops = device_mlp_operands(X, W1, W2)
    ref_bits = None
    for pol in POLICIES:
        d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, cs.LAUNCH_PERSISTENT, M=M, K=K, N1=N1, N2=N2, tile_n=tile_n,
                         cta_pair=pair)
        try:
            cs.cusync_plan_info(d)
        except cs.CusyncError as e:   # StridedSync needs a column-tile count divisible by G
            assert pol == "STRIDED" and e.status == cs.ERR_UNSUPPORTED
            continue
        H, Y, _ = run_mlp(d, *ops, runs=3)
        assert_within_tol(f64(H), H_ref, f"H {pol}")
        assert_within_tol(f64(Y), Y_ref, f"Y {pol}")
        b = (bits(H), bits(Y))
        if ref_bits is None:
            ref_bits = b
        else:
            assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), pol


def test_intermediate_never_holds_negative_zero():
    (X, W1, W2), _ = _mlp_case(256, 512, 1024, 256, seed=2)
    ops = device_mlp_operands(X, W1, W2)
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "SENTINEL", M=256, K=512, N1=1024, N2=256)
    H, _, _ = run_mlp(d, *ops)
    assert not np.any(bits(H).view(np.uint16) == 0x8000)


@pytest.mark.parametrize("M,K,N1,N2,tile_n", [(64, 256, 512, 256, 256), (200, 512, 384, 264, 256),
                                               (130, 256, 640, 128, 128)])
@pytest.mark.parametrize("pair", [1, 2])
def test_swiglu_all_policies(M, K, N1, N2, tile_n, pair):
    X, Wg, Wu, Wd = synth.mlp_swiglu_inputs(M, K, N1, N2, seed=3)
    H_ref, Y_ref = chains.mlp_swiglu(f64(X), f64(Wg), f64(Wu), f64(Wd))
    ops = device_mlp_operands(X, Wg, Wd, Wup=Wu)
    ref_bits = None
    for pol in POLICIES:
        d = cs.make_desc(cs.CHAIN_MLP_SWIGLU, pol, cs.LAUNCH_PERSISTENT, M=M, K=K, N1=N1, N2=N2, tile_n=tile_n,
                         cta_pair=pair)
        try:
            cs.cusync_plan_info(d)
        except cs.CusyncError as e:
            assert pol == "STRIDED" and e.status == cs.ERR_UNSUPPORTED
            continue
        H, Y, _ = run_mlp(d, *ops, runs=2)
        assert_within_tol(f64(H), H_ref, f"H {pol}")
        assert_within_tol(f64(Y), Y_ref, f"Y {pol}")
        b = (bits(H), bits(Y))
        if ref_bits is None:
            ref_bits = b
        else:
            assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), pol


@pytest.mark.parametrize("n,h,w,c,k,tile_n", [(2, 14, 14, 128, 128, 128), (3, 14, 14, 64, 256, 256),
                                              (2, 9, 30, 64, 128, 128), (1, 5, 100, 128, 64, 128)])
def test_conv_chain_all_policies(n, h, w, c, k, tile_n):
    x, w1, w2 = synth.conv_inputs(n, h, w, c, k, seed=4)
    H_ref, Y_ref = chains.conv_relu_chain(f64(x), f64(w1), f64(w2))
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_CONV_RELU, pol, launch, n=n, h=h, w=w, c=c, k_out=k, tile_n=tile_n)
            try:
                cs.cusync_plan_info(d)
            except cs.CusyncError as e:
                assert pol == "STRIDED" and e.status == cs.ERR_UNSUPPORTED
                continue
            y1, y2, _ = run_conv(d, x, w1, w2, runs=2)
            assert_within_tol(f64(y1), H_ref, f"y1 {pol} {launch}")
            assert_within_tol(f64(y2), Y_ref, f"y2 {pol} {launch}")
            b = (bits(y1), bits(y2))
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), (pol, launch)


def test_skipped_post_times_out_and_recovers():
    """A producer tile that never posts makes the consumer's bounded wait expire: the run
    reports CUSYNC_ERR_TIMEOUT (no hang, no trap), and the chain works again afterwards."""
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(256, 256, 1024, 256, seed=5)
    ops = device_mlp_operands(X, W1, W2)
    for pol in ("ROW", "TILE"):
        d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, M=256, K=256, N1=1024, N2=256, flags=cs.DEBUG_SKIP_POST,
                         timeout_ns=20_000_000)
        _, _, st = run_mlp(d, *ops, check=False)
        assert st == cs.ERR_TIMEOUT
        d.flags = 0
        H, Y, st = run_mlp(d, *ops)
        assert_within_tol(f64(Y), Y_ref, f"Y after timeout {pol}")
    # the same chain object, across the failure
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "TILE", M=256, K=256, N1=1024, N2=256, flags=cs.DEBUG_SKIP_POST,
                     timeout_ns=20_000_000)
    ch = cs.Chain(d)
    Hd = torch.empty((256, 1024), dtype=torch.bfloat16, device="cuda")
    Yd = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
    ch.run(*ops, Hd, Yd)
    st, code, detail = ch.check()
    assert st == cs.ERR_TIMEOUT and (code >> 24) == 1
    ch.close()


def test_withheld_split_sums_time_out_and_recover():
    """K split: a unit whose partial sums never arrive makes the next unit's bounded read of
    its workspace slot expire.  The run reports CUSYNC_ERR_TIMEOUT (no hang, no trap), again
    after cusync_chain_check's reset, and a chain without the fault computes the right
    result."""
    M, K, N1, N2 = 264, 2048, 1024, 512
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(M, K, N1, N2, seed=8)
    ops = device_mlp_operands(X, W1, W2)
    for pol, ks in (("ROW", 3), ("STREAM", 2)):
        d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, M=M, K=K, N1=N1, N2=N2, tile_n=256, ksplit=ks,
                         flags=cs.DEBUG_SKIP_SPLIT, timeout_ns=20_000_000)
        ch = cs.Chain(d)
        try:
            Hd = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
            Yd = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
            for _ in range(2):  # the chain stays usable: the same failure, reported the same way
                ch.run(*ops, Hd, Yd)
                st, code, detail = ch.check()
                # (the first wait to expire may be a consumer's on the semaphore that the
                # stalled tile never posts: the same class, a semaphore or slot timeout)
                assert st == cs.ERR_TIMEOUT and (code >> 24) == 1, (pol, st, hex(code), hex(detail))
        finally:
            ch.close()
        d.flags = 0
        H, Y, st = run_mlp(d, *ops, runs=2)
        assert_within_tol(f64(H), H_ref, f"H after split timeout {pol}")
        assert_within_tol(f64(Y), Y_ref, f"Y after split timeout {pol}")


def test_invalid_pointers_rejected():
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=64, K=256, N1=1024, N2=256)
    ch = cs.Chain(d)
    try:
        t = torch.empty(64 * 1024 + 8, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(cs.CusyncError) as e:
            ch.run(t.data_ptr() + 2, t, t, t, t)   # misaligned
        assert e.value.status == cs.ERR_INVALID_ARG
        with pytest.raises(cs.CusyncError) as e:
            ch.run(0, t, t, t, t)
        assert e.value.status == cs.ERR_INVALID_ARG
    finally:
        ch.close()


def test_tile_order_and_prefetch_do_not_change_results():
    """The raster group size and the L2 prefetch distance only change when and in which
    order tiles are computed, never a byte of H or Y."""
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(520, 512, 1536, 512, seed=6)
    ops = device_mlp_operands(X, W1, W2)
    ref = None
    for pol in ("STREAM", "ROW", "TILE"):
        for raster, pf in ((1, -1), (3, 8), (16, 2), (16, -1)):
            d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, M=520, K=512, N1=1536, N2=512, tile_n=256,
                             raster_rows=raster, l2_prefetch=pf)
            H, Y, _ = run_mlp(d, *ops, runs=2)
            b = (bits(H), bits(Y))
            if ref is None:
                assert_within_tol(f64(Y), Y_ref, "Y")
                ref = b
            assert np.array_equal(b[0], ref[0]) and np.array_equal(b[1], ref[1]), (pol, raster, pf)


def test_auto_policy_runs_the_predicted_policy():
    """CUSYNC_POLICY_AUTO creates the chain with the policy the latency model predicts
    fastest; its output is byte-identical to that policy's."""
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(520, 512, 1536, 512, seed=7)
    ops = device_mlp_operands(X, W1, W2)
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "AUTO", M=520, K=512, N1=1536, N2=512)
    chosen = cs.cusync_plan_info(d).policy
    assert chosen == cs.cusync_predict_policies(d).best
    H, Y, _ = run_mlp(d, *ops, runs=2)
    assert_within_tol(f64(Y), Y_ref, "Y auto")
    d2 = cs.make_desc(cs.CHAIN_MLP_GELU, chosen, M=520, K=512, N1=1536, N2=512)
    H2, Y2, _ = run_mlp(d2, *ops, runs=1)
    assert np.array_equal(bits(Y), bits(Y2)) and np.array_equal(bits(H), bits(H2))


def test_many_tiles_all_policies():
    """A long token dimension with small weights: 128 row tiles of 256 tokens and 256
    producer plus 256 consumer pair tiles, several waves of the persistent queue, row
    tiles taken in groups of 64 (half of them): every policy and launch mode byte-identical,
    the oracle on the first and last row of every tile."""
    M, K, N1, N2 = 32768, 256, 512, 512
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=27)
    ops = device_mlp_operands(X, W1, W2)
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2)
            info = cs.cusync_plan_info(d)
            assert info.cta_pair == 2 and info.m_tiles[0] == 128 and info.raster_rows == 64
            H, Y, _ = run_mlp(d, *ops, runs=2)
            b = (bits(H), bits(Y))
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), (pol, launch)
    rows = sorted({r for t0 in range(0, M, 256) for r in (t0, t0 + 255)})
    H_ref, Y_ref = chains.mlp_gelu(f64(X[rows]), f64(W1), f64(W2))
    assert_within_tol(f64(H[rows]), H_ref, "H sampled rows")
    assert_within_tol(f64(Y[rows]), Y_ref, "Y sampled rows")


@pytest.mark.parametrize("ksplit,skew", [(3, 3), (2, 6), (4, 2)])
@pytest.mark.parametrize("pair", [1, 2])
def test_graded_k_split_all_policies(ksplit, skew, pair):
    """Producer units of growing length (ksplit_skew; e.g. 7, 10 and 15 of 32 k-blocks):
    every policy and launch mode within tolerance of the oracle and byte-identical to one
    another."""
    M, K, N1, N2 = 264, 2048, 1024, 512
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(M, K, N1, N2, seed=18)
    ops = device_mlp_operands(X, W1, W2)
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2, tile_n=256, cta_pair=pair,
                             ksplit=ksplit, ksplit_skew=skew)
            info = cs.cusync_plan_info(d)
            assert (info.ksplit, info.ksplit_skew) == (ksplit, skew)
            H, Y, _ = run_mlp(d, *ops, runs=3)
            assert_within_tol(f64(H), H_ref, f"H {pol} {launch} ksplit={ksplit} skew={skew}")
            assert_within_tol(f64(Y), Y_ref, f"Y {pol} {launch} ksplit={ksplit} skew={skew}")
            b = (bits(H), bits(Y))
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), (pol, launch)


@pytest.mark.parametrize("ksplit", [0, 2, 3, 5])
@pytest.mark.parametrize("pair", [1, 2])
def test_k_split_producer_all_policies(ksplit, pair):
    """Producer tiles computed as K-split units (partial sums added in unit order by the
    tile's units, the last one applying GeLU and posting): every policy and launch mode
    within tolerance of the oracle and byte-identical to one another; ksplit 0 lets the
    planner choose (2 here)."""
    M, K, N1, N2 = 264, 2048, 1024, 512
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(M, K, N1, N2, seed=8)
    ops = device_mlp_operands(X, W1, W2)
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2, tile_n=256, cta_pair=pair,
                             ksplit=ksplit)
            assert cs.cusync_plan_info(d).ksplit == (ksplit or 2)
            H, Y, _ = run_mlp(d, *ops, runs=3)
            assert_within_tol(f64(H), H_ref, f"H {pol} {launch} ksplit={ksplit}")
            assert_within_tol(f64(Y), Y_ref, f"Y {pol} {launch} ksplit={ksplit}")
            b = (bits(H), bits(Y))
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), (pol, launch)


@pytest.mark.parametrize("ks,ks_prod,pair", [(2, 1, 1), (3, 2, 1), (3, 1, 2), (4, 2, 2)])
def test_k_split_consumer_all_policies(ks, ks_prod, pair):
    """Consumer tiles computed as K-split units, each waiting from its own first k-block
    for what it reads (StridedSync groups included): every policy and launch mode within
    tolerance of the oracle and byte-identical to one another; with a split producer too."""
    M, K, N1, N2 = 300, 1024, 2048, 512
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(M, K, N1, N2, seed=12)
    ops = device_mlp_operands(X, W1, W2)
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2, tile_n=256, cta_pair=pair,
                             ksplit=ks_prod, ksplit_consumer=ks)
            info = cs.cusync_plan_info(d)
            assert info.ksplit_consumer == ks and info.ksplit == ks_prod
            H, Y, _ = run_mlp(d, *ops, runs=3)
            assert_within_tol(f64(H), H_ref, f"H {pol} {launch}")
            assert_within_tol(f64(Y), Y_ref, f"Y {pol} {launch}")
            b = (bits(H), bits(Y))
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), (pol, launch)


def test_k_split_swiglu():
    M, K, N1, N2 = 200, 1024, 512, 256
    X, Wg, Wu, Wd = synth.mlp_swiglu_inputs(M, K, N1, N2, seed=9)
    H_ref, Y_ref = chains.mlp_swiglu(f64(X), f64(Wg), f64(Wu), f64(Wd))
    ops = device_mlp_operands(X, Wg, Wd, Wup=Wu)
    ref = None
    for pol in ("STREAM", "ROW", "TILE", "SENTINEL"):
        d = cs.make_desc(cs.CHAIN_MLP_SWIGLU, pol, M=M, K=K, N1=N1, N2=N2, tile_n=256, ksplit=3)
        H, Y, _ = run_mlp(d, *ops, runs=2)
        assert_within_tol(f64(H), H_ref, f"H {pol}")
        assert_within_tol(f64(Y), Y_ref, f"Y {pol}")
        b = (bits(H), bits(Y))
        ref = ref or b
        assert np.array_equal(b[0], ref[0]) and np.array_equal(b[1], ref[1]), pol


@pytest.mark.parametrize("M,K,N1,N2,ksplit,ksplit_consumer", [
    (256, 1024, 1152, 768, 0, 0),    # the planner's K split
    (520, 512, 1536, 512, 1, 0),     # several row tiles, ragged M
    (300, 384, 1000, 264, 1, 0),     # ragged N1 (the last producer tile is partly outside H) and N2
    (264, 2048, 1152, 512, 3, 2),    # K-split producer and consumer
])
def test_192_wide_pair_tiles_all_policies(M, K, N1, N2, ksplit, ksplit_consumer):
    """256 x 192 tiles on CTA pairs (the accumulators 256 TMEM columns apart, three
    64-column store boxes per tile, a consumer k-block reading producer column tile
    kb*64/192): every policy and launch mode within tolerance of the oracle and
    byte-identical to one another."""
    (X, W1, W2), (H_ref, Y_ref) = _mlp_case(M, K, N1, N2, seed=13)
    ops = device_mlp_operands(X, W1, W2)
    ref_bits = None
    for pol in POLICIES:
        for launch in LAUNCHES:
            if pol == "STREAM" and launch != cs.LAUNCH_PERSISTENT:
                continue
            d = cs.make_desc(cs.CHAIN_MLP_GELU, pol, launch, M=M, K=K, N1=N1, N2=N2, tile_n=192, cta_pair=2,
                             ksplit=ksplit, ksplit_consumer=ksplit_consumer)
            try:
                info = cs.cusync_plan_info(d)
            except cs.CusyncError as e:
                assert pol == "STRIDED" and e.status == cs.ERR_UNSUPPORTED
                continue
            assert info.tile_n == 192 and info.cta_pair == 2
            H, Y, _ = run_mlp(d, *ops, runs=3)
            assert_within_tol(f64(H), H_ref, f"H {pol} {launch}")
            assert_within_tol(f64(Y), Y_ref, f"Y {pol} {launch}")
            b = (bits(H), bits(Y))
            if ref_bits is None:
                ref_bits = b
            else:
                assert np.array_equal(b[0], ref_bits[0]) and np.array_equal(b[1], ref_bits[1]), (pol, launch)


def test_192_wide_tiles_only_for_gelu_pairs():
    for kw in (dict(kind=cs.CHAIN_MLP_GELU, cta_pair=1), dict(kind=cs.CHAIN_MLP_SWIGLU, cta_pair=2)):
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_plan_info(cs.make_desc(policy="ROW", M=256, K=512, N1=1152, N2=256, tile_n=192, **kw))
        assert e.value.status == cs.ERR_UNSUPPORTED
