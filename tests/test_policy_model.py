"""The policy-choice latency model: the oracle's model pinned to closed forms, to the
stream waves of the pages' Table tab:waves:mlp and to invariants; the library's model
(cusync_predict_policies, the same code path CUSYNC_POLICY_AUTO uses) checked against
the oracle on MLP, SwiGLU and conv chains for every policy."""

import math

import pytest

import tile_level_sync_gb300 as cs
from oracle import planner
from oracle import policy_model as pm

from test_oracle_planner_deps import _rows

POLICY_IDX = {"STREAM": 0, "ROW": 1, "TILE": 2, "STRIDED": 3, "SENTINEL": 4}


def _model(**kw):
    base = dict(kblock_ns=(10.0, 20.0), wait_kblock_ns=3.0, sentinel_kblock_ns=50.0, start_ns=100.0,
                epilogue_ns=(30.0, 40.0), post_ns=7.0, gap_ns=500.0, fill_ns_per_mb=11.0)
    base.update(kw)
    return pm.Model(**base)


def test_stream_closed_form_one_wave():
    """Every tile has its own CTA: T = (T_init + KB0 t0 + T_epi0) + gap + (T_init + KB1 t1 + T_epi1)."""
    prod, cons, dc = pm.gemm_chain(256, 1024, 512, 256, 256, 1, "ROW")
    ch = pm.Chain(prod, cons, (8, 16), dc)
    m = _model()
    want = (100 + 8 * 10 + 30) + 500 + (100 + 16 * 20 + 40)
    assert pm.predict_stream(ch, 152, 152, m) == pytest.approx(want, rel=1e-12)


def test_stream_waves_reproduce_table_waves_mlp():
    """ALCOP's batch model with T_init = T_epilogue = 0 and one time unit per tile: a
    stream-ordered chain takes the sum of the two kernels' wave counts ([cuSync] Table
    tab:waves:mlp, "StreamSync waves")."""
    m = _model(kblock_ns=(1.0, 1.0), start_ns=0.0, epilogue_ns=(0.0, 0.0), gap_ns=0.0)
    for row in _rows("tab_waves_mlp.txt"):
        _b, g1x, g1y, g1z, _w1, g2x, g2y, g2z, _w2, sw, _cw, cap = row
        t1 = planner.grid_tbs((g1x, g1y, g1z))
        t2 = planner.grid_tbs((g2x, g2y, g2z))
        ch = pm.Chain([(0, i) for i in range(t1)], list(range(t2)), (1, 1), None)
        assert pm.predict_stream(ch, int(cap), int(cap), m) == pytest.approx(int(sw), abs=1e-12)


def test_fused_row_one_wave_closed_form():
    """All tiles resident: every consumer waits for its row, then refills and runs."""
    prod, cons, dc = pm.gemm_chain(256, 1024, 512, 256, 256, 1, "ROW")
    ch = pm.Chain(prod, cons, (8, 16), dc)
    m = _model()
    prod_done = 100 + 8 * 10 + 30
    want = prod_done + 7 + 100 + 16 * 20 + 3 + 40   # post, refill, main loop (+ the waiting k-block), epilogue
    assert pm.predict_fused(ch, "ROW", 152, m) == pytest.approx(want, rel=1e-12)


def test_fused_tile_waits_column_by_column():
    """One CTA: the queue runs producer columns 0 and 1, then the consumer, which only
    waits where a k-block needs a producer tile (none are late, so no refill)."""
    prod, cons, dc = pm.gemm_chain(128, 256, 128, 128, 128, 1, "TILE")
    ch = pm.Chain(prod, cons, (4, 4), dc)
    m = _model()
    p0 = 100 + 4 * 10
    p1 = p0 + 4 * 10
    cons_start = p1
    # k-blocks 0 and 2 start a new producer column (128 / 64 = 2 k-blocks per column)
    main_end = cons_start + 4 * 20 + 2 * 3
    last_epi = max(p1, p0 + 30) + 30          # producer epilogues queue on the CTA
    want = max(main_end, last_epi) + 40
    assert pm.predict_fused(ch, "TILE", 1, m) == pytest.approx(want, rel=1e-12)


def test_fused_prediction_grows_with_post_latency():
    prod, cons, dc = pm.gemm_chain(512, 2048, 1024, 256, 256, 1, "TILE")
    ch = pm.Chain(prod, cons, (16, 32), dc)
    prev = None
    for post in (0.0, 50.0, 500.0, 5000.0):
        t = pm.predict_fused(ch, "TILE", 8, _model(post_ns=post))
        assert prev is None or t >= prev
        prev = t
    assert pm.predict_stream(ch, 8, 8, _model(post_ns=0.0)) == pm.predict_stream(ch, 8, 8, _model(post_ns=5e3))


def _oracle_predict(desc, info, model, policy):
    n_out = info.n_out[0]
    if desc.kind == cs.CHAIN_CONV_RELU:
        prod, cons, dc = pm.conv_chain(desc.n, desc.h, desc.w, desc.c, desc.k_out, info.tile_n,
                                       info.conv_rows_per_tile)
        h_mb = desc.n * desc.h * desc.w * desc.k_out * 2 / 1e6
    else:
        prod, cons, dc = pm.gemm_chain(desc.M, desc.N1, desc.N2, info.tile_n, n_out, info.cta_pair, policy,
                                       G=info.strided_group if policy == "STRIDED" else 2, raster=info.raster_rows)
        h_mb = desc.M * desc.N1 * 2 / 1e6
    G = info.strided_group if policy == "STRIDED" else 1
    ch = pm.Chain(prod, cons, tuple(info.k_blocks), dc, G=G, h_mb=h_mb, ksplit=info.ksplit,
                  kb_per_split=info.kb_per_split, kb_skew=info.ksplit_skew)
    mo = pm.Model(kblock_ns=tuple(model.kblock_ns), wait_kblock_ns=model.wait_kblock_ns,
                  sentinel_kblock_ns=model.sentinel_kblock_ns, start_ns=model.start_ns,
                  epilogue_ns=tuple(model.epilogue_ns), post_ns=model.post_ns, gap_ns=model.gap_ns,
                  fill_ns_per_mb=model.fill_ns_per_mb, tile_ns=model.tile_ns, tile_wait_ns=model.tile_wait_ns)
    slots = info.num_sms // info.cta_pair
    units = len(prod) * info.ksplit
    if policy == "STREAM":
        return pm.predict_stream(ch, min(slots, units), min(slots, len(cons)), mo) / 1e3
    return pm.predict_fused(ch, policy, min(slots, units + len(cons)), mo) / 1e3


CASES = [
    dict(kind=cs.CHAIN_MLP_GELU, M=512, K=512, N1=1024, N2=512, tile_n=256, cta_pair=1, num_sms=24),
    dict(kind=cs.CHAIN_MLP_GELU, M=384, K=256, N1=1024, N2=768, tile_n=128, cta_pair=1, num_sms=16),
    dict(kind=cs.CHAIN_MLP_GELU, M=1024, K=256, N1=1024, N2=512, tile_n=256, cta_pair=2, num_sms=20),
    dict(kind=cs.CHAIN_MLP_SWIGLU, M=256, K=256, N1=512, N2=256, tile_n=256, cta_pair=1, num_sms=12),
    dict(kind=cs.CHAIN_CONV_RELU, n=2, h=14, w=14, c=64, k_out=256, tile_n=128, num_sms=6),
    # K split: 2 x 2 producer tiles on 16 CTAs -> 4 units each (4 k-blocks per unit)
    dict(kind=cs.CHAIN_MLP_GELU, M=256, K=1024, N1=512, N2=512, tile_n=256, cta_pair=1, num_sms=16),
    dict(kind=cs.CHAIN_MLP_GELU, M=256, K=1024, N1=512, N2=512, tile_n=256, cta_pair=1, num_sms=40, ksplit=3),
    # graded K split: units of 2, 5 and 9 k-blocks
    dict(kind=cs.CHAIN_MLP_GELU, M=256, K=1024, N1=512, N2=512, tile_n=256, cta_pair=1, num_sms=40, ksplit=3,
         ksplit_skew=3),
]


@pytest.mark.parametrize("case", CASES)
def test_library_model_matches_oracle(case):
    base = cs.make_desc(policy="ROW", **case)
    model = cs.cusync_default_latency_model(base)
    pred = cs.cusync_predict_policies(base)
    assert pred.num_sms == case["num_sms"]
    for pol, idx in POLICY_IDX.items():
        d = cs.make_desc(policy=pol, **case)
        try:
            info = cs.cusync_plan_info(d)
        except cs.CusyncError as e:
            assert pol == "STRIDED" and e.status == cs.ERR_UNSUPPORTED
            assert pred.us[idx] == -1.0
            continue
        want = _oracle_predict(d, info, model, pol)
        assert pred.us[idx] == pytest.approx(want, rel=1e-9), pol
    valid = {p: pred.us[i] for p, i in POLICY_IDX.items() if pred.us[i] >= 0}
    assert pred.best == POLICY_IDX[min(valid, key=valid.get)]
    sync = {p: v for p, v in valid.items() if p != "STREAM"}
    assert pred.best_sync == POLICY_IDX[min(sync, key=sync.get)]


def test_custom_model_is_used():
    case = CASES[0]
    d = cs.make_desc(policy="ROW", **case)
    m = cs.cusync_default_latency_model(d)
    slow = cs.cusync_default_latency_model(d)
    slow.post_ns = m.post_ns + 1e6
    a = cs.cusync_predict_policies(d, m)
    b = cs.cusync_predict_policies(d, slow)
    assert b.us[POLICY_IDX["STREAM"]] == a.us[POLICY_IDX["STREAM"]]
    assert b.us[POLICY_IDX["ROW"]] > a.us[POLICY_IDX["ROW"]] + 900.0
    assert b.best == POLICY_IDX["STREAM"]


@pytest.mark.parametrize("case", CASES)
def test_auto_policy_resolves_to_the_predicted_best(case):
    d = cs.make_desc(policy="AUTO", **case)
    info = cs.cusync_plan_info(d)
    assert info.policy == cs.cusync_predict_policies(d).best
    # the resolved plan is the plan of that policy
    d2 = cs.make_desc(policy=info.policy, **case)
    assert cs.cusync_plan_info(d2).num_flags == info.num_flags


def test_default_model_is_calibrated_per_tiling():
    gelu = cs.cusync_default_latency_model(cs.make_desc(policy="ROW", M=256, K=256, N1=512, N2=256, tile_n=256,
                                                        cta_pair=1))
    pair = cs.cusync_default_latency_model(cs.make_desc(policy="ROW", M=1024, K=256, N1=512, N2=256, tile_n=256))
    conv = cs.cusync_default_latency_model(cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", n=1, h=14, w=14, c=64,
                                                        k_out=128, tile_n=128))
    # a pair k-block covers 256 rows in less than twice a single CTA's 128-row k-block
    assert gelu.kblock_ns[0] < 2 * pair.kblock_ns[0] and pair.kblock_ns[0] < 2 * gelu.kblock_ns[0]
    assert gelu.epilogue_ns[0] > gelu.epilogue_ns[1]         # GeLU epilogue vs plain store, same width
    assert conv.epilogue_ns[0] == pytest.approx(conv.epilogue_ns[1] * 22.0 / 17.0)
    for m in (gelu, pair, conv):
        assert m.sentinel_kblock_ns > m.kblock_ns[1] and m.start_ns > 0 and m.post_ns > 0


def test_k_split_closed_form():
    """Two units of one tile on two CTAs: each runs half of the k-blocks; the second
    unit's epilogue follows the first's; the consumer refills after the post."""
    prod, cons, dc = pm.gemm_chain(128, 256, 128, 256, 256, 1, "ROW")
    ch = pm.Chain(prod, cons, (8, 4), dc, ksplit=2, kb_per_split=4)
    m = _model()
    u0 = 100 + 4 * 10 + 30
    u1 = max(100 + 4 * 10, u0) + 30
    cons_start = 100 + 4 * 10             # CTA 0 frees up first and takes the consumer tile
    want = max(u1 + 7 + 100, cons_start) + 4 * 20 + 3
    want = max(want, u0) + 40
    assert pm.predict_fused(ch, "ROW", 2, m) == pytest.approx(want, rel=1e-12)


def test_graded_k_split_closed_form():
    """Three units of one tile of 24 k-blocks graded by 4 (4, 8, 12 k-blocks) on three
    CTAs, stream order: the units form a chain, so each unit's epilogue follows its own
    mainloop and the epilogue of the unit before it; the consumer launch follows the last
    epilogue.  With equal units (8 each) every mainloop ends at once and the three
    epilogues queue behind one another, so the chain ends later."""
    prod, cons, dc = pm.gemm_chain(128, 256, 128, 256, 256, 1, "ROW")
    ch = pm.Chain(prod, cons, (24, 4), dc, ksplit=3, kb_per_split=4, kb_skew=4)
    assert [n for _, _, n in pm._units(ch)] == [4, 8, 12]
    m = _model()
    u0 = 100 + 4 * 10 + 30
    u1 = max(100 + 8 * 10, u0) + 30
    u2 = max(100 + 12 * 10, u1) + 30
    want = u2 + 500 + (100 + 4 * 20 + 40)
    assert pm.predict_stream(ch, 3, 1, m) == pytest.approx(want, rel=1e-12)
    eq = pm.Chain(prod, cons, (24, 4), dc, ksplit=3, kb_per_split=8)
    e0 = 100 + 8 * 10 + 30
    e1 = max(100 + 8 * 10, e0) + 30
    e2 = max(100 + 8 * 10, e1) + 30
    assert pm.predict_stream(eq, 3, 1, m) == pytest.approx(e2 + 500 + (100 + 4 * 20 + 40), rel=1e-12)
    assert pm.predict_stream(eq, 3, 1, m) > pm.predict_stream(ch, 3, 1, m)


def test_grouped_queue_order():
    """The oracle model's queue order with row tiles in groups (column outer, row inner
    within a group), written out by hand for 3 row tiles x 2 columns in groups of 2, and
    equal to the library's tile order for the planner's groups."""
    assert pm._grouped_rows(3, 2, 2) == [(0, 0), (1, 0), (0, 1), (1, 1), (2, 0), (2, 1)]
    assert pm._grouped_rows(2, 3, 1) == [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 2)]
    for M in (1024, 2048, 1280):
        d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, K=256, N1=1024, N2=512, cta_pair=2, num_sms=148)
        info = cs.cusync_plan_info(d)
        assert info.raster_rows == (info.m_tiles[0] // 2 if info.m_tiles[0] >= 4 else 1)
        for stage in (0, 1):
            mt, nt = info.m_tiles[stage], info.n_tiles[stage]
            lib = [cs.cusync_tile_at(d, stage, u) for u in range(mt * nt)]
            assert lib == pm._grouped_rows(mt, nt, info.raster_rows)


def test_tile_costs_closed_form():
    """tile_ns and tile_wait_ns written out by hand: one CTA, two producer tiles of 4
    k-blocks, then one consumer tile that consults a semaphore at k-blocks 0 and 2."""
    prod, cons, dc = pm.gemm_chain(128, 256, 128, 128, 128, 1, "TILE")
    ch = pm.Chain(prod, cons, (4, 4), dc)
    m = _model(tile_ns=7.0, tile_wait_ns=11.0)
    p0 = 100 + 4 * 10                          # first tile: start_ns, then its k-blocks
    p1 = p0 + 7 + 4 * 10                       # a later tile: tile_ns before its k-blocks
    cons_start = p1 + 7
    main_end = cons_start + 11 + 4 * 20 + 2 * 3   # the first consult costs tile_wait_ns once
    last_epi = max(p1, p0 + 30) + 30
    want = max(main_end, last_epi) + 40
    assert pm.predict_fused(ch, "TILE", 1, m) == pytest.approx(want, rel=1e-12)
    # stream order: each later tile of a launch pays tile_ns, no consult
    s0 = 100 + 4 * 10
    s1 = s0 + 7 + 4 * 10
    e0 = max(s1, s0 + 30) + 30
    c0 = e0 + 500 + 100 + 4 * 20               # gap_ns, then the consumer launch's first tile
    assert pm.predict_stream(ch, 1, 1, m) == pytest.approx(c0 + 40, rel=1e-12)


def test_stack_closed_form_and_pair_consistency():
    """A two-stage stack is the convolution pair: the same tiles, waits and costs; stream
    order of a stack is its stages' launches gap_ns apart."""
    prod, cons, dc = pm.conv_chain(1, 4, 4, 64, 64, 64, 4)     # one 16-pixel tile per stage
    ch = pm.Chain(prod, cons, (9, 9), dc)
    m = _model()
    for pol in ("ROW", "TILE"):
        assert pm.predict_stack(2, prod, 9, dc, pol, 1, 1, m) == pytest.approx(pm.predict_fused(ch, pol, 1, m))
    assert pm.predict_stack(2, prod, 9, dc, "STREAM", 1, 1, m) == pytest.approx(pm.predict_stream(ch, 1, 1, m))
    one = 100 + 9 * 10 + 30                    # stage 0 alone: start, k-blocks, epilogue
    later = 100 + 9 * 20 + 30
    want = one + 500 + later + 500 + (100 + 9 * 20 + 40)
    assert pm.predict_stack(3, prod, 9, dc, "STREAM", 1, 1, m) == pytest.approx(want)


STACK_CASES = [dict(n=2, h=14, w=14, c=64, stages=4, tile_n=128, num_sms=8),
               dict(n=4, h=8, w=8, c=128, stages=3, tile_n=128, num_sms=6),
               dict(n=2, h=7, w=7, c=256, stages=5, tile_n=256, num_sms=4)]


@pytest.mark.parametrize("case", STACK_CASES)
def test_library_stack_model_matches_oracle(case):
    base = cs.make_desc(cs.CHAIN_CONV_STACK, "ROW", **case)
    model = cs.cusync_default_latency_model(base)
    pred = cs.cusync_predict_policies(base)
    mo = pm.Model(kblock_ns=tuple(model.kblock_ns), wait_kblock_ns=model.wait_kblock_ns,
                  sentinel_kblock_ns=model.sentinel_kblock_ns, start_ns=model.start_ns,
                  epilogue_ns=tuple(model.epilogue_ns), post_ns=model.post_ns, gap_ns=model.gap_ns,
                  fill_ns_per_mb=model.fill_ns_per_mb, tile_ns=model.tile_ns, tile_wait_ns=model.tile_wait_ns)
    for pol, idx in POLICY_IDX.items():
        d = cs.make_desc(cs.CHAIN_CONV_STACK, pol, **case)
        try:
            info = cs.cusync_plan_info(d)
        except cs.CusyncError as e:
            assert pol == "STRIDED" and e.status == cs.ERR_UNSUPPORTED
            assert pred.us[idx] == -1.0
            continue
        tiles, _, dc = pm.conv_chain(case["n"], case["h"], case["w"], case["c"], case["c"], info.tile_n,
                                     info.conv_rows_per_tile)
        units = len(tiles)
        fill = 0
        if pol == "SENTINEL":
            chunks = (case["stages"] - 1) * case["n"] * case["h"] * case["w"] * case["c"] // 8
            fill = -(-chunks // 4096)
        want = pm.predict_stack(case["stages"], tiles, info.k_blocks[0], dc, pol,
                                min(case["num_sms"], units * case["stages"]), min(case["num_sms"], units), mo,
                                fill_units=fill) / 1e3
        assert pred.us[idx] == pytest.approx(want, rel=1e-9), pol
