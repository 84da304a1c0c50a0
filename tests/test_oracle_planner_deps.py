"""Pins of the oracle's wave arithmetic (against the tables and worked examples printed in
[cuSync]), of its dependency sets (closed forms and policy invariants) and of the
sentinel example's expected output."""

import math
import os

import numpy as np
import pytest

from oracle import deps, planner, sentinel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_tab_intro():
    for batch, _gemm, gx, gy, gz, occ, w, util in _rows("tab_intro.txt"):
        tbs = planner.grid_tbs((gx, gy, gz))
        cap = planner.wave_capacity(int(occ), 80)
        assert cap == 160
        assert planner.fractional_waves(tbs, cap) == pytest.approx(float(w), abs=1e-12)
        assert round(100 * planner.utilisation(tbs, cap)) == int(util)


def test_tab_waves_mlp():
    for row in _rows("tab_waves_mlp.txt"):
        _b, g1x, g1y, g1z, w1, g2x, g2y, g2z, w2, sw, cw, cap = row
        t1 = planner.grid_tbs((g1x, g1y, g1z))
        t2 = planner.grid_tbs((g2x, g2y, g2z))
        cw_ = planner.chain_waves([t1, t2], int(cap))
        assert cw_.waves_frac[0] == pytest.approx(float(w1), abs=1e-12)
        assert cw_.waves_frac[1] == pytest.approx(float(w2), abs=1e-12)
        assert cw_.stream_waves == int(sw)
        assert cw_.fused_waves_frac == pytest.approx(float(cw), abs=1e-12)


def test_tab_waves_conv128():
    pinned = 0
    for B, gx, conv_w, sw, cw, ok in _rows("tab_waves_conv128.txt"):
        B, gx = int(B), int(gx)
        assert math.ceil(B * 28 * 28 / 64) == gx           # 64-pixel M tiles
        if ok != "yes":
            continue
        pinned += 1
        c = planner.chain_waves([gx, gx], 160)
        # printed to two digits (rounded or truncated)
        assert abs(c.waves_frac[0] - float(conv_w)) < 0.01
        assert abs(c.fused_waves_frac - float(cw)) < 0.015
        assert c.stream_waves == int(sw)
    assert pinned == 7


def test_worked_examples():
    for name, t1, t2, occ, sms, sw, fw, last, _src in _rows("worked_examples.txt"):
        c = planner.chain_waves([int(t1), int(t2)], planner.wave_capacity(int(occ), int(sms)))
        assert c.stream_waves == int(sw), name
        assert c.fused_waves == int(fw), name
        assert c.last_wave_tbs == int(last), name


def test_planner_edge_cases():
    assert planner.waves(0, 148) == 0
    assert planner.utilisation(0, 148) == 0.0
    assert planner.last_wave_tbs(296, 148) == 148
    assert planner.gemm_tiles(64, 1024, 128, 256) == 4          # ragged M: one partial row of tiles
    assert planner.gemm_tiles(1024, 6144, 128, 256) == 192


# ----------------------------------------------------------------------------- dependencies


def test_gemm_data_deps_closed_form():
    ch = deps.GemmChain(M=300, N1=512, BM=128, BNo=128, BK=64)   # ragged M
    for m in range(ch.m_tiles):
        for kb in range(ch.k_blocks):
            assert deps.data_deps(ch, m, kb) == {(m, kb // 2)}
    ch = deps.GemmChain(M=128, N1=200, BM=64, BNo=64, BK=64)     # ragged N1
    assert ch.k_blocks == 4 and ch.n_tiles == 4
    assert deps.data_deps(ch, 1, 3) == {(1, 3)}


def test_conv_data_deps_halo_closed_form():
    ch = deps.ConvChain(N=2, P=14, Q=14, C=128, TH=7, BNo=128, BK=64)
    assert ch.tiles_per_image == 2 and ch.k_blocks == 18
    cb_per_tap = 2
    for m in range(ch.m_tiles):
        n, hb = divmod(m, 2)
        p0, p1 = hb * 7, min(hb * 7 + 7, 14) - 1
        for kb in range(ch.k_blocks):
            tap = kb // cb_per_tap
            r = tap // 3
            lo, hi = max(p0 + r - 1, 0), min(p1 + r - 1, 13)
            want = {(n * 2 + t, 0) for t in range(lo // 7, hi // 7 + 1)}
            assert deps.data_deps(ch, m, kb) == want, (m, kb)
    # the halo: the first row-tile needs the second one only from filter row r = 2 on
    assert deps.data_deps(ch, 0, 0) == {(0, 0)}
    assert deps.data_deps(ch, 0, 12) == {(0, 0), (1, 0)}
    assert deps.data_deps(ch, 1, 0) == {(0, 0), (1, 0)}


def _union(sets):
    out = set()
    for s in sets:
        out |= s
    return out


@pytest.mark.parametrize("chain", [
    deps.GemmChain(M=256, N1=1024, BM=128, BNo=256, BK=64),
    deps.GemmChain(M=200, N1=512, BM=128, BNo=128, BK=64),
    deps.ConvChain(N=2, P=6, Q=5, C=128, TH=3, BNo=64, BK=64),
])
def test_policy_invariants(chain):
    nt = chain.n_tiles
    for m in range(chain.m_tiles):
        needed = [deps.data_deps(chain, m, kb) for kb in range(chain.k_blocks)]
        per_policy = {}
        for pol, G in [("TILE", 1), ("ROW", 1), ("STRIDED", 1), ("STRIDED", 2), ("STRIDED", nt), ("SENTINEL", 1)]:
            if pol == "STRIDED" and nt % G:
                continue
            ws = deps.wait_sets(chain, pol, m, G)
            # safety: everything a k-block reads has been waited for at or before it
            for kb in range(chain.k_blocks):
                assert needed[kb] <= _union(ws[:kb + 1]), (pol, G, m, kb)
            # no tile is waited for twice
            assert sum(len(s) for s in ws) == len(_union(ws))
            per_policy[(pol, G)] = ws
        tile = per_policy[("TILE", 1)]
        # TileSync waits for exactly the data dependencies, each when first needed
        assert _union(tile) == _union(needed)
        assert per_policy[("SENTINEL", 1)] == tile
        assert per_policy[("STRIDED", 1)] == tile
        if ("STRIDED", nt) in per_policy:
            # one group holding every column tile: the whole rows are waited for,
            # at the first k-block of each row, which for GEMM chains is RowSync
            assert _union(per_policy[("STRIDED", nt)]) == _union(per_policy[("ROW", 1)])
        row = per_policy[("ROW", 1)]
        assert all(not s for s in row[1:])
        assert _union(tile) <= row[0]


def test_strided_order_and_groups():
    ch = deps.GemmChain(M=128, N1=6 * 64, BM=128, BNo=64, BK=64)
    assert deps.strided_members(ch, 3, 4) == [0, 2, 4]
    assert deps.strided_members(ch, 2, 4) == [1, 4]
    assert deps.strided_producer_order(6, 3) == [0, 2, 4, 1, 3, 5]
    assert deps.strided_producer_order(6, 1) == list(range(6))
    assert sorted(deps.strided_producer_order(24, 2)) == list(range(24))


def test_sentinel_example_closed_form():
    inp = (np.arange(2048, dtype=np.float32) - 512.0) * 0.25
    inp[5] = -0.0
    out = sentinel.double_then_reverse(inp)
    i = np.arange(1024)
    want0 = 2 * 0.25 * (1023 - i - 512.0)
    want0[1023 - 5] = 0.0                      # input 5 was overwritten with -0.0
    np.testing.assert_array_equal(out[:1024], want0)
    np.testing.assert_array_equal(out[1024:], 2 * 0.25 * (2047 - i - 512.0))
    # element 1023 - 5 of tile 0 came from the -0.0 input and must be +0.0
    assert out[1018] == 0.0 and not np.signbit(out[1018])
    assert out[511] == 0.0 and not np.signbit(out[511])


@pytest.mark.parametrize("chain", [
    deps.ConvChain(N=2, P=6, Q=5, C=128, TH=2, BNo=64, BK=64),
    deps.ConvChain(N=1, P=7, Q=3, C=128, TH=3, BNo=128, BK=64),
    deps.ConvChain(N=1, P=5, Q=4, C=64, TH=1, BNo=64, BK=64),
])
@pytest.mark.parametrize("policy", ["ROW", "TILE"])
def test_two_buffer_rotation_is_covered_by_the_waits(chain, policy):
    """A stack whose intermediates alternate between two buffers overwrites, in stage
    s + 2, the buffer that stage s + 1 reads.  Before a stage-(s + 2) tile stores (after
    its last k-block) it has waited for every stage-(s + 1) tile its policy names; those
    must include every tile that reads the region it overwrites (a tile posts only after
    its own k-blocks have read their input)."""
    for m in range(chain.m_tiles):
        waited = set().union(*deps.wait_sets(chain, policy, m))
        for c in range(chain.n_tiles):
            readers = deps.war_readers(chain, m, c)
            assert readers, (m, c)
            assert readers <= waited, (m, c, sorted(readers - waited))


def test_two_buffer_rotation_needs_every_k_block_of_waits():
    """The property above holds only once all of a tile's k-blocks have waited: the
    TileSync waits before the first k-block alone miss readers (rows below the tile), so
    the store must follow the last wait."""
    chain = deps.ConvChain(N=1, P=6, Q=4, C=128, TH=2, BNo=64, BK=64)
    first = deps.wait_sets(chain, "TILE", 1)[0]
    assert not deps.war_readers(chain, 1, 0) <= first

