"""CPU tests of the C-ABI library: it builds, loads and exports every function the public
header declares; its host-side planner matches the oracle (and through it the tables of
[cuSync]); and the dependency logic the kernels execute (the same code, called on the
host) matches the oracle's brute-force dependency sets for every policy."""

import os
import re

import pytest

import tile_level_sync_gb300 as cs
from oracle import deps, planner

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(cusync_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_function():
    lib = cs.load()
    names = _declared_functions()
    assert len(names) >= 13
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def _header_constants():
    """CUSYNC_* enumerators (explicit values) and #define flags of the public header."""
    src = open(os.path.join(ROOT, "include", "cusync.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    vals = {k: int(v) for k, v in re.findall(r"\b(CUSYNC_[A-Z0-9_]+)\s*=\s*(\d+)", src)}
    for k, sh in re.findall(r"#define\s+(CUSYNC_[A-Z0-9_]+)\s+\(1u\s*<<\s*(\d+)\)", src):
        vals[k] = 1 << int(sh)
    for k, v in re.findall(r"#define\s+(CUSYNC_[A-Z0-9_]+)\s+(\d+)\s*$", src, flags=re.M):
        vals[k] = int(v)
    return vals


def test_binding_constants_match_header():
    vals = _header_constants()
    assert len(vals) >= 20
    for name, v in vals.items():
        py = name[len("CUSYNC_"):]
        if py.startswith("POLICY_") or py.startswith("CHAIN_") or py.startswith("LAUNCH_") or \
                py.startswith("FLAG_") or py.startswith("DEBUG_"):
            assert getattr(cs, py) == v, name
        elif py == "OK" or py.startswith("ERR_") or py.startswith("NOALLOC_"):
            assert getattr(cs, py) == v, name


def test_status_strings():
    assert cs.status_string(cs.OK) == "CUSYNC_OK"
    assert cs.status_string(cs.ERR_TIMEOUT) == "CUSYNC_ERR_TIMEOUT"


@pytest.mark.parametrize("tbs0,tbs1,occ,sms", [
    (192, 384, 2, 80), (72, 48, 3, 80), (6, 6, 1, 4), (240, 0, 2, 80), (0, 0, 1, 148),
    (48, 96, 1, 148), (384, 768, 1, 148), (1536, 3072, 1, 148), (296, 148, 1, 148), (1, 1, 1, 1),
])
def test_wave_stats_matches_oracle(tbs0, tbs1, occ, sms):
    r = cs.cusync_wave_stats(tbs0, tbs1, occ, sms)
    cap = planner.wave_capacity(occ, sms)
    o = planner.chain_waves([tbs0, tbs1], cap)
    assert r.cap == cap
    assert list(r.tbs) == [tbs0, tbs1]
    assert list(r.waves_ceil) == list(o.waves_ceil)
    assert list(r.waves) == pytest.approx(list(o.waves_frac), abs=1e-15)
    assert list(r.util) == pytest.approx(list(o.util), abs=1e-15)
    assert r.stream_waves == o.stream_waves
    assert r.fused_waves == o.fused_waves
    assert r.fused_waves_frac == pytest.approx(o.fused_waves_frac, abs=1e-15)
    assert r.last_wave_tbs == o.last_wave_tbs


def test_wave_stats_invalid():
    lib = cs.load()
    rep = cs.cusync_wave_report_t()
    import ctypes
    assert lib.cusync_wave_stats(-1, 0, 1, 1, ctypes.byref(rep)) == cs.ERR_INVALID_ARG
    assert lib.cusync_wave_stats(1, 0, 0, 1, ctypes.byref(rep)) == cs.ERR_INVALID_ARG
    assert lib.cusync_wave_stats(1, 0, 1, 0, ctypes.byref(rep)) == cs.ERR_INVALID_ARG
    assert lib.cusync_wave_stats(1, 0, 1, 1, None) == cs.ERR_INVALID_ARG


GPT = dict(K=12288, N1=6144, N2=12288)


@pytest.mark.parametrize("M,tile_n,prod,cons,stream,fused", [
    (64, 256, 4, 1, 2, 1),
    (256, 256, 48, 96, 2, 1),
    (512, 256, 96, 192, 3, 2),
    (1024, 256, 192, 384, 5, 4),
    (2048, 256, 384, 768, 9, 8),
    (4096, 256, 768, 1536, 17, 16),
    (256, 128, 96, 192, 3, 2),
    (1024, 128, 384, 768, 9, 8),
])
def test_plan_waves_gpt_mlp(M, tile_n, prod, cons, stream, fused):
    dims = dict(K=256, N1=1024, N2=256) if M == 64 else GPT
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, tile_n=tile_n, num_sms=148, cta_pair=1, ksplit=1,
                     ksplit_consumer=1, **dims)
    r = cs.cusync_plan_waves(d)
    assert (r.tbs[0], r.tbs[1]) == (prod, cons)
    assert r.tbs[0] == planner.gemm_tiles(M, dims["N1"], 128, tile_n)
    assert (r.stream_waves, r.fused_waves) == (stream, fused)
    assert (r.tile_m, r.tile_n, r.tile_k) == (128, tile_n, 64)


@pytest.mark.parametrize("M,prod,cons,stream,fused", [
    (256, 24, 48, 2, 1),
    (1024, 96, 192, 5, 4),
    (4096, 384, 768, 17, 16),
])
def test_plan_waves_cta_pairs(M, prod, cons, stream, fused):
    # a CTA pair computes a 256 x 256 tile and occupies two SMs: 74 pairs on 148 SMs
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, tile_n=256, num_sms=148, cta_pair=2, ksplit=1, ksplit_consumer=1, **GPT)
    r = cs.cusync_plan_waves(d)
    assert (r.tbs[0], r.tbs[1]) == (prod, cons)
    assert r.cap == 74
    assert (r.stream_waves, r.fused_waves) == (stream, fused)
    assert (r.tile_m, r.tile_n) == (256, 256)
    o = planner.chain_waves([prod, cons], 74)
    assert (o.stream_waves, o.fused_waves) == (stream, fused)
    info = cs.cusync_plan_info(d)
    assert info.cta_pair == 2 and info.grid[0] == 2 * min(74, prod + cons)


def test_cta_pairs_not_for_convolution_chains():
    d = cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", n=1, h=14, w=14, c=64, k_out=64, num_sms=148, cta_pair=2)
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(d)
    assert e.value.status == cs.ERR_UNSUPPORTED
    d.cta_pair = 0
    assert cs.cusync_plan_info(d).cta_pair == 1
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=64, K=64, N1=256, N2=64, num_sms=148)
    assert cs.cusync_plan_info(d).cta_pair == 1
    d.M = 1024
    assert cs.cusync_plan_info(d).cta_pair == 2
    d.M = 512
    assert cs.cusync_plan_info(d).cta_pair == 2
    d.M = 256
    assert cs.cusync_plan_info(d).cta_pair == 2
    d.M = 255
    assert cs.cusync_plan_info(d).cta_pair == 1
    d.M = 64
    d.cta_pair = 2
    assert cs.cusync_plan_info(d).cta_pair == 2


def test_plan_swiglu_and_conv():
    d = cs.make_desc(cs.CHAIN_MLP_SWIGLU, "TILE", M=256, K=8192, N1=3584, N2=8192, tile_n=256, num_sms=148,
                     cta_pair=1, ksplit=1, ksplit_consumer=1)
    r = cs.cusync_plan_waves(d)
    assert (r.tbs[0], r.tbs[1]) == (2 * 28, 2 * 32)
    d = cs.make_desc(cs.CHAIN_CONV_RELU, "TILE", n=32, h=14, w=14, c=256, k_out=256, tile_n=256, num_sms=148)
    info = cs.cusync_plan_info(d)
    assert info.conv_rows_per_tile == 7
    assert list(info.m_tiles) == [64, 64] and list(info.k_blocks) == [36, 36]
    r = cs.cusync_plan_waves(d)
    assert (r.tbs[0], r.tbs[1], r.stream_waves, r.fused_waves) == (64, 64, 2, 1)


def test_invalid_and_unsupported_descriptors():
    bad = [
        (cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=0, K=64, N1=64, N2=64, num_sms=148), cs.ERR_INVALID_ARG),
        (cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=8, K=60, N1=64, N2=64, num_sms=148), cs.ERR_UNSUPPORTED),
        (cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=8, K=64, N1=64, N2=64, tile_n=64, num_sms=148),
         cs.ERR_UNSUPPORTED),
        (cs.make_desc(cs.CHAIN_MLP_GELU, 9, M=8, K=64, N1=64, N2=64, num_sms=148), cs.ERR_INVALID_ARG),
        (cs.make_desc(cs.CHAIN_MLP_GELU, "STRIDED", M=8, K=64, N1=768, N2=64, tile_n=256, strided_group=2,
                      num_sms=148), cs.ERR_UNSUPPORTED),   # 3 column tiles, G = 2
        (cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", n=1, h=14, w=14, c=96, k_out=128, num_sms=148),
         cs.ERR_UNSUPPORTED),
        (cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", n=1, h=4, w=200, c=64, k_out=64, num_sms=148),
         cs.ERR_UNSUPPORTED),
    ]
    for d, want in bad:
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_plan_waves(d)
        assert e.value.status == want


# ------------------------------------------------------------------ dependency logic


def _members(policy, flag, nt, D, G):
    if policy == "TILE":
        return {(flag // nt, flag % nt)}
    if policy == "ROW":
        return {(flag, c) for c in range(nt)}
    if policy == "STRIDED":
        m, g = divmod(flag, D)
        return {(m, g + j * D) for j in range(G)}
    raise ValueError(policy)


def _oracle_chain(desc, info):
    if desc.kind == cs.CHAIN_CONV_RELU:
        return deps.ConvChain(N=desc.n, P=desc.h, Q=desc.w, C=desc.k_out, TH=info.conv_rows_per_tile,
                              BNo=info.n_out[0], BK=info.tile_k)
    return deps.GemmChain(M=desc.M, N1=desc.N1, BM=info.tile_m, BNo=info.n_out[0], BK=info.tile_k)


CASES = [
    dict(kind=cs.CHAIN_MLP_GELU, M=300, K=128, N1=1024, N2=256, tile_n=256),
    dict(kind=cs.CHAIN_MLP_GELU, M=256, K=128, N1=1536, N2=256, tile_n=128),
    dict(kind=cs.CHAIN_MLP_GELU, M=130, K=64, N1=640, N2=64, tile_n=128),           # ragged M and N1
    dict(kind=cs.CHAIN_MLP_GELU, M=520, K=128, N1=1152, N2=256, tile_n=192),        # 192-wide (pairs only)
    dict(kind=cs.CHAIN_MLP_GELU, M=300, K=128, N1=1000, N2=64, tile_n=192),         # ... with a ragged N1
    dict(kind=cs.CHAIN_MLP_SWIGLU, M=200, K=64, N1=512, N2=64, tile_n=256),
    dict(kind=cs.CHAIN_CONV_RELU, n=2, h=14, w=14, c=64, k_out=256, tile_n=128),
    dict(kind=cs.CHAIN_CONV_RELU, n=2, h=9, w=30, c=64, k_out=128, tile_n=128),     # 4 rows per tile
    dict(kind=cs.CHAIN_CONV_RELU, n=1, h=5, w=100, c=128, k_out=128, tile_n=128),   # 1 row per tile
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("policy,G", [("TILE", 1), ("ROW", 1), ("STRIDED", 2), ("STRIDED", 1)])
@pytest.mark.parametrize("pair", [1, 2])
def test_consumer_waits_match_oracle(case, policy, G, pair):
    if pair == 2 and case["kind"] == cs.CHAIN_CONV_RELU:
        pytest.skip("CTA pairs are for the MLP chains")
    desc = cs.make_desc(policy=policy, strided_group=G, num_sms=148, cta_pair=pair, **case)
    try:
        info = cs.cusync_plan_info(desc)
    except cs.CusyncError as e:
        # StridedSync needs a column-tile count divisible by G; 192-wide tiles need pairs
        assert (policy == "STRIDED" or (case["tile_n"] == 192 and pair == 1)) and e.status == cs.ERR_UNSUPPORTED
        return
    ch = _oracle_chain(desc, info)
    nt = info.n_tiles[0]
    assert ch.n_tiles == nt and ch.m_tiles == info.m_tiles[1] and ch.k_blocks == info.k_blocks[1]
    D, Gc = info.strided_distance, info.strided_group
    for m in range(ch.m_tiles):
        got = [set() for _ in range(ch.k_blocks)]
        for kb, flag, per_run in cs.cusync_consumer_waits(desc, m):
            mem = _members(policy, flag, nt, D, Gc)
            assert per_run == len(mem) * info.cta_pair   # every CTA of a tile posts
            assert 0 <= flag < info.num_flags
            got[kb] |= mem
        want = deps.wait_sets(ch, policy, m, Gc)
        assert got == want, (policy, m)


@pytest.mark.parametrize("case", CASES)
def test_sentinel_and_stream_wait_on_no_semaphore(case):
    for pol in ("SENTINEL", "STREAM"):
        desc = cs.make_desc(policy=pol, num_sms=148, **case)
        info = cs.cusync_plan_info(desc)
        assert info.num_flags == 0
        for m in range(info.m_tiles[1]):
            assert cs.cusync_consumer_waits(desc, m) == []
        assert cs.cusync_producer_flag(desc, 0, 0) == -1


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("policy,G", [("TILE", 1), ("ROW", 1), ("STRIDED", 2)])
@pytest.mark.parametrize("pair", [1, 2])
def test_producer_posts_and_order(case, policy, G, pair):
    if pair == 2 and case["kind"] == cs.CHAIN_CONV_RELU:
        pytest.skip("CTA pairs are for the MLP chains")
    desc = cs.make_desc(policy=policy, strided_group=G, num_sms=148, cta_pair=pair, **case)
    try:
        info = cs.cusync_plan_info(desc)
    except cs.CusyncError:
        return
    nt, D, Gc = info.n_tiles[0], info.strided_distance, info.strided_group
    posts = {}
    for m in range(info.m_tiles[0]):
        for c in range(nt):
            f = cs.cusync_producer_flag(desc, m, c)
            assert (m, c) in _members(policy, f, nt, D, Gc)
            posts[f] = posts.get(f, 0) + 1
    for f, n in posts.items():
        assert n == len(_members(policy, f, nt, D, Gc))
    order = [cs.cusync_producer_col(desc, y) for y in range(nt)]
    if policy == "STRIDED":
        assert order == deps.strided_producer_order(nt, Gc)
    else:
        assert order == list(range(nt))


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("policy,G", [("ROW", 1), ("STRIDED", 2), ("SENTINEL", 1)])
@pytest.mark.parametrize("raster", [1, 3, 16])
def test_tile_order_is_a_permutation(case, policy, G, raster):
    desc = cs.make_desc(policy=policy, strided_group=G, num_sms=148, raster_rows=raster, **case)
    try:
        info = cs.cusync_plan_info(desc)
    except cs.CusyncError:
        return
    for stage in (0, 1):
        mt, nt = info.m_tiles[stage], info.n_tiles[stage]
        seen = [cs.cusync_tile_at(desc, stage, u) for u in range(mt * nt)]
        assert sorted(seen) == [(m, n) for m in range(mt) for n in range(nt)]
        # rows are finished group by group: every tile of row group g precedes group g+1
        pos = {t: u for u, t in enumerate(seen)}
        for m in range(mt - 1):
            if (m // raster) != ((m + 1) // raster):
                assert max(pos[(m, n)] for n in range(nt)) < min(pos[(m + 1, n)] for n in range(nt))
        if raster == 1:
            order = deps.strided_producer_order(nt, info.strided_group) if (stage == 0 and policy == "STRIDED") \
                else list(range(nt))
            assert seen == [(m, order[y]) for m in range(mt) for y in range(nt)]


@pytest.mark.parametrize("kind,dims,pair,want", [
    (cs.CHAIN_MLP_GELU, dict(M=256, **GPT), 1, 3),            # 48 tiles on 152 SMs: 3 units each
    (cs.CHAIN_MLP_GELU, dict(M=512, **GPT), 1, 2),            # 96 tiles fill more than half a wave
    (cs.CHAIN_MLP_GELU, dict(M=1024, **GPT), 1, 1),           # 192 tiles: more than a wave
    (cs.CHAIN_MLP_GELU, dict(M=64, K=256, N1=1024, N2=256), 1, 1),   # 4 k-blocks: nothing to split
    (cs.CHAIN_MLP_GELU, dict(M=64, K=12288, N1=6144, N2=12288), 1, 4),  # 24 tiles: at most 4 units
    (cs.CHAIN_MLP_SWIGLU, dict(M=256, K=8192, N1=3584, N2=8192), 1, 2),
    (cs.CHAIN_MLP_GELU, dict(M=256, **GPT), 2, 3),            # 24 pair tiles on 76 pairs
])
def test_planner_k_split(kind, dims, pair, want):
    d = cs.make_desc(kind, "ROW", num_sms=152, cta_pair=pair, tile_n=256, **dims)
    info = cs.cusync_plan_info(d)
    assert info.ksplit == want
    lens = _unit_lengths(info)
    assert sum(lens) == info.k_blocks[0] and min(lens) >= 1
    if pair == 2 and want > 1:
        # graded split: each unit 8 k-blocks longer (short units: a quarter of one, even)
        assert info.ksplit_skew == max(2, min(8, info.k_blocks[0] // want // 4) & ~1)
        assert all(b - a == info.ksplit_skew for a, b in zip(lens[:-2], lens[1:-1])) and lens[-1] >= lens[-2]
    else:
        assert info.ksplit_skew == 0
        assert info.kb_per_split * want >= info.k_blocks[0] > info.kb_per_split * (want - 1)
    r = cs.cusync_plan_waves(d)
    assert r.tbs[0] == info.m_tiles[0] * info.n_tiles[0] * want   # the producer launch runs units
    assert r.tbs[0] * pair <= 2 * 152


def test_k_split_requests():
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=256, num_sms=152, ksplit=5, ksplit_skew=-1, tile_n=256, **GPT)
    info = cs.cusync_plan_info(d)
    assert info.ksplit == 5 and info.kb_per_split == 39            # 192 k-blocks in 5 equal units
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=256, num_sms=152, ksplit=5, tile_n=256, **GPT)
    info = cs.cusync_plan_info(d)
    assert (info.ksplit, info.kb_per_split, info.ksplit_skew) == (5, 22, 8)  # graded: 22, 30, 38, 46, 56
    assert _unit_lengths(info) == [22, 30, 38, 46, 56]
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=64, K=320, N1=512, N2=256, ksplit=4, num_sms=152)
    info = cs.cusync_plan_info(d)
    assert (info.ksplit, info.kb_per_split) == (3, 2)              # 5 k-blocks: no empty unit
    with pytest.raises(cs.CusyncError) as e:                       # more units than k-blocks
        cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=64, K=128, N1=512, N2=256, ksplit=3,
                                         num_sms=152))
    assert e.value.status == cs.ERR_UNSUPPORTED
    d = cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", n=1, h=14, w=14, c=64, k_out=128, ksplit=2, num_sms=152)
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(d)
    assert e.value.status == cs.ERR_UNSUPPORTED
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=64, K=64, N1=256, N2=64, ksplit=-1,
                                         num_sms=152))
    assert e.value.status == cs.ERR_INVALID_ARG


def _unit_lengths(info):
    """k-blocks of each producer unit, as the header defines the graded split."""
    S, K = info.ksplit, info.k_blocks[0]
    out, start = [], 0
    for k in range(S):
        n = K - start if k == S - 1 else min(info.kb_per_split + k * info.ksplit_skew, K - start)
        out.append(n)
        start += n
    return out


@pytest.mark.parametrize("S,skew,want", [(3, 8, [56, 64, 72]), (3, 16, [48, 64, 80]), (2, 10, [91, 101]),
                                         (4, 5, [40, 45, 50, 57]), (3, -1, [64, 64, 64])])
def test_graded_k_split(S, skew, want):
    """Each producer unit runs ksplit_skew k-blocks more than the one before it and the
    last takes the remainder; the units cover the 192 k-blocks of the GPT-3 slice once,
    in order."""
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=256, num_sms=152, ksplit=S, ksplit_skew=skew, tile_n=256, **GPT)
    info = cs.cusync_plan_info(d)
    assert info.ksplit == S and info.ksplit_skew == max(skew, 0)
    lens = _unit_lengths(info)
    assert lens == want and sum(lens) == info.k_blocks[0] == 192
    assert all(b > a for a, b in zip(lens, lens[1:])) or skew < 0


def test_graded_k_split_requests():
    for bad in (-2, 65):
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=256, num_sms=152, ksplit=3,
                                             ksplit_skew=bad, **GPT))
        assert e.value.status == cs.ERR_INVALID_ARG
    # a skew that leaves unit 0 without k-blocks
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=256, K=1024, N1=512, N2=512, num_sms=152,
                                         ksplit=4, ksplit_skew=6))
    assert e.value.status == cs.ERR_UNSUPPORTED
    # no split: the skew is ignored
    info = cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=256, num_sms=152, ksplit=1,
                                            ksplit_skew=8, **GPT))
    assert info.ksplit == 1 and info.ksplit_skew == 0


# ----------------------------------------------------------------- attention chain

ATTN_CASES = [
    dict(M=200, K=512, N1=512, N2=384, tile_n=256),     # ragged M; 6 QKV column tiles, 4 heads
    dict(M=256, K=256, N1=768, N2=256, tile_n=128),     # 18 QKV column tiles, 6 heads
    dict(M=64, K=128, N1=256, N2=128, tile_n=256),
]


@pytest.mark.parametrize("case", ATTN_CASES)
@pytest.mark.parametrize("policy", ["ROW", "TILE", "STRIDED"])
def test_attention_plan_and_pointwise_waits_match_oracle(case, policy):
    d = cs.make_desc(cs.CHAIN_ATTENTION, policy, num_sms=148, cta_pair=1, ksplit=1, **case)
    info = cs.cusync_plan_info(d)
    M, N1, tn = case["M"], case["N1"], case["tile_n"]
    assert info.nst == 3 and info.cta_pair == 1
    assert (info.n_tiles[0], info.n_tiles[1], info.n_tiles2) == (3 * N1 // tn, N1 // 128, -(-case["N2"] // tn))
    assert info.k_blocks[1] == 0 and info.n_out[1] == 128
    qc = deps.QkvChain(M=M, N1=N1, BM=128, BNo=tn)
    nt = info.n_tiles[0]
    for m in range(info.m_tiles[1]):
        for i in range(info.n_tiles[1]):
            got = set()
            for flag, per_run in cs.cusync_pointwise_waits(d, m, i):
                if policy == "TILE":
                    mem = {divmod(flag, nt)}
                    assert per_run == 1
                elif policy == "ROW":
                    mem = {(flag, c) for c in range(nt)}
                    assert per_run == nt
                else:
                    D = info.strided_distance_pw
                    assert info.strided_group_pw == 3 and D * 3 == nt
                    mp, g = divmod(flag, D)
                    mem = {(mp, g + j * D) for j in range(3)}
                    assert per_run == 3
                got |= mem
            assert got == deps.pointwise_wait_set(qc, policy, m, i), (m, i)


@pytest.mark.parametrize("case", ATTN_CASES)
@pytest.mark.parametrize("policy", ["ROW", "TILE", "STRIDED"])
def test_attention_output_gemm_waits_match_oracle(case, policy):
    """The output GEMM reads XDot: TileSync on the pointwise tiles (also under StridedSync,
    as in the pages' Strided+TileSync), or RowSync."""
    d = cs.make_desc(cs.CHAIN_ATTENTION, policy, num_sms=148, cta_pair=1, ksplit=1, **case)
    info = cs.cusync_plan_info(d)
    gc = deps.GemmChain(M=case["M"], N1=case["N1"], BM=128, BNo=128, BK=64)
    want_pol = "ROW" if policy == "ROW" else "TILE"
    nt = info.n_tiles[1]
    for m in range(info.m_tiles2):
        got = [set() for _ in range(info.k_blocks2)]
        for kb, flag, per_run in cs.cusync_consumer_waits(d, m):
            got[kb] |= {(flag, c) for c in range(nt)} if want_pol == "ROW" else {divmod(flag, nt)}
        assert got == deps.wait_sets(gc, want_pol, m), m


def test_attention_refusals():
    base = dict(M=64, K=128, N1=256, N2=128, tile_n=256, num_sms=148)
    for kw, status in [(dict(policy="SENTINEL"), cs.ERR_UNSUPPORTED), (dict(policy="ROW", N1=192), cs.ERR_UNSUPPORTED)]:
        args = dict(base, **kw)
        pol = args.pop("policy")
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_plan_info(cs.make_desc(cs.CHAIN_ATTENTION, pol, **args))
        assert e.value.status == status, kw
    # the latency model covers the two-stage chains only
    with pytest.raises(cs.CusyncError):
        cs.cusync_predict_policies(cs.make_desc(cs.CHAIN_ATTENTION, "ROW", **base))
    # CTA pairs: 256-row tiles in all three stages, every CTA of a pair posting; the
    # convolution chains keep single CTAs
    info = cs.cusync_plan_info(cs.make_desc(cs.CHAIN_ATTENTION, "ROW", **dict(base, M=600, cta_pair=2)))
    assert info.cta_pair == 2 and info.m_tiles[0] == info.m_tiles[1] == info.m_tiles2 == 3
    assert cs.cusync_pointwise_waits(cs.make_desc(cs.CHAIN_ATTENTION, "TILE", **dict(base, cta_pair=2)), 0, 0)[0][1] == 2
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", n=1, h=14, w=14, c=64, k_out=64, cta_pair=2))
    assert e.value.status == cs.ERR_UNSUPPORTED


STACK_CASES = [
    dict(n=2, h=14, w=14, c=128, stages=4, tile_n=128),   # two row tiles per image
    dict(n=1, h=9, w=30, c=64, stages=3, tile_n=128),     # 4 image rows per tile, ragged columns
    dict(n=1, h=5, w=100, c=128, stages=5, tile_n=256),   # 1 image row per tile
]


@pytest.mark.parametrize("case", STACK_CASES)
@pytest.mark.parametrize("policy", ["ROW", "TILE"])
def test_stack_waits_match_oracle_and_cover_rotation(case, policy):
    """Every stage of a convolution stack waits on the one before it exactly as the
    oracle's Conv2DTileSync sets say (one set of semaphores per boundary), and the union
    of a tile's waits covers every tile that reads what it overwrites when the
    intermediates alternate between two buffers."""
    desc = cs.make_desc(cs.CHAIN_CONV_STACK, policy, num_sms=148, **case)
    info = cs.cusync_plan_info(desc)
    stages = case["stages"]
    assert info.nst == stages and info.work_buffers == min(2, stages - 1)
    assert info.work_bytes == info.work_buffers * case["n"] * case["h"] * case["w"] * case["c"] * 2
    ch = deps.ConvChain(N=case["n"], P=case["h"], Q=case["w"], C=case["c"], TH=info.conv_rows_per_tile,
                        BNo=info.n_out[0], BK=info.tile_k)
    nt = info.n_tiles[0]
    assert ch.n_tiles == nt and ch.m_tiles == info.m_tiles[1] and ch.k_blocks == info.k_blocks[1]
    assert info.num_flags % (stages - 1) == 0
    stride = info.num_flags // (stages - 1)
    for m in range(ch.m_tiles):
        got = [set() for _ in range(ch.k_blocks)]
        for kb, flag, per_run in cs.cusync_consumer_waits(desc, m):
            mem = _members(policy, flag, nt, info.strided_distance, info.strided_group)
            assert per_run == len(mem) and 0 <= flag < stride
            got[kb] |= mem
        assert got == deps.wait_sets(ch, policy, m), (policy, m)
        waited = set().union(*got)
        for c in range(nt):
            assert deps.war_readers(ch, m, c) <= waited, (m, c)


def test_stack_plan_and_refusals():
    base = dict(n=2, h=14, w=14, c=256, num_sms=152)
    act = 2 * 14 * 14 * 256 * 2
    for pol, nbuf in (("ROW", 2), ("TILE", 2), ("STREAM", 2), ("SENTINEL", 22)):
        info = cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_STACK, pol, stages=12, **base))
        assert info.nst == 12 and info.work_buffers == nbuf and info.work_bytes == nbuf * act
        assert info.m_tiles[0] == info.m_tiles[1] and info.k_blocks[0] == info.k_blocks[1]  # uniform stages
        per = {"ROW": info.m_tiles[0], "TILE": info.m_tiles[0] * info.n_tiles[0]}.get(pol, 0)
        assert info.num_flags == per * 11
    info = cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_STACK, "ROW", stages=2, **base))
    assert info.work_buffers == 1 and info.work_bytes == act
    bad = [
        (dict(stages=1), cs.ERR_UNSUPPORTED), (dict(stages=17), cs.ERR_UNSUPPORTED),
        (dict(stages=4, k_out=128), cs.ERR_UNSUPPORTED),             # channels must stay equal
        (dict(stages=4, cta_pair=2), cs.ERR_UNSUPPORTED),
        (dict(stages=4, policy=cs.POLICY_STRIDED_TILE), cs.ERR_UNSUPPORTED),
        (dict(stages=4, ksplit=2), cs.ERR_UNSUPPORTED),
    ]
    for extra, status in bad:
        kw = dict(base)
        pol = extra.pop("policy", cs.POLICY_ROW)
        kw.update(extra)
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_STACK, pol, **kw))
        assert e.value.status == status, extra
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_STACK, "ROW", n=1, h=8, w=8, c=96, stages=3, num_sms=152))
    assert e.value.status == cs.ERR_UNSUPPORTED


@pytest.mark.parametrize("kind,dims,pair,want", [
    (cs.CHAIN_MLP_GELU, dict(M=256, **GPT), 2, 1),      # 48 pair tiles: more than half of 76 pairs
    (cs.CHAIN_MLP_GELU, dict(M=1024, **GPT), 2, 1),
    (cs.CHAIN_MLP_SWIGLU, dict(M=256, K=8192, N1=3584, N2=8192), 2, 1),   # CTA pairs keep whole tiles
    (cs.CHAIN_MLP_SWIGLU, dict(M=256, K=8192, N1=3584, N2=8192), 1, 2),   # 64 tiles on 152 SMs
    (cs.CHAIN_MLP_GELU, dict(M=64, K=12288, N1=6144, N2=12288), 1, 3),    # 48 tiles: 3 units fit in a wave
    (cs.CHAIN_MLP_GELU, dict(M=64, K=256, N1=1024, N2=256), 1, 1),        # 16 k-blocks: nothing to split
])
def test_planner_consumer_split(kind, dims, pair, want):
    d = cs.make_desc(kind, "ROW", num_sms=152, cta_pair=pair, tile_n=256, **dims)
    info = cs.cusync_plan_info(d)
    assert info.ksplit_consumer == want
    assert info.kb_per_split_consumer * want >= info.k_blocks[1] > info.kb_per_split_consumer * (want - 1)
    # the model plays whole consumer tiles, so its prediction does not depend on the split
    d1 = cs.make_desc(kind, "ROW", num_sms=152, cta_pair=pair, tile_n=256, ksplit_consumer=1, **dims)
    assert cs.cusync_predict_policies(d).us[cs.POLICY_ROW] == cs.cusync_predict_policies(d1).us[cs.POLICY_ROW]


def test_consumer_split_requests():
    base = dict(num_sms=152, tile_n=256, M=256, **GPT)
    assert cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", ksplit_consumer=2, **base)).ksplit_consumer == 2
    assert cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", ksplit_consumer=1, **base)).ksplit_consumer == 1
    for bad, status in ((dict(ksplit_consumer=-1), cs.ERR_INVALID_ARG), (dict(ksplit_consumer=17), cs.ERR_INVALID_ARG)):
        with pytest.raises(cs.CusyncError) as e:
            cs.cusync_plan_info(cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", **bad, **base))
        assert e.value.status == status
    # only the MLP chains split their consumer
    conv = dict(n=2, h=14, w=14, c=128, k_out=128, num_sms=152)
    assert cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", **conv)).ksplit_consumer == 1
    with pytest.raises(cs.CusyncError) as e:
        cs.cusync_plan_info(cs.make_desc(cs.CHAIN_CONV_RELU, "ROW", ksplit_consumer=2, **conv))
    assert e.value.status == cs.ERR_UNSUPPORTED


@pytest.mark.parametrize("case", [
    dict(M=300, K=128, N1=1024, N2=256, tile_n=256),
    dict(M=256, K=128, N1=1536, N2=256, tile_n=128),
    dict(M=130, K=64, N1=2304, N2=64, tile_n=128),
    dict(M=520, K=128, N1=2304, N2=256, tile_n=192, cta_pair=2),
])
@pytest.mark.parametrize("policy,G", [("TILE", 1), ("ROW", 1), ("STRIDED", 2), ("STRIDED", 3)])
@pytest.mark.parametrize("ks", [2, 3])
def test_consumer_unit_waits_match_oracle(case, policy, G, ks):
    """Every K-split unit of a consumer tile waits, from its own first k-block on, for the
    producer tiles the oracle's policy sets name for exactly the k-blocks it computes."""
    case = dict(case)
    pair = case.pop("cta_pair", 1)
    desc = cs.make_desc(cs.CHAIN_MLP_GELU, policy, strided_group=G, num_sms=148, cta_pair=pair, ksplit_consumer=ks,
                        **case)
    try:
        info = cs.cusync_plan_info(desc)
    except cs.CusyncError as e:
        assert policy == "STRIDED" and e.status == cs.ERR_UNSUPPORTED
        return
    ch = _oracle_chain(desc, info)
    nt, D, Gc = info.n_tiles[0], info.strided_distance, info.strided_group
    per = info.kb_per_split_consumer
    # units start on producer column tiles, which may leave fewer units than asked for
    assert 1 < info.ksplit_consumer <= ks and per % max(1, info.n_out[0] // 64) == 0
    for m in range(ch.m_tiles):
        for u in range(info.ksplit_consumer):
            kbs = list(range(u * per, min((u + 1) * per, ch.k_blocks)))
            got = {kb: set() for kb in kbs}
            for kb, flag, per_run in cs.cusync_consumer_unit_waits(desc, m, u):
                assert kb in got
                got[kb] |= _members(policy, flag, nt, D, Gc)
            want = deps.wait_sets(ch, policy, m, Gc, kbs=kbs)
            assert [got[kb] for kb in kbs] == want, (policy, m, u)


def test_noalloc_semaphore_limit_is_exact():
    """The allocation-free entry point accepts a plan of exactly
    CUSYNC_NOALLOC_MAX_SEMAPHORES semaphores (it gets past the size check to the pointer
    check: null operands are INVALID_ARG) and refuses one more as UNSUPPORTED, before it
    touches a device.  Single-CTA RowSync plans have one semaphore per 128-row tile."""
    import ctypes
    lib = cs.load()
    n = cs.NOALLOC_MAX_SEMAPHORES
    for tiles, want in ((n, cs.ERR_INVALID_ARG), (n + 1, cs.ERR_UNSUPPORTED)):
        d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=128 * tiles, K=64, N1=64, N2=64, cta_pair=1, tile_n=128,
                         num_sms=148)
        assert cs.cusync_plan_info(d).num_flags == tiles
        st = lib.cusync_run_mlp_noalloc(ctypes.byref(d), None, None, None, None, None, None, None)
        assert st == want, (tiles, cs.status_string(st))


def test_noalloc_refuses_k_split():
    """No workspace for K-split partial sums: a split of either GEMM is refused."""
    import ctypes
    lib = cs.load()
    for ks, ks1 in ((2, 0), (0, 2), (1, 3)):
        d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=256, K=2048, N1=1024, N2=512, tile_n=256, cta_pair=1,
                         ksplit=ks, ksplit_consumer=ks1, num_sms=148)
        st = lib.cusync_run_mlp_noalloc(ctypes.byref(d), None, None, None, None, None, None, None)
        assert st == cs.ERR_UNSUPPORTED, (ks, ks1, cs.status_string(st))


@pytest.mark.parametrize("M,pair,bands,group", [(1024, 2, 0, 2), (2048, 2, 0, 4), (4096, 2, 0, 8), (512, 2, 0, 1),
                                                (1024, 1, 0, 1), (1024, 2, 2, 1)])
def test_planner_default_tile_order(M, pair, bands, group):
    """The planner groups half of the row tiles (columns outer, rows inner) for MLP chains
    on CTA pairs with at least four row tiles and no row bands; row-major otherwise."""
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=M, K=512, N1=1024, N2=512, cta_pair=pair, num_sms=148,
                     bands=bands)
    info = cs.cusync_plan_info(d)
    for stage in (0, 1):
        order = [cs.cusync_tile_at(d, stage, u) for u in range(info.m_tiles[stage] * info.n_tiles[stage])]
        # the first `group` positions walk down the rows of column 0
        assert order[:group] == [(m, 0) for m in range(group)]
        if group < info.m_tiles[stage]:
            assert order[group] == (0, 1) if group > 1 else order[1] == (0, 1)
