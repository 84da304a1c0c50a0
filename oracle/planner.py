"""Thread-block wave arithmetic (oracle; test infrastructure).

[cuSync] §II-A, paragraph "Thread block Wave Execution": a GPU runs at most
occupancy x #SMs thread blocks at a time, so a grid of TBs thread blocks
needs ceil(TBs / (occupancy x #SMs)) waves.  Table ``tab:intro`` reports the
fractional wave count TBs / (occupancy x #SMs) and the utilisation
TBs / (ceil(waves) x occupancy x #SMs).

[cuSync] §III and §III-A ("Under-utilization in Training of GPT-3"): with
stream synchronisation the two kernels of a chain take the sum of their
ceilinged wave counts; with fine-grained synchronisation the thread blocks
of both kernels share waves, ceil((TBs_1 + TBs_2) / cap), and the last
wave holds (TBs_1 + TBs_2) mod cap thread blocks.  Table ``tab:waves:mlp``
reports the fused figure as the sum of the fractional waves.
"""

import math
from dataclasses import dataclass


def grid_tbs(grid):
    """Number of thread blocks of a grid given as (x, y, z) or any sequence."""
    n = 1
    for g in grid:
        n *= int(g)
    return n


def wave_capacity(occupancy, num_sms):
    return int(occupancy) * int(num_sms)


def fractional_waves(tbs, cap):
    return tbs / cap


def waves(tbs, cap):
    return math.ceil(tbs / cap)


def utilisation(tbs, cap):
    """TBs / (ceil(waves) * cap); 0 for an empty grid."""
    w = waves(tbs, cap)
    return 0.0 if w == 0 else tbs / (w * cap)


def last_wave_tbs(tbs, cap):
    """Thread blocks in the last wave (cap when the grid fills it exactly; 0 when empty)."""
    if tbs == 0:
        return 0
    r = tbs % cap
    return cap if r == 0 else r


@dataclass
class ChainWaves:
    tbs: tuple
    waves_frac: tuple
    waves_ceil: tuple
    util: tuple
    stream_waves: int        # sum of per-kernel ceilings (stream synchronisation)
    fused_waves_frac: float  # sum of fractional waves (tab:waves:mlp "cuSync Waves")
    fused_waves: int         # ceil(sum TBs / cap)
    last_wave_tbs: int       # thread blocks in the fused last wave
    cap: int


def chain_waves(tbs_list, cap):
    """Wave figures of a chain of dependent kernels that share one capacity."""
    tbs = tuple(int(t) for t in tbs_list)
    total = sum(tbs)
    return ChainWaves(
        tbs=tbs,
        waves_frac=tuple(fractional_waves(t, cap) for t in tbs),
        waves_ceil=tuple(waves(t, cap) for t in tbs),
        util=tuple(utilisation(t, cap) for t in tbs),
        stream_waves=sum(waves(t, cap) for t in tbs),
        fused_waves_frac=total / cap,
        fused_waves=waves(total, cap),
        last_wave_tbs=last_wave_tbs(total, cap),
        cap=cap,
    )


def gemm_tiles(m, n, tile_m, tile_n):
    """Output tiles of an [m, n] GEMM result cut into [tile_m, tile_n] tiles ([cuSync] §II-C)."""
    return math.ceil(m / tile_m) * math.ceil(n / tile_n)
