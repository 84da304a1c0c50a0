"""Expected output of the sentinel-protocol example (oracle; test infrastructure).

[CUDA-FGS] §4.6.6 (Example): a producer writes out = canonicalize(2 * in)
for fp32 data into a sentinel-initialised buffer, and a consumer reverses
each 1024-element tile of that buffer.  The consumer's output element
t*1024 + i is therefore canonicalize(2 * in[t*1024 + 1023 - i]), where
canonicalize turns -0.0 into +0.0 (§4.6.4.3).  Computed here in fp64 and
returned as float32 values; doubling is exact in binary floating point, so
the float32 result of the definition is unique.
"""

import numpy as np

TILE_ELEMS = 1024


def double_then_reverse(inp, tile=TILE_ELEMS):
    x = np.asarray(inp, dtype=np.float32).astype(np.float64)
    if x.size % tile:
        raise ValueError("input length must be a multiple of the tile size")
    doubled = 2.0 * x
    doubled = np.where(doubled == 0.0, 0.0, doubled)   # -0 -> +0
    out = doubled.reshape(-1, tile)[:, ::-1].reshape(-1)
    return out.astype(np.float32)
