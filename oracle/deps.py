"""Tile dependency sets of a producer -> consumer chain (oracle; test infrastructure).

[cuSync] §II-C (Tile based Computations): the producer's output H is cut
into tiles, each written by one thread block; a consumer tile of a GEMM
reads the whole row band of H its output rows belong to.  §IV-D
(Synchronizing Dependent Tiles): before the consumer loads a tile of its A
input it waits for the producer tiles that write it.  This module derives,
by brute force over the elements of H, exactly which producer tiles write
any element a consumer k-block reads (the *data dependencies*), and the
sets each policy of [cuSync] §IV-E waits for:

* TileSync  -- one semaphore per producer tile; wait on each tile the first
               time a k-block needs it.
* RowSync   -- one semaphore per producer row of tiles; wait once, before the
               first k-block, for every row the consumer tile will read.
* StridedSync(G) -- producer column tiles that are D = n_cols / G apart
               share one semaphore (group g = col mod D, G members); wait for
               the whole group the first time a k-block needs one member.
               The page's formulas for this policy disagree with its text; the
               reading used (G members per group, distance D) is recorded in
               the design notes.  G = 1 is TileSync and G = n_cols is
               RowSync.
* Sentinel  -- [CUDA-FGS] §4.6: no semaphore; the consumer checks the loaded
               data itself, which amounts to waiting on exactly the data
               dependencies of each k-block.

Two geometries are modelled:

* GEMM chain: H is [M, N1]; producer tiles are [BM, BNo] blocks (BNo = H
  columns written per producer tile); consumer row-tile m reads
  H[m*BM:(m+1)*BM, kb*BK:(kb+1)*BK] for its k-block kb.
* Conv chain (implicit GEMM, 3x3 or any RxS, stride 1): H is NHWC
  [N, P, Q, C]; a producer and a consumer row-tile both cover TH whole image
  rows of one image (tile (n, hb) = rows hb*TH .. hb*TH+TH-1 of image n) and
  all Q columns; the reduction index is k = (r*S + s)*C + c, cut into BK
  channel blocks per filter tap, so k-block kb reads, for tap (r, s) and
  channel block cb, H[n, p + r - pad, q + s - pad, cb*BK:(cb+1)*BK] for the
  tile's output pixels (p, q) that fall inside the image.  This is the
  halo-aware form of [cuSync] §IV-E "Conv2DTileSync", whose mapping from an output
  tile to the input-image tile it waits on divides the column index by the filter
  area and leaves out the spatial halo.
"""

import math
from dataclasses import dataclass

import numpy as np

POLICIES = ("TILE", "ROW", "STRIDED", "SENTINEL")


@dataclass(frozen=True)
class GemmChain:
    M: int
    N1: int      # columns of H
    BM: int      # rows per tile (producer and consumer)
    BNo: int     # H columns written by one producer tile
    BK: int      # H columns read by one consumer k-block

    @property
    def m_tiles(self):
        return math.ceil(self.M / self.BM)

    @property
    def n_tiles(self):
        return math.ceil(self.N1 / self.BNo)

    @property
    def k_blocks(self):
        return math.ceil(self.N1 / self.BK)

    def h_shape(self):
        return (self.M, self.N1)

    def writes(self, m, c):
        mask = np.zeros(self.h_shape(), dtype=bool)
        mask[m * self.BM:(m + 1) * self.BM, c * self.BNo:(c + 1) * self.BNo] = True
        return mask

    def reads(self, m, kb):
        mask = np.zeros(self.h_shape(), dtype=bool)
        mask[m * self.BM:(m + 1) * self.BM, kb * self.BK:(kb + 1) * self.BK] = True
        return mask


@dataclass(frozen=True)
class ConvChain:
    N: int
    P: int       # image rows of H (= output rows of both convolutions, stride 1)
    Q: int       # image columns
    C: int       # channels of H
    TH: int      # image rows per row-tile
    BNo: int     # H channels written by one producer tile
    BK: int      # channels per consumer k-block
    R: int = 3
    S: int = 3
    pad: int = 1

    @property
    def tiles_per_image(self):
        return math.ceil(self.P / self.TH)

    @property
    def m_tiles(self):
        return self.N * self.tiles_per_image

    @property
    def n_tiles(self):
        return math.ceil(self.C / self.BNo)

    @property
    def k_blocks(self):
        return self.R * self.S * math.ceil(self.C / self.BK)

    def h_shape(self):
        return (self.N, self.P, self.Q, self.C)

    def _rows(self, m):
        n, hb = divmod(m, self.tiles_per_image)
        return n, hb * self.TH, min((hb + 1) * self.TH, self.P)

    def writes(self, m, c):
        n, p0, p1 = self._rows(m)
        mask = np.zeros(self.h_shape(), dtype=bool)
        mask[n, p0:p1, :, c * self.BNo:(c + 1) * self.BNo] = True
        return mask

    def reads(self, m, kb):
        n, p0, p1 = self._rows(m)
        cblocks = math.ceil(self.C / self.BK)
        tap, cb = divmod(kb, cblocks)
        r, s = divmod(tap, self.S)
        mask = np.zeros(self.h_shape(), dtype=bool)
        for p in range(p0, p1):
            hp = p + r - self.pad
            if not 0 <= hp < self.P:
                continue
            for q in range(self.Q):
                wq = q + s - self.pad
                if 0 <= wq < self.Q:
                    mask[n, hp, wq, cb * self.BK:(cb + 1) * self.BK] = True
        return mask


def data_deps(chain, m, kb):
    """Producer tiles (m', c') that write any element consumer row-tile m reads in k-block kb."""
    rd = chain.reads(m, kb)
    out = set()
    for mp in range(chain.m_tiles):
        for c in range(chain.n_tiles):
            if np.any(chain.writes(mp, c) & rd):
                out.add((mp, c))
    return out


def war_readers(chain, m, c):
    """Buffer rotation: the tiles (m', c') of the stage that reads a buffer which stage
    s + 2 overwrites with its tile (m, c).  In a stack whose intermediates alternate
    between two buffers, stage s + 2 writes the buffer that stage s wrote and stage s + 1
    read; every consumer tile (m', c') reads all channels of its input rows, so it is a
    reader of the region when any of its k-blocks reads an element that (m, c) writes."""
    w = chain.writes(m, c)
    readers = set()
    for mp in range(chain.m_tiles):
        if any((chain.reads(mp, kb) & w).any() for kb in range(chain.k_blocks)):
            readers |= {(mp, cp) for cp in range(chain.n_tiles)}
    return readers


def strided_members(chain, G, c):
    """Producer column tiles sharing column c's StridedSync semaphore (distance D = n_tiles / G)."""
    if chain.n_tiles % G:
        raise ValueError("n_tiles must be a multiple of the group size G")
    D = chain.n_tiles // G
    g = c % D
    return [g + j * D for j in range(G)]


def strided_producer_order(n_tiles, G):
    """Column visited at position y of a producer row under StridedSync ([cuSync] Fig.
    ``fig:use-case:self-attention:strided``, ``prodOrder``, with G members per group):
    the G members of group 0 first, then those of group 1, and so on."""
    D = n_tiles // G
    return [(y % G) * D + y // G for y in range(n_tiles)]


def wait_sets(chain, policy, m, G=2, kbs=None):
    """For consumer row-tile m: list over k-blocks of the producer tiles newly waited for
    before that k-block's A load (cumulatively these must cover every data dependency).

    kbs: the k-blocks a work unit computes, in order (default: all of the tile's); a
    K-split unit of the consumer waits for what its own k-blocks read, from its first."""
    kbs = range(chain.k_blocks) if kbs is None else kbs
    deps = [data_deps(chain, m, kb) for kb in kbs]
    waited = set()
    out = []
    if policy in ("TILE", "SENTINEL"):
        for d in deps:
            new = d - waited
            waited |= new
            out.append(new)
    elif policy == "ROW":
        rows = sorted({mp for d in deps for (mp, _) in d})
        first = {(mp, c) for mp in rows for c in range(chain.n_tiles)}
        out = [first] + [set() for _ in deps[1:]]
    elif policy == "STRIDED":
        for d in deps:
            new = set()
            for (mp, c) in d:
                if (mp, c) not in waited:
                    new |= {(mp, cc) for cc in strided_members(chain, G, c)}
            new -= waited
            waited |= new
            out.append(new)
    else:
        raise ValueError(policy)
    return out


@dataclass(frozen=True)
class QkvChain:
    """The QKV GEMM -> pointwise step of the attention block ([cuSync] Fig.
    ``fig:use-case:self-attention:dependencies``): XQKV [M, 3*N1] is written in [BM, BNo]
    tiles; pointwise tile (m, i) reads rows m*BM.. and the columns of head i
    ([i*head, (i+1)*head)) of each of the three blocks."""
    M: int
    N1: int
    BM: int
    BNo: int
    head: int = 128

    @property
    def n_tiles(self):
        return math.ceil(3 * self.N1 / self.BNo)

    def writes(self, m, c):
        mask = np.zeros((self.M, 3 * self.N1), dtype=bool)
        mask[m * self.BM:(m + 1) * self.BM, c * self.BNo:(c + 1) * self.BNo] = True
        return mask

    def reads(self, m, i):
        mask = np.zeros((self.M, 3 * self.N1), dtype=bool)
        for b in range(3):
            c0 = b * self.N1 + i * self.head
            mask[m * self.BM:(m + 1) * self.BM, c0:c0 + self.head] = True
        return mask


def pointwise_wait_set(chain, policy, m, i):
    """Producer tiles a pointwise tile waits for: its data dependencies (TileSync), the
    whole row(s) of tiles (RowSync), or the StridedSync(G = 3) groups of its columns."""
    rd = chain.reads(m, i)
    data = {(mp, c) for mp in range(math.ceil(chain.M / chain.BM)) for c in range(chain.n_tiles)
            if np.any(chain.writes(mp, c) & rd)}
    if policy == "TILE":
        return data
    if policy == "ROW":
        return {(mp, c) for (mp, _) in data for c in range(chain.n_tiles)}
    if policy == "STRIDED":
        return {(mp, cc) for (mp, c) in data for cc in strided_members(chain, 3, c)}
    raise ValueError(policy)
