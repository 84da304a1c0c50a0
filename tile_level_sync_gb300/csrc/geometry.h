// Tile geometry, tile order and dependency tracking of a producer -> consumer chain.
//
// Everything here is plain integer logic compiled for both the host and the device:
// the chain kernel calls it to decide which semaphores to wait on and to post, and the
// host library exposes the same functions (cusync_consumer_waits,
// cusync_producer_flag) so that the dependency logic the GPU executes can be checked
// on a CPU.
//
// Sources:
//  * "A Framework for Fine-Grained Synchronization of Dependent GPU Kernels" (cuSync),
//    §II-C (tiled GEMM: tile C^{xy} reads a row of A tiles), §IV-C (tile processing
//    order), §IV-E (TileSync, RowSync, StridedSync, Conv2DTileSync; Fig. fig:ex and
//    Fig. fig:use-case:self-attention:strided).
#pragma once
#include <cstdint>

#if defined(__CUDACC__)
#define CUSYNC_HD __host__ __device__ __forceinline__
#else
#define CUSYNC_HD inline
#endif

namespace cusync {

// Policy and epilogue codes (same values as the public enums in cusync.h).
enum : int32_t { POL_STREAM = 0, POL_ROW = 1, POL_TILE = 2, POL_STRIDED = 3, POL_SENTINEL = 4 };
enum : int32_t { EPI_NONE = 0, EPI_GELU = 1, EPI_SWIGLU = 2, EPI_RELU = 3 };
// A operand of a stage: a GEMM, an implicit-GEMM convolution, or no GEMM at all (the
// attention chain's pointwise stage, computed by the epilogue warps).
enum : int32_t { AMODE_GEMM = 0, AMODE_CONV = 1, AMODE_POINTWISE = 2 };
// Width of a pointwise tile of the attention chain (one attention head).
constexpr int32_t kHead = 128;

constexpr int32_t kBM = 128;  // output rows (tokens / pixels) per tile: UMMA M
constexpr int32_t kBK = 64;   // reduction elements per k-block: one 128-byte swizzle row of bf16
constexpr int32_t kMaxConvColTiles = 16;
constexpr int32_t kMaxWaits = 4;

// One GEMM stage of the chain: out[M, N] = act(A[M, K] x B[N, K]^T).
// For a convolution stage, A is the implicit im2col matrix of an NHWC image and the
// M rows of a tile are `th` whole image rows of one image (th * img_w <= 128).
struct StageGeo {
  int32_t a_mode;    // AMODE_*
  int32_t epi;       // EPI_*
  int32_t M;         // output rows: tokens, or pixels N*P*Q
  int32_t N;         // output columns (channels)
  int32_t K;         // reduction length (conv: 9 * input channels)
  int32_t m_tiles;   // row tiles
  int32_t n_tiles;   // column tiles
  int32_t k_blocks;  // ceil(K / kBK)
  int32_t n_out;     // output columns written per tile (BN, or BN/2 for SwiGLU)
  int32_t raster;    // row tiles per raster group (see tile_at)
  // convolution only
  int32_t img_n, img_h, img_w, cin;  // input image (= output image: 3x3, stride 1, pad 1)
  int32_t th;                        // image rows per row tile
  int32_t tpi;                       // row tiles per image = ceil(img_h / th)
  int32_t cblocks;                   // cin / kBK channel blocks per filter tap
  // K split (GEMM producers): each tile is computed by ksplit work units over
  // consecutive k-block ranges (split_unit); their fp32 partial sums are added in unit
  // order and the last unit applies the epilogue.  1 = no split.  Unit 0 takes
  // kb_per_split k-blocks and each later unit kb_skew more than the one before it; the
  // last unit takes what remains.
  int32_t ksplit;
  int32_t kb_per_split;
  int32_t kb_skew;
};

// First k-block and k-block count of K-split unit ks of a stage.  With kb_skew = 0 the
// units are kb_per_split long but the last, which takes the remainder.
CUSYNC_HD void split_unit(const StageGeo& g, int32_t ks, int32_t* kb0, int32_t* nkb) {
  const int32_t k0 = ks * g.kb_per_split + g.kb_skew * (ks * (ks - 1) / 2);
  const int32_t rest = g.k_blocks - k0;
  const int32_t len = g.kb_per_split + ks * g.kb_skew;
  *kb0 = k0;
  *nkb = (ks == g.ksplit - 1 || rest < len) ? rest : len;
}

// Work units of a stage's queue: tiles x K-split units (the split units of one tile are
// consecutive in the queue).
CUSYNC_HD int64_t stage_units(const StageGeo& g) {
  return (int64_t)g.m_tiles * g.n_tiles * (g.ksplit > 1 ? g.ksplit : 1);
}

// Consumer-side view of the producer's semaphores.
struct DepCfg {
  int32_t policy;        // POL_*
  int32_t prod_m_tiles;  // producer row tiles
  int32_t prod_n_tiles;  // producer column tiles (nt)
  int32_t prod_n_out;    // H columns per producer tile
  int32_t G;             // StridedSync group size (tiles sharing one semaphore)
  int32_t D;             // StridedSync distance = nt / G
  int32_t posts;         // posts per producer tile (one per CTA computing it: 1 or 2)
};

struct Wait {
  int32_t flag;      // semaphore index
  uint32_t per_run;  // posts the semaphore receives per chain run
};

// Number of semaphores the policy needs.
CUSYNC_HD int64_t num_flags(const DepCfg& d) {
  switch (d.policy) {
    case POL_TILE: return (int64_t)d.prod_m_tiles * d.prod_n_tiles;
    case POL_ROW: return d.prod_m_tiles;
    case POL_STRIDED: return (int64_t)d.prod_m_tiles * d.D;
    default: return 0;
  }
}

// Producer column tile visited at position y of a row.  RowMajor for every policy but
// StridedSync, whose prodOrder visits the G members of group 0 (columns 0, D, 2D, ...)
// first, then those of group 1, and so on.
CUSYNC_HD int32_t producer_col(const DepCfg& d, int32_t y) {
  if (d.policy == POL_STRIDED) return (y % d.G) * d.D + y / d.G;
  return y;
}

// Tile at position u of a stage's queue.  Row tiles are taken in groups of `raster`
// rows; inside a group the column position is the outer index and the row the inner
// one, so the CTAs working at the same time share a few weight column tiles and a few
// activation row tiles in L2.  raster = 1 is the RowMajor order of cuSync §IV-C;
// within every group the rows still complete in order.  Writes the row tile and the
// column position (which a policy may permute, see producer_col).
CUSYNC_HD void tile_at(const StageGeo& g, int32_t u, int32_t* m, int32_t* y) {
  const int32_t gm = g.raster < 1 ? 1 : g.raster;
  const int32_t per_group = gm * g.n_tiles;
  const int32_t grp = u / per_group;
  const int32_t rows = (g.m_tiles - grp * gm) < gm ? (g.m_tiles - grp * gm) : gm;
  const int32_t idx = u - grp * per_group;
  *y = idx / rows;
  *m = grp * gm + idx % rows;
}

// Semaphore the producer posts after finishing tile (m, c); -1 if the policy posts none.
CUSYNC_HD int32_t producer_flag(const DepCfg& d, int32_t m, int32_t c) {
  switch (d.policy) {
    case POL_TILE: return m * d.prod_n_tiles + c;
    case POL_ROW: return m;
    case POL_STRIDED: return m * d.D + (c % d.D);
    default: return -1;
  }
}

// Image-row range (in producer row tiles) read by consumer row tile m for filter row r.
CUSYNC_HD void conv_row_tiles(const StageGeo& g, int32_t m, int32_t r, int32_t* lo_tile, int32_t* hi_tile) {
  const int32_t n = m / g.tpi, hb = m % g.tpi;
  const int32_t p0 = hb * g.th;
  int32_t p1 = p0 + g.th - 1;
  if (p1 > g.img_h - 1) p1 = g.img_h - 1;
  int32_t lo = p0 + r - 1, hi = p1 + r - 1;  // 3x3, pad 1
  if (lo < 0) lo = 0;
  if (hi > g.img_h - 1) hi = g.img_h - 1;
  if (hi < lo) {  // a tile whose shifted window lies wholly outside the image
    *lo_tile = 0;
    *hi_tile = -1;
    return;
  }
  *lo_tile = n * g.tpi + lo / g.th;
  *hi_tile = n * g.tpi + hi / g.th;
}

// Tracks which producer tiles a consumer row tile has already waited for, and yields
// the semaphore waits needed before each A k-block, in the consumer's fixed natural
// k order.  Each producer tile is waited for once, when a k-block first reads it
// (TileSync), or with its whole group (StridedSync), or all rows up front before the
// first k-block (RowSync).  Sentinel and stream-ordered chains wait on no semaphore.
//
// GEMM chains: consumer k-block kb reads producer column tile c = kb*kBK / prod_n_out
// of its own row tile, so at most one wait per k-block and only the last column waited
// needs remembering (register state only).
// A work unit's k-blocks are visited in increasing order from its first one (k-block 0 for
// a whole tile, a later one for a K-split unit of a consumer tile).
struct GemmDepTracker {
  int32_t last_c;
  uint64_t groups;  // StridedSync: groups already waited for (D <= 64)
  CUSYNC_HD void reset() {
    last_c = -1;
    groups = 0;
  }
  CUSYNC_HD int next(const DepCfg& d, int32_t m, int32_t kb, Wait* out) {
    const int32_t pol = d.policy;
    const uint32_t pp = (uint32_t)d.posts;
    if (pol == POL_ROW) {  // the whole row, before the unit's first k-block
      if (last_c != -1) return 0;
      last_c = 0;
      out[0] = Wait{m, (uint32_t)d.prod_n_tiles * pp};
      return 1;
    }
    if (pol != POL_TILE && pol != POL_STRIDED) return 0;
    const int32_t c = (kb * kBK) / d.prod_n_out;
    if (c == last_c) return 0;
    last_c = c;
    if (pol == POL_TILE) {
      out[0] = Wait{m * d.prod_n_tiles + c, pp};
      return 1;
    }
    // StridedSync: column c belongs to group c mod D, waited for at its first touch (from
    // column 0 on, group g is first touched at column g)
    const int32_t grp = c % d.D;
    if (d.D <= 64) {
      if ((groups >> grp) & 1ull) return 0;
      groups |= 1ull << grp;
    } else if (c >= d.D) {
      return 0;  // whole tiles only (a K split of the consumer needs D <= 64)
    }
    out[0] = Wait{m * d.D + grp, (uint32_t)d.G * pp};
    return 1;
  }
};

// Convolution chains (halo): the producer row tiles a k-block reads depend on its filter
// row; per producer column tile, the row tiles already waited for form one interval.
struct ConvDepTracker {
  int32_t lo[kMaxConvColTiles];  // waited producer row-tile interval per column tile
  int32_t hi[kMaxConvColTiles];

  CUSYNC_HD void reset() {
    for (int i = 0; i < kMaxConvColTiles; ++i) {
      lo[i] = 1;
      hi[i] = 0;  // empty interval
    }
  }

  CUSYNC_HD int next(const StageGeo& cons, const DepCfg& d, int32_t m, int32_t kb, Wait* out) {
    const int32_t pol = d.policy;
    if (pol != POL_TILE && pol != POL_ROW && pol != POL_STRIDED) return 0;
    int n = 0;
    // k = (r*3 + s)*cin + channel
    const int32_t tap = kb / cons.cblocks, cb = kb % cons.cblocks;
    const int32_t r = tap / 3;
    if (pol == POL_ROW) {
      if (kb != 0) return 0;
      // union over the three filter rows (consecutive windows overlap or touch, so the
      // union is one interval of row tiles)
      int32_t a = 0x7FFFFFFF, b = -1;
      for (int32_t rr = 0; rr < 3; ++rr) {
        int32_t lo_t, hi_t;
        conv_row_tiles(cons, m, rr, &lo_t, &hi_t);
        if (hi_t < lo_t) continue;
        if (lo_t < a) a = lo_t;
        if (hi_t > b) b = hi_t;
      }
      for (int32_t mp = a; mp <= b && n < kMaxWaits; ++mp)
        out[n++] = Wait{mp, (uint32_t)(d.prod_n_tiles * d.posts)};
      return n;
    }
    const int32_t c = (cb * kBK) / d.prod_n_out;
    int32_t a, b;
    conv_row_tiles(cons, m, r, &a, &b);
    for (int32_t mp = a; mp <= b && n < kMaxWaits; ++mp) {
      if (lo[c] <= mp && mp <= hi[c]) continue;
      if (pol == POL_TILE) {
        out[n++] = Wait{mp * d.prod_n_tiles + c, (uint32_t)d.posts};
        if (lo[c] > hi[c]) { lo[c] = mp; hi[c] = mp; }
        else { if (mp < lo[c]) lo[c] = mp; if (mp > hi[c]) hi[c] = mp; }
      } else {  // StridedSync: the whole group of column c, for row tile mp
        out[n++] = Wait{mp * d.D + (c % d.D), (uint32_t)(d.G * d.posts)};
        for (int32_t cc = c % d.D; cc < d.prod_n_tiles; cc += d.D) {
          if (lo[cc] > hi[cc]) { lo[cc] = mp; hi[cc] = mp; }
          else { if (mp < lo[cc]) lo[cc] = mp; if (mp > hi[cc]) hi[cc] = mp; }
        }
      }
    }
    return n;
  }
};

// Whether consumer k-block kb can need a semaphore that no earlier k-block of its tile
// needed; the trackers are consulted only at these k-blocks (on the device and in the
// host introspection alike).  RowSync waits once, before k-block 0.  A GEMM k-block
// starts reading a new producer column tile every prod_n_out / kBK k-blocks.  A conv
// k-block (filter tap r*3+s, channel block cb) reads the producer row tiles of filter
// row r, which change only when s returns to 0, and producer column tile
// cb*kBK / prod_n_out, which changes every prod_n_out / kBK channel blocks.
// (A K-split unit of a consumer tile also consults the tracker at its first k-block.)
CUSYNC_HD bool dep_kblock(const StageGeo& cons, const DepCfg& d, int32_t kb) {
  const int32_t pol = d.policy;
  if (pol != POL_TILE && pol != POL_ROW && pol != POL_STRIDED) return false;
  if (pol == POL_ROW) return kb == 0;
  const int32_t per_col = d.prod_n_out / kBK > 1 ? d.prod_n_out / kBK : 1;
  if (cons.a_mode == AMODE_GEMM) return kb % per_col == 0;
  const int32_t tap = kb / cons.cblocks, cb = kb % cons.cblocks;
  return tap % 3 == 0 && cb % per_col == 0;
}

// Whether a work unit of a GEMM consumer (KB k-blocks from k-block kb0 of its tile)
// consults its tracker before its k-block kb (counted from the unit's first): RowSync at
// the unit's first k-block, TileSync and StridedSync at every k-block that starts a
// producer column tile.  The planner makes kb0 a multiple of that period
// (kb_per_split_alignment), so the unit's first k-block is always one of them; the
// loader evaluates the same test.
CUSYNC_HD bool unit_dep_kblock(const DepCfg& d, int32_t kb0, int32_t KB, int32_t kb) {
  const int32_t pol = d.policy;
  if (pol != POL_TILE && pol != POL_ROW && pol != POL_STRIDED) return false;
  (void)kb0;
  const int32_t every = pol == POL_ROW ? KB + 1 : (d.prod_n_out / kBK > 1 ? d.prod_n_out / kBK : 1);
  return (kb % every) == 0;
}

// K-block period that a consumer's K-split units must start on: the k-blocks of one
// producer column tile.
CUSYNC_HD int32_t kb_per_split_alignment(int32_t prod_n_out) { return prod_n_out / kBK > 1 ? prod_n_out / kBK : 1; }

// Semaphore waits of the attention chain's pointwise tile (m, i) (head i of row tile m) on
// the QKV GEMM, whose output row holds the Q, V and K blocks of width nq = 3 * D column
// tiles apart (D = producer column tiles per block): the head reads column tile
// c = i * kHead / prod_n_out of each block.  RowSync: the whole row tile; TileSync: the
// three tiles; StridedSync (G = 3, distance D): the one semaphore the three share.
CUSYNC_HD int pointwise_waits(const DepCfg& d, int32_t m, int32_t i, Wait* out) {
  const int32_t c = i * kHead / d.prod_n_out;
  const int32_t third = d.prod_n_tiles / 3;
  switch (d.policy) {
    case POL_ROW:
      out[0] = Wait{m, (uint32_t)(d.prod_n_tiles * d.posts)};
      return 1;
    case POL_TILE:
      for (int j = 0; j < 3; ++j) out[j] = Wait{m * d.prod_n_tiles + c + j * third, (uint32_t)d.posts};
      return 3;
    case POL_STRIDED:
      out[0] = Wait{m * d.D + (c % d.D), (uint32_t)(d.G * d.posts)};
      return 1;
    default:
      return 0;
  }
}

// Either tracker, chosen by the consumer's A operand (used by the host introspection).
struct DepTracker {
  GemmDepTracker gemm;
  ConvDepTracker conv;
  CUSYNC_HD void reset() {
    gemm.reset();
    conv.reset();
  }
  CUSYNC_HD int next(const StageGeo& cons, const DepCfg& d, int32_t m, int32_t kb, Wait* out) {
    return cons.a_mode == AMODE_GEMM ? gemm.next(d, m, kb, out) : conv.next(cons, d, m, kb, out);
  }
};

}  // namespace cusync
