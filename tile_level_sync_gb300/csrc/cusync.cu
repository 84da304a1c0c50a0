// Host side of the C ABI declared in include/cusync.h: argument validation, the wave
// planner, chain state, TMA descriptors and kernel launches.
//
// Sources: "A Framework for Fine-Grained Synchronization of Dependent GPU Kernels"
// (cuSync) §II-A (waves), §III-A (fused waves), §IV-A..C (launch on separate streams,
// stage processing order, tile processing order), §V (optimisations); CUDA Programming
// Guide §4.6 (sentinel protocol, programmatic dependent launch, §4.6.5 progress).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/cusync.h"
#include "chain_kernel.cuh"
#include "geometry.h"
#include "policy_model.h"

using namespace cusync;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // one second
// L2 prefetch lead of the weight boxes (k-blocks ahead of the loader) that the planner
// gives MLP chains on CTA pairs whose producer GEMM is K-split (the weight-streaming
// slices): 5-6% faster there; the other chains measured equal or slower with it.
constexpr int32_t kDefaultPrefetch = 4;

bool log_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = std::getenv("CUSYNC_LOG");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}

#define CUSYNC_LOG(...)                          \
  do {                                           \
    if (log_enabled()) {                         \
      std::fprintf(stderr, "[cusync] " __VA_ARGS__); \
      std::fprintf(stderr, "\n");                \
    }                                            \
  } while (0)

cusync_status_t cuda_fail(cudaError_t e, const char* what) {
  CUSYNC_LOG("%s: %s", what, cudaGetErrorString(e));
  return CUSYNC_ERR_CUDA;
}

// ----------------------------------------------------------------------------- planning

struct Plan {
  int32_t bn;           // accumulator tile width (UMMA N)
  int32_t pair;         // CTAs per tile: 1, or 2 (a CTA pair computing a 256-row tile)
  int32_t nst;          // stages: 2, 3 (attention: QKV GEMM, pointwise, output GEMM), or
                        // a convolution stack's depth
  StageGeo geo[3];      // per stage; a stack: geo[0] its first stage, geo[1] every later one
  int32_t stack;        // convolution stack (stages 1 .. nst-1 share geo[1] and `dep`)
  int32_t nbuf;         // stack: intermediate buffers in the workspace
  int32_t rotate;       // stack under the sentinel policy: two sets of buffers used in turn
  int64_t flags_stride; // stack: semaphores per stage boundary
  DepCfg dep;           // the last stage's waits on the stage before it (a stack: every stage's)
  DepCfg dep_pw;        // attention: the pointwise stage's waits on the QKV GEMM
  int64_t num_flags;
  int64_t num_flags_pw;
  int64_t split_rows;   // K split: workspace row blocks (producer tiles x pair), else 0
  int64_t split_rows1;  // K split of the consumer: its row blocks, else 0
  int32_t n_bands;      // MLP chains: row bands of the output with their own semaphore, else 0
};

// Row bands of an MLP chain's output: band b covers consumer row tiles
// [b * m_tiles / n_bands, (b + 1) * m_tiles / n_bands) (the kernel maps a row tile to its band
// with the inverse of this split).
constexpr int32_t kMaxBands = 16;
int32_t band_lo(int32_t m_tiles, int32_t n_bands, int32_t b) { return (int32_t)((int64_t)b * m_tiles / n_bands); }

// Geometry of stage s.
const StageGeo& sgeo(const Plan& p, int s) { return p.geo[p.stack ? (s > 0 ? 1 : 0) : s]; }

// Work units of all stages (trace records of a run).
int64_t total_units(const Plan& p) {
  int64_t n = 0;
  for (int s = 0; s < p.nst; ++s) n += stage_units(sgeo(p, s));
  return n;
}

// Elements of one intermediate of a convolution stack.
int64_t stack_buf_elems(const cusync_chain_desc_t& d) { return (int64_t)d.n * d.h * d.w * d.c; }

// Words of a chain's device state: control words, semaphores and band semaphores.
int64_t state_words(const Plan& p) {
  return CTRL_WORDS + p.num_flags + p.num_flags_pw + p.n_bands;
}
// fp32 elements of the K-split workspace: ksplit - 1 slots of a 128-row accumulator per
// row block.
int64_t split_ws_floats0(const Plan& p) { return p.split_rows * (int64_t)(p.geo[0].ksplit - 1) * 128 * (int64_t)p.bn; }
int64_t split_ws_floats(const Plan& p) {
  return split_ws_floats0(p) + p.split_rows1 * (int64_t)(p.geo[1].ksplit - 1) * 128 * (int64_t)p.bn;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Image rows per row tile of a convolution: the fewest tiles per image whose rows fit
// the 128-row UMMA tile, then the rows spread evenly over them.
int32_t conv_rows_per_tile(int32_t h, int32_t w) {
  const int32_t max_rows = kBM / w;
  const int32_t tpi = (int32_t)ceil_div(h, max_rows);
  return (int32_t)ceil_div(h, tpi);
}

int query_num_sms(int32_t requested, int* out);

int32_t default_tile_n(const cusync_chain_desc_t& d) {
  if (d.tile_n) return d.tile_n;
  // A single-CTA MLP chain whose producer tiles at width 256 would occupy at most a
  // sixteenth of the SMs is bound by the latency of a few tiles: 128-wide tiles double
  // their number (the 64-token chain of 256 x 1024 x 256: 19.0 against 22.7 us, RowSync).
  const bool mlp = d.kind == CUSYNC_CHAIN_MLP_GELU || d.kind == CUSYNC_CHAIN_MLP_SWIGLU;
  const bool single = d.cta_pair == 1 || (d.cta_pair == 0 && d.M < 256);
  if (mlp && single && d.M > 0 && d.N1 > 0) {
    int sms = 0;
    if (query_num_sms(d.num_sms, &sms) != 0) sms = 148;
    const int64_t tiles = ((d.M + 127) / 128) * ((d.N1 + 255) / 256);
    if (16 * tiles <= sms) return 128;
  }
  return 256;
}

cusync_status_t resolve_auto(const cusync_chain_desc_t& d, cusync_chain_desc_t* out);

// Planner's graded split of a K-split producer on CTA pairs: each unit 8 k-blocks longer
// than the one before it (units shorter than 32 k-blocks: a quarter of one, even, at
// least 2).  Measured against equal units, same box: GPT-3 M=256 MLP slice (3 units of
// 64 k-blocks) 75.9 against 77.7 us, SwiGLU M=256 (2 x 64) 57.3 against 59.2, GPT-3 M=512
// (2 x 96, two waves) 120.1 against 123.8, GPT-3 attention M=256 (4 x 48) 78.4 against
// 82.9; skews of 4, 6, 10, 12 and 16 measured slower than 8 on the first and the last,
// 12 equal on the third.
int32_t default_split_skew(int32_t k_blocks, int32_t ksplit) {
  const int32_t per = k_blocks / ksplit;
  return std::max(2, std::min(8, per / 4) & ~1);
}

cusync_status_t make_plan(const cusync_chain_desc_t& d, Plan* p) {
  if (d.kind < CUSYNC_CHAIN_MLP_GELU || d.kind > CUSYNC_CHAIN_CONV_STACK) return CUSYNC_ERR_INVALID_ARG;
  if (d.policy == CUSYNC_POLICY_AUTO) {
    cusync_chain_desc_t r;
    cusync_status_t st = resolve_auto(d, &r);
    return st != CUSYNC_OK ? st : make_plan(r, p);
  }
  if (d.policy < CUSYNC_POLICY_STREAM || d.policy > CUSYNC_POLICY_SENTINEL) return CUSYNC_ERR_INVALID_ARG;
  if (d.launch != CUSYNC_LAUNCH_PERSISTENT && d.launch != CUSYNC_LAUNCH_PDL) return CUSYNC_ERR_INVALID_ARG;
  const int32_t bn = default_tile_n(d);
  if (bn != 128 && bn != 192 && bn != 256) return CUSYNC_ERR_UNSUPPORTED;
  const bool mlp = d.kind == CUSYNC_CHAIN_MLP_GELU || d.kind == CUSYNC_CHAIN_MLP_SWIGLU;
  const bool attn = d.kind == CUSYNC_CHAIN_ATTENTION;
  const bool stack = d.kind == CUSYNC_CHAIN_CONV_STACK;
  // CTA pairs (cta_group::2, 256-row tiles) for MLP and attention chains with at least
  // 256 tokens, where they measured faster on GB300 (GPT-3 MLP M=256: 91 against 97 us;
  // SwiGLU M=256 even; GPT-3 attention M=1024: 148.6 against 155.1 us, M=256 84.1 against
  // 85.9 us); single-CTA 128-row tiles otherwise.
  const int32_t pair = d.cta_pair ? d.cta_pair : (((mlp || attn) && d.M >= 256) ? 2 : 1);
  if (pair != 1 && pair != 2) return CUSYNC_ERR_INVALID_ARG;
  if (pair == 2 && !mlp && !attn) return CUSYNC_ERR_UNSUPPORTED;  // (convolutions: single CTAs)
  // 192-wide tiles: GeLU MLP chains on CTA pairs (a SwiGLU tile would write 96 columns, not
  // whole 64-column store boxes)
  if (bn == 192 && (pair != 2 || d.kind != CUSYNC_CHAIN_MLP_GELU)) return CUSYNC_ERR_UNSUPPORTED;
  std::memset(p, 0, sizeof(*p));
  p->bn = bn;
  p->pair = pair;
  StageGeo& g0 = p->geo[0];
  StageGeo& g1 = p->geo[1];
  StageGeo& g2 = p->geo[2];
  p->nst = attn ? 3 : 2;
  if (stack) {
    // [cuSync] Table tab:resnet-sizes: a ResNet-38 layer group is a run of 3x3
    // convolutions of equal channels; here `stages` of them in one chain
    if (d.n < 1 || d.h < 1 || d.w < 1 || d.c < 1 || d.stages < 1) return CUSYNC_ERR_INVALID_ARG;
    if (d.stages < 2 || d.stages > kMaxQueues) return CUSYNC_ERR_UNSUPPORTED;
    if (d.k_out != 0 && d.k_out != d.c) return CUSYNC_ERR_UNSUPPORTED;   // equal channels
    if (d.policy == CUSYNC_POLICY_STRIDED_TILE) return CUSYNC_ERR_UNSUPPORTED;
    if (d.c % kBK) return CUSYNC_ERR_UNSUPPORTED;
    if (d.w > kBM || d.w > 256) return CUSYNC_ERR_UNSUPPORTED;
    if ((int64_t)d.n * d.h * d.w > (1ll << 30)) return CUSYNC_ERR_UNSUPPORTED;
    if (ceil_div(d.c, bn) > kMaxConvColTiles) return CUSYNC_ERR_UNSUPPORTED;
    const int32_t th = conv_rows_per_tile(d.h, d.w);
    for (int s = 0; s < 2; ++s) {
      StageGeo& g = p->geo[s];
      g.a_mode = AMODE_CONV;
      g.epi = EPI_RELU;  // the kernel applies none after the last convolution
      g.M = d.n * d.h * d.w;
      g.N = d.c;
      g.K = 9 * d.c;
      g.n_out = bn;
      g.img_n = d.n;
      g.img_h = d.h;
      g.img_w = d.w;
      g.cin = d.c;
      g.th = th;
      g.tpi = (int32_t)ceil_div(d.h, th);
      g.cblocks = d.c / kBK;
      g.m_tiles = d.n * g.tpi;
      g.n_tiles = (int32_t)ceil_div(d.c, bn);
      g.k_blocks = 9 * g.cblocks;
    }
    p->nst = d.stages;
    p->stack = 1;
  } else if (attn) {
    // "A Framework for Fine-Grained Synchronization of Dependent GPU Kernels",
    // Fig. fig:gpt-3:attention: XQKV = X x QKV (one GEMM for the three blocks), the
    // pointwise dot-product kernel per head, XW2 = XDot x W2.
    if (d.M < 1 || d.K < 1 || d.N1 < 1 || d.N2 < 1) return CUSYNC_ERR_INVALID_ARG;
    if (d.K % 8 || d.N2 % 8 || d.N1 % bn || d.N1 % kHead) return CUSYNC_ERR_UNSUPPORTED;
    if (d.policy == CUSYNC_POLICY_SENTINEL) return CUSYNC_ERR_UNSUPPORTED;
    if (d.M > (1ll << 30) || d.K > (1ll << 30) || 3 * d.N1 > (1ll << 30) || d.N2 > (1ll << 30))
      return CUSYNC_ERR_UNSUPPORTED;
    g0.a_mode = AMODE_GEMM;
    g0.epi = EPI_NONE;
    g0.M = (int32_t)d.M;
    g0.N = (int32_t)(3 * d.N1);
    g0.K = (int32_t)d.K;
    g0.n_out = bn;
    g1.a_mode = AMODE_POINTWISE;
    g1.epi = EPI_NONE;
    g1.M = (int32_t)d.M;
    g1.N = (int32_t)d.N1;
    g1.K = (int32_t)(3 * d.N1);  // row length of the XQKV input
    g1.n_out = kHead;
    g2.a_mode = AMODE_GEMM;
    g2.epi = EPI_NONE;
    g2.M = (int32_t)d.M;
    g2.N = (int32_t)d.N2;
    g2.K = (int32_t)d.N1;
    g2.n_out = bn;
    for (StageGeo* g : {&g0, &g1, &g2}) {
      g->m_tiles = (int32_t)ceil_div(g->M, (int64_t)kBM * pair);
      g->n_tiles = (int32_t)ceil_div(g->N, g->n_out);
      g->k_blocks = g->a_mode == AMODE_POINTWISE ? 0 : (int32_t)ceil_div(g->K, kBK);
    }
  } else if (d.kind == CUSYNC_CHAIN_MLP_GELU || d.kind == CUSYNC_CHAIN_MLP_SWIGLU) {
    if (d.M < 1 || d.K < 1 || d.N1 < 1 || d.N2 < 1) return CUSYNC_ERR_INVALID_ARG;
    // TMA row strides and 16-byte output chunks need multiples of 8 bf16 elements.
    if (d.K % 8 || d.N1 % 8 || d.N2 % 8) return CUSYNC_ERR_UNSUPPORTED;
    if (d.M > (1ll << 30) || d.K > (1ll << 30) || d.N1 > (1ll << 30) || d.N2 > (1ll << 30))
      return CUSYNC_ERR_UNSUPPORTED;
    const bool swiglu = d.kind == CUSYNC_CHAIN_MLP_SWIGLU;
    g0.a_mode = AMODE_GEMM;
    g0.epi = swiglu ? EPI_SWIGLU : EPI_GELU;
    g0.M = (int32_t)d.M;
    g0.N = (int32_t)d.N1;
    g0.K = (int32_t)d.K;
    g0.n_out = swiglu ? bn / 2 : bn;
    g1.a_mode = AMODE_GEMM;
    g1.epi = EPI_NONE;
    g1.M = (int32_t)d.M;
    g1.N = (int32_t)d.N2;
    g1.K = (int32_t)d.N1;
    g1.n_out = bn;
    for (StageGeo* g : {&g0, &g1}) {
      g->m_tiles = (int32_t)ceil_div(g->M, (int64_t)kBM * pair);
      g->n_tiles = (int32_t)ceil_div(g->N, g->n_out);
      g->k_blocks = (int32_t)ceil_div(g->K, kBK);
    }
  } else {
    if (d.n < 1 || d.h < 1 || d.w < 1 || d.c < 1 || d.k_out < 1) return CUSYNC_ERR_INVALID_ARG;
    if (d.c % kBK || d.k_out % kBK) return CUSYNC_ERR_UNSUPPORTED;  // whole channel blocks per tap
    if (d.w > kBM || d.w > 256) return CUSYNC_ERR_UNSUPPORTED;       // one image row per box row run
    if ((int64_t)d.n * d.h * d.w > (1ll << 30)) return CUSYNC_ERR_UNSUPPORTED;
    if (ceil_div(d.k_out, bn) > kMaxConvColTiles) return CUSYNC_ERR_UNSUPPORTED;
    const int32_t th = conv_rows_per_tile(d.h, d.w);
    const int32_t tpi = (int32_t)ceil_div(d.h, th);
    const int32_t cins[2] = {d.c, d.k_out};
    for (int s = 0; s < 2; ++s) {
      StageGeo& g = p->geo[s];
      g.a_mode = AMODE_CONV;
      g.epi = s == 0 ? EPI_RELU : EPI_NONE;
      g.M = d.n * d.h * d.w;
      g.N = d.k_out;
      g.K = 9 * cins[s];
      g.n_out = bn;
      g.img_n = d.n;
      g.img_h = d.h;
      g.img_w = d.w;
      g.cin = cins[s];
      g.th = th;
      g.tpi = tpi;
      g.cblocks = cins[s] / kBK;
      g.m_tiles = d.n * tpi;
      g.n_tiles = (int32_t)ceil_div(d.k_out, bn);
      g.k_blocks = 9 * g.cblocks;
    }
  }
  // Tile order.  0 = planner: an MLP chain on CTA pairs with at least four row tiles takes
  // them in groups of half its row tiles (tile_at: columns outer, rows inner in a group),
  // so the CTAs running at the same time share each weight column tile and HBM delivers
  // it once per group instead of once per row tile: GPT-3 slices at M = 1024, 2048, 4096
  // measured 203.9 / 361.6 / 694.4 us against 215.0 / 391.6 / 744.7 us row-major (groups of
  // 2, 4 and 8), the SwiGLU M = 1024 chain 118.4 against 121.3 us.  The two halves of the
  // producer rows still complete one after the other, so RowSync consumers of the first
  // half start while the second is produced.  Otherwise (and for chains with row bands,
  // whose band semaphores need row-major order) one row tile per group.
  int32_t raster = d.raster_rows;
  if (raster == 0) {
    raster = 1;
    if (mlp && pair == 2 && d.bands == 0 && g0.m_tiles >= 4) raster = g0.m_tiles / 2;
  }
  g0.raster = raster < g0.m_tiles ? raster : g0.m_tiles;
  g1.raster = raster < g1.m_tiles ? raster : g1.m_tiles;
  g2.raster = raster < g2.m_tiles ? raster : g2.m_tiles;
  // K split of the producer GEMM (see cusync_chain_desc_t::ksplit)
  if (d.ksplit < 0 || d.ksplit > 16) return CUSYNC_ERR_INVALID_ARG;
  int32_t ks = d.ksplit;
  if (ks == 0) {
    ks = 1;
    if (mlp || attn) {
      int sms = 0;
      if (query_num_sms(d.num_sms, &sms) != 0) sms = 148;
      // Producer tiles that fill at most half of a wave: as many units per tile as fit in
      // the wave (at most 4, at least 16 k-blocks each).  Tiles that fill more than half
      // of it: 2 units per tile, whose second wave the fused queue fills with consumer
      // tiles (measured faster on GB300, e.g. the M=512 GPT-3 MLP slice).
      const int64_t slots = sms / pair;
      const int64_t t0 = (int64_t)g0.m_tiles * g0.n_tiles;
      int64_t want = 1;
      if (t0 > 0 && 2 * t0 <= slots) want = std::min<int64_t>(slots / t0, 4);
      else if (t0 > 0 && t0 <= slots) want = 2;
      ks = (int32_t)std::max<int64_t>(1, std::min<int64_t>(want, g0.k_blocks / 16));
    }
  }
  if (ks > 1 && !mlp && !attn) return CUSYNC_ERR_UNSUPPORTED;
  if (ks > g0.k_blocks) return CUSYNC_ERR_UNSUPPORTED;
  g0.ksplit = ks;
  g0.kb_per_split = (int32_t)ceil_div(g0.k_blocks, ks);
  g0.ksplit = (int32_t)ceil_div(g0.k_blocks, g0.kb_per_split);  // no empty unit
  // Graded split (cusync_chain_desc_t::ksplit_skew): each unit kb_skew k-blocks longer
  // than the one before it, so that the units finish one after the other and each
  // unit's exchange overlaps the mainloops of the units after it.
  if (d.ksplit_skew < -1 || d.ksplit_skew > 64) return CUSYNC_ERR_INVALID_ARG;
  int32_t skew = d.ksplit_skew;
  if (skew == 0) skew = ((mlp || attn) && pair == 2 && g0.ksplit > 1) ? default_split_skew(g0.k_blocks, g0.ksplit) : -1;
  if (skew > 0 && g0.ksplit > 1) {
    const int32_t S = g0.ksplit;
    const int32_t base = (g0.k_blocks - skew * (S * (S - 1) / 2)) / S;
    if (base < 1) return CUSYNC_ERR_UNSUPPORTED;
    g0.kb_per_split = base;
    g0.kb_skew = skew;
  }
  // K split of the consumer GEMM of an MLP chain (cusync_chain_desc_t::ksplit_consumer):
  // single-CTA consumer tiles that fill at most half of a wave get as many units per tile
  // as fit in one wave (at most 4, at least 16 k-blocks each).  CTA pairs keep whole
  // consumer tiles: with their two-k-block copies the SwiGLU M=256 slice (32 pair tiles
  // of 56 k-blocks) measured 60.7 us unsplit against 61.7 us with two units, and the
  // GPT-3 M=256 and M=512 slices 4-9% slower with three units.
  if (d.ksplit_consumer < 0 || d.ksplit_consumer > 16) return CUSYNC_ERR_INVALID_ARG;
  int32_t ks1 = d.ksplit_consumer;
  if (ks1 == 0) {
    ks1 = 1;
    if (mlp && pair == 1) {
      int sms = 0;
      if (query_num_sms(d.num_sms, &sms) != 0) sms = 148;
      const int64_t slots = std::max<int64_t>(1, sms / pair);
      const int64_t t1 = (int64_t)g1.m_tiles * g1.n_tiles;
      if (t1 > 0 && 2 * t1 <= slots)
        ks1 = (int32_t)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(slots / t1, 4), g1.k_blocks / 16));
    }
  }
  if (ks1 > 1 && !mlp) return CUSYNC_ERR_UNSUPPORTED;
  if (ks1 > 1 && ks1 > g1.k_blocks) return CUSYNC_ERR_UNSUPPORTED;
  g1.ksplit = 1;
  g1.kb_per_split = g1.k_blocks;
  if (ks1 > 1) {
    // units start on producer column tiles (kb_per_split_alignment), no empty unit
    const int32_t al = kb_per_split_alignment(g0.n_out);
    g1.kb_per_split = (int32_t)(ceil_div(ceil_div(g1.k_blocks, ks1), al) * al);
    g1.ksplit = (int32_t)ceil_div(g1.k_blocks, g1.kb_per_split);
  }
  g2.ksplit = 1;
  g2.kb_per_split = g2.k_blocks;
  // row bands of the output (MLP chains; cusync_chain_desc_t::bands)
  if (d.bands < 0) return CUSYNC_ERR_INVALID_ARG;
  if (d.bands > 0) {
    if (!mlp || d.bands > kMaxBands || d.bands > g1.m_tiles) return CUSYNC_ERR_UNSUPPORTED;
    if (g1.raster > 1) return CUSYNC_ERR_UNSUPPORTED;  // a band's tiles are consecutive in row-major order
    p->n_bands = d.bands;
  }
  if (d.l2_prefetch < -1 || d.l2_prefetch > 64) return CUSYNC_ERR_INVALID_ARG;
  if (attn) {
    // the pointwise stage waits on the QKV GEMM: StridedSync with G = 3 (the Q, V and K
    // tiles of a head share one semaphore), or RowSync / TileSync; the output GEMM waits on
    // the pointwise stage: TileSync (also under StridedSync, as in the pages'
    // Strided+TileSync), or RowSync
    DepCfg& dp = p->dep_pw;
    dp.policy = d.policy;
    dp.prod_m_tiles = g0.m_tiles;
    dp.prod_n_tiles = g0.n_tiles;
    dp.prod_n_out = g0.n_out;
    dp.G = 1;
    dp.D = g0.n_tiles;
    dp.posts = pair;
    if (d.policy == CUSYNC_POLICY_STRIDED_TILE) {
      if (g0.n_tiles % 3) return CUSYNC_ERR_UNSUPPORTED;
      dp.G = 3;
      dp.D = g0.n_tiles / 3;
    }
    DepCfg& dep = p->dep;
    dep.policy = d.policy == CUSYNC_POLICY_STRIDED_TILE ? CUSYNC_POLICY_TILE : d.policy;
    dep.prod_m_tiles = g1.m_tiles;
    dep.prod_n_tiles = g1.n_tiles;
    dep.prod_n_out = g1.n_out;
    dep.G = 1;
    dep.D = g1.n_tiles;
    dep.posts = pair;  // each CTA of a pair posts its 128 rows of the pointwise tile
    p->num_flags = num_flags(dep);
    p->num_flags_pw = num_flags(dp);
    if (p->num_flags + p->num_flags_pw > (1ll << 24)) return CUSYNC_ERR_UNSUPPORTED;
    p->split_rows = g0.ksplit > 1 ? (int64_t)g0.m_tiles * g0.n_tiles * pair : 0;
    return CUSYNC_OK;
  }
  DepCfg& dep = p->dep;
  dep.policy = d.policy;
  dep.prod_m_tiles = g0.m_tiles;
  dep.prod_n_tiles = g0.n_tiles;
  dep.prod_n_out = g0.n_out;
  dep.G = 1;
  dep.D = g0.n_tiles;
  dep.posts = pair;
  if (d.policy == CUSYNC_POLICY_STRIDED_TILE) {
    const int32_t G = d.strided_group ? d.strided_group : 2;
    if (G < 1 || g0.n_tiles % G) return CUSYNC_ERR_UNSUPPORTED;
    dep.G = G;
    dep.D = g0.n_tiles / G;
  }
  if (g1.ksplit > 1 && dep.policy == POL_STRIDED && dep.D > 64) {
    // a StridedSync unit remembers its waited groups in 64 bits
    if (d.ksplit_consumer > 1) return CUSYNC_ERR_UNSUPPORTED;
    g1.ksplit = 1;
    g1.kb_per_split = g1.k_blocks;
  }
  p->split_rows1 = g1.ksplit > 1 ? (int64_t)g1.m_tiles * g1.n_tiles * pair : 0;
  p->num_flags = num_flags(dep);
  if (stack) {
    // one set of semaphores per stage boundary; the intermediates alternate between two
    // buffers, except under the sentinel policy
    p->flags_stride = p->num_flags;
    p->num_flags = p->flags_stride * (p->nst - 1);
    // under the sentinel policy one buffer per intermediate, in two sets that alternate
    // between runs: each run's last launch writes the sentinel over the other set
    // ([CUDA-FGS] §4.6.4.5 "Buffer Reuse"), so no fill precedes a run
    p->rotate = d.policy == CUSYNC_POLICY_SENTINEL ? 1 : 0;
    p->nbuf = p->rotate ? 2 * (p->nst - 1) : std::min(2, p->nst - 1);
  }
  if (p->num_flags > (1ll << 24)) return CUSYNC_ERR_UNSUPPORTED;
  p->split_rows = g0.ksplit > 1 ? (int64_t)g0.m_tiles * g0.n_tiles * pair : 0;
  return CUSYNC_OK;
}

int query_num_sms(int32_t requested, int* out) {
  if (requested > 0) {
    *out = requested;
    return 0;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  *out = sms;
  return 0;
}

// ----------------------------------------------------------------------------- TMA maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

bool load_encoder() {
  std::lock_guard<std::mutex> lk(g_encode_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// cuStreamWaitValue32 (driver API) through the runtime's entry-point query.
PFN_cuStreamWaitValue32_v11070 g_wait_value = nullptr;

bool load_wait_value() {
  std::lock_guard<std::mutex> lk(g_encode_mu);
  if (g_wait_value) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_wait_value = reinterpret_cast<PFN_cuStreamWaitValue32_v11070>(fn);
  return true;
}

// 2-D row-major bf16 [rows, cols] with a [box_rows, 64] box, 128-byte swizzle.
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D NHWC bf16 image [n, h, w, c] with a [1, th, w, 64] box (all of an image row run,
// one 64-channel block), 128-byte swizzle; out-of-image elements read as zero.
bool encode_nhwc(CUtensorMap* m, const void* ptr, uint64_t n, uint64_t h, uint64_t w, uint64_t c, uint32_t th) {
  cuuint64_t dims[4] = {c, w, h, n};
  cuuint64_t strides[3] = {c * 2, w * c * 2, h * w * c * 2};
  cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)w, th, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A convolution stack's intermediates: `nbuf` NHWC images one after the other, as a 5-D
// map [nbuf, n, h, w, c] whose outermost coordinate selects the buffer; same box.
bool encode_nhwc_bufs(CUtensorMap* m, const void* ptr, uint64_t nbuf, uint64_t n, uint64_t h, uint64_t w, uint64_t c,
                      uint32_t th) {
  cuuint64_t dims[5] = {c, w, h, n, nbuf};
  cuuint64_t strides[4] = {c * 2, w * c * 2, h * w * c * 2, n * h * w * c * 2};
  cuuint32_t box[5] = {(cuuint32_t)kBK, (cuuint32_t)w, th, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A convolution stack's weights: `depth` row-major [rows, cols] matrices one after the
// other, as a 3-D map whose outermost coordinate selects the stage; [box_rows, 64] box.
bool encode_3d(CUtensorMap* m, const void* ptr, uint64_t depth, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[3] = {cols, rows, depth};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)kBK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D row-major bf16 [rows, cols] seen as 3-D [cols/64][rows][64] (cols a multiple of 64):
// a {64, box_rows, kps} box brings kps consecutive 64-column k-blocks of box_rows rows,
// laid out in shared memory one k-block after the other, each as a 2-D box would be.
bool encode_kview(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t kps) {
  cuuint64_t dims[3] = {(cuuint64_t)kBK, rows, cols / kBK};
  cuuint64_t strides[2] = {cols * 2, (cuuint64_t)kBK * 2};
  cuuint32_t box[3] = {(cuuint32_t)kBK, box_rows, kps};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A GEMM operand's map: the k-block view when the kernel's stages hold two k-blocks and
// the reduction length is a whole number of k-blocks (*kview = 1), else the 2-D map.
bool encode_operand(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, int32_t kps,
                    int32_t* kview) {
  *kview = (kps > 1 && cols % kBK == 0) ? 1 : 0;
  return *kview ? encode_kview(m, ptr, rows, cols, box_rows, (uint32_t)kps) : encode_2d(m, ptr, rows, cols, box_rows);
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int BN, int PAIR, bool CHECK>
cudaError_t set_kernel_attrs() {
  cudaError_t e = cudaFuncSetAttribute(chain_kernel<BN, PAIR, CHECK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       KCfg<BN, PAIR>::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chain_kernel<BN, PAIR, CHECK>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // Load the kernel now rather than at its first launch (CUDA-FGS §4.6.5, "Overlap").
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, chain_kernel<BN, PAIR, CHECK>);
}

template <bool CHECK>
cudaError_t set_kernel_attrs_all_tiles() {
  cudaError_t e = set_kernel_attrs<256, 1, CHECK>();
  if (e == cudaSuccess) e = set_kernel_attrs<128, 1, CHECK>();
  if (e == cudaSuccess) e = set_kernel_attrs<256, 2, CHECK>();
  if (e == cudaSuccess) e = set_kernel_attrs<192, 2, CHECK>();
  if (e == cudaSuccess) e = set_kernel_attrs<128, 2, CHECK>();
  return e;
}

cudaError_t set_all_kernel_attrs() {
  cudaError_t e = set_kernel_attrs_all_tiles<false>();
  if (e == cudaSuccess) e = set_kernel_attrs_all_tiles<true>();
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, sentinel_fill_kernel);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, band_release_kernel);
  return e;
}

// Clusters of two CTAs that can be resident at once (pair kernels), for the current device:
// the fewer of the instantiations with and without the sentinel checkers.
template <int BN, bool CHECK>
int max_pair_clusters_of() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(KCfg<BN, 2>::threads(CHECK));
  cfg.dynamicSmemBytes = KCfg<BN, 2>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, chain_kernel<BN, 2, CHECK>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int BN>
int max_pair_clusters() {
  return std::min(max_pair_clusters_of<BN, false>(), max_pair_clusters_of<BN, true>());
}

// Grid sizes (CTAs) of the fused launch and of the two separate launches.
struct Grids {
  int32_t fused;     // the one persistent launch of all stages
  int32_t stage[kMaxQueues];  // one launch per stage (stream order or programmatic dependent launch)
};

Grids make_grids(const Plan& p, int sms, int max_clusters) {
  int64_t t[kMaxQueues] = {}, total = 0;
  for (int s = 0; s < p.nst; ++s) total += (t[s] = stage_units(sgeo(p, s)));
  // one tile per CTA, or per CTA pair (cluster of two) resident at once
  const int64_t slots = p.pair == 2 ? std::max<int64_t>(1, std::min<int64_t>(sms / 2, max_clusters > 0 ? max_clusters
                                                                                                       : sms / 2))
                                    : sms;
  Grids g;
  g.fused = (int32_t)(p.pair * std::min<int64_t>(slots, total));
  for (int s = 0; s < kMaxQueues; ++s) g.stage[s] = (int32_t)(p.pair * std::min<int64_t>(slots, t[s]));
  return g;
}

// ----------------------------------------------------------------------------- latency model

// GB300 constants of the latency model for plan p, from the in-kernel trace of the bench
// workloads: mainloop ns per k-block (single CTAs 345-375; CTA pairs, whose stages of
// two k-blocks take one copy per operand, 320-360 per pair k-block; convolutions
// 355-400), a consumer
// k-block under the sentinel check once its data is valid (420-440 ns: two checker warps
// scan alternate stages), a tile's first copy about 1 us,
// the post seen by a consumer about 1.5 us after the stores, 2 us between stream-ordered
// kernels, and epilogue time per output column by activation (tanh-GeLU 22 ns, SwiGLU
// 26 ns, ReLU 22 ns, none 17 ns for a 128-row tile).
// Per-tile costs, from the same traces: a CTA's next tile starts its mainloop 2.2-2.9 us
// after the previous one's last k-block (stacks and the GPT-3 M = 1024 slice alike), and a
// consumer tile's first semaphore consult costs 1.8 us (CTA pairs) to 2.6 us (convolution
// tiles) even when the semaphores are already posted.
LatencyModel default_model(const Plan& p) {
  LatencyModel m;
  const bool conv = p.geo[0].a_mode == AMODE_CONV;
  if (conv) {
    m.kblock_ns[0] = 375.0;
    m.kblock_ns[1] = 375.0;
    m.sentinel_kblock_ns = 500.0;
    m.tile_ns = 2500.0;
    m.tile_wait_ns = 2600.0;
  } else if (p.pair == 2) {
    m.kblock_ns[0] = 340.0;
    m.kblock_ns[1] = 330.0;
    m.sentinel_kblock_ns = 435.0;
    m.tile_ns = 2700.0;
    m.tile_wait_ns = 1800.0;
  } else {
    m.kblock_ns[0] = p.bn == 128 ? 355.0 : 350.0;
    m.kblock_ns[1] = p.bn == 128 ? 365.0 : 370.0;
    m.sentinel_kblock_ns = 440.0;
    m.tile_ns = 2500.0;
    m.tile_wait_ns = 2000.0;
  }
  m.wait_kblock_ns = 150.0;
  m.start_ns = 1000.0;
  for (int s = 0; s < 2; ++s) {
    double per_col = 17.0;
    switch (p.geo[s].epi) {
      case EPI_GELU: per_col = 22.0; break;
      case EPI_SWIGLU: per_col = 26.0; break;
      case EPI_RELU: per_col = 22.0; break;
      default: break;
    }
    m.epilogue_ns[s] = per_col * p.geo[s].n_out;
  }
  m.post_ns = 1500.0;
  m.gap_ns = 2000.0;
  m.fill_ns_per_mb = 350.0;
  return m;
}

// Predicted us of one run under each policy (-1 where the plan is refused).
void predict_all(const cusync_chain_desc_t& d, const cusync_latency_model_t* model, int sms, double us[5]) {
  for (int pol = CUSYNC_POLICY_STREAM; pol <= CUSYNC_POLICY_SENTINEL; ++pol) {
    cusync_chain_desc_t c = d;
    c.policy = (cusync_policy_t)pol;
    c.ksplit_consumer = 1;  // the model plays whole consumer tiles
    Plan q;
    if (make_plan(c, &q) != CUSYNC_OK || (q.nst != 2 && !q.stack)) {  // two-stage chains and stacks
      us[pol] = -1.0;
      continue;
    }
    LatencyModel lm;
    if (model) std::memcpy(&lm, model, sizeof(lm));
    else lm = default_model(q);
    const Grids g = make_grids(q, sms, 0);
    if (q.stack) {
      ModelStack ms;
      ms.geo[0] = q.geo[0];
      ms.geo[1] = q.geo[1];
      ms.dep = q.dep;
      ms.stages = q.nst;
      ms.slots_fused = g.fused;
      ms.slots_stage = g.stage[0];
      ms.fill_units = 0;
      if (q.rotate) {
        const int64_t set_chunks = (int64_t)(q.nst - 1) * stack_buf_elems(c) / 8;
        ms.fill_units = (int32_t)ceil_div(set_chunks, 4096);
      }
      us[pol] = predict_stack_ns(ms, lm) / 1000.0;
      continue;
    }
    ModelChain mc;
    mc.geo[0] = q.geo[0];
    mc.geo[1] = q.geo[1];
    mc.dep = q.dep;
    mc.slots_fused = g.fused / q.pair;
    mc.slots[0] = g.stage[0] / q.pair;
    mc.slots[1] = g.stage[1] / q.pair;
    mc.h_mb = (double)q.geo[0].M * (double)q.geo[0].N * 2.0 / 1e6;
    us[pol] = predict_chain_ns(mc, lm) / 1000.0;
  }
}

cusync_status_t resolve_auto(const cusync_chain_desc_t& d, cusync_chain_desc_t* out) {
  int sms = 0;
  if (query_num_sms(d.num_sms, &sms) != 0) return CUSYNC_ERR_CUDA;
  double us[5];
  predict_all(d, nullptr, sms, us);
  int best = -1;
  for (int pol = CUSYNC_POLICY_STREAM; pol <= CUSYNC_POLICY_SENTINEL; ++pol)
    if (us[pol] >= 0.0 && (best < 0 || us[pol] < us[best])) best = pol;
  if (best < 0) return CUSYNC_ERR_UNSUPPORTED;
  *out = d;
  out->policy = (cusync_policy_t)best;
  return CUSYNC_OK;
}

// B box rows per CTA: BN (single), BN/2 (pair, or either SwiGLU half).
uint32_t b_box_rows(const Plan& p, bool swiglu) { return (uint32_t)((swiglu || p.pair == 2) ? p.bn / 2 : p.bn); }

}  // namespace

// ----------------------------------------------------------------------------- chain

struct cusync_chain {
  cusync_chain_desc_t d;
  Plan plan;
  int device;
  int num_sms;
  uint32_t* state;       // CTRL_WORDS control words and the semaphores
  float* split_ws;       // K-split fp32 workspace, or null
  TraceRec* trace;       // per-tile timeline (CUSYNC_FLAG_TRACE), or null
  Grids grids;
  // TMA descriptors cached by operand pointers
  const void* cached[6];
  bool maps_valid;
  ChainArgs args;
  const void* filled_ws;  // rotating sentinel stack: the workspace whose sets hold the sentinel
  bool need_fill;         // rotating sentinel stack: fill both sets before the next run
  cudaEvent_t band_ev;    // row bands: recorded after the band semaphores are cleared for a run
  bool bands_ready;       // row bands: a run with band semaphores was enqueued (band waits allowed)
};

namespace {

template <int BN, int PAIR, bool CHECK>
cudaError_t launch_chain(const ChainArgs& a, int grid, bool pdl_secondary, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(KCfg<BN, PAIR>::threads(CHECK));
  cfg.dynamicSmemBytes = KCfg<BN, PAIR>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR == 2) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl_secondary) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, chain_kernel<BN, PAIR, CHECK>, a);
}

template <bool CHECK>
cudaError_t launch_tiles(const Plan& p, const ChainArgs& a, int grid, bool pdl2, cudaStream_t s) {
  if (p.pair == 2) {
    if (p.bn == 192) return launch_chain<192, 2, CHECK>(a, grid, pdl2, s);
    return p.bn == 256 ? launch_chain<256, 2, CHECK>(a, grid, pdl2, s) : launch_chain<128, 2, CHECK>(a, grid, pdl2, s);
  }
  return p.bn == 256 ? launch_chain<256, 1, CHECK>(a, grid, pdl2, s) : launch_chain<128, 1, CHECK>(a, grid, pdl2, s);
}

cudaError_t launch_any(const Plan& p, const ChainArgs& a, int grid, bool pdl2, cudaStream_t s) {
  return a.sentinel_check ? launch_tiles<true>(p, a, grid, pdl2, s) : launch_tiles<false>(p, a, grid, pdl2, s);
}

// The launches of one chain run: sentinel fill, then one fused persistent kernel or the
// producer and consumer kernels (stream order, or programmatic dependent launch).
cusync_status_t launch_run(const cusync_chain_desc_t& d, const Plan& p, ChainArgs A, const Grids& g, void* h,
                           int sms, cudaStream_t stream, bool fill_sets = false) {
  cudaError_t e;
  // Sentinel fill before the run; a rotating stack fills both of its sets only when asked
  // (a new workspace, or after a reset), its runs otherwise fill the next run's set.
  const bool per_stage = d.policy == CUSYNC_POLICY_STREAM || d.launch == CUSYNC_LAUNCH_PDL;
  // Unless the caller opts out, the run's first launch is a programmatic dependent of the
  // kernel before it in the stream: its set-up overlaps that kernel's tail, and it waits
  // for that kernel's completion before it touches memory (pdl_role bit 2); the run's last
  // launch lets such a launch start once all of its tiles are claimed (bit 3).
  const bool overlap = !(d.flags & CUSYNC_FLAG_NO_RUN_OVERLAP);
  // A two-stage chain's fused run under the sentinel policy overlaps its fill: the fill is
  // a programmatic dependent of the kernel before it (it waits for that kernel's end, then
  // lets the chain start), and the chain waits for the fill only before it first stores
  // or loads the intermediate (pdl_role bit 4), so the producers' mainloops run meanwhile.
  const bool fill = d.policy == CUSYNC_POLICY_SENTINEL && !(d.flags & CUSYNC_DEBUG_SKIP_INIT) && (!p.rotate || fill_sets);
  const bool fill_overlap = fill && overlap && !per_stage && !p.stack && p.nst == 2;
  if (fill) {
    // the intermediate (a stack: all of its intermediates, one buffer each)
    const int64_t bytes = (int64_t)p.geo[0].M * p.geo[0].N * 2 * (p.stack ? p.nbuf : 1);
    const int64_t n16 = bytes / 16;
    int blocks = (int)std::min<int64_t>(ceil_div(n16, 256), (int64_t)sms * 8);
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = fill_overlap ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, sentinel_fill_kernel, reinterpret_cast<uint4*>(h), n16, fill_overlap ? 1 : 0);
    if (e != cudaSuccess) return cuda_fail(e, "sentinel fill launch");
  }
  if (!per_stage) {
    A.queue = 0;
    A.first_stage = 0;
    A.last_stage = p.nst - 1;
    A.pdl_role = fill_overlap ? (16 | 8) : (overlap ? (4 | 8) : 0);
    e = launch_any(p, A, g.fused, overlap, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fused chain launch");
    return CUSYNC_OK;
  }
  // One launch per stage; with programmatic dependent launch each one after the first is
  // a secondary of the one before it (triggered at that one's start).
  const bool pdl = d.policy != CUSYNC_POLICY_STREAM;
  for (int s = 0; s < p.nst; ++s) {
    A.queue = s;
    A.first_stage = s;
    A.last_stage = s;
    A.pdl_role = pdl ? ((s + 1 < p.nst ? 1 : 0) | (s > 0 ? 2 : 0)) : 0;
    if (overlap && s == 0) A.pdl_role |= 4;
    if (overlap && s == p.nst - 1) A.pdl_role |= 8;
    e = launch_any(p, A, g.stage[s], /*pdl2=*/(pdl && s > 0) || (overlap && s == 0), stream);
    if (e != cudaSuccess) return cuda_fail(e, s == 0 ? "producer launch" : "later stage launch");
  }
  return CUSYNC_OK;
}

// k-blocks per pipeline stage of the kernel that runs plan p (the sentinel policy runs the
// checked instantiation).
int32_t kernel_kps(const Plan& p, bool check) {
  if (p.pair == 2) {
    if (p.bn == 192) return KCfg<192, 2>::kps(check);
    return p.bn == 256 ? KCfg<256, 2>::kps(check) : KCfg<128, 2>::kps(check);
  }
  return p.bn == 256 ? KCfg<256, 1>::kps(check) : KCfg<128, 1>::kps(check);
}

// TMA descriptors of a run: k-block views or 2-D maps for GEMM operands (encode_operand),
// 4-D NHWC maps for conv images.
bool encode_maps(const cusync_chain_desc_t& d, const Plan& p, ChainArgs& A, const void* a0, const void* b0,
                 const void* b1, const void* h, const void* y, const void* h2 = nullptr) {
  bool ok = true;
  const int32_t kps = kernel_kps(p, d.policy == CUSYNC_POLICY_SENTINEL);
  for (int s = 0; s < 3; ++s) A.st[s].a3d = A.st[s].b3d = 0;
  if (d.kind == CUSYNC_CHAIN_ATTENTION) {
    // stage 0: XQKV = X x QKV; stage 1 reads XQKV and writes XDot (no maps);
    // stage 2: Y = XDot x W2
    const uint64_t n3 = (uint64_t)(3 * d.N1);
    A.st[0].a_ptr = static_cast<const uint16_t*>(a0);
    A.st[0].a_rows = (int32_t)d.M;
    A.st[0].b_ptr = static_cast<const uint16_t*>(b0);
    A.st[0].b_rows = (int32_t)n3;
    A.st[1].a_ptr = static_cast<const uint16_t*>(h);
    A.st[1].a_rows = (int32_t)d.M;
    A.st[2].a_ptr = static_cast<const uint16_t*>(h2);
    A.st[2].a_rows = (int32_t)d.M;
    A.st[2].b_ptr = static_cast<const uint16_t*>(b1);
    A.st[2].b_rows = (int32_t)d.N2;
    ok &= h2 != nullptr;
    ok &= encode_operand(&A.st[0].tmA, a0, (uint64_t)d.M, (uint64_t)d.K, 128u, kps, &A.st[0].a3d);
    ok &= encode_operand(&A.st[0].tmB, b0, n3, (uint64_t)d.K, b_box_rows(p, false), kps, &A.st[0].b3d);
    ok &= encode_2d(&A.st[0].tmO, h, (uint64_t)d.M, n3, 32u);
    ok &= encode_operand(&A.st[2].tmA, h2, (uint64_t)d.M, (uint64_t)d.N1, 128u, kps, &A.st[2].a3d);
    ok &= encode_operand(&A.st[2].tmB, b1, (uint64_t)d.N2, (uint64_t)d.N1, b_box_rows(p, false), kps, &A.st[2].b3d);
    ok &= encode_2d(&A.st[2].tmO, y, (uint64_t)d.M, (uint64_t)d.N2, 32u);
  } else if (d.kind == CUSYNC_CHAIN_CONV_STACK) {
    // stage 0 reads x, every later stage one of the workspace's buffers; all stages take
    // their weights from the stacked weights (a0 = x, b0 = weights, h = workspace)
    const StageGeo& g0 = p.geo[0];
    ok &= encode_nhwc(&A.st[0].tmA, a0, d.n, d.h, d.w, d.c, (uint32_t)g0.th);
    ok &= encode_nhwc_bufs(&A.st[1].tmA, h, (uint64_t)p.nbuf, d.n, d.h, d.w, d.c, (uint32_t)g0.th);
    ok &= encode_3d(&A.st[0].tmB, b0, (uint64_t)p.nst, (uint64_t)d.c, (uint64_t)9 * d.c, b_box_rows(p, false));
    A.st[1].tmB = A.st[0].tmB;
  } else if (d.kind == CUSYNC_CHAIN_CONV_RELU) {
    const StageGeo& g0 = p.geo[0];
    ok &= encode_nhwc(&A.st[0].tmA, a0, d.n, d.h, d.w, d.c, (uint32_t)g0.th);
    ok &= encode_operand(&A.st[0].tmB, b0, (uint64_t)d.k_out, (uint64_t)9 * d.c, b_box_rows(p, false), kps, &A.st[0].b3d);
    ok &= encode_nhwc(&A.st[1].tmA, h, d.n, d.h, d.w, d.k_out, (uint32_t)g0.th);
    ok &= encode_operand(&A.st[1].tmB, b1, (uint64_t)d.k_out, (uint64_t)9 * d.k_out, b_box_rows(p, false), kps,
                         &A.st[1].b3d);
  } else {
    const bool swiglu = d.kind == CUSYNC_CHAIN_MLP_SWIGLU;
    A.st[0].a_ptr = static_cast<const uint16_t*>(a0);
    A.st[0].a_rows = (int32_t)d.M;
    A.st[0].b_ptr = static_cast<const uint16_t*>(b0);
    A.st[0].b_rows = (int32_t)(swiglu ? 2 * d.N1 : d.N1);
    A.st[1].a_ptr = static_cast<const uint16_t*>(h);
    A.st[1].a_rows = (int32_t)d.M;
    A.st[1].b_ptr = static_cast<const uint16_t*>(b1);
    A.st[1].b_rows = (int32_t)d.N2;
    ok &= encode_operand(&A.st[0].tmA, a0, (uint64_t)d.M, (uint64_t)d.K, 128u, kps, &A.st[0].a3d);
    // a single CTA of a SwiGLU chain copies the gate and up halves of its weight tile
    // separately for every k-block (the 2-D map)
    ok &= encode_operand(&A.st[0].tmB, b0, (uint64_t)(swiglu ? 2 * d.N1 : d.N1), (uint64_t)d.K, b_box_rows(p, swiglu),
                         (swiglu && p.pair == 1) ? 1 : kps, &A.st[0].b3d);
    ok &= encode_operand(&A.st[1].tmA, h, (uint64_t)d.M, (uint64_t)d.N1, 128u, kps, &A.st[1].a3d);
    ok &= encode_operand(&A.st[1].tmB, b1, (uint64_t)d.N2, (uint64_t)d.N1, b_box_rows(p, false), kps, &A.st[1].b3d);
    ok &= encode_2d(&A.st[0].tmO, h, (uint64_t)d.M, (uint64_t)d.N1, 32u);
    ok &= encode_2d(&A.st[1].tmO, y, (uint64_t)d.M, (uint64_t)d.N2, 32u);
  }
  return ok;
}

// Kernel arguments that do not depend on the operand pointers.
void fill_static_args(const cusync_chain_desc_t& d, const Plan& p, uint32_t* state, float* split_ws, ChainArgs& A) {
  const int64_t t0 = stage_units(p.geo[0]);
  const int64_t t1 = stage_units(p.geo[1]);
  const uint64_t timeout = d.timeout_ns ? d.timeout_ns : kDefaultTimeoutNs;
  A.st[0].g = p.geo[0];
  A.st[1].g = p.geo[1];
  A.st[2].g = p.geo[2];
  A.st[0].b_half_rows = d.kind == CUSYNC_CHAIN_MLP_SWIGLU ? (int32_t)d.N1 : 0;
  A.nst = p.nst;
  A.dep = p.dep;
  A.dep_pw = p.dep_pw;
  A.ctrl = state;
  A.flags = state + CTRL_WORDS;
  A.flags_pw = state + CTRL_WORDS + p.num_flags;
  A.band_flags = p.n_bands > 0 ? state + CTRL_WORDS + p.num_flags + p.num_flags_pw : nullptr;
  A.n_bands = p.n_bands;
  A.split_ws = p.split_rows > 0 ? split_ws : nullptr;
  A.split_ws1 = p.split_rows1 > 0 ? split_ws + split_ws_floats0(p) : nullptr;
  A.tiles0 = (int32_t)t0;
  A.tiles1 = (int32_t)t1;
  A.tiles2 = (int32_t)stage_units(p.geo[2]);
  A.stack = p.stack;
  A.nbuf = p.stack ? p.nbuf : 1;
  A.flags_stride = (int32_t)p.flags_stride;
  A.buf_elems = p.stack ? stack_buf_elems(d) : 0;
  A.rotate = p.rotate;
  if (p.rotate) {
    A.set_chunks = (int64_t)(p.nst - 1) * A.buf_elems / 8;
    A.fill_unit_chunks = 4096;  // 64 KB per unit
    A.fill_units = (int32_t)ceil_div(A.set_chunks, A.fill_unit_chunks);
  }
  A.flags_bits = d.flags;
  A.sentinel_check = d.policy == CUSYNC_POLICY_SENTINEL ? 1 : 0;
  A.num_flags = (int32_t)p.num_flags;
  const bool streams_weights = (d.kind == CUSYNC_CHAIN_MLP_GELU || d.kind == CUSYNC_CHAIN_MLP_SWIGLU) && p.pair == 2 &&
                               p.geo[0].ksplit > 1;
  A.l2_prefetch = d.l2_prefetch < 0 ? 0 : (d.l2_prefetch == 0 ? (streams_weights ? kDefaultPrefetch : 0) : d.l2_prefetch);
  A.timeout_ns = timeout;
  A.pipe_timeout_ns = std::max<uint64_t>(4 * timeout, 2000000000ull);
}

cusync_status_t run_chain(cusync_chain* ch, const void* a0, const void* b0, const void* b1, void* h, void* h2,
                          void* y, cudaStream_t stream) {
  const cusync_chain_desc_t& d = ch->d;
  const Plan& p = ch->plan;
  if (!aligned16(a0) || !aligned16(b0) || !aligned16(b1) || !aligned16(h) || !aligned16(y))
    return CUSYNC_ERR_INVALID_ARG;
  if (h == y || h == a0 || y == a0) return CUSYNC_ERR_INVALID_ARG;
  if (p.nst == 3 && !p.stack && (!aligned16(h2) || h2 == h || h2 == y || h2 == a0)) return CUSYNC_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != ch->device) return CUSYNC_ERR_INVALID_ARG;
  ChainArgs& A = ch->args;
  const void* ptrs[6] = {a0, b0, b1, h, y, h2};
  if (!ch->maps_valid || std::memcmp(ptrs, ch->cached, sizeof(ptrs)) != 0) {
    if (!encode_maps(d, p, A, a0, b0, b1, h, y, h2)) {
      ch->maps_valid = false;
      return CUSYNC_ERR_INVALID_ARG;
    }
    std::memcpy(ch->cached, ptrs, sizeof(ptrs));
    ch->maps_valid = true;
  }
  A.st[0].out = h;
  A.st[1].out = (p.nst == 3 && !p.stack) ? h2 : y;
  A.st[2].out = (p.nst == 3 && !p.stack) ? y : nullptr;
  const bool fill_sets = p.rotate && (h != ch->filled_ws || ch->need_fill);
  const cusync_status_t st = launch_run(d, p, A, ch->grids, h, ch->num_sms, stream, fill_sets);
  if (st == CUSYNC_OK && p.rotate) {
    ch->filled_ws = h;
    ch->need_fill = false;
  }
  return st;
}

}  // namespace

extern "C" {

const char* cusync_status_string(cusync_status_t s) {
  switch (s) {
    case CUSYNC_OK: return "CUSYNC_OK";
    case CUSYNC_ERR_INVALID_ARG: return "CUSYNC_ERR_INVALID_ARG";
    case CUSYNC_ERR_UNSUPPORTED: return "CUSYNC_ERR_UNSUPPORTED";
    case CUSYNC_ERR_CUDA: return "CUSYNC_ERR_CUDA";
    case CUSYNC_ERR_NOMEM: return "CUSYNC_ERR_NOMEM";
    case CUSYNC_ERR_TIMEOUT: return "CUSYNC_ERR_TIMEOUT";
    case CUSYNC_ERR_DEVICE: return "CUSYNC_ERR_DEVICE";
  }
  return "CUSYNC_ERR_UNKNOWN";
}

// [cuSync] §II-A "Thread block Wave Execution" and §III-A.
cusync_status_t cusync_wave_stats(int64_t tbs0, int64_t tbs1, int32_t occupancy, int32_t num_sms,
                                  cusync_wave_report_t* out) {
  if (!out || tbs0 < 0 || tbs1 < 0 || occupancy < 1 || num_sms < 1) return CUSYNC_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  const int64_t cap = (int64_t)occupancy * num_sms;
  const int64_t tbs[2] = {tbs0, tbs1};
  int32_t stream = 0;
  for (int i = 0; i < 2; ++i) {
    out->tbs[i] = tbs[i];
    out->waves[i] = (double)tbs[i] / (double)cap;
    out->waves_ceil[i] = (int32_t)ceil_div(tbs[i], cap);
    out->util[i] = out->waves_ceil[i] ? (double)tbs[i] / ((double)out->waves_ceil[i] * (double)cap) : 0.0;
    stream += out->waves_ceil[i];
  }
  const int64_t total = tbs0 + tbs1;
  out->stream_waves = stream;
  out->fused_waves = (int32_t)ceil_div(total, cap);
  out->fused_waves_frac = (double)total / (double)cap;
  out->last_wave_tbs = total == 0 ? 0 : (total % cap == 0 ? cap : total % cap);
  out->cap = (int32_t)cap;
  out->occupancy = occupancy;
  out->num_sms = num_sms;
  return CUSYNC_OK;
}

cusync_status_t cusync_plan_waves(const cusync_chain_desc_t* d, cusync_wave_report_t* out) {
  if (!d || !out) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  int sms = 0;
  if (query_num_sms(d->num_sms, &sms) != 0) return CUSYNC_ERR_CUDA;
  const int64_t t0 = stage_units(p.geo[0]);
  const int64_t t1 = stage_units(p.geo[1]);
  // one tile per CTA, or per CTA pair: a pair occupies two SMs
  st = cusync_wave_stats(t0, t1, 1, p.pair == 2 ? sms / 2 : sms, out);
  if (st != CUSYNC_OK) return st;
  out->num_sms = sms;
  out->tile_m = kBM * p.pair;
  out->tile_n = p.bn;
  out->tile_k = kBK;
  return CUSYNC_OK;
}

cusync_status_t cusync_create_chain(const cusync_chain_desc_t* d, cusync_chain_t* out) {
  if (!d || !out) return CUSYNC_ERR_INVALID_ARG;
  *out = nullptr;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  if (!load_encoder()) return CUSYNC_ERR_CUDA;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    CUSYNC_LOG("device compute capability %d.%d; this library is built for sm_103a", major, minor);
    return CUSYNC_ERR_UNSUPPORTED;
  }
  int dev_sms = 0;
  if (query_num_sms(0, &dev_sms) != 0) return CUSYNC_ERR_CUDA;
  const int sms = d->num_sms > 0 ? std::min(d->num_sms, dev_sms) : dev_sms;
  if ((e = set_all_kernel_attrs()) != cudaSuccess) return cuda_fail(e, "kernel attributes");
  const int max_clusters = p.pair != 2 ? 0
                           : p.bn == 256 ? max_pair_clusters<256>()
                           : p.bn == 192 ? max_pair_clusters<192>()
                                         : max_pair_clusters<128>();
  if (p.pair == 2 && max_clusters < 1) {
    CUSYNC_LOG("no CTA-pair cluster can be resident on this device");
    return CUSYNC_ERR_UNSUPPORTED;
  }

  cusync_chain* ch = new (std::nothrow) cusync_chain();
  if (!ch) return CUSYNC_ERR_NOMEM;
  ch->d = *d;
  ch->d.policy = (cusync_policy_t)p.dep.policy;  // CUSYNC_POLICY_AUTO resolved
  if (ch->d.timeout_ns == 0) ch->d.timeout_ns = kDefaultTimeoutNs;
  ch->plan = p;
  ch->device = dev;
  ch->num_sms = sms;
  const size_t words = (size_t)state_words(p);
  ch->state = nullptr;
  ch->split_ws = nullptr;
  ch->trace = nullptr;
  if (cudaMalloc(&ch->state, words * sizeof(uint32_t)) != cudaSuccess) {
    delete ch;
    return CUSYNC_ERR_NOMEM;
  }
  if ((e = cudaMemset(ch->state, 0, words * sizeof(uint32_t))) != cudaSuccess) {
    cudaFree(ch->state);
    delete ch;
    return cuda_fail(e, "state clear");
  }
  if ((p.split_rows > 0 || p.split_rows1 > 0) &&
      cudaMalloc(&ch->split_ws, (size_t)split_ws_floats(p) * sizeof(float)) != cudaSuccess) {
    cudaFree(ch->state);
    delete ch;
    return CUSYNC_ERR_NOMEM;
  }
  // every K-split workspace word starts empty (all bits set: the kernel's empty mark)
  if (ch->split_ws && (e = cudaMemset(ch->split_ws, 0xFF, (size_t)split_ws_floats(p) * sizeof(float))) != cudaSuccess) {
    cudaFree(ch->split_ws);
    cudaFree(ch->state);
    delete ch;
    return cuda_fail(e, "K-split workspace clear");
  }
  if (d->flags & CUSYNC_FLAG_TRACE) {
    const size_t n = (size_t)total_units(p);
    if (cudaMalloc(&ch->trace, n * sizeof(TraceRec)) != cudaSuccess ||
        cudaMemset(ch->trace, 0, n * sizeof(TraceRec)) != cudaSuccess) {
      if (ch->trace) cudaFree(ch->trace);
      if (ch->split_ws) cudaFree(ch->split_ws);
      cudaFree(ch->state);
      delete ch;
      return CUSYNC_ERR_NOMEM;
    }
  }
  ch->grids = make_grids(p, sms, max_clusters);
  ChainArgs& A = ch->args;
  std::memset(&A, 0, sizeof(A));
  fill_static_args(ch->d, p, ch->state, ch->split_ws, A);
  A.trace = ch->trace;
  ch->maps_valid = false;
  ch->filled_ws = nullptr;
  ch->need_fill = true;
  ch->band_ev = nullptr;
  ch->bands_ready = false;
  if (p.n_bands > 0 && (e = cudaEventCreateWithFlags(&ch->band_ev, cudaEventDisableTiming)) != cudaSuccess) {
    if (ch->trace) cudaFree(ch->trace);
    if (ch->split_ws) cudaFree(ch->split_ws);
    cudaFree(ch->state);
    delete ch;
    return cuda_fail(e, "band event");
  }
  *out = ch;
  CUSYNC_LOG("chain kind=%d policy=%d launch=%d tiles=%d+%d bn=%d pair=%d sms=%d clusters=%d flags=%lld", d->kind,
             d->policy, d->launch, A.tiles0, A.tiles1, p.bn, p.pair, sms, max_clusters, (long long)p.num_flags);
  return CUSYNC_OK;
}

cusync_status_t cusync_run_mlp(cusync_chain_t ch, const void* X, const void* W1t, const void* W2t, void* H, void* Y,
                               cusync_stream_t stream) {
  if (!ch) return CUSYNC_ERR_INVALID_ARG;
  if (ch->d.kind != CUSYNC_CHAIN_MLP_GELU && ch->d.kind != CUSYNC_CHAIN_MLP_SWIGLU) return CUSYNC_ERR_INVALID_ARG;
  return run_chain(ch, X, W1t, W2t, H, nullptr, Y, reinterpret_cast<cudaStream_t>(stream));
}

cusync_status_t cusync_run_conv_chain(cusync_chain_t ch, const void* x, const void* w1, const void* w2, void* y1,
                                      void* y2, cusync_stream_t stream) {
  if (!ch) return CUSYNC_ERR_INVALID_ARG;
  if (ch->d.kind != CUSYNC_CHAIN_CONV_RELU) return CUSYNC_ERR_INVALID_ARG;
  return run_chain(ch, x, w1, w2, y1, nullptr, y2, reinterpret_cast<cudaStream_t>(stream));
}

cusync_status_t cusync_run_conv_stack(cusync_chain_t ch, const void* x, const void* w, void* work, void* y,
                                      cusync_stream_t stream) {
  if (!ch) return CUSYNC_ERR_INVALID_ARG;
  if (ch->d.kind != CUSYNC_CHAIN_CONV_STACK) return CUSYNC_ERR_INVALID_ARG;
  // the weights take the place of both weight operands (one stacked map serves all stages)
  return run_chain(ch, x, w, w, work, nullptr, y, reinterpret_cast<cudaStream_t>(stream));
}

cusync_status_t cusync_run_attention(cusync_chain_t ch, const void* X, const void* Wqkv_t, const void* W2t,
                                     void* XQKV, void* XDot, void* Y, cusync_stream_t stream) {
  if (!ch) return CUSYNC_ERR_INVALID_ARG;
  if (ch->d.kind != CUSYNC_CHAIN_ATTENTION) return CUSYNC_ERR_INVALID_ARG;
  return run_chain(ch, X, Wqkv_t, W2t, XQKV, XDot, Y, reinterpret_cast<cudaStream_t>(stream));
}

cusync_status_t cusync_chain_reset(cusync_chain_t ch, cusync_stream_t stream) {
  if (!ch) return CUSYNC_ERR_INVALID_ARG;
  const size_t words = (size_t)state_words(ch->plan);
  cudaError_t e = cudaMemsetAsync(ch->state, 0, words * sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "state reset");
  // a run that stopped early may have left K-split sums unread: mark every word empty
  if (ch->split_ws) {
    e = cudaMemsetAsync(ch->split_ws, 0xFF, (size_t)split_ws_floats(ch->plan) * sizeof(float),
                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "K-split workspace reset");
  }
  ch->need_fill = true;  // a run that stopped early may have left the next set unfilled
  ch->bands_ready = false;
  return CUSYNC_OK;
}

cusync_status_t cusync_chain_check(cusync_chain_t ch, cusync_stream_t stream, uint32_t* code, uint32_t* detail) {
  if (!ch) return CUSYNC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t w[2] = {0, 0};
  e = cudaMemcpy(w, ch->state, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "error word read");
  if (code) *code = w[0];
  if (detail) *detail = w[1];
  if (w[0] == 0) return CUSYNC_OK;
  const uint32_t cls = w[0] >> 24;
  CUSYNC_LOG("device error class %u tile %u detail 0x%x", cls, w[0] & 0xFFFFFFu, w[1]);
  cusync_status_t r = CUSYNC_ERR_DEVICE;
  if (cls == ERRC_FLAG_TIMEOUT || cls == ERRC_SENTINEL_TIMEOUT) r = CUSYNC_ERR_TIMEOUT;
  if (cusync_chain_reset(ch, stream) != CUSYNC_OK) return CUSYNC_ERR_CUDA;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
  return r;
}

cusync_status_t cusync_plan_info(const cusync_chain_desc_t* d, cusync_chain_info_t* out) {
  if (!d || !out) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  int sms = 0;
  if (query_num_sms(d->num_sms, &sms) != 0) return CUSYNC_ERR_CUDA;
  std::memset(out, 0, sizeof(*out));
  for (int s = 0; s < 2; ++s) {
    out->m_tiles[s] = p.geo[s].m_tiles;
    out->n_tiles[s] = p.geo[s].n_tiles;
    out->k_blocks[s] = p.geo[s].k_blocks;
    out->n_out[s] = p.geo[s].n_out;
  }
  out->tile_m = kBM * p.pair;
  out->tile_n = p.bn;
  out->tile_k = kBK;
  out->strided_group = p.dep.G;
  out->strided_distance = p.dep.D;
  out->num_flags = (int32_t)p.num_flags;
  const Grids g = make_grids(p, sms, 0);
  const bool two = p.dep.policy == POL_STREAM || d->launch == CUSYNC_LAUNCH_PDL;
  out->grid[0] = two ? g.stage[0] : g.fused;
  out->grid[1] = two ? g.stage[1] : 0;
  out->grid2 = two ? g.stage[2] : 0;
  out->cta_pair = p.pair;
  out->num_sms = sms;
  out->conv_rows_per_tile = d->kind == CUSYNC_CHAIN_CONV_RELU ? p.geo[0].th : 0;
  out->policy = p.nst == 3 ? p.dep_pw.policy : p.dep.policy;
  out->ksplit = p.geo[0].ksplit;
  out->kb_per_split = p.geo[0].kb_per_split;
  out->ksplit_skew = p.geo[0].kb_skew;
  out->ksplit_consumer = p.geo[1].ksplit;
  out->kb_per_split_consumer = p.geo[1].kb_per_split;
  out->raster_rows = p.geo[0].raster;
  out->nst = p.nst;
  out->m_tiles2 = p.geo[2].m_tiles;
  out->n_tiles2 = p.geo[2].n_tiles;
  out->k_blocks2 = p.geo[2].k_blocks;
  out->n_out2 = p.geo[2].n_out;
  out->num_flags_pw = (int32_t)p.num_flags_pw;
  out->strided_group_pw = p.dep_pw.G;
  out->strided_distance_pw = p.dep_pw.D;
  if (p.stack) {
    out->conv_rows_per_tile = p.geo[0].th;
    out->work_buffers = p.nbuf;
    out->work_bytes = (int64_t)p.nbuf * stack_buf_elems(*d) * 2;
    out->m_tiles2 = out->n_tiles2 = out->k_blocks2 = out->n_out2 = out->grid2 = 0;
  }
  return CUSYNC_OK;
}

cusync_status_t cusync_pointwise_waits(const cusync_chain_desc_t* d, int32_t m_tile, int32_t head, int32_t* flag,
                                       uint32_t* per_run, int32_t max, int32_t* n_out) {
  if (!d || !n_out || max < 0 || (max > 0 && (!flag || !per_run))) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  if (p.nst != 3) return CUSYNC_ERR_INVALID_ARG;
  if (m_tile < 0 || m_tile >= p.geo[1].m_tiles || head < 0 || head >= p.geo[1].n_tiles) return CUSYNC_ERR_INVALID_ARG;
  Wait w[3];
  const int n = pointwise_waits(p.dep_pw, m_tile, head, w);
  for (int i = 0; i < n && i < max; ++i) {
    flag[i] = w[i].flag;
    per_run[i] = w[i].per_run;
  }
  *n_out = n;
  return CUSYNC_OK;
}

cusync_status_t cusync_default_latency_model(const cusync_chain_desc_t* d, cusync_latency_model_t* out) {
  if (!d || !out) return CUSYNC_ERR_INVALID_ARG;
  cusync_chain_desc_t c = *d;
  if (c.policy == CUSYNC_POLICY_AUTO) c.policy = CUSYNC_POLICY_STREAM;  // the constants do not depend on it
  Plan p;
  cusync_status_t st = make_plan(c, &p);
  if (st != CUSYNC_OK) return st;
  const LatencyModel m = default_model(p);
  static_assert(sizeof(LatencyModel) == sizeof(cusync_latency_model_t), "latency model layout");
  std::memcpy(out, &m, sizeof(m));
  return CUSYNC_OK;
}

cusync_status_t cusync_predict_policies(const cusync_chain_desc_t* d, const cusync_latency_model_t* model,
                                        cusync_policy_prediction_t* out) {
  if (!d || !out) return CUSYNC_ERR_INVALID_ARG;
  int sms = 0;
  if (query_num_sms(d->num_sms, &sms) != 0) return CUSYNC_ERR_CUDA;
  std::memset(out, 0, sizeof(*out));
  predict_all(*d, model, sms, out->us);
  out->best = -1;
  out->best_sync = -1;
  for (int pol = CUSYNC_POLICY_STREAM; pol <= CUSYNC_POLICY_SENTINEL; ++pol) {
    if (out->us[pol] < 0.0) continue;
    if (out->best < 0 || out->us[pol] < out->us[out->best]) out->best = pol;
    if (pol != CUSYNC_POLICY_STREAM && (out->best_sync < 0 || out->us[pol] < out->us[out->best_sync]))
      out->best_sync = pol;
  }
  out->num_sms = sms;
  return out->best < 0 ? CUSYNC_ERR_UNSUPPORTED : CUSYNC_OK;
}

cusync_status_t cusync_consumer_waits(const cusync_chain_desc_t* d, int32_t m_tile, int32_t* kb, int32_t* flag,
                                      uint32_t* per_run, int32_t max, int32_t* n_out) {
  if (!d || !n_out || max < 0) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  const StageGeo& g = sgeo(p, p.nst - 1);  // the stage that waits on `dep`
  if (m_tile < 0 || m_tile >= g.m_tiles) return CUSYNC_ERR_INVALID_ARG;
  if (max > 0 && (!kb || !flag || !per_run)) return CUSYNC_ERR_INVALID_ARG;
  DepTracker dt;
  dt.reset();
  int32_t n = 0;
  for (int32_t k = 0; k < g.k_blocks; ++k) {
    if (!dep_kblock(g, p.dep, k)) continue;
    Wait w[kMaxWaits];
    const int c = dt.next(g, p.dep, m_tile, k, w);
    for (int i = 0; i < c; ++i, ++n) {
      if (n < max) {
        kb[n] = k;
        flag[n] = w[i].flag;
        per_run[n] = w[i].per_run;
      }
    }
  }
  *n_out = n;
  return CUSYNC_OK;
}

cusync_status_t cusync_consumer_unit_waits(const cusync_chain_desc_t* d, int32_t m_tile, int32_t unit, int32_t* kb,
                                           int32_t* flag, uint32_t* per_run, int32_t max, int32_t* n_out) {
  if (!d || !n_out || max < 0) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  if (p.stack || p.nst != 2) return CUSYNC_ERR_INVALID_ARG;
  const StageGeo& g = p.geo[1];
  if (g.a_mode != AMODE_GEMM) return CUSYNC_ERR_INVALID_ARG;
  if (m_tile < 0 || m_tile >= g.m_tiles || unit < 0 || unit >= g.ksplit) return CUSYNC_ERR_INVALID_ARG;
  if (max > 0 && (!kb || !flag || !per_run)) return CUSYNC_ERR_INVALID_ARG;
  int32_t kb0 = 0, nkb = 0;
  split_unit(g, unit, &kb0, &nkb);
  GemmDepTracker t;
  t.reset();
  int32_t n = 0;
  for (int32_t k = 0; k < nkb; ++k) {
    if (!unit_dep_kblock(p.dep, kb0, nkb, k)) continue;
    Wait w[kMaxWaits];
    const int c = t.next(p.dep, m_tile, kb0 + k, w);
    for (int i = 0; i < c; ++i, ++n) {
      if (n < max) {
        kb[n] = kb0 + k;
        flag[n] = w[i].flag;
        per_run[n] = w[i].per_run;
      }
    }
  }
  *n_out = n;
  return CUSYNC_OK;
}

cusync_status_t cusync_producer_flag(const cusync_chain_desc_t* d, int32_t m_tile, int32_t n_tile, int32_t* flag) {
  if (!d || !flag) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  const StageGeo& g = p.geo[0];
  if (m_tile < 0 || m_tile >= g.m_tiles || n_tile < 0 || n_tile >= g.n_tiles) return CUSYNC_ERR_INVALID_ARG;
  *flag = producer_flag(p.dep, m_tile, n_tile);
  return CUSYNC_OK;
}

cusync_status_t cusync_tile_at(const cusync_chain_desc_t* d, int32_t stage, int32_t u, int32_t* m_tile,
                               int32_t* n_tile) {
  if (!d || !m_tile || !n_tile || stage < 0 || stage > 1) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  const StageGeo& g = p.geo[stage];
  if (u < 0 || u >= g.m_tiles * g.n_tiles) return CUSYNC_ERR_INVALID_ARG;
  int32_t m, y;
  tile_at(g, u, &m, &y);
  *m_tile = m;
  *n_tile = stage == 0 ? producer_col(p.dep, y) : y;
  return CUSYNC_OK;
}

cusync_status_t cusync_producer_col(const cusync_chain_desc_t* d, int32_t y, int32_t* col) {
  if (!d || !col) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  if (y < 0 || y >= p.geo[0].n_tiles) return CUSYNC_ERR_INVALID_ARG;
  *col = producer_col(p.dep, y);
  return CUSYNC_OK;
}

// Posts a complete run makes on band b's semaphore: one per CTA of every consumer tile in
// the band (the last K-split unit of a tile posts).
static uint32_t band_posts(const Plan& p, int32_t b) {
  const StageGeo& g = p.geo[1];
  const int32_t rows = band_lo(g.m_tiles, p.n_bands, b + 1) - band_lo(g.m_tiles, p.n_bands, b);
  return (uint32_t)rows * (uint32_t)g.n_tiles * (uint32_t)p.pair;
}

static bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone;
}

cusync_status_t cusync_run_mlp_bands(cusync_chain_t ch, const void* X, const void* W1t, const void* W2t, void* H,
                                     void* Y, cusync_stream_t stream, cusync_stream_t band_stream) {
  if (!ch) return CUSYNC_ERR_INVALID_ARG;
  if (ch->d.kind != CUSYNC_CHAIN_MLP_GELU && ch->d.kind != CUSYNC_CHAIN_MLP_SWIGLU) return CUSYNC_ERR_INVALID_ARG;
  const Plan& p = ch->plan;
  if (p.n_bands < 1) return CUSYNC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t bs = reinterpret_cast<cudaStream_t>(band_stream);
  if (s == bs) return CUSYNC_ERR_INVALID_ARG;
  // band waits are stream memory operations that CUDA's graph dependencies do not see
  if (stream_capturing(s) || stream_capturing(bs)) return CUSYNC_ERR_UNSUPPORTED;
  if (!load_wait_value()) return CUSYNC_ERR_UNSUPPORTED;
  ch->bands_ready = false;
  uint32_t* const bands = ch->args.band_flags;
  cudaError_t e = cudaMemsetAsync(bands, 0, (size_t)p.n_bands * sizeof(uint32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "band semaphores clear");
  if ((e = cudaEventRecord(ch->band_ev, s)) != cudaSuccess) return cuda_fail(e, "band event record");
  const cusync_status_t st = run_chain(ch, X, W1t, W2t, H, nullptr, Y, s);
  BandTargets tg;
  std::memset(&tg, 0, sizeof(tg));
  for (int32_t b = 0; b < p.n_bands; ++b) tg.v[b] = band_posts(p, b);
  // launched whatever the run's launch status, so that band waits always end
  band_release_kernel<<<1, 32, 0, s>>>(bands, tg, p.n_bands);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "band release launch");
  if (st != CUSYNC_OK) return st;
  // the band stream's waits start only once this run's band semaphores are cleared
  if ((e = cudaStreamWaitEvent(bs, ch->band_ev, 0)) != cudaSuccess) return cuda_fail(e, "band stream wait");
  ch->bands_ready = true;
  return CUSYNC_OK;
}

cusync_status_t cusync_band_wait(cusync_chain_t ch, int32_t band, cusync_stream_t band_stream) {
  if (!ch || !ch->bands_ready) return CUSYNC_ERR_INVALID_ARG;
  const Plan& p = ch->plan;
  if (band < 0 || band >= p.n_bands) return CUSYNC_ERR_INVALID_ARG;
  cudaStream_t bs = reinterpret_cast<cudaStream_t>(band_stream);
  if (stream_capturing(bs)) return CUSYNC_ERR_UNSUPPORTED;
  const CUresult r = g_wait_value(reinterpret_cast<CUstream>(bs),
                                  reinterpret_cast<CUdeviceptr>(ch->args.band_flags + band), band_posts(p, band),
                                  CU_STREAM_WAIT_VALUE_GEQ);
  if (r != CUDA_SUCCESS) {
    CUSYNC_LOG("cuStreamWaitValue32: error %d", (int)r);
    return CUSYNC_ERR_CUDA;
  }
  return CUSYNC_OK;
}

cusync_status_t cusync_band_rows(const cusync_chain_desc_t* d, int32_t band, int64_t* row0, int64_t* rows) {
  if (!d || !row0 || !rows) return CUSYNC_ERR_INVALID_ARG;
  Plan p;
  cusync_status_t st = make_plan(*d, &p);
  if (st != CUSYNC_OK) return st;
  if (p.n_bands < 1 || band < 0 || band >= p.n_bands) return CUSYNC_ERR_INVALID_ARG;
  const int64_t tm = (int64_t)kBM * p.pair;
  const int64_t r0 = band_lo(p.geo[1].m_tiles, p.n_bands, band) * tm;
  const int64_t r1 = std::min<int64_t>((int64_t)band_lo(p.geo[1].m_tiles, p.n_bands, band + 1) * tm, p.geo[1].M);
  *row0 = r0;
  *rows = r1 - r0;
  return CUSYNC_OK;
}

cusync_status_t cusync_chain_trace(cusync_chain_t ch, cusync_stream_t stream, cusync_trace_rec_t* out, int32_t max,
                                   int32_t* n_out) {
  static_assert(sizeof(cusync_trace_rec_t) == sizeof(TraceRec), "trace record layout");
  if (!ch || !n_out || max < 0 || (max > 0 && !out) || !ch->trace) return CUSYNC_ERR_INVALID_ARG;
  const int32_t n = (int32_t)total_units(ch->plan);
  *n_out = n;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  const int32_t k = std::min(n, max);
  if (k > 0 && (e = cudaMemcpy(out, ch->trace, (size_t)k * sizeof(TraceRec), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "trace read");
  return CUSYNC_OK;
}

cusync_status_t cusync_destroy_chain(cusync_chain_t ch) {
  if (!ch) return CUSYNC_OK;
  cudaError_t e = cudaSuccess;
  if (ch->trace) cudaFree(ch->trace);
  if (ch->split_ws) cudaFree(ch->split_ws);
  if (ch->band_ev) cudaEventDestroy(ch->band_ev);
  if (ch->state) e = cudaFree(ch->state);
  delete ch;
  return e == cudaSuccess ? CUSYNC_OK : CUSYNC_ERR_CUDA;
}

}  // extern "C"

// ----------------------------------------------------------------------------- no-alloc entry
//
// Some callers of this library may not allocate device memory themselves: a plugin or
// operator running inside an inference runtime whose device memory is owned by the
// runtime's own pool, or a latency-critical serving loop where cudaMalloc / cudaFree
// would add device-wide synchronisation.  cusync_run_mlp_noalloc serves them: it runs
// the same chain kernel as cusync_run_mlp, but keeps the chain's synchronisation state
// (error word, tile counters, semaphores) in the fixed array below instead of in memory
// allocated by cusync_create_chain.  It allocates nothing.
//
// The array lives in every device that loads this library, until the process exits.
// All calls share it and it keeps the last call's contents, so every call clears the
// part it uses on its stream before launching; two calls whose work overlaps on the GPU
// (different streams, no ordering between them) race on it and must not be issued.

namespace {

constexpr int kNoAllocWords = 16384;  // 64 KiB: CTRL_WORDS control words + semaphores
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocWords];

constexpr int kMaxDevices = 64;
uint32_t* g_noalloc_ptr[kMaxDevices] = {};
int g_noalloc_clusters[kMaxDevices][3] = {};  // co-resident CTA-pair clusters (BN 256, 128, 192)
std::mutex g_noalloc_mu;

// Device address of the scratch array and the kernels' attributes for the current device,
// set up on the first call made with that device current.
cusync_status_t noalloc_setup(int dev, uint32_t** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (dev < 0 || dev >= kMaxDevices) return CUSYNC_ERR_UNSUPPORTED;
  if (g_noalloc_ptr[dev] == nullptr) {
    if (!load_encoder()) return CUSYNC_ERR_CUDA;
    cudaError_t e = set_all_kernel_attrs();
    if (e != cudaSuccess) return cuda_fail(e, "kernel attributes (no-alloc)");
    uint32_t* p = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_noalloc_clusters[dev][0] = max_pair_clusters<256>();
    g_noalloc_clusters[dev][1] = max_pair_clusters<128>();
    g_noalloc_clusters[dev][2] = max_pair_clusters<192>();
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return CUSYNC_OK;
}

}  // namespace

extern "C" cusync_status_t cusync_run_mlp_noalloc(const cusync_chain_desc_t* d, const void* X, const void* W1t,
                                                  const void* W2t, void* H, void* Y, cusync_stream_t stream,
                                                  uint32_t* error_word) {
  if (!d) return CUSYNC_ERR_INVALID_ARG;
  if (d->kind != CUSYNC_CHAIN_MLP_GELU && d->kind != CUSYNC_CHAIN_MLP_SWIGLU) return CUSYNC_ERR_INVALID_ARG;
  // No workspace to hold K-split partial sums: neither GEMM is split.  0 (the planner's
  // choice elsewhere) means 1 here.
  if (d->ksplit > 1 || d->ksplit_consumer > 1) return CUSYNC_ERR_UNSUPPORTED;
  cusync_chain_desc_t dd = *d;
  dd.ksplit = 1;
  dd.ksplit_consumer = 1;
  Plan p;
  cusync_status_t st = make_plan(dd, &p);
  if (st != CUSYNC_OK) return st;
  dd.policy = (cusync_policy_t)p.dep.policy;  // CUSYNC_POLICY_AUTO resolved
  // The fixed array bounds the chain's state: control words and every semaphore.
  static_assert(CUSYNC_NOALLOC_MAX_SEMAPHORES == kNoAllocWords - CTRL_WORDS, "no-alloc limit in cusync.h");
  const int64_t words = state_words(p);
  if (words > kNoAllocWords) {
    CUSYNC_LOG("no-alloc run needs %lld semaphores; the fixed scratch holds %d", (long long)(words - CTRL_WORDS),
               CUSYNC_NOALLOC_MAX_SEMAPHORES);
    return CUSYNC_ERR_UNSUPPORTED;
  }
  if (!aligned16(X) || !aligned16(W1t) || !aligned16(W2t) || !aligned16(H) || !aligned16(Y))
    return CUSYNC_ERR_INVALID_ARG;
  if (H == Y || H == X || Y == X) return CUSYNC_ERR_INVALID_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return CUSYNC_ERR_UNSUPPORTED;
  uint32_t* scratch = nullptr;
  if ((st = noalloc_setup(dev, &scratch)) != CUSYNC_OK) return st;
  int dev_sms = 0;
  if (query_num_sms(0, &dev_sms) != 0) return CUSYNC_ERR_CUDA;
  const int sms = d->num_sms > 0 ? std::min(d->num_sms, dev_sms) : dev_sms;

  ChainArgs A;
  std::memset(&A, 0, sizeof(A));
  if (!encode_maps(dd, p, A, X, W1t, W2t, H, Y)) return CUSYNC_ERR_INVALID_ARG;
  fill_static_args(dd, p, scratch, nullptr, A);
  A.st[0].out = H;
  A.st[1].out = Y;
  const int max_clusters = g_noalloc_clusters[dev][p.bn == 256 ? 0 : (p.bn == 128 ? 1 : 2)];
  if (p.pair == 2 && max_clusters < 1) return CUSYNC_ERR_UNSUPPORTED;
  const Grids grids = make_grids(p, sms, max_clusters);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Clear what must start at zero: error word, tile counters, run count, semaphores.
  e = cudaMemsetAsync(scratch, 0, (size_t)words * sizeof(uint32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "no-alloc scratch clear");
  if ((st = launch_run(dd, p, A, grids, H, sms, s)) != CUSYNC_OK) return st;
  if (error_word) {
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
    if ((e = cudaMemcpy(error_word, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost)) != cudaSuccess)
      return cuda_fail(e, "error word read");
    if (*error_word != 0) return (*error_word >> 24) == ERRC_PIPELINE ? CUSYNC_ERR_DEVICE : CUSYNC_ERR_TIMEOUT;
  }
  return CUSYNC_OK;
}
