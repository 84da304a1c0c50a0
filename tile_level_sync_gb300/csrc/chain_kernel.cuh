// The chain kernel: a persistent, warp-specialised tcgen05 GEMM that runs producer
// tiles, consumer tiles, or both from one tile queue, with the synchronisation of
// "A Framework for Fine-Grained Synchronization of Dependent GPU Kernels" (cuSync)
// and of the CUDA Programming Guide §4.6 "Fine-Grained Synchronization" (CUDA-FGS).
//
// One CTA per SM (PAIR = 1) or one CTA pair per two SMs in a cluster of 2 (PAIR = 2).
// Roles inside each CTA (256 threads):
//   warp 0, lane 0  TMA issuer (+ scheduler in the leader CTA).  The scheduler claims
//                   tiles from a global counter in queue order (cuSync §IV-C: each
//                   kernel takes its next tile from a per-stage counter) and hands them
//                   to every role of the CTA (and of the peer CTA) through a
//                   shared-memory ring.  The loader streams this CTA's rows of A and its
//                   share of B into a multi-stage shared-memory ring with TMA.  For a
//                   consumer tile it waits on the producer's semaphores before each A
//                   load and, while a semaphore is still short, issues the weight (B)
//                   loads of the next stages (cuSync §V, "Reorder Tile Loads and
//                   Synchronization").
//   warp 1          TMEM owner and (leader) MMA issuer.  It waits for each stage to land
//                   (or, for a tile under the sentinel check, to be checked); lane 0
//                   issues tcgen05.mma (128 x BN x 16 per CTA, or 256 x BN x 16 across
//                   the pair with cta_group::2, bf16 in, fp32 accumulate into TMEM) and
//                   commits each stage back to the loaders of both CTAs.
//   warp 7          sentinel checker (sentinel policy only).  It waits for each landed
//                   stage of a consumer tile, scans every A element for the 0x8000
//                   pattern and re-issues the A load while the pattern is present
//                   (CUDA-FGS §4.6.4.4 and §4.6.7, in software: sm_103a has no copy-time
//                   validity report), then arrives on the MMA issuer's `ready` barrier
//                   (the leader's, in a pair), so that the scan overlaps the MMAs of the
//                   stages before it.
//   warp 6          L2 prefetch of the weight boxes a few k-blocks ahead of the loader.
//   warps 2..5      epilogue.  tcgen05.ld of this CTA's 128 accumulator rows
//                   (double-buffered in TMEM so the next tile's mainloop overlaps this
//                   epilogue), GeLU / SwiGLU / ReLU, bf16 round-to-nearest-even, -0 -> +0
//                   (CUDA-FGS §4.6.4.3), then TMA stores of 32-row x 64-column boxes
//                   (GEMM outputs) or 16-byte stores (convolution outputs); for a
//                   producer tile one thread posts the tile's semaphore
//                   after all of the CTA's stores (cuSync §IV-E "Post": barrier,
//                   device-scope fence, atomic increment).  Each CTA of a pair posts its
//                   own half, so a pair tile's semaphore receives two posts.
//
// The pipelining follows the load-compute rules of "ALCOP: Automatic Load-COmpute
// Pipelining in Deep Learning Compiler for AI-GPUs" (pipelining rules): only buffers
// filled by asynchronous copies in a sequential k-loop are multi-buffered, each with its
// own barrier.
//
// Every wait is bounded by %globaltimer.  A semaphore or sentinel wait that expires
// records an error word and lets the CTA run to completion on whatever data is present;
// a pipeline (mbarrier) wait that expires also raises a CTA-local abort so the other
// roles drain.  Nothing traps.
#pragma once
#include <cuda_bf16.h>

#include "geometry.h"
#include "ptx.cuh"

namespace cusync {

// Control words in front of the semaphore array.
// Tile counters and exit counters: one per launch of a chain run (queue 0 .. kMaxQueues-1;
// a run launches at most one kernel per stage).
constexpr int kMaxQueues = 16;
enum : int {
  CTRL_ERR = 0,
  CTRL_ERR_DETAIL = 1,
  CTRL_RUNS = 8,
  CTRL_COUNTER = 16,
  CTRL_EXIT = CTRL_COUNTER + kMaxQueues,
  CTRL_WORDS = CTRL_EXIT + kMaxQueues
};
// Error classes (bits 31..24 of the error word; bits 23..0 hold the tile index).
enum : uint32_t { ERRC_FLAG_TIMEOUT = 1, ERRC_SENTINEL_TIMEOUT = 2, ERRC_PIPELINE = 3 };
// Flag bits shared with cusync.h.
constexpr uint32_t kFlagNoReorder = 1u << 0;
constexpr uint32_t kDebugSkipPost = 1u << 8;
constexpr uint32_t kDebugSkipSplit = 1u << 10;
// Semaphores read in one round trip when a wait finds its semaphore not yet known ready.
constexpr int kProbe = 32;

struct StageArgs {
  CUtensorMap tmA;       // activations: 2-D [M, K] or 4-D NHWC image
  CUtensorMap tmB;       // weights [N (or 2*N1), K]
  CUtensorMap tmO;       // GEMM output [M, N]: 64-column x 32-row store boxes, 128-byte swizzle
  void* out;             // bf16 [M, N] row-major (conv: [pixels, channels])
  const uint16_t* a_ptr; // activations [a_rows, K] row-major (read directly by the pointwise stage)
  const uint16_t* b_ptr; // weights [b_rows, K] row-major
  int32_t a_rows, b_rows;
  StageGeo g;
  int32_t b_half_rows;   // SwiGLU: row offset of the up-projection half of B
  // Operand maps that are 3-D k-block views [K/64][rows][64] (box {64, rows, KPS}): one
  // copy brings all of a pipeline stage's k-blocks.  Otherwise the map is 2-D (or the
  // convolution / stack map) and a stage takes one copy per k-block.
  int32_t a3d, b3d;
};

// One tile of a traced run (same layout as cusync_trace_rec_t).
struct TraceRec {
  uint32_t tile, smid, cta, stage;
  uint64_t t_claim, t_ready, t_mma0, t_mma1, t_epi, t_post;
  uint32_t polls, reloads;
  uint32_t land_clk, check_clk;
  uint64_t t_acc, t_xchg;
};

// A stage's weight (B) copies, armed by the loader and issued by the B-copy warp.
struct BCmd {
  const CUtensorMap* tm;
  int32_t kglob;        // the stage's first k-block in the tile's K
  int32_t nk;           // k-blocks of the stage
  int32_t brow0, brow1; // B rows of this CTA's share (brow1 >= 0: SwiGLU up rows on a single CTA)
  int32_t zs;           // stack: the weights' stage coordinate, else -1
  uint32_t mode;        // bit 0: one 3-D box of the stage; bit 1: complete on the pair leader's barrier
  int32_t _pad[2];
};

struct ChainArgs {
  StageArgs st[3];       // 0 = producer, nst - 1 = the GEMM consumer (attention: 1 = pointwise);
                         // convolution stack: 0 = the first stage, 1 = every later stage
  DepCfg dep;            // what the last stage waits for on the stage before it
  DepCfg dep_pw;         // attention: what the pointwise stage waits for on stage 0
  uint32_t* flags;       // semaphores of `dep`
  uint32_t* flags_pw;    // semaphores of `dep_pw`
  uint32_t* band_flags;  // MLP chains with row bands: one semaphore per band of consumer row tiles,
                         // posted once per CTA by each consumer tile of the band after its stores
  int32_t n_bands;
  uint32_t* ctrl;        // CTRL_* words
  TraceRec* trace;       // per-tile timeline, or null
  float* split_ws;       // K split: fp32 partial sums, per (tile, pair rank) ksplit-1 slots of 128 x BN;
                         // every word not holding a sum holds kSplitEmpty
  float* split_ws1;      // the same for a K-split consumer (stage 1 of a two-stage chain)
  int32_t queue;         // tile counter slot used by this launch
  int32_t first_stage;   // stages served by this launch: [first_stage, last_stage]
  int32_t last_stage;
  int32_t tiles0, tiles1, tiles2;
  int32_t nst;           // stages in the chain: 2, 3 (attention), or a stack's depth
  int32_t stack;         // convolution stack: stages 1 .. nst-1 share st[1], read the
                         // intermediate of the stage before them and write their own
  int32_t nbuf;          // stack: intermediate buffers in st[0].out; stage s writes s % nbuf
  int32_t flags_stride;  // stack: semaphores per stage boundary (boundary s at s * stride)
  int64_t buf_elems;     // stack: elements of one intermediate buffer
  // Stack under the sentinel policy: two sets of nst - 1 buffers used in turn, run r in
  // set r % 2; the launch that serves the last stage ends with fill units that write the
  // sentinel over the other set, ready for the next run.
  int32_t rotate;
  int32_t fill_units;
  int64_t fill_unit_chunks;  // 16-byte chunks per fill unit
  int64_t set_chunks;        // 16-byte chunks of one set
  uint32_t flags_bits;
  int32_t pdl_role;      // bit 0: trigger dependents at start; bit 1: wait on the primary at exit;
                         // bit 2: the run's first launch, started early (programmatic launch after
                         // the kernel before it in the stream): wait for that kernel before
                         // reading the run number or touching global memory;
                         // bit 3: the run's last launch: trigger dependents once this CTA has
                         // claimed its last tile;
                         // bit 4: started early after the sentinel fill of the intermediate (a
                         // programmatic dependent that lets this launch start once the run before
                         // has ended): wait for the fill before the first store or load of the
                         // intermediate
  int32_t sentinel_check;
  int32_t num_flags;     // semaphores in `flags`
  int32_t l2_prefetch;   // k-blocks the prefetch warp runs ahead of the loader (0: none)
  int32_t _pad;
  uint64_t timeout_ns;       // semaphore / sentinel waits
  uint64_t pipe_timeout_ns;  // shared-memory pipeline waits
};

template <int BN, int PAIR>
struct KCfg {
  static constexpr int kTileM = 128 * PAIR;          // output rows per tile (pair tile)
  static constexpr int kBRows = BN / PAIR;           // B rows held by each CTA
  static constexpr int kABytes = 128 * kBK * 2;      // this CTA's 128 rows of A
  static constexpr int kBBytes = kBRows * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (192 * 1024) / kStageBytes;  // 4, 6 or 8
  // k-blocks per pipeline stage: in a CTA pair two consecutive k-blocks share a stage and,
  // for GEMM operands, one copy (a 3-D box of two k-blocks).  Each copy costs the SM a
  // fixed time whatever its size (measured on a minimal copy->MMA pipeline of CTA pairs
  // with operands in L2: 417 ns per k-block with one copy per operand and k-block, 262 ns
  // with one per two k-blocks), so halving the copies lifts the mainloop towards the L2
  // port and tensor rates.  A single CTA keeps one k-block per stage: its stages of two
  // k-blocks measured 5-10% slower on the attention and convolution chains (a drained
  // stage is refilled only once both of its k-blocks are consumed, which leaves fewer
  // bytes in flight).  Sentinel-checked pair kernels take two k-blocks per stage too: both
  // checker warps then scan every stage, one k-block each.
  __host__ __device__ static constexpr int kps(bool check) { return (PAIR == 2 && kStages >= 6) ? 2 : 1; }
  // Two fp32 accumulators of BN columns, kAccStride columns apart.  A TMEM allocation is
  // a power of two of columns: a 192-wide tile's accumulators start at columns 0 and 256
  // of a 512-column allocation.
  static constexpr int kAccStride = (BN & (BN - 1)) == 0 ? BN : 256;
  static constexpr int kTmemCols = 2 * kAccStride;
  static constexpr int kSlots = 4;                   // tile hand-off ring
  // Warps: 0 loader, 1 MMA, 2..5 epilogue, 6 prefetch; then, under the sentinel policy,
  // the checkers (7..8 on single CTAs, 7..10 on CTA pairs, whose stages hold two k-blocks:
  // each checker scans half of one), and a second group of epilogue warps (two warps per
  // TMEM lane quarter, each storing every other 64-column box of a tile): 7..10 without
  // the checkers, 11..14 after them on CTA pairs (15 warps, 128 registers a thread; the
  // sentinel policy's GPT-3 M=256 / M=512 MLP chains 91.3 / 146.0 against 93.2 / 150.1 us
  // with one group).  Single-CTA sentinel kernels keep one group: 13 warps would also
  // cap them at 128 registers, where they spill.
  // Single-CTA kernels without the checkers issue each stage's weight (B) copies from
  // warp 11 (split_b): their loader, with one copy per operand and k-block, bounds the
  // mainloop, and the stacks of short convolution tiles measured 2-4% faster with the
  // second issuer (ResNet-38 28x28x128: 157.7 against 163.2 us); CTA pairs, which bring two
  // k-blocks per copy, measured 2-9% slower with it (GPT-3 M=1024: 226.4 against 208.6 us).
  __host__ __device__ static constexpr int epi_warps(bool check) { return (check && PAIR == 1) ? 4 : 8; }
  __host__ __device__ static constexpr int check_warps() { return PAIR == 2 ? 4 : 2; }
  // first warp of the second epilogue group: after the checkers when there are any
  __host__ __device__ static constexpr int epi2_warp(bool check) { return check ? 7 + check_warps() : 7; }
  __host__ __device__ static constexpr bool split_b(bool check) { return !check && PAIR == 1; }
  static constexpr int threads(bool check) {
    return 32 * (check ? 7 + check_warps() + (epi_warps(check) - 4) : (split_b(check) ? 12 : 11));
  }
  // epilogue staging for TMA stores: 32-row x 64-column bf16 boxes, 32 KB in all (two
  // boxes per epilogue warp with four warps, one with eight)
  static constexpr int kEpiBufBytes = 32 * 64 * 2;
  static constexpr int kEpiBytes = 8 * kEpiBufBytes;
  __host__ __device__ static constexpr int epi_bufs(bool check) { return 8 / epi_warps(check); }
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 1024 + kEpiBytes;
};

struct TileRef {
  int32_t s, m, c;
  int32_t ks;   // K-split unit of the tile (0 without a split)
  int32_t kb0;  // first k-block of the unit
  int32_t nkb;  // k-blocks of the unit
  int32_t q;    // the unit's position among the launch's work units (fill units not counted)
};

// Work units of stage s.
__device__ __forceinline__ int32_t stage_tiles(const ChainArgs& a, int32_t s) {
  return a.stack ? a.tiles0 : (s == 0 ? a.tiles0 : (s == 1 ? a.tiles1 : a.tiles2));
}

// Operands and geometry of stage s.
__device__ __forceinline__ const StageArgs& stage_args(const ChainArgs& a, int32_t s) {
  return a.st[a.stack ? (s > 0 ? 1 : 0) : s];
}

// Whether stage s reads the output of the stage before it (waits on it, or checks it).
__device__ __forceinline__ bool stage_consumes(const ChainArgs& a, int32_t s) {
  return a.stack ? s > 0 : s == a.nst - 1;
}

// Stack: the intermediate buffer that stage s (< nst - 1) writes.  With two buffers a
// stage overwrites the input of the stage before it; the tile's own waits have covered
// every reader of what it overwrites by the time it stores (it stores after its last
// k-block, and each semaphore it waited on was posted after that tile's reads).
// Under the sentinel policy the run's set comes first: run r uses set r % 2.
__device__ __forceinline__ int32_t stack_buf(const ChainArgs& a, int32_t s, uint32_t run) {
  return a.rotate ? (int32_t)(run & 1u) * (a.nst - 1) + s : s % a.nbuf;
}

// Fill units (see ChainArgs::rotate) follow the work units in the queue of the launch that
// serves the last stage, so the CTAs that run out of work in the last wave write them.
// They wait on nothing, so the order of the work units, and with it the argument that no
// wait can deadlock, is unchanged.
constexpr int32_t kFillStage = -1;

__device__ __forceinline__ TileRef decode_tile(const ChainArgs& a, int32_t t) {
  if (a.fill_units > 0 && a.last_stage == a.nst - 1) {
    int32_t units = 0;
    for (int32_t s = a.first_stage; s <= a.last_stage; ++s) units += stage_tiles(a, s);
    if (t >= units) return TileRef{kFillStage, t - units, 0, 0, 0, 0, -1};
  }
  const int32_t q = t;
  // the launch serves stages [first_stage, last_stage], their work units in that order
  int32_t s = a.first_stage, u = t;
  while (s < a.last_stage) {
    const int32_t n = stage_tiles(a, s);
    if (u < n) break;
    u -= n;
    ++s;
  }
  const StageGeo& g = stage_args(a, s).g;
  int32_t ks = 0, kb0 = 0, nkb = g.k_blocks;
  if (g.ksplit > 1) {
    ks = u % g.ksplit;
    u /= g.ksplit;
    split_unit(g, ks, &kb0, &nkb);
  }
  int32_t m, y;
  tile_at(g, u, &m, &y);
  // StridedSync's producer order applies to the stage whose semaphores it groups
  const DepCfg& pd = (a.nst == 3) ? a.dep_pw : a.dep;
  const int32_t c = (s == 0) ? producer_col(pd, y) : y;
  return TileRef{s, m, c, ks, kb0, nkb, q};
}

// Index of queue position t in the chain's tile numbering (producer tiles first).
__device__ __forceinline__ int32_t chain_tile(const ChainArgs& a, int32_t t) {
  for (int32_t s = 0; s < a.first_stage; ++s) t += stage_tiles(a, s);
  return t;
}

__device__ __forceinline__ uint32_t a_tile_bytes(const StageGeo& g) {
  return g.a_mode == AMODE_GEMM ? (uint32_t)(128 * kBK * 2) : (uint32_t)(g.img_w * g.th * kBK * 2);
}

// This CTA's A k-block: rows [m*tile_m + rank*128, +128) of a GEMM, or the conv box.
// With to_leader, the copy's completion is counted on the pair leader's barrier `bar`.
template <int PAIR>
__device__ __forceinline__ void issue_a(const ChainArgs& a, const TileRef& tr, int32_t kb, uint32_t rank, void* dst,
                                        uint64_t* bar, uint64_t pol, int32_t a_buf, bool to_leader = false) {
  const StageArgs& S = stage_args(a, tr.s);
  if (S.g.a_mode == AMODE_GEMM) {
    const int32_t row = tr.m * (128 * PAIR) + (int32_t)rank * 128;
    if (PAIR == 2 && to_leader) ptx::tma_load_2d_to_leader(dst, &S.tmA, ptx::mapa(bar, 0), kb * kBK, row, pol);
    else ptx::tma_load_2d(dst, &S.tmA, bar, kb * kBK, row, pol);
  } else {
    // implicit im2col: filter tap (r, s), channel block cb; the box is TH image rows of
    // one image shifted by (r-1, s-1); rows or columns outside the image are zero-filled.
    const int32_t tap = kb / S.g.cblocks, cb = kb % S.g.cblocks;
    const int32_t r = tap / 3, s = tap % 3;
    const int32_t n = tr.m / S.g.tpi, hb = tr.m % S.g.tpi;
    if (a_buf >= 0)  // the stack's intermediates: one more coordinate, the buffer
      ptx::tma_load_5d(dst, &S.tmA, bar, cb * kBK, s - 1, hb * S.g.th + r - 1, n, a_buf, pol);
    else
      ptx::tma_load_4d(dst, &S.tmA, bar, cb * kBK, s - 1, hb * S.g.th + r - 1, n, pol);
  }
}

// Row of B where this CTA's share of the weight tile starts.  A single CTA holds the BN
// rows of its column tile (SwiGLU: BN/2 gate rows then BN/2 up rows); in a pair the
// leader holds the first half and the peer the second, which for SwiGLU are the gate
// and up rows.
template <int BN, int PAIR>
__device__ __forceinline__ int32_t b_row(const StageArgs& S, const TileRef& tr, uint32_t rank, int half) {
  if (S.g.epi == EPI_SWIGLU) {
    const int32_t row0 = tr.c * (BN / 2);
    const int which = PAIR == 2 ? (int)rank : half;
    return which == 0 ? row0 : S.b_half_rows + row0;
  }
  return tr.c * BN + (PAIR == 2 ? (int32_t)rank * (BN / 2) : 0);
}

__device__ __forceinline__ void record_error(const ChainArgs& a, uint32_t cls, int32_t tile, int32_t detail) {
  const uint32_t w = (cls << 24) | ((uint32_t)tile & 0xFFFFFFu);
  if (atomicCAS(a.ctrl + CTRL_ERR, 0u, w) == 0u) atomicExch(a.ctrl + CTRL_ERR_DETAIL, (uint32_t)detail);
}

// Bit 15 (bit 31) of the result is set when the low (high) bf16 half of x is the sentinel
// 0x8000; the other bits are don't-care.  x ^ 0x80008000 turns a sentinel half into a zero
// half, and (t - 0x00010001) & ~t has the top bit of a half set exactly when some half is
// zero (a borrow out of a zero low half can only add a flag when one is already raised).
// Three integer operations per word, so results can be OR-ed together and tested once.
__device__ __forceinline__ uint32_t sentinel_bits_bf16x2(uint32_t x) {
  const uint32_t t = x ^ 0x80008000u;
  return (t - 0x00010001u) & ~t;
}


// K-split workspace words that hold no partial sum hold kSplitEmpty, a NaN (sign set,
// all payload bits set); a unit stores a sum equal to it as the canonical NaN instead,
// so a word holds either kSplitEmpty or a sum.
constexpr uint32_t kSplitEmpty = 0xFFFFFFFFu;
__device__ __forceinline__ uint32_t split_canon(uint32_t x) { return x == kSplitEmpty ? 0x7FFFFFFFu : x; }
__device__ __forceinline__ bool split_empty(const uint4& v) {
  return (v.x == kSplitEmpty) | (v.y == kSplitEmpty) | (v.z == kSplitEmpty) | (v.w == kSplitEmpty);
}

__device__ __forceinline__ uint32_t canon_bf16x2(uint32_t x) {
  uint32_t lo = x & 0xFFFFu, hi = x >> 16;
  lo = (lo == 0x8000u) ? 0u : lo;
  hi = (hi == 0x8000u) ? 0u : hi;
  return lo | (hi << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // round to nearest even; a -> low half
  return canon_bf16x2(*reinterpret_cast<uint32_t*>(&v));
}

// The activations use the hardware tanh approximation (PTX tanh.approx.f32, one MUFU
// operation; relative error about 2^-11, far below a bf16 half-ulp of 2^-9):
// tanh-GeLU 0.5 z (1 + tanh u) with u = sqrt(2/pi) (z + 0.044715 z^3), and
// silu(g) = g sigmoid(g) = 0.5 g (1 + tanh(g / 2)).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gelu_f(float z) {
  const float u = 0.7978845608028654f * fmaf(0.044715f * z, z * z, z);
  const float h = 0.5f * z;
  return fmaf(h, tanh_approx(u), h);
}
__device__ __forceinline__ float silu_f(float g) {
  const float h = 0.5f * g;
  return fmaf(h, tanh_approx(h), h);
}

// Attention chain, pointwise tile (m, head i), run by the 128 epilogue threads (one token
// row each): once the QKV GEMM's tiles it reads are posted (cuSync §IV-E waits on the
// semaphores of the policy -- StridedSync groups a head's three Q/V/K tiles), each thread
// computes s_j = q_j v_j over the head's kHead columns, p = softmax(s) over the head, and
// XDot_j = p_j k_j ("A Framework for Fine-Grained Synchronization of Dependent GPU
// Kernels", Fig. fig:gpt-3:attention, fused dot-product kernel; dropout is the identity
// of inference).  Two passes over the row: an online maximum and sum of exponentials,
// then the outputs.  Then cuSync §IV-E "Post" for the GEMM that reads XDot.
__device__ __noinline__ void pointwise_tile(const ChainArgs& args, const TileRef& tr, int32_t t, int64_t grow,
                                            uint64_t* pw_done, uint32_t pw_parity, uint32_t runs, bool leader,
                                            uint64_t pto, volatile int32_t* abort_flag) {
  const StageArgs& SA = stage_args(args, tr.s);
  const StageGeo& g = SA.g;
  Wait w[3];
  const int nw = pointwise_waits(args.dep_pw, tr.m, tr.c, w);
  for (int i = 0; i < nw; ++i) {
    const uint32_t target = runs * w[i].per_run;
    const uint64_t t0 = ptx::globaltimer();
    while ((int32_t)(ptx::ld_acquire_gpu(args.flags_pw + w[i].flag) - target) < 0) {
      __nanosleep(64);
      if (ptx::ld_relaxed_gpu(args.ctrl + CTRL_ERR) != 0u) break;
      if (ptx::globaltimer() - t0 > args.timeout_ns) {
        record_error(args, ERRC_FLAG_TIMEOUT, t, w[i].flag & 0xFFFF);
        break;
      }
    }
  }
  if (grow < g.M) {  // this thread's token row (a CTA of a pair holds 128 of the tile's 256)
    const int32_t n1 = g.N;
    const uint16_t* xr = SA.a_ptr + grow * (int64_t)g.K + (int64_t)tr.c * kHead;  // XQKV row: Q | V | K
    const uint4* qp = reinterpret_cast<const uint4*>(xr);
    const uint4* vp = reinterpret_cast<const uint4*>(xr + n1);
    const uint4* kp = reinterpret_cast<const uint4*>(xr + 2 * n1);
    auto lo = [](uint32_t x) { return __uint_as_float(x << 16); };
    auto hi = [](uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); };
    float mx = -INFINITY, sum = 0.0f;
    for (int j = 0; j < kHead / 8; ++j) {
      const uint4 a = __ldcg(qp + j), b = __ldcg(vp + j);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float sv = (e & 1) ? hi(av[e / 2]) * hi(bv[e / 2]) : lo(av[e / 2]) * lo(bv[e / 2]);
        if (sv > mx) {
          sum = sum * __expf(mx - sv) + 1.0f;
          mx = sv;
        } else {
          sum += __expf(sv - mx);
        }
      }
    }
    const float inv = 1.0f / sum;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(SA.out) + grow * (int64_t)n1 + (int64_t)tr.c * kHead;
    for (int j = 0; j < kHead / 8; ++j) {
      const uint4 a = __ldcg(qp + j), b = __ldcg(vp + j), c = __ldcg(kp + j);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w}, cv[4] = {c.x, c.y, c.z, c.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = __expf(lo(av[e]) * lo(bv[e]) - mx) * inv;
        const float p1 = __expf(hi(av[e]) * hi(bv[e]) - mx) * inv;
        o[e] = pack_bf16x2(p0 * lo(cv[e]), p1 * hi(cv[e]));
      }
      ptx::st_relaxed_gpu_b128(orow + j * 8, o[0], o[1], o[2], o[3]);
    }
  }
  ptx::mbar_arrive(pw_done);
  if (threadIdx.x == 64) {
    if (!ptx::mbar_wait_bounded(pw_done, pw_parity, pto)) {
      record_error(args, ERRC_PIPELINE, t, 8);
      *abort_flag = 1;
    } else {
      const int32_t flag = producer_flag(args.dep, tr.m, tr.c);
      if (flag >= 0) {
        ptx::fence_acq_rel_gpu();
        ptx::red_release_gpu_add(args.flags + flag, 1u);
      }
      if (args.trace && leader) {
        args.trace[chain_tile(args, tr.q)].t_epi = ptx::globaltimer();
        args.trace[chain_tile(args, tr.q)].t_post = ptx::globaltimer();
      }
    }
  }
  __syncwarp();
}

// Bounded waits on barriers that may receive arrivals from the other CTA of a pair use
// cluster-scope acquire.
template <int PAIR>
__device__ __forceinline__ bool xwait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (PAIR == 2) return ptx::mbar_wait_bounded_cluster(bar, parity, timeout_ns);
  return ptx::mbar_wait_bounded(bar, parity, timeout_ns);
}

// CHECK: the sentinel policy's instantiation, with the two checker warps (the host sets
// args.sentinel_check to match); every other policy runs without them.
template <int BN, int PAIR, bool CHECK>
__global__ void __launch_bounds__(KCfg<BN, PAIR>::threads(CHECK), 1) chain_kernel(const __grid_constant__ ChainArgs args) {
  using C = KCfg<BN, PAIR>;
  constexpr int S = C::kStages;          // k-block buffers of the ring
  constexpr int KPS = C::kps(CHECK);     // k-blocks per stage
  constexpr int NS = S / KPS;            // stages; stage st holds buffers st*KPS .. st*KPS+KPS-1
  static_assert(S % KPS == 0, "whole stages");
  constexpr uint32_t FULL = 0xFFFFFFFFu;
  constexpr bool kPair = PAIR == 2;
  constexpr int kEpiWarps = C::epi_warps(CHECK);
  constexpr int kEpiGroups = kEpiWarps / 4;  // epilogue warps per TMEM lane quarter
  constexpr int kEpi2 = C::epi2_warp(CHECK);  // first warp of the second epilogue group
  constexpr int kEpiBufs = C::epi_bufs(CHECK);  // staging boxes per epilogue warp

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::kStageBytes);
  uint64_t* full = bars;                  // [S]   this CTA's A+B (or A retry) landed
  uint64_t* empty = full + S;             // [S]   the MMA finished reading the stage
  uint64_t* ready = empty + S;            // [S]   checked tile: the stage passed the check (both CTAs')
  uint64_t* tfull = ready + S;            // [2]   accumulator ready
  uint64_t* tempty = tfull + 2;           // [2]   accumulator drained (leader in a pair)
  uint64_t* epi_done = tempty + 2;        // [2]   all epilogue threads of this CTA stored the tile
  uint64_t* qfull = epi_done + 2;         // [slots] tile index published
  uint64_t* qempty = qfull + C::kSlots;   // [slots] tile index consumed (leader in a pair)
  uint64_t* mma_done = qempty + C::kSlots;
  uint64_t* pw_done = mma_done + 1;       // attention: all epilogue threads stored a pointwise tile
  uint64_t* cfull = pw_done + 1;          // [S]   sentinel-checked tile: this CTA's A+B (or A retry) landed
  int32_t* qtile = reinterpret_cast<int32_t*>(cfull + S);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qtile + C::kSlots);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  volatile int32_t* it_issued = abort_flag + 1;
  volatile uint32_t* progress = reinterpret_cast<volatile uint32_t*>(it_issued + 1);  // k-blocks issued
  volatile uint32_t* run_no = progress + 1;  // this launch's run number, for every role
  // per stage: whether its last copy completes on cfull (1) or full (0)
  volatile uint8_t* stage_kind = reinterpret_cast<volatile uint8_t*>(run_no + 1);
  // pair, sentinel check: words the peer's checker stores into to signal `ready` (S <= 8)
  uint32_t* ready_sink = const_cast<uint32_t*>(run_no + 3);
  // sentinel check with two k-blocks per stage: each checker warp's finding per round (two
  // rounds in turn), and the barrier the checkers arrive on once they wrote it
  volatile uint32_t* scan_flag = run_no + 11;  // [2][4]
  // B copies issued by warp 11 (kernels without the checkers): commands armed by the loader
  // so far, whether the loader is done, and one command per stage slot
  volatile uint32_t* b_posted = run_no + 22;
  volatile uint32_t* b_stop = run_no + 23;
  BCmd* bcmd = reinterpret_cast<BCmd*>(reinterpret_cast<uint8_t*>(bars) + 512);
  uint64_t* scan_done = reinterpret_cast<uint64_t*>(const_cast<uint32_t*>(run_no + 20));  // 8-byte aligned
  uint8_t* epi_stage = smem + S * C::kStageBytes + 1024;  // 1024-byte aligned TMA store boxes

  // Stage st holds its k-blocks' A tiles one after the other, then their B tiles (the
  // layout of a 3-D box of KPS k-blocks); k-block h of the stage is at smem_a(st, h).
  auto smem_a = [&](int st, int h = 0) { return stage_base + st * KPS * C::kStageBytes + h * C::kABytes; };
  auto smem_b = [&](int st, int h = 0) {
    return stage_base + st * KPS * C::kStageBytes + KPS * C::kABytes + h * C::kBBytes;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  // A pair tile without the sentinel check is loaded "direct": the peer's copies complete
  // on the leader's `full` barriers, which count the bytes of both CTAs.  A consumer tile
  // under the sentinel policy is not: each CTA's copies complete locally, its checker
  // validates them and arrives on the leader's `ready` barrier.
  auto direct_tile = [&](const TileRef& tr) { return kPair && !(CHECK && stage_consumes(args, tr.s)); };

  // Run number of this launch.  Semaphores count up across runs (run r waits for r times
  // the posts of one run), and the count of finished runs lives in device memory, so the
  // same launch can be replayed from a CUDA graph.  Read before the first barrier: the
  // launch that increments it (below: the last stage's, once all of its CTAs have claimed
  // their last tile) does so only after every CTA of its own launch has passed that point,
  // and a later stage's launch starts only after every CTA of this one has triggered its
  // dependents, which it does after that barrier.
  uint32_t epoch = 0;

  if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < S; ++i) {
        ptx::mbar_init(&full[i], 1);
        ptx::mbar_init(&empty[i], 1);
        ptx::mbar_init(&ready[i], 1);
        ptx::mbar_init(&cfull[i], 1);
        stage_kind[i] = 0;
      }
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(&tfull[i], 1);
        ptx::mbar_init(&tempty[i], kPair ? 2 * kEpiWarps : 32 * kEpiWarps);
        ptx::mbar_init(&epi_done[i], 32 * kEpiWarps);
      }
      for (int i = 0; i < C::kSlots; ++i) {
        ptx::mbar_init(&qfull[i], 1);
        // consumers of a slot: MMA warp, the epilogue warps, the prefetch warp and, under
        // the sentinel policy, the two checker warps (+ the peer's loader and the same
        // warps in a pair)
        const uint32_t nloc = 2u + (uint32_t)kEpiWarps + (CHECK ? (uint32_t)C::check_warps() : 0u);
        ptx::mbar_init(&qempty[i], kPair ? 2u * nloc + 1u : nloc);
      }
      ptx::mbar_init(mma_done, 1);
      ptx::mbar_init(pw_done, 128);
      ptx::mbar_init(scan_done, (uint32_t)C::check_warps());
      *abort_flag = 0;
      *it_issued = 0;
      *progress = 0;
      *b_posted = 0;
      *b_stop = 0;
      ptx::mbar_init_fence();
    }
    __syncwarp();
    if (kPair) {
      ptx::tmem_alloc_pair(tmem_slot, C::kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, C::kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    for (int s = args.first_stage; s <= args.last_stage; ++s) {
      const StageArgs& S = stage_args(args, s);
      ptx::prefetch_tmap(&S.tmA);
      ptx::prefetch_tmap(&S.tmB);
      if (S.g.a_mode == AMODE_GEMM) ptx::prefetch_tmap(&S.tmO);
      if (args.stack && s >= 1) break;  // the later stages of a stack share these maps
    }
    // A run's first launch may start while the kernel before it in the stream (the last
    // launch of the previous run, or any kernel of the caller) is finishing: everything
    // above touches no global memory; from here on this CTA needs that kernel complete and
    // its writes visible (CUDA-FGS §4.6.5, programmatic dependent launch).
    if (args.pdl_role & 4) ptx::pdl_wait();
    epoch = ptx::ld_relaxed_gpu(args.ctrl + CTRL_RUNS) + 1u;
    *run_no = epoch;
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (kPair) ptx::cluster_sync();  // the peer's barriers exist before any remote arrive
  ptx::tc_fence_after();
  if (args.pdl_role & 1) ptx::pdl_launch_dependents();  // after this CTA read the run number
  const uint32_t tmem_base = *tmem_slot;

  int32_t total = 0;
  for (int s = args.first_stage; s <= args.last_stage; ++s) total += stage_tiles(args, s);
  if (args.last_stage == args.nst - 1) total += args.fill_units;
  const uint64_t pto = args.pipe_timeout_ns;

  // Arrive on "consumed" for ring slot `slot` (the leader's barrier in a pair).
  auto ring_release = [&](int slot) {
    if (kPair && !leader) ptx::mbar_arrive_cluster(ptx::mapa(&qempty[slot], 0));
    else ptx::mbar_arrive(&qempty[slot]);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA
    if (lane == 0) {
      const uint64_t pol_a = ptx::l2_policy_evict_last();
      const uint64_t pol_b = ptx::l2_policy_evict_normal();
      const bool reorder = !(args.flags_bits & kFlagNoReorder);
      uint32_t it = 0, tcount = 0, pw_seen = 0;  // it: stages armed (every tile starts a stage)
      uint32_t kit = 0;                           // k-blocks loaded, for the prefetch warp
      // ring cursors: the slot (and the parity of its `empty` phase) of the next stage to
      // arm, and the slot of the next stage to receive its A copies; they advance one stage
      // at a time, which spares the loader a division per stage
      int b_slot = 0, a_slot = 0;
      uint32_t b_par = 1u;
      bool ok = true;
      bool fill_seen = false;  // pdl_role bit 4: the intermediate's fill has ended
      while (true) {
        const int slot = tcount % C::kSlots;
        const uint32_t tpar = (tcount / C::kSlots) & 1u;
        int32_t t;
        bool done;
        if (leader) {
          // Every tile, the first included, is claimed from the launch's counter (cuSync
          // §IV-C), so a tile is only ever held by a CTA that is running: a wait (always on
          // tiles earlier in the queue) never depends on a CTA that has not started, and
          // the grid needs no co-residency guarantee.  (Issuing the first claim at kernel
          // entry instead, to overlap its round trip with the set-up, measured 3-7% slower
          // with CTA pairs.)
          t = (int32_t)atomicAdd(args.ctrl + CTRL_COUNTER + args.queue, 1u);
          done = t >= total || !ok || *abort_flag;
          if (!xwait<PAIR>(&qempty[slot], tpar ^ 1u, pto)) {
            record_error(args, ERRC_PIPELINE, 0xFFFFFF, 1);
            *abort_flag = 1;
            done = true;
          }
          qtile[slot] = done ? -1 : t;
          if (kPair) {
            ptx::st_cluster_u32(ptx::mapa(&qtile[slot], 1), (uint32_t)(done ? -1 : t));
            ptx::mbar_arrive_cluster(ptx::mapa(&qfull[slot], 1));
          }
          ptx::mbar_arrive(&qfull[slot]);
        } else {
          if (!xwait<PAIR>(&qfull[slot], tpar, pto)) {
            record_error(args, ERRC_PIPELINE, 0xFFFFFF, 6);
            *abort_flag = 1;
            t = -1;
          } else {
            t = qtile[slot];
          }
          done = t < 0;
          ring_release(slot);
        }
        ++tcount;
        if (done) break;

        const TileRef tr = decode_tile(args, t);
        if (tr.s == kFillStage) continue;  // written by this CTA's epilogue warps; nothing to load
        if ((args.pdl_role & 16) && tr.s > 0 && !fill_seen) {
          ptx::pdl_wait();  // the sentinel fill of the intermediate has ended (pdl_role bit 4)
          fill_seen = true;
        }
        const StageArgs& SA = stage_args(args, tr.s);
        const int32_t KB = tr.nkb;            // k-blocks of this work unit
        const int32_t kx0 = tr.kb0 * kBK;     // its first reduction coordinate
        const uint32_t abytes = a_tile_bytes(SA.g);
        TraceRec* trec = (args.trace && leader) ? args.trace + chain_tile(args, tr.q) : nullptr;
        if (trec) {
          trec->tile = (uint32_t)chain_tile(args, tr.q);
          trec->smid = ptx::smid();
          trec->cta = blockIdx.x;
          trec->stage = (uint32_t)tr.s;
          trec->t_claim = ptx::globaltimer();
          trec->t_post = 0;
          trec->polls = 0;
          trec->reloads = 0;
          trec->land_clk = 0;
          trec->check_clk = 0;
          trec->t_acc = 0;
          trec->t_xchg = 0;
        }
        if (SA.g.a_mode == AMODE_POINTWISE) {
          // Computed by this CTA's epilogue warps; nothing to load.  The next claim waits
          // until they are done, so that the pointwise tiles spread over the CTAs instead
          // of queueing behind one CTA's epilogue.
          if (!ptx::mbar_wait_bounded(pw_done, pw_seen & 1u, pto) || *abort_flag) {
            record_error(args, ERRC_PIPELINE, t, 9);
            *abort_flag = 1;
            ok = false;
          }
          ++pw_seen;
          continue;
        }
        const bool cons = stage_consumes(args, tr.s);
        GemmDepTracker gdt;
        gdt.reset();
        ConvDepTracker cdt;  // touched (stack arrays) only by convolution tiles
        if (SA.g.a_mode != AMODE_GEMM) cdt.reset();
        int32_t snext = 0;   // next stage of this tile to arm (its slot drained, its B copies issued)
        // Per-tile invariants of the k-loop, so that the single loader thread spends as few
        // instructions per k-block as possible (its latency is on the critical path).
        const bool gemm = SA.g.a_mode == AMODE_GEMM;
        const CUtensorMap* tmA = &SA.tmA;
        const CUtensorMap* tmB = &SA.tmB;
        const int32_t a_row = tr.m * (128 * PAIR) + (int32_t)rank * 128;
        const int32_t brow0 = b_row<BN, PAIR>(SA, tr, rank, 0);
        const int32_t brow1 = (PAIR == 1 && SA.g.epi == EPI_SWIGLU) ? b_row<BN, PAIR>(SA, tr, rank, 1) : -1;
        const bool direct = direct_tile(tr);
        const bool to_leader = direct && !leader;
        const int32_t NSK = (KB + KPS - 1) / KPS;  // stages of this work unit
        // bytes a stage of nk k-blocks brings into this CTA: a 3-D box always brings KPS
        // k-blocks (past the unit's or the tensor's end: unused, or zero-filled)
        const bool a3d = SA.a3d != 0, b3d = SA.b3d != 0;
        auto stage_bytes = [&](int32_t nk) -> uint32_t {
          const uint32_t b = (uint32_t)(a3d ? KPS : nk) * abytes + (uint32_t)(b3d ? KPS : nk) * (uint32_t)C::kBBytes;
          return direct ? 2u * b : b;  // a direct pair tile: the leader's barrier counts both CTAs
        };
        const uint32_t tx_full = stage_bytes(KPS);  // a whole stage (every stage when KPS = 1)
        // a tile that the checker warp validates completes its copies on cfull, which only
        // the checker waits on; every other tile on full, which only the MMA issuer waits on
        const bool checked = CHECK && cons;
        uint64_t* const lbar = checked ? cfull : full;
        // Stack: stage s waits on the semaphores of the boundary it consumes (s - 1), reads
        // its input from that stage's buffer (the fifth coordinate of the intermediates'
        // map) and its weights from slice s of the stacked weights (the third coordinate).
        const bool stacked = args.stack != 0;
        const uint32_t* const wflags = args.flags + (stacked && tr.s > 0 ? (tr.s - 1) * args.flags_stride : 0);
        const int32_t wnflags = stacked ? args.flags_stride : args.num_flags;
        const int32_t a_buf = stacked && tr.s > 0 ? stack_buf(args, tr.s - 1, epoch) : -1;
        // k-blocks at which the consumer may have to wait (dep_kblock): every dep_every-th
        // k-block of a GEMM; for a convolution the first 64 k-blocks by a bit mask, every
        // later one by dep_every = 1.
        const int32_t pol = args.dep.policy;
        int32_t dep_every = 0;
        uint64_t dep_mask = 0;
        if (cons && (pol == POL_ROW || pol == POL_TILE || pol == POL_STRIDED)) {
          if (gemm) {
            // (a K-split unit of the consumer starts at a multiple of the period: the
            // planner aligns kb_per_split, so the test below needs no offset)
            dep_every = pol == POL_ROW ? KB + 1 : max(1, args.dep.prod_n_out / kBK);
          } else {
            for (int32_t k = 0; k < KB && k < 64; ++k)
              if (dep_kblock(SA.g, args.dep, k)) dep_mask |= 1ull << k;
            dep_every = 1;
          }
        }
        // convolution A coordinates of k-block kb, advanced incrementally: channel block,
        // filter column s and filter row r; image and first image row of the tile
        int32_t cv_cb = 0, cv_s = 0, cv_r = 0, cv_img = 0, cv_h0 = 0;
        if (!gemm) {
          cv_img = tr.m / SA.g.tpi;
          cv_h0 = (tr.m % SA.g.tpi) * SA.g.th - 1;
        }
        // Arm stage sj of the tile: wait for its slot to drain (blocking) or return 0 if it
        // has not (non-blocking), set the bytes its barrier expects and issue its weight (B)
        // copies -- one 3-D box of KPS k-blocks, or one copy per k-block.
        auto arm_b = [&](int32_t sj, bool blocking) -> int {
          const int st = b_slot;  // the slot of stage it + sj (sj is always the next to arm)
          const uint32_t par = b_par;
          if (blocking) {
            const int32_t aborted = *abort_flag;  // read before the wait: off the critical path
            if (!ptx::mbar_wait_bounded(&empty[st], par, pto) || aborted) return -1;
          } else if (!ptx::mbar_test_wait(&empty[st], par)) {
            return 0;
          }
          if (++b_slot == NS) {
            b_slot = 0;
            b_par ^= 1u;
          }
          if (CHECK) stage_kind[st] = checked ? 1 : 0;  // (always 0 without the checkers)
          const int32_t kb = sj * KPS;
          const int32_t nk = KPS == 1 ? 1 : min(KPS, KB - kb);
          if (!to_leader) ptx::mbar_arrive_expect_tx(&lbar[st], (KPS == 1 || nk == KPS) ? tx_full : stage_bytes(nk));
          if constexpr (C::split_b(CHECK)) {
            // the copies are the B-copy warp's: one command per stage slot (a slot's command
            // is rewritten only once its stage was consumed, hence its copies issued)
            BCmd& c = bcmd[st];
            c.tm = tmB;
            c.kglob = tr.kb0 + kb;
            c.nk = nk;
            c.brow0 = brow0;
            c.brow1 = brow1;
            c.zs = stacked ? tr.s : -1;
            c.mode = ((KPS > 1 && b3d) ? 1u : 0u) | (to_leader ? 2u : 0u);
            __threadfence_block();
            *b_posted = *b_posted + 1u;
            return 1;
          }
          if (KPS > 1 && b3d) {
            if (to_leader) ptx::tma_load_3d_to_leader(smem_b(st), tmB, ptx::mapa(&full[st], 0), 0, brow0, tr.kb0 + kb, pol_b);
            else ptx::tma_load_3d(smem_b(st), tmB, &lbar[st], 0, brow0, tr.kb0 + kb, pol_b);
            return 1;
          }
#pragma unroll
          for (int32_t h = 0; h < KPS; ++h) {
            if (h >= nk) break;
            uint8_t* dst = smem_b(st, h);
            const int32_t x = kx0 + (kb + h) * kBK;
            if (stacked) {
              ptx::tma_load_3d(dst, tmB, &lbar[st], x, brow0, tr.s, pol_b);
            } else if (to_leader) {
              ptx::tma_load_2d_to_leader(dst, tmB, ptx::mapa(&full[st], 0), x, brow0, pol_b);
            } else {
              ptx::tma_load_2d(dst, tmB, &lbar[st], x, brow0, pol_b);
              if (brow1 >= 0) ptx::tma_load_2d(dst + (BN / 2) * 128, tmB, &lbar[st], x, brow1, pol_b);
            }
          }
          return 1;
        };
        // Semaphores already seen at their target during this tile: [rc_lo, rc_hi).
        int32_t rc_lo = 0, rc_hi = 0;
        uint32_t rc_target = 0;
        // Semaphore waits before A k-block kb (cuSync §IV-E "Wait", bounded).  A wait
        // first probes a run of up to kProbe consecutive semaphores with relaxed loads
        // (one round trip) and remembers which already reached the target; only a
        // semaphore still short of its target is polled, with exponential back-off.
        // While polling, the weight loads of the following stages are issued as their
        // slots drain (cuSync §V "Reorder Tile Loads and Synchronization").  One acquire
        // fence after the observations orders the A-tile reads after the producer's
        // releases, and a proxy fence orders them for the TMA (async proxy).
        auto wait_deps = [&](int32_t kb) {
          Wait w[kMaxWaits];
          const int n = gemm ? gdt.next(args.dep, tr.m, tr.kb0 + kb, w) : cdt.next(SA.g, args.dep, tr.m, kb, w);
          bool observed = false;
          for (int i = 0; i < n; ++i) {
            const int32_t f = w[i].flag;
            const uint32_t target = epoch * w[i].per_run;
            if (target == rc_target && rc_lo <= f && f < rc_hi) continue;
            uint32_t v[kProbe];
            const int32_t cnt = min(kProbe, wnflags - f);
#pragma unroll
            for (int q = 0; q < kProbe; ++q) v[q] = q < cnt ? ptx::ld_relaxed_gpu(wflags + f + q) : 0u;
            int32_t nready = 0;
#pragma unroll
            for (int q = 0; q < kProbe; ++q)
              if (nready == q && q < cnt && (int32_t)(v[q] - target) >= 0) nready = q + 1;
            observed = true;
            if (nready > 0) {
              rc_lo = f;
              rc_hi = f + nready;
              rc_target = target;
              continue;
            }
            const uint64_t t0 = ptx::globaltimer();
            uint32_t iter = 0, backoff = 64;
            while (true) {
              if (reorder && snext < min(NSK, kb / KPS + NS) && arm_b(snext, false) > 0) {
                ++snext;
              } else {
                __nanosleep(backoff);
                if (backoff < 256) backoff <<= 1;
              }
              if ((int32_t)(ptx::ld_relaxed_gpu(wflags + f) - target) >= 0) break;
              if ((++iter & 15u) == 0) {
                if (ptx::ld_relaxed_gpu(args.ctrl + CTRL_ERR) != 0u) break;
                if (ptx::globaltimer() - t0 > args.timeout_ns) {
                  record_error(args, ERRC_FLAG_TIMEOUT, t, (kb << 16) | (f & 0xFFFF));
                  break;
                }
              }
            }
            rc_lo = f;
            rc_hi = f + 1;
            rc_target = target;
            if (trec) trec->polls += iter + 1u;
          }
          if (observed) {
            ptx::fence_acq_rel_gpu();
            ptx::fence_proxy_async_global();
          }
        };
        // The loops visit the unit's stages.  Before a stage's A copies, the waits of each
        // of its k-blocks that can need a semaphore (the B copies go first: cuSync §V).  The
        // GEMM and convolution loops are kept apart: the single loader thread's instruction
        // latency per stage is on the critical path of the mainloop.
        if (gemm) {
          // the next k-block of the unit that consults the tracker: every dep_every-th
          // (unit_dep_kblock), kept as a running index because the loader thread's
          // instructions per stage are on the mainloop's critical path (one more term in
          // the test measured 9-12% slower with one k-block per stage)
          int32_t dep_next = dep_every > 0 ? 0 : 0x7FFFFFFF;
          for (int32_t sj = 0; sj < NSK; ++sj) {
            const int32_t kb = sj * KPS;
            const int32_t nk = KPS == 1 ? 1 : min(KPS, KB - kb);
            const bool dep_st = dep_next < kb + nk;
            auto deps_of_stage = [&]() {
              while (dep_next < kb + nk) {
                wait_deps(dep_next);
                dep_next += dep_every;
              }
            };
            if (dep_st && !reorder) deps_of_stage();
            if (snext == sj) {
              if (arm_b(sj, true) < 0) {
                record_error(args, ERRC_PIPELINE, t, 2);
                *abort_flag = 1;
                ok = false;
                break;
              }
              ++snext;
            }
            if (dep_st && reorder) deps_of_stage();
            if (kb == 0 && trec) trec->t_ready = ptx::globaltimer();
            const int st = a_slot;
            if (++a_slot == NS) a_slot = 0;
            if (KPS > 1 && a3d) {
              if (to_leader) ptx::tma_load_3d_to_leader(smem_a(st), tmA, ptx::mapa(&full[st], 0), 0, a_row, tr.kb0 + kb, pol_a);
              else ptx::tma_load_3d(smem_a(st), tmA, &lbar[st], 0, a_row, tr.kb0 + kb, pol_a);
            } else {
#pragma unroll
              for (int32_t h = 0; h < KPS; ++h) {
                if (h >= nk) break;
                if (to_leader)
                  ptx::tma_load_2d_to_leader(smem_a(st, h), tmA, ptx::mapa(&full[st], 0), kx0 + (kb + h) * kBK, a_row, pol_a);
                else
                  ptx::tma_load_2d(smem_a(st, h), tmA, &lbar[st], kx0 + (kb + h) * kBK, a_row, pol_a);
              }
            }
            *progress = kit + (uint32_t)(kb + nk);
          }
        } else {
          for (int32_t sj = 0; sj < NSK; ++sj) {
            const int32_t kb = sj * KPS;
            const int32_t nk = KPS == 1 ? 1 : min(KPS, KB - kb);
            bool dep_st = false;
#pragma unroll
            for (int h = 0; h < KPS; ++h)
              if (h < nk) dep_st |= (kb + h) < 64 ? ((dep_mask >> (kb + h)) & 1ull) != 0 : dep_every > 0;
            auto deps_of_stage = [&]() {
              for (int h = 0; h < nk; ++h)
                if ((kb + h) < 64 ? ((dep_mask >> (kb + h)) & 1ull) != 0 : dep_every > 0) wait_deps(kb + h);
            };
            if (dep_st && !reorder) deps_of_stage();
            if (snext == sj) {
              if (arm_b(sj, true) < 0) {
                record_error(args, ERRC_PIPELINE, t, 2);
                *abort_flag = 1;
                ok = false;
                break;
              }
              ++snext;
            }
            if (dep_st && reorder) deps_of_stage();
            if (kb == 0 && trec) trec->t_ready = ptx::globaltimer();
            const int st = a_slot;
            if (++a_slot == NS) a_slot = 0;
#pragma unroll
            for (int32_t h = 0; h < KPS; ++h) {
              if (h >= nk) break;
              if (a_buf >= 0)
                ptx::tma_load_5d(smem_a(st, h), tmA, &lbar[st], cv_cb * kBK, cv_s - 1, cv_h0 + cv_r, cv_img, a_buf, pol_a);
              else
                ptx::tma_load_4d(smem_a(st, h), tmA, &lbar[st], cv_cb * kBK, cv_s - 1, cv_h0 + cv_r, cv_img, pol_a);
              if (++cv_cb == SA.g.cblocks) {
                cv_cb = 0;
                if (++cv_s == 3) {
                  cv_s = 0;
                  ++cv_r;
                }
              }
            }
            *progress = kit + (uint32_t)(kb + nk);
          }
        }
        it += (uint32_t)snext;
        kit += (uint32_t)KB;
        *it_issued = (int32_t)it;
        if (!ok && leader) {
          // hand a terminator to the other roles so that they stop
          const int slot2 = tcount % C::kSlots;
          if (xwait<PAIR>(&qempty[slot2], ((tcount / C::kSlots) & 1u) ^ 1u, pto)) {
            qtile[slot2] = -1;
            if (kPair) {
              ptx::st_cluster_u32(ptx::mapa(&qtile[slot2], 1), (uint32_t)-1);
              ptx::mbar_arrive_cluster(ptx::mapa(&qfull[slot2], 1));
            }
            ptx::mbar_arrive(&qfull[slot2]);
          }
          break;
        }
        if (!ok) break;
      }
      // The run's last launch lets the next run's first launch start once every CTA has
      // claimed its last tile (that launch waits for this one before it touches memory).
      if (args.pdl_role & 8) ptx::pdl_launch_dependents();
      if constexpr (C::split_b(CHECK)) {
        __threadfence_block();
        *b_stop = 1u;  // every stage this loader armed has its command posted
      }
      if (leader) {
        // The last CTA (pair) to finish claiming resets this launch's tile counter.
        __threadfence();
        const uint32_t prev = atomicAdd(args.ctrl + CTRL_EXIT + args.queue, 1u);
        if (prev == gridDim.x / PAIR - 1) {
          atomicExch(args.ctrl + CTRL_COUNTER + args.queue, 0u);
          atomicExch(args.ctrl + CTRL_EXIT + args.queue, 0u);
          // Every CTA of the launch that serves the consumer has read the run number by now.
          if (args.last_stage == args.nst - 1) {
            __threadfence();
            atomicAdd(args.ctrl + CTRL_RUNS, 1u);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(128 * PAIR, BN);
    uint32_t it = 0, tcount = 0, acount = 0;
    uint32_t fpar = 0;  // parity of each stage's next `full` phase
    uint32_t rpar = 0;  // parity of each stage's next `ready` phase (checked tiles)
    bool ok = true;
    while (ok) {
      const int slot = tcount % C::kSlots;
      if (!xwait<PAIR>(&qfull[slot], (tcount / C::kSlots) & 1u, pto)) {
        ok = false;
        break;
      }
      const int32_t t = qtile[slot];
      __syncwarp();
      if (lane == 0) ring_release(slot);
      ++tcount;
      if (t < 0) break;
      const TileRef tr = decode_tile(args, t);
      if (tr.s == kFillStage) continue;
      const StageGeo& g = stage_args(args, tr.s).g;
      if (g.a_mode == AMODE_POINTWISE) continue;  // no MMA
      const int acc = acount & 1;
      const uint32_t apar = ((acount >> 1) & 1u) ^ 1u;
      ++acount;
      if (leader) {
        if (!xwait<PAIR>(&tempty[acc], apar, pto)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kAccStride);
      const bool checked = CHECK && stage_consumes(args, tr.s);
      // The peer of a pair issues nothing: its direct copies complete on the leader's
      // `full`, and its checker arrives on the leader's `ready`.
      if (!leader) {
        it += (uint32_t)((tr.nkb + KPS - 1) / KPS);
        continue;
      }
      uint32_t land_clk = 0;  // traced runs: SM cycles spent waiting for stages
      for (int32_t kb = 0; kb < tr.nkb; kb += KPS, ++it) {
        const int st = (int)(it % NS);
        const uint32_t c0 = args.trace ? (uint32_t)clock64() : 0u;
        bool landed;
        if (checked) {
          // every CTA's share of this stage landed and passed the sentinel check
          landed = xwait<PAIR>(&ready[st], (rpar >> st) & 1u, pto);
          rpar ^= 1u << st;
        } else {
          landed = ptx::mbar_wait_bounded(&full[st], (fpar >> st) & 1u, pto);
          fpar ^= 1u << st;
        }
        if (!landed) {
          ok = false;
          break;
        }
        if (args.trace) land_clk += (uint32_t)clock64() - c0;
        ptx::tc_fence_after();
        if (lane == 0 && kb == 0 && args.trace) args.trace[chain_tile(args, tr.q)].t_mma0 = ptx::globaltimer();
        if (lane == 0) {
          // the stage's k-blocks (the unit's last stage may hold fewer than KPS); the k-th
          // 16-wide slice of a 128-byte swizzled row starts 32 bytes further (+2 in the
          // descriptors' address field)
          const int nk = min(KPS, tr.nkb - kb);
#pragma unroll
          for (int h = 0; h < KPS; ++h) {
            if (h < nk) {
              const uint64_t da = ptx::smem_desc_k128(ptx::smem_u32(smem_a(st, h)));
              const uint64_t db = ptx::smem_desc_k128(ptx::smem_u32(smem_b(st, h)));
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {
                const uint32_t accum = (kb + h + k) != 0 ? 1u : 0u;
                if (kPair) ptx::umma_bf16_pair(d_tmem, da + 2u * k, db + 2u * k, idesc, accum);
                else ptx::umma_bf16(d_tmem, da + 2u * k, db + 2u * k, idesc, accum);
              }
            }
          }
          if (kPair) ptx::umma_commit_pair_multicast(&empty[st], 0x3);
          else ptx::umma_commit(&empty[st]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        if (kPair) ptx::umma_commit_pair_multicast(&tfull[acc], 0x3);
        else ptx::umma_commit(&tfull[acc]);
        if (args.trace) {
          TraceRec* r = args.trace + chain_tile(args, tr.q);
          r->t_mma1 = ptx::globaltimer();
          r->land_clk = land_clk;
        }
      }
      __syncwarp();
    }
    if (!ok) {
      record_error(args, ERRC_PIPELINE, 0xFFFFFF, 3);
      *abort_flag = 1;
    }
    if (leader && lane == 0) {
      // every MMA this thread issued has completed once mma_done flips
      if (kPair) ptx::umma_commit_pair_multicast(mma_done, 0x1);
      else ptx::umma_commit(mma_done);
      ptx::mbar_wait_bounded(mma_done, 0, pto);
    }
    __syncwarp();
    // Abnormal exit only: wait (bounded) for copies on `full` that were issued but not
    // consumed (the checker drains `cfull`).
    if (lane == 0 && !ok && leader) {
      const uint32_t issued = (uint32_t)*it_issued;
      for (uint32_t j = it; j < issued && j < it + NS; ++j) {
        const int st = (int)(j % NS);
        if (stage_kind[st] != 0) continue;
        ptx::mbar_wait_bounded(&full[st], (fpar >> st) & 1u, pto);
        fpar ^= 1u << st;
      }
    }
    __syncwarp();
  } else if (CHECK && warp >= 7 && warp < 7 + C::check_warps()) {
    // ------------------------------------------------------------ sentinel checkers
    // Under the sentinel policy every consumer k-block's A tile is validated here, off the
    // MMA issuer's path, and handed to it through `ready` (the leader's, in a pair).  With
    // one k-block per stage (single CTAs) warp 7 owns the even stages, warp 8 the odd ones
    // (the stage count is even, so a stage always belongs to the same warp and each warp's
    // barrier phases are its own); with two k-blocks per stage (pairs) both warps take
    // every stage (below).
    const int ck = warp - 7;
    const uint64_t pol_a = ptx::l2_policy_evict_last();
    // Whether k-block h of the A tile in stage sx still holds the sentinel anywhere (all
    // lanes).  Every bf16 element of the landed tile is inspected.  The PTX memory model
    // treats a vector store as independent scalar stores in no fixed order, so a copy that
    // overlaps the producer's 128-bit store of a chunk may bring some of its words written
    // and others not; a sampled word would then pass a chunk that is partly sentinel.
    // Scanning every word makes the check independent of how the producer's stores are
    // split: any element still holding 0x8000 sends the tile back.  Lane l reads 16-byte
    // chunk c = 32 i + l, so a warp's load covers 512 contiguous bytes without bank
    // conflicts.  Shared-memory loads are slow to return while TMA writes and the MMAs
    // read the same memory, so all of a 16 KB tile's loads (32 per lane) are issued before
    // the first one is tested.
    auto stage_has_sentinel = [&](int sx, int h, uint32_t nbytes) -> bool {
      uint32_t sbits = 0;
      const uint8_t* base = smem_a(sx, h);
      const uint32_t nchunks = nbytes / 16u;
      for (uint32_t c0 = (uint32_t)lane; c0 < nchunks; c0 += 32u * 32u) {
        uint4 v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t c = c0 + (uint32_t)j * 32u;
          v[j] = c < nchunks ? ptx::ld_shared_v4(base + c * 16u) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
          sbits |= sentinel_bits_bf16x2(v[j].x) | sentinel_bits_bf16x2(v[j].y) | sentinel_bits_bf16x2(v[j].z) |
                   sentinel_bits_bf16x2(v[j].w);
      }
      return __any_sync(FULL, (sbits & 0x80008000u) != 0u);
    };
    // The same for half (part 0 or 1) of a GEMM A k-block (128 rows x 64 = 16 KB, so 8 KB:
    // 16 loads per lane).
    auto half_has_sentinel = [&](int sx, int h, int part) -> bool {
      const uint8_t* base = smem_a(sx, h) + part * (C::kABytes / 2);
      uint4 v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = ptx::ld_shared_v4(base + ((uint32_t)lane + (uint32_t)j * 32u) * 16u);
      uint32_t sbits = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        sbits |= sentinel_bits_bf16x2(v[j].x) | sentinel_bits_bf16x2(v[j].y) | sentinel_bits_bf16x2(v[j].z) |
                 sentinel_bits_bf16x2(v[j].w);
      return __any_sync(FULL, (sbits & 0x80008000u) != 0u);
    };
    if constexpr (CHECK && KPS == 1) {
      static_assert(S % 2 == 0, "the checkers split the stages by parity");
      uint32_t it = 0, tcount = 0;
      uint32_t cpar = 0;  // parity of each stage's next `cfull` phase
      // Stages of later k-blocks of the current tile that were found landed and clean
      // while an earlier one was reloaded (their cfull phase is consumed).
      uint32_t clean_ahead = 0;
      bool ok = true;
      while (ok) {
        const int slot = tcount % C::kSlots;
        if (!xwait<PAIR>(&qfull[slot], (tcount / C::kSlots) & 1u, pto)) {
          ok = false;
          break;
        }
        const int32_t t = qtile[slot];
        __syncwarp();
        if (lane == 0) ring_release(slot);
        ++tcount;
        if (t < 0) break;
        const TileRef tr = decode_tile(args, t);
        if (tr.s == kFillStage) continue;
        const StageGeo& g = stage_args(args, tr.s).g;
        if (g.a_mode == AMODE_POINTWISE) continue;
        if (!stage_consumes(args, tr.s)) {
          it += (uint32_t)tr.nkb;  // loaded on `full`, consumed by the MMA issuer alone
          continue;
        }
        const uint32_t abytes = a_tile_bytes(g);
        const int32_t a_buf = args.stack ? stack_buf(args, tr.s - 1, *run_no) : -1;
        uint32_t check_clk = 0, reloads = 0;
        for (int32_t kb = 0; kb < tr.nkb; ++kb, ++it) {
          const int st = (int)(it % S);
          if ((st & 1) != ck) continue;  // the other checker's stage
          if ((clean_ahead >> st) & 1u) {
            clean_ahead &= ~(1u << st);
          } else {
            if (!ptx::mbar_wait_bounded(&cfull[st], (cpar >> st) & 1u, pto)) {
              ok = false;
              break;
            }
            cpar ^= 1u << st;
            const uint32_t c1 = args.trace ? (uint32_t)clock64() : 0u;
            // Software validity check of this CTA's landed A tile: while any element still
            // holds the sentinel, the A load is issued again.
            uint64_t t0 = 0;
            bool reloaded = false;
            while (true) {
              if (!stage_has_sentinel(st, 0, abytes)) break;
              if (ptx::ld_relaxed_gpu(args.ctrl + CTRL_ERR) != 0u) break;
              const uint64_t now = ptx::globaltimer();
              if (t0 == 0) t0 = now;
              if (now - t0 > args.timeout_ns) {
                if (lane == 0) record_error(args, ERRC_SENTINEL_TIMEOUT, t, kb);
                break;
              }
              if (lane == 0) {
                __nanosleep(128);
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive_expect_tx(&cfull[st], abytes);
                issue_a<PAIR>(args, tr, tr.kb0 + kb, rank, smem_a(st), &cfull[st], pol_a, a_buf);
              }
              ++reloads;
              __syncwarp();
              if (!ptx::mbar_wait_bounded(&cfull[st], (cpar >> st) & 1u, pto)) {
                ok = false;
                break;
              }
              cpar ^= 1u << st;
              reloaded = true;
            }
            if (!ok) break;
            if (reloaded) {
              // This k-block's data has just become valid.  The A tiles of the following
              // k-blocks of this tile that landed meanwhile were most likely copied before
              // their data was written too: check them now and issue the stale ones again
              // at once, so that their reloads overlap instead of following one another.
              for (int j = 2; j < S && kb + j < tr.nkb; j += 2) {
                const int sj = (int)((it + (uint32_t)j) % S);
                if ((clean_ahead >> sj) & 1u) continue;
                bool landed = false;
                if (lane == 0) landed = ptx::mbar_test_wait(&cfull[sj], (cpar >> sj) & 1u);
                if (!__shfl_sync(FULL, landed ? 1 : 0, 0)) continue;
                cpar ^= 1u << sj;
                if (stage_has_sentinel(sj, 0, abytes)) {
                  if (lane == 0) {
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive_expect_tx(&cfull[sj], abytes);
                    issue_a<PAIR>(args, tr, tr.kb0 + kb + j, rank, smem_a(sj), &cfull[sj], pol_a, a_buf);
                  }
                  ++reloads;
                } else {
                  clean_ahead |= 1u << sj;
                }
              }
              __syncwarp();
            }
            if (args.trace) check_clk += (uint32_t)clock64() - c1;
          }
          // Hand the checked stage to the MMA issuer.  In a pair the leader's checker
          // arrives and expects 4 bytes, which the peer's checker supplies with an
          // asynchronous store: a remote mbarrier.arrive.release would stall it for a
          // round trip between the SMs at every k-block.
          __syncwarp();
          if (lane == 0) {
            if (!kPair) ptx::mbar_arrive(&ready[st]);
            else if (leader) ptx::mbar_arrive_expect_tx(&ready[st], 4u);
            else ptx::st_async_u32(ptx::mapa(&ready_sink[st], 0), 1u, ptx::mapa(&ready[st], 0));
          }
        }
        if (!ok) break;
        if (args.trace && leader && lane == 0) {
          TraceRec* r = args.trace + chain_tile(args, tr.q);
          atomicAdd(&r->check_clk, check_clk);
          atomicAdd(&r->reloads, reloads);
        }
      }
      if (!ok) {
        record_error(args, ERRC_PIPELINE, 0xFFFFFF, 10);
        *abort_flag = 1;
        // wait (bounded) for copies on `cfull` that were issued but not consumed
        if (lane == 0) {
          const uint32_t issued = (uint32_t)*it_issued;
          for (uint32_t j = it; j < issued && j < it + S; ++j) {
            const int st = (int)(j % S);
            if ((st & 1) != ck || stage_kind[st] != 1 || ((clean_ahead >> st) & 1u)) continue;
            ptx::mbar_wait_bounded(&cfull[st], (cpar >> st) & 1u, pto);
            cpar ^= 1u << st;
          }
        }
      }
    } else if constexpr (CHECK) {
      // Two k-blocks per stage: checker warp 7 + c scans half c & 1 of k-block c >> 1 of
      // every checked stage.  The checkers combine their findings each round through
      // scan_flag and the scan_done barrier (bounded waits, one arrival per warp); warp 7
      // alone decides to reload the stage's A box or to give up after the timeout, and
      // hands the clean stage to the MMA issuer.  Every checker follows every stage and
      // round, so their barrier phases agree.
      constexpr int kCW = C::check_warps();
      static_assert(kCW == 2 * KPS, "two checkers per k-block of a stage");
      const int h_ck = ck >> 1;                // this warp's k-block of the stage
      uint32_t it = 0, tcount = 0, cpar = 0, xround = 0;
      bool ok = true;
      while (ok) {
        const int slot = tcount % C::kSlots;
        if (!xwait<PAIR>(&qfull[slot], (tcount / C::kSlots) & 1u, pto)) {
          ok = false;
          break;
        }
        const int32_t t = qtile[slot];
        __syncwarp();
        if (lane == 0) ring_release(slot);
        ++tcount;
        if (t < 0) break;
        const TileRef tr = decode_tile(args, t);
        if (tr.s == kFillStage) continue;
        const StageArgs& SA = stage_args(args, tr.s);
        const StageGeo& g = SA.g;
        if (g.a_mode == AMODE_POINTWISE) continue;
        const int32_t NSK = (tr.nkb + KPS - 1) / KPS;
        if (!stage_consumes(args, tr.s)) {
          it += (uint32_t)NSK;  // loaded on `full`, consumed by the MMA issuer alone
          continue;
        }
        const uint32_t abytes = a_tile_bytes(g);
        const int32_t a_row = tr.m * (128 * PAIR) + (int32_t)rank * 128;
        uint32_t check_clk = 0, reloads = 0;
        for (int32_t sj = 0; sj < NSK; ++sj, ++it) {
          const int st = (int)(it % NS);
          const int32_t kb = sj * KPS;
          const int32_t nk = min(KPS, tr.nkb - kb);
          if (!ptx::mbar_wait_bounded(&cfull[st], (cpar >> st) & 1u, pto)) {
            ok = false;
            break;
          }
          cpar ^= 1u << st;
          const uint32_t c1 = args.trace ? (uint32_t)clock64() : 0u;
          uint64_t t0 = 0;
          while (true) {
            // this warp's half k-block (only those of the unit: a box may reach into the next)
            const bool dirty = h_ck < nk && half_has_sentinel(st, h_ck, ck & 1);
            bool late = false;
            if (ck == 0 && t0 != 0)
              late = ptx::globaltimer() - t0 > args.timeout_ns || ptx::ld_relaxed_gpu(args.ctrl + CTRL_ERR) != 0u;
            if (lane == 0) {
              scan_flag[(xround & 1u) * kCW + (uint32_t)ck] = (dirty ? 1u : 0u) | (late ? 2u : 0u);
              ptx::mbar_arrive(scan_done);
            }
            if (!ptx::mbar_wait_bounded(scan_done, xround & 1u, pto)) {
              ok = false;
              break;
            }
            const uint32_t f0 = scan_flag[(xround & 1u) * kCW];
            uint32_t fa = 0;
#pragma unroll
            for (int c = 0; c < kCW; ++c) fa |= scan_flag[(xround & 1u) * kCW + (uint32_t)c];
            ++xround;
            if ((fa & 1u) == 0u) break;  // the stage is clean
            if (f0 & 2u) {
              if (ck == 0 && lane == 0) record_error(args, ERRC_SENTINEL_TIMEOUT, t, kb);
              break;
            }
            if (t0 == 0) t0 = ptx::globaltimer();
            // Load the stage's A box again (warp 7); both warps wait for it to land.
            if (ck == 0 && lane == 0) {
              __nanosleep(128);
              ptx::fence_proxy_async_smem();
              if (SA.a3d) {
                ptx::mbar_arrive_expect_tx(&cfull[st], (uint32_t)KPS * abytes);
                ptx::tma_load_3d(smem_a(st), &SA.tmA, &cfull[st], 0, a_row, tr.kb0 + kb, pol_a);
              } else {
                ptx::mbar_arrive_expect_tx(&cfull[st], (uint32_t)nk * abytes);
                for (int h = 0; h < nk; ++h)
                  ptx::tma_load_2d(smem_a(st, h), &SA.tmA, &cfull[st], (tr.kb0 + kb + h) * kBK, a_row, pol_a);
              }
            }
            ++reloads;
            __syncwarp();
            if (!ptx::mbar_wait_bounded(&cfull[st], (cpar >> st) & 1u, pto)) {
              ok = false;
              break;
            }
            cpar ^= 1u << st;
          }
          if (!ok) break;
          if (args.trace) check_clk += (uint32_t)clock64() - c1;
          // Hand the checked stage to the MMA issuer (warp 7; see the one-k-block path).
          __syncwarp();
          if (ck == 0 && lane == 0) {
            if (leader) ptx::mbar_arrive_expect_tx(&ready[st], 4u);
            else ptx::st_async_u32(ptx::mapa(&ready_sink[st], 0), 1u, ptx::mapa(&ready[st], 0));
          }
        }
        if (!ok) break;
        if (args.trace && leader && lane == 0) {
          TraceRec* r = args.trace + chain_tile(args, tr.q);
          atomicAdd(&r->check_clk, check_clk);
          if (ck == 0) atomicAdd(&r->reloads, reloads);
        }
      }
      if (!ok) {
        record_error(args, ERRC_PIPELINE, 0xFFFFFF, 10);
        *abort_flag = 1;
        // wait (bounded) for copies on `cfull` that were issued but not consumed
        if (ck == 0 && lane == 0) {
          const uint32_t issued = (uint32_t)*it_issued;
          for (uint32_t j = it; j < issued && j < it + NS; ++j) {
            const int st = (int)(j % NS);
            if (stage_kind[st] != 1) continue;
            ptx::mbar_wait_bounded(&cfull[st], (cpar >> st) & 1u, pto);
            cpar ^= 1u << st;
          }
        }
      }
    }
    __syncwarp();
  } else if (C::split_b(CHECK) && warp == 11) {
    // ------------------------------------------------------------ B-copy warp
    // Issues the weight (B) copies of the stages the loader armed, in order: the loader
    // keeps every barrier operation (the slot waits, the bytes each stage expects) and the
    // activation (A) copies, and hands the weight copies of each stage over, so that the
    // two kinds of copies are issued by two threads.  It never runs ahead of the loader.
    if (lane == 0) {
      const uint64_t pol_b = ptx::l2_policy_evict_normal();
      uint32_t done = 0;
      int slot = 0;
      uint64_t idle0 = 0;
      while (true) {
        const uint32_t posted = *b_posted;
        if (posted == done) {
          if (*b_stop && *b_posted == done) break;
          const uint64_t now = ptx::globaltimer();
          if (idle0 == 0) idle0 = now;
          if (now - idle0 > 2 * pto) {
            record_error(args, ERRC_PIPELINE, 0xFFFFFF, 13);
            *abort_flag = 1;
            break;
          }
          __nanosleep(32);
          continue;
        }
        idle0 = 0;
        __threadfence_block();
        while (done != posted) {
          const BCmd& c = bcmd[slot];
          uint64_t* bar = &full[slot];
          if (c.mode & 1u) {
            if (c.mode & 2u) ptx::tma_load_3d_to_leader(smem_b(slot), c.tm, ptx::mapa(bar, 0), 0, c.brow0, c.kglob, pol_b);
            else ptx::tma_load_3d(smem_b(slot), c.tm, bar, 0, c.brow0, c.kglob, pol_b);
          } else {
            for (int32_t h = 0; h < c.nk; ++h) {
              uint8_t* dst = smem_b(slot, h);
              const int32_t x = (c.kglob + h) * kBK;
              if (c.zs >= 0) {
                ptx::tma_load_3d(dst, c.tm, bar, x, c.brow0, c.zs, pol_b);
              } else if (c.mode & 2u) {
                ptx::tma_load_2d_to_leader(dst, c.tm, ptx::mapa(bar, 0), x, c.brow0, pol_b);
              } else {
                ptx::tma_load_2d(dst, c.tm, bar, x, c.brow0, pol_b);
                if (c.brow1 >= 0) ptx::tma_load_2d(dst + (BN / 2) * 128, c.tm, bar, x, c.brow1, pol_b);
              }
            }
          }
          if (++slot == NS) slot = 0;
          ++done;
        }
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ L2 prefetch warp
    // Follows the tile ring and, paced by the loader's progress counter, prefetches this
    // CTA's weight box of the k-blocks up to l2_prefetch ahead of the loader into L2, one
    // copy-engine prefetch per box.  The copies that follow then find the weights in L2
    // instead of waiting for HBM, which the shared-memory ring alone cannot hide when the
    // chain streams its weights (a few CTAs per weight tile, small M).
    const int32_t pd = args.l2_prefetch;
    uint32_t tcount = 0, it0 = 0;
    while (true) {
      const int slot = tcount % C::kSlots;
      if (!xwait<PAIR>(&qfull[slot], (tcount / C::kSlots) & 1u, pto)) break;
      const int32_t t = qtile[slot];
      __syncwarp();
      if (lane == 0) ring_release(slot);
      ++tcount;
      if (t < 0) break;
      const TileRef tr = decode_tile(args, t);
      if (tr.s == kFillStage) continue;
      const StageArgs& SA = stage_args(args, tr.s);
      const StageGeo& g = SA.g;
      const int32_t KB = tr.nkb;
      if (pd > 0 && g.a_mode == AMODE_GEMM) {
        const int32_t b0 = b_row<BN, PAIR>(SA, tr, rank, 0);
        const int32_t b1 = (PAIR == 1 && g.epi == EPI_SWIGLU) ? b_row<BN, PAIR>(SA, tr, rank, 1) : -1;
        bool live = true;
        for (int32_t kb = 0; kb < KB && live; ++kb) {
          const uint32_t j = it0 + (uint32_t)kb;
          if (lane == 0) {
            const uint64_t t0 = ptx::globaltimer();
            while ((int32_t)(j - *progress) >= pd) {
              __nanosleep(64);
              if (*abort_flag || ptx::globaltimer() - t0 > pto) {
                live = false;
                break;
              }
            }
          }
          live = __shfl_sync(FULL, live ? 1 : 0, 0) != 0;
          if (!live) break;
          // the weight tile's box through the copy engine: one instruction per box
          if (lane == 0 && !(SA.b3d && (kb & 1))) {
            if (SA.b3d) ptx::tma_prefetch_3d(&SA.tmB, 0, b0, tr.kb0 + kb);
            else if (!args.stack) {
              ptx::tma_prefetch_2d(&SA.tmB, (tr.kb0 + kb) * kBK, b0);
              if (b1 >= 0) ptx::tma_prefetch_2d(&SA.tmB, (tr.kb0 + kb) * kBK, b1);
            }
          }
        }
      }
      it0 += (uint32_t)KB;
    }
    __syncwarp();
  } else if ((warp >= 2 && warp <= 5) || (kEpiGroups == 2 && warp >= kEpi2 && warp < kEpi2 + 4)) {
    // ------------------------------------------------------------ epilogue (warps 2..5 and
    // 7..10; with the sentinel checkers, 2..5 and the four warps after the checkers)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int egrp = warp >= kEpi2 ? 1 : 0;        // this warp's group: it stores boxes egrp, egrp + kEpiGroups, ...
    const int ew = egrp * 4 + (warp - (egrp ? kEpi2 : 2));  // epilogue warp ordinal
    const int et = ew * 32 + lane;                 // epilogue thread ordinal
    uint32_t tcount = 0, acount = 0, pwcount = 0;  // pwcount: pointwise tiles done
    bool fill_seen = false;                        // pdl_role bit 4: the intermediate's fill has ended
    // Attention chain: a pointwise tile (see pointwise_tile) -- out of line, so that its
    // registers do not weigh on the GEMM epilogue.

    while (true) {
      const int slot = tcount % C::kSlots;
      if (!xwait<PAIR>(&qfull[slot], (tcount / C::kSlots) & 1u, pto)) break;
      const int32_t t = qtile[slot];
      __syncwarp();
      if (lane == 0) ring_release(slot);
      ++tcount;
      if (t < 0) break;
      const TileRef tr = decode_tile(args, t);
      if (tr.s == kFillStage) {
        // [CUDA-FGS] §4.6.4.5 "Buffer Reuse": the sentinel goes over the set of buffers
        // the next run will use while this run's tail is still computing; that set was
        // last read by the run before this one, which has finished.  Whole 16-byte chunks.
        const uint32_t next = (*run_no + 1u) & 1u;
        uint4* const base = reinterpret_cast<uint4*>(args.st[0].out) + (int64_t)next * args.set_chunks;
        const int64_t c0 = (int64_t)tr.m * args.fill_unit_chunks;
        const int64_t c1 = min(c0 + args.fill_unit_chunks, args.set_chunks);
        const uint4 v = make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
        // streaming stores: L2 keeps the lines of the stages still running, not these
        for (int64_t c = c0 + et; c < c1; c += 32 * kEpiWarps) __stcs(base + c, v);
        continue;
      }
      const StageArgs& SA = stage_args(args, tr.s);
      const StageGeo& g = SA.g;
      if (g.a_mode == AMODE_POINTWISE) {
        // one token row per thread of the first group (the second has nothing to do)
        if (egrp == 0)
          pointwise_tile(args, tr, t, (int64_t)tr.m * (128 * PAIR) + (int64_t)rank * 128 + row, pw_done,
                         pwcount & 1u, *run_no, leader, pto, abort_flag);
        ++pwcount;
        continue;
      }
      if ((args.pdl_role & 16) && !fill_seen) {
        ptx::pdl_wait();  // before this CTA's first store of the intermediate (pdl_role bit 4)
        fill_seen = true;
      }
      const int acc = acount & 1;
      const uint32_t apar = (acount >> 1) & 1u;
      ++acount;
      if (!ptx::mbar_wait_bounded(&tfull[acc], apar, pto)) {
        record_error(args, ERRC_PIPELINE, t, 4);
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const bool tracer = args.trace && leader && threadIdx.x == 64;  // records this tile's epilogue times
      if (tracer) args.trace[chain_tile(args, tr.q)].t_acc = ptx::globaltimer();
      uint64_t t_xchg = 0;

      int64_t grow;
      bool valid;
      if (g.a_mode == AMODE_GEMM) {
        grow = (int64_t)tr.m * (128 * PAIR) + (int64_t)rank * 128 + row;
        valid = grow < g.M;
      } else {
        const int32_t n = tr.m / g.tpi, hb = tr.m % g.tpi;
        const int32_t hl = row / g.img_w, w = row % g.img_w;
        const int32_t h = hb * g.th + hl;
        valid = (hl < g.th) && (h < g.img_h);
        grow = ((int64_t)n * g.img_h + h) * g.img_w + w;
      }
      // a stack's stage writes its intermediate buffer (the last stage: the output) and
      // applies no activation after the last convolution
      const bool stack_mid = args.stack && tr.s < args.nst - 1;
      const int32_t epi = (args.stack && !stack_mid) ? EPI_NONE : g.epi;
      __nv_bfloat16* const obase = stack_mid ? reinterpret_cast<__nv_bfloat16*>(args.st[0].out) +
                                                   (int64_t)stack_buf(args, tr.s, *run_no) * args.buf_elems
                                             : reinterpret_cast<__nv_bfloat16*>(SA.out);
      __nv_bfloat16* orow = obase + (valid ? grow * (int64_t)g.N : 0);
      const int32_t col0 = tr.c * g.n_out;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccStride);
      const int nchunks = g.n_out / 32;
      // GEMM outputs leave through TMA stores of 32-row x 64-column boxes staged in this
      // warp's shared-memory buffers; convolution outputs (a tile's pixels are not a box
      // of the output tensor) through 16-byte stores from registers.  With two warps per
      // lane quarter, each takes every other 64-column box (two 32-column chunks).  Under the
      // sentinel policy the consumer's check inspects every element it loads, so it does
      // not matter how the stores of the tile it checks are split.
      const bool tma_out = g.a_mode == AMODE_GEMM;
      uint8_t* ebuf = epi_stage + ew * kEpiBufs * C::kEpiBufBytes;
      const int32_t row_w0 = tr.m * (128 * PAIR) + (int32_t)rank * 128 + q * 32;
      // K split: unit k of a tile adds the running sum of units 0..k-1 to its fp32 partial
      // sums; the units other than the last store the result in their workspace slot, and
      // the last applies the epilogue to the total.  The slots mark their own readiness: a
      // word that holds no sum holds kSplitEmpty, a NaN that a sum never takes (the storing
      // unit writes any such value as the canonical NaN), so a unit re-reads a 16-byte
      // word of its predecessor's slot until it holds a sum, with no counter or fence
      // between the units, and writes kSplitEmpty back once it has read it ([CUDA-FGS]
      // §4.6.4 sentinel protocol, here for the partial sums rather than the intermediate).
      // A unit waits only on the unit before it in the queue, which is already running.
      const bool split = g.ksplit > 1;
      const bool last_unit = !split || tr.ks == g.ksplit - 1;
      float* const split_ws = tr.s == 0 ? args.split_ws : args.split_ws1;
      // Workspace layout per slot of a 128-row block: groups of 4 columns, then rows,
      // then the 4 columns -- a warp's 32 rows of one column group are 512 contiguous
      // bytes, so the 16-byte accesses below are fully coalesced.
      constexpr int kSlotF4 = 128 * BN / 4;  // 16-byte words per slot
      uint4* ws_row = nullptr;
      if (split) {
        const int64_t tile_id = ((int64_t)tr.m * g.n_tiles + tr.c) * PAIR + (int64_t)rank;
        ws_row = reinterpret_cast<uint4*>(split_ws) + tile_id * (g.ksplit - 1) * kSlotF4 + row;
      }
      const uint64_t split_t0 = (split && tr.ks > 0) ? ptx::globaltimer() : 0;
      // fault injection: the first unit of producer tile (0, 0) withholds its sums
      const bool split_skip = (args.flags_bits & kDebugSkipSplit) && tr.s == 0 && tr.ks == 0 && tr.m == 0 && tr.c == 0;
      bool split_late = false;  // a slot word stayed empty past the timeout (error recorded)
      // The 8 words of one slot at p (stride 128 words): split_issue loads them into v;
      // split_settle re-reads those that still hold kSplitEmpty and then marks the 8
      // words empty again for the next run.
      auto split_issue = [&](uint4 (&v)[8], const uint4* p) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = ptx::ld_relaxed_gpu_b128(p + i * 128);
      };
      auto split_settle = [&](uint4 (&v)[8], uint4* p) {
        auto any_empty = [&]() {
          bool e = false;
#pragma unroll
          for (int i = 0; i < 8; ++i) e |= split_empty(v[i]);
          return e;
        };
        uint32_t polls = 0;
        while (!split_late && any_empty()) {
          __nanosleep(128);
          if ((++polls & 15u) == 0 && ptx::ld_relaxed_gpu(args.ctrl + CTRL_ERR) != 0u) {
            split_late = true;  // another wait already failed: stop polling
            break;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (split_empty(v[i])) v[i] = ptx::ld_relaxed_gpu_b128(p + i * 128);
          if (ptx::globaltimer() - split_t0 > args.timeout_ns && any_empty()) {
            record_error(args, ERRC_FLAG_TIMEOUT, t, 0xFFFF);
            split_late = true;
          }
        }
        // the last unit marks the words as it reads them; a unit between the first and the
        // last marks them after all of its own slot's stores (below), which the next unit
        // is waiting for
        if (last_unit) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            ptx::st_relaxed_gpu_b128(p + i * 128, kSplitEmpty, kSplitEmpty, kSplitEmpty, kSplitEmpty);
        }
      };
      // 32 accumulator columns from `col` on.  The units form a chain: unit k > 0 adds
      // the running sum of units 0..k-1 from slot k-1 to its own sums (the same
      // association, ((p0 + p1) + p2) + ..., for every run and policy); a unit that is not
      // the last stores the result in its slot k.  Each unit reads one slot, chunk by
      // chunk as its predecessor writes it, so the units' epilogues overlap.
      auto split_add = [&](uint32_t (&x)[32], int col) {
        uint4* w = ws_row + (col / 4) * 128;  // column group col/4 + i is at w + i * 128
        if (tr.ks > 0) {
          uint4* prev = w + (tr.ks - 1) * kSlotF4;
          uint4 a[8];
          split_issue(a, prev);
          split_settle(a, prev);
          if (tracer) t_xchg = ptx::globaltimer();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            x[4 * i + 0] = __float_as_uint(__uint_as_float(a[i].x) + __uint_as_float(x[4 * i + 0]));
            x[4 * i + 1] = __float_as_uint(__uint_as_float(a[i].y) + __uint_as_float(x[4 * i + 1]));
            x[4 * i + 2] = __float_as_uint(__uint_as_float(a[i].z) + __uint_as_float(x[4 * i + 2]));
            x[4 * i + 3] = __float_as_uint(__uint_as_float(a[i].w) + __uint_as_float(x[4 * i + 3]));
          }
        }
        if (!last_unit && !split_skip) {
          uint4* ws = w + tr.ks * kSlotF4;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            ptx::st_relaxed_gpu_b128(ws + i * 128, split_canon(x[4 * i]), split_canon(x[4 * i + 1]),
                                     split_canon(x[4 * i + 2]), split_canon(x[4 * i + 3]));
        }
      };
      for (int j = 0; j < nchunks; ++j) {
        if (kEpiGroups > 1 && ((j >> 1) % kEpiGroups) != egrp) continue;  // the other group's box
        uint32_t v[32];
        float f[32];
        if (g.epi == EPI_SWIGLU) {
          uint32_t u[32];
          ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(j * 32), v);
          ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(BN / 2 + j * 32), u);
          ptx::tmem_ld_wait();
          if (split) {
            split_add(v, j * 32);
            split_add(u, BN / 2 + j * 32);
            if (!last_unit) continue;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = silu_f(__uint_as_float(v[i])) * __uint_as_float(u[i]);
        } else {
          ptx::tmem_ld_32x32b_x32(tbase + (uint32_t)(j * 32), v);
          ptx::tmem_ld_wait();
          if (split) {
            split_add(v, j * 32);
            if (!last_unit) continue;
          }
          if (epi == EPI_GELU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = gelu_f(__uint_as_float(v[i]));
          } else if (epi == EPI_RELU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = fmaxf(__uint_as_float(v[i]), 0.0f);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
          }
        }
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
        if (tma_out) {
          // Two 32-column chunks fill one 64-column box; each lane writes its row (128
          // bytes) with the 16-byte units permuted as the 128-byte swizzle expects, which
          // also spreads a warp's stores over all banks.
          const int box = j >> 1;
          const int lbox = box / kEpiGroups;  // this warp's box ordinal
          uint8_t* buf = ebuf + (lbox % kEpiBufs) * C::kEpiBufBytes;
          if ((j & 1) == 0 && lbox >= kEpiBufs) {
            if (lane == 0) ptx::bulk_wait_group_read<kEpiBufs - 1>();  // the store that last read `buf`
            __syncwarp();
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int u = (j & 1) * 4 + ch;
            ptx::st_shared_v4(buf + lane * 128 + ((u ^ (lane & 7)) << 4), p[4 * ch], p[4 * ch + 1], p[4 * ch + 2],
                              p[4 * ch + 3]);
          }
          if ((j & 1) == 1 || j == nchunks - 1) {
            ptx::fence_proxy_async_smem();  // this thread's writes before the async-proxy read
            __syncwarp();
            // boxes that start past the tensor's last row or column hold nothing to store
            if (lane == 0 && row_w0 < g.M && col0 + box * 64 < g.N) {
              ptx::tma_store_2d(&SA.tmO, buf, col0 + box * 64, row_w0);
              ptx::bulk_commit_group();
            }
          }
        } else if (valid) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int32_t col = col0 + j * 32 + ch * 8;
            if (col < g.N) ptx::st_relaxed_gpu_b128(orow + col, p[4 * ch], p[4 * ch + 1], p[4 * ch + 2], p[4 * ch + 3]);
          }
        }
      }
      if (split && !last_unit && tr.ks > 0) {
        // the predecessor's slot, read above, marked empty for the next run
        const int ncol = g.epi == EPI_SWIGLU ? 2 : 1;  // SwiGLU: gate and up columns
        for (int j = 0; j < nchunks; ++j) {
          if (kEpiGroups > 1 && ((j >> 1) % kEpiGroups) != egrp) continue;  // the other group's box
          for (int h = 0; h < ncol; ++h) {
            uint4* w = ws_row + ((h * (BN / 2) + j * 32) / 4) * 128 + (tr.ks - 1) * kSlotF4;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              ptx::st_relaxed_gpu_b128(w + i * 128, kSplitEmpty, kSplitEmpty, kSplitEmpty, kSplitEmpty);
          }
        }
      }
      if (tracer && t_xchg) args.trace[chain_tile(args, tr.q)].t_xchg = t_xchg;
      if (tma_out) {
        // The tile's stores have completed (not only read their source) before this warp
        // reports them done: the semaphore post below may follow right after.
        if (lane == 0) {
          ptx::bulk_wait_group_all();
          ptx::fence_proxy_async_global();
        }
        __syncwarp();
      }
      // Arrive on epi_done before releasing the accumulator: a thread can reach this
      // accumulator's next tile only after every thread released it, so each phase of
      // epi_done[acc] counts the arrivals of exactly one tile.
      ptx::mbar_arrive(&epi_done[acc]);
      ptx::tc_fence_before();
      if (kPair) {
        __syncwarp();
        if (lane == 0) {
          if (leader) ptx::mbar_arrive(&tempty[acc]);
          else ptx::mbar_arrive_cluster(ptx::mapa(&tempty[acc], 0));
        }
      } else {
        ptx::mbar_arrive(&tempty[acc]);
      }
      if (args.trace && leader && threadIdx.x == 64) {
        if (ptx::mbar_wait_bounded(&epi_done[acc], apar, pto))
          args.trace[chain_tile(args, tr.q)].t_epi = ptx::globaltimer();
      }
      if (!last_unit) {
        // K split: this unit's sums are in its workspace slot, which marks itself ready
      } else if (args.band_flags && tr.s == args.nst - 1 && threadIdx.x == 64) {
        // Row bands of the output: once all of this CTA's stores of the tile are complete
        // (the epi_done barrier; TMA stores waited for and proxy-fenced by each warp), one
        // device-scope release on the band's semaphore, so that a reduction of the band
        // across tensor-parallel shards can start while later bands are still computed.
        const int32_t mt = args.st[args.nst - 1].g.m_tiles;
        const int32_t band = (int32_t)(((int64_t)(tr.m + 1) * args.n_bands - 1) / mt);
        if (!ptx::mbar_wait_bounded(&epi_done[acc], apar, pto)) {
          record_error(args, ERRC_PIPELINE, t, 12);
          *abort_flag = 1;
        } else {
          ptx::fence_acq_rel_gpu();
          ptx::red_release_gpu_add(args.band_flags + band, 1u);
        }
      } else if ((args.stack ? stack_mid : tr.s == 0) && threadIdx.x == 64) {
        // stage 0 feeds the last stage (two-stage chains) or the pointwise stage (attention);
        // a stack's stage s feeds stage s + 1 through the semaphores of boundary s
        const bool to_pw = args.nst == 3 && !args.stack;
        const int32_t flag = producer_flag(to_pw ? args.dep_pw : args.dep, tr.m, tr.c);
        uint32_t* const fl = to_pw ? args.flags_pw : args.flags + (args.stack ? tr.s * args.flags_stride : 0);
        if (flag >= 0) {
          // cuSync §IV-E "Post": after all of this CTA's stores of the tile (the epi_done
          // barrier orders its 128 threads' stores before this thread), one device-scope
          // release.
          if (!ptx::mbar_wait_bounded(&epi_done[acc], apar, pto)) {
            record_error(args, ERRC_PIPELINE, t, 5);
            *abort_flag = 1;
          } else if (!((args.flags_bits & kDebugSkipPost) && tr.m == 0 && tr.c == 0)) {
            ptx::fence_acq_rel_gpu();
            ptx::red_release_gpu_add(fl + flag, 1u);
            if (args.trace && leader) args.trace[chain_tile(args, tr.q)].t_post = ptx::globaltimer();
          }
        }
      }
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (kPair) ptx::cluster_sync();  // both CTAs are done with the pair's TMEM and barriers
  if (warp == 1) {
    ptx::tc_fence_after();
    if (kPair) ptx::tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if ((args.pdl_role & 2) && threadIdx.x == 0) ptx::pdl_wait();
}

// After a run with row bands: raise each band semaphore to at least the count a complete
// run posts, so that every stream wait on a band ends even when a tile of this run gave up
// (its timeout is reported through the error word).  Normally the run has posted them all
// and this changes nothing.
struct BandTargets {
  uint32_t v[16];
};
__global__ void band_release_kernel(uint32_t* band_flags, BandTargets targets, int32_t n) {
  const int32_t i = (int32_t)threadIdx.x;
  if (i < n) atomicMax(band_flags + i, targets.v[i]);
}

// Fill a buffer with the bf16 sentinel 0x8000 using 16-byte stores (CUDA-FGS §4.6.4.2,
// initialisation "in a separate kernel").  overlap: launched as a programmatic dependent
// of the kernel before it, whose reads of the buffer must end first; once they have, the
// chain after this kernel may start (it waits for this fill before it touches the buffer).
__global__ void sentinel_fill_kernel(uint4* buf, int64_t n16, int32_t overlap) {
  if (overlap) {
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
  }
  const uint4 s = make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
    buf[i] = s;
}

}  // namespace cusync
