/*
 * cusync.h -- C ABI of a GB300 (sm_103a) library for tile-level synchronisation of a
 * chain of two dependent kernels: a producer GEMM (or implicit-GEMM convolution) with a
 * fused GeLU / SwiGLU / ReLU epilogue, and a consumer GEMM (or convolution) that reads
 * the producer's output.  Consumer thread blocks start on each input tile as soon as
 * that tile has been produced, instead of waiting for the whole producer grid, so the
 * under-filled last wave of one kernel overlaps the first wave of the next.
 *
 * Sources (cited by title and section):
 *  [cuSync]   "A Framework for Fine-Grained Synchronization of Dependent GPU Kernels"
 *             (arXiv 2305.13450).
 *  [CUDA-FGS] CUDA Programming Guide, section 4.6 "Fine-Grained Synchronization".
 *
 * Conventions shared by every entry point:
 *  - All tensors are bf16, row-major, device-resident, 16-byte aligned and owned by the
 *    caller.  The library never allocates or frees memory in a run call.
 *  - Weights are passed with the reduction dimension contiguous ("[out, in]", the
 *    layout torch.nn.Linear stores): W1t is [N1, K] where the chain computes X x W1.
 *  - Run calls are asynchronous on the caller's stream (a cudaStream_t passed as
 *    cusync_stream_t; NULL is the legacy default stream).  They return launch-time
 *    errors immediately; a device-side timeout is reported by cusync_chain_check.
 *  - A chain object owns its synchronisation state (semaphores, tile counters, error
 *    word) and is not thread-safe: use one chain per stream at a time.
 *  - Shapes the kernels cannot cover return CUSYNC_ERR_UNSUPPORTED; there is no
 *    fallback path.
 *  - Every synchronisation policy yields byte-identical outputs: the tiles, the k order
 *    inside a tile and the epilogue arithmetic do not depend on the policy.
 */
#ifndef CUSYNC_H_
#define CUSYNC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* cusync_stream_t;

/* Synchronisation policy between the producer and the consumer ([cuSync] §IV-E,
 * "Synchronization Policies"; [CUDA-FGS] §4.6.2, Table 14). */
typedef enum {
  /* Stream synchronisation ([cuSync] §II-A "Stream Synchronization"): the consumer
   * kernel is launched after the producer kernel on the same stream; the baseline. */
  CUSYNC_POLICY_STREAM = 0,
  /* RowSync: one semaphore per producer row of tiles; a consumer tile waits, before
   * its first k-block, until every tile of the rows it reads has been posted. */
  CUSYNC_POLICY_ROW = 1,
  /* TileSync: one semaphore per producer tile; a consumer tile waits on each producer
   * tile just before the first k-block that reads it. */
  CUSYNC_POLICY_TILE = 2,
  /* StridedSync: producer column tiles D = n_tiles/G apart share one semaphore (G
   * members per group), and the producer visits each group's members consecutively. */
  CUSYNC_POLICY_STRIDED_TILE = 3,
  /* Sentinel in data ([CUDA-FGS] §4.6.4): the intermediate buffer is filled with the
   * bf16 pattern 0x8000 (-0.0) before the producer runs, the producer never stores that
   * pattern, and the consumer re-loads an input tile while it still holds it.  On
   * sm_103a the check is done in software on every element of the landed tile (the
   * copy-time validity report of compute capability 10.7 is not used). */
  CUSYNC_POLICY_SENTINEL = 4,
  /* Whichever of the five the latency model (cusync_predict_policies, default model)
   * predicts fastest for the described shape, resolved when the chain is created; no
   * single policy is best for every shape ([cuSync] §VI-B). */
  CUSYNC_POLICY_AUTO = 5
} cusync_policy_t;

/* The chain computed ([cuSync] §II-B, Fig. fig:gpt-3:mlp, Table tab:resnet-sizes). */
typedef enum {
  /* H = GeLU_tanh(X x W1) (bf16), Y = H x W2.  X [M,K], W1t [N1,K], H [M,N1],
   * W2t [N2,N1], Y [M,N2]. */
  CUSYNC_CHAIN_MLP_GELU = 0,
  /* H = silu(X x Wgate) * (X x Wup) (bf16), Y = H x Wdown.  W1t [2*N1, K] holds the
   * rows of Wgate^T (0..N1-1) followed by those of Wup^T (N1..2*N1-1); W2t = Wdown^T
   * [N2, N1]. */
  CUSYNC_CHAIN_MLP_SWIGLU = 1,
  /* H = ReLU(conv3x3(x, w1)) (bf16), y = conv3x3(H, w2); stride 1, pad 1, NHWC images
   * x [n,h,w,c], H and y [n,h,w,k_out], KRSC weights w1 [k_out,3,3,c] and
   * w2 [k_out,3,3,k_out]. */
  CUSYNC_CHAIN_CONV_RELU = 2,
  /* Self-attention block of [cuSync] Fig. fig:gpt-3:attention, three dependent kernels:
   * XQKV = X x QKV (X [M,K]; W1t = QKV^T [3*N1, K], rows 0..N1-1 the XQ block, N1..2N1-1
   * the XV block, 2N1..3N1-1 the XK block, as the figure slices XQKV); then per head of
   * 128 columns and token row, XDot = softmax(XQ * XV) * XK (element-wise products,
   * softmax over the head's 128 values; dropout is the identity of inference); then
   * Y = XDot x W2 (W2t [N2, N1]).  Policies: ROW or TILE between both pairs of kernels,
   * STRIDED_TILE = StridedSync (G = 3: a head's Q, V and K tiles share one semaphore)
   * then TileSync, STREAM = three stream-ordered kernels; SENTINEL is not offered.
   * N1 must be a multiple of the tile width and of 128. */
  CUSYNC_CHAIN_ATTENTION = 3,
  /* A stack of `stages` 3x3 convolutions ([cuSync] Table tab:resnet-sizes: a ResNet-38
   * layer group repeats pairs of convolutions with equal channels): h_1 =
   * ReLU(conv(x, w_1)) (bf16), h_s = ReLU(conv(h_{s-1}, w_s)), y = conv(h_{N-1}, w_N);
   * stride 1, pad 1, NHWC images of c channels throughout (c == k_out), all in one
   * persistent kernel (or one kernel per stage under STREAM and PDL).  Every stage waits
   * on the one before it with the chain's policy (ROW, TILE or SENTINEL).  The
   * intermediates live in a caller-owned workspace (cusync_chain_info_t::work_bytes):
   * two buffers used in turn under ROW, TILE and STREAM (a stage overwrites the input of
   * the stage before it only after its own waits have covered every reader); under
   * SENTINEL one buffer per intermediate in each of two sets: run r uses set r % 2 and
   * its last launch writes the sentinel over the other set in its tail, so no fill
   * precedes a run (both sets are filled before the first run on a workspace, and after
   * cusync_chain_reset). */
  CUSYNC_CHAIN_CONV_STACK = 4
} cusync_chain_kind_t;

/* How the stages are launched so that a waiting consumer can never starve the producer
 * ([cuSync] §IV-B "Stage Processing Order"; [CUDA-FGS] §4.6.5). */
typedef enum {
  /* One persistent kernel with a single tile queue holding all producer tiles before all
   * consumer tiles; every tile is claimed from a counter by a running CTA, so every tile
   * a consumer waits on is already held by a running CTA (no co-residency needed). */
  CUSYNC_LAUNCH_PERSISTENT = 0,
  /* Two persistent kernels on one stream; the consumer is launched with programmatic
   * stream serialisation and the producer triggers its dependents at its start. */
  CUSYNC_LAUNCH_PDL = 1
} cusync_launch_t;

typedef enum {
  CUSYNC_OK = 0,
  CUSYNC_ERR_INVALID_ARG = 1, /* null, misaligned or inconsistent argument */
  CUSYNC_ERR_UNSUPPORTED = 2, /* shape or option the kernels do not cover */
  CUSYNC_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  CUSYNC_ERR_NOMEM = 4,       /* allocation of the chain's state failed */
  CUSYNC_ERR_TIMEOUT = 5,     /* a device wait on a semaphore or sentinel gave up */
  CUSYNC_ERR_DEVICE = 6       /* a device-internal wait gave up (pipeline fault) */
} cusync_status_t;

/* cusync_chain_desc_t.flags */
#define CUSYNC_FLAG_NO_REORDER (1u << 0)  /* disable [cuSync] §V "Reorder Tile Loads and
                                             Synchronization": weight tiles are then
                                             loaded only after the A-tile wait */
#define CUSYNC_FLAG_TRACE (1u << 1)       /* record a per-tile timeline (cusync_chain_trace) */
#define CUSYNC_FLAG_NO_RUN_OVERLAP (1u << 2) /* launch a run's first kernel in plain stream order
                                            (by default it is a programmatic dependent of the
                                            kernel before it in the stream: its set-up overlaps
                                            that kernel's tail, and it waits for that kernel
                                            to complete before touching memory) */
/* Fault injection for tests; each makes a device wait expire, never a GPU fault. */
#define CUSYNC_DEBUG_SKIP_POST (1u << 8)     /* the producer never posts tile (0,0) */
#define CUSYNC_DEBUG_SKIP_INIT (1u << 9)     /* SENTINEL: skip the sentinel fill */
#define CUSYNC_DEBUG_SKIP_SPLIT (1u << 10)   /* K split: the first unit of producer tile
                                                (0,0) stores no partial sums, so the next
                                                unit's bounded read of its slot expires */

typedef struct {
  int32_t kind;     /* cusync_chain_kind_t */
  int32_t policy;   /* cusync_policy_t */
  int32_t launch;   /* cusync_launch_t (ignored for CUSYNC_POLICY_STREAM) */
  int32_t _pad0;
  int64_t M, K, N1, N2;              /* MLP chains (see cusync_chain_kind_t) */
  int32_t n, h, w, c, k_out;         /* CONV_RELU: NHWC image and output channels */
  int32_t tile_n;                    /* accumulator tile width: 128, 192 (GeLU MLP chains
                                        on CTA pairs only) or 256; 0 = planner:
                                        128 for a single-CTA MLP chain whose producer
                                        tiles at 256 would fill at most 1/16 of the SMs,
                                        else 256 */
  int32_t strided_group;             /* G for STRIDED_TILE; 0 = 2 */
  uint32_t flags;                    /* CUSYNC_FLAG_* | CUSYNC_DEBUG_* */
  int32_t num_sms;                   /* SMs the kernels may use; 0 = all of the device */
  int32_t raster_rows;               /* tile order: row tiles per raster group (columns
                                        outer, rows inner within a group); 1 = plain
                                        row-major; 0 = planner: half the row tiles for an
                                        MLP chain on CTA pairs with at least four row
                                        tiles and no row bands, else row-major */
  uint64_t timeout_ns;               /* bound of every device wait on a semaphore or a
                                        sentinel; 0 = 1e9 (one second) */
  int32_t l2_prefetch;               /* k-blocks a prefetch warp runs ahead of the TMA
                                        loader, prefetching the weight boxes into L2
                                        through the copy engine; -1 = none; 0 = planner:
                                        4 for MLP chains on CTA pairs whose producer
                                        GEMM is K-split (weight streaming), else none */
  int32_t cta_pair;                  /* CTAs per tile: 1, or 2 = a CTA pair (cluster of
                                        two) computes a 256-row tile with cta_group::2
                                        MMAs, each CTA loading half of the weight tile
                                        (MLP and attention chains; in the attention
                                        chain's pointwise stage each CTA computes its
                                        128 rows); 0 = 2 for MLP and attention chains
                                        with M >= 256, else 1 */
  int32_t ksplit;                    /* K split of the producer GEMM (MLP chains): each
                                        producer tile is computed by this many work units
                                        over consecutive k-block ranges, whose fp32 partial
                                        sums are added in unit order (deterministic) before
                                        the last unit applies the epilogue and posts -- the
                                        z dimension of the first GEMM's grid in [cuSync]
                                        Table tab:waves:mlp.  0 = planner: when the
                                        producer tiles fill at most half of a wave, the
                                        largest split that keeps all units in it (at
                                        most 4); when they fill more than half of one
                                        wave, 2; else none; never fewer than 16 k-blocks
                                        per unit.  1 = none */
  int32_t stages;                    /* CONV_STACK: convolutions in the stack, 2..16 */
  int32_t ksplit_consumer;           /* K split of the consumer GEMM of an MLP chain, as
                                        ksplit: each consumer tile computed by this many
                                        units, added in unit order by the last.  0 =
                                        planner: when single-CTA consumer tiles fill at
                                        most half of a wave, as many units per tile as fit
                                        in one wave (at most 4, at least 16 k-blocks each);
                                        none on CTA pairs;
                                        none under STRIDED_TILE with more than 64 groups.
                                        1 = none */
  int32_t bands;                     /* MLP chains: row bands of the output Y, each with a
                                        semaphore that its consumer tiles post after their
                                        stores, for cusync_run_mlp_bands / cusync_band_wait
                                        (at most 16 and at most the consumer's row tiles;
                                        row-major tile order).  0 = none */
  int32_t ksplit_skew;               /* graded K split of the producer: each unit this
                                        many k-blocks longer than the one before it (the
                                        last takes the remainder), so the units finish one
                                        after the other and each exchange of partial sums
                                        overlaps the later units' mainloops.  0 =
                                        planner: 8 for MLP and attention chains on CTA
                                        pairs (a quarter of a unit, even, when units are
                                        shorter than 32 k-blocks), else none; -1 = equal
                                        units; at most 64 */
} cusync_chain_desc_t;

/* Wave arithmetic of a two-kernel chain ([cuSync] §II-A "Thread block Wave Execution",
 * Table tab:intro, §III-A). */
typedef struct {
  int64_t tbs[2];          /* thread blocks (tiles) of the producer and consumer */
  double waves[2];         /* fractional waves tbs / cap */
  int32_t waves_ceil[2];   /* ceil(tbs / cap) */
  double util[2];          /* tbs / (ceil(waves) * cap) */
  int32_t stream_waves;    /* waves_ceil[0] + waves_ceil[1]: stream synchronisation */
  int32_t fused_waves;     /* ceil((tbs[0] + tbs[1]) / cap): tile synchronisation */
  double fused_waves_frac; /* (tbs[0] + tbs[1]) / cap */
  int64_t last_wave_tbs;   /* thread blocks in the fused last wave */
  int32_t cap;             /* occupancy * num_sms */
  int32_t occupancy;
  int32_t num_sms;
  int32_t tile_m, tile_n, tile_k; /* tile chosen by cusync_plan_waves (0 from
                                     cusync_wave_stats) */
} cusync_wave_report_t;

/* One tile of a traced run (CUSYNC_FLAG_TRACE): %globaltimer stamps in nanoseconds taken
 * by the roles of the CTA that ran it.  Producer tiles come first (index < tbs[0]). */
typedef struct {
  uint32_t tile;      /* tile index in the chain (producer tiles, then consumer tiles) */
  uint32_t smid;      /* SM the tile ran on */
  uint32_t cta;       /* CTA (blockIdx.x) */
  uint32_t stage;     /* 0 producer, 1 consumer */
  uint64_t t_claim;   /* the scheduler claimed the tile */
  uint64_t t_ready;   /* the loader passed the waits before k-block 0 */
  uint64_t t_mma0;    /* the first stage of the tile landed */
  uint64_t t_mma1;    /* the last MMA of the tile was committed */
  uint64_t t_epi;     /* the epilogue finished the tile's stores */
  uint64_t t_post;    /* producer: the tile's semaphore was posted (0 if none) */
  uint32_t polls;     /* consumer: semaphore reads its waits took (probes and polls) */
  uint32_t reloads;   /* consumer, sentinel policy: A k-blocks loaded again */
  uint32_t land_clk;  /* SM cycles the MMA issuer waited for this tile's stages to land */
  uint32_t check_clk; /* SM cycles of the sentinel check of this tile (scans and reloads) */
  uint64_t t_acc;     /* the epilogue found the tile's accumulator complete */
  uint64_t t_xchg;    /* K split, a unit after the first: the epilogue (first warp) had read
                         every partial sum it adds from the unit before it (0 otherwise) */
} cusync_trace_rec_t;

/* Geometry of a chain (for tests and introspection). */
typedef struct {
  int32_t m_tiles[2], n_tiles[2], k_blocks[2];
  int32_t n_out[2];        /* output columns written per tile */
  int32_t tile_m, tile_n, tile_k;
  int32_t strided_group, strided_distance;
  int32_t num_flags;       /* semaphores of the policy */
  int32_t grid[2];         /* CTAs of the producer / consumer launch (fused: grid[0]) */
  int32_t num_sms;
  int32_t conv_rows_per_tile; /* CONV_RELU: image rows per row tile */
  int32_t cta_pair;           /* CTAs per tile (1 or 2); each posts its tile's semaphore */
  int32_t policy;             /* the policy the plan uses (CUSYNC_POLICY_AUTO resolved) */
  int32_t ksplit;             /* K-split units per producer tile (1 = none); the
                                 producer launch has m_tiles*n_tiles*ksplit units */
  int32_t kb_per_split;       /* k-blocks per unit (graded split: of unit 0) */
  /* ATTENTION (three stages): stage 1 is the pointwise kernel, stage 2 the output GEMM */
  int32_t nst;                /* stages of the chain: 2, or 3 */
  int32_t m_tiles2, n_tiles2, k_blocks2, n_out2, grid2;
  int32_t num_flags_pw;       /* semaphores the pointwise stage waits on */
  int32_t strided_group_pw, strided_distance_pw;
  int32_t work_buffers;       /* CONV_STACK: intermediate buffers in the workspace */
  int64_t work_bytes;         /* CONV_STACK: bytes of the caller's workspace (n*h*w*c
                                 bf16 per buffer) */
  int32_t ksplit_consumer;    /* K-split units per consumer tile (1 = none) */
  int32_t kb_per_split_consumer;
  int32_t raster_rows;        /* row tiles per group of the tile order (1 = row-major) */
  int32_t ksplit_skew;        /* k-blocks each producer unit adds to the one before it
                                 (kb_per_split is then unit 0's length) */
} cusync_chain_info_t;

/* Latency model of one chain run, in nanoseconds (cusync_predict_policies).  A tile
 * takes start_ns + k_blocks x kblock_ns + epilogue_ns ("ALCOP" analytical model, Table
 * I: initial phase, steady main loop, epilogue); the tiles are played out on the
 * launch's persistent CTAs in queue order, and a consumer k-block starts only after the
 * semaphores the device would wait on are posted ([cuSync] §IV-E). */
typedef struct {
  double kblock_ns[2];       /* mainloop time per 64-wide k-block of a producer / consumer
                                tile (of a CTA pair's 256-row tile with pairs) */
  double wait_kblock_ns;     /* extra time at each consumer k-block that consults a
                                semaphore (TileSync, StridedSync) */
  double sentinel_kblock_ns; /* consumer time per k-block under the sentinel policy */
  double start_ns;           /* a tile's first copy in flight; also the pipeline refill
                                after a consumer wait that blocked */
  double epilogue_ns[2];     /* last MMA to stores done, producer / consumer tile */
  double post_ns;            /* producer stores done to the post seen by a consumer */
  double gap_ns;             /* producer kernel end to consumer kernel start (stream) */
  double fill_ns_per_mb;     /* sentinel fill of the intermediate, per MB */
  double tile_ns;            /* a tile that is not its CTA's first: from the previous tile's
                                last k-block to its first (the next claim, the arming and
                                the first copy behind the previous tile's last copies) */
  double tile_wait_ns;       /* a consumer tile's first semaphore consult, even when the
                                semaphores are already posted (the probe's round trip, the
                                acquire and proxy fences) */
} cusync_latency_model_t;

typedef struct {
  double us[5];      /* predicted microseconds per run, indexed by cusync_policy_t
                        (STREAM..SENTINEL); -1 where the policy does not apply */
  int32_t best_sync; /* fastest tile-synchronised policy (ROW..SENTINEL) */
  int32_t best;      /* fastest policy, stream order included */
  int32_t num_sms;   /* SMs the prediction assumed */
} cusync_policy_prediction_t;

/* The model's constants for the chain described by *d, calibrated on GB300 (bench
 * traces: per-k-block mainloop times for single CTAs, CTA pairs and convolutions,
 * epilogue time per output column by activation).  Pure host computation. */
cusync_status_t cusync_default_latency_model(const cusync_chain_desc_t* d, cusync_latency_model_t* out);

/* Predicted time of one run of the chain described by *d (its policy field is ignored)
 * under each policy, with the persistent launch, on d->num_sms SMs (0: the current
 * device's count).  model NULL: cusync_default_latency_model.  Pure host computation. */
cusync_status_t cusync_predict_policies(const cusync_chain_desc_t* d, const cusync_latency_model_t* model,
                                        cusync_policy_prediction_t* out);

/* Status code as a static string. */
const char* cusync_status_string(cusync_status_t s);

/* Raw wave arithmetic for grids of tbs0 and tbs1 thread blocks with the given occupancy
 * (thread blocks per SM) on num_sms SMs.  tbs1 may be 0 (a single kernel).
 * INVALID_ARG if out is NULL, a count is negative or occupancy/num_sms < 1. */
cusync_status_t cusync_wave_stats(int64_t tbs0, int64_t tbs1, int32_t occupancy, int32_t num_sms,
                                  cusync_wave_report_t* out);

/* Tiles the chain described by *d would launch and their wave arithmetic on
 * d->num_sms SMs (0: the current device's count) at this library's occupancy of one
 * CTA per SM.  Pure host computation. */
cusync_status_t cusync_plan_waves(const cusync_chain_desc_t* d, cusync_wave_report_t* out);

/* Validate *d, allocate the chain's synchronisation state on the current device and
 * prepare the kernels.  *out receives an opaque handle owned by the caller (release it
 * with cusync_destroy_chain).  INVALID_ARG / UNSUPPORTED for bad descriptors, NOMEM or
 * CUDA on allocation or device errors. */
typedef struct cusync_chain* cusync_chain_t;
cusync_status_t cusync_create_chain(const cusync_chain_desc_t* d, cusync_chain_t* out);

/* Run an MLP chain (kinds MLP_GELU, MLP_SWIGLU) on `stream`: writes H (the
 * intermediate, caller-owned scratch of M*N1 bf16 that holds the producer's output on
 * return) and Y.  Pointers: X [M,K], W1t [N1,K] (SwiGLU: [2*N1,K]), W2t [N2,N1],
 * H [M,N1], Y [M,N2]; device memory, 16-byte aligned, not overlapping H or Y.
 * Asynchronous; INVALID_ARG / UNSUPPORTED / CUDA on launch-time errors.
 * Only kernel launches are enqueued on `stream`, so the call can be recorded by CUDA
 * stream capture; the run count that the semaphores are compared against lives in the
 * chain's device state, so each replay of a captured run is a new run.  Runs of one
 * chain must not overlap (one stream, or ordered streams). */
cusync_status_t cusync_run_mlp(cusync_chain_t chain, const void* X, const void* W1t, const void* W2t, void* H,
                               void* Y, cusync_stream_t stream);

/* Run a CONV_RELU chain: x [n,h,w,c], w1 [k_out,3,3,c], w2 [k_out,3,3,k_out] (KRSC),
 * y1 (intermediate, [n,h,w,k_out]) and y2 ([n,h,w,k_out]).  Same rules as
 * cusync_run_mlp. */
cusync_status_t cusync_run_conv_chain(cusync_chain_t chain, const void* x, const void* w1, const void* w2, void* y1,
                                      void* y2, cusync_stream_t stream);

/* Run a CONV_STACK chain: x [n,h,w,c], w [stages][c,3,3,c] (the stages' KRSC weights one
 * after the other), work (caller-owned workspace of cusync_chain_info_t::work_bytes, which
 * receives the intermediates; its contents on return are unspecified) and y
 * ([n,h,w,c], the last convolution).  Same rules as cusync_run_mlp. */
cusync_status_t cusync_run_conv_stack(cusync_chain_t chain, const void* x, const void* w, void* work, void* y,
                                      cusync_stream_t stream);

/* Run an ATTENTION chain on `stream` ([cuSync] Fig. fig:gpt-3:attention): writes XQKV
 * (first intermediate, [M, 3*N1] bf16: the XQ, XV and XK blocks side by side), XDot
 * (second intermediate, [M, N1] bf16) and Y [M, N2].  Inputs: X [M,K], Wqkv_t [3*N1,K]
 * (QKV^T, K contiguous), W2t [N2,N1].  Device memory, 16-byte aligned, caller-owned, the
 * outputs distinct from one another and from X.  Asynchronous, capturable like
 * cusync_run_mlp; INVALID_ARG / UNSUPPORTED / CUDA on launch-time errors. */
cusync_status_t cusync_run_attention(cusync_chain_t chain, const void* X, const void* Wqkv_t, const void* W2t,
                                     void* XQKV, void* XDot, void* Y, cusync_stream_t stream);

/* Synchronise `stream` and read the chain's device error word.  Returns OK, TIMEOUT (a
 * consumer gave up waiting on a semaphore or a sentinel: the outputs of that run are
 * not valid) or DEVICE.  After an error the chain's synchronisation state is reset, so
 * the next run starts clean.  If code/detail are non-NULL they receive the raw error
 * word and its detail (tile and k-block of the failing wait). */
cusync_status_t cusync_chain_check(cusync_chain_t chain, cusync_stream_t stream, uint32_t* code, uint32_t* detail);

/* Clear the chain's semaphores, tile counters and error word (stream-ordered). */
cusync_status_t cusync_chain_reset(cusync_chain_t chain, cusync_stream_t stream);

/* Geometry the chain described by *d would use (tiles, semaphores, grids on
 * d->num_sms SMs, or the current device's count when 0).  Pure host computation. */
cusync_status_t cusync_plan_info(const cusync_chain_desc_t* d, cusync_chain_info_t* out);

/* The semaphore waits the consumer performs for row tile m_tile of the chain described
 * by *d, in issue order: entry i is (kb[i], flag[i], per_run[i]): before loading A
 * k-block kb[i] it waits until semaphore flag[i] has received per_run[i] posts in the
 * current run.  Writes at most max entries and the total count to *n_out.  Pure host
 * computation with the same code the device runs. */
cusync_status_t cusync_consumer_waits(const cusync_chain_desc_t* d, int32_t m_tile, int32_t* kb, int32_t* flag,
                                      uint32_t* per_run, int32_t max, int32_t* n_out);

/* The waits of work unit `unit` (0 .. ksplit_consumer-1) of consumer tile m_tile of a
 * two-stage GEMM chain whose consumer is K-split: the same triples as
 * cusync_consumer_waits for the k-blocks the unit computes, as its loader performs them
 * (a unit waits before its own first k-block for what it reads there).  INVALID_ARG for
 * other chains or an out-of-range tile or unit. */
cusync_status_t cusync_consumer_unit_waits(const cusync_chain_desc_t* d, int32_t m_tile, int32_t unit, int32_t* kb,
                                           int32_t* flag, uint32_t* per_run, int32_t max, int32_t* n_out);

/* ATTENTION chains: the semaphore waits of pointwise tile (m_tile, head) on the QKV GEMM
 * ([cuSync] §IV-E; Fig. fig:use-case:self-attention:strided for StridedSync): entry i
 * is (flag[i], per_run[i]) -- semaphore flag[i] must have received per_run[i] posts in
 * the current run before the head is computed.  Writes at most max entries and the
 * count to *n_out.  Pure host computation with the code the device runs. */
cusync_status_t cusync_pointwise_waits(const cusync_chain_desc_t* d, int32_t m_tile, int32_t head, int32_t* flag,
                                       uint32_t* per_run, int32_t max, int32_t* n_out);

/* The semaphore producer tile (m_tile, n_tile) posts (-1 if the policy posts none), and
 * the producer column visited at position y of a row (the policy's tile order).  Pure
 * host computation. */
cusync_status_t cusync_producer_flag(const cusync_chain_desc_t* d, int32_t m_tile, int32_t n_tile, int32_t* flag);
cusync_status_t cusync_producer_col(const cusync_chain_desc_t* d, int32_t y, int32_t* col);

/* (row tile, column tile) at position u of stage `stage`'s tile queue (0 = producer,
 * 1 = consumer): the order in which the persistent CTAs claim tiles.  Pure host
 * computation. */
cusync_status_t cusync_tile_at(const cusync_chain_desc_t* d, int32_t stage, int32_t u, int32_t* m_tile,
                               int32_t* n_tile);

/* Semaphores that cusync_run_mlp_noalloc's fixed array holds: 16384 words less the 48
 * control words in front of the semaphores. */
#define CUSYNC_NOALLOC_MAX_SEMAPHORES 16336

/* Allocation-free variant of cusync_run_mlp, for callers that cannot allocate device
 * memory themselves (for example an operator running inside a runtime that owns the
 * device memory pool, or a serving loop that must avoid cudaMalloc's synchronisation).
 * The pages have no counterpart: it exists for such callers only.
 *
 * It needs no chain object: it plans the chain described by *d and runs it with the same
 * kernels, keeping the synchronisation state (error word, tile counters, semaphores) in a
 * fixed 64 KiB array inside the library (CUSYNC_NOALLOC_MAX_SEMAPHORES semaphores at
 * most; larger plans return CUSYNC_ERR_UNSUPPORTED).  It calls no cudaMalloc or
 * cudaFree.  Inputs and outputs are as for cusync_run_mlp.
 *  - There is no workspace for K-split partial sums: d->ksplit and d->ksplit_consumer
 *    must be 0 or 1 (CUSYNC_ERR_UNSUPPORTED otherwise), and 0 means 1 here, where
 *    cusync_run_mlp's planner may split.  With both set to 1, cusync_run_mlp on the same
 *    descriptor writes byte-identical H and Y.
 *  - The first call on each device looks up the array's device address and prepares the
 *    kernels for that device; make that first call before any stream capture.
 *  - Every call clears the part of the array it uses on `stream`, then launches; the
 *    array keeps the last call's contents.  Calls whose work may overlap on the GPU
 *    (e.g. on two unordered streams) race on the array: order them.
 *  - If error_word is non-NULL the call waits for the chain to finish and stores the
 *    device error word there (0 = no wait expired), returning CUSYNC_ERR_TIMEOUT or
 *    CUSYNC_ERR_DEVICE when it is set.  With NULL it returns after the launches. */
cusync_status_t cusync_run_mlp_noalloc(const cusync_chain_desc_t* d, const void* X, const void* W1t,
                                       const void* W2t, void* H, void* Y, cusync_stream_t stream,
                                       uint32_t* error_word);

/* Tensor-parallel MLP shard with the reduction of its output overlapped band by band.
 *
 * The pages' MLP block is one shard of a tensor-parallel layer: X x W1 split by columns,
 * x W2 split by rows, the shards' outputs summed across GPUs ([cuSync] §II-B "GPT-3", the
 * H/8 shard of Fig. fig:gpt-3:mlp); overlapping that communication with the computation is
 * the pages' next step ([cuSync] "Conclusion"), and [CUDA-FGS] §4.6 notes that the same
 * readiness protocol reaches another GPU when the consumer reads at a scope that covers
 * both.  Here each consumer tile posts its row band's semaphore after its stores, so a
 * reduction of band b (an all-reduce across the shards, on another stream) can start
 * while later bands are still being computed.
 *
 * cusync_run_mlp_bands runs the chain (chain created with desc.bands > 0) on `stream` as
 * cusync_run_mlp does, with band semaphores cleared first; band_stream (not `stream`) is
 * made to wait until they are cleared.  Then, for each band b in turn, the caller calls
 * cusync_band_wait(chain, b, band_stream) and enqueues its reduction of rows
 * cusync_band_rows(desc, b) of Y on band_stream.  After the run's kernels, `stream` runs a
 * one-thread-block kernel that raises every band semaphore to the count of a complete run,
 * so every band wait ends even if a tile of the run gave up waiting (reported by
 * cusync_chain_check); normally it changes nothing.
 *  - Before the next run of the chain, make `stream` wait for band_stream's work of this
 *    run: the next run overwrites Y and clears the semaphores.
 *  - Not inside CUDA stream capture (CUSYNC_ERR_UNSUPPORTED): a band wait is a stream
 *    memory operation (cuStreamWaitValue32), which graph dependencies do not see.
 *  - cusync_band_wait returns INVALID_ARG before a successful cusync_run_mlp_bands of the
 *    chain, for a band out of range, and after cusync_chain_reset. */
cusync_status_t cusync_run_mlp_bands(cusync_chain_t chain, const void* X, const void* W1t, const void* W2t,
                                     void* H, void* Y, cusync_stream_t stream, cusync_stream_t band_stream);
cusync_status_t cusync_band_wait(cusync_chain_t chain, int32_t band, cusync_stream_t band_stream);
/* Rows [*row0, *row0 + *rows) of Y in band `band` of the chain described by *d (pure host
 * computation). */
cusync_status_t cusync_band_rows(const cusync_chain_desc_t* d, int32_t band, int64_t* row0, int64_t* rows);

/* Copy the timeline of the last traced run into out[0..max) (one record per tile, in tile
 * order) after synchronising `stream`; *n_out receives the number of tiles.  INVALID_ARG
 * if the chain was created without CUSYNC_FLAG_TRACE. */
cusync_status_t cusync_chain_trace(cusync_chain_t chain, cusync_stream_t stream, cusync_trace_rec_t* out,
                                   int32_t max, int32_t* n_out);

/* Release the chain's device state.  NULL is accepted. */
cusync_status_t cusync_destroy_chain(cusync_chain_t chain);

#ifdef __cplusplus
}
#endif
#endif /* CUSYNC_H_ */
