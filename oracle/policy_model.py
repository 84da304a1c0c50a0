"""Latency model of one chain run under each synchronisation policy (oracle; test
infrastructure only).

[ALCOP] "ALCOP: Automatic Load-COmpute Pipelining in Deep Learning Compiler for
AI-GPUs", analytical model (Table I): the thread blocks of a kernel run in
threadblock batches that occupy all SMs, so a kernel takes (number of batches) x
(threadblock latency), and a threadblock's latency is the sum of an initial phase
(T_init, the first data requested and awaited), a steady main loop (T_main_loop) and
an epilogue (T_epilogue).

[cuSync] "A Framework for Fine-Grained Synchronization of Dependent GPU Kernels",
§III: with stream synchronisation the consumer kernel starts after the producer
kernel's last wave; with tile synchronisation consumer thread blocks share the waves of
the producer and each consumer tile only waits (§IV-E) for the producer tiles its policy
names.

The model written out here, step by step:

* a tile of stage s costs T_init (start_ns) when it is its CTA's first tile, then
  k_blocks(s) x kblock_ns[s] of main loop, then epilogue_ns[s]; a persistent CTA starts
  its next tile's main loop tile_ns after the previous one ends (the next claim, the
  arming and the first copy), and a tile's epilogue starts after both its main loop and
  the CTA's previous epilogue have finished;
* the queue holds the producer tiles (row-major, or row tiles taken in groups with the
  column outer within a group; StridedSync visits each group's columns one after
  another) before the consumer tiles (in the same row order); CTA q takes tile q
  first, and every later tile goes to the CTA whose main loop frees up first (the lowest
  index on a tie);
* with a K split of S, each producer tile is S consecutive queue entries over
  consecutive k-block ranges: entry k runs kb_per_split + k * kb_skew k-blocks (a graded
  split; kb_skew = 0: equal entries), and the last entry what remains; the entries form
  a chain: the epilogue of entry k > 0 (adding the running sum of the entries before it)
  also waits for entry k - 1's epilogue; only the last entry posts;
* a producer tile's post is seen post_ns after its epilogue; before consumer k-block kb
  the tile waits for the producer tiles its policy waits for there (``deps.wait_sets``);
  if they are posted later than the k-block could start, the k-block starts start_ns
  after the last post (the copy pipeline refills); a k-block that waited on anything
  costs wait_kblock_ns more (TileSync, StridedSync, RowSync's first k-block), and the
  first such k-block of a tile tile_wait_ns more before the wait (the probe of the
  semaphores and the fences after it, paid whether or not they are posted);
* the sentinel policy waits on exactly the producer tiles each k-block reads (the
  TileSync sets), costs sentinel_kblock_ns per consumer k-block and starts after the
  intermediate is filled (fill_ns_per_mb per MB);
* stream order runs the producer tiles as one launch, then, gap_ns after its last
  epilogue, the consumer tiles as a second launch with no waits;
* a convolution stack of S stages ([cuSync] §II-B "ResNet", Table ``tab:resnet-sizes``)
  is the same with every stage after the first a consumer of the stage before it: stream
  order runs S launches gap_ns apart; the fused launch queues stage 0's tiles, then stage
  1's, and so on (under the sentinel policy followed by fill units of 64 KB for the next
  run's intermediates, each fill_ns_per_mb x 0.065536 of epilogue time); the last stage's
  tiles take epilogue_ns[1], the others epilogue_ns[0].
"""

from dataclasses import dataclass

from oracle import deps


@dataclass
class Model:
    kblock_ns: tuple
    wait_kblock_ns: float
    sentinel_kblock_ns: float
    start_ns: float
    epilogue_ns: tuple
    post_ns: float
    gap_ns: float
    fill_ns_per_mb: float
    tile_ns: float = 0.0
    tile_wait_ns: float = 0.0


@dataclass
class Chain:
    """A chain's tiles: producer tiles (m, c) in queue order with k_blocks[0] each, consumer
    row tiles (m) in queue order with k_blocks[1] each, and the dependency geometry."""
    prod_tiles: list      # [(m, c)] in queue order
    cons_rows: list       # [m] in queue order
    k_blocks: tuple
    dep_chain: object     # deps.GemmChain / deps.ConvChain
    G: int = 1
    h_mb: float = 0.0
    ksplit: int = 1       # producer units per tile (K split), each over consecutive k-blocks
    kb_per_split: int = 0
    kb_skew: int = 0      # k-blocks each unit runs more than the one before it


def play(tiles, slots, t0, model, cost):
    """Run `tiles` (each passed to cost(tile, t_start) -> main-loop end) on `slots` CTAs
    from time t0.  Returns [(tile, main_end, done)] in queue order."""
    ctas = [{"free": t0, "last_done": t0, "used": False} for _ in range(max(1, min(slots, len(tiles))))]
    out = []
    for q, tile in enumerate(tiles):
        if q < len(ctas):
            k = q
        else:
            k = min(range(len(ctas)), key=lambda i: (ctas[i]["free"], i))
        c = ctas[k]
        start = c["free"] + model.tile_ns if c["used"] else c["free"] + model.start_ns
        c["used"] = True
        main_end = cost(tile, start)
        done = max(main_end, c["last_done"]) + model.epilogue_ns[tile[0]]
        c["free"] = main_end
        c["last_done"] = done
        out.append((tile, main_end, done))
    return out


def _units(chain):
    """Producer queue entries (tile, unit, k-blocks)."""
    S = max(1, chain.ksplit)
    total = chain.k_blocks[0]
    if S == 1:
        return [(t, 0, total) for t in chain.prod_tiles]
    lengths, start = [], 0
    for k in range(S):
        n = total - start if k == S - 1 else min(chain.kb_per_split + k * chain.kb_skew, total - start)
        lengths.append(n)
        start += n
    return [(t, k, lengths[k]) for t in chain.prod_tiles for k in range(S)]


def _play_producers(chain, slots, t0, model, ctas=None):
    """The producer entries on `slots` CTAs (or on the given CTA states); returns the
    CTA states, each tile's done time (its last unit's) and the latest done time."""
    S = max(1, chain.ksplit)
    units = _units(chain)
    if ctas is None:
        ctas = [{"free": t0, "last_done": t0, "used": False} for _ in range(max(1, min(slots, len(units))))]
    prev_done = {}
    tile_done = {}
    end = t0
    for q, (tile, k, nkb) in enumerate(units):
        i = q if q < len(ctas) else min(range(len(ctas)), key=lambda j: (ctas[j]["free"], j))
        c = ctas[i]
        start = c["free"] + model.tile_ns if c["used"] else c["free"] + model.start_ns
        c["used"] = True
        main_end = start + nkb * model.kblock_ns[0]
        ready = max(main_end, c["last_done"])
        if S > 1 and k > 0:
            ready = max(ready, prev_done[tile])   # the running sum of the entries before it
        done = ready + model.epilogue_ns[0]
        prev_done[tile] = done
        c["free"] = main_end
        c["last_done"] = done
        end = max(end, done)
        if k == S - 1:
            tile_done[tile] = done
    return ctas, tile_done, end


def predict_stream(chain, slots0, slots1, model):
    """Stream order: two launches, the second gap_ns after the first's last epilogue."""
    kb0, kb1 = chain.k_blocks
    _, _, end0 = _play_producers(chain, slots0, 0.0, model)
    r1 = play([(1, m) for m in chain.cons_rows], slots1, end0 + model.gap_ns, model,
              lambda tile, s: s + kb1 * model.kblock_ns[1])
    return max(d for _, _, d in r1) if r1 else end0 + model.gap_ns


def predict_fused(chain, policy, slots, model):
    """One persistent launch: producer entries, then consumer tiles that wait per policy."""
    kb1 = chain.k_blocks[1]
    sentinel = policy == "SENTINEL"
    wait_policy = "TILE" if sentinel else policy
    t0 = chain.h_mb * model.fill_ns_per_mb if sentinel else 0.0
    n_units = len(_units(chain))
    total = n_units + len(chain.cons_rows)
    ctas = [{"free": t0, "last_done": t0, "used": False} for _ in range(max(1, min(slots, total)))]
    # the producer entries come first in the queue, so every producer tile's post time
    # is known before the first consumer tile asks for it
    ctas, tile_done, end = _play_producers(chain, slots, t0, model, ctas)
    posted = {tile: d + model.post_ns for tile, d in tile_done.items()}
    wait_cache = {}
    for q, m in enumerate(chain.cons_rows, start=n_units):
        i = q if q < len(ctas) else min(range(len(ctas)), key=lambda j: (ctas[j]["free"], j))
        c = ctas[i]
        t = c["free"] + model.tile_ns if c["used"] else c["free"] + model.start_ns
        c["used"] = True
        if m not in wait_cache:
            wait_cache[m] = deps.wait_sets(chain.dep_chain, wait_policy, m, chain.G)
        consulted = False
        for kb in range(kb1):
            need = wait_cache[m][kb]
            if need:
                if not sentinel and not consulted:
                    t += model.tile_wait_ns
                    consulted = True
                ready = max(posted[p] for p in need)
                if ready > t:
                    t = ready + model.start_ns
            if sentinel:
                t += model.sentinel_kblock_ns
            else:
                t += model.kblock_ns[1] + (model.wait_kblock_ns if need else 0.0)
        done = max(t, c["last_done"]) + model.epilogue_ns[1]
        c["free"] = t
        c["last_done"] = done
        end = max(end, done)
    return end


def _grouped_rows(mt, nt, raster):
    """(row, column position) in queue order: row tiles taken in groups of `raster`, the
    column position outer and the row inner within a group; raster = 1 is row-major
    ([cuSync] §IV-C, tile processing order)."""
    out = []
    for g0 in range(0, mt, raster):
        rows = range(g0, min(g0 + raster, mt))
        out += [(m, y) for y in range(nt) for m in rows]
    return out


def gemm_chain(M, N1, N2, tile_n, n_out, pair, policy, G=2, raster=1):
    """Queue order of an MLP chain's tiles ([cuSync] §IV-C row-major, or grouped rows;
    StridedSync's producer order) and its dependency geometry."""
    bm = 128 * pair
    mt = -(-M // bm)
    nt0 = -(-N1 // n_out)
    nt1 = -(-N2 // tile_n)
    order = deps.strided_producer_order(nt0, G) if policy == "STRIDED" else list(range(nt0))
    prod = [(m, order[y]) for m, y in _grouped_rows(mt, nt0, raster)]
    cons = [m for m, _ in _grouped_rows(mt, nt1, raster)]
    return prod, cons, deps.GemmChain(M=M, N1=N1, BM=bm, BNo=n_out, BK=64)


def conv_chain(n, h, w, c, k, tile_n, th):
    """Queue order of a conv chain's tiles (row tiles of th image rows; row-major) and its
    halo-aware dependency geometry; th is the tiling's rows per tile."""
    tpi = -(-h // th)
    mt = n * tpi
    nt = -(-k // tile_n)
    prod = [(m, y) for m in range(mt) for y in range(nt)]
    cons = [m for m in range(mt) for _ in range(nt)]
    return prod, cons, deps.ConvChain(N=n, P=h, Q=w, C=k, TH=th, BNo=tile_n, BK=64)


def predict_stack(stages, tiles, k_blocks, dep_chain, policy, slots_fused, slots_stage, model, fill_units=0):
    """Predicted ns of one run of a convolution stack: `tiles` is one stage's (m, c) tiles in
    queue order (every stage has the same), `k_blocks` the k-blocks of a tile."""
    S = stages

    def run(queue, slots, t0, posts):
        ctas = [{"free": t0, "last_done": t0, "used": False} for _ in range(max(1, min(slots, len(queue))))]
        posted = {}
        end = t0
        for q, item in enumerate(queue):
            i = q if q < len(ctas) else min(range(len(ctas)), key=lambda j: (ctas[j]["free"], j))
            c = ctas[i]
            t = c["free"] + model.tile_ns if c["used"] else c["free"] + model.start_ns
            c["used"] = True
            if item is None:   # a fill unit: stores of the epilogue warps
                done = max(t, c["last_done"]) + model.fill_ns_per_mb * 65536 / 1e6
                c["last_done"] = done
                end = max(end, done)
                continue
            s, (m, col) = item
            if s == 0 or not posts:
                t += k_blocks * model.kblock_ns[0 if s == 0 else 1]
            else:
                sets = deps.wait_sets(dep_chain, "TILE" if policy == "SENTINEL" else policy, m, 1)
                consulted = False
                for kb in range(k_blocks):
                    need = sets[kb]
                    if need:
                        if policy != "SENTINEL" and not consulted:
                            t += model.tile_wait_ns
                            consulted = True
                        ready = max(posted[(s - 1, p)] for p in need)
                        if ready > t:
                            t = ready + model.start_ns
                    if policy == "SENTINEL":
                        t += model.sentinel_kblock_ns
                    else:
                        t += model.kblock_ns[1] + (model.wait_kblock_ns if need else 0.0)
            done = max(t, c["last_done"]) + model.epilogue_ns[0 if s < S - 1 else 1]
            c["free"] = t
            c["last_done"] = done
            end = max(end, done)
            if posts and s < S - 1:
                posted[(s, (m, col))] = done + model.post_ns
        return end

    if policy == "STREAM":
        t = 0.0
        for s in range(S):
            t = run([(s, tile) for tile in tiles], slots_stage, t + model.gap_ns if s else 0.0, False)
        return t
    queue = [(s, tile) for s in range(S) for tile in tiles]
    if policy == "SENTINEL":
        queue += [None] * fill_units
    return run(queue, slots_fused, 0.0, True)
