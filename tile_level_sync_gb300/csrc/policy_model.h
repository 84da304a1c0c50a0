// Latency model of a chain under each synchronisation policy, used to predict the
// fastest policy for a shape (host only).
//
// Sources:
//  * "ALCOP: Automatic Load-COmpute Pipelining in Deep Learning Compiler for AI-GPUs",
//    analytical model (Table I): a kernel's latency is its threadblock latency times the
//    number of threadblock batches, and a threadblock's latency is the sum of an initial
//    phase (the first copy in flight), a steady main loop and an epilogue.
//  * "A Framework for Fine-Grained Synchronization of Dependent GPU Kernels" (cuSync),
//    §III (stream synchronisation runs the kernels' waves one after the other; tile
//    synchronisation lets consumer tiles share waves with producer tiles), §IV-E (what a
//    consumer tile waits for under each policy), §VI-B ("no one policy" is best for
//    every shape).
//
// Here a tile's latency is T_start + (k-blocks x per-k-block time) + T_epilogue (with a
// K split, each unit of a producer tile runs its share of the k-blocks, and each unit's
// epilogue after the first -- adding the running sum of the units before it -- follows
// that of the unit before it), and the
// threadblock batches are not assumed but played out: a persistent CTA takes the next
// tile of the queue as soon as its mainloop finishes (its epilogue overlaps the next
// tile's mainloop) and starts its k-blocks tile_ns later (the claim, the arming and the
// first copy), the first tile of each CTA is its own index, later tiles go to the CTA that
// frees up first, and a consumer k-block cannot start before the semaphores it waits for
// (the same waits the device performs) are posted.  A tile's first semaphore consult costs
// tile_wait_ns whether or not they are posted (the probe and the fences), and a wait that
// blocks costs a pipeline refill (T_start) after the post is seen.  Convolution stacks
// (predict_stack_ns) chain the same rules over all of their stages.
#pragma once
#include <algorithm>
#include <cstdint>
#include <vector>

#include "geometry.h"

namespace cusync {

struct LatencyModel {
  double kblock_ns[2];        // mainloop ns per 64-wide k-block, producer / consumer tile
  double wait_kblock_ns;      // extra ns at each consumer k-block that consults a semaphore
  double sentinel_kblock_ns;  // consumer ns per k-block under the sentinel policy
  double start_ns;            // a tile's first copy in flight (also the refill after a wait)
  double epilogue_ns[2];      // last MMA to stores done, producer / consumer tile
  double post_ns;             // stores done to the post seen by a waiting consumer
  double gap_ns;              // end of one kernel to the start of the next (stream order)
  double fill_ns_per_mb;      // sentinel fill of the intermediate
  double tile_ns;             // a CTA's later tile: previous tile's last k-block to its first
  double tile_wait_ns;        // a consumer tile's first semaphore consult, posted or not
};

struct ModelChain {
  StageGeo geo[2];
  DepCfg dep;            // the policy's semaphore layout (dep.policy = the policy)
  int32_t slots_fused;   // CTAs (pairs) of the fused launch
  int32_t slots[2];      // CTAs (pairs) of the producer / consumer launch in stream order
  double h_mb;           // size of the intermediate (sentinel fill)
};

// One consumer tile's semaphore waits: for each k-block, the semaphores first needed
// there (the dependency trackers the device runs, at the k-blocks dep_kblock marks).
inline void consumer_wait_lists(const ModelChain& c, int32_t m, std::vector<std::vector<int32_t>>* out) {
  const StageGeo& g = c.geo[1];
  out->assign(g.k_blocks, {});
  DepTracker dt;
  dt.reset();
  for (int32_t kb = 0; kb < g.k_blocks; ++kb) {
    if (!dep_kblock(g, c.dep, kb)) continue;
    Wait w[kMaxWaits];
    const int n = dt.next(g, c.dep, m, kb, w);
    for (int i = 0; i < n; ++i) (*out)[kb].push_back(w[i].flag);
  }
}

struct SimCta {
  double free_main;  // its mainloop is free for the next tile
  double last_done;  // its last tile's stores are done
  bool used;
};

// Play one queue of tiles (stages [s0, s1]) on `slots` persistent CTAs from time t0.
// flag_ready[f] must hold the post time of every semaphore a consumer tile waits on
// (all producer tiles precede consumer tiles in the queue, so they are filled first).
inline double play_queue(const ModelChain& c, const LatencyModel& lm, int s0, int s1, int32_t slots, double t0,
                         bool sentinel, std::vector<double>* flag_ready) {
  const int64_t n0 = stage_units(c.geo[0]);
  const int64_t n1 = stage_units(c.geo[1]);
  const int32_t S = c.geo[0].ksplit > 1 ? c.geo[0].ksplit : 1;
  // K split: when the latest unit of each producer tile has stored its running sum (the
  // units of a tile form a chain)
  std::vector<double> unit_done(S > 1 ? (size_t)(n0 / S) : 0, 0.0);
  const int64_t total = (s0 == 0 ? n0 : 0) + (s1 == 1 ? n1 : 0);
  if (total == 0) return t0;
  std::vector<SimCta> cta((size_t)std::max<int64_t>(1, std::min<int64_t>(slots, total)));
  for (auto& x : cta) x = SimCta{t0, t0, false};
  const bool waits = s1 == 1 && s0 == 0 && c.dep.policy != POL_STREAM;
  double end = t0;
  std::vector<std::vector<int32_t>> wl;
  for (int64_t q = 0; q < total; ++q) {
    const int s = (s0 == 0 && q < n0) ? 0 : 1;
    int64_t u = (s == 0) ? q : (s0 == 0 ? q - n0 : q);
    int32_t ks = 0, nkb = c.geo[s].k_blocks;
    if (s == 0 && S > 1) {
      ks = (int32_t)(u % S);
      u /= S;
      int32_t kb0 = 0;
      split_unit(c.geo[0], ks, &kb0, &nkb);
    }
    int32_t m, y;
    tile_at(c.geo[s], (int32_t)u, &m, &y);
    const int32_t col = (s == 0) ? producer_col(c.dep, y) : y;
    // first tile of CTA q is tile q; later tiles go to the CTA that frees up first
    size_t k = 0;
    if (q < (int64_t)cta.size()) {
      k = (size_t)q;
    } else {
      for (size_t i = 1; i < cta.size(); ++i)
        if (cta[i].free_main < cta[k].free_main) k = i;
    }
    SimCta& x = cta[k];
    double t = x.used ? x.free_main + lm.tile_ns : x.free_main + lm.start_ns;
    x.used = true;
    const StageGeo& g = c.geo[s];
    if (s == 0 || !waits) {
      t += (double)nkb * lm.kblock_ns[s];
    } else {
      consumer_wait_lists(c, m, &wl);
      const double kb_ns = sentinel ? lm.sentinel_kblock_ns : lm.kblock_ns[1];
      bool consulted = false;
      for (int32_t kb = 0; kb < g.k_blocks; ++kb) {
        double ready = -1.0;
        for (int32_t f : wl[kb]) ready = std::max(ready, (*flag_ready)[(size_t)f]);
        if (!wl[kb].empty() && !sentinel && !consulted) {
          t += lm.tile_wait_ns;
          consulted = true;
        }
        if (ready > t) t = ready + lm.start_ns;  // the pipeline refills after the post
        t += kb_ns + ((!sentinel && !wl[kb].empty()) ? lm.wait_kblock_ns : 0.0);
      }
    }
    double ready = std::max(t, x.last_done);
    if (s == 0 && S > 1 && ks > 0) ready = std::max(ready, unit_done[(size_t)u]);  // the running sum before it
    const double done = ready + lm.epilogue_ns[s];
    if (s == 0 && S > 1) unit_done[(size_t)u] = done;
    x.free_main = t;
    x.last_done = done;
    end = std::max(end, done);
    if (s == 0 && flag_ready && ks == S - 1) {
      const int32_t f = producer_flag(c.dep, m, col);
      if (f >= 0) (*flag_ready)[(size_t)f] = std::max((*flag_ready)[(size_t)f], done + lm.post_ns);
    }
  }
  return end;
}

// Predicted ns of one run of the chain under c.dep.policy (POL_STREAM = stream order).
inline double predict_chain_ns(const ModelChain& c, const LatencyModel& lm) {
  if (c.dep.policy == POL_STREAM) {
    const double e0 = play_queue(c, lm, 0, 0, c.slots[0], 0.0, false, nullptr);
    return play_queue(c, lm, 1, 1, c.slots[1], e0 + lm.gap_ns, false, nullptr);
  }
  const bool sentinel = c.dep.policy == POL_SENTINEL;
  ModelChain cc = c;
  if (sentinel) cc.dep.policy = POL_TILE;  // the sentinel waits on exactly the data of each k-block
  const int64_t nflags = num_flags(cc.dep);
  std::vector<double> ready((size_t)std::max<int64_t>(1, nflags), 0.0);
  const double t0 = sentinel ? c.h_mb * lm.fill_ns_per_mb : 0.0;
  return play_queue(cc, lm, 0, 1, c.slots_fused, t0, sentinel, &ready);
}

// A convolution stack of `stages` dependent convolutions ([cuSync] §II-B "ResNet", Table
// tab:resnet-sizes): stage 0 reads the input, every later stage the stage before it (the
// halo dependency sets of the pair, `dep`); all stages have the same tiles.  Under the
// sentinel policy the intermediates of the next run are filled by fill units at the end of
// the run's queue (units of 64 KB, fill_ns_per_mb each).
struct ModelStack {
  StageGeo geo[2];       // stage 0; every later stage
  DepCfg dep;            // a stage's waits on the stage before it (dep.policy = the policy)
  int32_t stages;
  int32_t slots_fused;   // CTAs of the fused launch
  int32_t slots_stage;   // CTAs of one stage's launch in stream order
  int32_t fill_units;    // sentinel: fill units at the end of the queue
};

inline double predict_stack_ns(const ModelStack& c, const LatencyModel& lm) {
  const int32_t S = c.stages;
  const int64_t n = stage_units(c.geo[0]);
  const bool stream = c.dep.policy == POL_STREAM;
  const bool sentinel = c.dep.policy == POL_SENTINEL;
  DepCfg dep = c.dep;
  if (sentinel) dep.policy = POL_TILE;  // the sentinel waits on exactly the data of each k-block
  ModelChain mc;                        // for the consumer wait lists of stages >= 1
  mc.geo[0] = c.geo[0];
  mc.geo[1] = c.geo[1];
  mc.dep = dep;
  const int64_t nflags = std::max<int64_t>(1, num_flags(dep));
  std::vector<std::vector<double>> posted((size_t)S, std::vector<double>((size_t)nflags, 0.0));
  std::vector<std::vector<int32_t>> wl;
  const double fill_unit_ns = lm.fill_ns_per_mb * (65536.0 / 1e6);
  // one queue: the fused launch (stages 0 .. S-1, then fill units), or one stage of stream order
  auto play = [&](int32_t s0, int32_t s1, int32_t slots, double t0, int32_t fills) -> double {
    const int64_t total = (int64_t)(s1 - s0 + 1) * n + fills;
    std::vector<SimCta> cta((size_t)std::max<int64_t>(1, std::min<int64_t>(slots, total)));
    for (auto& x : cta) x = SimCta{t0, t0, false};
    double end = t0;
    for (int64_t q = 0; q < total; ++q) {
      size_t k = 0;
      if (q < (int64_t)cta.size()) {
        k = (size_t)q;
      } else {
        for (size_t i = 1; i < cta.size(); ++i)
          if (cta[i].free_main < cta[k].free_main) k = i;
      }
      SimCta& x = cta[k];
      double t = x.used ? x.free_main + lm.tile_ns : x.free_main + lm.start_ns;
      x.used = true;
      if (q >= (int64_t)(s1 - s0 + 1) * n) {  // a fill unit: the epilogue warps' stores
        const double done = std::max(t, x.last_done) + fill_unit_ns;
        x.last_done = done;
        end = std::max(end, done);
        continue;
      }
      const int32_t s = s0 + (int32_t)(q / n);
      int32_t m, y;
      tile_at(c.geo[s == 0 ? 0 : 1], (int32_t)(q % n), &m, &y);
      const StageGeo& g = c.geo[s == 0 ? 0 : 1];
      if (s == 0 || stream) {
        t += (double)g.k_blocks * lm.kblock_ns[s == 0 ? 0 : 1];
      } else {
        consumer_wait_lists(mc, m, &wl);
        const double kb_ns = sentinel ? lm.sentinel_kblock_ns : lm.kblock_ns[1];
        bool consulted = false;
        for (int32_t kb = 0; kb < g.k_blocks; ++kb) {
          double ready = -1.0;
          for (int32_t f : wl[kb]) ready = std::max(ready, posted[(size_t)(s - 1)][(size_t)f]);
          if (!wl[kb].empty() && !sentinel && !consulted) {
            t += lm.tile_wait_ns;
            consulted = true;
          }
          if (ready > t) t = ready + lm.start_ns;
          t += kb_ns + ((!sentinel && !wl[kb].empty()) ? lm.wait_kblock_ns : 0.0);
        }
      }
      const double done = std::max(t, x.last_done) + lm.epilogue_ns[s < S - 1 ? 0 : 1];
      x.free_main = t;
      x.last_done = done;
      end = std::max(end, done);
      if (!stream && s < S - 1) {
        const int32_t f = producer_flag(dep, m, y);
        if (f >= 0) posted[(size_t)s][(size_t)f] = std::max(posted[(size_t)s][(size_t)f], done + lm.post_ns);
      }
    }
    return end;
  };
  if (stream) {
    double t = 0.0;
    for (int32_t s = 0; s < S; ++s) t = play(s, s, c.slots_stage, s == 0 ? 0.0 : t + lm.gap_ns, 0);
    return t;
  }
  return play(0, S - 1, c.slots_fused, 0.0, sentinel ? c.fill_units : 0);
}

}  // namespace cusync
