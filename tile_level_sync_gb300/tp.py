"""Tensor-parallel MLP shard with the reduction of its output overlapped band by band.

The pages' MLP block is one shard of a tensor-parallel layer ("A Framework for
Fine-Grained Synchronization of Dependent GPU Kernels", §II-B "GPT-3": with 8-way tensor
parallelism each GPU holds H/8 columns of the first weight and H/8 rows of the second,
Fig. fig:gpt-3:mlp), whose outputs are summed across the GPUs; the pages name overlapping
that communication with the computation as their next step ("Conclusion").

Rank r of W ranks holds columns [r*N1/W, (r+1)*N1/W) of W1 (for SwiGLU: of both the gate
and the up projection) and the same rows of W2, computes its partial Y_r with the chain,
and the all-reduce (sum) of the Y_r over the ranks is the layer's output.  The chain's
consumer tiles post one semaphore per row band of Y; this module only orders host calls:
for each band it enqueues the library's wait on that band and then the band's reduction on
a side stream, so the reduction of early bands overlaps the computation of later ones.
The arithmetic runs in the library's kernels and in the collective library.
"""

import tile_level_sync_gb300 as cs


def shard_range(n, rank, world):
    """[lo, hi) of the rank's share of n columns (n divisible by world)."""
    if n % world:
        raise ValueError(f"{n} columns do not split evenly over {world} ranks")
    step = n // world
    return rank * step, (rank + 1) * step


def shard_mlp_weights(W1t, W2t, rank, world, swiglu=False):
    """The rank's weights in the library's layout: W1t [N1, K] (SwiGLU: [Wgate^T; Wup^T],
    [2*N1, K]) keeps the rows of its columns of H, W2t [N2, N1] the same columns."""
    n1 = W2t.shape[1]
    lo, hi = shard_range(n1, rank, world)
    if swiglu:
        w1 = W1t[lo:hi], W1t[n1 + lo:n1 + hi]
        w1s = w1[0].new_empty((2 * (hi - lo), W1t.shape[1]))
        w1s[:hi - lo] = w1[0]
        w1s[hi - lo:] = w1[1]
    else:
        w1s = W1t[lo:hi].contiguous()
    return w1s, W2t[:, lo:hi].contiguous()


def band_slices(desc):
    """(row0, rows) of each row band of the chain's output."""
    return [cs.cusync_band_rows(desc, b) for b in range(desc.bands)]


def reduce_bands(Y, slices, wait_band, reduce):
    """For each band in order: wait_band(b), then reduce(rows of Y in band b)."""
    for b, (r0, n) in enumerate(slices):
        wait_band(b)
        reduce(Y[r0:r0 + n])


class TensorParallelMLP:
    """One rank's shard of a tensor-parallel MLP: the chain on this rank's weights, then the
    all-reduce of Y over `group` (torch.distributed), one band at a time on a side stream
    as each band of Y is complete."""

    def __init__(self, desc, group=None):
        import torch
        if desc.bands < 1:
            raise ValueError("desc.bands must be at least 1")
        self.desc = desc
        self.group = group
        self.chain = cs.Chain(desc)
        self.side = torch.cuda.Stream()
        self.slices = band_slices(desc)

    def run(self, X, W1t, W2t, H, Y, reduce=None):
        """Enqueue one run and its band reductions; the current stream waits for the
        reductions at the end, so Y holds the summed output in stream order."""
        import torch
        import torch.distributed as dist
        cur = torch.cuda.current_stream()
        if reduce is None:
            def reduce(t):
                dist.all_reduce(t, group=self.group)
        cs.cusync_run_mlp_bands(self.chain.handle, X, W1t, W2t, H, Y, self.side, cur)
        with torch.cuda.stream(self.side):
            reduce_bands(Y, self.slices, lambda b: cs.cusync_band_wait(self.chain.handle, b, self.side), reduce)
        cur.wait_stream(self.side)

    def check(self):
        return self.chain.check()

    def close(self):
        self.chain.close()
