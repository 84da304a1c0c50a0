"""CPU oracle for tile-level synchronised GEMM/conv chains.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
its Python binding, ``smoke()``'s launch or ``bench.py``'s timed GPU arm)
imports, links or executes this package.  Only ``tests/``,
``__graft_entry__.smoke()`` (to check its result) and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may call it.

What it computes (all floating point in fp64, numpy):

* ``chains``      -- the three dependent chains the method synchronises:
                     GeLU MLP, SwiGLU MLP and the conv3x3 -> ReLU -> conv3x3
                     pair.  Tile-level synchronisation changes *when* a
                     consumer tile starts, never *what* it computes, so the
                     oracle is the plain definition of each chain.
* ``bf16``        -- round-to-nearest-even fp64 -> bf16 and the sign-of-zero
                     canonicalisation the sentinel protocol requires.
* ``activations`` -- tanh-GeLU, SiLU, ReLU.
* ``planner``     -- thread-block wave arithmetic (waves, utilisation,
                     stream-serialised vs. fused wave counts).
* ``deps``        -- per-consumer-tile data-dependency sets, derived by
                     brute force over the elements each tile reads and
                     writes, and the wait sets each synchronisation policy
                     implies.
* ``sentinel``    -- the expected output of the sentinel-protocol example
                     (double-then-reverse each 1024-element tile).

Pins (tests that tie each function to something other than itself) live in
``tests/test_oracle_*.py``.  Functions without such a pin say
"parity unpinned" in their docstring.

Sources, cited by title and section throughout:

* [cuSync] "A Framework for Fine-Grained Synchronization of Dependent GPU
  Kernels" (Jangda et al., arXiv 2305.13450).
* [CUDA-FGS] CUDA Programming Guide, section 4.6 "Fine-Grained
  Synchronization".
* [ALCOP] "ALCOP: Automatic Load-COmpute Pipelining in Deep Learning
  Compiler for AI-GPUs" (arXiv 2210.16691).
"""

from . import activations, bf16, chains, deps, planner, sentinel  # noqa: F401
