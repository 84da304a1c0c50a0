"""GPU test of cusync_run_mlp_noalloc, the entry point for callers that cannot allocate
device memory themselves (for example an operator inside a runtime that owns the device
memory pool, or a serving loop that must not pay cudaMalloc's synchronisation).  It keeps
the chain's synchronisation state in a fixed array inside the library instead of memory
from cusync_create_chain.

Two calls in a row, through the C ABI, must write exactly the bytes the regular entry
point cusync_run_mlp writes for the same descriptor (the same kernel and plan: no K split
on either path), and those bytes must match the oracle within the parity tests'
tolerance.  Cases: single CTAs at both tile widths (a 64-token chain among them), CTA
pairs, and the SwiGLU chain.  This file is named to be collected last."""

import ctypes

import pytest
import torch

import tile_level_sync_gb300 as cs
from oracle import chains
from tile_level_sync_gb300 import synth

from gpu_helpers import assert_within_tol, bits, device_mlp_operands, f64, run_mlp

pytestmark = pytest.mark.gpu

CASES = [
    # kind, policy, launch, M, K, N1, N2, tile_n, cta_pair
    ("gelu", "ROW", cs.LAUNCH_PERSISTENT, 200, 384, 640, 264, 256, 1),
    ("gelu", "TILE", cs.LAUNCH_PDL, 200, 384, 640, 264, 256, 1),
    ("gelu", "SENTINEL", cs.LAUNCH_PERSISTENT, 200, 384, 640, 264, 256, 1),
    ("gelu", "ROW", cs.LAUNCH_PERSISTENT, 64, 256, 1024, 256, 128, 1),
    ("gelu", "STRIDED", cs.LAUNCH_PERSISTENT, 520, 512, 1536, 512, 256, 2),
    ("gelu", "SENTINEL", cs.LAUNCH_PDL, 520, 512, 1536, 512, 256, 2),
    ("swiglu", "ROW", cs.LAUNCH_PERSISTENT, 200, 512, 384, 264, 256, 1),
    ("swiglu", "TILE", cs.LAUNCH_PERSISTENT, 264, 512, 512, 256, 256, 2),
]


@pytest.mark.parametrize("kind,policy,launch,M,K,N1,N2,tile_n,pair", CASES)
def test_noalloc_matches_regular_entry_point_twice(kind, policy, launch, M, K, N1, N2, tile_n, pair):
    if kind == "gelu":
        X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=7)
        H_ref, Y_ref = chains.mlp_gelu(f64(X), f64(W1), f64(W2))
        ops = device_mlp_operands(X, W1, W2)
        ck = cs.CHAIN_MLP_GELU
    else:
        X, Wg, Wu, Wd = synth.mlp_swiglu_inputs(M, K, N1, N2, seed=7)
        H_ref, Y_ref = chains.mlp_swiglu(f64(X), f64(Wg), f64(Wu), f64(Wd))
        ops = device_mlp_operands(X, Wg, Wd, Wup=Wu)
        ck = cs.CHAIN_MLP_SWIGLU
    # no K split on either path: the allocation-free one has no workspace for partial sums
    d = cs.make_desc(ck, policy, launch, M=M, K=K, N1=N1, N2=N2, tile_n=tile_n, cta_pair=pair, ksplit=1,
                     ksplit_consumer=1)
    H_reg, Y_reg, _ = run_mlp(d, *ops)          # regular entry point, chain-owned state
    for call in range(2):
        H = torch.full((M, N1), float("nan"), dtype=torch.bfloat16, device="cuda")
        Y = torch.full((M, N2), float("nan"), dtype=torch.bfloat16, device="cuda")
        st, err = cs.cusync_run_mlp_noalloc(d, *ops, H, Y, wait=True)
        assert st == cs.OK and err == 0, (call, st, hex(err))
        Hc, Yc = H.cpu(), Y.cpu()
        assert (bits(Hc) == bits(H_reg)).all(), f"call {call}: H differs from cusync_run_mlp"
        assert (bits(Yc) == bits(Y_reg)).all(), f"call {call}: Y differs from cusync_run_mlp"
        assert_within_tol(f64(Hc), H_ref, f"H call {call}")
        assert_within_tol(f64(Yc), Y_ref, f"Y call {call}")


def test_noalloc_rejects_plans_beyond_the_fixed_scratch():
    # one more single-CTA RowSync row tile than the array holds semaphores for
    tiles = cs.NOALLOC_MAX_SEMAPHORES + 1
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=128 * tiles, K=64, N1=64, N2=64, cta_pair=1, tile_n=128)
    st = cs.load().cusync_run_mlp_noalloc(ctypes.byref(d), None, None, None, None, None, None, None)
    assert st == cs.ERR_UNSUPPORTED
