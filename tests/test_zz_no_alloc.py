"""GPU test of cusync_run_mlp_noalloc, the entry point for callers that cannot allocate
device memory themselves (for example an operator inside a runtime that owns the device
memory pool).  It keeps the chain's synchronisation state in a fixed array inside the
library instead of memory from cusync_create_chain.  Two calls in a row, through the C
ABI, must give the same H and Y as the regular entry point cusync_run_mlp, within the
tolerance of the parity tests.  This file is named to be collected last."""

import pytest
import torch

import tile_level_sync_gb300 as cs
from tile_level_sync_gb300 import synth

from gpu_helpers import device_mlp_operands, f64, run_mlp, within_tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy,launch", [("ROW", cs.LAUNCH_PERSISTENT), ("TILE", cs.LAUNCH_PDL),
                                           ("SENTINEL", cs.LAUNCH_PERSISTENT)])
def test_noalloc_matches_regular_entry_point_twice(policy, launch):
    M, K, N1, N2 = 200, 384, 640, 264
    X, W1, W2 = synth.mlp_gelu_inputs(M, K, N1, N2, seed=7)
    ops = device_mlp_operands(X, W1, W2)
    d = cs.make_desc(cs.CHAIN_MLP_GELU, policy, launch, M=M, K=K, N1=N1, N2=N2, tile_n=256)
    H_ref, Y_ref, _ = run_mlp(d, *ops)          # regular entry point, chain-owned state
    for call in range(2):
        H = torch.full((M, N1), float("nan"), dtype=torch.bfloat16, device="cuda")
        Y = torch.full((M, N2), float("nan"), dtype=torch.bfloat16, device="cuda")
        st, err = cs.cusync_run_mlp_noalloc(d, *ops, H, Y, wait=True)
        assert st == cs.OK and err == 0, (call, st, hex(err))
        ok_h, worst_h = within_tol(f64(H.cpu()), f64(H_ref))
        ok_y, worst_y = within_tol(f64(Y.cpu()), f64(Y_ref))
        assert ok_h and ok_y, (call, worst_h, worst_y)


def test_noalloc_rejects_plans_beyond_the_fixed_scratch():
    # 16384 single-CTA row tiles of RowSync semaphores do not fit the 16368 the array holds
    d = cs.make_desc(cs.CHAIN_MLP_GELU, "ROW", M=128 * 16384, K=64, N1=64, N2=64, cta_pair=1)
    lib = cs.load()
    import ctypes
    st = lib.cusync_run_mlp_noalloc(ctypes.byref(d), None, None, None, None, None, None, None)
    assert st == cs.ERR_UNSUPPORTED
