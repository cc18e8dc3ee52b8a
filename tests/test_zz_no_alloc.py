"""attnres_backward_block_noalloc, for callers that cannot allocate device memory while they run
the block backward (a framework whose allocator owns every device byte, or a latency-critical
path that cannot take cudaMalloc's synchronisation): the same block backward with its scratch in
the library's own fixed device array.

Called through the C ABI twice in a row, with different upstream gradients, and compared after
each call with attnres_backward_block on a caller-provided workspace: the source and output
gradients bit for bit (same kernels, same inputs), the token sums (atomics) within 1e-5 of their
RMS.  The second call also shows that what the first one left in the shared array does no harm.
A block whose scratch would not fit is refused before anything runs.

This file is collected last, so that a run that stops at its first failure has run every other
test before it; it passes on its own in a fresh process as well."""
import numpy as np
import pytest
import torch

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B
from parity_util import to64
from synth import inputs as I

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    ar.library()
    return torch.device("cuda:0")


def _close_sum(got, want, what):
    g, w = to64(got), to64(want)
    scale = max(float(np.sqrt(np.mean(w * w))), 1.0)
    err = float(np.max(np.abs(g - w)))
    assert err <= 1e-5 * scale, f"{what}: max |err| = {err:.3e} > 1e-5 x {scale:.3e}"


@pytest.mark.parametrize("n,S,T,d,dt", [(9, 24, 37, 7168, "bf16"), (3, 4, 21, 256, "f32")])
def test_noalloc_matches_workspace_version_twice(dev, n, S, T, d, dt):
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    seed = 31337 + n
    assert ar.attnres_backward_block_workspace_size(n, S, T, d, dtype) <= (64 << 20)
    reps = torch.empty((n, T, d), dtype=dtype, device=dev)
    for j in range(n):
        I.fill_block_rep(reps[j], j, seed)
    v = torch.stack([I.normal((T, d), 1.0, seed, f"v{k}", dev, dtype) for k in range(S - 1)])
    W = I.queries(S, d, seed, "w", dev) * 3.0
    Gk = I.gains(S, d, 0.05, seed, "gk", dev)
    Gi = I.gains(S, d, 0.05, seed, "gi", dev)
    U = torch.empty_like(W)
    Us = torch.empty((2 * S, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, Gk, U, Us)
    us = Us if dt == "bf16" else None
    for call in range(2):
        gy = torch.stack([I.normal((T, d), 1.0 + call, seed, f"gy{call}/{i}", dev, dtype)
                          for i in range(S)])
        outs = []
        for fn in (ar.attnres_backward_block, ar.attnres_backward_block_noalloc):
            d_reps = torch.empty((n, T, d), dtype=dtype, device=dev)
            d_v = torch.empty((S - 1, T, d), dtype=dtype, device=dev)
            du = torch.zeros((S, d), device=dev)
            dgi = torch.zeros((S, d), device=dev)
            fn(reps, v, U, Gi, gy, d_reps, d_v, du, dgi, u_split=us, eps_key=EPS, eps_in=EPS)
            outs.append((d_reps, d_v, du, dgi))
        torch.cuda.synchronize()
        (r1, v1, u1, g1), (r2, v2, u2, g2) = outs
        assert torch.equal(r1, r2), f"call {call}: dL/db differs"
        assert torch.equal(v1, v2), f"call {call}: dL/dv differs"
        _close_sum(u2, u1, f"call {call}: dL/du")
        _close_sum(g2, g1, f"call {call}: dL/dgamma_in")
    ar.attnres_poll_device_errors()


def test_noalloc_refuses_a_block_beyond_its_scratch(dev):
    """A block whose scratch exceeds the fixed array is refused (ATTNRES_ERR_UNSUPPORTED) before
    anything runs; the same block runs through the workspace entry point."""
    n, S, T, d = 9, 24, 256, 7168
    assert ar.attnres_backward_block_workspace_size(n, S, T, d, torch.bfloat16) > (64 << 20)
    reps = torch.zeros((n, T, d), dtype=torch.bfloat16, device=dev)
    v = torch.zeros((S - 1, T, d), dtype=torch.bfloat16, device=dev)
    U = torch.zeros((S, d), device=dev)
    gy = torch.zeros((S, T, d), dtype=torch.bfloat16, device=dev)
    d_reps = torch.empty_like(reps)
    d_v = torch.empty_like(v)
    du = torch.zeros((S, d), device=dev)
    with pytest.raises(ar.AttnResError, match="ATTNRES_ERR_UNSUPPORTED"):
        ar.attnres_backward_block_noalloc(reps, v, U, None, gy, d_reps, d_v, du)
