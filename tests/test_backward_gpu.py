"""Backward of one sublayer's aggregation on the GPU (attnres_backward) against the fp64
oracle's chain rule (oracle.aggregate_backward, itself pinned to finite differences):
dL/dv_i element by element, and the token sums dL/du and dL/dgamma_in.

Tolerances are the method's: fp32 I/O 1e-5 x RMS, bf16 I/O 1e-2 x RMS (+ one bf16 ulp for the
bf16-stored source gradients).  The token sums are fp32 in both modes and are compared with
the fp32 bound in fp32 mode and the bf16 bound in bf16 mode."""
import numpy as np
import pytest
import torch

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B
import oracle.attnres_oracle as O
from parity_util import check_outputs, to64
from synth import inputs as I

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    ar.library()
    return torch.device("cuda:0")


def _rel_check(got, want, rel, what):
    g, w = to64(got), to64(want)
    rms = float(np.sqrt(np.mean(w * w)))
    err = float(np.max(np.abs(g - w)))
    assert np.all(np.isfinite(g)), what
    assert err <= rel * rms, f"{what}: max |err| = {err:.3e} > {rel:.0e} x RMS {rms:.3e}"


@pytest.mark.parametrize("n,T,d,dt", [(3, 24, 128, "f32"), (1, 5, 64, "f32"),
                                      (10, 37, 7168, "bf16"), (16, 20, 2048, "bf16"),
                                      (9, 300, 1024, "bf16"),
                                      (10, 700, 7168, "bf16"),   # several rows per CTA
                                      (1, 9, 4096, "bf16"), (13, 160, 6144, "bf16"),
                                      (4, 45, 4096, "f32")])     # 1024 vectors of fp32
def test_backward_matches_oracle(dev, n, T, d, dt):
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    seed = 8000 + n + d
    srcs = [I.normal((T, d), 1.0 + 0.1 * j, seed, f"v{j}", dev, dtype) for j in range(n)]
    W = I.queries(1, d, seed, "w", dev) * 3.0      # logits of order 1-3: non-uniform weights
    Gk = I.gains(1, d, 0.05, seed, "gk", dev)
    Gi = I.gains(1, d, 0.05, seed, "gi", dev)[0]
    U = torch.empty_like(W)
    ar.attnres_query_prep(W, Gk, U)
    gy = I.normal((T, d), 1.0, seed, "gy", dev, dtype)
    dsrcs = [torch.empty_like(s) for s in srcs]
    du = torch.zeros((d,), device=dev)
    dgi = torch.zeros((d,), device=dev)
    ar.attnres_backward(srcs, U[0], Gi, gy, dsrcs, du, dgi, eps_key=EPS, eps_in=EPS)
    torch.cuda.synchronize()
    G = O.aggregate_backward(np.stack([to64(s) for s in srcs]), to64(W[0]), to64(Gk[0]), EPS,
                             to64(Gi), EPS, to64(gy))
    for j in range(n):
        check_outputs(dsrcs[j], G.dsources[j], dt, f"dL/dv_{j}")
    rel = 1e-5 if dt == "f32" else 1e-2
    _rel_check(du, G.du, rel, "dL/du")
    _rel_check(dgi, G.dgamma_in, rel, "dL/dgamma_in")
    # the parameter gradients follow from du elementwise
    _rel_check(to64(Gk[0]) * to64(du), G.dw, rel, "dL/dw = gamma_key * du")


def test_backward_accumulates(dev):
    """du and dgamma_in are added to what the accumulators hold."""
    T, d, n = 16, 256, 4
    srcs = [I.normal((T, d), 1.0, 9, f"v{j}", dev, torch.float32) for j in range(n)]
    U = I.queries(1, d, 9, "w", dev)[0].contiguous()
    gy = I.normal((T, d), 1.0, 9, "gy", dev, torch.float32)
    dsrcs = [torch.empty_like(s) for s in srcs]
    du1 = torch.zeros((d,), device=dev)
    ar.attnres_backward(srcs, U, None, gy, dsrcs, du1)
    du2 = torch.full((d,), 0.5, device=dev)
    ar.attnres_backward(srcs, U, None, gy, dsrcs, du2)
    torch.cuda.synchronize()
    _rel_check(du2 - 0.5, du1, 1e-6, "accumulated")
