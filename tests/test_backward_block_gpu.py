"""Backward of one whole block (attnres_backward_block) on the GPU against the fp64 oracle's
chain rule composed over the block (oracle.block_backward, pinned to finite differences):
dL/db_j of the completed sources and dL/dv_k of the sublayer outputs element by element, and
the token sums dL/du_i and dL/dgamma_in,i of every sublayer.

Tolerances are the method's: fp32 I/O 1e-5 x RMS; bf16 I/O the bf16 output gate (within
max(1e-2 x RMS, one bf16 step) of the rounded oracle) for the stored gradients and 1e-2 x RMS
for the fp32 token sums."""
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


def _rel_check(got, want, rel, what, floor=1.0):
    """max |err| <= rel * max(RMS(want), floor): the floor (an absolute scale of the token
    sums) covers the degenerate block of one sublayer over one source, whose query gradient is
    exactly zero (a single source always has weight 1) and is met by fp32 rounding noise."""
    g, w = to64(got), to64(want)
    rms = float(np.sqrt(np.mean(w * w)))
    err = float(np.max(np.abs(g - w)))
    assert np.all(np.isfinite(g)), what
    scale = max(rms, floor)
    assert err <= rel * scale, f"{what}: max |err| = {err:.3e} > {rel:.0e} x {scale:.3e}"
    return err / scale


def _block_case(dev, n, S, T, d, dt, seed, qscale=3.0, split=True, stride_pad=0):
    dtype = torch.float32 if dt == "f32" else torch.bfloat16
    reps_all = torch.empty((n, T + stride_pad, d), dtype=dtype, device=dev)
    for j in range(n):
        I.fill_block_rep(reps_all[j], j, seed)
    reps = reps_all[:, :T]                                    # source stride (T + pad) d
    v = torch.stack([I.normal((T, d), 1.0, seed, f"v{k}", dev, dtype) for k in range(S)])
    W = I.queries(S, d, seed, "w", dev) * qscale              # logits of order 1-3
    Gk = I.gains(S, d, 0.05, seed, "gk", dev)
    Gi = I.gains(S, d, 0.05, seed, "gi", dev)
    U = torch.empty_like(W)
    Us = torch.empty((2 * S, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, Gk, U, Us)
    gy = torch.stack([I.normal((T, d), 1.0, seed, f"gy{i}", dev, dtype) for i in range(S)])
    d_reps = torch.empty((n, T, d), dtype=dtype, device=dev)
    d_v = torch.empty((max(S - 1, 1), T, d), dtype=dtype, device=dev)
    du = torch.zeros((S, d), device=dev)
    dgi = torch.zeros((S, d), device=dev)
    ar.attnres_backward_block(reps, v[:S - 1] if S > 1 else None, U, Gi, gy, d_reps,
                              d_v if S > 1 else None, du, dgi,
                              u_split=Us if (split and dt == "bf16") else None, eps_key=EPS,
                              eps_in=EPS)
    torch.cuda.synchronize()
    ar.attnres_poll_device_errors()
    G = O.block_backward(to64(reps), to64(v), to64(W), to64(Gk), to64(Gi), EPS, EPS, to64(gy))
    return d_reps, d_v, du, dgi, G, Gk


CASES = [
    # n, S, T, d, dtype
    (2, 3, 17, 128, "f32"),
    (3, 4, 24, 256, "f32"),
    (1, 1, 9, 64, "f32"),           # one sublayer: no partial source, no v
    (4, 2, 5, 96, "f32"),           # two sublayers, d not a multiple of 128
    (9, 24, 37, 7168, "bf16"),      # the long-context block shape, ragged T
    (4, 5, 50, 1024, "bf16"),
    (16, 2, 13, 512, "bf16"),       # n at its maximum
    (9, 18, 21, 2048, "bf16"),      # a tail block (S = 18)
    (1, 24, 8, 256, "bf16"),        # one completed source (the first block)
]


@pytest.mark.parametrize("n,S,T,d,dt", CASES)
def test_backward_block_matches_oracle(dev, n, S, T, d, dt):
    d_reps, d_v, du, dgi, G, Gk = _block_case(dev, n, S, T, d, dt, 9000 + n * 31 + S)
    for j in range(n):
        check_outputs(d_reps[j], G.dcompleted[j], dt, f"dL/db_{j}")
    for k in range(S - 1):
        check_outputs(d_v[k], G.dv[k], dt, f"dL/dv_{k + 1}")
    rel = 1e-5 if dt == "f32" else 1e-2
    _rel_check(du, G.du, rel, "dL/du")
    _rel_check(dgi, G.dgamma_in, rel, "dL/dgamma_in")
    _rel_check(to64(Gk) * to64(du), G.dw, rel, "dL/dw = gamma_key * du")


def test_backward_block_cuda_cores_and_source_stride(dev):
    """Phase 1 recomputed on the CUDA cores (no split queries), sources with a padded stride."""
    n, S, T, d = 5, 6, 19, 512
    d_reps, d_v, du, dgi, G, Gk = _block_case(dev, n, S, T, d, "bf16", 77, split=False,
                                              stride_pad=7)
    for j in range(n):
        check_outputs(d_reps[j], G.dcompleted[j], "bf16", f"dL/db_{j}")
    for k in range(S - 1):
        check_outputs(d_v[k], G.dv[k], "bf16", f"dL/dv_{k + 1}")
    _rel_check(du, G.du, 1e-2, "dL/du")


def test_backward_block_equals_per_sublayer_backward(dev):
    """The block backward equals the sum of the per-sublayer backward (attnres_backward over
    each sublayer's explicit source list) in fp32: every completed source's gradient is the sum
    over the sublayers, and dL/dv_k the sum of the partial gradients after k."""
    n, S, T, d = 3, 4, 12, 128
    seed = 4242
    reps = torch.stack([I.normal((T, d), 1.0 + 0.3 * j, seed, f"b{j}", dev) for j in range(n)])
    v = torch.stack([I.normal((T, d), 1.0, seed, f"v{k}", dev) for k in range(S)])
    W = I.queries(S, d, seed, "w", dev) * 3.0
    U = W.clone()
    gy = torch.stack([I.normal((T, d), 1.0, seed, f"gy{i}", dev) for i in range(S)])
    d_reps = torch.empty_like(reps)
    d_v = torch.empty((S - 1, T, d), device=dev)
    du = torch.zeros((S, d), device=dev)
    ar.attnres_backward_block(reps, v[:S - 1], U, None, gy, d_reps, d_v, du, eps_key=EPS,
                              eps_in=EPS)
    acc_b = torch.zeros_like(reps)
    acc_p = []
    du2 = torch.zeros((S, d), device=dev)
    for i in range(1, S + 1):
        srcs = [reps[j] for j in range(n)]
        if i >= 2:
            srcs.append(v[:i - 1].sum(dim=0))
        ds = [torch.empty_like(s) for s in srcs]
        ar.attnres_backward(srcs, U[i - 1], None, gy[i - 1], ds, du2[i - 1], eps_key=EPS,
                            eps_in=EPS)
        for j in range(n):
            acc_b[j] += ds[j]
        acc_p.append(ds[n] if i >= 2 else None)
    torch.cuda.synchronize()
    check_outputs(d_reps, to64(acc_b), "f32", "dL/db (block vs per sublayer)")
    for k in range(1, S):
        want = sum(to64(acc_p[i - 1]) for i in range(k + 1, S + 1))
        check_outputs(d_v[k - 1], want, "f32", f"dL/dv_{k} (block vs per sublayer)")
    _rel_check(du, du2, 1e-5, "dL/du (block vs per sublayer)")


def test_backward_block_accumulates_and_repeats(dev):
    """du and dgamma_in are added to what the accumulators hold; the source and output
    gradients of two calls agree bit for bit (only the token sums use atomics)."""
    n, S, T, d = 3, 5, 33, 256
    seed = 515
    reps = torch.stack([I.normal((T, d), 1.0, seed, f"b{j}", dev, torch.bfloat16)
                        for j in range(n)])
    v = torch.stack([I.normal((T, d), 1.0, seed, f"v{k}", dev, torch.bfloat16)
                     for k in range(S - 1)])
    W = I.queries(S, d, seed, "w", dev)
    Us = torch.empty((2 * S, d), dtype=torch.bfloat16, device=dev)
    U = torch.empty_like(W)
    ar.attnres_query_prep(W, None, U, Us)
    gy = torch.stack([I.normal((T, d), 1.0, seed, f"gy{i}", dev, torch.bfloat16)
                      for i in range(S)])
    outs = []
    for init in (0.0, 0.25):
        d_reps = torch.empty((n, T, d), dtype=torch.bfloat16, device=dev)
        d_v = torch.empty((S - 1, T, d), dtype=torch.bfloat16, device=dev)
        du = torch.full((S, d), init, device=dev)
        dgi = torch.full((S, d), init, device=dev)
        ar.attnres_backward_block(reps, v, U, None, gy, d_reps, d_v, du, dgi, u_split=Us)
        outs.append((d_reps, d_v, du - init, dgi - init))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    _rel_check(outs[1][2], outs[0][2], 1e-5, "du accumulated")
    _rel_check(outs[1][3], outs[0][3], 1e-5, "dgamma_in accumulated")
