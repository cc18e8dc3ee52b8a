"""The persistent row-ring aggregation kernel (one CTA per SM streaming whole source rows
through a ring of shared-memory slots; used for one head without a seeded partition, n <= 16
sources and rows of 512 to 1024 16-byte vectors) against the fp64 oracle, at token counts that
give every CTA several rows, so that the ring wraps and the per-row partial buffers alternate:
the direct path ("Attention Residuals" note §7) with h, y and alpha under each Table 4 variant,
and phase 1 with one query (the final aggregation: o, m, lse, alpha).  Tolerances:
parity_util.TOL."""
import numpy as np
import pytest
import torch

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B
import oracle.attnres_oracle as O
from parity_util import TOL, check_close, check_outputs, to64
from synth import inputs as I

pytestmark = pytest.mark.gpu

EPS = 1e-6
SIG, NOKN = ar.SIGMOID_WEIGHTS, ar.NO_KEY_NORM

# n, T, d, dtype, flags: T well above the 148 CTAs (several rows each, so the ring wraps);
# d = 7168 at n = 10 is the final aggregation's shape (15 slots); 512-vector rows (bf16 d = 4096,
# fp32 d = 2048) are the shortest the kernel takes, 1024 (bf16 d = 8192, fp32 d = 4096) the
# longest; n = 11 at d = 8192 leaves the ring its minimum of n + 2 slots.  bf16 rows of at most
# 896 vectors over at most 10 sources take the register-held kernel (the first six cases: it
# keeps eight sources in registers and the ninth and tenth in their slots, so n = 10, 9 and
# n <= 8 each take a different path through it), the rest the kernel that keeps a row's slots
# through both passes (n = 16, n = 11, 1024-vector bf16 rows at n = 4, and fp32).
CASES = [(10, 400, 7168, "bf16", 0), (10, 1200, 7168, "bf16", SIG | NOKN),
         (9, 640, 7168, "bf16", NOKN), (1, 300, 4096, "bf16", NOKN), (7, 1000, 6144, "bf16", SIG),
         (2, 777, 4096, "bf16", 0),
         (16, 700, 4096, "bf16", SIG), (3, 2000, 2048, "f32", NOKN),
         (11, 333, 8192, "bf16", SIG | NOKN), (4, 500, 8192, "bf16", 0),
         (5, 1500, 4096, "f32", 0)]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    ar.library()
    return torch.device("cuda:0")


def _dt(name):
    return torch.float32 if name == "f32" else torch.bfloat16


def _queries(d, dev, seed, flags):
    """w, gamma_key (None without the key norm) and the folded query u."""
    W = I.queries(1, d, seed, "w", dev)
    G = None if flags & NOKN else I.gains(1, d, 0.02, seed, "g", dev)
    U = torch.empty_like(W)
    ar.attnres_query_prep(W, G, U)
    return W, G, U


@pytest.mark.parametrize("n,T,d,dt,flags", CASES)
def test_full_path_many_rows_per_cta(dev, n, T, d, dt, flags):
    seed = 7100 + n + T
    dtype = _dt(dt)
    srcs = [I.normal((T, d), 1.0 + 0.05 * j, seed, f"v{j}", dev, dtype) for j in range(n)]
    W, G, U = _queries(d, dev, seed, flags)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    alpha = torch.empty((T, n), device=dev)
    ar.attnres_full_reference_path(srcs, U[0], G_in, h_out=h, y_out=y, alpha_out=alpha,
                                   eps_key=EPS, eps_in=EPS, flags=flags)
    torch.cuda.synchronize()
    ar.attnres_poll_device_errors()
    src64 = np.stack([to64(s) for s in srcs])
    weights = "sigmoid" if flags & SIG else "softmax"
    h_o, a_o, _ = O.aggregate_variant(src64, to64(W[0]), None if G is None else to64(G[0]), EPS,
                                      weights, not flags & NOKN)
    check_outputs(h, h_o, dt, "h")
    check_outputs(y, O.rmsnorm(h_o, to64(G_in), EPS), dt, "y")
    check_close(alpha, a_o.T, TOL[dt]["weight"], "alpha")


@pytest.mark.parametrize("n,T,d,dt,flags", CASES)
def test_final_aggregation_many_rows_per_cta(dev, n, T, d, dt, flags):
    """Phase 1 with one query over a [n, T, d] block-representation cache (the final
    aggregation): o = h, m, lse (softmax weights only) and alpha for every row."""
    seed = 7300 + n + T
    dtype = _dt(dt)
    reps = torch.empty((n, T, d), dtype=dtype, device=dev)
    for j in range(n):
        I.fill_block_rep(reps[j], j, seed)
    W, G, U = _queries(d, dev, seed, flags)
    o = torch.empty((1, T, d), dtype=dtype, device=dev)
    m = torch.empty((1, T), device=dev)
    lse = torch.full((1, T), 5.0, device=dev)
    alpha = torch.empty((1, T, n), device=dev)
    ar.attnres_phase1(reps, U, o, m, lse, alpha, eps=EPS, flags=flags)
    torch.cuda.synchronize()
    ar.attnres_poll_device_errors()
    weights = "sigmoid" if flags & SIG else "softmax"
    oo, om, olse, oa = O.phase1_variant(to64(reps), to64(W), None if G is None else to64(G), EPS,
                                        weights, not flags & NOKN)
    check_outputs(o, oo, dt, "o")
    check_close(m, om, TOL[dt]["stat"], "m")
    check_close(alpha, oa, TOL[dt]["weight"], "alpha")
    if flags & SIG:
        assert torch.all(lse == 5.0), "lse is not written with sigmoid weights"
    else:
        check_close(lse, olse, TOL[dt]["stat"], "lse")
