"""The Table 4 ablation variants ("Attention Residuals" note, result 4) on the GPU, through the
C ABI, against the fp64 oracle: sigmoid source weights, no key RMSNorm, and both together, in
phase 1 (both kernels), phase 2, the direct path and a whole block walk.  Tolerances:
parity_util.TOL (weights compared with the weight tolerance although they no longer sum to 1).

Without the key RMSNorm the key-norm gain goes with the norm, so the queries are folded with no
gain (the oracle gets gamma_key = None)."""
import numpy as np
import pytest
import torch

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B
from depth_wise_softmax_block_b300.schedule import BlockRunner, final_aggregation
import oracle.attnres_oracle as O
from parity_util import TOL, check_close, check_outputs, to64
from synth import inputs as I
from walk_util import partial_sources

pytestmark = pytest.mark.gpu
EPS = 1e-6
SIG, NOKN = ar.SIGMOID_WEIGHTS, ar.NO_KEY_NORM
VARIANTS = {"sigmoid": SIG, "no_key_norm": NOKN, "sigmoid_no_key_norm": SIG | NOKN}


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    ar.library()
    return torch.device("cuda:0")


def _dt(name):
    return torch.float32 if name == "f32" else torch.bfloat16


def _weights(flags):
    return "sigmoid" if flags & SIG else "softmax"


def _kn(flags):
    return not (flags & NOKN)


def make_reps(n, T, d, dtype, dev, seed):
    reps = torch.empty((n, T, d), dtype=dtype, device=dev)
    for j in range(n):
        I.fill_block_rep(reps[j], j, seed)
    return reps


def queries(S, d, dev, seed, flags):
    """W, G (None without the key norm), folded U and its bf16 split."""
    W = I.queries(S, d, seed, "w", dev)
    G = I.gains(S, d, 0.02, seed, "g", dev) if _kn(flags) else None
    U = torch.empty_like(W)
    us = torch.empty((2 * S, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, G, U, us)
    return W, G, U, us


def _g64(G, s=None):
    if G is None:
        return None
    return to64(G if s is None else G[s])


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("path", ["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("n,S,T,d,dt", [(9, 24, 37, 512, "bf16"), (4, 18, 21, 7168, "bf16"),
                                        (3, 5, 20, 128, "f32")])
def test_phase1_variant(dev, variant, path, n, S, T, d, dt):
    flags = VARIANTS[variant]
    seed = 4000 + n + S
    reps = make_reps(n, T, d, _dt(dt), dev, seed)
    W, G, U, us = queries(S, d, dev, seed, flags)
    o = torch.empty((S, T, d), dtype=reps.dtype, device=dev)
    m = torch.empty((S, T), device=dev)
    lse = torch.full((S, T), 7.0, device=dev)
    alpha = torch.empty((S, T, n), device=dev)
    ar.attnres_phase1(reps, U, o, m, lse, alpha, eps=EPS,
                      u_split=us if path == "tensor_cores" else None, flags=flags)
    torch.cuda.synchronize()
    oo, om, olse, oa = O.phase1_variant(to64(reps), to64(W), _g64(G), EPS, _weights(flags),
                                        _kn(flags))
    tol = TOL[dt]
    check_outputs(o, oo, dt, f"o ({variant}, {path})")
    check_close(m, om, tol["stat"], "m")
    check_close(alpha, oa, tol["weight"], "alpha")
    if flags & SIG:
        assert torch.all(lse == 7.0), "lse is not written with sigmoid weights"
    else:
        check_close(lse, olse, tol["stat"], "lse")


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("mode", ["first", "partial_only", "fused"])
@pytest.mark.parametrize("n,T,d,dt,ostore", [(9, 33, 7168, "bf16", "io"), (2, 40, 128, "f32", "io"),
                                              (9, 33, 7168, "bf16", "f32")])
def test_phase2_variant(dev, variant, mode, n, T, d, dt, ostore):
    flags = VARIANTS[variant]
    seed = 5000 + n + d
    dtype = _dt(dt)
    reps = make_reps(n, T, d, dtype, dev, seed)
    W, G, U, us = queries(1, d, dev, seed, flags)
    o = torch.empty((1, T, d), dtype=torch.float32 if ostore == "f32" else dtype, device=dev)
    lse = torch.empty((1, T), device=dev)
    ar.attnres_phase1(reps, U, o, lse_out=lse, eps=EPS, flags=flags)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    part = I.normal((T, d), 1.5, seed, "part", dev, dtype)
    vprev = I.normal((T, d), 1.0, seed, "vprev", dev, dtype)
    partial = part if mode in ("partial_only", "fused") else None
    v_prev = vprev if mode == "fused" else None
    pout = torch.empty_like(part) if mode == "fused" else None
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    ap = torch.empty((T,), device=dev)
    has_p = partial is not None
    ar.attnres_phase2_merge(o[0], None if flags & SIG else lse[0], partial, v_prev, pout, U[0],
                            G_in, y, h_out=h, alpha_p_out=ap if has_p else None, eps_key=EPS,
                            eps_in=EPS, flags=flags)
    torch.cuda.synchronize()
    p_exact = None
    if has_p:
        p_exact = to64(part) + (to64(vprev) if v_prev is not None else 0.0)
    h_m, y_m, a_m = O.merge_reference_variant(
        to64(o[0]), None if flags & SIG else to64(lse[0]), p_exact, to64(W[0]), _g64(G, 0), EPS,
        to64(G_in), EPS, _weights(flags), _kn(flags))
    check_outputs(h, h_m, dt, f"h ({variant}, {mode}, per call)")
    check_outputs(y, y_m, dt, f"y ({variant}, {mode}, per call)")
    if has_p:
        check_close(ap, a_m, TOL[dt]["weight"], "weight of the partial source")
    # end to end where the stored phase-1 output is fp32 (fp32 I/O, or ATTNRES_O_F32)
    if dt == "f32" or ostore == "f32":
        srcs = to64(reps) if p_exact is None else np.concatenate([to64(reps), p_exact[None]])
        h_d, a_d, _ = O.aggregate_variant(srcs, to64(W[0]), _g64(G, 0), EPS, _weights(flags),
                                          _kn(flags))
        check_outputs(h, h_d, dt, "h (two-phase vs direct)")
        check_outputs(y, O.rmsnorm(h_d, to64(G_in), EPS), dt, "y (two-phase vs direct)")
        if has_p:
            check_close(ap, a_d[-1], TOL[dt]["weight"], "weight of the partial (vs direct)")


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("n,T,d,dt", [(12, 40, 2048, "bf16"), (3, 64, 128, "f32")])
def test_full_path_variant(dev, variant, n, T, d, dt):
    flags = VARIANTS[variant]
    seed = 6000 + n
    dtype = _dt(dt)
    srcs = [I.normal((T, d), 1.0 + 0.05 * j, seed, f"v{j}", dev, dtype) for j in range(n)]
    W, G, U, _ = queries(1, d, dev, seed, flags)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    alpha = torch.empty((T, n), device=dev)
    ar.attnres_full_reference_path(srcs, U[0], G_in, h_out=h, y_out=y, alpha_out=alpha,
                                   eps_key=EPS, eps_in=EPS, flags=flags)
    torch.cuda.synchronize()
    src64 = np.stack([to64(s) for s in srcs])
    h_o, a_o, _ = O.aggregate_variant(src64, to64(W[0]), _g64(G, 0), EPS, _weights(flags),
                                      _kn(flags))
    check_outputs(h, h_o, dt, f"h ({variant})")
    check_outputs(y, O.rmsnorm(h_o, to64(G_in), EPS), dt, f"y ({variant})")
    check_close(alpha, a_o.T, TOL[dt]["weight"], "alpha")


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("dt,T,d,path", [("f32", 24, 128, "cuda_cores"),
                                         ("bf16", 40, 1024, "tensor_cores")])
def test_block_walk_variant(dev, variant, dt, T, d, path):
    """One block of S = 4 sublayers over n = 3 given sources through BlockRunner (phase 1,
    phase 2 with the fused partial update, the close) and the final aggregation, every
    element against the oracle's direct definition over the partial sums as the GPU stores
    them; phase 1's o is stored in fp32 (ATTNRES_O_F32), so no rounding sits between the
    phases."""
    flags = VARIANTS[variant]
    seed, n, S = 7000, 3, 4
    dtype = _dt(dt)
    reps = make_reps(n, T, d, dtype, dev, seed)
    W, G, U, us = queries(S, d, dev, seed, flags)
    G_in = I.gains(S, d, 0.05, seed, "gin", dev)
    v = torch.stack([I.normal((T, d), 1.0, seed, f"out{i}", dev, dtype) for i in range(S)])
    runner = BlockRunner(T, d, S, dtype, dev, keep_y=True, o_dtype=torch.float32)
    ys = torch.empty((S, T, d), dtype=dtype, device=dev)
    close = torch.empty((T, d), dtype=dtype, device=dev)

    def sub(i, y):
        ys[i - 1].copy_(y)
        return v[i - 1]

    runner.run_block(reps, U, G_in, sub, close, EPS, EPS,
                     U_split=us if path == "tensor_cores" else None, flags=flags)
    wf, gf = W[0], None if G is None else G[0]
    fin = torch.empty((T, d), dtype=dtype, device=dev)
    final_aggregation(torch.cat([reps, close[None]]), U[0], fin, EPS, flags=flags)
    torch.cuda.synchronize()
    # the GPU rounds the partial sums to the I/O type between sublayers; feed the oracle the
    # same rounded partials so the comparison is per call, not a drift measurement
    ps, close_want = partial_sources(v, dtype)
    r64 = to64(reps)
    for i in range(1, S + 1):
        srcs = r64 if ps[i - 1] is None else np.concatenate([r64, ps[i - 1][None]])
        h_o, _, _ = O.aggregate_variant(srcs, to64(W[i - 1]), _g64(G, i - 1), EPS,
                                        _weights(flags), _kn(flags))
        check_outputs(ys[i - 1], O.rmsnorm(h_o, to64(G_in[i - 1]), EPS), dt,
                      f"y_{i} ({variant})")
    assert torch.equal(close.cpu(), close_want), "closed block"
    fin_o, _, _ = O.aggregate_variant(np.concatenate([to64(reps), to64(close)[None]]), to64(wf),
                                      _g64(gf), EPS, _weights(flags), _kn(flags))
    check_outputs(fin, fin_o, dt, f"final ({variant})")
