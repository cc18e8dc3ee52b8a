"""Depth-attention heads (the multi-head variant of Table 4, "Attention Residuals" note,
result 4) on the GPU, through the C ABI, against the fp64 oracle's multi-head functions: phase 1
on both kernels (tensor cores: windows of whole heads per CTA; CUDA cores: one head per CTA
column), phase 2, the direct path, the grouped-schedule merge, a whole block walk and the
128K-prefill shape on sampled rows.  Tolerances: parity_util.TOL.

Reading of the pages (they name the variant but give no formula): head k owns the contiguous
features k*dh .. k*dh + dh - 1 (dh = d / H) and is a complete aggregation on them; the input
RMSNorm runs over the whole row."""
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
VARIANTS = {"softmax": 0, "sigmoid": SIG, "no_key_norm": NOKN}


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    ar.library()
    return torch.device("cuda:0")


def _dt(name):
    return torch.float32 if name == "f32" else torch.bfloat16


def _wk(flags):
    return dict(weights="sigmoid" if flags & SIG else "softmax", key_norm=not (flags & NOKN))


def make_reps(n, T, d, dtype, dev, seed):
    reps = torch.empty((n, T, d), dtype=dtype, device=dev)
    for j in range(n):
        I.fill_block_rep(reps[j], j, seed)
    return reps


def queries(S, d, dev, seed, flags=0):
    W = I.queries(S, d, seed, "w", dev)
    G = None if flags & NOKN else I.gains(S, d, 0.02, seed, "g", dev)
    U = torch.empty_like(W)
    us = torch.empty((2 * S, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, G, U, us)
    return W, G, U, us


def _g64(G, s=None):
    if G is None:
        return None
    return to64(G if s is None else G[s])


# (n, S, T, d, H, dtype): tensor-core windows (16 heads x 48 columns do not fit the 512
# tensor-memory columns, so two windows of 8), several M-tiles, heads whose width is not a
# multiple of a stage (CUDA cores, masked chunks), fp32.
P1_CASES = [(9, 24, 37, 1024, 16, "bf16"), (4, 6, 21, 7168, 16, "bf16"),
            (12, 8, 30, 512, 4, "bf16"), (33, 4, 19, 1024, 8, "bf16"),
            (5, 8, 23, 480, 4, "bf16"), (3, 5, 20, 160, 4, "f32"), (2, 3, 9, 128, 16, "f32")]


@pytest.mark.parametrize("path", ["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("n,S,T,d,H,dt", P1_CASES)
def test_phase1_heads(dev, path, n, S, T, d, H, dt):
    seed = 8000 + n + S + H
    reps = make_reps(n, T, d, _dt(dt), dev, seed)
    W, G, U, us = queries(S, d, dev, seed)
    o = torch.empty((S, T, d), dtype=reps.dtype, device=dev)
    m = torch.empty((S, H, T), device=dev)
    lse = torch.empty((S, H, T), device=dev)
    alpha = torch.empty((S, H, T, n), device=dev)
    ar.attnres_phase1(reps, U, o, m, lse, alpha, eps=EPS,
                      u_split=us if path == "tensor_cores" else None, heads=H)
    torch.cuda.synchronize()
    oo, om, olse, oa = O.multihead_phase1(to64(reps), to64(W), to64(G), EPS, H)
    tol = TOL[dt]
    check_outputs(o, oo, dt, f"o ({path}, H={H})")
    check_close(m, om, tol["stat"], "m")
    check_close(lse, olse, tol["stat"], "lse")
    check_close(alpha, oa, tol["weight"], "alpha")


@pytest.mark.parametrize("variant", ["sigmoid", "no_key_norm"])
@pytest.mark.parametrize("path", ["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("n,S,T,d,H,dt", [(9, 24, 37, 1024, 16, "bf16"),
                                          (3, 5, 20, 160, 4, "f32")])
def test_phase1_heads_variant(dev, variant, path, n, S, T, d, H, dt):
    flags = VARIANTS[variant]
    seed = 8100 + n + H
    reps = make_reps(n, T, d, _dt(dt), dev, seed)
    W, G, U, us = queries(S, d, dev, seed, flags)
    o = torch.empty((S, T, d), dtype=reps.dtype, device=dev)
    m = torch.empty((S, H, T), device=dev)
    alpha = torch.empty((S, H, T, n), device=dev)
    ar.attnres_phase1(reps, U, o, m, None, alpha, eps=EPS,
                      u_split=us if path == "tensor_cores" else None, flags=flags, heads=H)
    torch.cuda.synchronize()
    oo, om, _, oa = O.multihead_phase1(to64(reps), to64(W), _g64(G), EPS, H, **_wk(flags))
    check_outputs(o, oo, dt, f"o ({variant}, {path})")
    check_close(m, om, TOL[dt]["stat"], "m")
    check_close(alpha, oa, TOL[dt]["weight"], "alpha")


@pytest.mark.parametrize("path", ["tensor_cores", "cuda_cores"])
def test_phase1_heads_agree_with_one_head_per_slice(dev, path):
    """Head k of an H-head call equals a one-head call on the column slice of head k (the
    statistics and outputs of independent aggregations), element for element up to the
    tolerance."""
    n, S, T, d, H = 9, 24, 45, 2048, 4
    dh = d // H
    reps = make_reps(n, T, d, torch.bfloat16, dev, 8200)
    W, G, U, us = queries(S, d, dev, 8200)
    o = torch.empty((S, T, d), dtype=reps.dtype, device=dev)
    lse = torch.empty((S, H, T), device=dev)
    split = us if path == "tensor_cores" else None
    ar.attnres_phase1(reps, U, o, lse_out=lse, eps=EPS, u_split=split, heads=H)
    for k in range(H):
        sl = slice(k * dh, (k + 1) * dh)
        rk = reps[..., sl].contiguous()
        Uk = U[:, sl].contiguous()
        usk = us[:, sl].contiguous()
        ok = torch.empty((S, T, dh), dtype=reps.dtype, device=dev)
        lk = torch.empty((S, T), device=dev)
        ar.attnres_phase1(rk, Uk, ok, lse_out=lk, eps=EPS,
                          u_split=usk if split is not None else None)
        torch.cuda.synchronize()
        check_outputs(o[..., sl], to64(ok), "bf16", f"o head {k}")
        check_close(lse[:, k], to64(lk), TOL["bf16"]["stat"], f"lse head {k}")


# Row-wise kernels: one warp per head for H <= 16 heads of at most 128 16-byte vectors
# (d = 7168 / 16, 256 / 8, 96 / 3); otherwise the generic per-head reduction in shared memory
# (d = 7168 / 4: 224 vectors per head; 2048 / 32: more than 16 heads).
ROW_CASES = [(33, 7168, 16, "bf16"), (40, 256, 8, "f32"), (24, 96, 3, "f32"),
             (21, 7168, 4, "bf16"), (18, 2048, 32, "bf16")]


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("mode", ["first", "fused"])
@pytest.mark.parametrize("T,d,H,dt,ostore", [c + ("io",) for c in ROW_CASES] +
                         [c + ("f32",) for c in ROW_CASES if c[3] == "bf16"])
def test_phase2_heads(dev, variant, mode, T, d, H, dt, ostore):
    """Per call against the per-head merge of what the call received; with o stored in fp32
    (fp32 I/O, or ATTNRES_O_F32 with bf16 I/O) also h, y and the partial's weights end to end
    against the direct per-head aggregation."""
    flags = VARIANTS[variant]
    n, seed = 4, 8300 + d + H
    dtype = _dt(dt)
    reps = make_reps(n, T, d, dtype, dev, seed)
    W, G, U, _ = queries(1, d, dev, seed, flags)
    o = torch.empty((1, T, d), dtype=torch.float32 if ostore == "f32" else dtype, device=dev)
    lse = torch.empty((1, H, T), device=dev)
    ar.attnres_phase1(reps, U, o, lse_out=lse, eps=EPS, flags=flags, heads=H)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    part = I.normal((T, d), 1.5, seed, "part", dev, dtype)
    vprev = I.normal((T, d), 1.0, seed, "vprev", dev, dtype)
    fused = mode == "fused"
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    ap = torch.empty((H, T), device=dev)
    pout = torch.empty_like(part) if fused else None
    sig = bool(flags & SIG)
    ar.attnres_phase2_merge(o[0], None if sig else lse[0], part if fused else None,
                            vprev if fused else None, pout, U[0], G_in, y, h_out=h,
                            alpha_p_out=ap if fused else None, eps_key=EPS, eps_in=EPS,
                            flags=flags, heads=H)
    torch.cuda.synchronize()
    p = to64(part) + to64(vprev) if fused else None
    h_m, y_m, a_m = O.multihead_merge_reference(to64(o[0]), None if sig else to64(lse[0]), p,
                                                to64(W[0]), _g64(G, 0), EPS, to64(G_in), EPS, H,
                                                **_wk(flags))
    check_outputs(h, h_m, dt, f"h ({variant}, {mode}, per call)")
    check_outputs(y, y_m, dt, f"y ({variant}, {mode}, per call)")
    if fused:
        check_close(ap, a_m, TOL[dt]["weight"], "weights of the partial source")
    if dt == "f32" or ostore == "f32":   # two-phase against the direct per-head definition
        srcs = to64(reps) if p is None else np.concatenate([to64(reps), p[None]])
        h_d, a_d, _ = O.multihead_aggregate(srcs, to64(W[0]), _g64(G, 0), EPS, H, **_wk(flags))
        check_outputs(h, h_d, dt, "h (two-phase vs direct)")
        check_outputs(y, O.rmsnorm(h_d, to64(G_in), EPS), dt, "y (two-phase vs direct)")
        if fused:
            check_close(ap, a_d[:, -1], TOL[dt]["weight"], "weights of the partial (vs direct)")


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("n,T,d,H,dt", [(12, 40, 2048, 16, "bf16"), (3, 64, 128, 4, "f32"),
                                        (5, 17, 7168, 16, "bf16"), (4, 20, 7168, 4, "bf16"),
                                        (3, 16, 2048, 32, "bf16"), (64, 9, 512, 16, "f32")])
def test_full_path_heads(dev, variant, n, T, d, H, dt):
    flags = VARIANTS[variant]
    seed = 8400 + n + H
    dtype = _dt(dt)
    srcs = [I.normal((T, d), 1.0 + 0.05 * j, seed, f"v{j}", dev, dtype) for j in range(n)]
    W, G, U, _ = queries(1, d, dev, seed, flags)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    alpha = torch.empty((H, T, n), device=dev)
    ar.attnres_full_reference_path(srcs, U[0], G_in, h_out=h, y_out=y, alpha_out=alpha,
                                   eps_key=EPS, eps_in=EPS, flags=flags, heads=H)
    torch.cuda.synchronize()
    src64 = np.stack([to64(s) for s in srcs])
    h_o, a_o, _ = O.multihead_aggregate(src64, to64(W[0]), _g64(G, 0), EPS, H, **_wk(flags))
    check_outputs(h, h_o, dt, f"h ({variant})")
    check_outputs(y, O.rmsnorm(h_o, to64(G_in), EPS), dt, f"y ({variant})")
    check_close(alpha, np.transpose(a_o, (0, 2, 1)), TOL[dt]["weight"], "alpha")


@pytest.mark.parametrize("H", [8, 32])
@pytest.mark.parametrize("k", [0, 1, 3])
@pytest.mark.parametrize("dt,ostore", [("f32", "io"), ("bf16", "io"), ("bf16", "f32")])
def test_merge_sources_heads(dev, k, dt, ostore, H):
    """Grouped Full AttnRes phase 2 with heads: phase 1 over the history A per head, then the
    merge of k in-group sources; per call against the per-head partition merge of the stored
    (o, lse), and with o stored in fp32 (fp32 I/O, or ATTNRES_O_F32) against the direct
    per-head aggregation over A and B."""
    T, d, nA = 29, 512, 5
    dtype = _dt(dt)
    seed = 8500 + k
    A = torch.stack([I.normal((T, d), 1.0 + 0.1 * j, seed, f"a{j}", dev, dtype)
                     for j in range(nA)])
    Bs = [I.normal((T, d), 1.2, seed, f"b{j}", dev, dtype) for j in range(k)]
    W, G, U, us = queries(1, d, dev, seed)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    o = torch.empty((1, T, d), dtype=torch.float32 if ostore == "f32" else dtype, device=dev)
    lse = torch.empty((1, H, T), device=dev)
    ar.attnres_phase1(A, U, o, lse_out=lse, eps=EPS, heads=H)
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    alpha = torch.empty((H, T, max(k, 1)), device=dev)
    ar.attnres_phase2_merge_sources(o[0], lse[0], Bs, U[0], G_in, h_out=h, y_out=y,
                                    alpha_out=alpha[..., :k] if k else None, eps_key=EPS,
                                    eps_in=EPS, heads=H)
    torch.cuda.synchronize()
    B64 = np.stack([to64(b) for b in Bs]) if k else np.zeros((0, T, d))
    hm = np.zeros((T, d))
    am = np.zeros((H, k, T))
    o64, l64 = to64(o[0]), to64(lse[0])
    for hd, sl in enumerate(O.head_slices(d, H)):
        hk, _, ak, _ = O.merge_sources_reference(o64[:, sl], l64[hd], B64[..., sl],
                                                 to64(W[0])[sl], to64(G[0])[sl], EPS, None, EPS)
        hm[:, sl] = hk
        am[hd] = ak
    check_outputs(h, hm, dt, f"h (k={k}, per call)")
    check_outputs(y, O.rmsnorm(hm, to64(G_in), EPS), dt, f"y (k={k}, per call)")
    if k:
        check_close(alpha[..., :k], np.transpose(am, (0, 2, 1)), TOL[dt]["weight"], "alpha")
    if dt == "f32" or ostore == "f32":
        h_d, _, _ = O.multihead_aggregate(np.concatenate([to64(A), B64]), to64(W[0]),
                                          to64(G[0]), EPS, H)
        check_outputs(h, h_d, dt, "h (grouped vs direct)")
        check_outputs(y, O.rmsnorm(h_d, to64(G_in), EPS), dt, "y (grouped vs direct)")


@pytest.mark.parametrize("dt,T,d,H,path", [("f32", 24, 128, 4, "cuda_cores"),
                                           ("bf16", 40, 1024, 16, "tensor_cores")])
def test_block_walk_heads(dev, dt, T, d, H, path):
    """One block of S = 4 sublayers over n = 3 given sources through BlockRunner with H heads
    (phase 1, phase 2 with the fused partial update, the close) and the final aggregation,
    against the per-head direct definition with the sublayer outputs given."""
    seed, n, S = 8600, 3, 4
    dtype = _dt(dt)
    reps = make_reps(n, T, d, dtype, dev, seed)
    W, G, U, us = queries(S, d, dev, seed)
    G_in = I.gains(S, d, 0.05, seed, "gin", dev)
    v = torch.stack([I.normal((T, d), 1.0, seed, f"out{i}", dev, dtype) for i in range(S)])
    runner = BlockRunner(T, d, S, dtype, dev, keep_y=True, heads=H, o_dtype=torch.float32)
    ys = torch.empty((S, T, d), dtype=dtype, device=dev)
    close = torch.empty((T, d), dtype=dtype, device=dev)

    def sub(i, y):
        ys[i - 1].copy_(y)
        return v[i - 1]

    runner.run_block(reps, U, G_in, sub, close, EPS, EPS,
                     U_split=us if path == "tensor_cores" else None)
    fin = torch.empty((T, d), dtype=dtype, device=dev)
    final_aggregation(torch.cat([reps, close[None]]), U[0], fin, EPS, heads=H)
    torch.cuda.synchronize()
    # the partial sums as the GPU stores them (rounded to the I/O type between sublayers);
    # phase 1's o is stored in fp32 (ATTNRES_O_F32)
    r64 = to64(reps)
    ps, close_want = partial_sources(v, dtype)
    for i in range(1, S + 1):
        srcs = r64 if ps[i - 1] is None else np.concatenate([r64, ps[i - 1][None]])
        h_o, _, _ = O.multihead_aggregate(srcs, to64(W[i - 1]), to64(G[i - 1]), EPS, H)
        check_outputs(ys[i - 1], O.rmsnorm(h_o, to64(G_in[i - 1]), EPS), dt, f"y_{i}")
    assert torch.equal(close.cpu(), close_want), "closed block"
    fin_o, _, _ = O.multihead_aggregate(np.concatenate([r64, to64(close)[None]]), to64(W[0]),
                                        to64(G[0]), EPS, H)
    check_outputs(fin, fin_o, dt, "final")


def test_prefill_shape_heads_sampled(dev):
    """The 128K-prefill chunk shape with 16 heads (n = 9 sources, S = 24 queries, d = 7168),
    2048 tokens (256 token tiles x 2 head windows), on both phase-1 kernels; 24 sampled rows
    against the oracle, every row tensor cores against CUDA cores."""
    n, S, T, d, H = 9, 24, 2048, 7168, 16
    reps = make_reps(n, T, d, torch.bfloat16, dev, 8700)
    W, G, U, us = queries(S, d, dev, 8700)
    outs = {}
    for path in ("tensor_cores", "cuda_cores"):
        o = torch.empty((S, T, d), dtype=reps.dtype, device=dev)
        lse = torch.empty((S, H, T), device=dev)
        ar.attnres_phase1(reps, U, o, lse_out=lse, eps=EPS,
                          u_split=us if path == "tensor_cores" else None, heads=H)
        outs[path] = (o, lse)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(8700).choice(T, 24, replace=False))
    rows[0], rows[-1] = 0, T - 1
    oo, _, olse, _ = O.multihead_phase1(to64(reps[:, rows]), to64(W), to64(G), EPS, H)
    for path, (o, lse) in outs.items():
        check_outputs(o[:, rows], oo, "bf16", f"o ({path}, sampled rows)")
        check_close(lse[:, :, rows], olse, TOL["bf16"]["stat"], f"lse ({path})")
    (o1, l1), (o2, l2) = outs["tensor_cores"], outs["cuda_cores"]
    check_close(l1, to64(l2), TOL["bf16"]["stat"], "lse: tensor cores vs CUDA cores")
    check_outputs(o1, to64(o2), "bf16", "o: tensor cores vs CUDA cores")
