"""GPU kernels (through the C ABI) against the fp64 oracle, element by element, on seeded
inputs at sizes that span several tiles and a ragged tail.  Tolerances: parity_util.TOL."""
import numpy as np
import pytest
import torch

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B
import oracle.attnres_oracle as O
from parity_util import TOL, check_close, check_outputs, check_two_phase, to64
from synth import inputs as I

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    ar.library()
    return torch.device("cuda:0")


@pytest.fixture(params=["tensor_cores", "cuda_cores"])
def p1path(request):
    """Phase-1 kernel choice: with the split queries (tensor-core logits where the shape
    allows: bf16, 2 <= S <= 24, n <= 64) or without them (CUDA-core kernel for every shape)."""
    return request.param


def _dt(name):
    return torch.float32 if name == "f32" else torch.bfloat16


def make_reps(n, T, d, dtype, dev, seed, scale=1.0):
    reps = torch.empty((n, T, d), dtype=dtype, device=dev)
    for j in range(n):
        I.fill_block_rep(reps[j], j, seed)
    if scale != 1.0:
        reps = (reps.float() * scale).to(dtype)
    return reps


def make_queries(S, d, dev, seed, jitter=0.02, scale=1.0, zero=False):
    W = I.queries(S, d, seed, "w", dev, zero=zero) * scale
    G = I.gains(S, d, jitter, seed, "g", dev)
    U = torch.empty_like(W)
    ar.attnres_query_prep(W, G, U)
    return W, G, U


def split_of(U):
    """The bf16 hi/lo split of the queries U, as attnres_query_prep writes it."""
    us = torch.empty((2 * U.shape[0], U.shape[1]), dtype=torch.bfloat16, device=U.device)
    ar.attnres_query_prep(U, None, torch.empty_like(U), us)
    return us


def run_phase1(reps, U, path="cuda_cores", o_dtype=None):
    n, T, d = reps.shape
    S = U.shape[0]
    o = torch.empty((S, T, d), dtype=o_dtype or reps.dtype, device=reps.device)
    m = torch.empty((S, T), dtype=torch.float32, device=reps.device)
    lse = torch.empty_like(m)
    alpha = torch.empty((S, T, n), dtype=torch.float32, device=reps.device)
    us = split_of(U) if path == "tensor_cores" else None
    ar.attnres_phase1(reps, U, o, m, lse, alpha, eps=EPS, u_split=us)
    torch.cuda.synchronize()
    return o, m, lse, alpha


P1_CASES = [
    # n, S, T, d, dtype
    (1, 4, 64, 128, "f32"),
    (2, 4, 64, 128, "f32"),
    (3, 1, 64, 128, "f32"),
    (1, 1, 1, 8, "f32"),            # smallest shape
    (4, 64, 19, 256, "f32"),        # S at its maximum, ragged T
    (9, 24, 37, 7168, "bf16"),      # the long-context block shape, ragged T
    (9, 24, 100, 512, "bf16"),
    (5, 18, 50, 2048, "bf16"),      # a tail block (S = 18)
    (8, 24, 16, 200, "bf16"),       # d not a multiple of the 64-column stage
    (10, 1, 33, 7168, "bf16"),      # final aggregation over 10 sources
    (55, 1, 20, 2048, "bf16"),      # Full-AttnRes final aggregation (55 sources)
    (64, 1, 9, 64, "bf16"),         # n at its maximum
    (16, 64, 5, 64, "bf16"),        # largest n with S = 64
    (64, 2, 11, 64, "bf16"),        # n at its maximum with two queries
    (2, 2, 70, 136, "f32"),
    (7, 5, 23, 96, "f32"),
    (9, 24, 21, 320, "bf16"),       # the largest tensor-core tile with weights kept as pairs
    (16, 24, 21, 320, "bf16"),      # one full M-tile (16 sources x 8 tokens)
    (1, 2, 9, 64, "bf16"),          # its smallest (one source, two queries)
    (3, 7, 8, 136, "bf16"),         # odd S, ragged last column stage
    (17, 24, 12, 128, "bf16"),      # two M-tiles
    (33, 8, 19, 1024, "bf16"),      # three M-tiles
    (49, 16, 9, 2048, "bf16"),      # four M-tiles (the largest Full AttnRes history)
    (9, 24, 21, 512, "bf16"),       # ring slots in pairs (one copy takes two column stages)
    (2, 3, 17, 384, "bf16"),        # pairs, odd S, ragged token tile
]


@pytest.mark.parametrize("n,S,T,d,dt", P1_CASES)
def test_phase1_matches_oracle(dev, p1path, n, S, T, d, dt):
    seed = 1000 + n * 7 + S
    reps = make_reps(n, T, d, _dt(dt), dev, seed)
    W, G, U = make_queries(S, d, dev, seed)
    o, m, lse, alpha = run_phase1(reps, U, p1path)
    oo, om, olse, oalpha = O.phase1(to64(reps), to64(W), to64(G), EPS)
    tol = TOL[dt]
    check_outputs(o, oo, dt, "o")
    check_close(m, om, tol["stat"], "m")
    check_close(lse, olse, tol["stat"], "lse")
    check_close(alpha, oalpha, tol["weight"], "alpha")


O_F32_CASES = [(9, 24, 37, 7168), (9, 24, 100, 512), (5, 18, 50, 2048), (8, 24, 16, 200),
               (10, 1, 33, 7168), (3, 7, 8, 136), (17, 24, 12, 128), (55, 1, 20, 2048)]


@pytest.mark.parametrize("n,S,T,d", O_F32_CASES)
def test_phase1_o_f32(dev, p1path, n, S, T, d):
    """bf16 sources with phase 1's o stored in fp32 (ATTNRES_O_F32): o against the oracle at
    the bf16-mode bound without any storage rounding, the statistics as usual, and the fp32 o
    rounded to bf16 equal, bit for bit, to the o the same kernel stores in bf16 (the store is
    the only difference)."""
    seed = 1500 + n * 7 + S
    reps = make_reps(n, T, d, torch.bfloat16, dev, seed)
    W, G, U = make_queries(S, d, dev, seed)
    o32, m, lse, alpha = run_phase1(reps, U, p1path, torch.float32)
    o16, m2, lse2, alpha2 = run_phase1(reps, U, p1path)
    oo, om, olse, oalpha = O.phase1(to64(reps), to64(W), to64(G), EPS)
    check_outputs(o32, oo, "bf16", "o (fp32 store)")
    check_close(lse, olse, TOL["bf16"]["stat"], "lse")
    check_close(alpha, oalpha, TOL["bf16"]["weight"], "alpha")
    assert torch.equal(o32.to(torch.bfloat16), o16), "o: fp32 store rounded != bf16 store"
    assert torch.equal(lse, lse2) and torch.equal(alpha, alpha2)


def test_query_split(dev):
    """attnres_query_prep's split: hi = bf16(u), lo = bf16(u - hi), |u - hi - lo| <= 2^-16 |u|."""
    S, d = 24, 7168
    W = I.queries(S, d, 5, "w", dev)
    G = I.gains(S, d, 0.02, 5, "g", dev)
    U = torch.empty_like(W)
    us = torch.empty((2 * S, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, G, U, us)
    torch.cuda.synchronize()
    u = to64(U)
    hi, lo = to64(us[0::2]), to64(us[1::2])
    assert torch.equal(us[0::2], U.to(torch.bfloat16))                   # round to nearest even
    assert torch.equal(us[1::2], (U - us[0::2].float()).to(torch.bfloat16))
    assert np.all(np.abs(u - hi - lo) <= 2.0 ** -16 * np.abs(u))


def test_phase1_chunk_view(dev, p1path):
    """A token chunk of a larger cache: source stride != T*d and an offset base pointer."""
    n, Ttot, d, S = 9, 300, 512, 24
    reps_all = make_reps(n, Ttot, d, torch.bfloat16, dev, 77)
    W, G, U = make_queries(S, d, dev, 77)
    view = reps_all[:, 128:245]
    o, m, lse, alpha = run_phase1(view, U, p1path)
    oo, om, olse, oalpha = O.phase1(to64(view), to64(W), to64(G), EPS)
    check_outputs(o, oo, "bf16", "o (chunk view)")
    check_close(lse, olse, 1e-3, "lse (chunk view)")


def test_phase1_zero_queries_give_mean(dev):
    n, T, d, S = 6, 40, 256, 8
    reps = make_reps(n, T, d, torch.float32, dev, 5)
    W, G, U = make_queries(S, d, dev, 5, zero=True)
    o, m, lse, alpha = run_phase1(reps, U)
    check_close(alpha, np.full((S, T, n), 1.0 / n), 1e-6, "uniform weights")
    mean = to64(reps).mean(axis=0)
    check_outputs(o, np.broadcast_to(mean, (S, T, d)), "f32", "o = mean")
    check_close(lse, np.full((S, T), np.log(n)), 1e-5, "lse = ln n")


def test_phase1_extreme_logits(dev, p1path):
    """Large queries push the softmax towards one-hot; max subtraction keeps it finite."""
    n, T, d, S = 9, 24, 512, 24
    reps = make_reps(n, T, d, torch.bfloat16, dev, 9)
    W, G, U = make_queries(S, d, dev, 9, scale=60.0)
    o, m, lse, alpha = run_phase1(reps, U, p1path)
    oo, om, olse, oalpha = O.phase1(to64(reps), to64(W), to64(G), EPS)
    assert float(to64(alpha).max()) > 0.999
    check_outputs(o, oo, "bf16", "o (near one-hot)")
    check_close(alpha, oalpha, 1e-3, "alpha (near one-hot)")
    check_close(lse, olse, 2e-3 * max(1.0, float(np.abs(olse).max()) / 100), "lse")


def test_phase1_deterministic(dev, p1path):
    reps = make_reps(9, 50, 1024, torch.bfloat16, dev, 3)
    _, _, U = make_queries(24, 1024, dev, 3)
    a = run_phase1(reps, U, p1path)
    b = run_phase1(reps, U, p1path)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


P2_MODES = ["first", "partial_only", "vprev_only", "fused", "fused_inplace"]


@pytest.mark.parametrize("mode", P2_MODES)
@pytest.mark.parametrize("n,T,d,dt,ostore", [(2, 64, 128, "f32", "io"), (9, 45, 7168, "bf16", "io"),
                                              (3, 17, 2048, "bf16", "io"), (1, 5, 8, "f32", "io"),
                                              (9, 45, 7168, "bf16", "f32"),
                                              (3, 17, 2048, "bf16", "f32")])
def test_phase2_matches_oracle(dev, mode, n, T, d, dt, ostore):
    """Phase 1 then one phase-2 call.  Per call: h, y and the partial's weight against the
    pages' merge of exactly what the call received.  End to end, against the direct softmax
    over all the sources: the partial's weight at the weight tolerance; h and y at the output
    gate when o is stored in fp32 (ostore "f32", or fp32 I/O), and with the derived bound of
    the bf16 storage of o on the production path (bf16 I/O, ostore "io")."""
    seed = 2000 + n + d
    dtype = _dt(dt)
    reps = make_reps(n, T, d, dtype, dev, seed)
    W, G, U = make_queries(1, d, dev, seed)
    o, m, lse, _ = run_phase1(reps, U, o_dtype=torch.float32 if ostore == "f32" else None)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    part = I.normal((T, d), 1.5, seed, "part", dev, dtype)
    vprev = I.normal((T, d), 1.0, seed, "vprev", dev, dtype)
    partial = part if mode in ("partial_only", "fused", "fused_inplace") else None
    v_prev = vprev if mode in ("vprev_only", "fused", "fused_inplace") else None
    part_in = to64(part)
    if mode == "fused":
        pout = torch.empty_like(part)
    elif mode == "fused_inplace":
        pout = part
    else:
        pout = None
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    ap = torch.empty((T,), dtype=torch.float32, device=dev)
    has_p = partial is not None or v_prev is not None
    ar.attnres_phase2_merge(o[0], lse[0], partial, v_prev, pout, U[0], G_in, y, h_out=h,
                            alpha_p_out=ap if has_p else None, eps_key=EPS, eps_in=EPS)
    torch.cuda.synchronize()
    p_exact = None
    if has_p:
        p_exact = (part_in if partial is not None else 0.0) + \
                  (to64(vprev) if v_prev is not None else 0.0)
    # per call: the oracle gets exactly what the call received (o_l, lse_l, partial, v_prev)
    h_m, y_m, a_m = O.merge_reference(to64(o[0]), to64(lse[0]), p_exact, to64(W[0]),
                                      to64(G[0]), EPS, to64(G_in), EPS)
    check_outputs(h, h_m, dt, "h (per call)")
    check_outputs(y, y_m, dt, "y (per call)")
    if has_p:
        check_close(ap, a_m, TOL[dt]["weight"], "weight of the partial source")
    # end to end: phase 1 + phase 2 against the direct softmax over all the sources
    h_o, y_o, a_o, _ = O.phase2_reference(
        to64(reps), None if partial is None else part_in,
        None if v_prev is None else to64(vprev), to64(W[0]), to64(G[0]), EPS, to64(G_in), EPS)
    if has_p:
        check_close(ap, a_o[-1], TOL[dt]["weight"], "weight of the partial source (vs direct)")
    if dt == "f32" or ostore == "f32":
        check_outputs(h, h_o, dt, "h (vs direct)")
        check_outputs(y, y_o, dt, "y (vs direct)")
    else:
        oA, _, _, _ = O.phase1(to64(reps), to64(W[:1]), to64(G[:1]), EPS)
        wA = 1.0 - (a_o[-1] if has_p else 0.0)
        rh = O.rms(h_o, EPS)
        check_two_phase(y, y_o, oA[0], wA, rh, to64(G_in), dt, "y (two-phase vs direct)")
        check_two_phase(h, h_o, oA[0], wA, rh, to64(G_in), dt, "h (two-phase vs direct)",
                        h_only=True)
    if pout is not None:   # the fused update is exactly round(partial + v_prev)
        want = (torch.from_numpy(part_in).float() + vprev.float().cpu()).to(dtype)
        assert torch.equal(pout.cpu(), want)


@pytest.mark.parametrize("n,T,d,dt", [(3, 64, 128, "f32"), (12, 40, 2048, "bf16"),
                                       (55, 9, 2048, "bf16"), (1, 3, 7168, "bf16"),
                                       (64, 4, 64, "f32")])
def test_full_path_matches_oracle(dev, n, T, d, dt):
    seed = 3000 + n
    dtype = _dt(dt)
    srcs = [I.normal((T, d), 1.0 + 0.05 * j, seed, f"v{j}", dev, dtype) for j in range(n)]
    W, G, U = make_queries(1, d, dev, seed)
    G_in = I.gains(1, d, 0.05, seed, "gin", dev)[0]
    y = torch.empty((T, d), dtype=dtype, device=dev)
    h = torch.empty_like(y)
    alpha = torch.empty((T, n), dtype=torch.float32, device=dev)
    ar.attnres_full_reference_path(srcs, U[0], G_in, h_out=h, y_out=y, alpha_out=alpha,
                                   eps_key=EPS, eps_in=EPS)
    torch.cuda.synchronize()
    src64 = np.stack([to64(s) for s in srcs])
    h_o, y_o, a_o = O.sublayer_input(src64, to64(W[0]), to64(G[0]), EPS, to64(G_in), EPS)
    check_outputs(h, h_o, dt, "h")
    check_outputs(y, y_o, dt, "y")
    check_close(alpha, a_o.T, TOL[dt]["weight"], "alpha")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_partial_update_exact(dev, dt):
    dtype = _dt(dt)
    a = I.normal((333, 1024), 2.0, 1, "a", dev, dtype)
    b = I.normal((333, 1024), 1.0, 1, "b", dev, dtype)
    out = torch.empty_like(a)
    ar.attnres_partial_update(a, b, out)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), (a.float().cpu() + b.float().cpu()).to(dtype))


def test_query_prep_exact(dev):
    W = I.queries(24, 7168, 4, "w", dev)
    G = I.gains(24, 7168, 0.02, 4, "g", dev)
    U = torch.empty_like(W)
    ar.attnres_query_prep(W, G, U)
    U2 = W.clone()
    ar.attnres_query_prep(U2, None, U2)          # gamma NULL: copy, in place
    torch.cuda.synchronize()
    assert torch.equal(U.cpu(), W.cpu() * G.cpu())
    assert torch.equal(U2.cpu(), W.cpu())


def test_empty_T_is_a_noop(dev):
    reps = torch.empty((3, 0, 64), dtype=torch.bfloat16, device=dev)
    U = torch.zeros((2, 64), device=dev)
    o = torch.empty((2, 0, 64), dtype=torch.bfloat16, device=dev)
    ar.attnres_phase1(reps, U, o)
    torch.cuda.synchronize()


def test_scale_invariance_on_gpu(dev):
    """At eps = 0, scaling a source by a > 0 leaves every weight unchanged (RMS-normalised
    keys, raw values) -- checked on the GPU kernels directly."""
    n, T, d, S = 4, 30, 256, 6
    reps = make_reps(n, T, d, torch.float32, dev, 11)
    _, _, U = make_queries(S, d, dev, 11)
    base = torch.empty((S, T, n), device=dev)
    o = torch.empty((S, T, d), device=dev)
    ar.attnres_phase1(reps, U, o, alpha_out=base, eps=0.0)
    reps2 = reps.clone()
    reps2[2] *= 7.0
    scaled = torch.empty_like(base)
    ar.attnres_phase1(reps2, U, o, alpha_out=scaled, eps=0.0)
    torch.cuda.synchronize()
    check_close(scaled, base, 2e-6, "weights under source scaling")


def test_no_bounded_wait_gave_up(dev, p1path):
    """Every phase-1 launch above finished its copies: no bounded wait in a kernel timed out."""
    n, T, d, S = 9, 300, 7168, 24
    reps = make_reps(n, T, d, torch.bfloat16, dev, 31)
    W, G, U = make_queries(S, d, dev, 31)
    run_phase1(reps, U, p1path)
    ar.attnres_poll_device_errors()


@pytest.mark.parametrize("flags", [0, ar.SIGMOID_WEIGHTS])
@pytest.mark.parametrize("n,T", [(9, 256), (9, 520), (12, 256), (9, 1300)])
def test_phase1_tensor_cores_cluster_split(dev, n, T, flags):
    """Tensor-core phase 1 at token counts that select the cluster column split (T = 256: four
    CTAs per 8-token tile; T = 520: two) and at one that does not (T = 1300), d = 7168, S = 24:
    o, m, alpha (and lse with softmax weights) on sampled rows against the oracle, and every
    element against the CUDA-core kernel."""
    d, S = 7168, 24
    reps = make_reps(n, T, d, torch.bfloat16, dev, 90 + n + T)
    W, G, U = make_queries(S, d, dev, 90 + T)
    outs = {}
    for path in ("tensor_cores", "cuda_cores"):
        o = torch.empty((S, T, d), dtype=torch.bfloat16, device=dev)
        m = torch.empty((S, T), device=dev)
        lse = torch.full((S, T), 5.0, device=dev)
        alpha = torch.empty((S, T, n), device=dev)
        ar.attnres_phase1(reps, U, o, m, lse, alpha, eps=EPS,
                          u_split=split_of(U) if path == "tensor_cores" else None, flags=flags)
        outs[path] = (o, m, lse, alpha)
    torch.cuda.synchronize()
    ar.attnres_poll_device_errors()
    rows = np.sort(np.random.default_rng(T).choice(T, 12, replace=False))
    rows[0], rows[-1] = 0, T - 1
    wk = "sigmoid" if flags else "softmax"
    oo, om, olse, oa = O.phase1_variant(to64(reps[:, rows]), to64(W), to64(G), EPS, wk, True)
    o, m, lse, alpha = outs["tensor_cores"]
    check_outputs(o[:, rows], oo, "bf16", f"o (T={T}, n={n})")
    check_close(m[:, rows], om, TOL["bf16"]["stat"], "m")
    check_close(alpha[:, rows], oa, TOL["bf16"]["weight"], "alpha")
    if flags:
        assert torch.all(lse == 5.0), "lse is not written with sigmoid weights"
    else:
        check_close(lse[:, rows], olse, TOL["bf16"]["stat"], "lse")
    o2, m2, lse2, alpha2 = outs["cuda_cores"]
    check_outputs(o, to64(o2), "bf16", "o: tensor cores vs CUDA cores")
    check_close(alpha, to64(alpha2), TOL["bf16"]["weight"], "alpha: tensor cores vs CUDA cores")


TC2_CASES = [
    # n, S, T, d, weights, o stored in; T >= 600 keeps the cluster split (which keeps the
    # CUDA-core weighted sum) out
    (3, 5, 602, 640, "softmax", "bf16"),     # the fewest sources of the path, half a stage
    (7, 2, 601, 1024, "softmax", "bf16"),    # the fewest queries
    (8, 13, 603, 2112, "softmax", "bf16"),   # odd S; the last 128-column stage has one box
    (9, 23, 605, 704, "sigmoid", "bf16"),    # odd S, sigmoid weights, half a last stage
    (7, 24, 604, 960, "softmax", "f32"),     # o stored in fp32 (direct stores), half a stage
    (9, 24, 600, 7168, "softmax", "f32"),    # the block shape, o in fp32 (sampled rows)
]


@pytest.mark.parametrize("n,S,T,d,wk,ost", TC2_CASES)
def test_phase1_tensor_core_weighted_sum(dev, n, S, T, d, wk, ost):
    """The weighted sum of phase 1 on the tensor cores (one head, 3 to 9 sources, no cluster
    split): o, m, alpha and lse against the oracle, on every row (sampled rows at d = 7168), and
    every element of o against the CUDA-core kernel at the same gate."""
    flags = ar.SIGMOID_WEIGHTS if wk == "sigmoid" else 0
    odt = torch.float32 if ost == "f32" else torch.bfloat16
    seed = 7000 + n * 31 + S
    reps = make_reps(n, T, d, torch.bfloat16, dev, seed)
    W, G, U = make_queries(S, d, dev, seed)
    outs = {}
    for path in ("tensor_cores", "cuda_cores"):
        o = torch.empty((S, T, d), dtype=odt, device=dev)
        m = torch.empty((S, T), device=dev)
        lse = torch.full((S, T), 5.0, device=dev)
        alpha = torch.empty((S, T, n), device=dev)
        ar.attnres_phase1(reps, U, o, m, lse, alpha, eps=EPS,
                          u_split=split_of(U) if path == "tensor_cores" else None, flags=flags)
        outs[path] = (o, m, lse, alpha)
    torch.cuda.synchronize()
    ar.attnres_poll_device_errors()
    if d > 4096:
        rows = np.sort(np.random.default_rng(T).choice(T, 16, replace=False))
        rows[0], rows[-1] = 0, T - 1
    else:
        rows = np.arange(T)
    oo, om, olse, oa = O.phase1_variant(to64(reps[:, rows]), to64(W), to64(G), EPS, wk, True)
    o, m, lse, alpha = outs["tensor_cores"]
    check_outputs(o[:, rows], oo, "bf16", f"o (n={n}, S={S}, d={d}, {wk}, o {ost})")
    check_close(m[:, rows], om, TOL["bf16"]["stat"], "m")
    check_close(alpha[:, rows], oa, TOL["bf16"]["weight"], "alpha")
    if flags:
        assert torch.all(lse == 5.0), "lse is not written with sigmoid weights"
    else:
        check_close(lse[:, rows], olse, TOL["bf16"]["stat"], "lse")
    o2 = outs["cuda_cores"][0]
    check_outputs(o, to64(o2), "bf16", "o: tensor cores vs CUDA cores")


@pytest.mark.parametrize("polls", [0, 1000])
def test_wait_timeout_is_reported_and_context_survives(dev, polls):
    """The timeout path, made to run out on purpose without a real hang: a kernel whose bounded
    wait cannot succeed (an mbarrier that nothing arrives on) gives up after `polls` polls and
    counts the event; the poll reports ATTNRES_ERR_TIMEOUT once, the next poll is clean, and the
    context still computes phase 1 correctly afterwards."""
    ar.attnres_poll_device_errors()                       # start from a clean word
    ar.attnres_selftest_wait_timeout(polls)
    torch.cuda.synchronize()
    with pytest.raises(ar.AttnResError, match="ATTNRES_ERR_TIMEOUT"):
        ar.attnres_poll_device_errors()
    ar.attnres_poll_device_errors()                       # read and cleared
    n, S, T, d = 3, 4, 40, 512
    reps = make_reps(n, T, d, torch.bfloat16, dev, 77)
    W, G, U = make_queries(S, d, dev, 77)
    o, m, lse, alpha = run_phase1(reps, U, "tensor_cores")
    oo, om, olse, oa = O.phase1(to64(reps), to64(W), to64(G), EPS)
    check_outputs(o, oo, "bf16", "o after the timeout self-test")
    check_close(lse, olse, TOL["bf16"]["stat"], "lse after the timeout self-test")
    ar.attnres_poll_device_errors()                       # no wait of phase 1 gave up
