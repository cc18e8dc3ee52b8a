"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each ``pin_*`` takes the oracle module and raises AssertionError when the oracle disagrees
with a closed form, an invariant, a special case that reduces to a textbook or library
routine, or a brute-force enumeration.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutations.py`` plants plausible mistakes in a copy of the oracle and checks that
some pin fails for each.  Pages are cited by title and section:

  page 1  "Attention Residuals 阅读补充"
  page 2  "Attention Residuals" (note on arXiv 2603.15031)
"""
from __future__ import annotations

import itertools
import math

import numpy as np

RNG_SEED = 1234


def _rng(k=0):
    return np.random.default_rng(RNG_SEED + k)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max |diff| = {err:.3e} > {tol:.1e}"


# --- RMSNorm (page 1, "RMSNorm 的数学原理") --------------------------------------------------
def pin_rms_moments(O):
    """m_2 = sigma^2 + mu^2 (page 1, "二阶原点矩与方差"): r_0(x)^2 equals numpy's variance plus
    squared mean; with eps, r_eps^2 = m_2 + eps."""
    r = _rng(1)
    for d in (1, 3, 128, 7168):
        x = r.normal(0.7, 2.0, size=(5, d))
        m2 = np.var(x, axis=-1) + np.mean(x, axis=-1) ** 2
        _close(O.rms(x, 0.0) ** 2, m2, 1e-12 * max(1.0, m2.max()), f"r_0^2 vs var+mean^2 d={d}")
        _close(O.rms(x, 0.25) ** 2, m2 + 0.25, 1e-12 * max(1.0, m2.max()), "r_eps^2 = m2 + eps")


def pin_rmsnorm_sphere(O):
    """At gamma = 1, eps = 0 the normalised vector has length sqrt(d) and mean square 1
    (page 1, "从均方根到欧氏范数")."""
    r = _rng(2)
    for d in (2, 17, 128, 2048):
        x = r.normal(0.3, 3.0, size=(7, d))
        y = O.rmsnorm(x, None, 0.0)
        _close(np.linalg.norm(y, axis=-1), np.full(7, math.sqrt(d)), 1e-10 * math.sqrt(d),
               f"|RMSNorm(x)| = sqrt(d), d={d}")
        _close(np.mean(y * y, axis=-1), np.ones(7), 1e-12, "mean square 1")


def pin_rmsnorm_eps_length(O):
    """With eps > 0, |x~|^2 = d |x|^2 / (|x|^2 + d eps) < d (page 1, "ε 与 γ 改变了什么")."""
    r = _rng(3)
    d = 64
    x = r.normal(0.0, 0.1, size=(9, d))
    for eps in (1e-3, 0.01, 0.5):
        y = O.rmsnorm(x, None, eps)
        n2 = np.sum(x * x, axis=-1)
        _close(np.sum(y * y, axis=-1), d * n2 / (n2 + d * eps), 1e-10 * d, f"eps length {eps}")


def pin_rmsnorm_scale_sign(O):
    """RMSNorm(a x) = RMSNorm(x) for a > 0 and = -RMSNorm(x) for a < 0 at eps = 0; with
    eps > 0 the identity is only approximate (page 1, "尺度变化与平移")."""
    r = _rng(4)
    x = r.normal(0.0, 1.0, size=(4, 96))
    g = r.normal(1.0, 0.3, size=96)
    base = O.rmsnorm(x, g, 0.0)
    for a in (1e-3, 0.5, 3.0, 1e4):
        _close(O.rmsnorm(a * x, g, 0.0), base, 1e-11, f"scale invariance a={a}")
        _close(O.rmsnorm(-a * x, g, 0.0), -base, 1e-11, f"sign flip a={-a}")
    # eps > 0 breaks exact invariance when a^2 m2 is comparable to eps
    diff = np.max(np.abs(O.rmsnorm(1e-3 * x, g, 1e-6) - O.rmsnorm(x, g, 1e-6)))
    assert diff > 1e-3, "eps must enter the scale (page 1: approximate for eps > 0)"


def pin_rmsnorm_shift(O):
    """A shift x + c 1 changes m_2 to m_2 + 2 c mu + c^2 (page 1, "尺度变化与平移")."""
    r = _rng(5)
    x = r.normal(0.4, 1.5, size=(6, 50))
    mu = np.mean(x, axis=-1)
    m2 = O.rms(x, 0.0) ** 2
    for c in (-2.0, 0.3, 5.0):
        _close(O.rms(x + c, 0.0) ** 2, m2 + 2 * c * mu + c * c, 1e-10 * (1 + c * c), f"shift {c}")


def pin_rmsnorm_basis_gamma(O):
    """Closed form on a scaled basis vector: RMSNorm(c e_k; gamma) = sign(c) gamma_k sqrt(d)
    e_k at eps = 0 (page 1 definition; gamma acts per feature)."""
    d = 12
    g = np.linspace(0.5, 2.0, d)
    for k, c in ((0, 3.0), (5, -0.25), (11, 7e3)):
        x = np.zeros(d)
        x[k] = c
        want = np.zeros(d)
        want[k] = math.copysign(1.0, c) * g[k] * math.sqrt(d)
        _close(O.rmsnorm(x, g, 0.0), want, 1e-12 * math.sqrt(d), f"basis k={k}")


# --- depth softmax (page 2 §7) ---------------------------------------------------------------
def _sources(r, n, T, d, shift=True):
    v = r.normal(0.0, 1.0, size=(n, T, d)) * np.sqrt(np.arange(1, n + 1))[:, None, None]
    if shift:
        v = v + r.normal(0.0, 0.5, size=(n, T, 1))
    return v


def pin_softmax_simplex(O):
    """alpha > 0 and sum_i alpha_i = 1 for every token (page 2 §7), also with large logits."""
    r = _rng(6)
    v = _sources(r, 7, 11, 40)
    for scale in (1.0, 30.0):
        w = r.normal(0.0, scale / math.sqrt(40), size=40)
        _, alpha, _ = O.aggregate(v, w, None, 1e-6)
        assert alpha.shape == (7, 11)
        assert np.all(alpha > 0.0), "weights must be positive"
        _close(alpha.sum(axis=0), np.ones(11), 1e-13, "weights sum to 1")


def pin_zero_query_mean(O):
    """Zero pseudo-queries give the uniform mean of the sources (page 2 §7, zero init)."""
    r = _rng(7)
    v = _sources(r, 5, 9, 33)
    for g in (None, r.normal(1.0, 0.2, size=33)):
        h, alpha, _ = O.aggregate(v, np.zeros(33), g, 1e-6)
        _close(alpha, np.full((5, 9), 0.2), 1e-14, "uniform weights")
        _close(h, v.mean(axis=0), 1e-12, "h = mean of sources")


def pin_convex_bound(O):
    """|h_l| <= max_i |v_i| (page 2 §7, convex-combination bound)."""
    r = _rng(8)
    v = _sources(r, 6, 20, 24)
    w = r.normal(0.0, 2.0, size=24)
    h, _, _ = O.aggregate(v, w, None, 1e-6)
    assert np.all(np.linalg.norm(h, axis=-1) <= np.linalg.norm(v, axis=-1).max(axis=0) + 1e-12)


def rational_case(O, gamma):
    """Sources on distinct scaled basis vectors, queries chosen so z_j = ln p_j exactly:
    then alpha_j = p_j / sum p and h[k_j] = c_j p_j / sum p.  Returns (got, want) pairs."""
    d = 8
    ks = [1, 6, 3, 4]
    cs = [2.5, -0.75, 40.0, -3.0]
    ps = [1.0, 2.0, 3.0, 4.0]
    T = 1
    v = np.zeros((4, T, d))
    for j, (k, c) in enumerate(zip(ks, cs)):
        v[j, 0, k] = c
    g = np.ones(d) if gamma is None else gamma
    w = np.zeros(d)
    for k, c, p in zip(ks, cs, ps):
        w[k] = math.log(p) / (math.copysign(1.0, c) * math.sqrt(d) * g[k])
    h, alpha, z = O.aggregate(v, w, gamma, 0.0)
    tot = sum(ps)
    want_alpha = np.array(ps)[:, None] / tot
    want_h = np.zeros((T, d))
    for k, c, p in zip(ks, cs, ps):
        want_h[0, k] = c * p / tot
    return (z, np.log(np.array(ps))[:, None]), (alpha, want_alpha), (h, want_h)


def pin_rational_case(O):
    """Exact closed form (see rational_case); also with a non-uniform key gain."""
    for gamma in (None, np.linspace(0.5, 1.5, 8)):
        (z, zw), (a, aw), (h, hw) = rational_case(O, gamma)
        _close(z, zw, 1e-12, "z = ln p")
        _close(a, aw, 1e-13, "alpha = p / sum p")
        _close(h, hw, 1e-11, "h = sum alpha v")


def pin_one_hot_limit(O):
    """A query aligned with source j's normalised direction and scaled up drives alpha_j -> 1
    and h -> v_j (limit of the softmax)."""
    r = _rng(9)
    v = _sources(r, 4, 1, 64)
    j = 2
    u = O.rmsnorm(v[j, 0], None, 0.0) / math.sqrt(64)
    h, alpha, _ = O.aggregate(v, 400.0 * u, None, 0.0)
    assert alpha[j, 0] > 1 - 1e-9, f"alpha_j = {alpha[j, 0]}"
    _close(h[0], v[j, 0], 1e-6 * np.abs(v[j, 0]).max(), "h -> v_j")


def pin_scale_invariance_weights(O):
    """Scaling one source by a > 0 leaves every weight unchanged at eps = 0, because the key
    is RMS-normalised while the value is not (page 1, "回到 AttnRes")."""
    r = _rng(10)
    v = _sources(r, 5, 6, 30)
    w = r.normal(0.0, 0.5, size=30)
    h0, a0, _ = O.aggregate(v, w, None, 0.0)
    for a in (0.01, 9.0):
        v2 = v.copy()
        v2[3] *= a
        h1, a1, _ = O.aggregate(v2, w, None, 0.0)
        _close(a1, a0, 1e-13, f"weights invariant, a={a}")
        _close(h1, h0 + (a - 1.0) * a0[3][:, None] * v[3], 1e-10 * a, "h shifts by source 3 only")


# --- two-phase statistics and merge (page 1 two-phase section; page 2 §10) --------------------
def pin_partition_merge(O):
    """Merging the statistics of any split A | B with the pages' formula
        h = (e^{m_A-m} o_A + e^{m_B-m} o_B) / (e^{m_A-m} l_A + e^{m_B-m} l_B)
    (o unnormalised) equals the direct softmax over A u B.  Brute force over every split of
    n = 5 sources."""
    r = _rng(11)
    n, T, d = 5, 4, 16
    v = _sources(r, n, T, d)
    w = r.normal(0.0, 1.0, size=d)
    g = r.normal(1.0, 0.1, size=d)
    h_direct, a_direct, _ = O.aggregate(v, w, g, 1e-6)
    for k in range(1, n):
        for A in itertools.combinations(range(n), k):
            B = [i for i in range(n) if i not in A]
            oA, mA, lseA, aA = O.partition_stats(v[list(A)], w, g, 1e-6)
            oB, mB, lseB, aB = O.partition_stats(v[B], w, g, 1e-6)
            lA, lB = np.exp(lseA - mA), np.exp(lseB - mB)     # exp-sums from the lse
            m = np.maximum(mA, mB)
            ca, cb = np.exp(mA - m) * lA, np.exp(mB - m) * lB
            h = (ca[:, None] * oA + cb[:, None] * oB) / (ca + cb)[:, None]
            _close(h, h_direct, 1e-12, f"merge split {A}")
            _close(aA * (ca / (ca + cb)), a_direct[list(A)], 1e-13, "merged weights A")
            _close(aB * (cb / (ca + cb)), a_direct[B], 1e-13, "merged weights B")


def pin_lse_bruteforce(O):
    """lse = ln sum exp z by a scalar fsum loop, and 0 <= lse - m <= ln n."""
    r = _rng(12)
    n, T, d = 6, 5, 10
    v = _sources(r, n, T, d)
    w = r.normal(0.0, 2.0, size=d)
    o, m, lse, alpha = O.partition_stats(v, w, None, 1e-6)
    z = O.depth_logits(v, w, None, 1e-6)
    for t in range(T):
        assert abs(lse[t] - O.logsumexp_bruteforce(z[:, t])) < 1e-12
        assert abs(m[t] - max(z[:, t])) == 0.0
    assert np.all(lse - m >= 0.0) and np.all(lse - m <= math.log(n) + 1e-15)
    # partition statistics over the full set reproduce the direct aggregation
    h, a2, _ = O.aggregate(v, w, None, 1e-6)
    _close(o, h, 1e-12, "o_A over all sources = h")
    _close(alpha, a2, 1e-14, "alpha_A over all sources = alpha")


def pin_phase1_per_query(O):
    """phase1() returns, per query s, the partition statistics of that query alone, with
    alpha laid out [S, T, n] (checked against a single-query partition_stats call and the
    rational closed form placed at query 2)."""
    r = _rng(13)
    n, T, d, S = 4, 1, 8, 3
    (_, _), (_, aw), (_, hw) = rational_case(O, None)
    v = np.zeros((n, T, d))
    for j, (k, c) in enumerate(zip([1, 6, 3, 4], [2.5, -0.75, 40.0, -3.0])):
        v[j, 0, k] = c
    W = r.normal(0.0, 1.0, size=(S, d))
    W[2] = 0.0
    for k, c, p in zip([1, 6, 3, 4], [2.5, -0.75, 40.0, -3.0], [1.0, 2.0, 3.0, 4.0]):
        W[2, k] = math.log(p) / (math.copysign(1.0, c) * math.sqrt(d))
    o, m, lse, alpha = O.phase1(v, W, None, 0.0)
    assert o.shape == (S, T, d) and m.shape == (S, T) and alpha.shape == (S, T, n)
    _close(o[2], hw, 1e-11, "phase1 o for the rational query")
    _close(alpha[2, 0], aw[:, 0], 1e-13, "phase1 alpha layout [S,T,n]")
    _close(lse[2], [math.log(10.0)], 1e-12, "lse = ln sum p")


# --- block structure (page 2 §8) -------------------------------------------------------------
def _walk_inputs(r, L, T, d, n_given):
    b0 = r.normal(0.0, 1.0, size=(T, d)) + r.normal(0.0, 0.5, size=(T, 1))
    v = r.normal(0.0, 1.0, size=(L, T, d))
    given = r.normal(0.0, 2.0, size=(n_given, T, d))
    W = r.normal(0.0, 1.0 / math.sqrt(d), size=(L, d)) * 8.0
    Gk = r.normal(1.0, 0.1, size=(L, d))
    Gi = r.normal(1.0, 0.1, size=(L, d))
    wf = r.normal(0.0, 1.0, size=d)
    gf = r.normal(1.0, 0.1, size=d)
    return b0, v, given, W, Gk, Gi, wf, gf


def pin_block_equals_full(O):
    """N = L (one sublayer per block) recovers Full AttnRes exactly (page 2 §8, the two
    extremes): the block walk and the full walk build their source lists differently."""
    r = _rng(14)
    L, T, d = 6, 5, 16
    b0, v, given, W, Gk, Gi, wf, gf = _walk_inputs(r, L, T, d, L)
    blk = O.block_attnres_walk(b0, given, v, 1, W, Gk, Gi, wf, gf, 1e-6, 1e-6, consistent=True)
    full = O.full_attnres_walk(b0, v, W, Gk, Gi, wf, gf, 1e-6, 1e-6)
    for l in range(L):
        _close(blk.h[l], full.h[l], 1e-12, f"h_{l+1}")
        _close(blk.y[l], full.y[l], 1e-12, f"y_{l+1}")
        assert blk.n_sources[l] == full.n_sources[l] == l + 1
    _close(blk.final, full.final, 1e-12, "final aggregation")


def pin_single_block_standard_residual(O):
    """N = 1 with zero queries and eps = 0: every sublayer averages the embedding and the
    partial sum, and after the input RMSNorm this equals RMSNorm of the standard residual
    stream h_l = h_1 + sum_{i<l} f_i(h_i) (page 2 §6 unrolled residual; page 2 §8 'N = 1';
    page 1 "回到 AttnRes", a positive overall scale is cancelled by the next RMSNorm)."""
    r = _rng(15)
    L, T, d = 5, 3, 20
    b0, v, given, _, _, Gi, wf, gf = _walk_inputs(r, L, T, d, 1)
    W = np.zeros((L, d))
    walk = O.block_attnres_walk(b0, given, v, L, W, None, Gi, wf, gf, 0.0, 0.0, consistent=True)
    stream = b0.copy()
    for l in range(L):
        ref = O.rmsnorm(stream, Gi[l], 0.0)
        _close(walk.y[l], ref, 1e-11, f"standard residual at l={l+1}")
        want_n = 1 if l == 0 else 2
        assert walk.n_sources[l] == want_n, "embedding + partial (none for the first sublayer)"
        stream = stream + v[l]


def pin_full_zero_init(O):
    """Full AttnRes with all w_l = 0: h_l = (1/l)(h_1 + sum_{i<l} v_i) (page 2 §7)."""
    r = _rng(16)
    L, T, d = 5, 4, 12
    v0 = r.normal(size=(T, d))
    v = r.normal(size=(L, T, d))
    W = np.zeros((L, d))
    walk = O.full_attnres_walk(v0, v, W, None, None, np.zeros(d), None, 1e-6, 1e-6)
    acc = v0.copy()
    for l in range(1, L + 1):
        _close(walk.h[l - 1], acc / l, 1e-12, f"h_{l} = mean")
        acc = acc + v[l - 1]
    _close(walk.final, acc / (L + 1), 1e-12, "final = mean of all")


def pin_block_score_count(O):
    """The number of logits of the block walk matches page 2 §8's count
    sum_{n=1}^{N} [n + (S-1)(n+1)] (plus the final aggregation's N + 1), and each sublayer
    scores n sources (first of the block) or n + 1 (later ones)."""
    for L, S in ((8, 4), (12, 3), (186 - 18, 24), (6, 1)):
        N = L // S
        want = sum(n + (S - 1) * (n + 1) for n in range(1, N + 1)) + N + 1
        assert O.block_score_count(L, S) == want, (L, S)
    r = _rng(17)
    L, S, T, d = 7, 3, 2, 8
    b0, v, given, W, Gk, Gi, wf, gf = _walk_inputs(r, L, T, d, 3)
    walk = O.block_attnres_walk(b0, given, v, S, W, Gk, Gi, wf, gf, 1e-6, 1e-6)
    want_counts = [1, 2, 2, 2, 3, 3, 3]          # blocks of 3, 3, 1 sublayers
    assert walk.n_sources == want_counts, walk.n_sources
    assert len(walk.closed) == 3


def pin_partials_and_given(O):
    """Inside block n the partial source of position i is the sum of the block's earlier
    outputs (b_n^0 = 0 means no source at i = 1); with ``consistent=False`` the completed
    blocks are the given tensors (page 2 §8 definitions)."""
    r = _rng(18)
    L, S, T, d = 6, 3, 2, 8
    b0, v, given, W, Gk, Gi, wf, gf = _walk_inputs(r, L, T, d, 2)
    walk = O.block_attnres_walk(b0, given, v, S, W, Gk, Gi, wf, gf, 1e-6, 1e-6)
    assert walk.partials[0] is None and walk.partials[3] is None
    _close(walk.partials[1], v[0], 0.0, "b_1^1 = v_1")
    _close(walk.partials[2], v[0] + v[1], 1e-15, "b_1^2")
    _close(walk.partials[5], v[3] + v[4], 1e-15, "b_2^2")
    # sublayer 4 (block 2, first) sees [b_0, given b_1] only
    h4, _, _ = O.aggregate(np.stack([b0, given[0]]), W[3], Gk[3], 1e-6)
    _close(walk.h[3], h4, 1e-13, "block 2 first sublayer uses the given b_1")
    fin, _, _ = O.aggregate(np.stack([b0, given[0], given[1]]), wf, gf, 1e-6)
    _close(walk.final, fin, 1e-13, "final aggregation over b_0 .. b_N")


def pin_input_norm(O):
    """y = RMSNorm_in(h): length sqrt(d) at gamma_in = 1, eps_in = 0, and parallel to h."""
    r = _rng(19)
    v = _sources(r, 3, 4, 32)
    h, y, _ = O.sublayer_input(v, r.normal(size=32), None, 1e-6, None, 0.0)
    _close(np.linalg.norm(y, axis=-1), np.full(4, math.sqrt(32)), 1e-11, "|y| = sqrt(d)")
    cos = np.sum(h * y, axis=-1) / (np.linalg.norm(h, axis=-1) * np.linalg.norm(y, axis=-1))
    _close(cos, np.ones(4), 1e-12, "y parallel to h")


def pin_phase2_reference(O):
    """phase2_reference forms the partial as partial_prev + v_prev, and with neither it is the
    first sublayer (no partial source; page 2 §8, V_first)."""
    r = _rng(20)
    reps = _sources(r, 3, 4, 16)
    pp, vp = r.normal(size=(4, 16)), r.normal(size=(4, 16))
    w = r.normal(size=16)
    h, _, a, p = O.phase2_reference(reps, pp, vp, w, None, 1e-6, None, 1e-6)
    _close(p, pp + vp, 1e-15, "partial = prev + v")
    h2, _, _ = O.aggregate(np.concatenate([reps, (pp + vp)[None]]), w, None, 1e-6)
    _close(h, h2, 1e-13, "four sources")
    h1, _, a1, p1 = O.phase2_reference(reps, None, None, w, None, 1e-6, None, 1e-6)
    assert p1 is None and a1.shape[0] == 3


def pin_single_block_matches_walk(O):
    """The one-block function over given sources equals the depth walk's first block when
    the given source is the embedding alone (two code paths build the same source lists)."""
    r = _rng(21)
    L, T, d = 5, 3, 16
    b0, v, given, W, Gk, Gi, wf, gf = _walk_inputs(r, L, T, d, 1)
    walk = O.block_attnres_walk(b0, given, v, L, W, Gk, Gi, wf, gf, 1e-6, 1e-6, consistent=True)
    one = O.single_block(b0[None], v, W, Gk, Gi, wf, gf, 1e-6, 1e-6)
    for l in range(L):
        _close(one.y[l], walk.y[l], 1e-13, f"y_{l+1}")
        assert one.n_sources[l] == walk.n_sources[l]
    _close(one.closed[0], v.sum(axis=0), 1e-12, "closed block = sum of outputs")
    _close(one.final, walk.final, 1e-13, "final aggregation")


def pin_merge_reference(O):
    """Phase 2 by the merge formula, fed phase 1's statistics of A, equals the direct
    softmax over A plus the partial source (brute force over several A and p), and without a
    partial it returns o_A itself."""
    r = _rng(22)
    n, T, d = 4, 6, 24
    A = _sources(r, n, T, d)
    w = r.normal(0.0, 0.5, size=d)
    gk = r.normal(1.0, 0.1, size=d)
    gi = r.normal(1.0, 0.1, size=d)
    o, m, lse, _ = O.partition_stats(A, w, gk, 1e-6)
    for scale in (0.1, 1.0, 10.0):
        p = r.normal(0.0, scale, size=(T, d))
        h, y, ap = O.merge_reference(o, lse, p, w, gk, 1e-6, gi, 1e-6)
        h2, y2, a2 = O.sublayer_input(np.concatenate([A, p[None]]), w, gk, 1e-6, gi, 1e-6)
        _close(h, h2, 1e-12 * scale, f"merge = direct, scale {scale}")
        _close(y, y2, 1e-11, "y")
        _close(ap, a2[-1], 1e-13, "weight of the partial")
    h0, y0, a0 = O.merge_reference(o, lse, None, w, gk, 1e-6, gi, 1e-6)
    _close(h0, o, 0.0, "no partial: h = o_A")
    assert np.all(a0 == 0.0)


# --- multi-head depth attention (Table 4 variant; reading in the oracle) ---------------------
def pin_multihead_one_head(O):
    """H = 1 is the single-head aggregation, phase 1 and merge."""
    r = _rng(60)
    v = _sources(r, 4, 5, 24)
    W = r.normal(0.0, 0.5, size=(3, 24))
    G = r.normal(1.0, 0.1, size=(3, 24))
    h1, a1, _ = O.multihead_aggregate(v, W[0], G[0], 1e-6, 1)
    h0, a0, _ = O.aggregate(v, W[0], G[0], 1e-6)
    _close(h1, h0, 0.0, "h")
    _close(a1[0], a0, 0.0, "alpha")
    o, m, lse, al = O.multihead_phase1(v, W, G, 1e-6, 1)
    o0, m0, l0, al0 = O.phase1(v, W, G, 1e-6)
    _close(o, o0, 0.0, "o")
    _close(lse[:, 0], l0, 0.0, "lse")


def pin_multihead_scalar_heads(O):
    """H = d: every head is one feature, whose RMSNorm at eps = 0 is sign(v_k) gamma_k, so the
    logit of source i in head k is w_k gamma_k sign(v_ik) and head k's output is the softmax of
    those logits over the sources applied to v_ik (closed form, element by element)."""
    r = _rng(61)
    n, T, d = 3, 2, 6
    v = _sources(r, n, T, d)
    w = r.normal(0.0, 1.0, size=d)
    g = r.normal(1.0, 0.3, size=d)
    h, alpha, z = O.multihead_aggregate(v, w, g, 0.0, d)
    zw = (w * g)[None, None, :] * np.sign(v)                 # [n, T, d]
    e = np.exp(zw - zw.max(axis=0, keepdims=True))
    a = e / e.sum(axis=0, keepdims=True)
    _close(np.moveaxis(z, 0, -1), zw, 1e-12, "scalar-head logits")
    _close(h, np.sum(a * v, axis=0), 1e-12, "scalar-head outputs")


def pin_multihead_heads_independent(O):
    """Changing one head's slice of the query or of a source changes only that head's output
    slice (heads do not mix), and zero queries give the mean in every head."""
    r = _rng(62)
    n, T, d, H = 4, 3, 24, 3
    v = _sources(r, n, T, d)
    w = r.normal(0.0, 0.8, size=d)
    h0, _, _ = O.multihead_aggregate(v, w, None, 1e-6, H)
    w2 = w.copy()
    w2[8:16] *= -3.0                    # head 1
    v2 = v.copy()
    v2[2, :, 16:24] += 5.0              # head 2
    h1, _, _ = O.multihead_aggregate(v2, w2, None, 1e-6, H)
    _close(h1[..., 0:8], h0[..., 0:8], 0.0, "head 0 unchanged")
    assert np.max(np.abs(h1[..., 8:16] - h0[..., 8:16])) > 1e-3
    assert np.max(np.abs(h1[..., 16:24] - h0[..., 16:24])) > 1e-3
    hz, _, _ = O.multihead_aggregate(v, np.zeros(d), None, 1e-6, H)
    _close(hz, v.mean(axis=0), 1e-12, "zero queries: mean")


def pin_multihead_merge(O):
    """Per-head phase 1 over A plus the per-head merge of a partial source equals the direct
    per-head aggregation over A plus the partial, then the whole-vector input RMSNorm."""
    r = _rng(63)
    n, T, d, H = 4, 3, 32, 4
    A = _sources(r, n, T, d)
    p = r.normal(0.0, 2.0, size=(T, d))
    W = r.normal(0.0, 0.5, size=(1, d))
    G = r.normal(1.0, 0.1, size=(1, d))
    gi = r.normal(1.0, 0.1, size=d)
    o, m, lse, _ = O.multihead_phase1(A, W, G, 1e-6, H)
    h, y, ap = O.multihead_merge_reference(o[0], lse[0], p, W[0], G[0], 1e-6, gi, 1e-6, H)
    hd, ad, _ = O.multihead_aggregate(np.concatenate([A, p[None]]), W[0], G[0], 1e-6, H)
    _close(h, hd, 1e-12, "merge = direct")
    _close(y, O.rmsnorm(hd, gi, 1e-6), 1e-12, "y")
    _close(ap, ad[:, -1], 1e-14, "weights of the partial")


# --- backward (page 2 §7 logit gradient; page 1 "梯度沿切向传播") ------------------------------
def _fd_grad(f, x, h=1e-6):
    """Central finite differences of the scalar f at x (any shape), in fp64."""
    x = np.array(x, dtype=np.float64)
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        g[i] = (f(xp) - f(xm)) / (2 * h)
    return g


def pin_rmsnorm_backward(O):
    """The RMSNorm input gradient against finite differences (with gain and eps), and the
    pages' radial property: at eps = 0 the Jacobian maps x to 0, so x^T dL/dx = 0; with eps the
    radial eigenvalue is eps / r^3 (page 1, "梯度沿切向传播")."""
    r = _rng(50)
    d = 6
    x = r.normal(0.3, 1.2, size=d)
    g = r.normal(0.0, 1.0, size=d)
    gam = r.normal(1.0, 0.2, size=d)
    for eps in (0.0, 0.3):
        dx, dg = O.rmsnorm_backward(x, gam, eps, g)
        fd = _fd_grad(lambda xx: float(np.sum(g * O.rmsnorm(xx, gam, eps))), x)
        _close(dx, fd, 1e-8, f"dL/dx eps={eps}")
        fdg = _fd_grad(lambda gg: float(np.sum(g * O.rmsnorm(x, gg, eps))), gam)
        _close(dg, fdg, 1e-8, "dL/dgamma")
    dx, _ = O.rmsnorm_backward(x, None, 0.0, g)
    assert abs(float(np.dot(x, dx))) < 1e-12, "radial component at eps = 0"
    eps = 0.3
    rr = float(O.rms(x, eps))
    dx, _ = O.rmsnorm_backward(x, None, eps, g)
    _close(np.dot(x, dx), eps / rr ** 3 * np.dot(x, g), 1e-12, "radial eigenvalue eps / r^3")


def pin_aggregate_backward_fd(O):
    """Every gradient of the aggregation (sources, query, both gains) against central finite
    differences of L = sum g_y ⊙ y computed by the forward oracle."""
    r = _rng(51)
    n, T, d = 3, 2, 5
    v = _sources(r, n, T, d)
    w = r.normal(0.0, 0.7, size=d)
    gk = r.normal(1.0, 0.2, size=d)
    gi = r.normal(1.0, 0.2, size=d)
    gy = r.normal(0.0, 1.0, size=(T, d))
    ek, ei = 1e-3, 2e-3
    G = O.aggregate_backward(v, w, gk, ek, gi, ei, gy)

    def loss(vv=v, ww=w, kk=gk, ii=gi):
        _, y, _ = O.sublayer_input(vv, ww, kk, ek, ii, ei)
        return float(np.sum(gy * y))
    _close(G.dsources, _fd_grad(lambda x: loss(vv=x), v), 1e-7, "dL/dv")
    _close(G.dw, _fd_grad(lambda x: loss(ww=x), w), 1e-7, "dL/dw")
    _close(G.dgamma_key, _fd_grad(lambda x: loss(kk=x), gk), 1e-7, "dL/dgamma_key")
    _close(G.dgamma_in, _fd_grad(lambda x: loss(ii=x), gi), 1e-7, "dL/dgamma_in")
    # the folded query: z_i = u . v_i / r_i with u = w ⊙ gamma_key
    _close(G.dw, gk * G.du, 1e-13, "dw = gamma_key ⊙ du")
    _close(G.dgamma_key, w * G.du, 1e-13, "dgamma_key = w ⊙ du")


def pin_backward_scale_invariance(O):
    """At eps = 0 both norms are scale invariant, so the key-path gradient of each source is
    orthogonal to it (v_i^T (dv_i - alpha_i g_h) = 0) and the norm's input gradient is
    orthogonal to h (h^T g_h = 0); and the logit gradients sum to 0 over the sources
    (softmax: sum_i alpha_i (v_i - h) = 0)."""
    r = _rng(52)
    n, T, d = 4, 3, 16
    v = _sources(r, n, T, d)
    w = r.normal(0.0, 0.5, size=d)
    gy = r.normal(0.0, 1.0, size=(T, d))
    G = O.aggregate_backward(v, w, None, 0.0, None, 0.0, gy)
    _, alpha, _ = O.aggregate(v, w, None, 0.0)
    h, _, _ = O.aggregate(v, w, None, 0.0)
    key_path = G.dsources - alpha[..., None] * G.g_h[None]
    _close(np.sum(key_path * v, axis=-1), np.zeros((n, T)), 1e-12, "v_i . key-path gradient")
    _close(np.sum(G.g_h * h, axis=-1), np.zeros(T), 1e-12, "h . g_h")
    _close(G.dz.sum(axis=0), np.zeros(T), 1e-12, "sum_i dz_i")


def pin_block_backward_fd(O):
    """The block's backward composed over its S sublayers (every completed source collects the
    gradients of all S sublayers; the partial source of sublayer i passes its gradient to each
    v_k it sums, k < i) against central finite differences of L = sum_i g_i ⊙ y_i computed by
    the forward oracle's block (``single_block``), for the completed sources, the sublayer
    outputs and every per-sublayer parameter."""
    r = _rng(53)
    n, S, T, d = 2, 3, 2, 5
    comp = _sources(r, n, T, d)
    v = r.normal(0.0, 1.0, size=(S, T, d))
    W = r.normal(0.0, 0.7, size=(S, d))
    Gk = r.normal(1.0, 0.2, size=(S, d))
    Gi = r.normal(1.0, 0.2, size=(S, d))
    gy = r.normal(0.0, 1.0, size=(S, T, d))
    ek, ei = 1e-3, 2e-3
    G = O.block_backward(comp, v, W, Gk, Gi, ek, ei, gy)

    def loss(cc=comp, vv=v, ww=W, kk=Gk, ii=Gi):
        b = O.single_block(cc, vv, ww, kk, ii, W[0], None, ek, ei)
        return float(sum(np.sum(gy[i] * b.y[i]) for i in range(S)))
    _close(G.dcompleted, _fd_grad(lambda x: loss(cc=x), comp), 1e-7, "dL/db_j")
    _close(G.dv, _fd_grad(lambda x: loss(vv=x), v), 1e-7, "dL/dv_k")
    _close(G.dw, _fd_grad(lambda x: loss(ww=x), W), 1e-7, "dL/dw_i")
    _close(G.dgamma_key, _fd_grad(lambda x: loss(kk=x), Gk), 1e-7, "dL/dgamma_key,i")
    _close(G.dgamma_in, _fd_grad(lambda x: loss(ii=x), Gi), 1e-7, "dL/dgamma_in,i")
    _close(G.dw, Gk * G.du, 1e-13, "dw_i = gamma_key,i ⊙ du_i")
    assert np.all(G.dv[-1] == 0.0) and np.all(G.dpartial[0] == 0.0)
    # dv_k is the sum of the partial gradients of the sublayers after k
    _close(G.dv[:-1], np.cumsum(G.dpartial[::-1], axis=0)[::-1][1:], 1e-13, "dv = suffix sums")


# --- grouped two-phase Full AttnRes (page 1, "静态 Query 与两阶段计算") ------------------------
def pin_grouped_full_equals_direct(O):
    """The grouped two-phase schedule reproduces the direct Full AttnRes walk for every group
    size, including S = 1 (phase 1 alone) and S = L (one group, phase 2 merges up to L - 1
    in-group sources)."""
    r = _rng(40)
    L, T, d = 7, 3, 16
    v0 = r.normal(0.0, 1.0, size=(T, d))
    v = r.normal(0.0, 1.0, size=(L, T, d)) * (1.0 + 0.1 * np.arange(1, L + 1))[:, None, None]
    W = r.normal(0.0, 0.5, size=(L, d))
    Gk = r.normal(1.0, 0.1, size=(L, d))
    Gi = r.normal(1.0, 0.1, size=(L, d))
    full = O.full_attnres_walk(v0, v, W, Gk, Gi, None, None, 1e-6, 1e-6)
    for S in (1, 2, 3, L):
        g = O.grouped_full_walk(v0, v, W, Gk, Gi, S, 1e-6, 1e-6)
        for l in range(L):
            _close(g.y[l], full.y[l], 1e-12, f"S={S} y_{l + 1}")
            _close(g.h[l], full.h[l], 1e-12, f"S={S} h_{l + 1}")
            _close(g.alpha[l], full.alpha[l], 1e-14, f"S={S} alpha_{l + 1}")


def pin_merge_sources(O):
    """Merging partition A with a list B of in-group sources equals the direct softmax over
    A u B for every split of 5 sources; with one source it is merge_reference; with none it
    returns o_A."""
    r = _rng(41)
    n, T, d = 5, 4, 12
    v = _sources(r, n, T, d)
    w = r.normal(0.0, 1.0, size=d)
    g = r.normal(1.0, 0.1, size=d)
    gi = r.normal(1.0, 0.1, size=d)
    h_d, a_d, _ = O.aggregate(v, w, g, 1e-6)
    for k in range(1, n):
        o, m, lse, aA = O.partition_stats(v[:k], w, g, 1e-6)
        h, y, aB, wA = O.merge_sources_reference(o, lse, v[k:], w, g, 1e-6, gi, 1e-6)
        _close(h, h_d, 1e-12, f"A = first {k}")
        _close(aB, a_d[k:], 1e-14, "in-group weights")
        _close(aA * wA, a_d[:k], 1e-14, "history weights")
        _close(y, O.rmsnorm(h_d, gi, 1e-6), 1e-12, "y")
    o, m, lse, _ = O.partition_stats(v[:4], w, g, 1e-6)
    h1, y1, aB, _ = O.merge_sources_reference(o, lse, v[4:], w, g, 1e-6, gi, 1e-6)
    h2, y2, ap = O.merge_reference(o, lse, v[4], w, g, 1e-6, gi, 1e-6)
    _close(h1, h2, 1e-13, "one source = merge_reference")
    _close(aB[0], ap, 1e-15, "its weight")
    h0, _, aB0, wA0 = O.merge_sources_reference(o, lse, v[:0], w, g, 1e-6, gi, 1e-6)
    _close(h0, o, 0.0, "no source: o_A")
    assert aB0.shape[0] == 0 and np.all(wA0 == 1.0)


# --- Table 4 ablation variants (page 2 "Attention Residuals" note, result 4) -------------------
def pin_sigmoid_zero_query_half(O):
    """Sigmoid weights with zero queries: every weight is sigmoid(0) = 1/2 (no sum-to-1), so
    h = (1/2) sum_i v_i."""
    r = _rng(30)
    v = _sources(r, 5, 7, 20)
    for kn in (True, False):
        h, alpha, _ = O.aggregate_variant(v, np.zeros(20), None, 1e-6, "sigmoid", kn)
        _close(alpha, np.full((5, 7), 0.5), 0.0, "alpha = 1/2")
        _close(h, 0.5 * v.sum(axis=0), 1e-12, "h = half the sum")


def pin_sigmoid_rational(O):
    """Sources on distinct scaled basis vectors and queries with z_j = ln(p_j / (1 - p_j)):
    then alpha_j = p_j exactly and h[k_j] = c_j p_j (sigmoid weights, key RMSNorm at eps = 0,
    where RMSNorm(c e_k) = sign(c) sqrt(d) gamma_k e_k)."""
    d = 8
    ks, cs, ps = [2, 5, 7], [3.0, -0.5, 12.0], [0.2, 0.5, 0.9]
    v = np.zeros((3, 1, d))
    for j, (k, c) in enumerate(zip(ks, cs)):
        v[j, 0, k] = c
    g = np.linspace(0.5, 1.5, d)
    w = np.zeros(d)
    for k, c, p in zip(ks, cs, ps):
        w[k] = math.log(p / (1 - p)) / (math.copysign(1.0, c) * math.sqrt(d) * g[k])
    h, alpha, _ = O.aggregate_variant(v, w, g, 0.0, "sigmoid", True)
    _close(alpha[:, 0], np.array(ps), 1e-14, "alpha = p")
    want = np.zeros(d)
    for k, c, p in zip(ks, cs, ps):
        want[k] = c * p
    _close(h[0], want, 1e-13, "h[k_j] = c_j p_j")


def pin_sigmoid_reflection(O):
    """sigmoid(z) + sigmoid(-z) = 1, so h(w) + h(-w) = sum_i v_i for any sources."""
    r = _rng(31)
    v = _sources(r, 6, 5, 16)
    w = r.normal(0.0, 1.0, size=16)
    for kn in (True, False):
        h1, _, _ = O.aggregate_variant(v, w, None, 1e-6, "sigmoid", kn)
        h2, _, _ = O.aggregate_variant(v, -w, None, 1e-6, "sigmoid", kn)
        _close(h1 + h2, v.sum(axis=0), 1e-12, "h(w) + h(-w)")


def pin_sigmoid_partitions_add(O):
    """With sigmoid weights the partitions of any split simply add (brute force over every
    split of 5 sources), and the phase-2 merge of phase 1's partition plus a partial source
    equals the direct aggregation over both."""
    r = _rng(32)
    n, T, d = 5, 3, 12
    v = _sources(r, n, T, d)
    W = r.normal(0.0, 1.0, size=(2, d))
    G = r.normal(1.0, 0.1, size=(2, d))
    for kn in (True, False):
        o_all, _, lse, _ = O.phase1_variant(v, W, G, 1e-6, "sigmoid", kn)
        assert lse is None
        for s in range(2):
            h, _, _ = O.aggregate_variant(v, W[s], G[s], 1e-6, "sigmoid", kn)
            _close(o_all[s], h, 1e-12, "phase 1 over all = direct")
        for k in range(1, n):
            for A in itertools.combinations(range(n), k):
                B = [i for i in range(n) if i not in A]
                oA = O.phase1_variant(v[list(A)], W, G, 1e-6, "sigmoid", kn)[0]
                oB = O.phase1_variant(v[B], W, G, 1e-6, "sigmoid", kn)[0]
                _close(oA + oB, o_all, 1e-12, f"split {A}")
        gi = r.normal(1.0, 0.1, size=d)
        p = r.normal(0.0, 2.0, size=(T, d))
        oA = O.phase1_variant(v[:3], W[:1], G[:1], 1e-6, "sigmoid", kn)[0][0]
        h, y, ap = O.merge_reference_variant(oA, None, p, W[0], G[0], 1e-6, gi, 1e-6, "sigmoid",
                                             kn)
        h2, a2, _ = O.aggregate_variant(np.concatenate([v[:3], p[None]]), W[0], G[0], 1e-6,
                                        "sigmoid", kn)
        _close(h, h2, 1e-12, "merge = direct")
        _close(ap, a2[-1], 1e-15, "weight of the partial")
        _close(y, O.rmsnorm(h2, gi, 1e-6), 1e-12, "y")


def pin_raw_logits(O):
    """No key RMSNorm: the logit of c e_k is w_k c exactly, and scaling one source by a scales
    its logit by a (the magnitude enters the score, unlike the normalised key)."""
    d = 10
    w = np.arange(1.0, d + 1.0) / 7.0
    for k, c in ((0, 2.0), (4, -3.5), (9, 0.25)):
        v = np.zeros((1, 1, d))
        v[0, 0, k] = c
        _close(O.depth_logits_raw(v, w), [[w[k] * c]], 1e-15, "z = w_k c")
    r = _rng(33)
    v = _sources(r, 4, 6, d)
    z0 = O.variant_logits(v, w, None, 1e-6, False)
    v2 = v.copy()
    v2[1] *= -2.5
    z1 = O.variant_logits(v2, w, None, 1e-6, False)
    _close(z1[1], -2.5 * z0[1], 1e-12, "z scales with the source")
    _close(np.delete(z1, 1, 0), np.delete(z0, 1, 0), 0.0, "other logits unchanged")


def pin_raw_equals_scaled_query(O):
    """When every source row has the same RMS r (eps = 0, no gain), w^T v = r w^T RMSNorm(v),
    so dropping the key norm equals keeping it with the query scaled by r."""
    r = _rng(34)
    v = _sources(r, 5, 4, 32)
    rr = 1.7
    v = v / O.rms(v, 0.0)[..., None] * rr
    w = r.normal(0.0, 0.3, size=32)
    for weights in ("softmax", "sigmoid"):
        h1, a1, z1 = O.aggregate_variant(v, w, None, 0.0, weights, False)
        h2, a2, z2 = O.aggregate_variant(v, rr * w, None, 0.0, weights, True)
        _close(z1, z2, 1e-12, "logits")
        _close(h1, h2, 1e-12, f"h ({weights})")


def pin_variant_defaults(O):
    """The variant functions with softmax weights and the key RMSNorm are the default ones."""
    r = _rng(35)
    v = _sources(r, 4, 5, 24)
    W = r.normal(0.0, 0.5, size=(3, 24))
    G = r.normal(1.0, 0.1, size=(3, 24))
    gi = r.normal(1.0, 0.1, size=24)
    h, a, z = O.aggregate(v, W[0], G[0], 1e-6)
    h2, a2, z2 = O.aggregate_variant(v, W[0], G[0], 1e-6)
    _close(h2, h, 0.0, "h")
    _close(a2, a, 0.0, "alpha")
    base = O.phase1(v, W, G, 1e-6)
    var = O.phase1_variant(v, W, G, 1e-6)
    for x, y, nm in zip(var, base, ("o", "m", "lse", "alpha")):
        _close(x, y, 1e-14, f"phase1 {nm}")
    p = r.normal(0.0, 1.0, size=(5, 24))
    m1 = O.merge_reference(base[0][0], base[2][0], p, W[0], G[0], 1e-6, gi, 1e-6)
    m2 = O.merge_reference_variant(base[0][0], base[2][0], p, W[0], G[0], 1e-6, gi, 1e-6)
    for x, y in zip(m2, m1):
        _close(x, y, 0.0, "merge")
    vv = r.normal(0.0, 1.0, size=(3, 5, 24))
    ys, hs, closed = O.single_block_variant(v[:2], vv, W, G, np.stack([gi] * 3), 1e-6, 1e-6)
    for i in range(3):
        srcs = O.block_sources(list(v[:2]), None if i == 0 else vv[:i].sum(axis=0))
        _, y, _ = O.sublayer_input(srcs, W[i], G[i], 1e-6, gi, 1e-6)
        _close(ys[i], y, 1e-13, f"single_block_variant y_{i + 1}")
    _close(closed, vv.sum(axis=0), 1e-12, "closed block")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
