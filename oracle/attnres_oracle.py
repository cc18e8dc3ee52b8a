"""Plain, slow, fp64 CPU oracle for Attention Residuals (AttnRes) residual aggregation.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links this file:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.
It shares no code, header, table or helper with the CUDA library; both sides only share the
seeded input generators in ``synth/``.

Everything here is the *direct* definition written out in float64 numpy, with no blocking,
fusion or reordering: the two-phase schedule is exact in real arithmetic (page 1 "Attention
Residuals 阅读补充", section "静态 Query 与两阶段计算", the merge identity; page 2 "Attention
Residuals" note, §10), so the oracle for every phase is the plain softmax over the sources the
definition names.  Vectorising over tokens is not a reordering: depth attention never mixes
tokens (page 2 §7: "only aggregates along depth"; page 5 "ML 研究者的三层基本功", system layer,
sequence sharding).

Pages cited (titles as they appear on the pages):
  page 1  "Attention Residuals 阅读补充" (chlience.com reading notes)
  page 2  "Attention Residuals" (papers.chlience.com note on arXiv 2603.15031)
  page 3  CSDN/gitcode overview article of the AttnRes report
  page 4  "Kimi K3 模型结构（4）：深度维度，Attention Residuals"

Readings of points the pages leave open (each is also listed in the design notes):
  * phase 1 returns the *normalised* partial output o_A / l_A plus m_A and a true
    log-sum-exp lse_A = m_A + ln l_A (page 2 §10 calls l both an exp-sum and a log-sum-exp;
    page 3 section 4.2 says "max, log-sum-exp");
  * the first sublayer of a block has no partial-sum source at all (page 2 §8, V_first);
  * eps sits inside the square root, added to the mean square (page 1, definition of r_eps);
  * the key-norm gain gamma belongs to the target sublayer l (page 1, "Full AttnRes" cost
    section: one query vector and one set of RMSNorm gains per layer);
  * no 1/sqrt(d) scale and no temperature (page 2 §7);
  * the norm fused after the merge is the input RMSNorm of sublayer l, y = RMSNorm_in(h)
    (page 3 section 4.2 kernel fusion; page 1 "回到 AttnRes", f(z) = F(RMSNorm(z)));
  * the final output aggregates the embedding and all complete blocks with one extra
    pseudo-query w_{L+1} (page 2 §8, last sentence of the block definition).

Parity status: every function below is pinned by ``tests/test_oracle_pins.py`` (closed forms,
invariants, special cases, brute force) and by ``tests/test_oracle_mutations.py`` (planted
mistakes that the pins must catch).  No function here is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F64 = np.float64


def _f64(x):
    return np.asarray(x, dtype=F64)


# ---------------------------------------------------------------------------------------------
# RMSNorm (page 1, section "RMSNorm 的数学原理")
# ---------------------------------------------------------------------------------------------
def rms(x, eps: float):
    """r_eps(x) = sqrt( (1/d) * sum_k x_k^2 + eps ), over the last axis (the d features of one
    token).  Page 1, "RMSNorm 的数学原理", definition of the root mean square with eps."""
    x = _f64(x)
    d = x.shape[-1]
    return np.sqrt(np.sum(x * x, axis=-1) / d + eps)


def rmsnorm(x, gamma, eps: float):
    """RMSNorm(x) = gamma ⊙ x / r_eps(x).  ``gamma=None`` stands for all ones.
    Page 1, "RMSNorm 的数学原理", the normalisation with the learnable per-feature gain."""
    x = _f64(x)
    y = x / rms(x, eps)[..., None]
    if gamma is not None:
        y = y * _f64(gamma)
    return y


# ---------------------------------------------------------------------------------------------
# Depth attention for one target sublayer (page 2 §7, Full AttnRes equations)
# ---------------------------------------------------------------------------------------------
def depth_logits(sources, w, gamma_key, eps: float):
    """z_i = w^T RMSNorm(v_i) for every source i.

    sources: [n, T, d] (source-major), w: [d], gamma_key: [d] or None.  Returns z: [n, T].
    Page 2 §7: the keys are the RMS-normalised sources, the query is the static w_l, no scale.
    """
    keys = rmsnorm(sources, gamma_key, eps)            # [n, T, d]
    return np.sum(keys * _f64(w), axis=-1)             # [n, T]


def depth_softmax(z):
    """alpha_i = exp(z_i) / sum_j exp(z_j) over the source axis (axis 0).  The max is taken
    out first only to keep exp in range; it cancels exactly.  Page 2 §7."""
    z = _f64(z)
    e = np.exp(z - np.max(z, axis=0, keepdims=True))
    return e / np.sum(e, axis=0, keepdims=True)


def aggregate(sources, w, gamma_key, eps: float):
    """h = sum_i alpha_i v_i with alpha = softmax_i(w^T RMSNorm(v_i)).

    The values are the raw sources (not normalised).  Page 2 §7 (the h_l equation); page 1
    "回到 AttnRes" (the a_{t+1,s} kernel).  Returns (h [T,d], alpha [n,T], z [n,T]).
    """
    src = _f64(sources)
    z = depth_logits(src, w, gamma_key, eps)
    alpha = depth_softmax(z)
    h = np.sum(alpha[..., None] * src, axis=0)
    return h, alpha, z


def partition_stats(sources, w, gamma_key, eps: float):
    """Softmax statistics of one source partition X (page 1, two-phase section; page 2 §10):

        m_X = max_i z_i,   l_X = sum_i exp(z_i - m_X),   o_X = sum_i exp(z_i - m_X) v_i.

    Returned as phase 1 hands them over (reading of the l / log-sum-exp naming clash):
    (o_X / l_X  [T,d],  m_X [T],  lse_X = m_X + ln l_X [T],  alpha_X = e / l_X [n,T]).
    """
    src = _f64(sources)
    z = depth_logits(src, w, gamma_key, eps)
    m = np.max(z, axis=0)
    e = np.exp(z - m)
    ell = np.sum(e, axis=0)
    o = np.sum(e[..., None] * src, axis=0) / ell[..., None]
    return o, m, m + np.log(ell), e / ell


def sublayer_input(sources, w, gamma_key, eps_key: float, gamma_in, eps_in: float):
    """The input of sublayer l: h_l by depth attention, then its input RMSNorm y_l.

    Returns (h [T,d], y [T,d], alpha [n,T]).  Page 2 §7 for h; page 1 "回到 AttnRes"
    (f(z) = F(RMSNorm(z))) for y.
    """
    h, alpha, _ = aggregate(sources, w, gamma_key, eps_key)
    y = rmsnorm(h, gamma_in, eps_in)
    return h, y, alpha


def phase1(reps, W, G_key, eps: float):
    """What phase 1 of one block returns, by the definition: for each of the S queries of the
    block, the softmax statistics over the partition A = {b_0 .. b_{n-1}} (page 2 §10 step 1;
    page 1 two-phase section, step 1).

    reps: [n, T, d]; W: [S, d]; G_key: [S, d] or None.
    Returns o [S,T,d], m [S,T], lse [S,T], alpha [S,T,n].
    """
    reps = _f64(reps)
    S = np.shape(W)[0]
    outs = []
    for s in range(S):
        g = None if G_key is None else _f64(G_key)[s]
        outs.append(partition_stats(reps, _f64(W)[s], g, eps))
    o = np.stack([x[0] for x in outs])
    m = np.stack([x[1] for x in outs])
    lse = np.stack([x[2] for x in outs])
    alpha = np.stack([np.moveaxis(x[3], 0, -1) for x in outs])
    return o, m, lse, alpha


# ---------------------------------------------------------------------------------------------
# Block AttnRes depth walk (page 2 §8; page 3 section 3.2; page 4 block structure)
# ---------------------------------------------------------------------------------------------
def block_of(l: int, S: int):
    """Sublayer l (1-based) sits in block n = ceil(l / S) at position i = l - (n-1) S.
    Block boundaries fall at multiples of S; the last block may be shorter (page 4: K3 has
    seven full blocks and a shorter tail)."""
    n = (l - 1) // S + 1
    return n, l - (n - 1) * S


def block_sources(completed, partial):
    """Sources of a sublayer in block n (page 2 §8, V_first / V_later):
    [b_0, ..., b_{n-1}] and, from the second sublayer of the block on, the partial b_n^{i-1}.
    ``partial=None`` is the first sublayer: the partial is absent, not a zero source."""
    srcs = [_f64(b) for b in completed]
    if partial is not None:
        srcs.append(_f64(partial))
    return np.stack(srcs)


@dataclass
class BlockWalk:
    """Everything the direct-definition walk produces, for parity and pins."""
    h: list = field(default_factory=list)          # h_l [T,d] for l = 1..L
    y: list = field(default_factory=list)          # y_l = RMSNorm_in(h_l)
    alpha: list = field(default_factory=list)      # alpha over the sources of l, [n_l, T]
    n_sources: list = field(default_factory=list)  # number of sources scored by sublayer l
    partials: list = field(default_factory=list)   # b_n^{i-1} used by l (None when i = 1)
    closed: list = field(default_factory=list)     # b_n = b_n^{S_n} for every block n
    final: np.ndarray | None = None                # final aggregation over b_0 .. b_N
    final_alpha: np.ndarray | None = None


def block_attnres_walk(b0, given_blocks, v, S: int, W, G_key, G_in, w_final, g_final,
                       eps_key: float, eps_in: float, consistent: bool = False) -> BlockWalk:
    """Walk L sublayers of Block AttnRes by the direct definition.

    b0: embedding b_0 [T,d].  v: [L, T, d], v[l-1] stands in for f_l(h_l), the output of
    sublayer l.  given_blocks: completed block representations b_1 .. b_N ([N,T,d]) used as
    sources when ``consistent`` is False (the synthetic workloads give them directly);
    when ``consistent`` is True every completed block is the sum of its own sublayer outputs,
    b_n = sum_{j in B_n} v_j, as page 2 §8 defines it.  W, G_key, G_in: [L, d] (None = ones
    for the gains).  w_final / g_final: the extra pseudo-query of the final aggregation.

    Within block n: b_n^0 = 0, b_n^i = b_n^{i-1} + v_{(n,i)}  (page 2 §8).
    """
    v = _f64(v)
    L = v.shape[0]
    N = (L + S - 1) // S
    out = BlockWalk()
    completed = [_f64(b0)]
    partial = None
    for l in range(1, L + 1):
        n, i = block_of(l, S)
        srcs = block_sources(completed, partial if i >= 2 else None)
        gk = None if G_key is None else _f64(G_key)[l - 1]
        gi = None if G_in is None else _f64(G_in)[l - 1]
        h, y, alpha = sublayer_input(srcs, _f64(W)[l - 1], gk, eps_key, gi, eps_in)
        out.h.append(h)
        out.y.append(y)
        out.alpha.append(alpha)
        out.n_sources.append(srcs.shape[0])
        out.partials.append(None if i == 1 else partial)
        # partial-sum update with this sublayer's output
        partial = v[l - 1].copy() if i == 1 else partial + v[l - 1]
        block_len = min(S, L - (n - 1) * S)
        if i == block_len:                      # block n closes
            out.closed.append(partial)
            completed.append(partial if consistent else _f64(given_blocks[n - 1]))
            partial = None
    assert len(completed) == N + 1
    fin, fin_alpha, _ = aggregate(np.stack(completed), w_final, g_final, eps_key)
    out.final, out.final_alpha = fin, fin_alpha
    return out


def block_score_count(L: int, S: int) -> int:
    """Number of (source, target) logits the block walk computes, counted from the source
    lists above (first sublayer of block n: n sources, later ones n + 1), plus the final
    aggregation over N + 1 sources."""
    total = 0
    for l in range(1, L + 1):
        n, i = block_of(l, S)
        total += n if i == 1 else n + 1
    N = (L + S - 1) // S
    return total + N + 1


# ---------------------------------------------------------------------------------------------
# Full AttnRes depth walk (page 2 §7)
# ---------------------------------------------------------------------------------------------
def full_attnres_walk(v0, v, W, G_key, G_in, w_final, g_final, eps_key: float, eps_in: float):
    """Full AttnRes: v_0 = h_1 (embedding), v_i = f_i(h_i); sublayer l reads v_0 .. v_{l-1}.

    v: [L, T, d] with v[i-1] = v_i.  The final aggregation reads v_0 .. v_L.
    Returns a BlockWalk with one 'block' per sublayer (closed = v_l).
    """
    v = _f64(v)
    L = v.shape[0]
    out = BlockWalk()
    hist = [_f64(v0)]
    for l in range(1, L + 1):
        srcs = np.stack(hist)
        gk = None if G_key is None else _f64(G_key)[l - 1]
        gi = None if G_in is None else _f64(G_in)[l - 1]
        h, y, alpha = sublayer_input(srcs, _f64(W)[l - 1], gk, eps_key, gi, eps_in)
        out.h.append(h)
        out.y.append(y)
        out.alpha.append(alpha)
        out.n_sources.append(len(hist))
        out.partials.append(None)
        out.closed.append(v[l - 1])
        hist.append(v[l - 1])
    fin, fin_alpha, _ = aggregate(np.stack(hist), w_final, g_final, eps_key)
    out.final, out.final_alpha = fin, fin_alpha
    return out


# ---------------------------------------------------------------------------------------------
# Multi-head depth attention (page 2 "Attention Residuals" note, result 4, Table 4: "Block,
# multi-head H = 16 adds depth attention heads"; no formula on the pages).  Reading: the d
# features split into H contiguous slices of d / H; each head is a complete AttnRes
# aggregation on its slice (the key is the RMSNorm of the source's slice with the slice of the
# gain, the logit uses the slice of the query, the softmax runs per head) and the heads'
# outputs are concatenated; the sublayer's input RMSNorm then normalises the whole vector.
# ---------------------------------------------------------------------------------------------
def head_slices(d: int, H: int):
    """The H contiguous feature slices of a d-vector."""
    assert d % H == 0
    dh = d // H
    return [slice(k * dh, (k + 1) * dh) for k in range(H)]


def multihead_aggregate(sources, w, gamma_key, eps: float, H: int, weights: str = "softmax",
                        key_norm: bool = True):
    """h = concat_k aggregate_k, each head k on its feature slice.  Returns (h [T,d],
    alpha [H,n,T], z [H,n,T])."""
    src = _f64(sources)
    d = src.shape[-1]
    h = np.zeros(src.shape[1:])
    al, zz = [], []
    for sl in head_slices(d, H):
        g = None if gamma_key is None else _f64(gamma_key)[sl]
        hk, ak, zk = aggregate_variant(src[..., sl], _f64(w)[sl], g, eps, weights, key_norm)
        h[..., sl] = hk
        al.append(ak)
        zz.append(zk)
    return h, np.stack(al), np.stack(zz)


def multihead_phase1(reps, W, G_key, eps: float, H: int, weights: str = "softmax",
                     key_norm: bool = True):
    """Phase 1 per head: for each query s and head k, the partition statistics of the head's
    slice (phase1, or phase1_variant under a Table 4 variant).  Returns o [S,T,d] (heads
    concatenated), m and lse [S,H,T] (lse None with sigmoid weights), alpha [S,H,T,n]."""
    reps = _f64(reps)
    S, d = np.shape(W)
    o = np.zeros((S,) + reps.shape[1:])
    m = np.zeros((S, H, reps.shape[1]))
    lse = np.zeros_like(m)
    alpha = np.zeros((S, H, reps.shape[1], reps.shape[0]))
    plain = weights == "softmax" and key_norm
    for k, sl in enumerate(head_slices(d, H)):
        gk = None if G_key is None else _f64(G_key)[:, sl]
        if plain:
            ok, mk, lk, ak = phase1(reps[..., sl], _f64(W)[:, sl], gk, eps)
        else:
            ok, mk, lk, ak = phase1_variant(reps[..., sl], _f64(W)[:, sl], gk, eps, weights,
                                            key_norm)
        o[..., sl] = ok
        m[:, k], alpha[:, k] = mk, ak
        if lk is not None:
            lse[:, k] = lk
    return o, m, (lse if weights == "softmax" else None), alpha


def multihead_merge_reference(o_A, lse_A, p, w, gamma_key, eps_key: float, gamma_in,
                              eps_in: float, H: int, weights: str = "softmax",
                              key_norm: bool = True):
    """Phase 2 per head: each head merges its slice of phase 1's result (o_A, lse_A [H,T])
    with its slice of the partial source p (merge_reference on the slice, or
    merge_reference_variant under a Table 4 variant); the heads are concatenated and the input
    RMSNorm normalises the whole h.  Returns (h, y, weights of p [H,T])."""
    o_A = _f64(o_A)
    d = o_A.shape[-1]
    h = np.zeros_like(o_A)
    ap = np.zeros((H,) + o_A.shape[:-1])
    plain = weights == "softmax" and key_norm
    for k, sl in enumerate(head_slices(d, H)):
        g = None if gamma_key is None else _f64(gamma_key)[sl]
        pk = None if p is None else _f64(p)[..., sl]
        lk = None if lse_A is None else _f64(lse_A)[k]
        if plain:
            hk, _, ak = merge_reference(o_A[..., sl], lk, pk, _f64(w)[sl], g, eps_key, None,
                                        eps_in)
        else:
            hk, _, ak = merge_reference_variant(o_A[..., sl], lk, pk, _f64(w)[sl], g, eps_key,
                                                None, eps_in, weights, key_norm)
        h[..., sl] = hk
        ap[k] = ak
    return h, rmsnorm(h, gamma_in, eps_in), ap


# ---------------------------------------------------------------------------------------------
# Backward of one aggregation (page 2 §7, the logit gradient; page 1, "梯度沿切向传播", the
# RMSNorm input gradient).  The chain rule written out; pinned against finite differences.
# ---------------------------------------------------------------------------------------------
def rmsnorm_backward(x, gamma, eps: float, g):
    """dL/dx for y = gamma ⊙ x / r_eps(x) and upstream g = dL/dy, over the last axis.  Page 1
    ("梯度沿切向传播"): the upstream gradient is first multiplied by gamma, then with
    yhat = x / r,  dL/dx = (1/r) (g' - yhat (yhat^T g') / d).  Also returns dL/dgamma = g ⊙ yhat
    (per token, not summed)."""
    x, g = _f64(x), _f64(g)
    d = x.shape[-1]
    r = rms(x, eps)[..., None]
    yhat = x / r
    gp = g if gamma is None else g * _f64(gamma)
    dx = (gp - yhat * np.sum(yhat * gp, axis=-1, keepdims=True) / d) / r
    return dx, g * yhat


@dataclass
class AggregateGrads:
    dsources: np.ndarray      # [n, T, d]  dL/dv_i (value path + key path)
    dw: np.ndarray            # [d]  dL/dw, summed over tokens
    dgamma_key: np.ndarray    # [d]  or None when gamma_key is None
    dgamma_in: np.ndarray     # [d]  or None when gamma_in is None
    du: np.ndarray            # [d]  dL/du for the folded query u = w ⊙ gamma_key
    dz: np.ndarray            # [n, T] dL/dz_i
    g_h: np.ndarray           # [T, d] dL/dh


def aggregate_backward(sources, w, gamma_key, eps_key: float, gamma_in, eps_in: float, g_y):
    """Gradients of y = RMSNorm_in(h), h = sum_i alpha_i v_i, alpha = softmax(z),
    z_i = w^T RMSNorm_key(v_i), for the upstream gradient g_y = dL/dy [T, d]:
      g_h   = RMSNorm backward of the input norm (page 1);
      dz_i  = alpha_i g_h^T (v_i - h)                     (page 2 §7);
      dv_i  = alpha_i g_h  (value path)  +  RMSNorm backward of the key norm with upstream
              dz_i w  (key path);
      dw    = sum_{t,i} dz_i RMSNorm_key(v_i);  dgamma_key = sum_{t,i} dz_i w ⊙ v_i / r_i;
      dgamma_in = sum_t g_y ⊙ h / r_h;  du = sum_{t,i} dz_i v_i / r_i."""
    v = _f64(sources)
    w = _f64(w)
    keys = rmsnorm(v, gamma_key, eps_key)
    z = np.sum(keys * w, axis=-1)
    alpha = depth_softmax(z)
    h = np.sum(alpha[..., None] * v, axis=0)
    g_h, dgi = rmsnorm_backward(h, gamma_in, eps_in, g_y)
    dz = alpha * np.sum(g_h[None] * (v - h[None]), axis=-1)
    dv = alpha[..., None] * g_h[None]
    dkey = dz[..., None] * w
    dv_key, dgk = rmsnorm_backward(v, gamma_key, eps_key, dkey)
    dv = dv + dv_key
    dw = np.sum(dz[..., None] * keys, axis=(0, 1))
    r = rms(v, eps_key)[..., None]
    du = np.sum(dz[..., None] * v / r, axis=(0, 1))
    return AggregateGrads(
        dsources=dv, dw=dw,
        dgamma_key=None if gamma_key is None else np.sum(dgk, axis=(0, 1)),
        dgamma_in=None if gamma_in is None else np.sum(dgi, axis=0),
        du=du, dz=dz, g_h=g_h)


@dataclass
class BlockGrads:
    dcompleted: np.ndarray    # [n, T, d]  dL/db_j of the block's completed sources
    dv: np.ndarray            # [S, T, d]  dL/dv_k through the block's sublayer inputs (dv_S = 0)
    dpartial: np.ndarray      # [S, T, d]  dL/dp_i of sublayer i's partial source (dp_1 = 0)
    du: np.ndarray            # [S, d]     dL/du_i, summed over tokens
    dw: np.ndarray            # [S, d]
    dgamma_key: np.ndarray    # [S, d] or None
    dgamma_in: np.ndarray     # [S, d] or None


def block_backward(completed, v, W, G_key, G_in, eps_key: float, eps_in: float, g_y):
    """Gradients of one block of Block AttnRes (page 2 §8) for the upstream gradients
    g_y[i] = dL/dy_i of its S sublayer inputs, by the chain rule composed over the block.

    Forward (the direct definition): sublayer i reads the completed sources b_0 .. b_{n-1} and,
    for i >= 2, the partial sum p_i = b^{i-1} = v_1 + ... + v_{i-1} (page 2 §8: b_n^i =
    b_n^{i-1} + f_i(h_i)); y_i = RMSNorm_in(h_i) with h_i the depth softmax over those sources.
    Backward: each sublayer's aggregation backward (``aggregate_backward``) gives the gradient
    of every source it read; the completed sources collect theirs over all S sublayers, the
    partial source of sublayer i hands its gradient to every v_k it sums (k < i), and the
    parameter gradients stay per sublayer.  v_S enters no sublayer input of the block (only
    the closed block b^S, which later blocks read), so dv_S = 0 here.

    completed [n, T, d]; v [S, T, d]; W, G_key, G_in [S, d] (gains may be None); g_y [S, T, d].
    """
    comp = _f64(completed)
    v = _f64(v)
    g_y = _f64(g_y)
    W = _f64(W)
    S = v.shape[0]
    n = comp.shape[0]
    dcomp = np.zeros_like(comp)
    dv = np.zeros_like(v)
    dpart = np.zeros_like(v)
    du = np.zeros((S, comp.shape[-1]))
    dw = np.zeros_like(du)
    dgk = None if G_key is None else np.zeros_like(du)
    dgi = None if G_in is None else np.zeros_like(du)
    partial = None
    for i in range(1, S + 1):
        srcs = block_sources(list(comp), partial)
        gk = None if G_key is None else _f64(G_key)[i - 1]
        gi = None if G_in is None else _f64(G_in)[i - 1]
        G = aggregate_backward(srcs, W[i - 1], gk, eps_key, gi, eps_in, g_y[i - 1])
        dcomp += G.dsources[:n]
        if partial is not None:
            dpart[i - 1] = G.dsources[n]
            dv[:i - 1] += G.dsources[n][None]
        du[i - 1], dw[i - 1] = G.du, G.dw
        if dgk is not None:
            dgk[i - 1] = G.dgamma_key
        if dgi is not None:
            dgi[i - 1] = G.dgamma_in
        partial = v[i - 1].copy() if partial is None else partial + v[i - 1]
    return BlockGrads(dcompleted=dcomp, dv=dv, dpartial=dpart, du=du, dw=dw, dgamma_key=dgk,
                      dgamma_in=dgi)


# ---------------------------------------------------------------------------------------------
# Full AttnRes with the grouped two-phase schedule (page 1, "静态 Query 与两阶段计算": the L
# layers fall into G scheduling groups of S = L / G; phase 1 scores the S queries of a group
# against the history in one pass and keeps the softmax statistics; phase 2 takes the layers
# of the group one by one and merges the representations the group has produced so far by
# online softmax)
# ---------------------------------------------------------------------------------------------
def merge_sources_reference(o_A, lse_A, sources_B, w, gamma_key, eps_key: float, gamma_in,
                            eps_in: float):
    """Phase 2 of one layer of a group: partition A as phase 1 hands it over (normalised o_A
    [T,d], lse_A [T]) merged with the in-group sources B ([k,T,d], k >= 0) by the partition
    merge of page 1: with m = max(lse_A, max_{i in B} z_i),
        h = (e^{lse_A - m} o_A + sum_{i in B} e^{z_i - m} v_i)
            / (e^{lse_A - m} + sum_{i in B} e^{z_i - m}).
    Returns (h, y = RMSNorm_in(h), alpha_B [k,T], weight of A [T])."""
    o_A, lse_A = _f64(o_A), _f64(lse_A)
    B = _f64(sources_B).reshape((-1,) + o_A.shape)
    if B.shape[0] == 0:
        return o_A, rmsnorm(o_A, gamma_in, eps_in), np.zeros((0,) + lse_A.shape), \
            np.ones_like(lse_A)
    z = depth_logits(B, w, gamma_key, eps_key)              # [k, T]
    m = np.maximum(lse_A, np.max(z, axis=0))
    ca = np.exp(lse_A - m)
    cb = np.exp(z - m)
    den = ca + np.sum(cb, axis=0)
    h = (ca[..., None] * o_A + np.sum(cb[..., None] * B, axis=0)) / den[..., None]
    return h, rmsnorm(h, gamma_in, eps_in), cb / den, ca / den


def grouped_full_walk(v0, v, W, G_key, G_in, S: int, eps_key: float, eps_in: float):
    """Full AttnRes (page 2 §7: layer l reads v_0 .. v_{l-1}) run by the grouped two-phase
    schedule with groups of S layers (the last group may be shorter): for group g starting at
    layer l0 + 1, phase 1 = partition_stats over A = [v_0 .. v_{l0}] for each of its queries;
    layer l0 + i then merges B = [v_{l0+1} .. v_{l0+i-1}].
    v: [L, T, d] (v[i-1] = v_i).  Returns a BlockWalk (h, y, and alpha over A followed by B)."""
    v = _f64(v)
    L = v.shape[0]
    hist = [_f64(v0)] + [v[i] for i in range(L)]
    out = BlockWalk()
    for l0 in range(0, L, S):
        A = np.stack(hist[:l0 + 1])
        for l in range(l0 + 1, min(l0 + S, L) + 1):
            gk = None if G_key is None else _f64(G_key)[l - 1]
            gi = None if G_in is None else _f64(G_in)[l - 1]
            o, m, lse, aA = partition_stats(A, _f64(W)[l - 1], gk, eps_key)
            B = np.stack(hist[l0 + 1:l]) if l > l0 + 1 else np.zeros((0,) + A.shape[1:])
            h, y, aB, wA = merge_sources_reference(o, lse, B, _f64(W)[l - 1], gk, eps_key, gi,
                                                   eps_in)
            out.h.append(h)
            out.y.append(y)
            out.alpha.append(np.concatenate([aA * wA, aB]))
            out.n_sources.append(l)
    return out


# ---------------------------------------------------------------------------------------------
# Ablation variants of the report's Table 4 (page 2 "Attention Residuals" note, result 4):
# "sigmoid weights" (no softmax competition between sources, no sum-to-1 constraint) and
# "no key RMSNorm" (the source magnitude enters the score directly).  The pages give one line
# per variant; the readings taken here:
#   * sigmoid weights: alpha_i = sigmoid(z_i) = 1 / (1 + exp(-z_i)) for every source on its
#     own, h = sum_i alpha_i v_i with no normalisation;
#   * no key RMSNorm: z_i = w^T v_i.  The key-norm gain is part of that RMSNorm, so it goes
#     with it (a caller folds no gain into the query).
# ---------------------------------------------------------------------------------------------
def depth_logits_raw(sources, w):
    """No key RMSNorm: z_i = w^T v_i for every source i.  sources [n,T,d], w [d] -> z [n,T]."""
    return np.sum(_f64(sources) * _f64(w), axis=-1)


def depth_sigmoid(z):
    """alpha_i = 1 / (1 + exp(-z_i)), each source on its own (no sum over sources)."""
    return 1.0 / (1.0 + np.exp(-_f64(z)))


def variant_logits(sources, w, gamma_key, eps: float, key_norm: bool):
    """z with the key RMSNorm (page 2 §7) or without it (Table 4 variant)."""
    if key_norm:
        return depth_logits(sources, w, gamma_key, eps)
    return depth_logits_raw(sources, w)


def variant_weights(z, weights: str):
    """softmax over the sources (page 2 §7) or the per-source sigmoid (Table 4 variant)."""
    if weights == "softmax":
        return depth_softmax(z)
    if weights == "sigmoid":
        return depth_sigmoid(z)
    raise ValueError(weights)


def aggregate_variant(sources, w, gamma_key, eps: float, weights: str = "softmax",
                      key_norm: bool = True):
    """h = sum_i alpha_i v_i with the variant's logits and weights.  Returns (h, alpha, z)."""
    src = _f64(sources)
    z = variant_logits(src, w, gamma_key, eps, key_norm)
    alpha = variant_weights(z, weights)
    return np.sum(alpha[..., None] * src, axis=0), alpha, z


def phase1_variant(reps, W, G_key, eps: float, weights: str = "softmax", key_norm: bool = True):
    """Phase 1 of one block under a variant, per query s over the partition A = reps:
    softmax weights -> (o normalised, m, lse, alpha) exactly as phase1(); sigmoid weights ->
    o = sum_{i in A} sigmoid(z_i) v_i (the partition's contribution; no statistics are needed
    to merge sums), m = max_i z_i, lse = None, alpha = sigmoid(z).
    reps: [n,T,d]; W: [S,d]; G_key: [S,d] or None.  o [S,T,d], m [S,T], alpha [S,T,n]."""
    reps = _f64(reps)
    S = np.shape(W)[0]
    o, m, lse, alpha = [], [], [], []
    for s in range(S):
        g = None if G_key is None else _f64(G_key)[s]
        z = variant_logits(reps, _f64(W)[s], g, eps, key_norm)
        mz = np.max(z, axis=0)
        if weights == "softmax":
            e = np.exp(z - mz)
            ell = np.sum(e, axis=0)
            a = e / ell
            lse.append(mz + np.log(ell))
        else:
            a = depth_sigmoid(z)
        o.append(np.sum(a[..., None] * reps, axis=0))
        m.append(mz)
        alpha.append(np.moveaxis(a, 0, -1))
    return (np.stack(o), np.stack(m), np.stack(lse) if lse else None, np.stack(alpha))


def merge_reference_variant(o_A, lse_A, p, w, gamma_key, eps_key: float, gamma_in,
                            eps_in: float, weights: str = "softmax", key_norm: bool = True):
    """Phase 2 of one sublayer under a variant, on the inputs it receives.  Softmax weights:
    the partition merge of merge_reference() with the variant's logit for p.  Sigmoid
    weights: the weights do not depend on each other, so the two partitions simply add,
    h = o_A + sigmoid(z_p) p (o_A as phase1_variant returns it).
    Returns (h, y = RMSNorm_in(h), weight of p)."""
    o_A = _f64(o_A)
    if p is None:
        return o_A, rmsnorm(o_A, gamma_in, eps_in), np.zeros(o_A.shape[:-1])
    p = _f64(p)
    z = variant_logits(p[None], w, gamma_key, eps_key, key_norm)[0]
    if weights == "sigmoid":
        a_p = depth_sigmoid(z)
        h = o_A + a_p[..., None] * p
    else:
        lse_A = _f64(lse_A)
        M = np.maximum(lse_A, z)
        ca, cb = np.exp(lse_A - M), np.exp(z - M)
        h = (ca[..., None] * o_A + cb[..., None] * p) / (ca + cb)[..., None]
        a_p = cb / (ca + cb)
    return h, rmsnorm(h, gamma_in, eps_in), a_p


def single_block_variant(completed, v, W, G_key, G_in, eps_key: float, eps_in: float,
                         weights: str = "softmax", key_norm: bool = True):
    """single_block() under a variant (direct definition for every sublayer of one block):
    returns (y per sublayer [S][T,d], h per sublayer, closed block b^S)."""
    completed = [_f64(b) for b in completed]
    v = _f64(v)
    ys, hs = [], []
    partial = None
    for i in range(1, v.shape[0] + 1):
        srcs = block_sources(completed, partial)
        gk = None if G_key is None else _f64(G_key)[i - 1]
        gi = None if G_in is None else _f64(G_in)[i - 1]
        h, _, _ = aggregate_variant(srcs, _f64(W)[i - 1], gk, eps_key, weights, key_norm)
        hs.append(h)
        ys.append(rmsnorm(h, gi, eps_in))
        partial = v[i - 1].copy() if partial is None else partial + v[i - 1]
    return ys, hs, partial


# ---------------------------------------------------------------------------------------------
# Reference values for one phase-2 call and one partial update, on given inputs
# ---------------------------------------------------------------------------------------------
def phase2_reference(reps, partial_prev, v_prev, w, gamma_key, eps_key, gamma_in, eps_in):
    """What the sublayer input is by definition when the block's completed sources are
    ``reps`` [n,T,d] and the partial source is b^{i-1} = partial_prev + v_prev (either may be
    None; both None is the first sublayer of the block, which has no partial source).

    Returns (h, y, alpha [n(+1), T], p) with p the partial source used (None if absent).
    """
    if partial_prev is None and v_prev is None:
        p = None
    elif partial_prev is None:
        p = _f64(v_prev)
    elif v_prev is None:
        p = _f64(partial_prev)
    else:
        p = _f64(partial_prev) + _f64(v_prev)
    srcs = block_sources(list(_f64(reps)), p)
    h, y, alpha = sublayer_input(srcs, w, gamma_key, eps_key, gamma_in, eps_in)
    return h, y, alpha, p


def logsumexp_bruteforce(z_row) -> float:
    """ln sum_i exp(z_i) for a short list, with math.fsum over math.exp: a slow scalar
    cross-check of the vectorised statistics (used only on tiny inputs)."""
    return math.log(math.fsum(math.exp(float(zi)) for zi in z_row))


def single_block(completed, v, W, G_key, G_in, w_final, g_final, eps_key: float,
                 eps_in: float) -> BlockWalk:
    """One block over the given completed sources b_0 .. b_{n-1} ([n, T, d]): sublayer i
    (1-based) reads the completed sources plus the partial b^{i-1} for i >= 2 (page 2 §8),
    the block closes with b^S = sum of its outputs, and the final aggregation reads
    b_0 .. b_{n-1}, b^S with the extra query (page 2 §8, last sentence).
    v: [S, T, d]; W, G_key, G_in: [S, d] (None = ones for the gains)."""
    completed = [_f64(b) for b in completed]
    v = _f64(v)
    out = BlockWalk()
    partial = None
    for i in range(1, v.shape[0] + 1):
        srcs = block_sources(completed, partial)
        gk = None if G_key is None else _f64(G_key)[i - 1]
        gi = None if G_in is None else _f64(G_in)[i - 1]
        h, y, alpha = sublayer_input(srcs, _f64(W)[i - 1], gk, eps_key, gi, eps_in)
        out.h.append(h)
        out.y.append(y)
        out.alpha.append(alpha)
        out.n_sources.append(srcs.shape[0])
        out.partials.append(partial)
        partial = v[i - 1].copy() if partial is None else partial + v[i - 1]
    out.closed.append(partial)
    fin, fin_alpha, _ = aggregate(np.stack(completed + [partial]), w_final, g_final, eps_key)
    out.final, out.final_alpha = fin, fin_alpha
    return out


def merge_reference(o_A, lse_A, p, w, gamma_key, eps_key: float, gamma_in, eps_in: float):
    """Phase 2 of one sublayer on the inputs it receives: the statistics of partition A as
    phase 1 hands them over (normalised o_A [T,d], lse_A [T]) and the partial source p [T,d]
    (partition B = {p}, or None when the block has no partial yet).

    The pages merge two partitions X in {A, B} from (m_X, l_X, o_X unnormalised) with the
    common max m (page 1 two-phase section; page 2 §10).  A normalised o_A with its
    log-sum-exp carries the same information: e^{m_A - m} o_A,unnorm = e^{lse_A - m} o_A and
    e^{m_A - m} l_A = e^{lse_A - m}.  Partition B has m_B = z_p, l_B = 1, o_B = p, so
        M = max(lse_A, z_p),  h = (e^{lse_A - M} o_A + e^{z_p - M} p) / (e^{lse_A - M} + e^{z_p - M}).
    Returns (h, y = RMSNorm_in(h), weight of p)."""
    o_A = _f64(o_A)
    lse_A = _f64(lse_A)
    if p is None:
        h = o_A
        a_p = np.zeros(o_A.shape[:-1])
    else:
        p = _f64(p)
        z = depth_logits(p[None], w, gamma_key, eps_key)[0]
        M = np.maximum(lse_A, z)
        ca = np.exp(lse_A - M)
        cb = np.exp(z - M)
        h = (ca[..., None] * o_A + cb[..., None] * p) / (ca + cb)[..., None]
        a_p = cb / (ca + cb)
    return h, rmsnorm(h, gamma_in, eps_in), a_p
