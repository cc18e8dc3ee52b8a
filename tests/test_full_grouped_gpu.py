"""Full AttnRes by the grouped two-phase schedule on the GPU ("Attention Residuals 阅读补充",
section "静态 Query 与两阶段计算"): phase 1 over the history for a group's queries, then the
multi-source phase-2 merge (attnres_phase2_merge_sources) layer by layer, against the fp64
oracle.  Each call is checked against the oracle's merge fed the call's exact inputs (o, lse
as stored), and each layer end to end against the direct Full AttnRes definition."""
import numpy as np
import pytest
import torch

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B
from depth_wise_softmax_block_b300.schedule import FullGroupedRunner
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


def _setup(T, d, L, dtype, dev, seed):
    hist = torch.empty((L + 1, T, d), dtype=dtype, device=dev)
    hist[0].copy_(I.normal((T, d), 1.0, seed, "v0", dev, dtype))
    v = torch.stack([I.normal((T, d), 1.0 + 0.05 * l, seed, f"v{l}", dev, dtype)
                     for l in range(1, L + 1)])
    W = I.queries(L, d, seed, "w", dev)
    Gk = I.gains(L, d, 0.02, seed, "gk", dev)
    Gi = I.gains(L, d, 0.02, seed, "gi", dev)
    U = torch.empty_like(W)
    Us = torch.empty((2 * L, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, Gk, U, Us)
    return hist, v, W, Gk, Gi, U, Us


def _run(hist, v, U, Gi, S, dtype, split, snap=None, o_dtype=None):
    L, T, d = v.shape
    runner = FullGroupedRunner(T, d, S, dtype, hist.device, o_dtype=o_dtype)
    ys = torch.empty((L, T, d), dtype=dtype, device=hist.device)

    def sub(l, y):
        if snap is not None:   # the stored phase-1 result this layer merged from
            i = (l - 1) % S
            snap[l] = (runner.o[i].clone(), runner.lse[i, 0].clone())   # one head
        return v[l - 1]

    runner.run(hist, U, Gi, ys, sub, EPS, EPS, U_split=split)
    torch.cuda.synchronize()
    return ys


@pytest.mark.parametrize("S", [1, 3, 8])
def test_grouped_full_f32_every_element(dev, S):
    T, d, L = 24, 128, 8
    hist, v, W, Gk, Gi, U, _ = _setup(T, d, L, torch.float32, dev, 11)
    ys = _run(hist, v, U, Gi, S, torch.float32, None)
    walk = O.full_attnres_walk(to64(hist[0]), to64(v), to64(W), to64(Gk), to64(Gi), None, None,
                               EPS, EPS)
    for l in range(L):
        check_outputs(ys[l], walk.y[l], "f32", f"y_{l + 1} (S={S})")


@pytest.mark.parametrize("T,d,L,S,rows_k,split", [(40, 2048, 20, 8, 0, True),
                                                  (8192, 2048, 54, 8, 12, True),
                                                  (8192, 2048, 54, 16, 12, False)])
@pytest.mark.parametrize("ostore", ["o_bf16", "o_f32"])
def test_grouped_full_bf16(dev, T, d, L, S, rows_k, split, ostore):
    """bf16: every call against the merge of its own stored inputs; every layer against the
    direct definition, at the output gate when phase 1's o is stored in fp32 (ATTNRES_O_F32)
    and with the two-phase storage term when it is stored in bf16 (the production path)."""
    hist, v, W, Gk, Gi, U, Us = _setup(T, d, L, torch.bfloat16, dev, 12)
    snap = {}
    o32 = ostore == "o_f32"
    ys = _run(hist, v, U, Gi, S, torch.bfloat16, Us if split else None, snap,
              torch.float32 if o32 else None)
    rows = np.arange(T) if rows_k == 0 else np.unique(
        np.concatenate([[0, T - 1], np.random.default_rng(5).integers(0, T, rows_k)]))
    h64 = to64(hist[:, rows])
    W64, Gk64, Gi64 = to64(W), to64(Gk), to64(Gi)
    for l in range(1, L + 1):
        l0 = (l - 1) // S * S
        o_g, lse_g = snap[l]
        B64 = h64[l0 + 1:l]
        h_m, y_m, _, _ = O.merge_sources_reference(to64(o_g[rows]), to64(lse_g[rows]), B64,
                                                   W64[l - 1], Gk64[l - 1], EPS, Gi64[l - 1],
                                                   EPS)
        check_outputs(ys[l - 1][rows], y_m, "bf16", f"y_{l} per call")
        # end to end: direct softmax over v_0 .. v_{l-1}
        h_d, y_d, a_d = O.sublayer_input(h64[:l], W64[l - 1], Gk64[l - 1], EPS, Gi64[l - 1],
                                         EPS)
        if o32:
            check_outputs(ys[l - 1][rows], y_d, "bf16", f"y_{l} (vs direct)")
        else:
            oA, _, _, _ = O.partition_stats(h64[:l0 + 1], W64[l - 1], Gk64[l - 1], EPS)
            wA = np.sum(a_d[:l0 + 1], axis=0)
            check_two_phase(ys[l - 1][rows], y_d, oA, wA, O.rms(h_d, EPS), Gi64[l - 1], "bf16",
                            f"y_{l} (two-phase vs direct)")


def test_merge_sources_weights_and_empty(dev):
    """k = 0 returns o_l itself; the in-group weights match the oracle's."""
    T, d = 33, 512
    g = torch.Generator(device="cpu").manual_seed(3)
    o = torch.randn((T, d), generator=g).to(dev)
    lse = (torch.randn((T,), generator=g) + 1.0).to(dev)
    srcs = [torch.randn((T, d), generator=g).to(dev) * (1 + j) for j in range(4)]
    u = (torch.randn((d,), generator=g) / d ** 0.5).to(dev)
    h = torch.empty_like(o)
    alpha = torch.empty((T, 4), device=dev)
    ar.attnres_phase2_merge_sources(o, lse, [], u, None, h_out=h)
    torch.cuda.synchronize()
    assert torch.equal(h, o)
    ar.attnres_phase2_merge_sources(o, lse, srcs, u, None, h_out=h, alpha_out=alpha, eps_key=EPS)
    torch.cuda.synchronize()
    hh, _, aB, _ = O.merge_sources_reference(to64(o), to64(lse), np.stack([to64(s) for s in srcs]),
                                             to64(u), None, EPS, None, EPS)
    check_outputs(h, hh, "f32", "h")
    check_close(alpha, aB.T, TOL["f32"]["weight"], "in-group weights")
