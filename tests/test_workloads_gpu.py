"""The five workloads on the GPU against the oracle.

  tiny_block_f32       every element of every sublayer, Block walk vs the oracle walk
                       (given and consistent block sums), plus the zero-query model
  prefill_chunk_bf16   T = 16384, d = 7168, 186 sublayers: per-call parity on sampled rows
  full_attnres_bf16    T = 8192, d = 2048, 54 sublayers: the direct path per sublayer, and
                       the Block path with one sublayer per block equal to it (N = L)
  decode_bf16          T = 256, d = 7168, 186 sublayers: per-call parity on sampled rows
  longctx_prefill_bf16 the bench step (8 chunks of 16384 tokens over a [10, 131072, 7168]
                       cache) in the launch configuration the bench times, sampled rows
"""
import numpy as np
import pytest
import torch

import depth_wise_softmax_block_b300 as ar
from depth_wise_softmax_block_b300 import build as B
from depth_wise_softmax_block_b300.schedule import BlockRunner, final_aggregation
import oracle.attnres_oracle as O
from parity_util import TOL, check_close, check_outputs, record_parity, sample_rows, to64
from synth import inputs as I
from walk_util import run_checked_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.build()
    ar.library()
    return torch.device("cuda:0")


def folded(P, dev):
    """Folded queries U [L, d], the final query, and U's bf16 hi/lo split [2L, d] (which the
    bf16 walks pass to phase 1, as the bench does)."""
    U = torch.empty_like(P.W)
    U_split = torch.empty((2 * U.shape[0], U.shape[1]), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(P.W, P.G_key, U, U_split)
    uf = torch.empty_like(P.w_final)
    ar.attnres_query_prep(P.w_final.view(1, -1), P.g_final.view(1, -1), uf.view(1, -1))
    return U, uf, U_split


def gpu_block_walk(wl, reps, v, P, U, uf, dev, consistent=False, U_split=None):
    """The whole depth on the GPU.  reps: [N+1, T, d] (slot 0 = b_0, given blocks after);
    v: [L, T, d].  Returns (ys [L, T, d], final [T, d], closed blocks)."""
    T, d, L, S = wl.T, wl.d, wl.L, wl.S
    N = wl.n_blocks
    runner = BlockRunner(T, d, S, wl.torch_dtype, dev, keep_y=True)
    ys = torch.empty((L, T, d), dtype=wl.torch_dtype, device=dev)
    src = reps.clone()
    closed = torch.empty((N, T, d), dtype=wl.torch_dtype, device=dev)
    for n in range(1, N + 1):
        l0 = (n - 1) * S
        Sn = min(S, L - l0)

        def sublayer(i, y, l0=l0):
            ys[l0 + i - 1].copy_(y)
            return v[l0 + i - 1]

        us = None if U_split is None else U_split[2 * l0:2 * (l0 + Sn)]
        runner.run_block(src[:n], U[l0:l0 + Sn], P.G_in[l0:l0 + Sn], sublayer, closed[n - 1],
                         U_split=us)
        if consistent:
            src[n].copy_(closed[n - 1])
    fin = torch.empty((T, d), dtype=wl.torch_dtype, device=dev)
    final_aggregation(src[:N + 1], uf, fin)
    torch.cuda.synchronize()
    return ys, fin, closed


@pytest.mark.parametrize("zero", [False, True])
@pytest.mark.parametrize("consistent", [False, True])
def test_tiny_block_f32_every_element(dev, zero, consistent):
    wl = I.TINY_BLOCK_F32
    N = wl.n_blocks
    reps = I.make_reps(wl, N + 1, dev)
    v = I.make_outputs(wl, 1, wl.L, dev)
    P = I.block_params(wl, dev, zero_queries=zero)
    U, uf, _ = folded(P, dev)
    ys, fin, closed = gpu_block_walk(wl, reps, v, P, U, uf, dev, consistent)
    ow = O.block_attnres_walk(to64(reps[0]), to64(reps[1:]), to64(v), wl.S, to64(P.W),
                              to64(P.G_key), to64(P.G_in), to64(P.w_final), to64(P.g_final),
                              wl.eps, wl.eps, consistent=consistent)
    for l in range(wl.L):
        check_outputs(ys[l], ow.y[l], "f32", f"y_{l + 1}")
    for n in range(N):
        check_outputs(closed[n], ow.closed[n], "f32", f"b_{n + 1}")
    check_outputs(fin, ow.final, "f32", "final aggregation")


def _block_walk_checked(wl, dev, rows_k, report, o_dtype=None):
    T, d, L, S = wl.T, wl.d, wl.L, wl.S
    N = wl.n_blocks
    rows = sample_rows(T, rows_k, seed=wl.seed)
    reps = I.make_reps(wl, N + 1, dev)
    P = I.block_params(wl, dev)
    U, uf, U_split = folded(P, dev)
    runner = BlockRunner(T, d, S, wl.torch_dtype, dev, o_dtype=o_dtype, extra_outputs=True)
    vbuf = torch.empty((S, T, d), dtype=wl.torch_dtype, device=dev)
    close = torch.empty((T, d), dtype=wl.torch_dtype, device=dev)
    for n in range(1, N + 1):
        l0 = (n - 1) * S
        Sn = min(S, L - l0)
        for i in range(Sn):
            I.fill_sublayer_output(vbuf[i], l0 + i + 1, wl.seed)
        run_checked_block(runner, reps[:n], U[l0:l0 + Sn], P.W[l0:l0 + Sn],
                          P.G_key[l0:l0 + Sn], P.G_in[l0:l0 + Sn], vbuf[:Sn], close, "bf16",
                          rows, report=report, U_split=U_split[2 * l0:2 * (l0 + Sn)])
    fin = torch.empty((T, d), dtype=wl.torch_dtype, device=dev)
    final_aggregation(reps[:N + 1], uf, fin)
    torch.cuda.synchronize()
    want, _, _ = O.aggregate(to64(reps[:N + 1, rows]), to64(P.w_final), to64(P.g_final), wl.eps)
    check_outputs(fin[rows], want, "bf16", "final aggregation", report)


# Phase 1's o stored in bf16 (the production path the bench times) or in fp32 (ATTNRES_O_F32:
# no rounding between the phases, so every output meets the plain gate against the direct
# definition).
O_STORE = {"o_bf16": None, "o_f32": torch.float32}


def _summary(report, wl_name, ostore):
    """Literal max |gpu - oracle| / RMS per gate kind over the walk (printed; the numbers in
    the design notes come from this line)."""
    kinds = {}
    for k, v in report.items():
        kind = k.split(" ", 1)[1] if k[:2] in ("y_", "h_") else k
        kinds[kind] = max(kinds.get(kind, 0.0), v)
    items = ", ".join(f"{k}: {v:.3e}" for k, v in sorted(kinds.items()))
    print(f"PARITY {wl_name} {ostore}: {items}")
    record_parity(f"{wl_name} {ostore}", kinds)


@pytest.mark.parametrize("ostore", sorted(O_STORE))
def test_prefill_chunk_bf16_sampled(dev, ostore):
    report = {}
    _block_walk_checked(I.PREFILL_CHUNK_BF16, dev, 40, report, O_STORE[ostore])
    assert len([k for k in report if k.startswith("y_")]) > 0
    _summary(report, I.PREFILL_CHUNK_BF16.name, ostore)


@pytest.mark.parametrize("ostore", sorted(O_STORE))
def test_decode_bf16_sampled(dev, ostore):
    report = {}
    _block_walk_checked(I.DECODE_BF16, dev, 24, report, O_STORE[ostore])
    _summary(report, I.DECODE_BF16.name, ostore)


def test_full_attnres_bf16(dev):
    wl = I.FULL_INTERP_BF16
    T, d, L = wl.T, wl.d, wl.L
    rows = sample_rows(T, 32, seed=wl.seed)
    hist = torch.empty((L + 1, T, d), dtype=torch.bfloat16, device=dev)
    I.fill_sublayer_output(hist[0], 0, wl.seed, 0.0)               # v_0 ~ N(0, 1)
    for l in range(1, L + 1):
        I.fill_sublayer_output(hist[l], l, wl.seed, wl.v_growth)    # v_l ~ N(0,1)(1 + 0.05 l)
    P = I.block_params(wl, dev)
    U, uf, _ = folded(P, dev)
    y_full = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    h_full = torch.empty_like(y_full)
    o = torch.empty((1, T, d), dtype=torch.float32, device=dev)      # ATTNRES_O_F32
    lse = torch.empty((1, T), device=dev)
    y_blk = torch.empty_like(y_full)
    h64 = to64(hist[:, rows])
    for l in range(1, L + 1):
        srcs = [hist[j] for j in range(l)]
        ar.attnres_full_reference_path(srcs, U[l - 1], P.G_in[l - 1], h_out=h_full, y_out=y_full)
        # Block AttnRes with one sublayer per block: phase 1 over the same l sources, then
        # phase 2 without a partial source
        ar.attnres_phase1(hist[:l], U[l - 1:l], o, lse_out=lse)
        ar.attnres_phase2_merge(o[0], lse[0], None, None, None, U[l - 1], P.G_in[l - 1], y_blk)
        if l in (1, 2, 9, 27, 54) or l % 13 == 0:
            _, y_o, _ = O.sublayer_input(h64[:l], to64(P.W[l - 1]), to64(P.G_key[l - 1]), wl.eps,
                                         to64(P.G_in[l - 1]), wl.eps)
            check_outputs(y_full[rows], y_o, "bf16", f"full y_{l}")
            check_outputs(y_blk[rows], y_o, "bf16", f"block(N=L) y_{l}")
        # the two GPU paths agree everywhere within the bf16 tolerance
        check_outputs(y_blk, y_full, "bf16", f"block(N=L) vs full, l={l}")
    fin = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    final_aggregation(hist, uf, fin)
    torch.cuda.synchronize()
    want, _, _ = O.aggregate(h64, to64(P.w_final), to64(P.g_final), wl.eps)
    check_outputs(fin[rows], want, "bf16", "final aggregation (55 sources)")


@pytest.mark.parametrize("ostore", sorted(O_STORE))
def test_longctx_prefill_bench_step_sampled(dev, ostore):
    """The step the bench times, checked on sampled rows of every chunk: the same calls in the
    same launch configuration, through a runner that also writes h and the partial's weight
    (o_bf16: the bench's own o storage; o_f32: o stored in fp32).  With o in bf16 the timed
    step itself (no hooks, no extra outputs) then reproduces the checked outputs bit for bit."""
    import bench
    from depth_wise_softmax_block_b300.schedule import final_aggregation
    wl = I.LONGCTX_PREFILL_BF16
    st = bench.LongContextStep(wl, dev)
    chk_runner = BlockRunner(wl.chunk, wl.d, wl.S, torch.bfloat16, dev, o_dtype=O_STORE[ostore],
                             extra_outputs=True)
    rows = sample_rows(wl.chunk, 12, seed=1)
    report = {}
    st.prep()
    for c in range(st.nchunks):
        reps_c, close_c, all_c, out_c = st.chunk_views(c)
        rep = {}
        run_checked_block(chk_runner, reps_c, st.U, st.P.W, st.P.G_key, st.P.G_in, st.vbuf,
                          close_c, "bf16", rows, wl.eps, rep, U_split=st.U_split)
        final_aggregation(all_c, st.uf[0], out_c, wl.eps)
        torch.cuda.synchronize()
        want, _, _ = O.aggregate(to64(all_c[:, rows]), to64(st.P.w_final), to64(st.P.g_final),
                                 wl.eps)
        check_outputs(out_c[rows], want, "bf16", f"final chunk {c}", rep)
        report.update({f"{k} chunk {c}": v for k, v in rep.items()})
    assert len([k for k in report if k[:2] in ("y_", "h_")]) == st.nchunks * 8 * wl.S
    _summary({k.rsplit(" chunk ", 1)[0]: v for k, v in report.items()}, wl.name, ostore)
    if ostore == "o_bf16":
        # the timed step itself (no hooks) reproduces the checked outputs bit for bit
        ref = st.out.clone()
        st.run()
        torch.cuda.synchronize()
        assert torch.equal(st.out, ref)


def test_depth_walk_cuda_graph_replay_matches_eager(dev):
    """The block schedule captured as one CUDA graph (the library launches on the caller's
    stream and allocates nothing) replays bit for bit what the eager walk computes: 256 tokens,
    two blocks of 24 sublayers, bf16, tensor-core phase 1."""
    T, d, S, L = 256, 1024, 24, 48
    N = L // S
    reps = torch.empty((N + 1, T, d), dtype=torch.bfloat16, device=dev)
    for j in range(N + 1):
        I.fill_block_rep(reps[j], j, 77)
    W = I.queries(L, d, 77, "w", dev)
    G = I.gains(L, d, 0.02, 77, "g", dev)
    Gi = I.gains(L, d, 0.02, 77, "gi", dev)
    U = torch.empty_like(W)
    Us = torch.empty((2 * L, d), dtype=torch.bfloat16, device=dev)
    ar.attnres_query_prep(W, G, U, Us)
    vbuf = torch.stack([I.normal((T, d), 1.0, 77, f"v{i}", dev, torch.bfloat16) for i in range(S)])
    runner = BlockRunner(T, d, S, torch.bfloat16, dev, keep_y=True)
    fin = torch.empty((T, d), dtype=torch.bfloat16, device=dev)

    def walk():
        for n in range(1, N + 1):
            l0 = (n - 1) * S
            runner.run_block(reps[:n], U[l0:l0 + S], Gi[l0:l0 + S], lambda i, y: vbuf[i - 1],
                             reps[n], U_split=Us[2 * l0:2 * (l0 + S)])
        final_aggregation(reps[:N + 1], U[0], fin)

    walk()
    torch.cuda.synchronize()
    eager = (fin.clone(), runner.y.clone(), reps.clone())
    fin.zero_()
    runner.y.zero_()
    reps[1:].zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        walk()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        walk()
    fin.zero_()
    runner.y.zero_()
    reps[1:].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(fin, eager[0]), "final aggregation differs under graph replay"
    assert torch.equal(runner.y, eager[1]), "sublayer inputs differ under graph replay"
    assert torch.equal(reps, eager[2]), "block closes differ under graph replay"
