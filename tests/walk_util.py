"""Run Block AttnRes blocks on the GPU through the schedule the bench times, and check every
call against the oracle on sampled token rows (per-call parity: the oracle gets the exact
tensors each GPU call received, restricted to the sampled rows)."""
from __future__ import annotations

import numpy as np
import torch

import oracle.attnres_oracle as O
from parity_util import TOL, check_close, check_outputs, to64


class BlockChecker:
    """Checks one block run by ``BlockRunner.run_block`` on rows ``rows``."""

    def __init__(self, reps, W, Gk, Gin, dtype: str, rows, eps=1e-6, report=None):
        self.rows = rows
        self.reps64 = to64(reps[:, rows])          # [n, k, d]
        self.W, self.Gk = to64(W), to64(Gk)
        self.Gin = None if Gin is None else to64(Gin)
        self.dt = dtype
        self.eps = eps
        self.pending = None
        self.report = {} if report is None else report
        self.calls = 0

    def snap(self, t):
        return None if t is None else to64(t[self.rows])

    def before(self, i, args):
        """on_call hook: remember the exact inputs of phase-2 call i."""
        self.pending = (i, self.snap(args["partial"]), self.snap(args["v_prev"]))

    def after(self, i, y):
        """Check the y_i just written against the oracle on the same inputs."""
        j, part, vprev = self.pending
        assert j == i
        g_in = None if self.Gin is None else self.Gin[i - 1]
        _, y_o, _, _ = O.phase2_reference(self.reps64, part, vprev, self.W[i - 1],
                                          self.Gk[i - 1], self.eps, g_in, self.eps)
        rel = check_outputs(y[self.rows], y_o, self.dt, f"y_{i}")
        self.report[f"y_{i}"] = rel
        self.calls += 1

    def check_phase1(self, o, lse):
        oo, _, olse, _ = O.phase1(self.reps64, self.W, self.Gk, self.eps)
        check_outputs(o[:, self.rows], oo, self.dt, "phase-1 o")
        check_close(lse[:, self.rows], olse, TOL[self.dt]["stat"], "phase-1 lse")


def run_checked_block(runner, reps, U, W, Gk, Gin, vbuf, close_out, dtype, rows, eps=1e-6,
                      report=None):
    """Run one block with per-call checks.  vbuf: [S, T, d] stand-in sublayer outputs."""
    chk = BlockChecker(reps, W, Gk, Gin, dtype, rows, eps, report)
    S = U.shape[0]
    last_partial = {}

    def sublayer(i, y):
        chk.after(i, y)
        return vbuf[i - 1]

    def on_call(i, args):
        chk.before(i, args)
        last_partial["p"] = args["partial"]

    runner.run_block(reps, U, Gin, sublayer, close_out, eps, eps, on_call=on_call)
    torch.cuda.synchronize()
    chk.check_phase1(runner.o[:S], runner.lse[:S])
    # the close is exactly round(b^{S-1} + v_S) of the stored tensors
    if S >= 2:
        # b^{S-1} is runner.partial (S >= 3) or v_1 (S == 2); both still hold it
        prev = vbuf[0] if S == 2 else runner.partial
        want = (prev[rows].float() + vbuf[S - 1][rows].float()).to(close_out.dtype)
        assert torch.equal(close_out[rows], want), "block close"
    assert chk.calls == S
    return chk
