"""Run Block AttnRes blocks on the GPU through the schedule the bench times, and check every
call against the oracle on sampled token rows.

Two checks per phase-2 call:
  per call    the oracle is given exactly what the call received (the phase-1 row block o_l
              and lse_l, the partial and v_prev, restricted to the sampled rows) and applies
              the pages' merge (``merge_reference``); gate: parity_util.TOL;
  end to end  the direct softmax over all the block's sources (``phase2_reference``); gate:
              the per-call tolerance plus the derived bound for the bf16 storage of o_l
              (parity_util.check_two_phase).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.attnres_oracle as O
from parity_util import TOL, check_close, check_outputs, check_two_phase, to64


class BlockChecker:
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
        self.o_gpu = self.lse_gpu = None
        self.oA = None

    def snap(self, t):
        return None if t is None else to64(t[self.rows])

    def phase1_done(self, o, lse):
        """Snapshot the phase-1 outputs (rows) and check them against the oracle."""
        self.o_gpu = to64(o[:, self.rows])
        self.lse_gpu = to64(lse[:, 0, self.rows])    # one head
        oo, _, olse, _ = O.phase1(self.reps64, self.W, self.Gk, self.eps)
        self.oA = oo
        check_outputs(self.o_gpu, oo, self.dt, "phase-1 o")
        check_close(self.lse_gpu, olse, TOL[self.dt]["stat"], "phase-1 lse")

    def before(self, i, args):
        """on_call hook: remember the exact inputs of phase-2 call i."""
        self.pending = (i, self.snap(args["partial"]), self.snap(args["v_prev"]))

    def after(self, i, y):
        j, part, vprev = self.pending
        assert j == i
        if part is None and vprev is None:
            p = None
        else:
            p = (0.0 if part is None else part) + (0.0 if vprev is None else vprev)
        g_in = None if self.Gin is None else self.Gin[i - 1]
        yg = y[self.rows]
        _, y_m, _ = O.merge_reference(self.o_gpu[i - 1], self.lse_gpu[i - 1], p, self.W[i - 1],
                                      self.Gk[i - 1], self.eps, g_in, self.eps)
        self.report[f"y_{i}"] = check_outputs(yg, y_m, self.dt, f"y_{i} (per call)")
        h_d, y_d, a_d, _ = O.phase2_reference(self.reps64, part, vprev, self.W[i - 1],
                                              self.Gk[i - 1], self.eps, g_in, self.eps)
        w_A = 1.0 - (a_d[-1] if p is not None else 0.0)
        self.report[f"y_{i} direct"] = check_two_phase(yg, y_d, self.oA[i - 1], w_A,
                                                       O.rms(h_d, self.eps), g_in, self.dt,
                                                       f"y_{i} (two-phase vs direct)")
        self.calls += 1


def run_checked_block(runner, reps, U, W, Gk, Gin, vbuf, close_out, dtype, rows, eps=1e-6,
                      report=None, U_split=None):
    """Run one block with per-call checks.  vbuf: [S, T, d] stand-in sublayer outputs;
    U_split: the queries' bf16 split (tensor-core phase 1) or None."""
    chk = BlockChecker(reps, W, Gk, Gin, dtype, rows, eps, report)
    S = U.shape[0]

    def sublayer(i, y):
        chk.after(i, y)
        return vbuf[i - 1]

    def on_call(i, args):
        if i == 1:
            chk.phase1_done(runner.o[:S], runner.lse[:S])
        chk.before(i, args)

    runner.run_block(reps, U, Gin, sublayer, close_out, eps, eps, on_call=on_call,
                     U_split=U_split)
    torch.cuda.synchronize()
    # the close is exactly round(b^{S-1} + v_S) of the stored tensors
    if S >= 2:
        prev = runner.last_partial      # b^{S-1}: v_1 when S == 2
        want = (prev[rows].float() + vbuf[S - 1][rows].float()).to(close_out.dtype)
        assert torch.equal(close_out[rows], want), "block close"
    assert chk.calls == S
    return chk
