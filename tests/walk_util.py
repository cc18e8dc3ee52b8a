"""Run Block AttnRes blocks on the GPU through the schedule the bench times, and check every
call against the oracle on sampled token rows.

Checks per phase-2 call (the runner writes h and the partial's weight besides y):
  per call    the oracle is given exactly what the call received (the phase-1 row block o_l
              and lse_l, the partial and v_prev, restricted to the sampled rows) and applies
              the pages' merge (``merge_reference``): y and h, parity_util's output gate;
  end to end  the direct softmax over all the block's sources (``phase2_reference``):
                - the weight of the partial source, at the weight tolerance (it does not
                  depend on how o_l is stored);
                - y and h: with phase 1's o stored in fp32 (ATTNRES_O_F32) at the plain
                  output gate; with o stored in bf16 (the production path) at the output gate
                  plus the derived bound for that storage (parity_util.check_two_phase).
"""
from __future__ import annotations

import torch

import oracle.attnres_oracle as O
from parity_util import LAST, TOL, check_close, check_outputs, check_two_phase, to64


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
        self.o_stored = None
        self.oA = None

    def put(self, key, rel):
        """Keep the largest literal error seen under ``key`` (blocks reuse the call keys), and
        for the output checks also the largest distance from the correctly rounded result."""
        self.report[key] = max(self.report.get(key, 0.0), rel)
        if not key.startswith("partial weight"):
            k2 = key + " [vs rne(oracle)]"
            self.report[k2] = max(self.report.get(k2, 0.0), LAST["vs_rounded"])

    def snap(self, t):
        return None if t is None else to64(t[self.rows])

    def phase1_done(self, o, lse):
        """Snapshot the phase-1 outputs (rows) and check them against the oracle."""
        self.o_stored = "bf16" if o.dtype == torch.bfloat16 else "f32"
        self.o_gpu = to64(o[:, self.rows])
        self.lse_gpu = to64(lse[:, 0, self.rows])    # one head
        oo, _, olse, _ = O.phase1(self.reps64, self.W, self.Gk, self.eps)
        self.oA = oo
        self.put(f"phase-1 o ({self.o_stored})",
                 check_outputs(self.o_gpu, oo, self.dt, f"phase-1 o ({self.o_stored})",
                               stored=self.o_stored))
        check_close(self.lse_gpu, olse, TOL[self.dt]["stat"], "phase-1 lse")

    def before(self, i, args):
        """on_call hook: remember the exact inputs of phase-2 call i."""
        self.pending = (i, self.snap(args["partial"]), self.snap(args["v_prev"]))

    def after(self, i, y, h, alpha_p):
        """Called right after phase-2 call i with its outputs y, h ([T, d]) and the partial's
        weight alpha_p ([1, T]; not written for i = 1)."""
        j, part, vprev = self.pending
        assert j == i
        if part is None and vprev is None:
            p = None
        else:
            p = (0.0 if part is None else part) + (0.0 if vprev is None else vprev)
        g_in = None if self.Gin is None else self.Gin[i - 1]
        yg, hg = y[self.rows], h[self.rows]
        tag = f"o {self.o_stored}"
        # per call: the pages' merge on the inputs the call received
        h_m, y_m, a_m = O.merge_reference(self.o_gpu[i - 1], self.lse_gpu[i - 1], p,
                                          self.W[i - 1], self.Gk[i - 1], self.eps, g_in, self.eps)
        self.put(f"y_{i} per call ({tag})", check_outputs(yg, y_m, self.dt, f"y_{i} (per call)"))
        self.put(f"h_{i} per call ({tag})", check_outputs(hg, h_m, self.dt, f"h_{i} (per call)"))
        # end to end: the direct softmax over all the sources of the sublayer
        h_d, y_d, a_d, _ = O.phase2_reference(self.reps64, part, vprev, self.W[i - 1],
                                              self.Gk[i - 1], self.eps, g_in, self.eps)
        if p is not None:
            self.put("partial weight abs err (vs direct)",
                     check_close(alpha_p[0, self.rows], a_d[-1], TOL[self.dt]["weight"],
                                 f"weight of the partial source, call {i} (vs direct)"))
        if self.o_stored == "f32" or self.dt == "f32":
            self.put(f"y_{i} direct ({tag})",
                     check_outputs(yg, y_d, self.dt, f"y_{i} (vs direct)"))
            self.put(f"h_{i} direct ({tag})",
                     check_outputs(hg, h_d, self.dt, f"h_{i} (vs direct)"))
        else:
            w_A = 1.0 - (a_d[-1] if p is not None else 0.0)
            rh = O.rms(h_d, self.eps)
            self.put(f"y_{i} direct two-phase bound ({tag})", check_two_phase(
                yg, y_d, self.oA[i - 1], w_A, rh, g_in, self.dt, f"y_{i} (two-phase vs direct)"))
            self.put(f"h_{i} direct two-phase bound ({tag})", check_two_phase(
                hg, h_d, self.oA[i - 1], w_A, rh, g_in, self.dt, f"h_{i} (two-phase vs direct)",
                h_only=True))
        self.calls += 1


def partial_sources(v, dtype):
    """The partial-sum sources of one block's phase-2 calls as the GPU forms them, in fp64:
    [None, v_1, b^1 + v_2, b^2 + v_3, ...] where the stored partials are b^1 = v_1 and
    b^k = round(b^{k-1} + v_k) (the fp32 sum of the two stored values rounded to the I/O type
    ``dtype``); and the stored close b^S.  v: [S, T, d] tensor of the I/O type."""
    vc = v.float().cpu()
    S = vc.shape[0]
    ps, stored = [None], None
    for i in range(2, S + 1):
        if i == 2:
            ps.append(vc[0].double().numpy())
            stored = vc[0].to(dtype)
        else:
            ps.append(stored.double().numpy() + vc[i - 2].double().numpy())
            stored = (stored.float() + vc[i - 2]).to(dtype)
    close = vc[0].to(dtype) if S == 1 else (stored.float() + vc[S - 1]).to(dtype)
    return ps, close


def run_checked_block(runner, reps, U, W, Gk, Gin, vbuf, close_out, dtype, rows, eps=1e-6,
                      report=None, U_split=None):
    """Run one block with per-call checks.  vbuf: [S, T, d] stand-in sublayer outputs;
    U_split: the queries' bf16 split (tensor-core phase 1) or None.  The runner must have been
    made with ``extra_outputs=True``."""
    assert runner.h is not None and runner.alpha_p is not None
    chk = BlockChecker(reps, W, Gk, Gin, dtype, rows, eps, report)
    S = U.shape[0]

    def sublayer(i, y):
        chk.after(i, y, runner.h, runner.alpha_p)
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
