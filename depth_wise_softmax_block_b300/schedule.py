"""Block AttnRes schedule on the GPU, driven through the C ABI.

One block of S sublayers (page "Attention Residuals" note, §8 block definition and §10
two-phase schedule):

  1. phase 1: the block's S queries against the n completed sources b_0 .. b_{n-1};
  2. for i = 1 .. S, phase 2 merges the partial source b^{i-1} and writes the sublayer input
     y_i = RMSNorm_in(h_i).  The partial is built inside phase 2 from the previous sublayer's
     output: b^1 = v_1 needs no write, b^{i-1} = b^{i-2} + v_{i-1} is written in place;
  3. the block closes with b^S = b^{S-1} + v_S (the new completed source).

Sublayer outputs v_i come from a caller-supplied function of y_i (the model's attention or
MLP), which is where a real model would run f_i; the synthetic workloads hand back stand-ins.
All buffers are allocated once by the caller-facing ``BlockRunner`` so a step allocates
nothing.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

from . import (attnres_full_reference_path, attnres_partial_update, attnres_phase1,
               attnres_phase2_merge, attnres_phase2_merge_sources)


class KernelTimer:
    """CUDA events around each launch, on the current (launching) stream, grouped by kind.
    Durations are read after the caller synchronises."""

    def __init__(self):
        self.events = {}

    def wrap(self, kind: str, fn, *args, **kw):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        r = fn(*args, **kw)
        b.record()
        self.events.setdefault(kind, []).append((a, b))
        return r

    def totals_ms(self):
        return {k: (sum(a.elapsed_time(b) for a, b in v), len(v)) for k, v in self.events.items()}

    def clear(self):
        self.events.clear()


def _call(timer, kind, fn, *args, **kw):
    return fn(*args, **kw) if timer is None else timer.wrap(kind, fn, *args, **kw)


class BlockRunner:
    """Work buffers for blocks of up to ``S_max`` sublayers over ``T`` tokens, with ``heads``
    depth-attention heads (per-head log-sum-exps).

    ``o_dtype``: the type phase 1's output is stored in (the I/O type by default; fp32 removes
    the rounding between the two phases, ATTNRES_O_F32).  ``extra_outputs``: every phase-2 call
    also writes h (``self.h``) and the weight of the partial source (``self.alpha_p``), which
    the caller may read in the sublayer callback."""

    def __init__(self, T: int, d: int, S_max: int, dtype, device, keep_y: bool = False,
                 timer: Optional[KernelTimer] = None, heads: int = 1, o_dtype=None,
                 extra_outputs: bool = False):
        self.timer = timer
        self.T, self.d, self.S_max, self.heads = T, d, S_max, heads
        self.o = torch.empty((S_max, T, d), dtype=o_dtype or dtype, device=device)
        self.lse = torch.empty((S_max, heads, T), dtype=torch.float32, device=device)
        self.partial = torch.empty((T, d), dtype=dtype, device=device)
        self.keep_y = keep_y
        n_y = S_max if keep_y else 1
        self.y = torch.empty((n_y, T, d), dtype=dtype, device=device)
        self.h = torch.empty((T, d), dtype=dtype, device=device) if extra_outputs else None
        self.alpha_p = (torch.empty((heads, T), dtype=torch.float32, device=device)
                        if extra_outputs else None)

    def y_buffer(self, i: int) -> torch.Tensor:
        return self.y[i - 1] if self.keep_y else self.y[0]

    def run_block(self, reps: torch.Tensor, U: torch.Tensor, G_in: Optional[torch.Tensor],
                  sublayer: Callable[[int, torch.Tensor], torch.Tensor], close_out: torch.Tensor,
                  eps_key: float = 1e-6, eps_in: float = 1e-6,
                  on_call: Optional[Callable] = None,
                  U_split: Optional[torch.Tensor] = None, flags: int = 0) -> None:
        """Run one block.

        reps: [n, T, d] completed sources (any source stride); U: [S, d] folded queries;
        G_in: [S, d] input-norm gains or None; sublayer(i, y_i) -> v_i ([T, d], 1-based i);
        close_out: [T, d] receives b^S.  ``on_call(i, kind, args)`` is invoked before each
        phase-2 call (tests use it to snapshot the exact inputs).  U_split: [2S, d] bf16
        hi/lo split of U (attnres_query_prep), which puts phase 1's logits on the tensor cores.
        flags: variant flags (sigmoid weights, no key RMSNorm) for every call of the block.
        """
        S = U.shape[0]
        assert S <= self.S_max
        o, lse = self.o[:S], self.lse[:S]
        tm = self.timer
        _call(tm, "phase1", attnres_phase1, reps, U, o, lse_out=lse, eps=eps_key, u_split=U_split,
              flags=flags, heads=self.heads)
        v_prev = None       # v_{i-1}
        part = None         # tensor holding b^{i-2} (None while it is zero)
        for i in range(1, S + 1):
            y = self.y_buffer(i)
            g = None if G_in is None else G_in[i - 1]
            if i == 1:
                args = dict(partial=None, v_prev=None, partial_out=None)
            elif i == 2:
                args = dict(partial=v_prev, v_prev=None, partial_out=None)   # b^1 = v_1
            else:
                args = dict(partial=part, v_prev=v_prev, partial_out=self.partial)
            if on_call is not None:
                on_call(i, args)
            kind = "phase2_first" if i == 1 else ("phase2" if i == 2 else "phase2_fused")
            _call(tm, kind, attnres_phase2_merge, o[i - 1], lse[i - 1], args["partial"],
                  args["v_prev"], args["partial_out"], U[i - 1], g, y, h_out=self.h,
                  alpha_p_out=self.alpha_p if i > 1 else None, eps_key=eps_key,
                  eps_in=eps_in, flags=flags, heads=self.heads)
            # b^{i-1} now lives in args["partial"] (i == 2) or args["partial_out"] (i >= 3)
            if i == 2:
                part = v_prev
            elif i >= 3:
                part = args["partial_out"]
            v_prev = sublayer(i, y)
        self.last_partial = part  # b^{S-1} (None when S == 1)
        # close: b^S = b^{S-1} + v_S  (b^{S-1} = v_1 when S == 2; b^1 = v_1 when S == 1)
        if S == 1:
            close_out.copy_(v_prev)
        else:
            _call(tm, "close", attnres_partial_update, part, v_prev, close_out)


def final_aggregation(reps: torch.Tensor, u_final: torch.Tensor, out: torch.Tensor,
                      eps: float = 1e-6, timer: Optional[KernelTimer] = None,
                      flags: int = 0, heads: int = 1) -> torch.Tensor:
    """Final output over b_0 .. b_N: phase 1 with the single extra pseudo-query."""
    _call(timer, "final", attnres_phase1, reps, u_final.view(1, -1), out.view(1, *out.shape),
          eps=eps, flags=flags, heads=heads)
    return out


def full_attnres_sublayer(history, u_l, g_in, y_out, h_out=None, alpha_out=None,
                          eps_key: float = 1e-6, eps_in: float = 1e-6):
    """Full AttnRes input of one sublayer over the explicit history v_0 .. v_{l-1}."""
    return attnres_full_reference_path(list(history), u_l, g_in, h_out=h_out, y_out=y_out,
                                       alpha_out=alpha_out, eps_key=eps_key, eps_in=eps_in)


class FullGroupedRunner:
    """Full AttnRes (layer l reads v_0 .. v_{l-1}) by the grouped two-phase schedule ("Attention
    Residuals 阅读补充", section "静态 Query 与两阶段计算"): groups of S layers; phase 1
    scores a group's queries against the history [v_0 .. v_{l0}] in one pass; layer l0 + i then
    merges the group's own outputs v_{l0+1} .. v_{l0+i-1} into phase 1's result.

    ``hist`` [L + 1, T, d] holds v_0 in slot 0; slot l receives v_l = sublayer(l, y_l) (the
    model's attention or MLP; a stand-in for the synthetic workloads)."""

    def __init__(self, T: int, d: int, S: int, dtype, device, timer: Optional[KernelTimer] = None,
                 heads: int = 1, o_dtype=None):
        self.S, self.timer, self.heads = S, timer, heads
        self.o = torch.empty((S, T, d), dtype=o_dtype or dtype, device=device)
        self.lse = torch.empty((S, heads, T), dtype=torch.float32, device=device)

    def run(self, hist: torch.Tensor, U: torch.Tensor, G_in: Optional[torch.Tensor],
            y_out: torch.Tensor, sublayer: Callable[[int, torch.Tensor], torch.Tensor],
            eps_key: float = 1e-6, eps_in: float = 1e-6, U_split: Optional[torch.Tensor] = None,
            flags: int = 0) -> None:
        """U [L, d] folded queries; y_out [L, T, d] receives every layer's input y_l;
        U_split [2L, d] (optional) puts phase 1's logits on the tensor cores where the shape
        allows."""
        L = U.shape[0]
        tm = self.timer
        for l0 in range(0, L, self.S):
            Sg = min(self.S, L - l0)
            o, lse = self.o[:Sg], self.lse[:Sg]
            us = None if U_split is None else U_split[2 * l0:2 * (l0 + Sg)]
            _call(tm, "phase1", attnres_phase1, hist[:l0 + 1], U[l0:l0 + Sg], o, lse_out=lse,
                  eps=eps_key, u_split=us, flags=flags, heads=self.heads)
            for i in range(1, Sg + 1):
                l = l0 + i
                g = None if G_in is None else G_in[l - 1]
                srcs = [hist[j] for j in range(l0 + 1, l)]
                _call(tm, "phase2_sources", attnres_phase2_merge_sources, o[i - 1], lse[i - 1],
                      srcs, U[l - 1], g, y_out=y_out[l - 1], eps_key=eps_key, eps_in=eps_in,
                      flags=flags, heads=self.heads)
                v = sublayer(l, y_out[l - 1])
                if v.data_ptr() != hist[l].data_ptr():
                    hist[l].copy_(v)

