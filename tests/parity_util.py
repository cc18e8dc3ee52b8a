"""Tolerances and comparison helpers for GPU-vs-oracle parity.

Tolerances (stated for the method: outputs within 1e-5 x output RMS in fp32 mode and within
1e-2 x output RMS in bf16 mode; softmax weights within 1e-5 (fp32) and 1e-3 (bf16)):

  fp32 I/O   |gpu - oracle| <= 1e-5 * RMS(oracle)                                 outputs
             |gpu - oracle| <= 1e-5                                               weights, m, lse
  bf16 I/O, output stored in bf16
             |gpu - rne_bf16(oracle)| <= max(1e-2 * RMS(oracle), ulp_bf16(oracle))  outputs
  bf16 I/O, output stored in fp32 (phase 1's o with ATTNRES_O_F32)
             |gpu - oracle| <= 1e-2 * RMS(oracle)                                 outputs
             |gpu - oracle| <= 1e-3                                               weights, m, lse

The bf16-stored form compares with the oracle rounded to bf16 (round to nearest even) and
allows one bf16 step where that step is larger than 1e-2 x RMS: above 1.28 x RMS one step of
bf16 exceeds 1e-2 x RMS, so no bf16 store of a large element could meet the bare bound, and
the nearest bf16 value of the exact result is what a correct kernel stores.  Every check also
reports the literal max |gpu - oracle| / RMS against the unrounded fp64 oracle.

RMS = sqrt(mean(oracle^2)) over the compared tensor.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = {
    "f32": dict(out_rel=1e-5, ulps=0.0, weight=1e-5, stat=1e-5),
    "bf16": dict(out_rel=1e-2, ulps=1.0, weight=1e-3, stat=1e-3),
}


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    _, e = np.frexp(np.where(ax > 0, ax, 1.0))     # ax = m 2^e, m in [0.5, 1)
    u = np.ldexp(1.0, e - 8)
    return np.where(ax > 0, u, np.ldexp(1.0, -133))


def rne_bf16(x: np.ndarray) -> np.ndarray:
    """x rounded to the nearest bfloat16 value, ties to even (exact for normal numbers: the
    spacing is a power of two, so x / spacing is exact and rint rounds half to even)."""
    x = np.asarray(x, dtype=np.float64)
    u = ulp_bf16(x)
    return np.rint(x / u) * u


def _stored(got, stored):
    if stored is not None:
        return stored
    if isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16:
        return "bf16"
    return "f32"


GATES = {}     # what -> literal max |gpu - oracle| / RMS of the last check of that name
# max |gpu - rne_bf16(oracle)| / RMS of the last bf16-stored output check (the distance from
# the correctly rounded result; 0 when every element is the nearest bf16 value)
LAST = {"vs_rounded": 0.0}


def _report(what, rel, report):
    GATES[what] = rel
    if report is not None:
        report[what] = rel


def output_gate(g, w, dtype: str, stored: str, extra=0.0):
    """(err, bound, rms, literal) of GPU values g against oracle values w (fp64 arrays)."""
    tol = TOL[dtype]
    rms = float(np.sqrt(np.mean(w * w))) if w.size else 0.0
    lit = np.abs(g - w)
    if stored == "bf16":
        ref = rne_bf16(w)
        err = np.abs(g - ref)
        bound = np.maximum(tol["out_rel"] * rms, ulp_bf16(np.maximum(np.abs(w), np.abs(ref))))
    else:
        err = lit
        bound = tol["out_rel"] * rms
    rel = float(lit.max() / rms) if lit.size and rms > 0 else 0.0
    LAST["vs_rounded"] = float(err.max() / rms) if err.size and rms > 0 else 0.0
    return err, bound + extra, rms, rel


def check_outputs(got, want, dtype: str, what: str, report: dict | None = None,
                  stored: str | None = None):
    """Element-wise output check with the dtype's tolerance (module docstring); ``stored`` is
    the type the GPU stored ``got`` in ("bf16" or "f32"; by default ``got``'s dtype).  Returns
    the literal max |gpu - oracle| / RMS."""
    st = _stored(got, stored)
    g, w = to64(got), to64(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err, bound, rms, rel = output_gate(g, w, dtype, st)
    _report(what, rel, report)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max |err|/RMS = {rel:.3e} (RMS {rms:.3e})")
    return rel


def check_two_phase(got, y_direct, o_A, w_A, r_h, gamma_in, dtype: str, what: str,
                    report: dict | None = None, h_only: bool = False):
    """End-to-end check of a phase-2 output of the production path (phase 1's o stored in the
    I/O type) against the direct (one-softmax) definition.

    Besides the output gate of ``check_outputs``, the two-phase composition carries the storage
    rounding of the phase-1 output o_A when it is stored in bf16: |delta o_i| <= ulp(o_i) / 2
    enters h with the weight w_A of partition A, and y = gamma h / r(h) turns it into
        |delta y_i| <= w_A (|gamma_i| |delta o_i| + |y_i| RMS(delta o)) / r(h)
    (the second term bounds the change of r(h) by Cauchy-Schwarz); for h itself (h_only) the
    term is w_A |delta o_i|.  A full ulp is used for the half-ulp rounding as margin.  With o
    stored in fp32 (ATTNRES_O_F32), or in fp32 mode, there is no such term: use
    ``check_outputs`` against the direct definition instead."""
    g, w = to64(got), to64(y_direct)
    extra = 0.0
    if dtype == "bf16":
        uo = ulp_bf16(to64(o_A))
        wa = to64(w_A)[..., None]
        if h_only:
            extra = wa * uo
        else:
            gam = np.ones(w.shape[-1]) if gamma_in is None else np.abs(to64(gamma_in))
            rh = to64(r_h)[..., None]
            rms_uo = np.sqrt(np.mean(uo * uo, axis=-1, keepdims=True))
            extra = wa * (gam * uo + np.abs(w) * rms_uo) / rh
    err, bound, rms, rel = output_gate(g, w, dtype, _stored(got, None), extra)
    _report(what, rel, report)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements beyond the "
                           f"two-phase bound; max |err|/RMS = {rel:.3e}")
    return rel


def record_parity(what: str, values: dict):
    """Append one line {what: {gate: literal max error}} to the file named by the environment
    variable ATTNRES_PARITY_REPORT, if it is set (a record of the literal errors of a run)."""
    import json
    import os
    path = os.environ.get("ATTNRES_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({what: values}) + "\n")


def check_close(got, want, atol: float, what: str):
    g, w = to64(got), to64(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    err = float(np.max(np.abs(g - w))) if g.size else 0.0
    assert err <= atol, f"{what}: max |err| = {err:.3e} > {atol:.1e}"
    return err


def sample_rows(T: int, k: int, seed: int = 0) -> torch.Tensor:
    """Row indices to check at full size: first, last, a ragged spread, and random ones."""
    g = np.random.default_rng(seed)
    idx = {0, T - 1, T // 2, max(0, T - 7)}
    idx |= set(g.choice(T, size=min(T, k), replace=False).tolist())
    return torch.tensor(sorted(idx), dtype=torch.long)
