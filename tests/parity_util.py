"""Tolerances and comparison helpers for GPU-vs-oracle parity.

Tolerances (stated for the method: outputs within 1e-5 x output RMS in fp32 mode and within
1e-2 x output RMS in bf16 mode; softmax weights within 1e-5 (fp32) and 1e-3 (bf16)):

  fp32 I/O   |gpu - oracle| <= 1e-5 * RMS(oracle)                           outputs
             |gpu - oracle| <= 1e-5                                         weights, m, lse
  bf16 I/O   |gpu - oracle| <= 1e-2 * RMS(oracle) + ulp_bf16(oracle)        outputs
             |gpu - oracle| <= 1e-3                                         weights, m, lse

The extra ulp in bf16 mode is storage, not arithmetic: an output stored in bf16 is off by
up to half an ulp from any real value, and phase 2 reads the phase-1 output that was itself
stored in bf16 (another half ulp, relative to the same magnitude).  Above 2.56 x RMS half an
ulp alone exceeds 1e-2 x RMS, so without the term no bf16 store of a large element could
pass.  The literal max |gpu - oracle| / RMS is reported by every check.
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


def check_outputs(got, want, dtype: str, what: str, report: dict | None = None):
    """Element-wise output check with the dtype's tolerance; returns max err / RMS."""
    g, w = to64(got), to64(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    tol = TOL[dtype]
    rms = float(np.sqrt(np.mean(w * w))) if w.size else 0.0
    err = np.abs(g - w)
    bound = tol["out_rel"] * rms + (tol["ulps"] * ulp_bf16(w) if tol["ulps"] else 0.0)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    bad = err > bound
    rel = float(err.max() / rms) if err.size and rms > 0 else 0.0
    if report is not None:
        report[what] = rel
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max |err|/RMS = {rel:.3e} (RMS {rms:.3e})")
    return rel


def check_two_phase(got, y_direct, o_A, w_A, r_h, gamma_in, dtype: str, what: str,
                    report: dict | None = None):
    """End-to-end check of a phase-2 output against the direct (one-softmax) definition.

    Besides the per-call tolerance, the two-phase composition carries the storage rounding of
    the phase-1 output o_A (bf16 when the I/O is bf16): |delta o_i| <= ulp(o_i) / 2 enters h
    with the weight w_A of partition A, and y = gamma h / r(h) turns it into
        |delta y_i| <= w_A (|gamma_i| |delta o_i| + |y_i| RMS(delta o)) / r(h)
    (the second term bounds the change of r(h) by Cauchy-Schwarz).  A full ulp is used for
    the half-ulp rounding as margin.  In fp32 mode the term is below 1e-6 and is dropped."""
    g, w = to64(got), to64(y_direct)
    tol = TOL[dtype]
    rms = float(np.sqrt(np.mean(w * w)))
    bound = tol["out_rel"] * rms
    if dtype == "bf16":
        uo = ulp_bf16(to64(o_A))
        gam = np.ones(w.shape[-1]) if gamma_in is None else np.abs(to64(gamma_in))
        wa = to64(w_A)[..., None]
        rh = to64(r_h)[..., None]
        rms_uo = np.sqrt(np.mean(uo * uo, axis=-1, keepdims=True))
        bound = bound + ulp_bf16(w) + wa * (gam * uo + np.abs(w) * rms_uo) / rh
    err = np.abs(g - w)
    rel = float(err.max() / rms) if err.size else 0.0
    if report is not None:
        report[what] = rel
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements beyond the "
                           f"two-phase bound; max |err|/RMS = {rel:.3e}")
    return rel


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
