"""Algorithmic byte and flop counts of the AttnRes residual-aggregation path.

These are the counts the bench divides by measured time to report achieved GB/s (and the
roofline fraction), plus the pages' own analytic cost formulas, which the tests check against
the numbers the pages print.

Per-token algorithmic bytes of each kernel (E = bytes per stored element, 2 for bf16 and 4
for fp32; statistics are fp32):
  phase 1, n sources, S queries:            (n + S) d E + 4 S (lse) [+ 4 S (m)] [+ 4 S n (alpha)]
  phase 2, no partial source (i = 1):       2 d E                      (read o, write y)
  phase 2, partial given as one tensor:     3 d E + 4                  (read o, lse, p; write y)
  phase 2, fused partial update:            5 d E + 4                  (+ read v, write p)
  partial update / block close:             3 d E
  full reference path, n sources:           (n + 1) d E (+ d E with h)
With H depth-attention heads every statistic (lse, m, alpha) is kept per head: H times the
4-byte terms above.
"""
from __future__ import annotations

from dataclasses import dataclass


def phase1_bytes(n: int, S: int, d: int, E: int, with_m: bool = False, with_lse: bool = True,
                 with_alpha: bool = False, heads: int = 1) -> int:
    b = (n + S) * d * E
    b += 4 * S * heads * (int(with_m) + int(with_lse))
    if with_alpha:
        b += 4 * S * heads * n
    return b


def phase2_bytes(d: int, E: int, has_partial: bool, fused_update: bool,
                 write_h: bool = False, heads: int = 1) -> int:
    if not has_partial:
        b = 2 * d * E
    else:
        b = 3 * d * E + 4 * heads
        if fused_update:
            b += 2 * d * E
    if write_h:
        b += d * E
    return b


def partial_update_bytes(d: int, E: int) -> int:
    return 3 * d * E


def full_path_bytes(n: int, d: int, E: int, write_h: bool = False, write_y: bool = True) -> int:
    return (n + int(write_h) + int(write_y)) * d * E


def phase1_flops(n: int, S: int, d: int) -> int:
    """Per token: S n d multiply-adds for the logits, S n d for the weighted sum, n d for the
    squares (2 flops each)."""
    return 2 * (2 * S * n * d + n * d)


@dataclass(frozen=True)
class BlockStepBytes:
    phase1: int
    phase2: int
    close: int
    final: int

    @property
    def total(self) -> int:
        return self.phase1 + self.phase2 + self.close + self.final


def block_step_bytes(n: int, S: int, d: int, E: int, final_sources: int,
                     heads: int = 1) -> BlockStepBytes:
    """Per-token bytes of one block of the chunked-prefill step: phase 1 over n sources with
    S queries; phase 2 for i = 1 (no partial), i = 2 (partial = v_1, nothing to write) and
    i = 3 .. S (fused partial update); the block close b^S = b^{S-1} + v_S; the final
    aggregation (phase 1 with one query over ``final_sources`` sources, no statistics)."""
    p1 = phase1_bytes(n, S, d, E, heads=heads)
    p2 = phase2_bytes(d, E, False, False)
    if S >= 2:
        p2 += phase2_bytes(d, E, True, False, heads=heads)
    p2 += max(0, S - 2) * phase2_bytes(d, E, True, True, heads=heads)
    close = partial_update_bytes(d, E)
    final = phase1_bytes(final_sources, 1, d, E, with_lse=False) if final_sources else 0
    return BlockStepBytes(p1, p2, close, final)


# --- the pages' analytic formulas (checked against their printed numbers in tests) ---------
def io_per_layer_standard(d):
    """Standard residual: 3d per layer (page 2 §10 table)."""
    return 3 * d


def io_per_layer_full_two_phase(S, N, d):
    """Full AttnRes with the two-phase schedule: (S + N) d (page 2 §10 table; N here is the
    number of scheduling groups)."""
    return (S + N) * d


def io_per_layer_block_two_phase(S, N, d):
    """Block AttnRes with the two-phase schedule: (N / S + 5) d (page 2 §10 table)."""
    return (N / S + 5) * d


def io_per_layer_mhc(m, d):
    """mHC: (8m + 2) d + 2 m^2 + 4 m (page 2 §10 table)."""
    return (8 * m + 2) * d + 2 * m * m + 4 * m


def block_cache_bytes(B, N, T, d, P=1, E=2):
    """Block-representation prefill cache, E B N (T / P) d bytes (page 1, Block AttnRes
    memory section; page 2 §10)."""
    return E * B * N * (T / P) * d


def full_history_bytes(B, T, L, d, E=2):
    """Full AttnRes prefill history 2 B T (L + 1) d bytes in bf16 (page 1, Full AttnRes)."""
    return E * B * T * (L + 1) * d


def n_pairs(L):
    """Source-target pairs of Full AttnRes, L (L + 1) / 2 (page 1, Full AttnRes arithmetic)."""
    return L * (L + 1) // 2


def full_fwd_flops_per_token(L, d):
    """About 4 d N_pair = 2 L (L + 1) d flops per token (page 1, Full AttnRes arithmetic)."""
    return 4 * d * n_pairs(L)


def pp_comm_naive(P, V, Np=1, d=1):
    """C (C - 1) / 2 N_p d with C = P V (page 2 §9)."""
    C = P * V
    return C * (C - 1) // 2 * Np * d


def pp_comm_cached(P, V, Np=1, d=1):
    """P (P - 1) / 2 N_p d + (V - 1) P^2 N_p d (page 2 §9; page 1 prints (V - 1) P^2 / 2 for
    the second term, page 2's form matches its own P = 4, V = 2 example)."""
    return P * (P - 1) // 2 * Np * d + (V - 1) * P * P * Np * d
