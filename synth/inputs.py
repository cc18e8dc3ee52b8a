"""Seeded synthetic workloads for AttnRes residual aggregation.

Holds shapes, value distributions and seeds only -- none of the method's arithmetic.  The
same generators serve the CUDA path and the fp64 oracle: tensors are drawn once (on the GPU
for the large workloads) and the oracle is handed the exact stored values.

Value recipe (the pages fix no data; these follow the workload shapes of the Kimi K2/K3
dimensions the pages quote -- d = 7168, 93 decoder layers = 186 sublayers, 9 sources):
  * block representation b_n (slot n = 0 is the embedding):  N(0, n + 1) plus a per-(slot,
    token) mean shift drawn from N(0, 0.25) and added to all d features;
  * sublayer outputs v (stand-ins for f_l):  N(0, 1)  (the Full-AttnRes workload scales
    v_i by (1 + 0.05 i));
  * pseudo-queries w_l:  N(0, 1/d);
  * RMSNorm gains:  1, or 1 + N(0, 0.02^2) where the workload says so;
  * eps = 1e-6 for both the key norm and the input norm.

Every tensor has its own stream: ``torch.Generator(device).manual_seed(mix(seed, tag))``.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" or "bf16": storage type of every [T, d] tensor
    T: int                # tokens
    d: int                # hidden size
    L: int                # sublayers
    S: int                # sublayers per block (1 = Full AttnRes)
    seed: int
    gamma_jitter: float   # std of the RMSNorm gains around 1 (0 = all ones)
    v_growth: float = 0.0 # v_i scaled by (1 + v_growth * i)
    chunk: int = 0        # tokens per chunk for chunked prefill (0 = no chunking)
    eps: float = 1e-6

    @property
    def n_blocks(self) -> int:
        return (self.L + self.S - 1) // self.S

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five workloads.  Names say what they are.
TINY_BLOCK_F32 = Workload("tiny_block_f32_T64_d128_L8_S4", "f32", 64, 128, 8, 4, seed=0,
                          gamma_jitter=0.0)
PREFILL_CHUNK_BF16 = Workload("prefill_chunk_bf16_T16384_d7168_L186_S24", "bf16", 16384, 7168,
                              186, 24, seed=2, gamma_jitter=0.02)
FULL_INTERP_BF16 = Workload("full_attnres_bf16_T8192_d2048_L54", "bf16", 8192, 2048, 54, 1,
                            seed=3, gamma_jitter=0.0, v_growth=0.05)
DECODE_BF16 = Workload("decode_bf16_T256_d7168_L186_S24", "bf16", 256, 7168, 186, 24, seed=4,
                       gamma_jitter=0.0)
LONGCTX_PREFILL_BF16 = Workload("longctx_prefill_bf16_T131072_chunk16384_d7168_S24_n9", "bf16",
                                131072, 7168, 24, 24, seed=5, gamma_jitter=0.02, chunk=16384)

WORKLOADS = {w.name: w for w in (TINY_BLOCK_F32, PREFILL_CHUNK_BF16, FULL_INTERP_BF16,
                                 DECODE_BF16, LONGCTX_PREFILL_BF16)}


def _stream(seed: int, tag: str, device) -> torch.Generator:
    h = hashlib.sha256(f"{seed}/{tag}".encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def normal(shape, std: float, seed: int, tag: str, device="cpu", dtype=torch.float32,
           mean: float = 0.0) -> torch.Tensor:
    """N(mean, std^2) draws of ``shape``, rounded once to ``dtype``."""
    g = _stream(seed, tag, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(dtype)


def fill_block_rep(out: torch.Tensor, slot: int, seed: int, tag: str = "rep") -> None:
    """Write block representation b_slot into ``out`` ([T, d], any dtype): N(0, slot+1) plus a
    per-token mean shift N(0, 0.25).  Drawn in token slabs to bound the fp32 temporary."""
    T, d = out.shape
    dev = out.device
    g_val = _stream(seed, f"{tag}/{slot}/val", dev)
    g_shift = _stream(seed, f"{tag}/{slot}/shift", dev)
    shift = torch.randn((T, 1), generator=g_shift, device=dev, dtype=torch.float32) * 0.5
    std = float(slot + 1) ** 0.5
    slab = max(1, (1 << 28) // d)
    for t0 in range(0, T, slab):
        t1 = min(T, t0 + slab)
        x = torch.randn((t1 - t0, d), generator=g_val, device=dev, dtype=torch.float32)
        x.mul_(std).add_(shift[t0:t1])
        out[t0:t1].copy_(x.to(out.dtype))


def fill_sublayer_output(out: torch.Tensor, l: int, seed: int, growth: float = 0.0,
                         tag: str = "v") -> None:
    """Write v_l (stand-in output of sublayer l) into ``out``: N(0,1) * (1 + growth * l)."""
    T, d = out.shape
    dev = out.device
    g = _stream(seed, f"{tag}/{l}", dev)
    scale = 1.0 + growth * l
    slab = max(1, (1 << 28) // d)
    for t0 in range(0, T, slab):
        t1 = min(T, t0 + slab)
        x = torch.randn((t1 - t0, d), generator=g, device=dev, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        out[t0:t1].copy_(x.to(out.dtype))


def queries(n: int, d: int, seed: int, tag: str, device="cpu", zero: bool = False):
    """Pseudo-queries w: [n, d] fp32, N(0, 1/d) (or all zero, the zero-initialised model)."""
    if zero:
        return torch.zeros((n, d), dtype=torch.float32, device=device)
    return normal((n, d), d ** -0.5, seed, tag, device)


def gains(n: int, d: int, jitter: float, seed: int, tag: str, device="cpu"):
    """RMSNorm gains: [n, d] fp32, 1 + N(0, jitter^2) (all ones when jitter == 0)."""
    if jitter == 0.0:
        return torch.ones((n, d), dtype=torch.float32, device=device)
    return normal((n, d), jitter, seed, tag, device, mean=1.0)


@dataclass
class BlockParams:
    """Per-sublayer parameters of a depth walk (all fp32, on one device)."""
    W: torch.Tensor        # [L, d] pseudo-queries
    G_key: torch.Tensor    # [L, d] key-norm gains
    G_in: torch.Tensor     # [L, d] input-norm gains
    w_final: torch.Tensor  # [d] final-aggregation query
    g_final: torch.Tensor  # [d] its key-norm gain


def block_params(wl: Workload, device="cpu", zero_queries: bool = False) -> BlockParams:
    L, d, s = wl.L, wl.d, wl.seed
    W = queries(L + 1, d, s, "w", device, zero_queries)
    Gk = gains(L + 1, d, wl.gamma_jitter, s, "gamma_key", device)
    Gi = gains(L, d, wl.gamma_jitter, s, "gamma_in", device)
    return BlockParams(W[:L].contiguous(), Gk[:L].contiguous(), Gi, W[L].contiguous(),
                       Gk[L].contiguous())


def make_reps(wl: Workload, n_slots: int, device="cpu", T: int | None = None) -> torch.Tensor:
    """Block-representation cache [n_slots, T, d] in the workload's dtype (slot 0 = b_0)."""
    T = wl.T if T is None else T
    reps = torch.empty((n_slots, T, wl.d), dtype=wl.torch_dtype, device=device)
    for j in range(n_slots):
        fill_block_rep(reps[j], j, wl.seed)
    return reps


def make_outputs(wl: Workload, first: int, count: int, device="cpu",
                 T: int | None = None) -> torch.Tensor:
    """Sublayer outputs v_first .. v_{first+count-1}: [count, T, d] in the workload dtype."""
    T = wl.T if T is None else T
    v = torch.empty((count, T, wl.d), dtype=wl.torch_dtype, device=device)
    for k in range(count):
        fill_sublayer_output(v[k], first + k, wl.seed, wl.v_growth)
    return v
