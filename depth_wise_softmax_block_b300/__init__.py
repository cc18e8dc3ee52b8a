"""B300 (sm_103a) Attention Residuals aggregation: Python binding of ``libattnres.so``.

The functions below carry the names of the C entry points in ``include/attnres.h`` and do
argument marshalling only (shapes, strides, dtypes, the current CUDA stream); every step of
the computation runs in the library's CUDA kernels.  PyTorch provides device memory and
streams.  There is no CPU fallback: if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattnres.so")

F32, BF16 = 0, 1
SIGMOID_WEIGHTS, NO_KEY_NORM = 0x1, 0x2   # variant flags (include/attnres.h)
O_F32 = 0x4                               # phase 1's output o stored in fp32
_U = ctypes.c_uint
STATUS = {0: "ATTNRES_OK", 1: "ATTNRES_ERR_INVALID_ARG", 2: "ATTNRES_ERR_UNSUPPORTED",
          3: "ATTNRES_ERR_MISALIGNED", 4: "ATTNRES_ERR_CUDA", 5: "ATTNRES_ERR_TIMEOUT"}

# C signatures (argument types, in order) of every exported symbol of include/attnres.h.
_P, _I, _I64, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
SIGNATURES = {
    "attnres_abi_version": ([], _I),
    "attnres_status_string": ([_I], ctypes.c_char_p),
    "attnres_last_cuda_error": ([], ctypes.c_char_p),
    "attnres_poll_device_errors": ([], _I),
    "attnres_selftest_wait_timeout": ([_U, _P], _I),
    "attnres_query_prep": ([_P, _P, _P, _P, _I, _I, _P], _I),
    "attnres_phase1": ([_P, _I64, _I, _I64, _I, _I, _P, _P, _I, _F, _P, _P, _P, _P, _U, _I,
                        _P], _I),
    "attnres_phase2_merge": ([_P, _P, _P, _P, _P, _I64, _I, _I, _P, _F, _P, _F, _P, _P, _P, _U,
                              _I, _P], _I),
    "attnres_partial_update": ([_P, _P, _P, _I64, _I, _I, _P], _I),
    "attnres_full_reference_path": ([_P, _I, _I64, _I, _I, _P, _F, _P, _F, _P, _P, _P, _U, _I,
                                     _P], _I),
    "attnres_phase2_merge_sources": ([_P, _P, _P, _I, _I64, _I, _I, _P, _F, _P, _F, _P, _P, _P, _U,
                                      _I, _P], _I),
    "attnres_backward": ([_P, _I, _I64, _I, _I, _P, _F, _P, _F, _P, _P, _P, _P, _P], _I),
    "attnres_backward_block_workspace_size": ([_I, _I, _I64, _I, _I, _P], _I),
    "attnres_backward_block": ([_P, _I64, _I, _P, _I64, _I, _I64, _I, _I, _P, _P, _F, _P, _F, _P,
                                _P, _P, _I64, _P, _P, _P, ctypes.c_uint64, _P], _I),
    "attnres_backward_block_noalloc": ([_P, _I64, _I, _P, _I64, _I, _I64, _I, _I, _P, _P, _F, _P,
                                        _F, _P, _P, _P, _I64, _P, _P, _P], _I),
}


class AttnResError(RuntimeError):
    """A library call returned a non-OK status."""


_lib = None


def library() -> ctypes.CDLL:
    """The loaded ``libattnres.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m depth_wise_softmax_block_b300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        msg = STATUS.get(status, str(status))
        if status == 4:
            msg += ": " + library().attnres_last_cuda_error().decode()
        raise AttnResError(f"{what} failed: {msg}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _io(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _rows(t: torch.Tensor, T: int, d: int, name: str):
    if t is None:
        return
    if tuple(t.shape[-2:]) != (T, d) or t.stride(-1) != 1 or t.stride(-2) != d:
        raise ValueError(f"{name}: expected rows of shape [{T}, {d}] with row stride {d}")


def _stats(t: torch.Tensor, numel: int, name: str):
    """A statistics output must be a contiguous fp32 tensor of the expected size."""
    if t is None:
        return
    if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != numel:
        raise ValueError(f"{name}: expected a contiguous fp32 tensor of {numel} elements")


def attnres_poll_device_errors():
    """Raise if a kernel's bounded wait gave up since the previous poll (synchronises)."""
    _check(library().attnres_poll_device_errors(), "attnres_poll_device_errors")


def attnres_selftest_wait_timeout(polls=1000, stream=None):
    """Launch the library's timeout self-test: a kernel whose bounded wait cannot succeed gives
    up after ``polls`` polls; the next attnres_poll_device_errors raises (ATTNRES_ERR_TIMEOUT)."""
    _check(library().attnres_selftest_wait_timeout(polls, _stream(stream)),
           "attnres_selftest_wait_timeout")


def attnres_query_prep(w, gamma_key, u_out, u_split_out=None, stream=None):
    """u = w ⊙ gamma_key (query with the key-norm gain folded in), [rows, d] fp32; optionally
    its bf16 hi/lo split [2 * rows, d] for the tensor-core phase 1."""
    rows, d = w.shape
    if u_split_out is not None:
        if (tuple(u_split_out.shape) != (2 * rows, d) or u_split_out.dtype != torch.bfloat16
                or not u_split_out.is_contiguous()):
            raise ValueError("u_split_out must be a contiguous bf16 [2 * rows, d] tensor")
    _check(library().attnres_query_prep(_ptr(w), _ptr(gamma_key), _ptr(u_out),
                                        _ptr(u_split_out), rows, d, _stream(stream)),
           "attnres_query_prep")
    return u_out


def _o_flag(o, io_dtype) -> int:
    """ATTNRES_O_F32 when phase 1's output ``o`` is fp32 and the I/O type is not."""
    if o.dtype == io_dtype:
        return 0
    if o.dtype == torch.float32:
        return O_F32
    raise TypeError(f"phase-1 output of dtype {o.dtype} with I/O dtype {io_dtype}")


def attnres_phase1(reps, u, o_out, m_out=None, lse_out=None, alpha_out=None, eps=1e-6,
                   u_split=None, flags=0, heads=1, stream=None):
    """Phase 1 over ``reps`` [n, T, d] (any source stride, rows of stride d) for the S queries
    ``u`` [S, d]; writes o [S, T, d] and the optional statistics (m, lse [S, heads, T], alpha
    [S, heads, T, n]; with one head the head axis may be left out).  ``u_split`` ([2S, d]
    bf16, from attnres_query_prep) puts the logits on the tensor cores where the shape
    allows.  An fp32 ``o_out`` with bf16 sources stores o in fp32 (ATTNRES_O_F32)."""
    n, T, d = reps.shape
    S = u.shape[0]
    if u_split is not None and (tuple(u_split.shape) != (2 * S, d) or not u_split.is_contiguous()
                                or u_split.dtype != torch.bfloat16):
        raise ValueError("u_split must be a contiguous bf16 [2S, d] tensor")
    _rows(reps[0], T, d, "reps")
    if tuple(o_out.shape) != (S, T, d) or not o_out.is_contiguous():
        raise ValueError("o_out must be a contiguous [S, T, d] tensor")
    src_stride = reps.stride(0) if n > 1 else T * d
    for name, t, per in (("m_out", m_out, 1), ("lse_out", lse_out, 1), ("alpha_out", alpha_out, n)):
        _stats(t, S * heads * T * per, name)
    flags |= _o_flag(o_out, reps.dtype)
    _check(library().attnres_phase1(_ptr(reps), src_stride, n, T, d, _io(reps), _ptr(u),
                                    _ptr(u_split), S, eps, _ptr(o_out), _ptr(m_out), _ptr(lse_out),
                                    _ptr(alpha_out), flags, heads, _stream(stream)),
           "attnres_phase1")
    return o_out


def attnres_phase2_merge(o_l, lse_l, partial, v_prev, partial_out, u_l, gamma_in, y_out,
                         h_out=None, alpha_p_out=None, eps_key=1e-6, eps_in=1e-6, flags=0,
                         heads=1, stream=None):
    """Phase 2 for one sublayer: merge the partial-sum source (partial + v_prev) into the
    phase-1 result and apply the input RMSNorm.  Tensors are [T, d]; lse_l and alpha_p_out
    are [heads, T] (or [T] with one head).  The I/O type is y_out's; an fp32 ``o_l`` with bf16
    I/O is read as fp32 (ATTNRES_O_F32)."""
    T, d = o_l.shape
    for name, t in (("o_l", o_l), ("partial", partial), ("v_prev", v_prev),
                    ("partial_out", partial_out), ("y_out", y_out), ("h_out", h_out)):
        _rows(t, T, d, name)
    _stats(lse_l, heads * T, "lse_l")
    _stats(alpha_p_out, heads * T, "alpha_p_out")
    flags |= _o_flag(o_l, y_out.dtype)
    _check(library().attnres_phase2_merge(
        _ptr(o_l), _ptr(lse_l), _ptr(partial), _ptr(v_prev), _ptr(partial_out), T, d, _io(y_out),
        _ptr(u_l), eps_key, _ptr(gamma_in), eps_in, _ptr(h_out), _ptr(y_out), _ptr(alpha_p_out),
        flags, heads, _stream(stream)), "attnres_phase2_merge")
    return y_out


def attnres_partial_update(partial, v, out, stream=None):
    """out = partial + v (partial-sum update / block close)."""
    T, d = partial.shape
    for name, t in (("partial", partial), ("v", v), ("out", out)):
        _rows(t, T, d, name)
    _check(library().attnres_partial_update(_ptr(partial), _ptr(v), _ptr(out), T, d,
                                            _io(partial), _stream(stream)),
           "attnres_partial_update")
    return out


def attnres_full_reference_path(srcs, u_l, gamma_in, h_out=None, y_out=None, alpha_out=None,
                                eps_key=1e-6, eps_in=1e-6, flags=0, heads=1, stream=None):
    """Direct single-pass aggregation over the list of [T, d] source tensors ``srcs``;
    alpha_out is [heads, T, n] (or [T, n] with one head)."""
    T, d = srcs[0].shape
    for t in srcs:
        _rows(t, T, d, "srcs[j]")
    _stats(alpha_out, heads * T * len(srcs), "alpha_out")
    arr = (ctypes.c_void_p * len(srcs))(*[t.data_ptr() for t in srcs])
    _check(library().attnres_full_reference_path(
        arr, len(srcs), T, d, _io(srcs[0]), _ptr(u_l), eps_key, _ptr(gamma_in), eps_in,
        _ptr(h_out), _ptr(y_out), _ptr(alpha_out), flags, heads, _stream(stream)),
        "attnres_full_reference_path")
    return h_out if y_out is None else y_out


def attnres_phase2_merge_sources(o_l, lse_l, srcs, u_l, gamma_in, h_out=None, y_out=None,
                                 alpha_out=None, eps_key=1e-6, eps_in=1e-6, flags=0, heads=1,
                                 stream=None):
    """Grouped Full AttnRes phase 2 for one layer: merge phase 1's (o_l, lse_l) with the
    group's in-group sources ``srcs`` (a list of [T, d] tensors, possibly empty); lse_l is
    [heads, T] and alpha_out [heads, T, k] (head axis optional with one head).  The I/O type is
    that of the outputs; an fp32 ``o_l`` with bf16 I/O is read as fp32 (ATTNRES_O_F32)."""
    T, d = o_l.shape
    io_dtype = (y_out if y_out is not None else h_out).dtype
    flags |= _o_flag(o_l, io_dtype)
    for name, t in [("o_l", o_l), ("h_out", h_out), ("y_out", y_out)] + \
            [("srcs[j]", t) for t in srcs]:
        _rows(t, T, d, name)
    _stats(lse_l, heads * T, "lse_l")
    _stats(alpha_out, heads * T * len(srcs), "alpha_out")
    arr = (ctypes.c_void_p * max(1, len(srcs)))(*[t.data_ptr() for t in srcs])
    _check(library().attnres_phase2_merge_sources(
        _ptr(o_l), _ptr(lse_l), arr if srcs else None, len(srcs), T, d,
        BF16 if io_dtype == torch.bfloat16 else F32, _ptr(u_l), eps_key, _ptr(gamma_in), eps_in,
        _ptr(h_out), _ptr(y_out), _ptr(alpha_out), flags, heads, _stream(stream)),
        "attnres_phase2_merge_sources")
    return h_out if y_out is None else y_out


def attnres_backward(srcs, u, gamma_in, g_y, dsrcs, du, dgamma_in=None, eps_key=1e-6,
                     eps_in=1e-6, stream=None):
    """Backward of one sublayer's aggregation over ``srcs`` ([T, d] tensors): writes dL/dv_i
    into ``dsrcs`` and ADDS dL/du (and dL/dgamma_in) into the fp32 [d] accumulators."""
    T, d = srcs[0].shape
    for name, t in [("g_y", g_y)] + [("srcs[j]", t) for t in srcs] + \
            [("dsrcs[j]", t) for t in dsrcs]:
        _rows(t, T, d, name)
    if len(dsrcs) != len(srcs):
        raise ValueError("one gradient tensor per source")
    a_src = (ctypes.c_void_p * len(srcs))(*[t.data_ptr() for t in srcs])
    a_dst = (ctypes.c_void_p * len(dsrcs))(*[t.data_ptr() for t in dsrcs])
    _check(library().attnres_backward(a_src, len(srcs), T, d, _io(srcs[0]), _ptr(u), eps_key,
                                      _ptr(gamma_in), eps_in, _ptr(g_y), a_dst, _ptr(du),
                                      _ptr(dgamma_in), _stream(stream)), "attnres_backward")
    return dsrcs



def attnres_backward_block_workspace_size(n_src, S, T, d, dtype) -> int:
    """Bytes of device workspace attnres_backward_block needs for these sizes."""
    out = ctypes.c_uint64(0)
    _check(library().attnres_backward_block_workspace_size(
        n_src, S, T, d, BF16 if dtype == torch.bfloat16 else F32, ctypes.byref(out)),
        "attnres_backward_block_workspace_size")
    return int(out.value)


def attnres_backward_block(reps, v, u, gamma_in, g_y, d_reps, d_v, du, dgamma_in=None,
                           u_split=None, eps_key=1e-6, eps_in=1e-6, workspace=None, stream=None):
    """Backward of one block: ``reps`` [n, T, d] completed sources (any source stride),
    ``v`` [S-1, T, d] the sublayer outputs v_1 .. v_{S-1} (None when S == 1), ``u`` [S, d] the
    folded queries, ``g_y`` [S, T, d] = dL/dy_i.  Writes d_reps [n, T, d] (contiguous) and d_v
    [S-1, T, d]; ADDS du and dgamma_in ([S, d] fp32).  ``workspace``: a uint8 device tensor of
    at least attnres_backward_block_workspace_size() bytes (made here when None)."""
    n, T, d = reps.shape
    S = u.shape[0]
    _rows(reps[0], T, d, "reps")
    if g_y.shape != (S, T, d) or not g_y.is_contiguous():
        raise ValueError("g_y must be a contiguous [S, T, d] tensor")
    if d_reps.shape != (n, T, d) or not d_reps.is_contiguous():
        raise ValueError("d_reps must be a contiguous [n, T, d] tensor")
    if S > 1:
        for name, t in (("v", v), ("d_v", d_v)):
            if t is None or t.shape[0] < S - 1 or tuple(t.shape[1:]) != (T, d):
                raise ValueError(f"{name} must hold S - 1 rows of [T, d]")
            _rows(t[0], T, d, name)
    need = attnres_backward_block_workspace_size(n, S, T, d, reps.dtype)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=reps.device)
    src_stride = reps.stride(0) if n > 1 else T * d
    v_stride = v.stride(0) if (v is not None and v.shape[0] > 1) else T * d
    dv_stride = d_v.stride(0) if (d_v is not None and d_v.shape[0] > 1) else T * d
    _check(library().attnres_backward_block(
        _ptr(reps), src_stride, n, _ptr(v), v_stride, S, T, d, _io(reps), _ptr(u), _ptr(u_split),
        eps_key, _ptr(gamma_in), eps_in, _ptr(g_y), _ptr(d_reps), _ptr(d_v), dv_stride, _ptr(du),
        _ptr(dgamma_in), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "attnres_backward_block")
    return d_reps


def attnres_backward_block_noalloc(reps, v, u, gamma_in, g_y, d_reps, d_v, du, dgamma_in=None,
                                   u_split=None, eps_key=1e-6, eps_in=1e-6, stream=None):
    """attnres_backward_block for callers that cannot allocate device memory while it runs: the
    scratch is the library's own fixed device array (ATTNRES_NOALLOC_SCRATCH_BYTES), so nothing
    is allocated here or in the library.  Blocks whose scratch would not fit raise
    (ATTNRES_ERR_UNSUPPORTED).  Calls whose work overlaps on the GPU share that array and race:
    order them.  The first call on a device looks up the array's address; make it before any
    stream capture."""
    n, T, d = reps.shape
    S = u.shape[0]
    _rows(reps[0], T, d, "reps")
    if g_y.shape != (S, T, d) or not g_y.is_contiguous():
        raise ValueError("g_y must be a contiguous [S, T, d] tensor")
    if d_reps.shape != (n, T, d) or not d_reps.is_contiguous():
        raise ValueError("d_reps must be a contiguous [n, T, d] tensor")
    if S > 1:
        for name, t in (("v", v), ("d_v", d_v)):
            if t is None or t.shape[0] < S - 1 or tuple(t.shape[1:]) != (T, d):
                raise ValueError(f"{name} must hold S - 1 rows of [T, d]")
            _rows(t[0], T, d, name)
    src_stride = reps.stride(0) if n > 1 else T * d
    v_stride = v.stride(0) if (v is not None and v.shape[0] > 1) else T * d
    dv_stride = d_v.stride(0) if (d_v is not None and d_v.shape[0] > 1) else T * d
    _check(library().attnres_backward_block_noalloc(
        _ptr(reps), src_stride, n, _ptr(v), v_stride, S, T, d, _io(reps), _ptr(u), _ptr(u_split),
        eps_key, _ptr(gamma_in), eps_in, _ptr(g_y), _ptr(d_reps), _ptr(d_v), dv_stride, _ptr(du),
        _ptr(dgamma_in), _stream(stream)), "attnres_backward_block_noalloc")
    return d_reps
