"""GB300 (sm_103a) Lightning Attention chunkwise prefill and speculative-decoding ops.

``la_prefill_fwd`` (include/la_prefill.h), ``la_prefill_bwd`` (include/la_backward.h),
``la_prefill_fwd_segmented``,
``la_prefill_fwd_segmented_static`` and ``la_prefill_segmented_workspace``
(include/la_segment.h) and ``la_decode_mtp``,
``la_verify``, ``la_commit`` (include/la_decode.h) are thin ctypes bindings of the C
entry points of the same names: they check dtypes and shapes of torch tensors, pass their device
pointers and the current CUDA stream, and raise on a non-OK status.  Every step of the
computation runs in the library's CUDA kernels; there is no other implementation in
this package and no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = ["la_prefill_fwd", "la_prefill_fwd_segmented", "la_prefill_fwd_segmented_static", "la_prefill_bwd",
           "la_prefill_bwd_workspace", "la_prefill_fwd_d256", "la_prefill_d256_workspace",
           "la_prefill_fwd_d256_segmented", "la_prefill_d256_segmented_workspace",
           "la_prefill_segmented_workspace", "la_decode_mtp", "la_verify", "la_commit", "LaError", "load_library", "SCHEDULES", "DEV_ERR_BAD_SEQLENS",
           "DEV_ERR_BAD_INDEX", "DEV_ERR_TIMEOUT", "EXPORTED_SYMBOLS"]

SCHEDULES = {"auto": 0, "persistent": 1, "non_persistent": 2}
DEV_ERR_BAD_SEQLENS = 1
DEV_ERR_BAD_INDEX = 2
DEV_ERR_TIMEOUT = 4
EXPORTED_SYMBOLS = ("la_prefill_fwd", "la_status_string", "la_last_error", "la_prefill_smem_bytes",
                    "la_decode_mtp", "la_verify",
                    "la_commit", "la_prefill_segmented_workspace", "la_prefill_fwd_segmented",
                    "la_prefill_fwd_segmented_static", "la_prefill_bwd_workspace", "la_prefill_bwd",
                    "la_prefill_d256_workspace", "la_prefill_fwd_d256", "la_prefill_d256_segmented_workspace",
                    "la_prefill_fwd_d256_segmented")

_lock = threading.Lock()
_lib = None


class LaError(RuntimeError):
    """A non-OK la_status returned by the C library."""

    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}")
        self.status = status
        self.name = name


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libla_prefill.so (building it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if build_if_missing:
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path} (run linear_attention_prefill_chunkwise_gb300.build)")
            lib = ctypes.CDLL(path)
            vp, i32p, fp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            lib.la_prefill_fwd.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, i32p, i32p, vp, fp] + \
                [ctypes.c_int] * 8 + [ctypes.c_int, vp, vp]
            lib.la_prefill_fwd.restype = ctypes.c_int
            lib.la_status_string.argtypes = [ctypes.c_int]
            lib.la_status_string.restype = ctypes.c_char_p
            lib.la_last_error.argtypes = []
            lib.la_last_error.restype = ctypes.c_char_p
            lib.la_prefill_smem_bytes.argtypes = []
            lib.la_prefill_smem_bytes.restype = ctypes.c_int
            ints = [ctypes.c_int] * 7  # B, T, H, HV, D, V, pool_size
            lib.la_decode_mtp.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, i32p, vp] + ints + [vp, vp]
            lib.la_decode_mtp.restype = ctypes.c_int
            lib.la_verify.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, i32p, vp, vp, vp] + ints + [vp, vp]
            lib.la_verify.restype = ctypes.c_int
            lib.la_commit.argtypes = [fp, i32p, vp, vp, i32p, fp] + ints + [vp, vp]
            lib.la_commit.restype = ctypes.c_int
            lib.la_prefill_segmented_workspace.argtypes = [ctypes.c_int] * 6 + [vp, vp]
            lib.la_prefill_segmented_workspace.restype = ctypes.c_int
            lib.la_prefill_fwd_segmented.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, i32p, i32p, vp, fp] + \
                [ctypes.c_int] * 9 + [vp, ctypes.c_size_t, vp, vp]
            lib.la_prefill_fwd_segmented.restype = ctypes.c_int
            lib.la_prefill_fwd_segmented_static.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, i32p, i32p, vp,
                                                            fp] + [ctypes.c_int] * 9 + [vp, vp]
            lib.la_prefill_fwd_segmented_static.restype = ctypes.c_int
            lib.la_prefill_bwd_workspace.argtypes = [ctypes.c_int] * 8 + [vp]
            lib.la_prefill_bwd_workspace.restype = ctypes.c_int
            lib.la_prefill_bwd.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, vp, fp, i32p, i32p, vp, vp, vp, fp] + \
                [ctypes.c_int] * 8 + [vp, ctypes.c_size_t, vp, vp]
            lib.la_prefill_bwd.restype = ctypes.c_int
            lib.la_prefill_d256_workspace.argtypes = [ctypes.c_int] * 5 + [vp]
            lib.la_prefill_d256_workspace.restype = ctypes.c_int
            lib.la_prefill_fwd_d256.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, i32p, i32p, vp, fp] + \
                [ctypes.c_int] * 8 + [vp, ctypes.c_size_t, vp, vp]
            lib.la_prefill_fwd_d256.restype = ctypes.c_int
            lib.la_prefill_d256_segmented_workspace.argtypes = [ctypes.c_int] * 7 + [vp, vp]
            lib.la_prefill_d256_segmented_workspace.restype = ctypes.c_int
            lib.la_prefill_fwd_d256_segmented.argtypes = [vp, vp, vp, fp, ctypes.c_float, fp, i32p, i32p, vp, fp] + \
                [ctypes.c_int] * 9 + [vp, ctypes.c_size_t, vp, vp]
            lib.la_prefill_fwd_d256_segmented.restype = ctypes.c_int
            _lib = lib
        return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, ndim):
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o, h_final, seq_len, dev_error, stream):
    """Checks shared by the prefill entry points; returns (o, B, T, N, H, HV, D, V, pool, stream)."""
    import torch
    _check(q, "q", torch.bfloat16, 3)
    _check(k, "k", torch.bfloat16, 3)
    _check(v, "v", torch.bfloat16, 3)
    _check(slopes, "slopes", torch.float32, 1)
    _check(h0, "h0", torch.float32, 4)
    _check(h_final, "h_final", torch.float32, 4)
    _check(state_indices, "state_indices", torch.int32, 1)
    _check(cu_seqlens, "cu_seqlens", torch.int32, 1)
    tokens, H, D = q.shape
    _, HV, V = v.shape
    if k.shape != q.shape or v.shape[0] != tokens:
        raise ValueError("q, k, v token counts / shapes disagree")
    if slopes.shape[0] != HV:
        raise ValueError("slopes must have HV entries")
    if o is None:
        o = torch.empty((tokens, HV, V), dtype=torch.bfloat16, device=q.device)
    _check(o, "o", torch.bfloat16, 3)
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
        B, T = 1, tokens
    else:
        if seq_len is None:
            raise ValueError("fixed-length mode needs seq_len")
        T = int(seq_len)
        if T == 0:
            raise ValueError("seq_len must be positive in fixed-length mode")
        if tokens % T:
            raise ValueError("tokens must be a multiple of seq_len")
        B = tokens // T
        N = B
    pool = 0
    for t in (h0, h_final):
        if t is not None:
            if tuple(t.shape[1:]) != (HV, V, D):
                raise ValueError("state tensors must be [P, HV, V, D]")
            pool = t.shape[0] if pool == 0 else min(pool, t.shape[0])
    if h0 is not None and h_final is not None and h0.shape[0] != h_final.shape[0]:
        raise ValueError("h0 and h_final must have the same number of slots")
    if state_indices is not None and state_indices.shape[0] != N:
        raise ValueError("state_indices must have N entries")
    if dev_error is not None:
        _check(dev_error, "dev_error", torch.int32, 1)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    return o, B, T, N, H, HV, D, V, pool, stream


def la_prefill_fwd(q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None, o=None,
                   h_final=None, seq_len=None, schedule="auto", dev_error=None, stream=None):
    """Lightning Attention chunkwise prefill (forward) on the current CUDA device.

    q, k: bf16 [tokens, H, 128]; v: bf16 [tokens, HV, 128]; slopes: fp32 [HV];
    h0 / h_final: fp32 [P, HV, 128, 128] ([V, K] per state) or None;
    state_indices: int32 [N] or None (negative = padded sequence);
    cu_seqlens: int32 [N + 1] or None.  Without cu_seqlens the batch is fixed
    length: ``seq_len`` tokens per sequence (tokens must be a multiple of it).
    ``o`` (bf16 [tokens, HV, 128]) is allocated when not given.  h_final may be
    the same tensor as h0 (in-place state pool).  Returns ``o``.
    """
    lib = load_library()
    o, B, T, N, H, HV, D, V, pool, stream = _prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o,
                                                          h_final, seq_len, dev_error, stream)
    if isinstance(schedule, str):
        schedule = SCHEDULES[schedule]
    st = lib.la_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale), _ptr(h0),
                            _ptr(state_indices), _ptr(cu_seqlens), _ptr(o), _ptr(h_final),
                            int(B), int(T), int(N), int(H), int(HV), int(D), int(V), int(pool),
                            int(schedule), _ptr(dev_error), ctypes.c_void_p(stream))
    if st != 0:
        _raise(lib, st)
    return o


def la_prefill_segmented_workspace(B, T, N, HV, packed, segment_len=0):
    """(workspace bytes, resolved segment length) of la_prefill_fwd_segmented for these sizes.

    segment_len 0 = automatic (uses the current device's SM count); both values are 0 when
    the call would run la_prefill_fwd unchanged."""
    lib = load_library()
    nbytes = ctypes.c_size_t(0)
    seg = ctypes.c_int(0)
    st = lib.la_prefill_segmented_workspace(int(B), int(T), int(N), int(HV), int(bool(packed)), int(segment_len),
                                            ctypes.byref(nbytes), ctypes.byref(seg))
    if st != 0:
        _raise(lib, st)
    return nbytes.value, seg.value


def la_prefill_fwd_segmented(q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None, o=None,
                             h_final=None, seq_len=None, segment_len=0, workspace=None, dev_error=None,
                             stream=None):
    """la_prefill_fwd with every sequence cut into segments of ``segment_len`` tokens (0 =
    automatic) that run in parallel from their exact initial states.

    Arguments as la_prefill_fwd; ``workspace`` is a CUDA uint8 tensor of at least
    la_prefill_segmented_workspace(...)[0] bytes, allocated here when None.  Returns ``o``."""
    import torch
    lib = load_library()
    o, B, T, N, H, HV, D, V, pool, stream = _prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o,
                                                          h_final, seq_len, dev_error, stream)
    if workspace is None:
        nbytes, _ = la_prefill_segmented_workspace(B, T, N, HV, cu_seqlens is not None, segment_len)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device) if nbytes else None
    if workspace is not None:
        _check(workspace, "workspace", torch.uint8, 1)
    st = lib.la_prefill_fwd_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale), _ptr(h0),
                                      _ptr(state_indices), _ptr(cu_seqlens), _ptr(o), _ptr(h_final),
                                      int(B), int(T), int(N), int(H), int(HV), int(D), int(V), int(pool),
                                      int(segment_len), _ptr(workspace),
                                      ctypes.c_size_t(0 if workspace is None else workspace.numel()),
                                      _ptr(dev_error), ctypes.c_void_p(stream))
    if st != 0:
        _raise(lib, st)
    return o


def la_prefill_fwd_segmented_static(q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None,
                                    o=None, h_final=None, seq_len=None, segment_len=0, dev_error=None,
                                    stream=None):
    """la_prefill_fwd_segmented with the scratch taken from the library's built-in 16 MiB
    device buffer instead of a workspace, for callers that cannot allocate device memory.
    Calls share that buffer: calls that overlap on the GPU race.  Returns ``o``."""
    lib = load_library()
    o, B, T, N, H, HV, D, V, pool, stream = _prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o,
                                                          h_final, seq_len, dev_error, stream)
    st = lib.la_prefill_fwd_segmented_static(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale),
                                             _ptr(h0), _ptr(state_indices), _ptr(cu_seqlens), _ptr(o),
                                             _ptr(h_final), int(B), int(T), int(N), int(H), int(HV), int(D),
                                             int(V), int(pool), int(segment_len), _ptr(dev_error),
                                             ctypes.c_void_p(stream))
    if st != 0:
        _raise(lib, st)
    return o


def la_prefill_d256_workspace(B, T, N, HV, has_state):
    """Bytes of device workspace la_prefill_fwd_d256 needs for these sizes."""
    lib = load_library()
    nbytes = ctypes.c_size_t(0)
    st = lib.la_prefill_d256_workspace(int(B), int(T), int(N), int(HV), int(bool(has_state)), ctypes.byref(nbytes))
    if st != 0:
        _raise(lib, st)
    return nbytes.value


def la_prefill_fwd_d256(q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None, o=None,
                        h_final=None, seq_len=None, workspace=None, dev_error=None, stream=None):
    """la_prefill_fwd at head dimension D = V = 256 (q, k [tokens, H, 256], v [tokens, HV, 256],
    states [P, HV, 256, 256]), run as four 128 x 128 state blocks by the D = 128 kernel.

    Arguments as la_prefill_fwd; ``workspace`` is a CUDA uint8 tensor of at least
    la_prefill_d256_workspace(...) bytes, allocated here when None.  Returns ``o``."""
    import torch
    lib = load_library()
    o, B, T, N, H, HV, D, V, pool, stream = _prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o,
                                                          h_final, seq_len, dev_error, stream)
    if workspace is None:
        nbytes = la_prefill_d256_workspace(B, T, N, HV, h0 is not None or h_final is not None)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8, 1)
    st = lib.la_prefill_fwd_d256(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale), _ptr(h0),
                                 _ptr(state_indices), _ptr(cu_seqlens), _ptr(o), _ptr(h_final), int(B), int(T),
                                 int(N), int(H), int(HV), int(D), int(V), int(pool), _ptr(workspace),
                                 ctypes.c_size_t(workspace.numel()), _ptr(dev_error), ctypes.c_void_p(stream))
    if st != 0:
        _raise(lib, st)
    return o


def la_prefill_d256_segmented_workspace(B, T, N, HV, packed, segment_len, has_state):
    """(bytes, resolved segment length) of device workspace la_prefill_fwd_d256_segmented needs."""
    lib = load_library()
    nbytes, res = ctypes.c_size_t(0), ctypes.c_int(0)
    st = lib.la_prefill_d256_segmented_workspace(int(B), int(T), int(N), int(HV), int(bool(packed)), int(segment_len),
                                                 int(bool(has_state)), ctypes.byref(nbytes), ctypes.byref(res))
    if st != 0:
        _raise(lib, st)
    return nbytes.value, res.value


def la_prefill_fwd_d256_segmented(q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None, o=None,
                                  h_final=None, seq_len=None, segment_len=0, workspace=None, dev_error=None,
                                  stream=None):
    """la_prefill_fwd_d256 with every sequence cut into segments of ``segment_len`` tokens (0 =
    automatic) that run in parallel from their exact initial states; ``workspace`` as
    la_prefill_d256_segmented_workspace(...)[0] bytes, allocated here when None.  Returns ``o``."""
    import torch
    lib = load_library()
    o, B, T, N, H, HV, D, V, pool, stream = _prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, o,
                                                          h_final, seq_len, dev_error, stream)
    if workspace is None:
        nbytes, _ = la_prefill_d256_segmented_workspace(B, T, N, HV, cu_seqlens is not None, segment_len,
                                                        h0 is not None or h_final is not None)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8, 1)
    st = lib.la_prefill_fwd_d256_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale), _ptr(h0),
                                           _ptr(state_indices), _ptr(cu_seqlens), _ptr(o), _ptr(h_final), int(B),
                                           int(T), int(N), int(H), int(HV), int(D), int(V), int(pool),
                                           int(segment_len), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                           _ptr(dev_error), ctypes.c_void_p(stream))
    if st != 0:
        _raise(lib, st)
    return o


def la_prefill_bwd_workspace(B, T, H, HV, D, pool_size, has_h0, has_dh_final):
    """Bytes of device workspace la_prefill_bwd needs for these sizes."""
    lib = load_library()
    nbytes = ctypes.c_size_t(0)
    st = lib.la_prefill_bwd_workspace(int(B), int(T), int(H), int(HV), int(D), int(pool_size), int(bool(has_h0)),
                                      int(bool(has_dh_final)), ctypes.byref(nbytes))
    if st != 0:
        _raise(lib, st)
    return nbytes.value


def la_prefill_bwd(q, k, v, slopes, scale, dout, h0=None, dh_final=None, state_indices=None, cu_seqlens=None,
                   dq=None, dk=None, dv=None, dh0=None, seq_len=None, workspace=None, dev_error=None, stream=None):
    """Gradients of the prefill (include/la_backward.h): given dout = dL/do [tokens, HV, D] BF16
    and dh_final = dL/dh_final [P, HV, D, D] FP32 (or None), returns (dq, dk, dv, dh0) with the
    layouts of q, k, v and h0 (dh0 only when a tensor is passed in).  HV a multiple of H (GVA);
    the other arguments as la_prefill_fwd.  ``workspace`` is a CUDA uint8 tensor of at least
    la_prefill_bwd_workspace(...) bytes, allocated here when None."""
    import torch
    lib = load_library()
    _check(dout, "dout", torch.bfloat16, 3)
    _check(dh_final, "dh_final", torch.float32, 4)
    _check(dh0, "dh0", torch.float32, 4)
    if dout is None or dout.shape != v.shape:
        raise ValueError("dout must have the shape of v")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, name, ref in ((dq, "dq", q), (dk, "dk", k), (dv, "dv", v)):
        _check(t, name, torch.bfloat16, 3)
        if t.shape != ref.shape:
            raise ValueError(f"{name} must have the shape of its input")
    # the forward's checks and sizes: dv has the layout of o, dh0 (else dh_final) that of h_final
    _, B, T, N, H, HV, D, V, pool, stream = _prefill_args(q, k, v, slopes, h0, state_indices, cu_seqlens, dv,
                                                          dh0 if dh0 is not None else dh_final, seq_len, dev_error,
                                                          stream)
    if workspace is None:
        nbytes = la_prefill_bwd_workspace(B, T, H, HV, D, pool, h0 is not None, dh_final is not None)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8, 1)
    st = lib.la_prefill_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale), _ptr(h0), _ptr(dout),
                            _ptr(dh_final), _ptr(state_indices), _ptr(cu_seqlens), _ptr(dq), _ptr(dk), _ptr(dv),
                            _ptr(dh0), int(B), int(T), int(N), int(H), int(HV), int(D), int(V), int(pool),
                            _ptr(workspace), ctypes.c_size_t(workspace.numel()), _ptr(dev_error),
                            ctypes.c_void_p(stream))
    if st != 0:
        _raise(lib, st)
    return dq, dk, dv, dh0


def _decode_common(q, k, v, slopes, state, state_indices, T, dev_error, stream):
    """Shape checks shared by the speculative-decoding ops; returns (lib, B, H, HV, pool, stream)."""
    import torch
    lib = load_library()
    for t, name, dt, nd in ((q, "q", torch.bfloat16, 3), (k, "k", torch.bfloat16, 3), (v, "v", torch.bfloat16, 3),
                            (slopes, "slopes", torch.float32, 1), (state, "state", torch.float32, 4),
                            (state_indices, "state_indices", torch.int32, 1), (dev_error, "dev_error", torch.int32, 1)):
        _check(t, name, dt, nd)
    T = int(T)
    if T < 1:
        raise ValueError("T must be >= 1")
    tokens, H, D = q.shape
    _, HV, V = v.shape
    if k.shape != q.shape or v.shape[0] != tokens or tokens % T:
        raise ValueError("q, k: [B*T, H, D]; v: [B*T, HV, V] with the same B*T")
    B = tokens // T
    if tuple(state.shape[1:]) != (HV, V, D):
        raise ValueError("state must be [P, HV, V, D]")
    if state_indices is not None and state_indices.shape[0] != B:
        raise ValueError("state_indices must have B entries")
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    return lib, B, H, HV, state.shape[0], stream


def _raise(lib, st):
    if st != 0:
        raise LaError(st, lib.la_status_string(st).decode(), lib.la_last_error().decode())


def la_decode_mtp(q, k, v, slopes, scale, state, T, state_indices=None, o=None, dev_error=None, stream=None):
    """Multi-token decode: advance each request's pooled state over its T draft tokens (in
    place) and return the outputs o (bf16 [B*T, HV, V]; D = V = 128 or 64)."""
    import torch
    lib, B, H, HV, pool, stream = _decode_common(q, k, v, slopes, state, state_indices, T, dev_error, stream)
    if o is None:
        o = torch.empty(v.shape, dtype=torch.bfloat16, device=q.device)
    _check(o, "o", torch.bfloat16, 3)
    _raise(lib, lib.la_decode_mtp(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale), _ptr(state),
                                  _ptr(state_indices), _ptr(o), B, int(T), H, HV, q.shape[2], v.shape[2], pool,
                                  _ptr(dev_error), ctypes.c_void_p(stream)))
    return o


def la_verify(q, k, v, slopes, scale, state, T, state_indices=None, o=None, kbuf=None, vbuf=None, dev_error=None,
              stream=None):
    """Parallel verify: the outputs of all T draft tokens from the pooled states, which are
    left untouched; with kbuf/vbuf (bf16 [P, T, H, D] / [P, T, HV, V]) the draft k, v
    are copied to the request's slot for la_commit.  Returns o."""
    import torch
    lib, B, H, HV, pool, stream = _decode_common(q, k, v, slopes, state, state_indices, T, dev_error, stream)
    if o is None:
        o = torch.empty(v.shape, dtype=torch.bfloat16, device=q.device)
    _check(o, "o", torch.bfloat16, 3)
    _check(kbuf, "kbuf", torch.bfloat16, 4)
    _check(vbuf, "vbuf", torch.bfloat16, 4)
    _raise(lib, lib.la_verify(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), ctypes.c_float(scale), _ptr(state),
                              _ptr(state_indices), _ptr(o), _ptr(kbuf), _ptr(vbuf), B, int(T), H, HV, q.shape[2],
                              v.shape[2], pool, _ptr(dev_error), ctypes.c_void_p(stream)))
    return o


def la_commit(state, kbuf, vbuf, accepted_len, slopes, state_indices=None, dev_error=None, stream=None):
    """Commit: advance each request's pooled state (in place) by its accepted prefix of the
    draft tokens held in kbuf/vbuf; accepted_len is int32 [B] (0 = no-op)."""
    import torch
    lib = load_library()
    _check(state, "state", torch.float32, 4)
    _check(kbuf, "kbuf", torch.bfloat16, 4)
    _check(vbuf, "vbuf", torch.bfloat16, 4)
    _check(accepted_len, "accepted_len", torch.int32, 1)
    _check(slopes, "slopes", torch.float32, 1)
    _check(state_indices, "state_indices", torch.int32, 1)
    _check(dev_error, "dev_error", torch.int32, 1)
    P, T, H, D = kbuf.shape
    HV, V = state.shape[1], state.shape[2]
    if tuple(vbuf.shape) != (P, T, HV, V) or state.shape[0] != P:
        raise ValueError("kbuf [P, T, H, D], vbuf [P, T, HV, V] and state [P, HV, V, D] must agree")
    B = accepted_len.shape[0]
    if stream is None:
        stream = torch.cuda.current_stream(state.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    _raise(lib, lib.la_commit(_ptr(state), _ptr(state_indices), _ptr(kbuf), _ptr(vbuf), _ptr(accepted_len),
                              _ptr(slopes), B, T, H, HV, D, V, P, _ptr(dev_error), ctypes.c_void_p(stream)))
    return state


def la_prefill_fwd_raw(*args):
    """Call the C entry point with raw integers / pointers (argument order of the header)."""
    return load_library().la_prefill_fwd(*args)
