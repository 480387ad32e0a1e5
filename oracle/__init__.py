"""Plain, slow, FP64 CPU oracle for the Lightning Attention chunkwise prefill.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA path and never imports it.

Contents:
  * ``tokenwise`` / ``chunked`` -- ctypes wrappers over ``la_oracle.c``: the
    decayed recurrence h_t = lambda h_{t-1} + k_t^T v_t, o_t = scale q_t h_t
    (page "[Lightning Attention] Add Hopper SM90 CuTe DSL prefill",
    Description), evaluated token by token, and in the chunkwise form
    (intra (QK^T masked by the causal decay) V + inter lambda^(s+1) Q S, one
    state advance per chunk).
  * ``backward`` -- gradients of a scalar loss through the same recurrence (dq, dk, dv and
    dh0 from dL/do and dL/dh_final), one forward and one reverse sweep per unit.
  * ``closed_form`` -- the direct O(T^2) sum printed on page "[LA] Lightning
    Attention MTP decode + KVBuffer parallel verify / commit", Description
    ("Closed form used by verify"):
        o_t = lambda^(t+1) scale (h0 . q_t) + sum_{i<=t} lambda^(t-i) scale (q_t . k_i) v_i
    written with numpy, for one (sequence, head) at a time, tiny T only.

State orientation is [V, K] (page "[Lightning Attention] Add Hopper SM90 CuTe
DSL prefill", Reviewer notes): S[v][k] multiplies q[k] and produces o[v].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblaoracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {-1: "bad shape", -2: "bad cu_seqlens", -3: "state index out of range", -4: "out of memory"}


def build(force: bool = False) -> str:
    """Compile la_oracle.c into oracle/_build/liblaoracle.so (FP64, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            fp = ctypes.POINTER(ctypes.c_float)
            ip = ctypes.POINTER(ctypes.c_int32)
            dp = ctypes.POINTER(ctypes.c_double)
            common = [fp, fp, fp, fp, ctypes.c_double, dp, ip, ip] + [ctypes.c_int] * 7 + [dp, dp]
            lib.la_oracle_tokenwise.argtypes = common + [ctypes.c_int]
            lib.la_oracle_tokenwise.restype = ctypes.c_int
            lib.la_oracle_chunked.argtypes = common + [ctypes.c_int, ctypes.c_int]
            lib.la_oracle_chunked.restype = ctypes.c_int
            lib.la_oracle_backward.argtypes = [fp, fp, fp, fp, ctypes.c_double, dp, fp, dp, ip, ip] + \
                [ctypes.c_int] * 7 + [dp, dp, dp, dp, ctypes.c_int]
            lib.la_oracle_backward.restype = ctypes.c_int
            lib.la_oracle_max_threads.argtypes = []
            lib.la_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
        return _lib


def max_threads() -> int:
    return int(_load().la_oracle_max_threads())


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _run(kind, q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None, T=None,
         o=None, h_final=None, want_state=True, chunk=64, nthreads=0):
    q, k, v, slopes = _f32(q), _f32(k), _f32(v), _f32(slopes)
    h0 = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
    tokens, H, D = q.shape
    _, HV, V = v.shape
    if cu_seqlens is not None:
        cu_seqlens = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = cu_seqlens.shape[0] - 1
        T = 0
    else:
        if T is None:
            raise ValueError("fixed-length mode needs T")
        N = tokens // T if T > 0 else 0
    if state_indices is not None:
        state_indices = np.ascontiguousarray(state_indices, dtype=np.int32)
        if h0 is not None:
            pool = h0.shape[0]
        elif h_final is not None:
            pool = h_final.shape[0]
        else:
            pool = int(state_indices.max(initial=-1)) + 1
    else:
        pool = N
    if o is None:
        o = np.full((tokens, HV, V), np.nan, dtype=np.float64)
    if h_final is None and want_state:
        h_final = np.full((pool, HV, V, D), np.nan, dtype=np.float64)
    if h_final is not None:
        assert h_final.dtype == np.float64 and h_final.flags.c_contiguous
    assert o.dtype == np.float64 and o.flags.c_contiguous
    lib = _load()
    args = [_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
            _ptr(slopes, ctypes.c_float), float(scale), _ptr(h0, ctypes.c_double),
            _ptr(state_indices, ctypes.c_int32), _ptr(cu_seqlens, ctypes.c_int32),
            int(N), int(T), int(H), int(HV), int(D), int(V), int(pool),
            _ptr(o, ctypes.c_double), _ptr(h_final, ctypes.c_double)]
    if kind == "tokenwise":
        rc = lib.la_oracle_tokenwise(*args, int(nthreads))
    else:
        rc = lib.la_oracle_chunked(*args, int(chunk), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the problem: {ERRORS.get(rc, rc)}")
    return o, h_final


def tokenwise(q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None, T=None,
              o=None, h_final=None, want_state=True, nthreads=0):
    """Tokenwise FP64 recurrence.

    q, k: [tokens, H, D]; v: [tokens, HV, V] (float32 values of the BF16 inputs);
    slopes: [HV]; h0: [P, HV, V, D] or None.  Returns (o [tokens, HV, V] f64,
    h_final [P, HV, V, D] f64 or None).  Rows of padded sequences and pool slots
    not selected keep the value of ``o`` / ``h_final`` passed in (NaN when the
    oracle allocates them).
    """
    return _run("tokenwise", q, k, v, slopes, scale, h0, state_indices, cu_seqlens, T, o,
                h_final, want_state, nthreads=nthreads)


def chunked(q, k, v, slopes, scale, h0=None, state_indices=None, cu_seqlens=None, T=None,
            o=None, h_final=None, want_state=True, chunk=64, nthreads=0):
    """Chunkwise FP64 evaluation (intra + inter + one state advance per chunk)."""
    return _run("chunked", q, k, v, slopes, scale, h0, state_indices, cu_seqlens, T, o,
                h_final, want_state, chunk=chunk, nthreads=nthreads)


def closed_form(q, k, v, slope, scale, h0=None):
    """Direct closed-form sum for one (sequence, head), numpy FP64, tiny T only.

    q, k: [T, D]; v: [T, V]; h0: [V, D] or None.  Returns (o [T, V], h_T [V, D]),
    where h_T = lambda^T h0 + sum_i lambda^(T-1-i) v_i k_i^T is the state the
    same sum implies after the last token.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, D = q.shape
    V = v.shape[1]
    lam = np.exp(-np.float64(slope))
    h0 = np.zeros((V, D)) if h0 is None else np.asarray(h0, dtype=np.float64)
    o = np.zeros((T, V))
    for t in range(T):
        term1 = lam ** (t + 1) * scale * (h0 @ q[t])
        term2 = np.zeros(V)
        for i in range(t + 1):
            term2 += lam ** (t - i) * scale * float(q[t] @ k[i]) * v[i]
        o[t] = term1 + term2
    hT = lam ** T * h0
    for i in range(T):
        hT = hT + lam ** (T - 1 - i) * np.outer(v[i], k[i])
    return o, hT


def backward(q, k, v, slopes, scale, dout, h0=None, dh_final=None, state_indices=None, cu_seqlens=None,
             T=None, want_dh0=True, nthreads=0):
    """Gradients of a scalar loss L through the recurrence, FP64 (``la_oracle.c``,
    la_oracle_backward): given dout = dL/do [tokens, HV, V] and dh_final = dL/dh_final
    [P, HV, V, D] (or None = 0), returns (dq [tokens, H, D], dk [tokens, H, D],
    dv [tokens, HV, V], dh0 [P, HV, V, D] or None).  Rows of padded sequences and unselected
    slots are NaN."""
    q, k, v, slopes, dout = _f32(q), _f32(k), _f32(v), _f32(slopes), _f32(dout)
    h0 = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
    dh_final = None if dh_final is None else np.ascontiguousarray(dh_final, dtype=np.float64)
    tokens, H, D = q.shape
    _, HV, V = v.shape
    if cu_seqlens is not None:
        cu_seqlens = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = cu_seqlens.shape[0] - 1
        T = 0
    else:
        if T is None:
            raise ValueError("fixed-length mode needs T")
        N = tokens // T if T > 0 else 0
    if state_indices is not None:
        state_indices = np.ascontiguousarray(state_indices, dtype=np.int32)
        pool = next((a.shape[0] for a in (h0, dh_final) if a is not None), int(state_indices.max(initial=-1)) + 1)
    else:
        pool = N
    dq = np.full((tokens, H, D), np.nan)
    dk = np.full((tokens, H, D), np.nan)
    dv = np.full((tokens, HV, V), np.nan)
    dh0 = np.full((pool, HV, V, D), np.nan) if want_dh0 else None
    lib = _load()
    rc = lib.la_oracle_backward(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                                _ptr(slopes, ctypes.c_float), float(scale), _ptr(h0, ctypes.c_double),
                                _ptr(dout, ctypes.c_float), _ptr(dh_final, ctypes.c_double),
                                _ptr(state_indices, ctypes.c_int32), _ptr(cu_seqlens, ctypes.c_int32),
                                int(N), int(T), int(H), int(HV), int(D), int(V), int(pool),
                                _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
                                _ptr(dh0, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the problem: {ERRORS.get(rc, rc)}")
    return dq, dk, dv, dh0
