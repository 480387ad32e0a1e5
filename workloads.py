"""Seeded synthetic inputs for the Lightning Attention prefill.

This module only draws and rounds random numbers: it holds none of the
method's arithmetic and is the one piece both the oracle-side tests and the
CUDA-side tests and benchmark use.

Recipe (the workloads named on page "[Lightning Attention] Add Hopper SM90 CuTe
DSL prefill", Description and Canonical CuTe vs FLA baseline: BF16 Q/K/V, FP32
decay and state, D = V = 128):
  * numpy ``default_rng(seed)``; draws in float32, then round-to-nearest-even
    to BF16;
  * q, k ~ N(0, 1), each (token, head) row divided by its L2 norm before the
    rounding; v ~ N(0, 1);
  * slope_h = 2^(-8 (h + 1) / Hs) per value head, Hs the number of value heads;
  * initial states ~ N(0, 0.02^2) in float32 (0.02 read as the standard
    deviation).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

D = 128
V = 128


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (uint16), round to nearest, ties to even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True)).astype(np.float32)
    return x / n


def slopes_for(hs: int) -> np.ndarray:
    return np.array([2.0 ** (-8.0 * (h + 1) / hs) for h in range(hs)], dtype=np.float32)


@dataclass
class Problem:
    """One prefill call's inputs (host arrays) and how to interpret them."""
    name: str
    q_bits: np.ndarray                  # uint16 [tokens, H, D]
    k_bits: np.ndarray                  # uint16 [tokens, H, D]
    v_bits: np.ndarray                  # uint16 [tokens, HV, V]
    slopes: np.ndarray                  # float32 [HV]
    scale: float
    H: int
    HV: int
    B: int                              # fixed mode: batch; packed: 1
    T: int                              # fixed mode: length; packed: total tokens
    cu_seqlens: Optional[np.ndarray] = None      # int32 [N+1]
    state_indices: Optional[np.ndarray] = None   # int32 [N]
    h0: Optional[np.ndarray] = None              # float32 [P, HV, V, D]
    want_final: bool = True
    in_place: bool = False              # final states scattered into the h0 pool
    extra: dict = field(default_factory=dict)
    D: int = 128                        # q/k head dimension
    V: int = 128                        # value head dimension

    @property
    def tokens(self) -> int:
        return int(self.q_bits.shape[0])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1) if self.cu_seqlens is not None else self.B

    @property
    def pool_size(self) -> int:
        if self.h0 is not None:
            return int(self.h0.shape[0])
        return self.N

    def q(self):
        return bf16_to_f32(self.q_bits)

    def k(self):
        return bf16_to_f32(self.k_bits)

    def v(self):
        return bf16_to_f32(self.v_bits)

    def lengths(self) -> np.ndarray:
        if self.cu_seqlens is not None:
            return np.diff(self.cu_seqlens.astype(np.int64))
        return np.full(self.B, self.T, dtype=np.int64)


def make_qkv(rng, tokens, H, HV, d=D, v_dim=V):
    q = bf16_bits(_unit_rows(rng, (tokens, H, d)))
    k = bf16_bits(_unit_rows(rng, (tokens, H, d)))
    v = bf16_bits(rng.standard_normal((tokens, HV, v_dim), dtype=np.float32))
    return q, k, v


def make_states(rng, P, HV, std=0.02, d=D, v_dim=V):
    return (rng.standard_normal((P, HV, v_dim, d), dtype=np.float32) * np.float32(std)).astype(np.float32)


def custom(seed, lengths=None, B=None, T=None, H=4, HV=4, scale=None, with_h0=True,
           pool=None, indices=None, want_final=True, in_place=False, slopes=None, name="custom", D=D):
    """A small problem of any shape: fixed (B, T) or packed (``lengths``); head dimension
    D = V (128 or 64)."""
    rng = np.random.default_rng(seed)
    if lengths is not None:
        lengths = np.asarray(lengths, dtype=np.int64)
        cu = np.zeros(len(lengths) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        tokens = int(cu[-1])
        N = len(lengths)
        Bv, Tv = 1, tokens
    else:
        cu = None
        tokens = B * T
        N = B
        Bv, Tv = B, T
    d = D
    q, k, v = make_qkv(rng, tokens, H, HV, d, d)
    sl = slopes_for(HV) if slopes is None else np.asarray(slopes, dtype=np.float32)
    sc = 1.0 / math.sqrt(d) if scale is None else scale
    P = pool if pool is not None else N
    h0 = make_states(rng, P, HV, d=d, v_dim=d) if with_h0 else None
    idx = None if indices is None else np.asarray(indices, dtype=np.int32)
    return Problem(name, q, k, v, sl, sc, H, HV, Bv, Tv, cu, idx, h0, want_final, in_place, D=d, V=d)


def config(i: int) -> Problem:
    """The five benchmark workloads, seeded with 1000 + i (i = 1..5)."""
    rng = np.random.default_rng(1000 + i)
    if i == 1:
        B, T, H, HV = 1, 256, 4, 4
        q, k, v = make_qkv(rng, B * T, H, HV)
        return Problem("tiny fixed B=1 T=256 H=HV=4", q, k, v, slopes_for(HV), 1.0, H, HV, B, T)
    if i == 2:
        B, T, H, HV = 2, 8192, 64, 64
        q, k, v = make_qkv(rng, B * T, H, HV)
        h0 = make_states(rng, B, HV)
        return Problem("fixed MHA B=2 T=8192 H=HV=64, h0 + final state", q, k, v, slopes_for(HV),
                       1.0 / math.sqrt(D), H, HV, B, T, h0=h0)
    if i == 3:
        N, H, HV, P = 32, 32, 32, 64
        lengths = rng.integers(1, 4097, N)
        cu = np.zeros(N + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        tokens = int(cu[-1])
        q, k, v = make_qkv(rng, tokens, H, HV)
        h0 = make_states(rng, P, HV)
        idx = rng.permutation(P)[:N].astype(np.int32)
        return Problem("packed varlen N=32 len~U[1,4096] H=HV=32, 64-slot pool in place", q, k, v,
                       slopes_for(HV), 1.0 / math.sqrt(D), H, HV, 1, tokens, cu, idx, h0,
                       in_place=True)
    if i == 4:
        B, T, H, HV = 4, 16384, 16, 64
        q, k, v = make_qkv(rng, B * T, H, HV)
        return Problem("GVA B=4 T=16384 H=16 HV=64, zero h0, final state", q, k, v,
                       slopes_for(HV), 1.0 / math.sqrt(D), H, HV, B, T)
    if i == 5:
        N, T, H, HV, P = 128, 8, 64, 64, 256
        cu = np.arange(N + 1, dtype=np.int32) * T
        q, k, v = make_qkv(rng, N * T, H, HV)
        h0 = make_states(rng, P, HV)
        idx = rng.permutation(P)[:N].astype(np.int32)
        pad = rng.choice(N, 16, replace=False)
        idx[pad] = -1
        return Problem("short packed N=128 T=8 H=HV=64, 256-slot pool, 16 padded", q, k, v,
                       slopes_for(HV), 1.0 / math.sqrt(D), H, HV, 1, N * T, cu, idx, h0,
                       in_place=True)
    raise ValueError(f"no workload {i}")
