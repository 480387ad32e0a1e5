"""Seeded random problems through the prefill, segmented-prefill and backward entry points,
each compared with the FP64 oracle element by element.

Each case draws, from its own seed, a batch that the hand-picked cases may not reach:
- fixed or packed, with sequence lengths from 0 to a few hundred tokens (so empty, short and
  ragged sequences, and both the tokenwise and the chunkwise kernel);
- 1 to 3 q/k heads with 1 to 3 value heads each;
- D = 128 or 64;
- an optional state pool with padded (-1) indices, updated in place or written to separate
  final states, with or without h0 and h_final;
- slopes mixing the workloads' default slopes with 0 (lambda = 1) and large values.

Bounds are those of the hand-picked cases (harness.check_output / check_state and the
backward's). Rows that are not written and slots that are not selected must stay untouched.
"""
import numpy as np
import pytest

import workloads as W
from harness import compare_full, run_gpu, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SEEDS = list(range(64))


def _draw(seed):
    """(keyword arguments of workloads.custom, segment length) for one random case."""
    rng = np.random.default_rng(20261203 + seed)
    D = int(rng.choice([128, 64]))
    H = int(rng.integers(1, 4))
    HV = H * int(rng.integers(1, 4))
    kw = dict(H=H, HV=HV, D=D)
    packed = bool(rng.integers(0, 2))
    if packed:
        n = int(rng.integers(1, 7))
        # lengths: mostly a few chunks, some short or empty
        lens = [int(x) for x in rng.choice([0, 1, 7, 31, 32, 33, 63, 64, 65, 127, 200, 333, 400], size=n)]
        kw["lengths"] = lens
    else:
        n = int(rng.integers(1, 4))
        kw["B"] = n
        kw["T"] = int(rng.choice([1, 17, 32, 33, 64, 100, 191, 256, 300]))
    kw["with_h0"] = bool(rng.random() < 0.8)
    if rng.integers(0, 2):
        # a pool holds initial states (its size is h0's first dimension)
        pool = n + int(rng.integers(0, 4))
        idx = rng.permutation(pool)[:n].astype(np.int64)
        pad = rng.random(n) < 0.25
        idx[pad] = -1
        kw["pool"] = pool
        kw["indices"] = [int(x) for x in idx]
        kw["in_place"] = bool(rng.integers(0, 2))
        kw["with_h0"] = True
    kw["want_final"] = bool(rng.random() < 0.85)
    if rng.random() < 0.4:
        sl = W.slopes_for(HV).astype(np.float32)
        special = rng.random(HV) < 0.5
        sl[special] = rng.choice([0.0, 1.0 / 256, 0.5, 3.0, 100.0], size=int(special.sum())).astype(np.float32)
        kw["slopes"] = [float(x) for x in sl]
    seg = int(rng.choice([0, 64, 128, 192, 320]))
    return kw, seg


@pytest.mark.parametrize("seed", SEEDS)
def test_random_prefill(seed):
    kw, _ = _draw(seed)
    p = W.custom(seed=seed, name=f"random {seed}", **kw)
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, f"random {seed} {kw}")


@pytest.mark.parametrize("seed", SEEDS)
def test_random_segmented(seed):
    import linear_attention_prefill_chunkwise_gb300 as lap
    kw, seg = _draw(seed)
    p = W.custom(seed=seed, name=f"random segmented {seed}", **kw)
    d = upload(p)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lap.la_prefill_fwd_segmented(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], state_indices=d["idx"],
                                 cu_seqlens=d["cu"], o=d["o"], h_final=d["h_final"],
                                 seq_len=None if p.cu_seqlens is not None else p.T, segment_len=seg, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    compare_full(p, d, f"random segmented {seed} (segment {seg}) {kw}")


@pytest.mark.parametrize("seed", SEEDS)
def test_random_backward(seed):
    from test_gpu_backward import _compare
    kw, _ = _draw(seed)
    # the backward has no in-place pool and no h_final; dL/dh_final stands in for the latter
    kw.pop("in_place", None)
    with_dhf = kw.pop("want_final")
    rng = np.random.default_rng(7000 + seed)
    p = W.custom(seed=seed, name=f"random backward {seed}", **kw)
    dout = W.bf16_bits(rng.standard_normal((p.tokens, p.HV, p.V), dtype=np.float32))
    dhf = (rng.standard_normal((p.pool_size, p.HV, p.V, p.D), dtype=np.float32) * np.float32(0.1)) if with_dhf else None
    _compare(p, dout, dhf, f"random backward {seed} {kw}", want_dh0=bool(seed % 3))


def _draw_decode(seed):
    """Arguments of test_gpu_decode.make_case for one random speculative-decoding batch: up to
    40 requests of 1 to 17 draft tokens (both sides of the tensor-core verify's 8-token limit),
    GVA groups, a pool larger than the batch with padded requests, mixed special slopes, and
    D = V = 128, 64 or 256."""
    rng = np.random.default_rng(31000 + seed)
    H = int(rng.integers(1, 5))
    HV = H * int(rng.integers(1, 4))
    B = int(rng.integers(1, 41))
    T = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 12, 16, 17]))
    kw = dict(seed=32000 + seed, B=B, T=T, H=H, HV=HV, P=B + int(rng.integers(0, 9)),
              n_pad=int(rng.integers(0, B // 4 + 1)))
    if rng.random() < 0.4:
        sl = W.slopes_for(HV).astype(np.float32)
        special = rng.random(HV) < 0.5
        sl[special] = rng.choice([0.0, 1e-4, 0.7, 5.0, 40.0, 200.0], size=int(special.sum())).astype(np.float32)
        kw["slopes"] = [float(x) for x in sl]
    kw["D"] = int(rng.choice([128, 128, 64, 256]))
    return kw


@pytest.mark.parametrize("seed", range(32))
def test_random_decode_ops(seed):
    from test_gpu_decode import check_decode_mtp, check_verify_then_commit, make_case
    kw = _draw_decode(seed)
    c = make_case(**kw)
    check_decode_mtp(c, f"random decode {seed} {kw}")
    check_verify_then_commit(c, f"random verify/commit {seed} {kw}", 33000 + seed)
