"""The backward pass (include/la_backward.h) through the C ABI against the FP64 oracle's
backward, which finite differences of the forward oracle pin (tests/test_oracle.py).

dq, dk and dv are BF16 like the forward's output and get its bounds (rel RMS <= 2e-3, max
|error| <= 1e-2 max |g| per tensor); dh0 is FP32 like the final state (rel RMS <= 1e-3, or
within 1e-30 where the exact values lie below FP32's normal range).  Rows of padded sequences and unselected slots must stay untouched.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from harness import O_MAX_ABS_FRAC, O_REL_RMS, STATE_REL_RMS, rel_rms, to_torch_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _grad_problem(seed, D=128, with_dhf=True, **kw):
    p = W.custom(seed=seed, D=D, **kw)
    rng = np.random.default_rng(seed + 1)
    dout = W.bf16_bits(rng.standard_normal((p.tokens, p.HV, p.V), dtype=np.float32))
    dhf = (rng.standard_normal((p.pool_size, p.HV, p.V, p.D), dtype=np.float32) * np.float32(0.1)) if with_dhf else None
    return p, dout, dhf


def _run(p, dout, dhf, want_dh0=True):
    import linear_attention_prefill_chunkwise_gb300 as lap
    dev = "cuda"
    q, k, v = (to_torch_bf16(b, dev) for b in (p.q_bits, p.k_bits, p.v_bits))
    sl = torch.from_numpy(p.slopes).to(dev)
    h0 = None if p.h0 is None else torch.from_numpy(p.h0).to(dev)
    dh_final = None if dhf is None else torch.from_numpy(dhf).to(dev)
    idx = None if p.state_indices is None else torch.from_numpy(p.state_indices).to(dev)
    cu = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).to(dev)
    poison = float("nan")
    dq, dk, dv = (torch.full_like(t, poison) for t in (q, k, v))
    dh0 = torch.full((p.pool_size, p.HV, p.V, p.D), poison, dtype=torch.float32, device=dev) if want_dh0 else None
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lap.la_prefill_bwd(q, k, v, sl, p.scale, to_torch_bf16(dout, dev), h0=h0, dh_final=dh_final, state_indices=idx,
                       cu_seqlens=cu, dq=dq, dk=dk, dv=dv, dh0=dh0, seq_len=None if cu is not None else p.T,
                       dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return (dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy(),
            None if dh0 is None else dh0.cpu().numpy())


def _check_grad(name, g, ref, label):
    live = ~np.isnan(ref[:, 0, 0])
    assert np.all(np.isnan(g[~live])), f"{label}: {name} written for padded rows"
    if not live.any():
        return
    g, ref = g[live], ref[live]
    assert np.all(np.isfinite(g)), f"{label}: non-finite {name}"
    r = rel_rms(g, ref)
    ma = float(np.max(np.abs(g - ref)))
    assert r <= O_REL_RMS, f"{label}: {name} rel RMS {r:.3e}"
    assert ma <= O_MAX_ABS_FRAC * float(np.max(np.abs(ref))) + 1e-30, f"{label}: {name} max abs {ma:.3e}"


def _compare(p, dout, dhf, label, want_dh0=True):
    dq, dk, dv, dh0 = _run(p, dout, dhf, want_dh0)
    rq, rk, rv, rh = oracle.backward(p.q(), p.k(), p.v(), p.slopes, p.scale, W.bf16_to_f32(dout),
                                     h0=None if p.h0 is None else p.h0.astype(np.float64),
                                     dh_final=None if dhf is None else dhf.astype(np.float64),
                                     state_indices=p.state_indices, cu_seqlens=p.cu_seqlens,
                                     T=None if p.cu_seqlens is not None else p.T, want_dh0=want_dh0)
    for name, g, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _check_grad(name, g, ref, label)
    if want_dh0:
        sel = ~np.isnan(rh[:, 0, 0, 0])
        assert np.all(np.isnan(dh0[~sel])), f"{label}: dh0 written for unselected slots"
        if sel.any():
            # states below FP32's normal range (lambda^n with large slopes) only need to be tiny
            r = rel_rms(dh0[sel], rh[sel])
            ma = float(np.max(np.abs(dh0[sel] - rh[sel])))
            assert r <= STATE_REL_RMS or ma <= 1e-30, f"{label}: dh0 rel RMS {r:.3e}, max abs {ma:.3e}"
    return dq, dk, dv, dh0


BWD_CASES = {
    "fixed_T300": dict(B=2, T=300, H=2, HV=2),
    "packed_ragged_pool": dict(lengths=[1, 63, 64, 65, 130, 0, 200, 31], H=2, HV=2, pool=11,
                               indices=[3, 10, -1, 0, 7, 5, 1, 9]),
    "no_h0_no_dh_final": dict(lengths=[70, 3, 129], H=1, HV=1, with_h0=False),
    "lambda_one": dict(lengths=[150, 20], H=2, HV=2, slopes=[0.0, 0.0]),
    "lambda_zero": dict(lengths=[150, 20], H=2, HV=2, slopes=[100.0, 100.0]),
    "short_sequences": dict(lengths=[5, 20, 3, 31, 1, 40, 16], H=2, HV=2),
    # GVA: dq and dk summed over each q/k head's value heads
    "gva_fixed_T300": dict(B=2, T=300, H=1, HV=4),
    "gva_packed_ragged_pool": dict(lengths=[1, 63, 64, 65, 130, 0, 200, 31], H=2, HV=6, pool=11,
                                   indices=[3, 10, -1, 0, 7, 5, 1, 9]),
    "gva_short_sequences": dict(lengths=[5, 20, 3, 31, 1, 40, 16], H=2, HV=4),
    "gva_lambda_zero_and_one": dict(lengths=[150, 20], H=1, HV=4, slopes=[100.0, 0.0, 100.0, 0.5]),
}


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("name", sorted(BWD_CASES))
def test_backward_cases(name, D):
    kw = dict(BWD_CASES[name])
    with_dhf = name != "no_h0_no_dh_final"
    p, dout, dhf = _grad_problem(zlib.crc32(f"bwd{name}{D}".encode()) % 10000, D=D, with_dhf=with_dhf, **kw)
    _compare(p, dout, dhf, f"backward {name} D={D}")


def test_backward_without_dh0():
    p, dout, dhf = _grad_problem(4401, lengths=[90, 40], H=2, HV=2)
    _compare(p, dout, dhf, "backward, dh0 not requested", want_dh0=False)


def test_backward_bench_shape_every_unit():
    # B=2, T=8192, H=64 with h0 and dh_final: every (sequence, head) unit within the bounds
    p, dout, dhf = _grad_problem(4402, B=2, T=8192, H=64, HV=64)
    dq, dk, dv, dh0 = _compare(p, dout, dhf, "backward B=2 T=8192 H=64")
    assert np.all(np.isfinite(dh0))


def test_backward_is_deterministic():
    p, dout, dhf = _grad_problem(4403, lengths=[300, 77, 129], H=2, HV=2)
    a = _run(p, dout, dhf)
    b = _run(p, dout, dhf)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_backward_gva_long_sequence():
    # B=1, T=4096, H=4 q/k heads with HV=16 value heads, h0 and dh_final: every unit within bounds
    p, dout, dhf = _grad_problem(4406, B=1, T=4096, H=4, HV=16)
    _compare(p, dout, dhf, "backward GVA B=1 T=4096 H=4 HV=16")


@pytest.mark.parametrize("D,HV", [(128, 2), (64, 2), (128, 4)])
def test_backward_nonfinite_sequence_does_not_reach_its_neighbours(D, HV):
    """A packed sequence whose q, k, v and dout hold infinities and NaNs leaves the gradients of
    every other sequence bitwise as they are with finite values there: the reverse runs read,
    in a sequence's last (ragged) chunk, rows of the next sequence, which must stay out."""
    import dataclasses
    p, dout, dhf = _grad_problem(4405, D=D, lengths=[70, 100, 45, 130], H=2, HV=HV, pool=6, indices=[4, 1, 5, 0])
    clean = _run(p, dout, dhf)
    a, b = int(p.cu_seqlens[1]), int(p.cu_seqlens[2])
    bits = {n: getattr(p, n).copy() for n in ("q_bits", "k_bits", "v_bits")}
    inf, nan, ninf = np.uint16(0x7F80), np.uint16(0x7FC0), np.uint16(0xFF80)
    bits["q_bits"][a] = ninf
    bits["k_bits"][a + 3, :, :5] = inf
    bits["v_bits"][b - 1] = nan
    dout_bad = dout.copy()
    dout_bad[a + 50] = inf
    bad = _run(dataclasses.replace(p, **bits), dout_bad, dhf)
    keep = np.r_[0:a, b:p.tokens]
    for name, x, y in zip(("dq", "dk", "dv"), clean[:3], bad[:3]):
        assert np.array_equal(x[keep].view(np.uint32), y[keep].view(np.uint32)), f"{name} of a neighbour changed"
    slots = [4, 5, 0]  # the other sequences' slots
    assert np.array_equal(clean[3][slots].view(np.uint32), bad[3][slots].view(np.uint32)), "dh0 of a neighbour changed"


def test_backward_gva_in_a_cuda_graph():
    """The whole GVA backward (chunkwise runs, FP32 parts, group sums, state kernels) captured in
    one CUDA graph replays bitwise like the eager call: no host synchronisation, no allocation."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    p, dout, dhf = _grad_problem(4407, lengths=[90, 40, 130], H=1, HV=2, pool=4, indices=[3, 0, 1])
    eager = _run(p, dout, dhf)
    dev = "cuda"
    q, k, v = (to_torch_bf16(b, dev) for b in (p.q_bits, p.k_bits, p.v_bits))
    sl = torch.from_numpy(p.slopes).to(dev)
    h0 = torch.from_numpy(p.h0).to(dev)
    dh_final = torch.from_numpy(dhf).to(dev)
    idx = torch.from_numpy(p.state_indices).to(dev)
    cu = torch.from_numpy(p.cu_seqlens).to(dev)
    do = to_torch_bf16(dout, dev)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    dh0 = torch.full((p.pool_size, p.HV, p.V, p.D), float("nan"), dtype=torch.float32, device=dev)
    nbytes = lap.la_prefill_bwd_workspace(1, p.tokens, p.H, p.HV, p.D, p.pool_size, True, True)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lap.la_prefill_bwd(q, k, v, sl, p.scale, do, h0=h0, dh_final=dh_final, state_indices=idx, cu_seqlens=cu,
                           dq=dq, dk=dk, dv=dv, dh0=dh0, workspace=ws)
    for _ in range(3):
        for t in (dq, dk, dv, dh0):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for got, want in zip((dq, dk, dv, dh0), eager):
            assert np.array_equal(got.float().cpu().numpy().view(np.uint32), want.view(np.uint32))
