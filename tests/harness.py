"""Helpers shared by the GPU tests: upload a seeded problem, run the CUDA path,
run the oracle on the whole problem or on sampled (sequence, head) units, and
the accuracy metrics the acceptance bounds are stated in."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W

# Acceptance bounds for the BF16 output and the FP32 final state, measured against
# the FP64 oracle on the same BF16-rounded inputs.
O_REL_RMS = 2e-3
O_MAX_ABS_FRAC = 1e-2
STATE_REL_RMS = 1e-3


def rel_rms(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.sum(ref ** 2))
    return float(np.sqrt(np.sum((x - ref) ** 2)) / max(den, 1e-300))


def check_output(o_gpu, o_ref, label=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert np.all(np.isfinite(o_gpu)), f"{label}: non-finite output"
    r = rel_rms(o_gpu, o_ref)
    ma = float(np.max(np.abs(o_gpu - o_ref))) if o_ref.size else 0.0
    mref = float(np.max(np.abs(o_ref))) if o_ref.size else 0.0
    assert r <= O_REL_RMS, f"{label}: output rel RMS {r:.3e} > {O_REL_RMS}"
    assert ma <= O_MAX_ABS_FRAC * mref + 1e-30, f"{label}: output max abs {ma:.3e} > 1e-2 * {mref:.3e}"
    return r, ma


def check_state(h_gpu, h_ref, label=""):
    h_gpu = np.asarray(h_gpu, dtype=np.float64)
    assert np.all(np.isfinite(h_gpu)), f"{label}: non-finite state"
    r = rel_rms(h_gpu, h_ref)
    assert r <= STATE_REL_RMS, f"{label}: state rel RMS {r:.3e} > {STATE_REL_RMS}"
    return r


def to_torch_bf16(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_f32(t):
    """BF16 device tensor -> float32 numpy (the conversion is exact)."""
    return t.float().cpu().numpy()


def upload(p: W.Problem, device="cuda", poison_o=True):
    """Device tensors for a problem: q, k, v, slopes, h0 (or None), idx, cu, o, h_final."""
    import torch
    d = {}
    d["q"] = to_torch_bf16(p.q_bits, device)
    d["k"] = to_torch_bf16(p.k_bits, device)
    d["v"] = to_torch_bf16(p.v_bits, device)
    d["slopes"] = torch.from_numpy(p.slopes).to(device)
    d["h0"] = None if p.h0 is None else torch.from_numpy(p.h0).to(device)
    d["idx"] = None if p.state_indices is None else torch.from_numpy(p.state_indices).to(device)
    d["cu"] = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).to(device)
    o = torch.empty((p.tokens, p.HV, p.V), dtype=torch.bfloat16, device=device)
    if poison_o:
        o.fill_(float("nan"))
    d["o"] = o
    if p.want_final:
        if p.in_place and d["h0"] is not None:
            d["h_final"] = d["h0"]
        else:
            d["h_final"] = torch.full((p.pool_size, p.HV, p.V, p.D), float("nan"), dtype=torch.float32,
                                      device=device)
    else:
        d["h_final"] = None
    return d


def run_gpu(p: W.Problem, d, schedule="auto", dev_error=None, stream=None):
    import linear_attention_prefill_chunkwise_gb300 as lap
    return lap.la_prefill_fwd(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], state_indices=d["idx"],
                              cu_seqlens=d["cu"], o=d["o"], h_final=d["h_final"],
                              seq_len=None if p.cu_seqlens is not None else p.T, schedule=schedule,
                              dev_error=dev_error, stream=stream)


def oracle_full(p: W.Problem, nthreads=0):
    """The oracle over the whole problem: (o [tokens, HV, V] f64 with NaN at unwritten rows,
    h_final [P, HV, V, D] f64 with h0 (or NaN) in unselected slots)."""
    h0 = None if p.h0 is None else p.h0.astype(np.float64)
    hf_init = None
    if p.want_final:
        hf_init = h0.copy() if (p.in_place and h0 is not None) else np.full((p.pool_size, p.HV, p.V, p.D), np.nan)
    return oracle.tokenwise(p.q(), p.k(), p.v(), p.slopes, p.scale, h0=h0, state_indices=p.state_indices,
                            cu_seqlens=p.cu_seqlens, T=None if p.cu_seqlens is not None else p.T,
                            h_final=hf_init, want_state=p.want_final, nthreads=nthreads)


def unit_bounds(p: W.Problem, n):
    if p.cu_seqlens is not None:
        return int(p.cu_seqlens[n]), int(p.cu_seqlens[n + 1])
    return n * p.T, (n + 1) * p.T


def oracle_unit(p: W.Problem, n, hv):
    """Oracle for one (sequence, value head): (o [L, V], h_final [V, D]) in f64, or None if padded."""
    a, b = unit_bounds(p, n)
    G = p.HV // p.H
    hq = hv // G
    slot = n if p.state_indices is None else int(p.state_indices[n])
    if slot < 0:
        return None
    h0 = None if p.h0 is None else p.h0[slot:slot + 1, hv:hv + 1].astype(np.float64)
    L = b - a
    if L == 0:
        hf = np.zeros((p.V, p.D)) if h0 is None else h0[0, 0].copy()
        return np.zeros((0, p.V)), hf
    o, hf = oracle.tokenwise(W.bf16_to_f32(p.q_bits[a:b, hq:hq + 1]), W.bf16_to_f32(p.k_bits[a:b, hq:hq + 1]),
                             W.bf16_to_f32(p.v_bits[a:b, hv:hv + 1]), p.slopes[hv:hv + 1], p.scale, h0=h0, T=L)
    return o[:, 0], hf[0, 0]


def compare_full(p, d, label):
    """Whole-problem comparison with the oracle: written rows within the output bounds, padded
    rows still poisoned, selected state slots within the state bound, the others untouched."""
    import torch
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_full(p)
    o_gpu = bf16_tensor_to_f32(d["o"])
    written = ~np.isnan(o_ref[:, 0, 0])
    # rows the oracle leaves unwritten (padded sequences) must stay poisoned
    assert np.all(np.isnan(o_gpu[~written])), f"{label}: padded rows were written"
    if written.any():
        check_output(o_gpu[written], o_ref[written], label)
    if d["h_final"] is not None:
        h_gpu = d["h_final"].cpu().numpy()
        sel = ~np.isnan(h_ref[:, 0, 0, 0])
        if p.in_place and p.h0 is not None:
            # unselected slots keep their initial value bit for bit
            unsel = np.ones(p.pool_size, bool)
            unsel[[s for s in (p.state_indices if p.state_indices is not None else range(p.N)) if s >= 0]] = False
            assert np.array_equal(h_gpu[unsel], p.h0[unsel]), f"{label}: unselected pool slots changed"
            sel = ~unsel
        else:
            assert np.all(np.isnan(h_gpu[~sel])), f"{label}: unselected h_final slots were written"
        if sel.any():
            check_state(h_gpu[sel], h_ref[sel], label)


def compare_sampled(p, d, units, label):
    """Comparison with the oracle on the given (sequence, value head) units, each computed alone."""
    import torch
    torch.cuda.synchronize()
    o_gpu_t = d["o"]
    hf = d["h_final"]
    for (n, hv) in units:
        res = oracle_unit(p, n, hv)
        if res is None:
            continue
        o_ref, h_ref = res
        a, b = unit_bounds(p, n)
        o_gpu = o_gpu_t[a:b, hv].float().cpu().numpy()
        check_output(o_gpu, o_ref, f"{label} unit (n={n}, hv={hv})")
        if hf is not None:
            slot = n if p.state_indices is None else int(p.state_indices[n])
            check_state(hf[slot, hv].cpu().numpy(), h_ref, f"{label} state (n={n}, hv={hv})")


def unit_metrics(o_gpu, o_ref):
    """(rel RMS, max abs error, max |o_ref|) of one unit's output rows."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    diff = o_gpu - o_ref
    den = np.sqrt(np.sum(o_ref ** 2))
    return (float(np.sqrt(np.sum(diff ** 2)) / max(den, 1e-300)), float(np.max(np.abs(diff))),
            float(np.max(np.abs(o_ref))))


def compare_every_unit(p, d, label, nthreads=0):
    """The whole problem against the oracle, unit by unit: every (sequence, value head) unit's
    output rows and final state must meet the output and state bounds on their own, rows of
    padded sequences must stay poisoned and state slots no sequence selects must keep their
    initial value bit for bit (or stay poisoned).  A failure lists every failing (n, hv) unit
    with its figures.  Returns the worst unit's (output rel RMS, state rel RMS)."""
    import torch
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_full(p, nthreads=nthreads)
    o_gpu = d["o"].float().cpu().numpy()
    hf = None if d["h_final"] is None else d["h_final"].cpu().numpy()
    slots = list(p.state_indices) if p.state_indices is not None else list(range(p.N))
    bad, worst_o, worst_s = [], 0.0, 0.0
    for n in range(p.N):
        a, b = unit_bounds(p, n)
        slot = int(slots[n])
        if slot < 0:
            if b > a and not np.all(np.isnan(o_gpu[a:b])):
                bad.append(f"(n={n}) padded sequence has written rows")
            continue
        for hv in range(p.HV):
            if b > a:
                og = o_gpu[a:b, hv]
                if not np.all(np.isfinite(og)):
                    bad.append(f"(n={n}, hv={hv}) non-finite output")
                    continue
                r, ma, mref = unit_metrics(og, o_ref[a:b, hv])
                worst_o = max(worst_o, r)
                if r > O_REL_RMS or ma > O_MAX_ABS_FRAC * mref + 1e-30:
                    bad.append(f"(n={n}, hv={hv}) output rel RMS {r:.3e}, max abs {ma:.3e} vs max |o| {mref:.3e}")
            if hf is not None:
                hs = hf[slot, hv]
                if not np.all(np.isfinite(hs)):
                    bad.append(f"(n={n}, hv={hv}) non-finite state")
                    continue
                rs = rel_rms(hs, h_ref[slot, hv])
                worst_s = max(worst_s, rs)
                if rs > STATE_REL_RMS:
                    bad.append(f"(n={n}, hv={hv}) state rel RMS {rs:.3e}")
    if hf is not None:
        live = [int(s) for s in slots if s >= 0]
        unsel = np.ones(hf.shape[0], bool)
        unsel[live] = False
        if p.in_place and p.h0 is not None:
            if not np.array_equal(hf[unsel].view(np.uint32), p.h0[unsel].view(np.uint32)):
                bad.append("state slots no sequence selects were changed")
        elif not np.all(np.isnan(hf[unsel])):
            bad.append("state slots no sequence selects were written")
    assert not bad, f"{label}: {len(bad)} failing units:\n  " + "\n  ".join(bad[:40])
    return worst_o, worst_s
