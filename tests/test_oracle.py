"""Pins for the FP64 oracle (CPU only).

The oracle is only trusted once it agrees with things other than itself:
hand-worked examples, the pages' closed form brute-forced on tiny inputs, the
special cases lambda = 1 (plain causal linear attention, a masked matmul) and
lambda = 0 (o_t = scale (q_t . k_t) v_t), and invariants (chunked == tokenwise,
packed == each sequence alone, pool isolation, GVA == repeated q/k heads,
continuation).  Each pin is chosen so that a plausible slip in the oracle
(update after read, exponent offset, transposed state, wrong head mapping,
dropped scale) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.sqrt(np.sum((a - b) ** 2)) / max(np.sqrt(np.sum(b ** 2)), 1e-300))


def rand_problem(seed, lengths, H, HV, D=16, V=24, with_h0=True, slopes=None, scale=0.37):
    """Small generic problem (any D, V) drawn here for oracle-only checks."""
    rng = np.random.default_rng(seed)
    tokens = int(np.sum(lengths))
    q = rng.standard_normal((tokens, H, D)).astype(np.float32)
    k = rng.standard_normal((tokens, H, D)).astype(np.float32) * np.float32(0.3)
    v = rng.standard_normal((tokens, HV, V)).astype(np.float32)
    if slopes is None:
        slopes = rng.uniform(0.01, 0.7, HV).astype(np.float32)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    h0 = rng.standard_normal((len(lengths), HV, V, D)) * 0.5 if with_h0 else None
    return q, k, v, np.asarray(slopes, dtype=np.float32), scale, h0, cu


# ---- hand-worked examples -------------------------------------------------------

@pytest.mark.parametrize("fn", ["tokenwise", "chunked"])
def test_golden_worked_examples(fn):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        q = np.array(c["q"], dtype=np.float32)[:, None, :]
        k = np.array(c["k"], dtype=np.float32)[:, None, :]
        v = np.array(c["v"], dtype=np.float32)[:, None, :]
        h0 = np.array(c["h0"], dtype=np.float64)[None, None]
        T = q.shape[0]
        kw = dict(chunk=2) if fn == "chunked" else {}
        o, hf = getattr(oracle, fn)(q, k, v, np.array([c["slope"]], np.float32), c["scale"],
                                    h0=h0, T=T, **kw)
        exp_o = np.array(c["o"])
        exp_h = np.array(c["h_final"])
        tol = c["tol"]
        assert np.allclose(o[:, 0, :], exp_o, rtol=tol, atol=tol), (c["name"], o[:, 0, :], exp_o)
        assert np.allclose(hf[0, 0], exp_h, rtol=tol, atol=tol), (c["name"], hf[0, 0], exp_h)


# ---- the pages' closed form, brute force -------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_closed_form_matches_tokenwise(seed):
    lengths = [1, 7, 32, 19]
    H, HV = 2, 4  # GVA, G = 2
    q, k, v, slopes, scale, h0, cu = rand_problem(seed, lengths, H, HV)
    o, hf = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu)
    G = HV // H
    for n, L in enumerate(lengths):
        a, b = cu[n], cu[n + 1]
        for hv in range(HV):
            hq = hv // G
            o_cf, h_cf = oracle.closed_form(q[a:b, hq], k[a:b, hq], v[a:b, hv], slopes[hv], scale,
                                            h0[n, hv])
            assert rel(o[a:b, hv], o_cf) < 1e-12
            assert rel(hf[n, hv], h_cf) < 1e-12


def test_closed_form_catches_plausible_slips():
    """The closed form separates the correct recurrence from its near misses."""
    q, k, v, slopes, scale, h0, cu = rand_problem(5, [12], 1, 1, D=16, V=16)
    lam = float(np.exp(-np.float64(slopes[0])))
    o_cf, _ = oracle.closed_form(q[:, 0], k[:, 0], v[:, 0], slopes[0], scale, h0[0, 0])
    q64, k64, v64 = (x[:, 0].astype(np.float64) for x in (q, k, v))
    # read-before-update (o_t would miss k_t v_t and use lambda^t on h0)
    S = h0[0, 0].copy()
    slip = []
    for t in range(12):
        slip.append(scale * S @ q64[t])
        S = lam * S + np.outer(v64[t], k64[t])
    assert rel(np.array(slip), o_cf) > 1e-3
    # transposed initial state
    o_t, _ = oracle.closed_form(q[:, 0], k[:, 0], v[:, 0], slopes[0], scale, h0[0, 0].T.copy())
    assert rel(o_t, o_cf) > 1e-3
    # exponent offset 0 on h0 instead of 1
    o_e, _ = oracle.closed_form(q[:, 0], k[:, 0], v[:, 0], slopes[0], scale, h0[0, 0] / lam)
    assert rel(o_e, o_cf) > 1e-3


# ---- special cases -----------------------------------------------------------------

def test_lambda_one_is_causal_linear_attention():
    lengths = [40, 9]
    q, k, v, _, scale, h0, cu = rand_problem(11, lengths, 2, 2, slopes=np.zeros(2))
    o, hf = oracle.tokenwise(q, k, v, np.zeros(2, np.float32), scale, h0=h0, cu_seqlens=cu)
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        for h in range(2):
            Q, K, Vv = (x[a:b, h].astype(np.float64) for x in (q, k, v))
            ref = scale * (np.tril(Q @ K.T) @ Vv + Q @ h0[n, h].T)
            assert rel(o[a:b, h], ref) < 1e-12
            assert rel(hf[n, h], h0[n, h] + Vv.T @ K) < 1e-12


def test_lambda_zero_keeps_only_current_token():
    lengths = [5, 1, 70]
    q, k, v, _, scale, h0, cu = rand_problem(12, lengths, 1, 2)
    sl = np.full(2, 800.0, np.float32)  # exp(-800) == 0 in double
    for fn in (oracle.tokenwise, oracle.chunked):
        o, hf = fn(q, k, v, sl, scale, h0=h0, cu_seqlens=cu)
        for n in range(len(lengths)):
            a, b = cu[n], cu[n + 1]
            for hv in range(2):
                Q = q[a:b, 0].astype(np.float64)
                K = k[a:b, 0].astype(np.float64)
                Vv = v[a:b, hv].astype(np.float64)
                ref = scale * np.sum(Q * K, axis=1)[:, None] * Vv
                assert rel(o[a:b, hv], ref) < 1e-12
                assert rel(hf[n, hv], np.outer(Vv[-1], K[-1])) < 1e-12


# ---- invariants -------------------------------------------------------------------

@pytest.mark.parametrize("chunk", [64, 16, 5])
def test_chunked_equals_tokenwise(chunk):
    lengths = [1, 63, 64, 65, 130, 200, 0, 3]
    q, k, v, slopes, scale, h0, cu = rand_problem(21, lengths, 2, 4, D=32, V=16)
    o1, h1 = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu)
    o2, h2 = oracle.chunked(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu, chunk=chunk)
    assert rel(o2, o1) < 1e-10
    assert rel(h2, h1) < 1e-10


def test_empty_sequence_returns_initial_state():
    lengths = [0, 4]
    q, k, v, slopes, scale, h0, cu = rand_problem(22, lengths, 1, 1)
    for fn in (oracle.tokenwise, oracle.chunked):
        o, hf = fn(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu)
        assert np.array_equal(hf[0], h0[0])
        assert not np.isnan(o).any()


def test_varlen_equals_each_sequence_alone():
    lengths = [17, 64, 3, 100]
    q, k, v, slopes, scale, h0, cu = rand_problem(31, lengths, 2, 2, D=32, V=32)
    o, hf = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu)
    for n, L in enumerate(lengths):
        a, b = cu[n], cu[n + 1]
        o1, h1 = oracle.tokenwise(q[a:b], k[a:b], v[a:b], slopes, scale, h0=h0[n:n + 1], T=L)
        assert np.array_equal(o[a:b], o1)
        assert np.array_equal(hf[n], h1[0])


def test_fixed_equals_packed_uniform():
    lengths = [48, 48, 48]
    q, k, v, slopes, scale, h0, cu = rand_problem(32, lengths, 1, 3)
    o1, h1 = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu)
    o2, h2 = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, T=48)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


def test_pool_gather_scatter_isolation_and_padding():
    lengths = [10, 30, 5, 64]
    H = HV = 2
    q, k, v, slopes, scale, _, cu = rand_problem(41, lengths, H, HV)
    rng = np.random.default_rng(7)
    P = 9
    pool = rng.standard_normal((P, HV, 24, 16))
    idx = np.array([6, -1, 2, 4], dtype=np.int32)
    o_init = np.full((q.shape[0], HV, 24), 123.0)
    hf_init = pool.copy()
    o, hf = oracle.tokenwise(q, k, v, slopes, scale, h0=pool, state_indices=idx, cu_seqlens=cu,
                             o=o_init.copy(), h_final=hf_init.copy())
    untouched = [s for s in range(P) if s not in (6, 2, 4)]
    assert np.array_equal(hf[untouched], pool[untouched])
    a, b = cu[1], cu[2]
    assert np.all(o[a:b] == 123.0)  # padded sequence: output rows untouched
    # selected slots equal running each sequence alone from its slot
    for n, s in enumerate(idx):
        if s < 0:
            continue
        a, b = cu[n], cu[n + 1]
        o1, h1 = oracle.tokenwise(q[a:b], k[a:b], v[a:b], slopes, scale, h0=pool[s:s + 1],
                                  T=int(lengths[n]))
        assert np.array_equal(o[a:b], o1)
        assert np.array_equal(hf[s], h1[0])


def test_out_of_range_index_rejected():
    q, k, v, slopes, scale, _, cu = rand_problem(42, [4], 1, 1)
    pool = np.zeros((2, 1, 24, 16))
    with pytest.raises(ValueError):
        oracle.tokenwise(q, k, v, slopes, scale, h0=pool, state_indices=np.array([2], np.int32),
                         cu_seqlens=cu)


def test_gva_is_contiguous_group_repeat():
    lengths = [33, 70]
    H, HV = 2, 6  # G = 3
    q, k, v, slopes, scale, h0, cu = rand_problem(51, lengths, H, HV)
    o, hf = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu)
    qr, kr = np.repeat(q, 3, axis=1), np.repeat(k, 3, axis=1)
    o2, h2 = oracle.tokenwise(qr, kr, v, slopes, scale, h0=h0, cu_seqlens=cu)
    assert np.array_equal(o, o2) and np.array_equal(hf, h2)
    # the other plausible mapping (hv % H) gives a different answer on these inputs
    qm, km = np.tile(q, (1, 3, 1)), np.tile(k, (1, 3, 1))
    o3, _ = oracle.tokenwise(qm, km, v, slopes, scale, h0=h0, cu_seqlens=cu)
    assert rel(o3, o) > 1e-2


def test_continuation():
    L1, L2 = 37, 91
    q, k, v, slopes, scale, h0, _ = rand_problem(61, [L1 + L2], 1, 2)
    o, hf = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, T=L1 + L2)
    oa, ha = oracle.tokenwise(q[:L1], k[:L1], v[:L1], slopes, scale, h0=h0, T=L1)
    ob, hb = oracle.tokenwise(q[L1:], k[L1:], v[L1:], slopes, scale, h0=ha, T=L2)
    assert rel(np.concatenate([oa, ob]), o) < 1e-12
    assert rel(hb, hf) < 1e-12


def test_segmented_scan_decomposition():
    """The segment-parallel form of the recurrence (page "linear_attention: add a Hopper (sm90) KDA
    prefill path - #1017", How: the segmented affine scan, applied to the scalar decay): each
    segment's local state from a zero start equals the closed form
    sum_j lambda^(L-1-j) v_j k_j^T; chaining H_{i+1} = lambda^{L_i} H_i + Sloc_i gives every
    segment's exact initial state; running each segment from it reproduces the whole
    sequence's outputs and final state."""
    seg = [64 * 3, 64 * 3, 64 + 17]
    total = sum(seg)
    # small slopes keep lambda^L away from 0, so the initial state still matters at every boundary
    q, k, v, slopes, scale, h0, _ = rand_problem(81, [total], 1, 2, slopes=[0.003, 0.02])
    o, hf = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, T=total)
    H = h0[0].copy()  # [HV, V, D]
    outs = []
    a = 0
    for L in seg:
        b = a + L
        _, sloc = oracle.tokenwise(q[a:b], k[a:b], v[a:b], slopes, scale, h0=None, T=L)
        for hv in range(2):
            _, hT = oracle.closed_form(q[a:b, 0], k[a:b, 0], v[a:b, hv], slopes[hv], scale)
            assert rel(sloc[0, hv], hT) < 1e-12
        oi, hi = oracle.tokenwise(q[a:b], k[a:b], v[a:b], slopes, scale, h0=H[None], T=L)
        outs.append(oi)
        lamL = np.exp(-slopes.astype(np.float64) * L)[:, None, None]
        H = lamL * H + sloc[0]
        assert rel(H, hi[0]) < 1e-12
        a = b
    assert rel(np.concatenate(outs), o) < 1e-12
    assert rel(H, hf[0]) < 1e-12
    # the plausible slip of decaying the local state by lambda^(L-1) instead of lambda^L
    lam_wrong = np.exp(-slopes.astype(np.float64) * (seg[0] - 1))[:, None, None]
    _, s0 = oracle.tokenwise(q[:seg[0]], k[:seg[0]], v[:seg[0]], slopes, scale, h0=None, T=seg[0])
    _, h_true = oracle.tokenwise(q[:seg[0]], k[:seg[0]], v[:seg[0]], slopes, scale, h0=h0, T=seg[0])
    assert rel(lam_wrong * h0[0] + s0[0], h_true[0]) > 1e-6


def test_scale_is_linear():
    q, k, v, slopes, _, h0, cu = rand_problem(71, [20], 1, 1)
    o1, h1 = oracle.tokenwise(q, k, v, slopes, 1.0, h0=h0, cu_seqlens=cu)
    o2, h2 = oracle.tokenwise(q, k, v, slopes, 0.25, h0=h0, cu_seqlens=cu)
    assert rel(o2, 0.25 * o1) < 1e-15 and np.array_equal(h1, h2)


# ---- the BF16 output floor on the tiny workload -----------------------------------

def test_bf16_output_floor_tiny_workload():
    """Rounding the exact output to BF16 alone costs ~1e-3 relative RMS; the
    2e-3 acceptance bound must leave room above it."""
    p = W.config(1)
    o, hf = oracle.tokenwise(p.q(), p.k(), p.v(), p.slopes, p.scale, T=p.T)
    ob = W.bf16_to_f32(W.bf16_bits(o.astype(np.float32))).astype(np.float64)
    floor = rel(ob, o)
    assert 5e-4 < floor < 2e-3, floor


# ---- backward: the oracle's gradients against finite differences of its forward pass ----
#
# L = sum_t o_t . dout_t + sum over selected slots of h_final . dh_final is linear in every
# single element of q, k, v and h0 (o_t is a sum of products with one factor from each of
# q, k, v, or of q and h0), so a central difference with any step is exact up to rounding.

def _fd_loss(q, k, v, sl, scale, h0, idx, cu, dout, dhf):
    o, hf = oracle.tokenwise(q, k, v, sl, scale, h0=h0, state_indices=idx, cu_seqlens=cu,
                             h_final=np.zeros_like(h0))
    sel = [int(s) for s in idx if s >= 0]
    live_rows = ~np.isnan(o[:, 0, 0])
    return float(np.sum(o[live_rows] * dout[live_rows])) + float(np.sum(hf[sel] * dhf[sel]))


def test_backward_matches_finite_differences_of_the_forward():
    rng = np.random.default_rng(71)
    lengths = [3, 0, 4, 2]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    tok, H, HV, D, V, P = int(cu[-1]), 1, 2, 3, 2, 6
    q = rng.standard_normal((tok, H, D)).astype(np.float32)
    k = rng.standard_normal((tok, H, D)).astype(np.float32)
    v = rng.standard_normal((tok, HV, V)).astype(np.float32)
    dout = rng.standard_normal((tok, HV, V)).astype(np.float32)
    sl = np.array([0.3, 1.1], np.float32)
    h0 = rng.standard_normal((P, HV, V, D))
    dhf = rng.standard_normal((P, HV, V, D))
    idx = np.array([4, 1, -1, 0], np.int32)  # sequence 2 padded
    scale = 0.75
    dq, dk, dv, dh0 = oracle.backward(q, k, v, sl, scale, dout, h0=h0, dh_final=dhf, state_indices=idx,
                                      cu_seqlens=cu)
    base = (q, k, v, sl, scale, h0, idx, cu, dout, dhf)
    eps = 0.5  # exact in float32; L is linear in each element

    def fd(pos, index):
        # the steps actually taken (x +- eps rounds in float32): L is linear in the element, so
        # the difference quotient over the exact step is the derivative
        args = list(base)
        x = args[pos].copy()
        x0 = float(x[index])
        x[index] = x0 + eps
        up = float(x[index])
        args[pos] = x
        lp = _fd_loss(*args)
        x[index] = x0 - eps
        dn = float(x[index])
        lm = _fd_loss(*args)
        return (lp - lm) / (up - dn)

    live = np.ones(tok, bool)
    live[cu[2]:cu[3]] = False
    for name, pos, grad in (("q", 0, dq), ("k", 1, dk), ("v", 2, dv)):
        for index in np.ndindex(*grad.shape):
            if not live[index[0]]:
                assert np.isnan(grad[index]), f"d{name} written for a padded row"
                continue
            ref = fd(pos, index)
            assert abs(grad[index] - ref) <= 1e-9 * (1 + abs(ref)), (name, index, grad[index], ref)
    for slot in range(P):
        for index in np.ndindex(HV, V, D):
            if slot not in (4, 1, 0):
                assert np.isnan(dh0[(slot,) + index]), "dh0 written for an unselected slot"
                continue
            ref = fd(5, (slot,) + index)
            assert abs(dh0[(slot,) + index] - ref) <= 1e-9 * (1 + abs(ref)), ("h0", slot, index)


def test_backward_lambda_one_matches_masked_linear_attention_gradients():
    # slope 0: o = scale (tril(Q K^T) V + Q h0^T) and h_final = h0 + V^T K, whose gradients are
    # plain masked matrix products
    rng = np.random.default_rng(72)
    T, D, V = 9, 5, 4
    q = rng.standard_normal((T, 1, D)).astype(np.float32)
    k = rng.standard_normal((T, 1, D)).astype(np.float32)
    v = rng.standard_normal((T, 1, V)).astype(np.float32)
    dout = rng.standard_normal((T, 1, V)).astype(np.float32)
    h0 = rng.standard_normal((1, 1, V, D))
    dhf = rng.standard_normal((1, 1, V, D))
    scale = 0.6
    dq, dk, dv, dh0 = oracle.backward(q, k, v, np.zeros(1, np.float32), scale, dout, h0=h0, dh_final=dhf, T=T)
    Q, K, Vm, dO = (x[:, 0].astype(np.float64) for x in (q, k, v, dout))
    Mk = np.tril(np.ones((T, T)))
    H0, dHf = h0[0, 0], dhf[0, 0]
    dq_ref = scale * (Mk * (dO @ Vm.T)) @ K + scale * dO @ H0
    dk_ref = scale * (Mk * (dO @ Vm.T)).T @ Q + Vm @ dHf
    dv_ref = scale * (Mk * (Q @ K.T)).T @ dO + K @ dHf.T
    dh0_ref = scale * dO.T @ Q + dHf
    assert np.allclose(dq[:, 0], dq_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(dk[:, 0], dk_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(dv[:, 0], dv_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(dh0[0, 0], dh0_ref, rtol=1e-12, atol=1e-12)


# ---- the block decomposition the D = 256 prefill relies on ---------------------------

def test_key_and_value_halves_decompose_the_recurrence():
    """S[v][k] += v_t[v] k_t[k] updates every state element on its own, and q . k splits over
    any partition of the key dimension, so the recurrence at head dimension D equals the sum over
    key halves b of the recurrences on (q[b half], k[b half]) from the state columns of that half,
    with the final state assembled block by block, for each half of the value dimension alike.
    A slip that mixes the halves (a cross term, one scale or decay applied twice) breaks it."""
    lengths = [9, 0, 14]
    q, k, v, slopes, scale, h0, cu = rand_problem(41, lengths, 2, 4, D=12, V=10)
    o, hf = oracle.tokenwise(q, k, v, slopes, scale, h0=h0, cu_seqlens=cu)
    half = 6
    o_sum = np.zeros_like(o)
    hf_blocks = np.zeros_like(hf)
    for b in range(2):
        ks = slice(b * half, (b + 1) * half)
        for a, vs in enumerate((slice(0, 4), slice(4, 10))):  # uneven value halves: rows are independent
            ob, hb = oracle.tokenwise(np.ascontiguousarray(q[:, :, ks]), np.ascontiguousarray(k[:, :, ks]),
                                      np.ascontiguousarray(v[:, :, vs]), slopes, scale,
                                      h0=np.ascontiguousarray(h0[:, :, vs, ks]), cu_seqlens=cu)
            o_sum[:, :, vs] += ob
            hf_blocks[:, :, vs, ks] = hb
    assert rel(o_sum, o) < 1e-12
    assert rel(hf_blocks, hf) < 1e-12
    # one key half alone is far from the whole (the test would catch a dropped half)
    o_half, _ = oracle.tokenwise(np.ascontiguousarray(q[:, :, :half]), np.ascontiguousarray(k[:, :, :half]), v,
                                 slopes, scale, h0=np.ascontiguousarray(h0[:, :, :, :half]), cu_seqlens=cu)
    assert rel(o_half, o) > 0.1
