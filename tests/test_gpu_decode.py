"""GPU parity of the speculative-decoding ops (include/la_decode.h) against the FP64 oracle.

Page "[LA] Lightning Attention MTP decode + KVBuffer parallel verify / commit", Description
and Tests: MTP decode advances each request's pooled state over its T draft tokens; verify
produces every draft token's output from the pooled state without changing it (optionally
copying k, v into a pooled KV buffer); commit advances the pooled state by the per-request
accepted prefix read from that buffer (L = 0 is a no-op, padded requests are skipped).

The oracle is the tokenwise FP64 recurrence on the same BF16 inputs: a request of T tokens
is a packed sequence of length T, and committing L tokens is the same recurrence over the
first L tokens.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import workloads as W
from harness import check_output, check_state, to_torch_bf16

pytestmark = pytest.mark.gpu


def make_case(seed, B, T, H, HV, P, n_pad=0, scale=None, slopes=None, D=W.D):
    rng = np.random.default_rng(seed)
    q, k, v = W.make_qkv(rng, B * T, H, HV, d=D, v_dim=D)
    pool = W.make_states(rng, P, HV, d=D, v_dim=D)
    idx = rng.permutation(P)[:B].astype(np.int32)
    if n_pad:
        idx[rng.choice(B, n_pad, replace=False)] = -1
    sl = W.slopes_for(HV) if slopes is None else np.asarray(slopes, dtype=np.float32)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    return dict(q=q, k=k, v=v, pool=pool, idx=idx, slopes=sl, scale=sc, B=B, T=T, H=H, HV=HV, P=P, D=D)


def oracle_run(c, lengths=None):
    """Outputs and final pool of the tokenwise oracle, each request of ``lengths`` tokens
    (default T) taken from the start of its T-token block."""
    B, T = c["B"], c["T"]
    L = np.full(B, T, dtype=np.int64) if lengths is None else np.asarray(lengths, dtype=np.int64)
    rows = np.concatenate([np.arange(b * T, b * T + L[b]) for b in range(B)]).astype(np.int64)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(L)
    q, k, v = (W.bf16_to_f32(c[n][rows]) for n in ("q", "k", "v"))
    o, h = oracle.tokenwise(q, k, v, c["slopes"], c["scale"], h0=c["pool"], state_indices=c["idx"],
                            cu_seqlens=cu, h_final=c["pool"].astype(np.float64).copy())
    return o, h, rows


def upload(c, device="cuda"):
    import torch
    d = {n: to_torch_bf16(c[n], device) for n in ("q", "k", "v")}
    d["slopes"] = torch.from_numpy(c["slopes"]).to(device)
    d["pool"] = torch.from_numpy(c["pool"]).to(device)
    d["idx"] = torch.from_numpy(c["idx"]).to(device)
    return d


def live_rows(c):
    return np.concatenate([np.arange(b * c["T"], (b + 1) * c["T"]) for b in range(c["B"]) if c["idx"][b] >= 0])


VERIFY_TC_MAX_T = 8  # la_verify's tensor-core closed form serves requests of at most 8 tokens

CASES = {
    "verify_shape_B128_T8_H64_pool256_pad16": dict(seed=5001, B=128, T=8, H=64, HV=64, P=256, n_pad=16),
    "T1": dict(seed=5002, B=5, T=1, H=4, HV=4, P=8, n_pad=1),
    "T3_gva": dict(seed=5003, B=6, T=3, H=2, HV=8, P=9, n_pad=2),
    "T17_tiles": dict(seed=5004, B=3, T=17, H=4, HV=4, P=4),
    "T40_slow_decay_lambda1": dict(seed=5005, B=2, T=40, H=2, HV=2, P=2, slopes=[0.0, 0.0]),
    "T5_gva_lambda_edges": dict(seed=5006, B=7, T=5, H=2, HV=6, P=11, n_pad=2,
                                slopes=[0.0, 1e-4, 0.7, 5.0, 40.0, 200.0]),
    "T8_gva_pool": dict(seed=5007, B=40, T=8, H=4, HV=16, P=64, n_pad=5),
    "T2_single_request": dict(seed=5008, B=1, T=2, H=1, HV=1, P=1),
    # D = V = 64: one CTA per (request, value head), and verify always tokenwise
    "D64_T1": dict(seed=5101, B=5, T=1, H=4, HV=4, P=8, n_pad=1, D=64),
    "D64_T5_gva_lambda_edges": dict(seed=5102, B=7, T=5, H=2, HV=6, P=11, n_pad=2,
                                    slopes=[0.0, 1e-4, 0.7, 5.0, 40.0, 200.0], D=64),
    "D64_T8_gva_pool": dict(seed=5103, B=40, T=8, H=4, HV=16, P=64, n_pad=5, D=64),
    "D64_T17_tiles": dict(seed=5104, B=3, T=17, H=4, HV=4, P=4, D=64),
    # D = V = 256: eight CTAs of 32 rows per (request, value head), row groups of 16 lanes
    "D256_T1": dict(seed=5201, B=5, T=1, H=2, HV=2, P=8, n_pad=1, D=256),
    "D256_T5_gva_lambda_edges": dict(seed=5202, B=7, T=5, H=2, HV=6, P=11, n_pad=2,
                                     slopes=[0.0, 1e-4, 0.7, 5.0, 40.0, 200.0], D=256),
    "D256_T8_gva_pool": dict(seed=5203, B=24, T=8, H=2, HV=8, P=32, n_pad=3, D=256),
    "D256_T17_tiles": dict(seed=5204, B=3, T=17, H=2, HV=2, P=4, D=256),
}


def check_decode_mtp(c, name):
    """la_decode_mtp on case c against the oracle: outputs, advanced slots, untouched rest."""
    import torch
    import linear_attention_prefill_chunkwise_gb300 as lap
    d = upload(c)
    o = torch.full((c["B"] * c["T"], c["HV"], c["D"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lap.la_decode_mtp(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], c["T"], state_indices=d["idx"],
                      o=o, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, h_ref, _ = oracle_run(c)
    rows = live_rows(c)
    check_output(o.float().cpu().numpy()[rows], o_ref[rows], f"{name} o")
    pool = d["pool"].cpu().numpy()
    sel = c["idx"][c["idx"] >= 0]
    check_state(pool[sel], h_ref[sel], f"{name} state")
    # padded requests: their o rows are not written; unselected slots are bit-identical
    pad_rows = np.setdiff1d(np.arange(c["B"] * c["T"]), rows)
    assert np.all(np.isnan(o.float().cpu().numpy()[pad_rows]))
    untouched = np.setdiff1d(np.arange(c["P"]), sel)
    assert np.array_equal(pool[untouched], c["pool"][untouched])


def check_verify_then_commit(c, name, seed):
    """la_verify then la_commit of a random accepted prefix (0 and T included) on case c: the
    outputs against the oracle and decode, the KV buffer, the committed slots against the
    oracle, bitwise where nothing or everything is accepted, and the untouched rest."""
    import torch
    import linear_attention_prefill_chunkwise_gb300 as lap
    B, T, H, HV, P = c["B"], c["T"], c["H"], c["HV"], c["P"]
    d = upload(c)
    # decode on a copy of the pool: the reference for verify's outputs and a full commit's state
    dec_pool = d["pool"].clone()
    o_dec = lap.la_decode_mtp(d["q"], d["k"], d["v"], d["slopes"], c["scale"], dec_pool, T, state_indices=d["idx"])
    kbuf = torch.zeros((P, T, H, c["D"]), dtype=torch.bfloat16, device="cuda")
    vbuf = torch.zeros((P, T, HV, c["D"]), dtype=torch.bfloat16, device="cuda")
    o = lap.la_verify(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], T, state_indices=d["idx"],
                      kbuf=kbuf, vbuf=vbuf)
    torch.cuda.synchronize()
    rows = live_rows(c)
    # verify: pool untouched, KV buffer = the draft k, v at the slot; the outputs match the oracle
    # (below) and, where verify runs the same tokenwise recurrence as decode (T > 8, or D = 64),
    # are bitwise decode's; for T <= 8 at D = 128 verify evaluates the closed form with the state
    # as a TF32 operand
    if T > VERIFY_TC_MAX_T or c["D"] != 128:
        assert torch.equal(o[rows], o_dec[rows])
    else:
        check_output(o.float().cpu().numpy()[rows], o_dec.float().cpu().numpy()[rows].astype(np.float64),
                     f"{name} verify vs decode")
    assert np.array_equal(d["pool"].cpu().numpy(), c["pool"])
    kb, vb = kbuf.cpu().view(torch.int16).numpy(), vbuf.cpu().view(torch.int16).numpy()
    for b in range(B):
        s = c["idx"][b]
        if s < 0:
            continue
        assert np.array_equal(kb[s], c["k"][b * T:(b + 1) * T].view(np.int16))
        assert np.array_equal(vb[s], c["v"][b * T:(b + 1) * T].view(np.int16))
    o_ref, _, _ = oracle_run(c)
    check_output(o.float().cpu().numpy()[rows], o_ref[rows], f"{name} verify o")
    # commit a random accepted prefix per request (0 and T included)
    rng = np.random.default_rng(seed)
    acc = rng.integers(0, T + 1, B).astype(np.int32)
    acc[0] = T
    if B > 1:
        acc[1] = 0
    acc_d = torch.from_numpy(acc).cuda()
    lap.la_commit(d["pool"], kbuf, vbuf, acc_d, d["slopes"], state_indices=d["idx"])
    torch.cuda.synchronize()
    pool = d["pool"].cpu().numpy()
    _, h_ref, _ = oracle_run(c, lengths=acc)
    sel = c["idx"][c["idx"] >= 0]
    check_state(pool[sel], h_ref[sel], f"{name} commit state")
    dec = dec_pool.cpu().numpy()
    for b in range(B):
        s = c["idx"][b]
        if s < 0:
            continue
        if acc[b] == 0:  # nothing accepted: the slot is bit-identical
            assert np.array_equal(pool[s], c["pool"][s])
        if acc[b] == T:  # everything accepted: bitwise the state decode leaves
            assert np.array_equal(pool[s], dec[s])
    untouched = np.setdiff1d(np.arange(P), sel)
    assert np.array_equal(pool[untouched], c["pool"][untouched])


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_mtp_matches_oracle(name):
    check_decode_mtp(make_case(**CASES[name]), name)


@pytest.mark.parametrize("name", sorted(CASES))
def test_verify_then_commit(name):
    c = make_case(**CASES[name])
    check_verify_then_commit(c, name, c["B"] * 131 + c["T"])


def test_decode_without_indices_and_bad_index_flag():
    import torch
    import linear_attention_prefill_chunkwise_gb300 as lap
    c = make_case(seed=5010, B=3, T=4, H=2, HV=2, P=3)
    c["idx"] = np.arange(3, dtype=np.int32)
    d = upload(c)
    o = lap.la_decode_mtp(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], c["T"])  # slot = request
    o_ref, h_ref, _ = oracle_run(c)
    check_output(o.float().cpu().numpy(), o_ref, "no indices o")
    check_state(d["pool"].cpu().numpy(), h_ref, "no indices state")
    # an index past the pool is skipped and flagged on the device, never read
    bad = torch.tensor([0, 7, 2], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = d["pool"].clone()
    lap.la_decode_mtp(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], c["T"], state_indices=bad,
                      dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lap.DEV_ERR_BAD_INDEX
    assert torch.equal(d["pool"][1], before[1])


@pytest.mark.parametrize("T", [3, 8])
def test_verify_nonfinite_request_does_not_reach_its_neighbours(T):
    """A request whose draft q, k, v hold Inf and NaN leaves every other request's outputs
    bitwise as they are without it: the tensor-core path reads the next request's token rows
    past a short request's end, which must stay out of its outputs."""
    import torch
    import linear_attention_prefill_chunkwise_gb300 as lap
    c = make_case(seed=5020 + T, B=6, T=T, H=2, HV=4, P=8, n_pad=1)
    d = upload(c)
    o_clean = lap.la_verify(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], T, state_indices=d["idx"])
    bad_b = 2 if c["idx"][2] >= 0 else 3
    for n in ("q", "k", "v"):
        x = d[n].clone()
        x[bad_b * T] = float("inf")
        x[bad_b * T + T - 1, 0, :7] = float("nan")
        d[n] = x
    o_bad = lap.la_verify(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], T, state_indices=d["idx"])
    torch.cuda.synchronize()
    rows = np.array([r for r in live_rows(c) if r // T != bad_b])
    assert torch.equal(o_bad[rows].view(torch.int16), o_clean[rows].view(torch.int16))
    assert bool(torch.isfinite(o_clean[rows].float()).all())


def test_verify_without_kv_buffer_and_bad_index_flag():
    import torch
    import linear_attention_prefill_chunkwise_gb300 as lap
    c = make_case(seed=5030, B=4, T=6, H=2, HV=4, P=5)
    d = upload(c)
    o = lap.la_verify(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], c["T"], state_indices=d["idx"])
    o_ref, _, _ = oracle_run(c)
    rows = live_rows(c)
    check_output(o.float().cpu().numpy()[rows], o_ref[rows], "verify without KV buffer o")
    bad = torch.tensor([c["idx"][0], 9, c["idx"][2], c["idx"][3]], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o2 = torch.full_like(o, float("nan"))
    lap.la_verify(d["q"], d["k"], d["v"], d["slopes"], c["scale"], d["pool"], c["T"], state_indices=bad, o=o2,
                  dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lap.DEV_ERR_BAD_INDEX
    T = c["T"]
    assert bool(torch.isnan(o2[T:2 * T].float()).all())  # the skipped request's rows are not written
    keep = np.r_[0:T, 2 * T:4 * T]
    assert torch.equal(o2[keep].view(torch.int16), o[keep].view(torch.int16))


def test_verify_and_commit_in_a_cuda_graph():
    """Verify (tensor-core closed form) and commit captured in one CUDA graph replay bitwise like
    the eager calls: neither synchronises with the host nor allocates."""
    import torch
    import linear_attention_prefill_chunkwise_gb300 as lap
    c = make_case(seed=5040, B=12, T=8, H=2, HV=4, P=16, n_pad=2)
    B, T, H, HV, P = c["B"], c["T"], c["H"], c["HV"], c["P"]
    d = upload(c)
    pool0 = d["pool"].clone()
    acc = torch.from_numpy(np.random.default_rng(5041).integers(0, T + 1, B).astype(np.int32)).cuda()

    def buffers():
        return (torch.full((B * T, HV, W.V), float("nan"), dtype=torch.bfloat16, device="cuda"),
                torch.zeros((P, T, H, W.D), dtype=torch.bfloat16, device="cuda"),
                torch.zeros((P, T, HV, W.V), dtype=torch.bfloat16, device="cuda"), pool0.clone())

    def calls(o, kbuf, vbuf, pool):
        lap.la_verify(d["q"], d["k"], d["v"], d["slopes"], c["scale"], pool, T, state_indices=d["idx"], o=o,
                      kbuf=kbuf, vbuf=vbuf)
        lap.la_commit(pool, kbuf, vbuf, acc, d["slopes"], state_indices=d["idx"])

    ref = buffers()
    calls(*ref)
    torch.cuda.synchronize()
    bufs = buffers()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(*bufs)
    rows = live_rows(c)
    for _ in range(3):
        bufs[3].copy_(pool0)
        bufs[0].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(bufs[0][rows].view(torch.int16), ref[0][rows].view(torch.int16))
        assert torch.equal(bufs[3].view(torch.int32), ref[3].view(torch.int32))
