"""CUDA path vs the FP64 oracle, element by element, on seeded inputs.

Small problems are compared in full (several chunks, ragged tails, empty and
padded sequences, GVA, state pools), and so are the five benchmark workloads at
full size: every (sequence, value head) unit's output rows and final state must
meet the bounds on its own, padded rows stay unwritten and unselected pool slots
keep their initial value bit for bit.
"""
import zlib

import numpy as np
import pytest

import workloads as W
from harness import compare_every_unit, compare_full, run_gpu, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_tiny_workload_full():
    p = W.config(1)
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, "tiny B=1 T=256 H=4")
    compare_every_unit(p, d, "tiny B=1 T=256 H=4")


EDGE_CASES = {
    "ragged_lengths_h0": dict(lengths=[1, 63, 64, 65, 130, 0, 200], H=2, HV=2),
    "gva_g2": dict(lengths=[100, 37, 64], H=2, HV=4),
    "gva_g4": dict(lengths=[129, 5], H=1, HV=4),
    "no_h0": dict(lengths=[70, 3], H=2, HV=2, with_h0=False),
    "no_final": dict(lengths=[70, 3], H=2, HV=2, want_final=False),
    "pool_padded_in_place": dict(lengths=[10, 30, 5, 64, 90], H=2, HV=2, pool=9,
                                 indices=[6, -1, 2, 4, -1], in_place=True),
    "pool_out_of_place": dict(lengths=[33, 0, 77], H=1, HV=2, pool=5, indices=[4, 0, -1]),
    "fixed_T100": dict(B=3, T=100, H=2, HV=2),
    "fixed_T64": dict(B=2, T=64, H=2, HV=2),
    "fixed_T1": dict(B=4, T=1, H=1, HV=1),
    "unit_scale": dict(lengths=[300], H=1, HV=1, scale=1.0),
    "lambda_one": dict(lengths=[150, 20], H=1, HV=2, slopes=[0.0, 0.0]),
    "lambda_zero": dict(lengths=[150, 20], H=1, HV=2, slopes=[100.0, 100.0]),
    "long_two_chunks_plus": dict(lengths=[64 * 9 + 17], H=1, HV=1),
    # sequences of at most 32 tokens run in the tokenwise kernel, longer ones in the chunkwise one
    "short_long_boundary": dict(lengths=[32, 33, 31, 16, 17, 0, 100, 1, 64], H=2, HV=4, pool=11,
                                indices=[3, 10, -1, 0, 7, 5, 1, 9, 2], in_place=True),
    "fixed_T32_tokenwise": dict(B=3, T=32, H=2, HV=2),
    "fixed_T33_chunkwise": dict(B=3, T=33, H=2, HV=2),
    "short_no_h0": dict(lengths=[5, 20, 0, 3, 32], H=1, HV=2, with_h0=False),
    "short_no_final": dict(lengths=[5, 20, 3, 31], H=2, HV=2, want_final=False),
    "fixed_T8_gva_pool": dict(B=4, T=8, H=1, HV=4, pool=6, indices=[5, -1, 0, 3], in_place=True),
    # packed batches of at most 256 sequences run a longest-first unit schedule; ties in length
    # are ranked by sequence index, padded sequences count as empty
    "packed_tied_lengths": dict(lengths=[100] * 6 + [37] * 5 + [300, 0, 100], H=1, HV=2, pool=16,
                                indices=[0, 1, 2, 3, 4, 5, 6, 7, 8, 9, -1, 11, 12, 13], in_place=True),
    # more than 256 sequences: round robin
    "packed_300_sequences": dict(lengths=[(37 * i) % 211 for i in range(300)], H=1, HV=2),
}


@pytest.mark.parametrize("name", sorted(EDGE_CASES))
def test_edge_cases_full(name):
    kw = dict(EDGE_CASES[name])
    p = W.custom(seed=zlib.crc32(name.encode()) % 10000, name=name, **kw)
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, name)


# The four large workloads, every (sequence, value head) unit against the oracle run over the
# whole problem (0.5 to 2 s of host time each on 16 cores).


def test_fixed_mha_b2_t8192_every_unit():
    p = W.config(2)
    d = upload(p)
    run_gpu(p, d)
    compare_every_unit(p, d, "B=2 T=8192 H=64")


def test_packed_varlen_pool_every_unit():
    p = W.config(3)
    d = upload(p)
    run_gpu(p, d)
    # all 32 sequences x 32 heads, the 32 slots not selected bit-identical to their initial value
    compare_every_unit(p, d, "packed N=32 H=32")


def test_gva_long_every_unit():
    p = W.config(4)
    d = upload(p)
    run_gpu(p, d)
    compare_every_unit(p, d, "GVA B=4 T=16384 H=16 HV=64")


def test_short_sequences_pool_every_unit():
    p = W.config(5)
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, "short packed N=128 T=8")
    compare_every_unit(p, d, "short packed N=128 T=8")


@pytest.mark.parametrize("which", ["small", "packed_full"])
def test_persistent_equals_non_persistent_bitwise(which):
    if which == "small":
        p = W.custom(seed=5, lengths=[1, 63, 64, 65, 130, 0, 200, 17, 64 * 5], H=2, HV=4, pool=12,
                     indices=[3, 11, -1, 0, 7, 5, 1, 2, 9])
    else:
        p = W.config(3)
    outs = []
    for sched in ("persistent", "non_persistent"):
        d = upload(p)
        run_gpu(p, d, schedule=sched)
        torch.cuda.synchronize()
        outs.append((d["o"].view(torch.int16).cpu().numpy(), d["h_final"].view(torch.int32).cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


def test_device_error_word_bad_seqlens_and_index():
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=9, lengths=[40, 50, 60], H=1, HV=1, pool=4, indices=[0, 1, 2])
    d = upload(p)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_cu = d["cu"].clone()
    bad_cu[2] = bad_cu[1] - 1  # sequence 1 has negative length
    lap.la_prefill_fwd(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], state_indices=d["idx"],
                       cu_seqlens=bad_cu, o=d["o"], h_final=d["h_final"], dev_error=err)
    torch.cuda.synchronize()
    assert err.item() & lap.DEV_ERR_BAD_SEQLENS
    err.zero_()
    bad_idx = d["idx"].clone()
    bad_idx[0] = 4  # == pool size
    lap.la_prefill_fwd(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], state_indices=bad_idx,
                       cu_seqlens=d["cu"], o=d["o"], h_final=d["h_final"], dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == lap.DEV_ERR_BAD_INDEX


def test_device_error_word_all_short_batch():
    """A packed batch of sequences of at most 32 tokens runs in the tokenwise kernel, and the
    chunkwise kernel launched beside it returns at once unless a sequence is long or its bounds
    are bad: bad bounds are still reported, a bad index too, and the valid sequences computed."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=19, lengths=[5, 20, 31, 12], H=2, HV=2, pool=6, indices=[3, 0, 5, 1])
    d = upload(p)
    run_gpu(p, d)
    torch.cuda.synchronize()
    compare_full(p, d, "all short packed")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_cu = d["cu"].clone()
    bad_cu[2] = bad_cu[1] - 1  # sequence 1 has negative length
    lap.la_prefill_fwd(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], state_indices=d["idx"],
                       cu_seqlens=bad_cu, o=d["o"], h_final=d["h_final"], dev_error=err)
    torch.cuda.synchronize()
    assert err.item() & lap.DEV_ERR_BAD_SEQLENS
    err.zero_()
    bad_idx = d["idx"].clone()
    bad_idx[2] = 6  # == pool size
    lap.la_prefill_fwd(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], state_indices=bad_idx,
                       cu_seqlens=d["cu"], o=d["o"], h_final=d["h_final"], dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == lap.DEV_ERR_BAD_INDEX


def test_cuda_graph_capture_and_replay_deterministic():
    p = W.custom(seed=13, lengths=[1, 100, 64, 257], H=2, HV=2, pool=6, indices=[5, 0, 3, -1])
    d = upload(p)
    h0 = d["h0"].clone()
    hf = torch.empty_like(h0)
    run_gpu(p, {**d, "h_final": hf})  # warm-up outside capture
    torch.cuda.synchronize()
    o_ref = d["o"].clone()
    hf_ref = hf.clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_gpu(p, {**d, "h_final": hf}, stream=s)
    for _ in range(5):
        d["o"].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(d["o"].view(torch.int16)[~torch.isnan(o_ref[:, 0, 0])],
                           o_ref.view(torch.int16)[~torch.isnan(o_ref[:, 0, 0])])
        assert torch.equal(hf[[5, 0, 3]].view(torch.int32), hf_ref[[5, 0, 3]].view(torch.int32))


@pytest.mark.parametrize("cfg", [2, 4])
def test_back_to_back_calls_bitwise(cfg):
    # Calls on one stream overlap their launches (programmatic stream serialization): each waits
    # for the previous kernel before touching memory, so back-to-back calls into separate output
    # buffers must agree bit for bit (GVA: two units per CTA on part of the SMs).
    p = W.config(cfg)
    d = upload(p)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(4):
            o = torch.empty_like(d["o"])
            hf = torch.empty_like(d["h_final"])
            run_gpu(p, {**d, "o": o, "h_final": hf}, stream=s.cuda_stream)
            outs.append((o, hf))
    torch.cuda.synchronize()
    for o, hf in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(hf.view(torch.int32), outs[0][1].view(torch.int32))


def test_two_streams_concurrent_equals_serial():
    pa = W.custom(seed=21, lengths=[300, 70, 1], H=2, HV=2)
    pb = W.custom(seed=22, B=2, T=200, H=1, HV=2)
    da, db = upload(pa), upload(pb)
    run_gpu(pa, da)
    run_gpu(pb, db)
    torch.cuda.synchronize()
    ref = [da["o"].clone(), da["h_final"].clone(), db["o"].clone(), db["h_final"].clone()]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(10):
        for t in (da["o"], db["o"]):
            t.fill_(float("nan"))
        torch.cuda.synchronize()
        run_gpu(pa, da, stream=s1)
        run_gpu(pb, db, stream=s2)
        torch.cuda.synchronize()
        got = [da["o"], da["h_final"], db["o"], db["h_final"]]
        for x, y in zip(got, ref):
            assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                               y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))


def test_rejected_shapes_return_status_without_launch():
    import linear_attention_prefill_chunkwise_gb300 as lap
    q = torch.zeros((64, 1, 32), dtype=torch.bfloat16, device="cuda")  # D = V = 32: not implemented
    v = torch.zeros((64, 1, 32), dtype=torch.bfloat16, device="cuda")
    sl = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(lap.LaError) as e:
        lap.la_prefill_fwd(q, q, v, sl, 1.0, seq_len=64)
    assert e.value.name == "LA_ERR_UNSUPPORTED"
    q = torch.zeros((64, 1, 64), dtype=torch.bfloat16, device="cuda")  # D = 64 with V = 128
    v = torch.zeros((64, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lap.LaError) as e:
        lap.la_prefill_fwd(q, q, v, sl, 1.0, seq_len=64)
    assert e.value.name == "LA_ERR_UNSUPPORTED"
    q = torch.zeros((64, 3, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((64, 4, 128), dtype=torch.bfloat16, device="cuda")
    sl = torch.ones(4, dtype=torch.float32, device="cuda")
    with pytest.raises(lap.LaError) as e:
        lap.la_prefill_fwd(q, q, v, sl, 1.0, seq_len=64)
    assert e.value.name == "LA_ERR_UNSUPPORTED"
    # misaligned q (offset by one element)
    qq = torch.zeros((64 * 4 * 128 + 1,), dtype=torch.bfloat16, device="cuda")[1:].view(64, 4, 128)
    with pytest.raises(lap.LaError) as e:
        lap.la_prefill_fwd(qq, qq, v, sl, 1.0, seq_len=64)
    assert e.value.name == "LA_ERR_INVALID_ARGUMENT"


# Packed sequences are unrelated requests: a non-finite value in one must not reach another.
# Sequence 2 holds +inf keys, NaN values and -inf queries; sequence 1 (77 tokens) ends inside a
# chunk whose tile rows past its end are sequence 2's, and sequence 4 (40 tokens) likewise reads
# sequence 5's clean rows.  Every other sequence must be bit-identical to running it alone.
ISOLATION_LENGTHS = [100, 77, 150, 64, 40, 200, 33, 65]
POISONED = 2


def _poisoned_problem():
    p = W.custom(seed=4242, lengths=ISOLATION_LENGTHS, H=2, HV=4)
    a, b = int(p.cu_seqlens[POISONED]), int(p.cu_seqlens[POISONED + 1])
    p.k_bits[a:b] = 0x7F80  # +inf
    p.v_bits[a:b] = 0x7FC0  # NaN
    p.q_bits[a:b] = 0xFF80  # -inf
    return p


def _alone(p, n):
    a, b = int(p.cu_seqlens[n]), int(p.cu_seqlens[n + 1])
    return W.Problem(f"sequence {n} alone", p.q_bits[a:b].copy(), p.k_bits[a:b].copy(), p.v_bits[a:b].copy(),
                     p.slopes, p.scale, p.H, p.HV, 1, b - a, np.array([0, b - a], dtype=np.int32), None,
                     p.h0[n:n + 1].copy())


def _run_path(path, p, d):
    import linear_attention_prefill_chunkwise_gb300 as lap
    if path == "prefill":
        run_gpu(p, d)
    else:
        lap.la_prefill_fwd_segmented(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], cu_seqlens=d["cu"],
                                     o=d["o"], h_final=d["h_final"], segment_len=64)
    torch.cuda.synchronize()


@pytest.mark.parametrize("path", ["prefill", "segmented"])
def test_nonfinite_sequence_does_not_reach_its_neighbours(path):
    p = _poisoned_problem()
    d = upload(p)
    _run_path(path, p, d)
    o_all = d["o"].view(torch.int16).cpu().numpy()
    h_all = d["h_final"].view(torch.int32).cpu().numpy()
    for n in range(len(ISOLATION_LENGTHS)):
        if n == POISONED:
            continue
        a, b = int(p.cu_seqlens[n]), int(p.cu_seqlens[n + 1])
        pa = _alone(p, n)
        da = upload(pa)
        _run_path(path, pa, da)
        o_one = da["o"].view(torch.int16).cpu().numpy()
        h_one = da["h_final"].view(torch.int32).cpu().numpy()
        assert np.array_equal(o_all[a:b], o_one), f"{path}: sequence {n} output differs from running it alone"
        assert np.array_equal(h_all[n], h_one[0]), f"{path}: sequence {n} final state differs from running it alone"


def test_rows_past_two_to_the_31_elements():
    """A packed batch of 2^20 tokens with 32 heads: q, k, v and o each hold 2^32 elements (8 GiB).
    Its first sequence is padded (never read or written); the second, the last 100 tokens, lies
    past element 2^31 of every tensor, so its loads, stores and state slots exercise 64-bit
    offsets: outputs and final state against the oracle, the padded rows and slot untouched."""
    import oracle
    import linear_attention_prefill_chunkwise_gb300 as lap
    from harness import check_output, check_state, to_torch_bf16
    tokens, H, HV, L = 1 << 20, 32, 32, 100
    assert (tokens - L) * HV * 128 > 2 ** 31
    dev = "cuda"
    rng = np.random.default_rng(31)
    qb, kb, vb = W.make_qkv(rng, L, H, HV)
    h0_np = W.make_states(rng, 2, HV)
    slopes = W.slopes_for(HV)
    scale = 1.0 / np.sqrt(128.0)
    q = torch.empty((tokens, H, 128), dtype=torch.bfloat16, device=dev)
    k = torch.empty_like(q)
    v = torch.empty((tokens, HV, 128), dtype=torch.bfloat16, device=dev)
    q[-L:] = to_torch_bf16(qb, dev)
    k[-L:] = to_torch_bf16(kb, dev)
    v[-L:] = to_torch_bf16(vb, dev)
    o = torch.full((tokens, HV, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    h0 = torch.from_numpy(h0_np).to(dev)
    hf = torch.full_like(h0, float("nan"))
    idx = torch.tensor([-1, 1], dtype=torch.int32, device=dev)
    cu = torch.tensor([0, tokens - L, tokens], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lap.la_prefill_fwd(q, k, v, torch.from_numpy(slopes).to(dev), scale, h0=h0, state_indices=idx, cu_seqlens=cu,
                       o=o, h_final=hf, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    o_ref, h_ref = oracle.tokenwise(W.bf16_to_f32(qb), W.bf16_to_f32(kb), W.bf16_to_f32(vb), slopes, scale,
                                    h0=h0_np[1:2].astype(np.float64), cu_seqlens=np.array([0, L], dtype=np.int32))
    check_output(o[-L:].float().cpu().numpy(), o_ref, "rows past 2^31 elements")
    check_state(hf[1].cpu().numpy(), h_ref[0], "state of the sequence past 2^31 elements")
    assert bool(torch.isnan(hf[0]).all())
    for r in (0, tokens // 2, tokens - L - 1):
        assert bool(torch.isnan(o[r].float()).all())
    del q, k, v, o
    torch.cuda.empty_cache()
