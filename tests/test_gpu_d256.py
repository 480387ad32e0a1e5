"""Head dimension D = V = 256 (include/la_d256.h) against the FP64 oracle.

la_prefill_fwd_d256 evaluates the 256 x 256 state as four independent 128 x 128 blocks with the
D = 128 chunkwise kernel and adds the two key halves of every output in FP32 before one rounding.
The oracle runs the D = 256 recurrence itself, so these cases check the decomposition as well as
the kernels: ragged and packed batches, a pool in place with padding, GVA, no h0, no final state,
lambda = 1 and lambda -> 0, a bad state index, isolation from a non-finite neighbour, and two
calls bitwise equal; the short fixed-length and packed split paths (tokenwise kernel); the
segmented form; and the decoding ops at D = 256 in a CUDA graph.
"""
import zlib

import numpy as np
import pytest

import workloads as W
from harness import compare_full, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def run_d256(p, d, dev_error=None, workspace=None):
    import linear_attention_prefill_chunkwise_gb300 as lap
    return lap.la_prefill_fwd_d256(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], state_indices=d["idx"],
                                   cu_seqlens=d["cu"], o=d["o"], h_final=d["h_final"],
                                   seq_len=None if p.cu_seqlens is not None else p.T, dev_error=dev_error,
                                   workspace=workspace)


D256_CASES = {
    "fixed_T300": dict(B=2, T=300, H=2, HV=2),
    "fixed_T64": dict(B=3, T=64, H=1, HV=2),
    "ragged_pool_in_place_gva": dict(lengths=[1, 63, 64, 65, 130, 0, 200, 31], H=2, HV=4, pool=11,
                                     indices=[3, 10, -1, 0, 7, 5, 1, 9], in_place=True),
    "gva_three_heads_per_group": dict(lengths=[150, 77], H=1, HV=3),
    "pool_out_of_place": dict(lengths=[333, 0, 777], H=1, HV=2, pool=5, indices=[4, 0, -1]),
    "no_h0": dict(lengths=[70, 3, 129], H=2, HV=2, with_h0=False),
    "no_final": dict(lengths=[70, 3], H=2, HV=2, want_final=False),
    "lambda_one": dict(lengths=[150, 20], H=1, HV=2, slopes=[0.0, 0.0]),
    "lambda_zero": dict(lengths=[150, 20], H=1, HV=2, slopes=[100.0, 100.0]),
    "long_nine_chunks": dict(lengths=[64 * 9 + 17], H=1, HV=1),
    "short_sequences": dict(lengths=[5, 20, 3, 31, 1, 40], H=2, HV=2),
    "empty_sequences_with_final": dict(lengths=[0, 0, 5], H=1, HV=2),
    # fixed length, T <= 32: the tokenwise kernel's D = 256 instance on whole states
    "short_fixed_T32_tokenwise": dict(B=3, T=32, H=2, HV=4),
    "short_fixed_T1_tokenwise": dict(B=4, T=1, H=1, HV=2),
    "short_fixed_T17_pool_in_place_tokenwise": dict(B=3, T=17, H=1, HV=2, pool=5, indices=[4, -1, 1],
                                                    in_place=True),
    "short_fixed_T8_no_h0_tokenwise": dict(B=2, T=8, H=2, HV=2, with_h0=False),
    # packed, at most 64 tokens per sequence on average: the short ones on the tokenwise kernel
    "split_pool_in_place_padded": dict(lengths=[9, 32, 0, 17, 33, 2, 100], H=1, HV=2, pool=9,
                                       indices=[4, 0, 8, -1, 2, 6, 1], in_place=True),
    "split_gva_no_h0": dict(lengths=[8, 8, 70, 8, 8, 8], H=2, HV=4, with_h0=False),
}


@pytest.mark.parametrize("name", sorted(D256_CASES))
def test_d256_cases_full(name):
    p = W.custom(seed=zlib.crc32(("d256" + name).encode()) % 10000, name=name, D=256, **D256_CASES[name])
    d = upload(p)
    run_d256(p, d)
    compare_full(p, d, f"D=256 {name}")


def test_d256_fixed_b2_t2048_h4_full():
    p = W.custom(seed=4002, B=2, T=2048, H=4, HV=4, D=256, name="D=256 B=2 T=2048 H=4")
    d = upload(p)
    run_d256(p, d)
    compare_full(p, d, p.name)


def test_d256_bad_index_flagged_others_intact():
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=4003, lengths=[100, 65, 30], H=1, HV=2, D=256, pool=4, indices=[2, 0, 3])
    d = upload(p)
    run_d256(p, d)
    o_ref = d["o"].clone()
    hf_ref = d["h_final"].clone()
    d2 = upload(p)
    d2["idx"] = torch.tensor([2, 9, 3], dtype=torch.int32, device="cuda")  # slot 9 is past the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_d256(p, d2, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lap.DEV_ERR_BAD_INDEX
    a, b = int(p.cu_seqlens[1]), int(p.cu_seqlens[2])
    keep = np.r_[0:a, b:p.tokens]
    assert torch.equal(d2["o"][keep].view(torch.int16), o_ref[keep].view(torch.int16))
    assert bool(torch.isnan(d2["o"][a:b].float()).all())  # the skipped sequence's rows are not written
    for slot in (2, 3):
        assert torch.equal(d2["h_final"][slot].view(torch.int32), hf_ref[slot].view(torch.int32))


def test_d256_nonfinite_sequence_does_not_reach_its_neighbours():
    lengths = [100, 77, 150, 64, 40]
    p = W.custom(seed=4004, lengths=lengths, H=1, HV=2, D=256)
    a, b = int(p.cu_seqlens[2]), int(p.cu_seqlens[3])
    p.k_bits[a:b] = 0x7F80
    p.v_bits[a:b] = 0x7FC0
    d = upload(p)
    run_d256(p, d)
    torch.cuda.synchronize()
    o_all = d["o"].view(torch.int16).cpu().numpy()
    for n in (0, 1, 3, 4):
        s, e = int(p.cu_seqlens[n]), int(p.cu_seqlens[n + 1])
        pa = W.Problem("alone", p.q_bits[s:e].copy(), p.k_bits[s:e].copy(), p.v_bits[s:e].copy(), p.slopes,
                       p.scale, p.H, p.HV, 1, e - s, np.array([0, e - s], dtype=np.int32), None,
                       p.h0[n:n + 1].copy(), D=256, V=256)
        da = upload(pa)
        run_d256(pa, da)
        torch.cuda.synchronize()
        assert np.array_equal(o_all[s:e], da["o"].view(torch.int16).cpu().numpy()), f"sequence {n}"
        assert np.array_equal(d["h_final"][n].view(torch.int32).cpu().numpy(),
                              da["h_final"][0].view(torch.int32).cpu().numpy()), f"sequence {n} state"


def test_d256_two_calls_bitwise_and_garbage_workspace():
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=4005, lengths=[300, 1, 129], H=2, HV=4, D=256, pool=6, indices=[5, -1, 2])
    nbytes = lap.la_prefill_d256_workspace(p.B, p.T, p.N, p.HV, True)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")  # NaN-like garbage
    outs = []
    for _ in range(2):
        d = upload(p)
        run_d256(p, d, workspace=ws)
        torch.cuda.synchronize()
        outs.append((d["o"].view(torch.int16).clone(), d["h_final"].view(torch.int32).clone()))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("seed", range(12))
def test_d256_random(seed):
    """Random batches (the generator of tests/test_gpu_random.py) at D = V = 256."""
    from test_gpu_random import _draw
    kw, _ = _draw(seed)
    kw["D"] = 256
    p = W.custom(seed=seed, name=f"random d256 {seed}", **kw)
    d = upload(p)
    run_d256(p, d)
    compare_full(p, d, f"random D=256 {seed} {kw}")


def test_d256_in_a_cuda_graph():
    """The five kernels of one call captured in a CUDA graph replay bitwise like the eager call:
    the call neither synchronises with the host nor allocates."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=4006, lengths=[200, 0, 65], H=1, HV=2, D=256, pool=4, indices=[3, -1, 1], in_place=True)
    ref = upload(p)
    run_d256(p, ref)
    torch.cuda.synchronize()
    d = upload(p)
    h0_init = d["h0"].clone()
    ws = torch.empty(lap.la_prefill_d256_workspace(p.B, p.T, p.N, p.HV, True), dtype=torch.uint8, device="cuda")
    run_d256(p, d, workspace=ws)  # warm-up outside the capture (first-call setup)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_d256(p, d, workspace=ws)
    for _ in range(2):
        d["h0"].copy_(h0_init)
        d["o"].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(d["o"].view(torch.int16), ref["o"].view(torch.int16))
        assert torch.equal(d["h0"].view(torch.int32), ref["h0"].view(torch.int32))


def run_d256_seg(p, d, segment_len, dev_error=None):
    import linear_attention_prefill_chunkwise_gb300 as lap
    return lap.la_prefill_fwd_d256_segmented(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"],
                                             state_indices=d["idx"], cu_seqlens=d["cu"], o=d["o"],
                                             h_final=d["h_final"], seq_len=None if p.cu_seqlens is not None else p.T,
                                             segment_len=segment_len, dev_error=dev_error)


@pytest.mark.parametrize("name", ["fixed_gva_ragged", "packed_pool_padded_in_place", "one_chunk_segments_no_h0",
                                  "no_final_state", "pool_out_of_place", "lambda_one", "lambda_zero",
                                  "segment_longer_than_some"])
def test_d256_segmented_full(name):
    """The segmented prefill's edge cases (tests/test_gpu_segment.py) at D = V = 256."""
    from test_gpu_segment import CASES
    kw, seg = CASES[name]
    p = W.custom(seed=zlib.crc32(("d256seg" + name).encode()) % 10000, name=name, D=256, **kw)
    d = upload(p)
    run_d256_seg(p, d, seg)
    compare_full(p, d, f"D=256 segmented {name} S={seg}")


def test_d256_segmented_auto_length_full():
    """B=1, T=8192, H=HV=2: 8 block chains, so the automatic length segments."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=4010, B=1, T=8192, H=2, HV=2, D=256)
    nbytes, seg = lap.la_prefill_d256_segmented_workspace(1, 8192, 1, 2, False, 0, True)
    assert seg > 0 and seg % 64 == 0 and seg < 8192
    d = upload(p)
    run_d256_seg(p, d, 0)
    compare_full(p, d, f"D=256 segmented auto S={seg}")


def test_d256_segmented_close_to_plain_d256():
    p = W.custom(seed=4011, lengths=[3000, 17, 2100], H=1, HV=2, D=256)
    d1 = upload(p)
    run_d256(p, d1)
    d2 = upload(p)
    run_d256_seg(p, d2, 256)
    torch.cuda.synchronize()
    from harness import rel_rms
    assert rel_rms(d2["o"].float().cpu().numpy(), d1["o"].float().cpu().numpy()) < 2e-3
    assert rel_rms(d2["h_final"].cpu().numpy(), d1["h_final"].cpu().numpy()) < 1e-4


def test_d256_segmented_two_calls_share_a_garbage_workspace():
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=4012, lengths=[700, 0, 333], H=1, HV=2, D=256, pool=5, indices=[4, -1, 0])
    nbytes, seg = lap.la_prefill_d256_segmented_workspace(p.B, p.T, p.N, p.HV, True, 128, True)
    assert seg == 128
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        d = upload(p)
        lap.la_prefill_fwd_d256_segmented(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"],
                                          state_indices=d["idx"], cu_seqlens=d["cu"], o=d["o"], h_final=d["h_final"],
                                          segment_len=128, workspace=ws)
        torch.cuda.synchronize()
        outs.append((d["o"].view(torch.int16).clone(), d["h_final"].view(torch.int32).clone()))
        compare_full(p, d, "D=256 segmented, garbage workspace")
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])


def test_d256_decode_and_commit_in_a_cuda_graph():
    """MTP decode and commit at D = 256 (the tokenwise kernel's 256-thread instance) captured in
    one CUDA graph replay bitwise like the eager calls."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    from test_gpu_decode import make_case
    from test_gpu_decode import upload as dec_upload
    c = make_case(seed=4013, B=6, T=5, H=1, HV=2, P=8, n_pad=1, D=256)
    d = dec_upload(c)
    pool0 = d["pool"].clone()
    B, T, H, HV, P = c["B"], c["T"], c["H"], c["HV"], c["P"]
    kbuf = torch.zeros((P, T, H, 256), dtype=torch.bfloat16, device="cuda")
    vbuf = torch.zeros((P, T, HV, 256), dtype=torch.bfloat16, device="cuda")
    acc = torch.tensor([5, 0, 3, 5, 1, 2], dtype=torch.int32, device="cuda")

    def calls(o, pool):
        lap.la_verify(d["q"], d["k"], d["v"], d["slopes"], c["scale"], pool, T, state_indices=d["idx"], o=o,
                      kbuf=kbuf, vbuf=vbuf)
        lap.la_commit(pool, kbuf, vbuf, acc, d["slopes"], state_indices=d["idx"])

    o_ref = torch.full((B * T, HV, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool_ref = pool0.clone()
    calls(o_ref, pool_ref)
    torch.cuda.synchronize()
    o = torch.full_like(o_ref, float("nan"))
    pool = pool0.clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(o, pool)
    for _ in range(2):
        pool.copy_(pool0)
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(pool.view(torch.int32), pool_ref.view(torch.int32))


def test_d256_parts_past_two_to_the_31_elements():
    """A packed batch of 266,240 tokens with 16 value heads at D = 256: the FP32 parts of o
    (tokens x 64 block heads x 128) hold 2.18e9 elements.  The first sequence is padded (never
    read or written); the second, the last 100 tokens, lies past element 2^31 of the parts, so
    their stores, the sum's loads and the output rows exercise 64-bit offsets: outputs and final
    state against the oracle, the padded rows and slot untouched."""
    import oracle
    from harness import check_output, check_state, to_torch_bf16
    tokens, H, HV, L = (1 << 18) + (1 << 12), 16, 16, 100
    assert (tokens - L) * 4 * HV * 128 > 2 ** 31
    dev = "cuda"
    rng = np.random.default_rng(41)
    qb, kb, vb = W.make_qkv(rng, L, H, HV, d=256, v_dim=256)
    h0_np = W.make_states(rng, 2, HV, d=256, v_dim=256)
    slopes = W.slopes_for(HV)
    scale = 1.0 / 16.0
    q = torch.empty((tokens, H, 256), dtype=torch.bfloat16, device=dev)
    k = torch.empty_like(q)
    v = torch.empty((tokens, HV, 256), dtype=torch.bfloat16, device=dev)
    q[-L:] = to_torch_bf16(qb, dev)
    k[-L:] = to_torch_bf16(kb, dev)
    v[-L:] = to_torch_bf16(vb, dev)
    o = torch.full((tokens, HV, 256), float("nan"), dtype=torch.bfloat16, device=dev)
    h0 = torch.from_numpy(h0_np).to(dev)
    hf = torch.full_like(h0, float("nan"))
    idx = torch.tensor([-1, 1], dtype=torch.int32, device=dev)
    cu = torch.tensor([0, tokens - L, tokens], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    import linear_attention_prefill_chunkwise_gb300 as lap
    lap.la_prefill_fwd_d256(q, k, v, torch.from_numpy(slopes).to(dev), scale, h0=h0, state_indices=idx,
                            cu_seqlens=cu, o=o, h_final=hf, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    o_ref, h_ref = oracle.tokenwise(W.bf16_to_f32(qb), W.bf16_to_f32(kb), W.bf16_to_f32(vb), slopes, scale,
                                    h0=h0_np[1:2].astype(np.float64), cu_seqlens=np.array([0, L], dtype=np.int32))
    check_output(o[-L:].float().cpu().numpy(), o_ref, "D=256 rows past 2^31 part elements")
    check_state(hf[1].cpu().numpy(), h_ref[0], "D=256 state of the sequence past 2^31 part elements")
    assert bool(torch.isnan(hf[0]).all())
    for r in (0, tokens // 2, tokens - L - 1):
        assert bool(torch.isnan(o[r].float()).all())
    del q, k, v, o
    torch.cuda.empty_cache()
