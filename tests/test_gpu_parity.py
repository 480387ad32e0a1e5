"""CUDA path vs the FP64 oracle, element by element, on seeded inputs.

Small problems are compared in full (several chunks, ragged tails, empty and
padded sequences, GVA, state pools); the five benchmark workloads at full size
are compared on sampled (sequence, value head) units the oracle computes one by
one, plus properties that hold at any size (untouched pool slots and padded
rows, finite outputs everywhere they are written).
"""
import zlib

import numpy as np
import pytest

import workloads as W
from harness import compare_full, compare_sampled, run_gpu, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_tiny_workload_full():
    p = W.config(1)
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, "tiny B=1 T=256 H=4")


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
}


@pytest.mark.parametrize("name", sorted(EDGE_CASES))
def test_edge_cases_full(name):
    kw = dict(EDGE_CASES[name])
    p = W.custom(seed=zlib.crc32(name.encode()) % 10000, name=name, **kw)
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, name)


def test_fixed_mha_b2_t8192_sampled():
    p = W.config(2)
    d = upload(p)
    run_gpu(p, d)
    compare_sampled(p, d, [(0, 0), (1, 63), (0, 31), (1, 1), (1, 40)], "B=2 T=8192 H=64")
    assert not torch.isnan(d["o"]).any().item()


def test_packed_varlen_pool_sampled():
    p = W.config(3)
    h0_before = p.h0.copy()
    d = upload(p)
    run_gpu(p, d)
    lengths = p.lengths()
    order = np.argsort(lengths)
    picks = [(int(order[-1]), 0), (int(order[-1]), 31), (int(order[0]), 5), (int(order[1]), 16),
             (int(order[len(order) // 2]), 7)]
    compare_sampled(p, d, picks, "packed N=32 H=32")
    assert not torch.isnan(d["o"]).any().item()
    h_gpu = d["h_final"].cpu().numpy()
    unsel = np.setdiff1d(np.arange(p.pool_size), p.state_indices)
    assert np.array_equal(h_gpu[unsel], h0_before[unsel])


def test_gva_long_sampled():
    p = W.config(4)
    d = upload(p)
    run_gpu(p, d)
    compare_sampled(p, d, [(0, 0), (3, 63), (2, 17)], "GVA B=4 T=16384 H=16 HV=64")


def test_short_sequences_pool_full():
    p = W.config(5)
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, "short packed N=128 T=8")


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
    q = torch.zeros((64, 1, 64), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((64, 1, 64), dtype=torch.bfloat16, device="cuda")
    sl = torch.ones(1, dtype=torch.float32, device="cuda")
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
