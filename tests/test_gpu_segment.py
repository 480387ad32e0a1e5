"""Segmented-sequence prefill (include/la_segment.h) vs the FP64 oracle.

The segmented path computes the same outputs and final states as the plain prefill, so
it is held to the same oracle and the same bounds: small problems in full (segments
ending inside a chunk, sequences shorter than one segment, empty and padded sequences,
GVA, in-place pools, no h0 / no final state, lambda = 1 and lambda = 0) at D = V = 128 and
64, a long few-head batch with the automatic segment length on sampled units, the device
error word, and two calls sharing one workspace.
"""
import zlib

import numpy as np
import pytest

import workloads as W
from harness import compare_full, compare_sampled, rel_rms, run_gpu, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def run_seg(p, d, segment_len, workspace=None, dev_error=None):
    import linear_attention_prefill_chunkwise_gb300 as lap
    return lap.la_prefill_fwd_segmented(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"],
                                        state_indices=d["idx"], cu_seqlens=d["cu"], o=d["o"], h_final=d["h_final"],
                                        seq_len=None if p.cu_seqlens is not None else p.T,
                                        segment_len=segment_len, workspace=workspace, dev_error=dev_error)


CASES = {
    # name: (problem arguments, segment length)
    "fixed_gva_ragged": (dict(B=2, T=1000, H=2, HV=4), 192),
    "packed_pool_padded_in_place": (dict(lengths=[0, 1, 63, 64, 65, 500, 1300, 64 * 7], H=2, HV=2, pool=12,
                                         indices=[3, 11, -1, 0, 7, 5, 1, 9], in_place=True), 128),
    "one_chunk_segments_no_h0": (dict(lengths=[700, 333], H=1, HV=4, with_h0=False), 64),
    "no_final_state": (dict(lengths=[900, 250], H=2, HV=2, want_final=False), 128),
    "pool_out_of_place": (dict(lengths=[333, 0, 777], H=1, HV=2, pool=5, indices=[4, 0, -1]), 256),
    "lambda_one": (dict(lengths=[900, 20], H=1, HV=2, slopes=[0.0, 0.0]), 256),
    "lambda_zero": (dict(lengths=[900, 20], H=1, HV=2, slopes=[100.0, 100.0]), 256),
    "segment_longer_than_some": (dict(lengths=[5000, 40, 3000], H=1, HV=1), 1024),
}


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("name", sorted(CASES))
def test_segmented_full(name, D):
    kw, seg = CASES[name]
    p = W.custom(seed=zlib.crc32(name.encode()) % 10000 + (D != 128), name=name, D=D, **kw)
    d = upload(p)
    run_seg(p, d, seg)
    compare_full(p, d, f"segmented {name} S={seg} D={D}")


@pytest.mark.parametrize("D", [128, 64])
def test_segmented_auto_length_full(D):
    """B=1, T=16384, H=HV=4: 4 chains, far fewer than SMs, so the automatic length segments."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=77, B=1, T=16384, H=4, HV=4, D=D)
    nbytes, seg = lap.la_prefill_segmented_workspace(1, 16384, 1, 4, False, 0)
    assert seg > 0 and seg % 64 == 0 and seg < 16384 and nbytes > 0
    d = upload(p)
    run_seg(p, d, 0)
    compare_full(p, d, f"segmented auto S={seg} D={D}")


@pytest.mark.parametrize("D", [128, 64])
def test_segmented_auto_short_first_segments_full(D):
    """B=1, T=4096, H=HV=64: two segments per chain would leave the local-state pass on 64
    SMs, so the automatic plan cuts the first half of each chain in two and keeps a long last
    segment; every unit against the oracle."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=81, B=1, T=4096, H=64, HV=64, D=D)
    nbytes, seg = lap.la_prefill_segmented_workspace(1, 4096, 1, 64, False, 0)
    if seg == 0:
        pytest.skip("this device has too few SMs for 64 chains to be segmented")
    d = upload(p)
    run_seg(p, d, 0)
    compare_full(p, d, f"segmented auto short first segments S={seg} D={D}")


def test_segmented_long_few_heads_sampled():
    """B=1, T=65536, H=HV=8 (a tensor-parallel shard of a 64-head layer), automatic length."""
    p = W.custom(seed=78, B=1, T=65536, H=8, HV=8)
    d = upload(p)
    run_seg(p, d, 0)
    compare_sampled(p, d, [(0, 0), (0, 7), (0, 3)], "segmented B=1 T=65536 H=8")
    assert not torch.isnan(d["o"]).any().item()


def test_segmented_close_to_plain():
    p = W.custom(seed=79, lengths=[3000, 17, 4100], H=2, HV=4)
    d1 = upload(p)
    run_gpu(p, d1)
    d2 = upload(p)
    run_seg(p, d2, 256)
    torch.cuda.synchronize()
    o1, o2 = d1["o"].float().cpu().numpy(), d2["o"].float().cpu().numpy()
    assert rel_rms(o2, o1) < 2e-3
    assert rel_rms(d2["h_final"].cpu().numpy(), d1["h_final"].cpu().numpy()) < 1e-4


def test_segmented_auto_falls_back_to_plain_bitwise():
    """With as many chains as SMs would fill, the automatic length runs the plain kernel."""
    import linear_attention_prefill_chunkwise_gb300 as lap
    p = W.custom(seed=80, B=2, T=300, H=64, HV=64)
    assert lap.la_prefill_segmented_workspace(2, 300, 2, 64, False, 0) == (0, 0)
    d1 = upload(p)
    run_gpu(p, d1)
    d2 = upload(p)
    run_seg(p, d2, 0)
    torch.cuda.synchronize()
    assert torch.equal(d1["o"].view(torch.int16), d2["o"].view(torch.int16))
    assert torch.equal(d1["h_final"].view(torch.int32), d2["h_final"].view(torch.int32))


def test_segmented_device_error_bad_seqlens_and_index():
    p = W.custom(seed=81, lengths=[400, 500, 600], H=1, HV=1, pool=4, indices=[0, 1, 2])
    d = upload(p)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = d["cu"].clone()
    cu[3] = cu[3] + 100  # sequence 2 ends beyond the batch; it overlaps no other sequence
    d["cu"] = cu
    run_seg(p, d, 128, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() & 1
    # the other sequences are intact and still correct
    compare_sampled(p, d, [(0, 0), (1, 0)], "segmented, bad bounds elsewhere")
    assert torch.isnan(d["o"][900:]).all().item()  # the skipped sequence's rows are not written

    d = upload(p)
    idx = d["idx"].clone()
    idx[2] = 9  # beyond the 4-slot pool
    d["idx"] = idx
    err.zero_()
    run_seg(p, d, 128, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() & 2
    compare_sampled(p, d, [(0, 0), (1, 0)], "segmented, bad index elsewhere")


def test_segmented_two_calls_share_a_workspace():
    import linear_attention_prefill_chunkwise_gb300 as lap
    pa = W.custom(seed=82, lengths=[1500, 64, 900], H=2, HV=2)
    pb = W.custom(seed=83, lengths=[10, 2000, 700], H=2, HV=2, with_h0=False)
    nbytes, _ = lap.la_prefill_segmented_workspace(1, max(pa.tokens, pb.tokens), 3, 2, True, 192)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")  # garbage on entry
    da, db = upload(pa), upload(pb)
    run_seg(pa, da, 192, workspace=ws)
    run_seg(pb, db, 192, workspace=ws)
    compare_full(pa, da, "first call")
    compare_full(pb, db, "second call, same workspace")
