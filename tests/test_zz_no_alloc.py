"""la_prefill_fwd_segmented_static: the segmented prefill for callers that cannot allocate
device memory (a plugin whose host framework owns all device memory, a path that must not
call cudaMalloc).  Its scratch is a 16 MiB buffer built into the library instead of a
caller workspace.

Checked here: through the C ABI, two calls in a row give bit for bit what
la_prefill_fwd_segmented gives with a caller-allocated workspace (both build the same plan
and run the same deterministic kernels, so any leftover state of the shared buffer would
show), and each is within the oracle's bounds on its own; a plan larger than the buffer is
refused on the host before anything is launched, and an invalid call is reported as invalid
whatever its size.  This file is collected last, so a run that stops at its first failure has
run every other test first.
"""
import ctypes

import numpy as np
import pytest

import linear_attention_prefill_chunkwise_gb300 as lap
import workloads as W

LA_INVALID, LA_UNSUPPORTED = 1, 2
FAKE = 0x10000  # never dereferenced: the calls below are refused on the host


def _static_call(lib, q=FAKE, slopes=FAKE, T=1 << 20):
    return lib.la_prefill_fwd_segmented_static(q, FAKE, FAKE, slopes, ctypes.c_float(1.0), None, None, None, FAKE,
                                               None, 1, T, 1, 64, 64, 128, 128, 0, 64, None, None)


def test_plan_beyond_the_buffer_is_refused_on_the_host():
    lib = lap.load_library()
    # 1M tokens in 64-token segments over 64 heads: 16384 x 64 states of 64 KiB, far over 16 MiB
    assert _static_call(lib) == LA_UNSUPPORTED
    assert b"scratch" in lib.la_last_error()


def test_invalid_arguments_are_reported_before_the_size_check():
    lib = lap.load_library()
    assert _static_call(lib, q=FAKE + 2) == LA_INVALID  # misaligned q
    assert _static_call(lib, slopes=None) == LA_INVALID
    assert b"scratch" not in lib.la_last_error()


@pytest.mark.gpu
def test_static_scratch_matches_caller_workspace_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    from harness import compare_full, upload

    problems = [
        (W.custom(seed=91, B=1, T=20000, H=4, HV=4), 0),  # automatic segment length
        (W.custom(seed=92, lengths=[3000, 5, 2500, 640], H=2, HV=4, pool=6, indices=[5, 0, -1, 2],
                  in_place=True), 256),
    ]
    runs = []
    for p, seg in problems:  # the built-in buffer, two calls back to back on one stream
        d = upload(p)
        lap.la_prefill_fwd_segmented_static(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"],
                                            state_indices=d["idx"], cu_seqlens=d["cu"], o=d["o"],
                                            h_final=d["h_final"], seq_len=None if p.cu_seqlens is not None else p.T,
                                            segment_len=seg)
        runs.append(d)
    torch.cuda.synchronize()
    for (p, seg), d in zip(problems, runs):
        ref = upload(p)
        lap.la_prefill_fwd_segmented(ref["q"], ref["k"], ref["v"], ref["slopes"], p.scale, h0=ref["h0"],
                                     state_indices=ref["idx"], cu_seqlens=ref["cu"], o=ref["o"],
                                     h_final=ref["h_final"], seq_len=None if p.cu_seqlens is not None else p.T,
                                     segment_len=seg)
        torch.cuda.synchronize()
        assert torch.equal(d["o"].view(torch.int16), ref["o"].view(torch.int16)), \
            f"{p.name}: built-in scratch output differs from the caller-workspace output"
        assert torch.equal(d["h_final"].view(torch.int32), ref["h_final"].view(torch.int32)), \
            f"{p.name}: built-in scratch final states differ from the caller-workspace ones"
        compare_full(p, d, f"{p.name}: built-in scratch vs the oracle")
