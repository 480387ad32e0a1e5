"""The kernels' timeout exit, exercised without hanging anything.

Every pipeline wait in the kernels is bounded: past its limit the CTA raises its abort flag,
every role leaves its loop, the CTA waits for its own loads and MMAs in flight, frees its
tensor memory and returns, and LA_DEV_ERR_TIMEOUT is set in the caller's error word.  The
normal limit (one second) is never reached by a healthy pipeline, so this test builds the
prefill entry point with a 100 ns limit, which ordinary waits (a tile arriving from HBM, an
MMA group) exceed.  The call must return LA_OK, the error word must carry the timeout bit,
and the CUDA context must stay usable: the normal library then computes the same problem
within the oracle's bounds.
"""
import ctypes

import pytest

import workloads as W
from harness import compare_full, run_gpu, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _short_limit_library():
    from linear_attention_prefill_chunkwise_gb300 import build as b
    lib = ctypes.CDLL(b.build(wait_limit_ns=100))
    vp, ip = ctypes.c_void_p, ctypes.c_void_p
    # q, k, v, slopes, scale, h0, state_indices, cu_seqlens, o, h_final, B, T, N, H, HV, D, V, pool_size,
    # schedule, dev_error, stream
    lib.la_prefill_fwd.argtypes = [vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp] + [ctypes.c_int] * 9 + [ip, vp]
    lib.la_prefill_fwd.restype = ctypes.c_int
    return lib


def test_wait_limit_exit_sets_the_timeout_bit_and_leaves_the_context_usable():
    import linear_attention_prefill_chunkwise_gb300 as lap
    lib = _short_limit_library()
    p = W.custom(seed=77, lengths=[300, 200, 129, 64], H=2, HV=2)  # chunkwise kernel only
    d = upload(p)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.la_prefill_fwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["slopes"].data_ptr(),
                            p.scale, d["h0"].data_ptr(), None, d["cu"].data_ptr(), d["o"].data_ptr(),
                            d["h_final"].data_ptr(), 1, p.tokens, p.N, p.H, p.HV, 128, 128, p.pool_size, 0,
                            err.data_ptr(), stream)
    assert st == 0
    torch.cuda.synchronize()  # raises if the kernel had faulted and the context were lost
    assert err.item() & lap.DEV_ERR_TIMEOUT, f"error word {err.item()}: the short limit never tripped"
    # the context and the device are intact: the normal build computes the problem correctly
    d2 = upload(p)
    run_gpu(p, d2)
    compare_full(p, d2, "after a timeout exit")
