"""Head dimension D = V = 64 through the same C ABI, against the FP64 oracle.

The chunkwise kernel's D = 64 instance uses the D = 128 tile and tensor-memory layout with
the second 64-wide box of every head row unused: Q, K and V load one box per row, the score
and O_inter contractions run over K = 64, dS has N = 64, and the state is the top-left 64 x 64
block of the 128 x 128 register and TMEM layout.  Short sequences take the tokenwise kernel's
D = 64 instance (one CTA per (sequence, value head), 8 columns of each state row per thread),
as at D = 128.  The segmented path at D = 64 is tested with the D = 128 cases in
test_gpu_segment.py.  The oracle computes in FP64 at any D.
"""
import zlib

import numpy as np
import pytest

import workloads as W
from harness import compare_every_unit, compare_full, run_gpu, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

D64_CASES = {
    "fixed_T300": dict(B=2, T=300, H=2, HV=2),
    "fixed_T64": dict(B=3, T=64, H=1, HV=2),
    "ragged_pool_in_place_gva": dict(lengths=[1, 63, 64, 65, 130, 0, 200, 31], H=2, HV=4, pool=11,
                                     indices=[3, 10, -1, 0, 7, 5, 1, 9], in_place=True),
    "no_h0": dict(lengths=[70, 3, 129], H=2, HV=2, with_h0=False),
    "no_final": dict(lengths=[70, 3], H=2, HV=2, want_final=False),
    "lambda_one": dict(lengths=[150, 20], H=1, HV=2, slopes=[0.0, 0.0]),
    "lambda_zero": dict(lengths=[150, 20], H=1, HV=2, slopes=[100.0, 100.0]),
    "long_nine_chunks": dict(lengths=[64 * 9 + 17], H=1, HV=1),
    "short_sequences": dict(lengths=[5, 20, 3, 31, 1, 40], H=2, HV=2),
    "short_fixed_T32_tokenwise": dict(B=3, T=32, H=2, HV=4),
    "short_fixed_T1_tokenwise": dict(B=5, T=1, H=1, HV=1),
    "short_pool_in_place_tokenwise": dict(lengths=[9, 32, 0, 17, 33, 2], H=1, HV=3, pool=9,
                                          indices=[4, 0, 8, -1, 2, 6], in_place=True),
    "short_no_h0_tokenwise": dict(B=2, T=24, H=1, HV=2, with_h0=False),
    "many_sequences": dict(lengths=[(37 * i) % 211 for i in range(300)], H=1, HV=2),
}


@pytest.mark.parametrize("name", sorted(D64_CASES))
def test_d64_cases_full(name):
    p = W.custom(seed=zlib.crc32(("d64" + name).encode()) % 10000, name=name, D=64, **D64_CASES[name])
    d = upload(p)
    run_gpu(p, d)
    compare_full(p, d, f"D=64 {name}")


def test_d64_fixed_b2_t8192_h64_every_unit():
    p = W.custom(seed=3002, B=2, T=8192, H=64, HV=64, D=64, name="D=64 B=2 T=8192 H=64")
    d = upload(p)
    run_gpu(p, d)
    compare_every_unit(p, d, p.name)


def test_d64_packed_varlen_every_unit():
    rng = np.random.default_rng(3003)
    lengths = rng.integers(1, 4097, 32)
    p = W.custom(seed=3003, lengths=lengths, H=32, HV=32, D=64, pool=64,
                 indices=rng.permutation(64)[:32], in_place=True, name="D=64 packed N=32 H=32")
    d = upload(p)
    run_gpu(p, d)
    compare_every_unit(p, d, p.name)


def test_d64_persistent_equals_non_persistent_bitwise():
    p = W.custom(seed=3004, lengths=[1, 63, 64, 65, 130, 0, 200, 17, 64 * 5], H=2, HV=4, pool=12,
                 indices=[3, 11, -1, 0, 7, 5, 1, 2, 9], D=64)
    outs = []
    for sched in ("persistent", "non_persistent"):
        d = upload(p)
        run_gpu(p, d, schedule=sched)
        torch.cuda.synchronize()
        outs.append((d["o"].view(torch.int16).cpu().numpy(), d["h_final"].view(torch.int32).cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


def _run_path(path, p, d):
    import linear_attention_prefill_chunkwise_gb300 as lap
    if path == "prefill":
        run_gpu(p, d)
    else:
        lap.la_prefill_fwd_segmented(d["q"], d["k"], d["v"], d["slopes"], p.scale, h0=d["h0"], cu_seqlens=d["cu"],
                                     o=d["o"], h_final=d["h_final"], segment_len=64)
    torch.cuda.synchronize()


@pytest.mark.parametrize("path", ["prefill", "segmented"])
def test_d64_nonfinite_sequence_does_not_reach_its_neighbours(path):
    lengths = [100, 77, 150, 64, 40]
    p = W.custom(seed=3005, lengths=lengths, H=2, HV=2, D=64)
    a, b = int(p.cu_seqlens[2]), int(p.cu_seqlens[3])
    p.k_bits[a:b] = 0x7F80
    p.v_bits[a:b] = 0x7FC0
    d = upload(p)
    _run_path(path, p, d)
    o_all = d["o"].view(torch.int16).cpu().numpy()
    for n in (0, 1, 3, 4):
        s, e = int(p.cu_seqlens[n]), int(p.cu_seqlens[n + 1])
        pa = W.Problem("alone", p.q_bits[s:e].copy(), p.k_bits[s:e].copy(), p.v_bits[s:e].copy(), p.slopes,
                       p.scale, p.H, p.HV, 1, e - s, np.array([0, e - s], dtype=np.int32), None,
                       p.h0[n:n + 1].copy(), D=64, V=64)
        da = upload(pa)
        _run_path(path, pa, da)
        assert np.array_equal(o_all[s:e], da["o"].view(torch.int16).cpu().numpy()), f"{path}: sequence {n}"
        assert np.array_equal(d["h_final"][n].view(torch.int32).cpu().numpy(),
                              da["h_final"][0].view(torch.int32).cpu().numpy()), f"{path}: sequence {n} state"
