"""The Python binding's own checks (CPU): it marshals arguments only, so every malformed call
must be refused before the C library is reached, with a plain Python error."""
import pytest

torch = pytest.importorskip("torch")

import linear_attention_prefill_chunkwise_gb300 as lap  # noqa: E402


def cpu_problem(tokens=64, H=2, HV=2):
    q = torch.zeros((tokens, H, 128), dtype=torch.bfloat16)
    k = torch.zeros_like(q)
    v = torch.zeros((tokens, HV, 128), dtype=torch.bfloat16)
    slopes = torch.zeros(HV, dtype=torch.float32)
    return q, k, v, slopes


@pytest.mark.parametrize("fn", [lap.la_prefill_fwd, lap.la_prefill_fwd_segmented, lap.la_prefill_fwd_segmented_static])
def test_host_tensors_are_refused(fn):
    q, k, v, slopes = cpu_problem()
    with pytest.raises(ValueError, match="CUDA tensor"):
        fn(q, k, v, slopes, 1.0, seq_len=64)


@pytest.mark.parametrize("fn", [lap.la_prefill_fwd, lap.la_prefill_fwd_segmented])
def test_wrong_dtype_and_rank_are_refused(fn):
    q, k, v, slopes = cpu_problem()
    with pytest.raises(TypeError, match="bfloat16"):
        fn(q.float(), k, v, slopes, 1.0, seq_len=64)
    with pytest.raises(ValueError, match="3 dims"):
        fn(q[0], k, v, slopes, 1.0, seq_len=64)
    with pytest.raises(TypeError, match="must be a torch.Tensor"):
        fn([0], k, v, slopes, 1.0, seq_len=64)


def test_exported_symbols_are_declared_and_bound():
    lib = lap.load_library()
    for name in lap.EXPORTED_SYMBOLS:
        assert hasattr(lib, name)
    assert "la_prefill_fwd_segmented_static" in lap.__all__
