"""The C-ABI library on the CPU: it builds for sm_103a, loads without a GPU,
exports every entry point the header declares, and rejects bad arguments on
the host with the documented status before touching any device state."""
import ctypes
import os
import re

import pytest

import linear_attention_prefill_chunkwise_gb300 as lap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]

LA_OK, LA_INVALID, LA_UNSUPPORTED, LA_CUDA = 0, 1, 2, 3


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(", text, re.M):
            names.append(m.group(1))
    return names


def test_header_declares_entry_points():
    names = declared_functions()
    assert "la_prefill_fwd" in names
    assert set(lap.EXPORTED_SYMBOLS) <= set(names)


def test_library_loads_and_exports_every_declared_symbol():
    lib = lap.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    assert lib.la_prefill_smem_bytes() <= 227 * 1024
    assert lib.la_status_string(LA_UNSUPPORTED) == b"LA_ERR_UNSUPPORTED"


FAKE = 0x10000  # never dereferenced: every call below is rejected on the host
# distinct fake buffers, 2^40 bytes apart, so that the check that outputs share no memory with
# inputs or with each other passes unless a case sets two of them to overlap
(Q, K, VV, SL, H0, O, HF, IDX, CU, ERR, WS, DOUT, DQ, DK, DV, DH0, DHF, KB, VB, ACC, ST) = (
    FAKE + (i + 1) * (1 << 40) for i in range(21))


def call(**over):
    args = dict(q=Q, k=K, v=VV, slopes=SL, scale=1.0, h0=None, idx=None, cu=None, o=O, hf=None,
                B=2, T=128, N=2, H=2, HV=2, D=128, V=128, P=0, sched=0, err=None, stream=None)
    args.update(over)
    a = args
    return lap.la_prefill_fwd_raw(a["q"], a["k"], a["v"], a["slopes"], ctypes.c_float(a["scale"]), a["h0"], a["idx"],
                                  a["cu"], a["o"], a["hf"], a["B"], a["T"], a["N"], a["H"], a["HV"], a["D"], a["V"],
                                  a["P"], a["sched"], a["err"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(D=64), LA_UNSUPPORTED),                # D != V
    (dict(V=256), LA_UNSUPPORTED),
    (dict(D=256, V=256), LA_UNSUPPORTED),
    (dict(D=32, V=32), LA_UNSUPPORTED),
    (dict(D=64, V=64, N=3), LA_INVALID),         # D = V = 64 passes the shape check
    # size limits: token rows (TMA coordinates) and units must stay within int32
    (dict(B=1, T=2**31 - 64, N=1), LA_UNSUPPORTED),
    (dict(B=2**16, T=2**15, N=2**16), LA_UNSUPPORTED),
    (dict(cu=FAKE, B=1, T=1000, N=2**30, HV=4, H=4), LA_UNSUPPORTED),
    (dict(B=2**20, T=1, N=2**20, H=2**12, HV=2**12), LA_UNSUPPORTED),  # N * HV units
    (dict(H=3, HV=4), LA_UNSUPPORTED),
    (dict(H=0), LA_INVALID),
    (dict(N=-1), LA_INVALID),
    (dict(N=3), LA_INVALID),                     # fixed mode needs N == B
    (dict(cu=FAKE, B=2), LA_INVALID),            # packed mode needs B == 1
    (dict(q=FAKE + 2), LA_INVALID),              # misaligned
    (dict(h0=FAKE + 8), LA_INVALID),
    (dict(slopes=None), LA_INVALID),
    (dict(o=None), LA_INVALID),
    (dict(sched=7), LA_INVALID),
    (dict(h0=FAKE, P=1), LA_INVALID),            # pool smaller than N without indices
    (dict(h0=FAKE, idx=FAKE, P=0), LA_INVALID),  # empty pool with indices
])
def test_host_validation(over, status):
    assert call(**over) == status
    assert lap.load_library().la_last_error() != b""


# B=2, T=128, H=HV=2, D=128: q, k, v and o are 128 KiB each, a state slot 128 KiB (2 heads)
@pytest.mark.parametrize("over", [
    dict(o=Q),                                   # o is q
    dict(o=VV + 128 * 1024 - 16),                # o starts inside v's last 16 bytes
    dict(o=K - 128 * 1024 + 16),                 # o ends inside k
    dict(o=SL - 64),                             # o covers slopes
    dict(hf=VV + 4096, P=2),                     # h_final inside v
    dict(h0=H0, hf=H0 + 65536, P=2),             # h_final overlaps h0 without being h0
    dict(hf=O + 1024, P=2),                      # the two outputs overlap
    dict(err=O + 16),                            # dev_error inside o
    dict(cu=O + 32, B=1, T=256, N=2),            # cu_seqlens inside o
    dict(idx=HF + 16, hf=HF, P=4),               # state_indices inside h_final
])
def test_outputs_may_not_overlap_inputs(over):
    assert call(**over) == LA_INVALID
    assert b"overlaps" in lap.load_library().la_last_error()


def test_in_place_pool_is_not_an_overlap():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # h_final == h0 (an in-place pool) passes every host check; without a device the call then
    # fails on the device query, not on the overlap check
    assert call(h0=H0, hf=H0, P=2) == LA_CUDA
    assert call(h0=H0, hf=H0, idx=IDX, P=8) == LA_CUDA


def test_empty_batch_is_a_no_op():
    assert call(N=0, B=0) == LA_OK
    assert call(cu=FAKE, B=1, T=0, N=1) == LA_OK  # no tokens and no state requested


def test_no_device_is_reported_not_hidden():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call() == LA_CUDA
    assert b"cuda" in lap.load_library().la_last_error().lower() or b"device" in lap.load_library().la_last_error()


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "linear_attention_prefill_chunkwise_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"


def call_decode(fn="la_decode_mtp", **over):
    a = dict(q=Q, k=K, v=VV, slopes=SL, scale=1.0, state=ST, idx=None, o=O, kbuf=None, vbuf=None,
             acc=ACC, B=2, T=8, H=2, HV=2, D=128, V=128, P=2, err=None, stream=None)
    a.update(over)
    lib = lap.load_library()
    ints = (a["B"], a["T"], a["H"], a["HV"], a["D"], a["V"], a["P"])
    if fn == "la_decode_mtp":
        return lib.la_decode_mtp(a["q"], a["k"], a["v"], a["slopes"], ctypes.c_float(a["scale"]), a["state"], a["idx"],
                                 a["o"], *ints, a["err"], a["stream"])
    if fn == "la_verify":
        return lib.la_verify(a["q"], a["k"], a["v"], a["slopes"], ctypes.c_float(a["scale"]), a["state"], a["idx"],
                             a["o"], a["kbuf"], a["vbuf"], *ints, a["err"], a["stream"])
    return lib.la_commit(a["state"], a["idx"], a["kbuf"], a["vbuf"], a["acc"], a["slopes"], *ints, a["err"],
                         a["stream"])


@pytest.mark.parametrize("fn,over,status", [
    ("la_decode_mtp", dict(D=64), LA_UNSUPPORTED),        # D != V
    ("la_decode_mtp", dict(D=32, V=32), LA_UNSUPPORTED),
    ("la_decode_mtp", dict(D=512, V=512), LA_UNSUPPORTED),
    ("la_decode_mtp", dict(D=64, V=64, P=1), LA_INVALID),  # D = V = 64 passes the shape check
    ("la_decode_mtp", dict(D=256, V=256, P=1), LA_INVALID),  # and D = V = 256
    ("la_commit", dict(D=64, V=64, kbuf=FAKE, vbuf=FAKE, acc=None), LA_INVALID),
    ("la_decode_mtp", dict(H=3, HV=4), LA_UNSUPPORTED),
    ("la_decode_mtp", dict(T=0), LA_INVALID),
    ("la_decode_mtp", dict(B=-1), LA_INVALID),
    ("la_decode_mtp", dict(P=1), LA_INVALID),             # pool smaller than B without indices
    ("la_decode_mtp", dict(idx=FAKE, P=0), LA_INVALID),   # empty pool with indices
    ("la_decode_mtp", dict(state=None), LA_INVALID),
    ("la_decode_mtp", dict(o=FAKE + 4), LA_INVALID),      # misaligned
    ("la_verify", dict(kbuf=FAKE), LA_INVALID),           # kbuf without vbuf
    ("la_verify", dict(V=64), LA_UNSUPPORTED),
    ("la_commit", dict(kbuf=FAKE, vbuf=FAKE, acc=None), LA_INVALID),
    ("la_commit", dict(kbuf=None, vbuf=FAKE), LA_INVALID),
    ("la_commit", dict(kbuf=FAKE, vbuf=FAKE, acc=FAKE + 2), LA_INVALID),
])
def test_decode_host_validation(fn, over, status):
    assert call_decode(fn, **over) == status
    assert lap.load_library().la_last_error() != b""


# B=2, T=8, H=HV=2: q, k, v and o are 8 KiB each, a pool slot 128 KiB, a KV-buffer slot 8 KiB
@pytest.mark.parametrize("fn,over", [
    ("la_decode_mtp", dict(o=VV)),               # o is v
    ("la_decode_mtp", dict(state=Q + 4096)),     # the pool overlaps q
    ("la_decode_mtp", dict(o=ST + 16)),          # o inside the pool
    ("la_decode_mtp", dict(err=ST + 16)),        # dev_error inside the pool
    ("la_verify", dict(kbuf=K, vbuf=VB)),        # the KV buffer is the draft k itself
    ("la_verify", dict(kbuf=KB, vbuf=KB + 1024)),  # the two KV buffers overlap
    ("la_verify", dict(kbuf=KB, vbuf=VB, o=ST - 16)),  # o ends inside the pool (read here)
    ("la_commit", dict(kbuf=ST, vbuf=VB)),       # the pool overlaps the KV buffer it reads
    ("la_commit", dict(kbuf=KB, vbuf=VB, acc=ST + 64)),
])
def test_decode_outputs_may_not_overlap_inputs(fn, over):
    assert call_decode(fn, **over) == LA_INVALID
    assert b"overlaps" in lap.load_library().la_last_error()


def test_decode_empty_batch_is_a_no_op():
    for fn in ("la_decode_mtp", "la_verify", "la_commit"):
        assert call_decode(fn, B=0, kbuf=FAKE, vbuf=FAKE) == LA_OK


def test_decode_no_device_is_reported():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_decode("la_decode_mtp") == LA_CUDA


# ---- segmented prefill (include/la_segment.h)

def _ws_bytes(nseg, HV, N):
    a = lambda x: (x + 255) // 256 * 256
    return a(nseg * HV * 128 * 128 * 4) + a((nseg + 1) * 4) + 2 * a(nseg * 4) + a((N + 1) * 4) + a(N * 4)


@pytest.mark.parametrize("B,T,N,HV,packed,S,nseg", [
    (2, 1000, 2, 4, 0, 192, 12),      # fixed: B * ceil(T / S)
    (1, 5000, 7, 2, 1, 128, 46),      # packed: N + floor(tokens / S)
    (3, 64 * 9, 3, 1, 0, 64, 27),
])
def test_segmented_workspace_size(B, T, N, HV, packed, S, nseg):
    nbytes, seg = lap.la_prefill_segmented_workspace(B, T, N, HV, packed, S)
    assert seg == S
    assert nbytes == _ws_bytes(nseg, HV, N)


def test_segmented_workspace_none_when_every_sequence_fits_one_segment():
    assert lap.la_prefill_segmented_workspace(2, 1000, 2, 4, 0, 1024) == (0, 0)
    assert lap.la_prefill_segmented_workspace(1, 1000, 3, 4, 1, 1024) == (0, 0)
    assert lap.la_prefill_segmented_workspace(0, 0, 0, 4, 0, 64) == (0, 0)


@pytest.mark.parametrize("seg", [100, -64, 32])
def test_segmented_workspace_rejects_bad_segment_len(seg):
    with pytest.raises(lap.LaError) as e:
        lap.la_prefill_segmented_workspace(2, 1000, 2, 4, 0, seg)
    assert e.value.status == LA_INVALID


def call_segmented(**over):
    a = dict(q=Q, k=K, v=VV, slopes=SL, scale=1.0, h0=None, idx=None, cu=None, o=O, hf=None,
             B=2, T=1000, N=2, H=2, HV=2, D=128, V=128, P=0, seg=128, ws=WS, wsb=1 << 30, err=None, stream=None)
    a.update(over)
    lib = lap.load_library()
    return lib.la_prefill_fwd_segmented(a["q"], a["k"], a["v"], a["slopes"], ctypes.c_float(a["scale"]), a["h0"],
                                        a["idx"], a["cu"], a["o"], a["hf"], a["B"], a["T"], a["N"], a["H"], a["HV"],
                                        a["D"], a["V"], a["P"], a["seg"], a["ws"], a["wsb"], a["err"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(D=64), LA_UNSUPPORTED),
    (dict(D=32, V=32), LA_UNSUPPORTED),
    (dict(D=64, V=64, wsb=1024), LA_INVALID),  # D = V = 64 passes the shape check
    (dict(H=3, HV=4), LA_UNSUPPORTED),
    (dict(N=3), LA_INVALID),
    (dict(seg=100), LA_INVALID),        # not a multiple of 64
    (dict(ws=None), LA_INVALID),        # workspace needed
    (dict(wsb=1024), LA_INVALID),       # workspace too small
    (dict(ws=FAKE + 16), LA_INVALID),   # workspace not 256-byte aligned
    (dict(q=FAKE + 2), LA_INVALID),
])
def test_segmented_host_validation(over, status):
    assert call_segmented(**over) == status
    assert lap.load_library().la_last_error() != b""


def test_segmented_workspace_may_not_overlap_the_buffers():
    assert call_segmented(ws=O - 256) == LA_INVALID     # the workspace runs into o
    assert call_segmented(o=Q) == LA_INVALID
    assert b"overlaps" in lap.load_library().la_last_error()


def test_segmented_empty_batch_is_a_no_op():
    assert call_segmented(N=0, B=0, T=0) == LA_OK


def test_segmented_no_device_is_reported():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_segmented() == LA_CUDA          # workspace fine: the first device query fails
    assert call_segmented(seg=0) == LA_CUDA     # automatic length needs the device


def call_backward(**over):
    a = dict(q=Q, k=K, v=VV, slopes=SL, scale=1.0, h0=None, dout=DOUT, dhf=None, idx=None, cu=None,
             dq=DQ, dk=DK, dv=DV, dh0=None, B=2, T=128, N=2, H=2, HV=2, D=128, V=128, P=0, ws=WS,
             wsb=1 << 39, err=None, stream=None)
    a.update(over)
    lib = lap.load_library()
    return lib.la_prefill_bwd(a["q"], a["k"], a["v"], a["slopes"], ctypes.c_float(a["scale"]), a["h0"], a["dout"],
                              a["dhf"], a["idx"], a["cu"], a["dq"], a["dk"], a["dv"], a["dh0"], a["B"], a["T"],
                              a["N"], a["H"], a["HV"], a["D"], a["V"], a["P"], a["ws"], a["wsb"], a["err"],
                              a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(H=2, HV=3), LA_UNSUPPORTED),           # HV must be a multiple of H
    (dict(D=64), LA_UNSUPPORTED),                # D != V
    (dict(D=256, V=256), LA_UNSUPPORTED),
    (dict(dout=None), LA_INVALID),
    (dict(dk=FAKE + 2), LA_INVALID),             # misaligned
    (dict(dhf=FAKE, scale=0.0, h0=FAKE, P=2), LA_INVALID),  # dh_final needs scale != 0
    (dict(wsb=1024, h0=FAKE, P=2), LA_INVALID),  # workspace too small (it holds h0 transposed)
    (dict(ws=FAKE + 16), LA_INVALID),            # workspace not 256-byte aligned
    (dict(N=3), LA_INVALID),
])
def test_backward_host_validation(over, status):
    assert call_backward(**over) == status
    assert lap.load_library().la_last_error() != b""


@pytest.mark.parametrize("over", [
    dict(dq=DK),                                 # two gradients in one buffer
    dict(dv=DOUT),                               # dv written over dout
    dict(dk=K),                                  # dk written over k
    dict(ws=DQ - 1024, h0=H0, P=2),              # the workspace (h0 transposed) runs into dq
    dict(dh0=H0, h0=H0, P=2),                    # dh0 written over h0 (read until the end)
    dict(err=DV + 4),
])
def test_backward_outputs_may_not_overlap_inputs(over):
    assert call_backward(**over) == LA_INVALID
    assert b"overlaps" in lap.load_library().la_last_error()


def test_backward_empty_batch_is_a_no_op():
    assert call_backward(N=0, B=0) == LA_OK


def test_backward_workspace_size():
    # a transposed h0 and two forms of dh_final, P x HV states of D x D FP32 each; with HV > H one
    # [tokens, HV, D] FP32 buffer more for the value heads' parts of dq and dk
    nbytes = lap.la_prefill_bwd_workspace(2, 8192, 64, 64, 128, 2, True, True)
    assert nbytes == 3 * 2 * 64 * 128 * 128 * 4
    assert lap.la_prefill_bwd_workspace(2, 8192, 64, 64, 128, 2, True, False) == 2 * 64 * 128 * 128 * 4
    assert lap.la_prefill_bwd_workspace(1, 100, 2, 2, 64, 3, False, True) == 2 * 3 * 2 * 64 * 64 * 4
    assert lap.la_prefill_bwd_workspace(1, 100, 2, 2, 64, 0, False, False) == 0
    align = lambda x: (x + 255) // 256 * 256
    assert lap.la_prefill_bwd_workspace(4, 1000, 16, 64, 128, 4, True, False) == \
        align(4 * 64 * 128 * 128 * 4) + align(4000 * 64 * 128 * 4)
    with pytest.raises(lap.LaError):
        lap.la_prefill_bwd_workspace(1, 100, 3, 4, 64, 0, False, False)  # HV not a multiple of H


def test_backward_without_states_needs_no_workspace():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # past every host check (no workspace needed without h0 and dh_final): the device query fails
    assert call_backward(ws=None, wsb=0) == LA_CUDA


# ---- D = 256 prefill (include/la_d256.h)

def call_d256(**over):
    a = dict(q=Q, k=K, v=VV, slopes=SL, scale=1.0, h0=None, idx=None, cu=None, o=O, hf=None,
             B=2, T=128, N=2, H=2, HV=2, D=256, V=256, P=0, ws=WS, wsb=1 << 30, err=None, stream=None)
    a.update(over)
    lib = lap.load_library()
    return lib.la_prefill_fwd_d256(a["q"], a["k"], a["v"], a["slopes"], ctypes.c_float(a["scale"]), a["h0"], a["idx"],
                                   a["cu"], a["o"], a["hf"], a["B"], a["T"], a["N"], a["H"], a["HV"], a["D"],
                                   a["V"], a["P"], a["ws"], a["wsb"], a["err"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(D=128, V=128), LA_UNSUPPORTED),    # the D = 128 entry point is la_prefill_fwd
    (dict(V=128), LA_UNSUPPORTED),
    (dict(D=64, V=64), LA_UNSUPPORTED),
    (dict(H=3, HV=4), LA_UNSUPPORTED),
    (dict(N=3), LA_INVALID),                 # fixed length needs N == B
    (dict(ws=None), LA_INVALID),
    (dict(wsb=1024), LA_INVALID),            # workspace too small
    (dict(ws=WS + 16), LA_INVALID),          # not 256-byte aligned
    (dict(q=Q + 2), LA_INVALID),             # misaligned
    (dict(h0=H0, P=1), LA_INVALID),          # pool smaller than N without indices
    (dict(o=Q), LA_INVALID),                 # the output overlaps an input
    (dict(ws=Q), LA_INVALID),                # the workspace overlaps an input
])
def test_d256_host_validation(over, status):
    assert call_d256(**over) == status
    assert lap.load_library().la_last_error() != b""


def test_d256_nothing_to_do():
    assert call_d256(N=0, B=0) == LA_OK


def test_d256_workspace_size():
    # FP32 parts: tokens x 4 HV x 128 floats; blocks: N x 4 HV x 128 x 128 floats (with a state)
    parts = 2 * 8192 * 4 * 16 * 128 * 4
    blocks = 2 * 4 * 16 * 128 * 128 * 4
    n0 = lap.la_prefill_d256_workspace(2, 8192, 2, 16, False)
    n1 = lap.la_prefill_d256_workspace(2, 8192, 2, 16, True)
    assert parts <= n0 < parts + 4096
    assert n1 - n0 >= blocks and n1 - n0 < blocks + 4096
    with pytest.raises(lap.LaError) as e:
        lap.la_prefill_d256_workspace(-1, 8, 1, 1, False)
    assert e.value.status == LA_INVALID


def call_d256_seg(**over):
    a = dict(q=Q, k=K, v=VV, slopes=SL, scale=1.0, h0=None, idx=None, cu=None, o=O, hf=None,
             B=1, T=4096, N=1, H=2, HV=2, D=256, V=256, P=0, seg=512, ws=WS, wsb=1 << 34, err=None, stream=None)
    a.update(over)
    lib = lap.load_library()
    return lib.la_prefill_fwd_d256_segmented(a["q"], a["k"], a["v"], a["slopes"], ctypes.c_float(a["scale"]), a["h0"],
                                             a["idx"], a["cu"], a["o"], a["hf"], a["B"], a["T"], a["N"], a["H"],
                                             a["HV"], a["D"], a["V"], a["P"], a["seg"], a["ws"], a["wsb"], a["err"],
                                             a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(D=128, V=128), LA_UNSUPPORTED),
    (dict(H=3, HV=4), LA_UNSUPPORTED),
    (dict(seg=100), LA_INVALID),             # not a multiple of 64
    (dict(ws=None), LA_INVALID),
    (dict(wsb=1024), LA_INVALID),
    (dict(ws=WS + 16), LA_INVALID),
    (dict(ws=Q), LA_INVALID),                # the workspace overlaps an input
])
def test_d256_segmented_host_validation(over, status):
    assert call_d256_seg(**over) == status
    assert lap.load_library().la_last_error() != b""


def test_d256_segmented_workspace_adds_the_segment_states():
    # an explicit segment length needs no device: 1 x 4096 tokens, 2 value heads, 512-token segments
    n_seg, s_seg = lap.la_prefill_d256_segmented_workspace(1, 4096, 1, 2, False, 512, True)
    n_plain = lap.la_prefill_d256_workspace(1, 4096, 1, 2, True)
    seg_bytes, s2 = lap.la_prefill_segmented_workspace(1, 4096, 1, 8, False, 512)
    assert s_seg == s2 == 512
    assert n_seg == n_plain + seg_bytes
