"""The allocation-free dynamic quantiser, through the C ABI.

fp8_quantize_fused_dynamic_noalloc exists for callers that may not allocate
device memory themselves — a host framework that hands out every byte of the
GPU from a pool planned at start-up and forbids libraries from allocating, or
a plain C caller with no allocator that must not pull in cudaMalloc and the
synchronisation that comes with it.  It keeps its scratch (barrier words and
per-CTA partial maxima) in the library's own static device memory.

Checked here: two calls in a row on the same and on different inputs give the
same bytes, amax and scales as the workspace-taking entry point (the
quantiser's results are exact, so the comparison is bit for bit, the bar the
other quantiser tests use); at 8192 x 8192, where each CTA of the persistent
grid walks several tiles and casts most of them after the grid barrier, the
same bits as the oracle; and after the grid barrier's wait has been made to
run out (a wait limit of 1 ns, FP8_ERR_TIMEOUT reported), the next call starts
clean and is bit-exact again.  The file is collected last so that a run which
stops at the first failure has run everything else already; it also passes on
its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev_bf16(h):
    return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.fixture(scope="module")
def lib():
    from scaled_linear_layers_gb300 import _lib
    return _lib.load()


def _outputs(R, C):
    f = dict(dtype=torch.float32, device="cuda")
    return (torch.empty((R, C), dtype=torch.uint8, device="cuda"),
            torch.empty((C, R), dtype=torch.uint8, device="cuda"),
            torch.empty(1, **f), torch.empty(1, **f), torch.empty(1, **f))


def test_noalloc_matches_workspace_entry_point_twice(lib):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.zeros(lib.fp8_quantize_fused_workspace_bytes() // 4, dtype=torch.int32,
                     device="cuda")
    shapes = [(1024, 768), (1024, 768), (4096, 2048)]
    for call, (R, C) in enumerate(shapes):
        x = _dev_bf16(synth.normal_with_outliers_bf16((R, C), 0.7, seed=11 + (call == 2), tensor="x"))
        q, qt, s, si, a = _outputs(R, C)
        rq, rqt, rs, rsi, ra = _outputs(R, C)
        st = lib.fp8_quantize_fused_dynamic_noalloc(_p(x), R, C, _p(s), _p(si), _p(q), _p(qt),
                                                    _p(a), stream)
        assert st == 0, lib.fp8_last_error().decode()
        st = lib.fp8_quantize_fused_dynamic(_p(x), R, C, _p(rs), _p(rsi), _p(rq), _p(rqt),
                                            _p(ra), _p(ws), stream)
        assert st == 0, lib.fp8_last_error().decode()
        assert lib.fp8_check_device_status(stream) == 0, lib.fp8_last_error().decode()
        assert torch.equal(q, rq) and torch.equal(qt, rqt), f"call {call}: bytes differ"
        assert torch.equal(a, ra) and torch.equal(s, rs) and torch.equal(si, rsi), f"call {call}"


def test_noalloc_rejects_bad_arguments_on_the_host(lib):
    bad = ctypes.c_void_p(0x1001)
    good = ctypes.c_void_p(0x2000)
    assert lib.fp8_quantize_fused_dynamic_noalloc(good, 24, 16, good, good, good, None, good,
                                                  None) == 3
    assert lib.fp8_quantize_fused_dynamic_noalloc(bad, 16, 16, good, good, good, None, good,
                                                  None) == 3
    assert lib.fp8_quantize_fused_dynamic_noalloc(good, 16, 16, good, good, None, None, good,
                                                  None) == 1


def _host_u8(t):
    return t.cpu().numpy()


def _call(lib, x, R, C, stream):
    q, qt, s, si, a = _outputs(R, C)
    st = lib.fp8_quantize_fused_dynamic_noalloc(_p(x), R, C, _p(s), _p(si), _p(q), _p(qt), _p(a),
                                                stream)
    assert st == 0, lib.fp8_last_error().decode()
    return q, qt, s, si, a


def test_noalloc_multi_tile_grid_matches_the_oracle_twice(lib):
    """8192 x 8192 = 4096 tiles of 128 x 128, several per CTA of the
    persistent grid (one CTA per SM times the resident CTAs per SM): the
    held-tile / reverse re-read path.  Two calls in a row, full bytes of q and
    qt, amax and both scales against the oracle's current scaling."""
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    R = C = 8192
    assert (R // 128) * (C // 128) > torch.cuda.get_device_properties(0).multi_processor_count * 4
    for call in range(2):
        xh = synth.normal_with_outliers_bf16((R, C), 1.0 + call, seed=21, tensor="x", step=call)
        q, qt, s, si, a = _call(lib, _dev_bf16(xh), R, C, stream)
        assert lib.fp8_check_device_status(stream) == 0, lib.fp8_last_error().decode()
        rq, rs, rsi, ra = oracle.quantize_dynamic(xh)
        assert np.array_equal(_host_u8(q), rq), f"call {call}: q differs from the oracle"
        assert np.array_equal(_host_u8(qt), rq.T), f"call {call}: qt differs from the oracle"
        assert a.item() == ra and s.item() == rs and si.item() == rsi, f"call {call}"


def test_noalloc_recovers_after_a_barrier_timeout(lib):
    """The grid barrier's bounded wait is driven into its timeout path with a
    1 ns wait limit (no fault, no hang: waiting CTAs give up at once and
    return).  fp8_check_device_status reports FP8_ERR_TIMEOUT; with the
    default limit back, the next call (which clears the barrier words itself)
    gives the workspace entry point's bits and the oracle's."""
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    R, C = 8192, 4096
    xh = synth.normal_with_outliers_bf16((R, C), 0.5, seed=23, tensor="x")
    x = _dev_bf16(xh)
    timed_out = False
    prev = lib.fp8_set_wait_limit_ns(1)
    try:
        for _ in range(5):
            _call(lib, x, R, C, stream)
            st = lib.fp8_check_device_status(stream)
            if st == 6:  # FP8_ERR_TIMEOUT
                timed_out = True
                break
            assert st == 0, lib.fp8_last_error().decode()
    finally:
        torch.cuda.synchronize()
        lib.fp8_set_wait_limit_ns(prev)
    assert timed_out, "a 1 ns limit never ran out"
    assert lib.fp8_check_device_status(stream) == 0
    q, qt, s, si, a = _call(lib, x, R, C, stream)
    ws = torch.zeros(lib.fp8_quantize_fused_workspace_bytes() // 4, dtype=torch.int32,
                     device="cuda")
    rq, rqt, rs, rsi, ra = _outputs(R, C)
    st = lib.fp8_quantize_fused_dynamic(_p(x), R, C, _p(rs), _p(rsi), _p(rq), _p(rqt), _p(ra),
                                        _p(ws), stream)
    assert st == 0, lib.fp8_last_error().decode()
    assert lib.fp8_check_device_status(stream) == 0, lib.fp8_last_error().decode()
    assert torch.equal(q, rq) and torch.equal(qt, rqt)
    assert torch.equal(a, ra) and torch.equal(s, rs) and torch.equal(si, rsi)
    oq, os_, osi, oa = oracle.quantize_dynamic(xh)
    assert np.array_equal(_host_u8(q), oq) and s.item() == os_ and a.item() == oa
