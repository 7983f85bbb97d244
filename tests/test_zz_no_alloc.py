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
other quantiser tests use).  The file is collected last so that a run which
stops at the first failure has run everything else already; it also passes on
its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

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
