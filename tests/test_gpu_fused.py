"""GPU parity of the single-launch dynamic quantiser (amax, grid barrier, cast)
against the oracle's current-scaling quantiser and against the two-pass GPU
path, through the C ABI: bytes, amax and scales bit for bit, repeated calls
on one workspace, q-only / qt-only outputs and grids with one and with many
tiles per CTA."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_bf16, host_u8, f32, u8

import scaled_linear_layers_gb300 as fp8

pytestmark = pytest.mark.gpu


def bits(v):
    return np.float32(v).view(np.uint32)


def workspace():
    n = fp8.fp8_quantize_fused_workspace_bytes()
    return torch.zeros(n // 4, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("shape", [(16, 16), (128, 128), (144, 272), (1024, 4096), (4096, 4096),
                                   (8192, 8192)])
def test_fused_dynamic_matches_oracle(shape):
    R, C = shape
    x = synth.normal_bf16(shape, 1.0, seed=R + C, tensor="x")
    ws = workspace()
    q, qt = u8(R, C), u8(C, R)
    s, si, a = f32(), f32(), f32()
    fp8.fp8_quantize_fused_dynamic(dev_bf16(x), s, si, q, qt, a, ws)
    fp8.fp8_check_device_status()
    if R * C <= 4096 * 4096:
        ref_q, ref_s, ref_si, ref_a = oracle.quantize_dynamic(x)
        assert np.array_equal(host_u8(q), ref_q)
        assert np.array_equal(host_u8(qt), ref_q.T)
    else:  # oracle on sampled rows, with the oracle's own amax and scale
        ref_a = oracle.amax(x)
        ref_s, ref_si = oracle.scale_from_amax(ref_a)
        rows = np.random.default_rng(0).choice(R, 8, replace=False)
        rq, _ = oracle.quantize(np.ascontiguousarray(x[rows]), ref_si)
        assert np.array_equal(host_u8(q)[rows], rq)
        assert np.array_equal(host_u8(qt)[:, rows], rq.T)
    assert bits(a.item()) == bits(ref_a)
    assert bits(s.item()) == bits(ref_s) and bits(si.item()) == bits(ref_si)


def test_fused_dynamic_equals_two_pass_and_reuses_its_workspace():
    ws = workspace()
    for trial in range(4):
        R, C = [(512, 768), (4096, 1024), (16, 4096), (2048, 2048)][trial]
        x = synth.normal_with_outliers_bf16((R, C), 0.3, seed=trial, tensor="g")
        xd = dev_bf16(x)
        q1, qt1, q2, qt2 = u8(R, C), u8(C, R), u8(R, C), u8(C, R)
        s1, si1, a1, s2, si2, a2 = f32(), f32(), f32(), f32(), f32(), f32()
        fp8.fp8_quantize_fused_dynamic(xd, s1, si1, q1, qt1, a1, ws)
        fp8.fp8_quantize_transpose(xd, fp8.DYNAMIC, s2, si2, q2, qt2, amax_out=a2)
        fp8.fp8_check_device_status()
        assert torch.equal(q1, q2) and torch.equal(qt1, qt2)
        assert torch.equal(s1, s2) and torch.equal(si1, si2) and torch.equal(a1, a2)
    # the barrier words are back at "no arrivals" after every call
    assert ws[0].item() == 0


def test_fused_dynamic_single_outputs_and_zero_tensor():
    ws = workspace()
    x = synth.normal_bf16((256, 384), 2.0, seed=5, tensor="x")
    ref_q, ref_s, _, _ = oracle.quantize_dynamic(x)
    q = u8(256, 384)
    s, si, a = f32(), f32(), f32()
    fp8.fp8_quantize_fused_dynamic(dev_bf16(x), s, si, q, None, a, ws)
    assert np.array_equal(host_u8(q), ref_q) and s.item() == ref_s
    qt = u8(384, 256)
    fp8.fp8_quantize_fused_dynamic(dev_bf16(x), s, si, None, qt, a, ws)
    assert np.array_equal(host_u8(qt), ref_q.T)
    z = np.zeros((64, 64), np.uint16)
    qz = u8(64, 64)
    fp8.fp8_quantize_fused_dynamic(dev_bf16(z), s, si, qz, None, a, ws)
    _, zs, zsi, _ = oracle.quantize_dynamic(z)
    assert a.item() == 0.0 and s.item() == zs and si.item() == zsi and not host_u8(qz).any()
    fp8.fp8_check_device_status()
