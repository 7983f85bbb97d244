"""The one-launch current-scaling fprop for linears that fit one output tile
(fp8_linear_fprop_dynamic_small), through the C ABI: amaxes, scales and the
e4m3 bytes bit for bit as the oracle's current scaling, y within the stated
tolerance and the derived fp32/bf16 bound of the oracle's fp64 GEMM, and the
same bits as the three-call path it replaces (the single-launch dynamic
quantiser on x and on w, then fp8_linear_fprop).  Shapes: the first
configuration (X [64,256], W [256,256], seed 0), the tile's limits, and shapes
whose rows, columns and contraction end inside a tile or a 128-byte block."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_bf16, host_u8, f32, u8, bf16_out

import scaled_linear_layers_gb300 as fp8

pytestmark = pytest.mark.gpu

SHAPES = [(64, 256, 256), (16, 16, 16), (48, 80, 112), (128, 256, 512), (112, 240, 496),
          (128, 16, 256), (16, 256, 32)]


def f32bits(v):
    return np.float32(v).view(np.uint32)


def check_gemm(got, ref, k):
    _, ref_b, bound = ref
    ok = oracle.gemm_tolerance_ok(got, ref_b, bound)
    assert ok.all(), f"{(~ok).sum()} outside the stated tolerance"
    ok = oracle.gemm_derived_ok(got, ref_b, bound, k)
    assert ok.all(), f"{(~ok).sum()} outside the derived bound"


def three_call_path(x, w, M, N, K, bias=None):
    n = fp8.fp8_quantize_fused_workspace_bytes() // 4
    ws = torch.zeros(2 * n, dtype=torch.int32, device="cuda")
    sx, six, ax, sw, siw, aw = (f32() for _ in range(6))
    xq, wq = u8(M, K), u8(N, K)
    fp8.fp8_quantize_fused_dynamic(x, sx, six, xq, None, ax, ws[:n])
    fp8.fp8_quantize_fused_dynamic(w, sw, siw, wq, None, aw, ws[n:])
    y = bf16_out(M, N)
    fp8.fp8_linear_fprop(xq, sx, wq, sw, M, N, K, fp8.DYNAMIC, bias, y)
    return y, xq, wq


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("with_bias", [False, True])
def test_small_fprop_matches_oracle_and_three_call_path(shape, with_bias):
    M, N, K = shape
    if shape == (64, 256, 256):  # the first configuration, as the pages' workload
        c = synth.CONFIG1
        xh = synth.normal_bf16((M, K), c["x_sigma"], c["seed"], "x")
        wh = synth.normal_bf16((N, K), c["w_sigma"], c["seed"], "w")
    else:
        xh = synth.normal_with_outliers_bf16((M, K), 1.0, M + K, "x")
        wh = synth.normal_bf16((N, K), 0.02, N + K, "w")
    bh = synth.normal_bf16((N,), 0.1, 3, "bias") if with_bias else None
    x, w = dev_bf16(xh), dev_bf16(wh)
    b = dev_bf16(bh) if with_bias else None
    scales, amax = f32(4), f32(2)
    xq, wq = u8(M, K), u8(N, K)
    y = bf16_out(M, N)
    fp8.fp8_linear_fprop_dynamic_small(x, w, scales, y, bias=b, amax=amax, xq=xq, wq=wq)
    fp8.fp8_check_device_status()
    rxq, rsx, rsix, rax = oracle.quantize_dynamic(xh)
    rwq, rsw, rsiw, raw = oracle.quantize_dynamic(wh)
    sc, am = scales.cpu().numpy(), amax.cpu().numpy()
    assert [f32bits(v) for v in sc] == [f32bits(v) for v in (rsx, rsix, rsw, rsiw)]
    assert [f32bits(v) for v in am] == [f32bits(rax), f32bits(raw)]
    assert np.array_equal(host_u8(xq), rxq) and np.array_equal(host_u8(wq), rwq)
    check_gemm(y.float().cpu().numpy(), oracle.gemm(rxq, rwq, rsx, rsw, bh), K)
    y3, xq3, wq3 = three_call_path(x, w, M, N, K, b)
    fp8.fp8_check_device_status()
    assert torch.equal(xq3, xq) and torch.equal(wq3, wq)
    assert torch.equal(y3, y), "the one-launch fprop differs from the three-call path"


def test_small_fprop_optional_outputs_and_repeat():
    """Without amax, xq and wq the result is the same; two calls in a row on
    new inputs leave nothing behind."""
    M, N, K = 64, 256, 256
    for t in range(2):
        xh = synth.normal_bf16((M, K), 1.0 + t, 5, "x", t)
        wh = synth.normal_bf16((N, K), 0.02, 5, "w", t)
        scales, y = f32(4), bf16_out(M, N)
        fp8.fp8_linear_fprop_dynamic_small(dev_bf16(xh), dev_bf16(wh), scales, y)
        fp8.fp8_check_device_status()
        rxq, rsx, _, _ = oracle.quantize_dynamic(xh)
        rwq, rsw, _, _ = oracle.quantize_dynamic(wh)
        check_gemm(y.float().cpu().numpy(), oracle.gemm(rxq, rwq, rsx, rsw), K)


def test_small_fprop_zero_input_uses_the_clamped_scale():
    M, N, K = 32, 64, 128
    xh = np.zeros((M, K), np.uint16)
    wh = synth.normal_bf16((N, K), 0.02, 6, "w")
    scales, y = f32(4), bf16_out(M, N)
    fp8.fp8_linear_fprop_dynamic_small(dev_bf16(xh), dev_bf16(wh), scales, y)
    fp8.fp8_check_device_status()
    rs, rsi = oracle.scale_from_amax(np.float32(0.0))
    sc = scales.cpu().numpy()
    assert f32bits(sc[0]) == f32bits(rs) and f32bits(sc[1]) == f32bits(rsi)
    assert not (y.float() != 0).any().item()
