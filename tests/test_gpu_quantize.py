"""GPU parity of the HBM-bound kernels against the oracle, through the C ABI:
amax, tensorwise quantise (delayed and dynamic), fused quantise+transpose,
1x128 / 128x1 / 128x128 block quantisation and token padding.  Every byte,
amax and scale must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_bf16, host_bf16, host_u8, f32, u8, first_diff

pytestmark = pytest.mark.gpu

import scaled_linear_layers_gb300 as fp8  # noqa: E402  (built by conftest)


def amax_bits(v):
    return np.float32(v).view(np.uint32)


def _all_bf16_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


@pytest.mark.parametrize("n", [0, 1, 7, 8, 15, 16, 17, 1000, 65536 + 3, 1 << 22])
def test_amax_exact(n):
    x = synth.normal_bf16((n,), 1.0, seed=n, tensor="x")
    a = f32()
    fp8.fp8_amax(dev_bf16(x), a)
    assert amax_bits(a.item()) == amax_bits(oracle.amax(x))


def test_amax_special_values():
    x = synth.normal_bf16((4096,), 1.0, seed=1, tensor="x")
    x[77] = 0xFF80  # -inf
    a = f32()
    fp8.fp8_amax(dev_bf16(x), a)
    assert a.item() == np.inf
    x[1234] = 0x7FC1  # a NaN
    fp8.fp8_amax(dev_bf16(x), a)
    assert amax_bits(a.item()) == amax_bits(oracle.amax(x))


@pytest.mark.parametrize("scale_inv", [1.0, 448.0 / 3.7, 3.3e-3, 1e10, 2.0 ** -20, 7.25])
def test_quantize_every_bf16_pattern(scale_inv):
    """The cast over all 65536 bf16 inputs (NaN, inf, -0, subnormals
    included) times several scales: every byte equals the oracle's."""
    x = _all_bf16_patterns()
    si = torch.tensor([scale_inv], dtype=torch.float32, device="cuda")
    q = u8(x.size)
    a = f32()
    fp8.fp8_quantize(dev_bf16(x), fp8.DELAYED, None, si, q, a)
    ref, ref_amax = oracle.quantize(x, np.float32(scale_inv))
    got = host_u8(q)
    assert np.array_equal(got, ref), first_diff(got, ref)
    assert amax_bits(a.item()) == amax_bits(ref_amax)


@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (64, 256), (77, 1000), (4096, 4096)])
@pytest.mark.parametrize("recipe", ["delayed", "dynamic"])
def test_quantize_tensorwise(shape, recipe):
    x = synth.normal_bf16(shape, 1.0, seed=sum(shape), tensor="x")
    xd = dev_bf16(x)
    q = u8(*shape)
    s, si, a = f32(), f32(), f32()
    if recipe == "delayed":
        si_val = np.float32(448.0) / np.float32(2.5)
        si.fill_(float(si_val))
        fp8.fp8_quantize(xd, fp8.DELAYED, None, si, q, a)
        ref_q, ref_a = oracle.quantize(x, si_val)
    else:
        fp8.fp8_quantize(xd, fp8.DYNAMIC, s, si, q, a)
        ref_q, ref_s, ref_si, ref_a = oracle.quantize_dynamic(x)
        assert amax_bits(s.item()) == amax_bits(ref_s)
        assert amax_bits(si.item()) == amax_bits(ref_si)
    got = host_u8(q)
    assert np.array_equal(got, ref_q), first_diff(got, ref_q)
    assert amax_bits(a.item()) == amax_bits(ref_a)


def test_quantize_dynamic_zero_tensor():
    x = np.zeros((32, 32), np.uint16)
    q = u8(32, 32)
    s, si, a = f32(), f32(), f32()
    fp8.fp8_quantize(dev_bf16(x), fp8.DYNAMIC, s, si, q, a)
    ref_q, ref_s, ref_si, _ = oracle.quantize_dynamic(x)
    assert a.item() == 0.0 and s.item() == ref_s and si.item() == ref_si
    assert not host_u8(q).any()


@pytest.mark.parametrize("shape", [(16, 16), (128, 128), (144, 272), (272, 144), (1024, 4096),
                                   (4096, 4096)])
@pytest.mark.parametrize("recipe", ["delayed", "dynamic"])
def test_quantize_transpose_tensorwise(shape, recipe):
    R, C = shape
    x = synth.normal_bf16(shape, 0.02 if recipe == "delayed" else 1.0, seed=R + 3 * C, tensor="w")
    xd = dev_bf16(x)
    q, qt = u8(R, C), u8(C, R)
    s, si, a = f32(), f32(), f32()
    if recipe == "delayed":
        si_val = np.float32(448.0) / np.float32(0.0937)
        si.fill_(float(si_val))
        fp8.fp8_quantize_transpose(xd, fp8.DELAYED, None, si, q, qt, amax_out=a)
        ref_q, ref_a = oracle.quantize(x, si_val)
    else:
        fp8.fp8_quantize_transpose(xd, fp8.DYNAMIC, s, si, q, qt, amax_out=a)
        ref_q, ref_s, ref_si, ref_a = oracle.quantize_dynamic(x)
        assert s.item() == ref_s and si.item() == ref_si
    got, got_t = host_u8(q), host_u8(qt)
    assert np.array_equal(got, ref_q), first_diff(got, ref_q)
    ref_t = oracle.transpose_u8(ref_q)
    assert np.array_equal(got_t, ref_t), first_diff(got_t, ref_t)
    assert amax_bits(a.item()) == amax_bits(ref_a)


def test_quantize_transpose_without_q():
    x = synth.normal_bf16((64, 48), 1.0, seed=9, tensor="x")
    qt = u8(48, 64)
    si = torch.full((1,), 3.0, dtype=torch.float32, device="cuda")
    fp8.fp8_quantize_transpose(dev_bf16(x), fp8.DELAYED, None, si, None, qt)
    ref_q, _ = oracle.quantize(x, np.float32(3.0))
    assert np.array_equal(host_u8(qt), ref_q.T)


@pytest.mark.parametrize("shape", [(16, 16), (144, 272), (1024, 4096), (3872, 4096)])
@pytest.mark.parametrize("recipe", ["delayed", "dynamic"])
def test_quantize_transpose_dbias(shape, recipe):
    """G's cast+transpose with the bias gradient (column sums of G) fused in:
    bytes, amax and scales as the plain cast+transpose; dbias within the
    fp32-summation bound of the oracle's exact sums; zero pad rows appended
    to G change no bit of dbias."""
    R, C = shape
    g = synth.normal_with_outliers_bf16(shape, 1e-3, seed=R + C, tensor="g")
    q, qt, s, si, a = u8(R, C), u8(C, R), f32(), f32(), f32()
    db = torch.empty(C, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(fp8.fp8_dbias_workspace_bytes(R, C) // 4, dtype=torch.float32, device="cuda")
    rec = fp8.DELAYED if recipe == "delayed" else fp8.DYNAMIC
    if recipe == "delayed":
        si.fill_(float(np.float32(448.0) / np.float32(0.01)))
    fp8.fp8_quantize_transpose_dbias(dev_bf16(g), rec, s, si, q, qt, db, ws, amax_out=a)
    q2, qt2, s2, si2, a2 = u8(R, C), u8(C, R), f32(), f32(), f32()
    si2.copy_(si) if recipe == "delayed" else None
    fp8.fp8_quantize_transpose(dev_bf16(g), rec, s2, si2, q2, qt2, amax_out=a2)
    fp8.fp8_check_device_status()
    assert torch.equal(q, q2) and torch.equal(qt, qt2) and torch.equal(a, a2)
    _, ref_db, mag = oracle.bias_grad(g)
    got = host_bf16(db).astype(np.uint32) << 16
    got = got.view(np.float32).astype(np.float64)
    ok = oracle.bias_grad_tolerance_ok(got, ref_db, mag, R)
    assert ok.all(), f"{(~ok).sum()} columns outside; first {np.argwhere(~ok)[:3].ravel()}"
    # padding: zero rows append zero tile sums (or add +0 within the last tile)
    gp = oracle.pad_rows(g, 256)
    Rp = gp.shape[0]
    dbp = torch.empty(C, dtype=torch.bfloat16, device="cuda")
    wsp = torch.empty(fp8.fp8_dbias_workspace_bytes(Rp, C) // 4, dtype=torch.float32,
                      device="cuda")
    fp8.fp8_quantize_transpose_dbias(dev_bf16(gp), rec, f32(), si.clone(), u8(Rp, C), u8(C, Rp),
                                     dbp, wsp, amax_out=f32())
    assert torch.equal(db, dbp)


def test_quantize_transpose_dbias_empty_rows():
    db = torch.full((32,), 1.0, dtype=torch.bfloat16, device="cuda")
    si = torch.ones(1, device="cuda")
    fp8.fp8_quantize_transpose_dbias(torch.empty((0, 32), dtype=torch.bfloat16, device="cuda"),
                                     fp8.DELAYED, None, si, None, u8(32, 0), db, None)
    assert not db.float().any()


# 78003 tiles: more than one pass of the persistent grid (152 SMs x 8 CTAs x
# 64 tiles) and a last group of 8 tiles that is only partly filled
@pytest.mark.parametrize("shape", [(1, 128), (5, 384), (256, 1024), (333, 4096), (26001, 384)])
def test_quantize_rowtiles(shape):
    R, C = shape
    x = synth.normal_with_outliers_bf16(shape, 1.0, seed=R, tensor="x")
    q = u8(R, C)
    s, si, a = f32(R, C // 128), f32(R, C // 128), f32()
    fp8.fp8_quantize(dev_bf16(x), fp8.BLOCK, s, si, q, a)
    ref_q, ref_s, ref_si = oracle.quantize_rowtiles(x, 128)
    assert np.array_equal(host_u8(q), ref_q), first_diff(host_u8(q), ref_q)
    assert np.array_equal(s.cpu().numpy(), ref_s) and np.array_equal(si.cpu().numpy(), ref_si)
    assert amax_bits(a.item()) == amax_bits(oracle.amax(x))


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 256), (1024, 2048)])
def test_quantize_transpose_block_rowcol(shape):
    R, C = shape
    x = synth.normal_with_outliers_bf16(shape, 1.0, seed=C, tensor="g")
    q, qt = u8(R, C), u8(C, R)
    s, si = f32(R, C // 128), f32(R, C // 128)
    st, sit = f32(R // 128, C), f32(R // 128, C)  # block-major column-tile scales
    a = f32()
    fp8.fp8_quantize_transpose(dev_bf16(x), fp8.BLOCK, s, si, q, qt, st, sit, a)
    ref_q, ref_s, ref_si = oracle.quantize_rowtiles(x, 128)
    ref_qt, ref_st, ref_sit = oracle.quantize_coltiles_t(x, 128)
    assert np.array_equal(host_u8(q), ref_q), first_diff(host_u8(q), ref_q)
    assert np.array_equal(s.cpu().numpy(), ref_s) and np.array_equal(si.cpu().numpy(), ref_si)
    assert np.array_equal(host_u8(qt), ref_qt), first_diff(host_u8(qt), ref_qt)
    assert np.array_equal(st.cpu().numpy(), ref_st.T) and np.array_equal(sit.cpu().numpy(), ref_sit.T)
    assert amax_bits(a.item()) == amax_bits(oracle.amax(x))


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (1024, 512)])
def test_quantize_block_2d(shape):
    R, C = shape
    x = synth.normal_with_outliers_bf16(shape, 0.02, seed=R * 7, tensor="w")
    q, qt = u8(R, C), u8(C, R)
    s, si = f32(R // 128, C // 128), f32(R // 128, C // 128)
    fp8.fp8_quantize_transpose(dev_bf16(x), fp8.BLOCK_2D, s, si, q, qt)
    ref_q, ref_s, ref_si = oracle.quantize_sqtiles(x, 128)
    assert np.array_equal(host_u8(q), ref_q), first_diff(host_u8(q), ref_q)
    assert np.array_equal(host_u8(qt), ref_q.T)
    assert np.array_equal(s.cpu().numpy(), ref_s) and np.array_equal(si.cpu().numpy(), ref_si)
    q2 = u8(R, C)
    s2, si2 = f32(R // 128, C // 128), f32(R // 128, C // 128)
    fp8.fp8_quantize(dev_bf16(x), fp8.BLOCK_2D, s2, si2, q2)
    assert np.array_equal(host_u8(q2), ref_q) and np.array_equal(s2.cpu().numpy(), ref_s)


@pytest.mark.parametrize("rows,cols", [(0, 16), (1, 16), (3858, 64), (40, 7), (16, 4096)])
def test_pad_tokens(rows, cols):
    x = synth.normal_bf16((rows, cols), 1.0, seed=rows, tensor="x")
    padded = fp8.fp8_padded_rows(rows, 16)
    out = torch.full((padded, cols), 7.0, dtype=torch.bfloat16, device="cuda")
    got_rows = fp8.fp8_pad_tokens(dev_bf16(x), 16, out)
    assert got_rows == padded
    ref = oracle.pad_rows(x, 16)
    assert np.array_equal(host_bf16(out), ref)


def test_timeout_path_reports_and_leaves_the_context_usable():
    fp8.fp8_selftest_wait_timeout(2000)  # 2 ms bounded wait on a barrier nobody completes
    with pytest.raises(fp8.Fp8Error) as e:
        fp8.fp8_check_device_status()
    assert e.value.status == 6 and "selftest" in str(e.value)
    fp8.fp8_check_device_status()  # cleared
    a = f32()
    x = synth.normal_bf16((1024,), 1.0, seed=5, tensor="x")
    fp8.fp8_amax(dev_bf16(x), a)
    assert a.item() == oracle.amax(x)


def test_injected_launch_failure_is_reported_and_recovers():
    """Host-side fault injection: a failing launch surfaces as FP8_ERR_CUDA
    with the entry point's name; the next call runs normally."""
    from scaled_linear_layers_gb300 import _lib
    lib = _lib.load()
    x = synth.normal_bf16((4096,), 1.0, seed=6, tensor="x")
    a = f32()
    assert lib.fp8_inject_launch_failures(1) == 0
    with pytest.raises(fp8.Fp8Error) as e:
        fp8.fp8_amax(dev_bf16(x), a)
    assert e.value.status == 5 and "fp8_amax" in str(e.value)
    fp8.fp8_amax(dev_bf16(x), a)
    fp8.fp8_check_device_status()
    assert a.item() == oracle.amax(x)
    assert lib.fp8_inject_launch_failures(-1) == 2


def test_multi_amax_scales_many_tensors():
    """One pass over many weights (more than one launch's 64), sizes with
    ragged tails, an empty tensor and special values: every amax and scale
    bit for bit as the oracle's per-tensor amax and scale rule."""
    shapes = [(4096, 4096), (3, 7), (0, 16), (1, 8), (65536 + 3,), (1024, 1000)] + \
        [(17 * (i + 1), 9) for i in range(66)]
    hs = []
    for i, sh in enumerate(shapes):
        h = synth.normal_with_outliers_bf16(sh, 0.02 * (1 + i % 5), seed=i, tensor="w")
        hs.append(h)
    hs[1] = hs[1].copy()
    hs[1].ravel()[5] = 0xFF80  # -inf
    ds = [dev_bf16(h) for h in hs]
    n = len(ds)
    amax, s, si = (torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3))
    fp8.fp8_multi_amax_scales(ds, amax, s, si)
    fp8.fp8_check_device_status()
    a_h, s_h, si_h = amax.cpu().numpy(), s.cpu().numpy(), si.cpu().numpy()
    for i, h in enumerate(hs):
        ra = oracle.amax(h.ravel())
        rs, rsi = oracle.scale_from_amax(ra)
        assert amax_bits(a_h[i]) == amax_bits(ra), (i, a_h[i], ra)
        assert amax_bits(s_h[i]) == amax_bits(rs) and amax_bits(si_h[i]) == amax_bits(rsi), i


@pytest.mark.parametrize("shape", [(3, 5, 16, 1, 4), (2, 3858, 64, 2, 2), (16, 1, 8, 1, 4),
                                   (1, 128, 4096, 1, 1)])
def test_pad_tokens_bshd(shape):
    B, T, H, cp, tp = shape
    x = synth.normal_bf16((B, T, H), 1.0, seed=B + T, tensor="x")
    Tp = oracle.padded_seq_len(B, T, cp, tp)
    out = torch.full((B, Tp, H), 7.0, dtype=torch.bfloat16, device="cuda")
    got_tp = fp8.fp8_pad_tokens_bshd(dev_bf16(x), cp, tp, out)
    assert got_tp == Tp
    assert np.array_equal(host_bf16(out), oracle.pad_bshd(x, Tp))


def test_quantize_transpose_largest_sweep_size_sampled():
    """The sweep's largest size, 2^30 elements as [262144, 4096] (64 stacked
    copies of one seeded block plus one planted maximum far down): the amax
    bit for bit, and q / qᵀ on sampled rows against the oracle."""
    base = synth.normal_bf16((4096, 4096), 1.0, seed=30, tensor="x")
    x = np.tile(base, (64, 1))
    x[200003, 4001] = synth.f32_to_bf16_bits(np.array([-37.5], np.float32))[0]
    R, C = x.shape
    xd = dev_bf16(x)
    amax_ref = oracle.amax(x)
    assert amax_ref == np.float32(37.5)
    _, si_ref = oracle.scale_from_amax(amax_ref)
    q, qt, si, a = u8(R, C), u8(C, R), f32(), f32()
    si.fill_(float(si_ref))
    fp8.fp8_quantize_transpose(xd, fp8.DELAYED, None, si, q, qt, amax_out=a)
    fp8.fp8_check_device_status()
    assert amax_bits(a.item()) == amax_bits(amax_ref)
    rows = np.array([0, 4095, 4096, 131071, 200003, 262143])
    ref, _ = oracle.quantize(np.ascontiguousarray(x[rows]), si_ref)
    idx = torch.from_numpy(rows).cuda()
    assert np.array_equal(host_u8(q.index_select(0, idx)), ref)
    assert np.array_equal(host_u8(qt.index_select(1, idx)), ref.T)
