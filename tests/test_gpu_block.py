"""GPU parity of the block-scaled FP8 GEMMs (1x128 activation/gradient tiles,
128x128 weight tiles; the TE "recipe=block" of the NeMo SALMAutomodel page)
against the oracle's per-block fp64 GEMM, through the C ABI.  Operands and
scales come from the oracle's block quantisers, so only the GEMM is tested
here (the quantisers have their own bit-exact tests)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_out

import scaled_linear_layers_gb300 as fp8

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


KERNELS = ["one_cta", "cta_pair", "one_cta_n256", "cta_pair_n256", "one_cta_n256_s",
           "cta_pair_n256_s"]


def use_kernel(mp, name):
    mp.setenv("FP8LINEAR_BLOCK_PAIR", "1" if "pair" in name else "0")
    mp.setenv("FP8LINEAR_BLOCK_BN", "256" if "n256" in name else "128")
    mp.setenv("FP8LINEAR_BLOCK_ACC", "1" if name.endswith("_s") else "0")


@pytest.fixture(params=KERNELS)
def kernel(request, monkeypatch):
    """Runs a test on the one-CTA kernel and on the CTA-pair kernel (256-row
    pair tiles; with M a multiple of 128 but not of 256 the last pair's peer
    rows lie past the matrix), each with 128- and 256-column tiles (with N a
    multiple of 128 but not of 256 the last tile's right half lies past the
    matrix), and the 256-column tiles with packed or scalar fp32 accumulators
    ("_s")."""
    use_kernel(monkeypatch, request.param)
    return request.param


def check(got, ref, bound, k=None):
    """The stated tolerance, and the derived fp32/bf16 bound when the
    contraction length k is given."""
    ok = oracle.gemm_tolerance_ok(got, ref, bound)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance; first {np.argwhere(~ok)[:3]}"
    if k is not None:
        ok = oracle.gemm_derived_ok(got, ref, bound, k)
        assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the derived bound (k={k})"


SHAPES = [(128, 128, 128), (256, 384, 512), (384, 256, 1024), (1024, 512, 768),
          (640, 1152, 384)]


def operands(M, N, K, seed):
    x = synth.normal_with_outliers_bf16((M, K), 1.0, seed, "x")
    w = synth.normal_with_outliers_bf16((N, K), 1.0, seed, "w")
    g = synth.normal_with_outliers_bf16((M, N), 1.0, seed, "g")
    return x, w, g


def all_entries(R, C):
    ii, jj = np.meshgrid(np.arange(R), np.arange(C), indexing="ij")
    return ii.ravel(), jj.ravel()


@pytest.mark.parametrize("shape", SHAPES)
def test_block_fprop(shape, kernel):
    M, N, K = shape
    x, w, _ = operands(M, N, K, 1)
    xq, xs, _ = oracle.quantize_rowtiles(x, 128)
    wq, ws, _ = oracle.quantize_sqtiles(w, 128)
    y = bf16_out(M, N)
    fp8.fp8_linear_fprop(dev(xq), dev(xs), dev(wq), dev(ws), M, N, K, fp8.BLOCK, None, y)
    ii, jj = all_entries(M, N)
    _, ref, bound = oracle.gemm_block_entries(xq, wq, xs, ws, 128, ii, jj)
    check(y.float().cpu().numpy().ravel(), ref, bound, K)


@pytest.mark.parametrize("shape", SHAPES)
def test_block_dgrad(shape, kernel):
    M, N, K = shape
    _, w, g = operands(M, N, K, 2)
    gq, gs, _ = oracle.quantize_rowtiles(g, 128)
    wq, ws, _ = oracle.quantize_sqtiles(w, 128)
    wqt = oracle.transpose_u8(wq)
    dx = bf16_out(M, K)
    fp8.fp8_linear_dgrad(dev(gq), dev(gs), dev(wqt), dev(ws), M, N, K, fp8.BLOCK, dx)
    ii, jj = all_entries(M, K)
    # B = Wqᵀ [K, N]: its 128x128 tile grid is the transpose of W's
    _, ref, bound = oracle.gemm_block_entries(gq, wqt, gs, np.ascontiguousarray(ws.T), 128, ii, jj)
    check(dx.float().cpu().numpy().ravel(), ref, bound, N)


@pytest.mark.parametrize("shape", SHAPES)
def test_block_wgrad(shape, kernel):
    M, N, K = shape
    x, _, g = operands(M, N, K, 3)
    gqt, gst, _ = oracle.quantize_coltiles_t(g, 128)   # [N, M], scales [N, M/128]
    xqt, xst, _ = oracle.quantize_coltiles_t(x, 128)   # [K, M], scales [K, M/128]
    dw = bf16_out(N, K)
    # the library takes column-tile scales block-major: [M/128, N] and [M/128, K]
    fp8.fp8_linear_wgrad(dev(gqt), dev(np.ascontiguousarray(gst.T)), dev(xqt),
                         dev(np.ascontiguousarray(xst.T)), M, N, K, fp8.BLOCK, dw)
    ii, jj = all_entries(N, K)
    _, ref, bound = oracle.gemm_block_entries(gqt, xqt, gst, xst, 1, ii, jj)
    check(dw.float().cpu().numpy().ravel(), ref, bound, M)


def test_block_equal_scales_match_tensorwise_gemm(kernel):
    """With every tile scale equal, the block GEMM reduces to the tensorwise
    one: both kernels must agree within the tolerance (and the oracle's two
    GEMMs agree exactly, pinned on the CPU)."""
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(4)
    A = rng.integers(0, 0x7E, (M, K), dtype=np.uint8)
    B = rng.integers(0, 0x7E, (N, K), dtype=np.uint8)
    sa = np.full((M, K // 128), 0.03, np.float32)
    sb = np.full((N // 128, K // 128), 0.5, np.float32)
    y_blk = bf16_out(M, N)
    fp8.fp8_linear_fprop(dev(A), dev(sa), dev(B), dev(sb), M, N, K, fp8.BLOCK, None, y_blk)
    y_t = bf16_out(M, N)
    fp8.fp8_linear_fprop(dev(A), dev(sa[:1, :1].ravel()), dev(B), dev(sb[:1, :1].ravel()), M, N, K,
                         fp8.DELAYED, None, y_t)
    _, ref, bound = oracle.gemm(A, B, np.float32(0.03), np.float32(0.5))
    check(y_blk.float().cpu().numpy(), ref, bound)
    check(y_t.float().cpu().numpy(), ref, bound)


def test_block_full_size_sampled(kernel):
    """The block workload's fprop shape (M=32768, K=N=8192) on sampled rows."""
    M, N, K = 32768, 8192, 8192
    rng = np.random.default_rng(5)
    A = rng.integers(0, 0x7E, (M, K), dtype=np.uint8) | (rng.integers(0, 2, (M, K), dtype=np.uint8) << 7)
    B = rng.integers(0, 0x7E, (N, K), dtype=np.uint8)
    sa = rng.uniform(1e-3, 1e-1, (M, K // 128)).astype(np.float32)
    sb = rng.uniform(1e-3, 1e-1, (N // 128, K // 128)).astype(np.float32)
    y = bf16_out(M, N)
    fp8.fp8_linear_fprop(dev(A), dev(sa), dev(B), dev(sb), M, N, K, fp8.BLOCK, None, y)
    rows = rng.choice(M, 2, replace=False)
    ii = np.concatenate([rng.integers(0, M, 2048), np.repeat(rows, N)])
    jj = np.concatenate([rng.integers(0, N, 2048), np.tile(np.arange(N), 2)])
    _, ref, bound = oracle.gemm_block_entries(A, B, sa, sb, 128, ii, jj)
    check(y.float().cpu().numpy()[ii, jj], ref, bound, K)


def _random_block_operands(rng, R, C):
    q = rng.integers(0, 0x7E, (R, C), dtype=np.uint8) | (rng.integers(0, 2, (R, C), dtype=np.uint8) << 7)
    return q


def test_block_wgrad_full_size_sampled(kernel):
    """The block workload's wgrad shape: dW [8192, 8192] over M = 32768 tokens,
    both operands with per-row scales of every 128-token block, on sampled
    entries and two full rows."""
    M, N, K = 32768, 8192, 8192
    rng = np.random.default_rng(6)
    A = _random_block_operands(rng, N, M)           # Gqᵀ [N, M]
    B = _random_block_operands(rng, K, M)           # Xqᵀ [K, M]
    sa = rng.uniform(1e-3, 1e-1, (M // 128, N)).astype(np.float32)   # block-major
    sb = rng.uniform(1e-3, 1e-1, (M // 128, K)).astype(np.float32)
    dw = bf16_out(N, K)
    fp8.fp8_linear_wgrad(dev(A), dev(sa), dev(B), dev(sb), M, N, K, fp8.BLOCK, dw)
    rows = rng.choice(N, 2, replace=False)
    ii = np.concatenate([rng.integers(0, N, 2048), np.repeat(rows, K)])
    jj = np.concatenate([rng.integers(0, K, 2048), np.tile(np.arange(K), 2)])
    _, ref, bound = oracle.gemm_block_entries(A, B, np.ascontiguousarray(sa.T),
                                              np.ascontiguousarray(sb.T), 1, ii, jj)
    check(dw.float().cpu().numpy()[ii, jj], ref, bound, M)


@pytest.mark.parametrize("which", ["fprop", "wgrad"])
def test_block_kernels_give_identical_bits(which, monkeypatch):
    """Every kernel variant computes the same fp32 operations in the same
    order (per 128-deep block: the partial, times its scale product, added to
    the running sum), so their outputs agree bit for bit."""
    M, N, K = 640, 1152, 768
    rng = np.random.default_rng(7)
    if which == "fprop":
        A, B = _random_block_operands(rng, M, K), _random_block_operands(rng, N, K)
        sa = rng.uniform(1e-3, 1e-1, (M, K // 128)).astype(np.float32)
        sb = rng.uniform(1e-3, 1e-1, (N // 128, K // 128)).astype(np.float32)
        out_shape = (M, N)
    else:
        A, B = _random_block_operands(rng, N, M), _random_block_operands(rng, K, M)
        sa = rng.uniform(1e-3, 1e-1, (M // 128, N)).astype(np.float32)
        sb = rng.uniform(1e-3, 1e-1, (M // 128, K)).astype(np.float32)
        out_shape = (N, K)
    outs = {}
    for name in KERNELS:
        use_kernel(monkeypatch, name)
        o = bf16_out(*out_shape)
        if which == "fprop":
            fp8.fp8_linear_fprop(dev(A), dev(sa), dev(B), dev(sb), M, N, K, fp8.BLOCK, None, o)
        else:
            fp8.fp8_linear_wgrad(dev(A), dev(sa), dev(B), dev(sb), M, N, K, fp8.BLOCK, o)
        fp8.fp8_check_device_status()
        outs[name] = o
    first = outs[KERNELS[0]]
    for name, o in outs.items():
        assert torch.equal(o, first), f"{name} differs from {KERNELS[0]}"
