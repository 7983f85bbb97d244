"""GPU parity of the tcgen05 scaled FP8 GEMMs (fprop, dgrad, wgrad) against
the oracle's fp64 GEMM, through the C ABI.

Tolerance (stated for the method): |D_gpu - bf16(D_ref)| <= 1e-2 * s_A s_B
sum_k |a_ik||b_kj| + 1e-3 elementwise.  On integer-valued operands whose
exact results are representable in bf16 the result must be exact."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_bf16, host_u8, f32, u8, bf16_out

import scaled_linear_layers_gb300 as fp8

pytestmark = pytest.mark.gpu


def to_dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def scal(v):
    return torch.tensor([float(v)], dtype=torch.float32, device="cuda")


def run_tensor_gemm(A, B, sa, sb, bias=None, which="fprop"):
    """D = sa*sb*A·Bᵀ via the given entry point, A [rows,K], B [cols,K]."""
    rows, K = A.shape
    cols = B.shape[0]
    D = bf16_out(rows, cols)
    Ad, Bd = to_dev_u8(A), to_dev_u8(B)
    if which == "fprop":      # M=rows, N=cols, K=K
        fp8.fp8_linear_fprop(Ad, scal(sa), Bd, scal(sb), rows, cols, K, fp8.DELAYED,
                             None if bias is None else dev_bf16(bias), D)
    elif which == "dgrad":    # dX[M,K'] with M=rows, K'=cols, contraction N=K
        fp8.fp8_linear_dgrad(Ad, scal(sa), Bd, scal(sb), rows, K, cols, fp8.DELAYED, D)
    else:                     # dW[N',K'] with N'=rows, K'=cols, contraction M=K
        fp8.fp8_linear_wgrad(Ad, scal(sa), Bd, scal(sb), K, rows, cols, fp8.DELAYED, D)
    return D.float().cpu().numpy()


def random_codes(rng, shape):
    c = rng.integers(0, 256, shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    return c


@pytest.mark.parametrize("which", ["fprop", "dgrad", "wgrad"])
@pytest.mark.parametrize("shape", [(16, 16, 16), (128, 256, 128), (64, 256, 256), (144, 272, 400),
                                   (256, 512, 1024), (400, 48, 2048), (1008, 528, 336)])
def test_gemm_random_codes_within_tolerance(shape, which):
    M, N, K = shape
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = random_codes(rng, (M, K))
    B = random_codes(rng, (N, K))
    sa, sb = np.float32(0.0123), np.float32(3.5e-4)
    got = run_tensor_gemm(A, B, sa, sb, which=which)
    _, ref, bound = oracle.gemm(A, B, sa, sb)
    ok = oracle.gemm_tolerance_ok(got, ref, bound)
    assert ok.all(), f"{(~ok).sum()} bad; first {np.argwhere(~ok)[:3]}"
    # much tighter in practice: fp32 accumulation of exact products
    assert np.max(np.abs(got - ref) / (bound + 1e-30)) < 1e-2


@pytest.mark.parametrize("bn", [256, 224, 192, 160, 128])
@pytest.mark.parametrize("which", ["fprop", "wgrad"])
def test_gemm_every_tile_width(bn, which, monkeypatch):
    """Each N-tile variant of the one-CTA kernel on shapes with ragged M/N/K tails."""
    monkeypatch.setenv("FP8LINEAR_GEMM_PAIR", "0")
    monkeypatch.setenv("FP8LINEAR_GEMM_BN", str(bn))
    rng = np.random.default_rng(bn)
    for M, N, K in [(400, 1008, 272), (128, 224, 128), (1152, 480, 640)]:
        A = random_codes(rng, (M, K))
        B = random_codes(rng, (N, K))
        got = run_tensor_gemm(A, B, 0.05, 0.002, which=which)
        _, ref, bound = oracle.gemm(A, B, np.float32(0.05), np.float32(0.002))
        ok = oracle.gemm_tolerance_ok(got, ref, bound)
        assert ok.all(), f"BN={bn} {(M, N, K)}: {(~ok).sum()} bad"


@pytest.mark.parametrize("bn", [256, 224, 192, 160, 128])
@pytest.mark.parametrize("which", ["fprop", "dgrad", "wgrad"])
def test_gemm_pair_kernel_every_tile_width(bn, which, monkeypatch):
    """The 2-SM (CTA pair) kernel, forced on, on shapes with ragged tails,
    including M smaller than the pair's 256 rows and a single-pair grid."""
    monkeypatch.setenv("FP8LINEAR_GEMM_PAIR", "1")
    monkeypatch.setenv("FP8LINEAR_GEMM_BN", str(bn))
    rng = np.random.default_rng(bn + 7)
    for M, N, K in [(400, 1008, 272), (128, 224, 128), (1152, 480, 640), (2048, 2048, 1024)]:
        A = random_codes(rng, (M, K))
        B = random_codes(rng, (N, K))
        got = run_tensor_gemm(A, B, 0.05, 0.002, which=which)
        _, ref, bound = oracle.gemm(A, B, np.float32(0.05), np.float32(0.002))
        ok = oracle.gemm_tolerance_ok(got, ref, bound)
        assert ok.all(), f"pair BN={bn} {(M, N, K)}: {(~ok).sum()} bad"


@pytest.mark.parametrize("n", [384, 400])
def test_gemm_pair_kernel_bias(n, monkeypatch):
    """Bias in the 2-SM kernel's epilogue; N = 400 ends in a 16-column chunk,
    whose upper half (past the bias array) is neither read nor stored."""
    monkeypatch.setenv("FP8LINEAR_GEMM_PAIR", "1")
    rng = np.random.default_rng(3)
    A = random_codes(rng, (512, 512))
    B = random_codes(rng, (n, 512))
    bias = synth.normal_bf16((n,), 1.0, seed=4, tensor="bias")
    got = run_tensor_gemm(A, B, 0.01, 0.02, bias=bias)
    _, ref, bound = oracle.gemm(A, B, np.float32(0.01), np.float32(0.02), bias)
    assert oracle.gemm_tolerance_ok(got, ref, bound).all()


def test_gemm_exact_on_integer_operands():
    """Values in -16..16 with K=256: every partial sum is an integer below
    2^16, exact in fp32, and the results fit bf16's 8 bits only when small;
    compare against the oracle's bf16 rounding of the exact value."""
    rng = np.random.default_rng(0)
    table = oracle.e4m3_decode_table()
    ints = [c for c in range(256) if np.isfinite(table[c]) and table[c] == int(table[c])
            and abs(table[c]) <= 4 and c != 0x80]
    A = rng.choice(ints, (256, 256)).astype(np.uint8)
    B = rng.choice(ints, (512, 256)).astype(np.uint8)
    got = run_tensor_gemm(A, B, 1.0, 1.0)
    _, ref, _ = oracle.gemm(A, B, np.float32(1.0), np.float32(1.0))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("n", [384, 400])
def test_gemm_bias(n, monkeypatch):
    """Bias in the one-CTA kernel's epilogue (N = 400: a last chunk of 16
    columns)."""
    monkeypatch.setenv("FP8LINEAR_GEMM_PAIR", "0")
    rng = np.random.default_rng(3)
    A = random_codes(rng, (256, 512))
    B = random_codes(rng, (n, 512))
    bias = synth.normal_bf16((n,), 1.0, seed=3, tensor="bias")
    got = run_tensor_gemm(A, B, 0.01, 0.02, bias=bias)
    _, ref, bound = oracle.gemm(A, B, np.float32(0.01), np.float32(0.02), bias)
    assert oracle.gemm_tolerance_ok(got, ref, bound).all()


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (16384, 4096, 4096)])
def test_gemm_full_size_sampled(shape, pair, monkeypatch):
    """Full-size GEMM in the benchmark's launch configuration; 4096 sampled
    entries plus 4 whole row panels against the oracle, for both kernels."""
    monkeypatch.setenv("FP8LINEAR_GEMM_PAIR", pair)
    M, N, K = shape
    rng = np.random.default_rng(M + K)
    x = synth.normal_bf16((M, K), 1.0, seed=1, tensor="x")
    w = synth.normal_bf16((N, K), 0.02, seed=1, tensor="w")
    xq, sx, _, _ = oracle.quantize_dynamic(x)
    wq, sw, _, _ = oracle.quantize_dynamic(w)
    Y = bf16_out(M, N)
    fp8.fp8_linear_fprop(to_dev_u8(xq), scal(sx), to_dev_u8(wq), scal(sw), M, N, K, fp8.DELAYED,
                         None, Y)
    got = Y.float().cpu().numpy()
    ii = rng.integers(0, M, 4096)
    jj = rng.integers(0, N, 4096)
    rows = rng.choice(M, 4, replace=False)
    ii = np.concatenate([ii, np.repeat(rows, N)])
    jj = np.concatenate([jj, np.tile(np.arange(N), 4)])
    _, ref, bound = oracle.gemm_entries(xq, wq, sx, sw, ii, jj)
    ok = oracle.gemm_tolerance_ok(got[ii, jj], ref, bound)
    assert ok.all(), f"{(~ok).sum()} bad"


def test_gemm_zero_k_tail_and_ragged_tiles():
    """M, N not multiples of the 128x256 tile and K not a multiple of 128:
    the TMA zero-fill must add nothing and the stores must stay in bounds."""
    rng = np.random.default_rng(11)
    M, N, K = 272, 304, 176
    A = random_codes(rng, (M, K))
    B = random_codes(rng, (N, K))
    D = torch.full((M + 16, N), 123.0, dtype=torch.bfloat16, device="cuda")
    fp8.fp8_linear_fprop(to_dev_u8(A), scal(1.0), to_dev_u8(B), scal(1.0), M, N, K, fp8.DELAYED,
                         None, D)
    got = D.float().cpu().numpy()
    _, ref, bound = oracle.gemm(A, B, np.float32(1.0), np.float32(1.0))
    assert oracle.gemm_tolerance_ok(got[:M], ref, bound).all()
    assert np.all(got[M:] == 123.0)  # rows past M untouched


@pytest.mark.parametrize("mode", ["auto", "pair"])
@pytest.mark.parametrize("shape", [(256, 256, 256), (384, 640, 1152), (1024, 512, 768),
                                   (2048, 4096, 1024)])
def test_dgrad_wgrad_in_one_launch(shape, mode, monkeypatch):
    """fp8_linear_dgrad_wgrad: dX = gs*ws Gq Wq and dW = gs*xs Gqᵀ Xq against
    the oracle, and bit-equal to the two single calls.  "pair" forces the
    shared 2-SM launch (with 256-row tiles: M=384 leaves half a tile of
    dgrad rows past the matrix); "auto" lets the library choose."""
    if mode == "pair":
        monkeypatch.setenv("FP8LINEAR_GEMM_PAIR", "1")
    M, N, K = shape
    rng = np.random.default_rng(M + 3 * N + 5 * K)
    G = random_codes(rng, (M, N))
    W = random_codes(rng, (N, K))
    X = random_codes(rng, (M, K))
    gs, ws, xs = np.float32(0.0031), np.float32(0.07), np.float32(0.0009)
    Gt, Wt, Xt = (np.ascontiguousarray(a.T) for a in (G, W, X))
    dx, dw = bf16_out(M, K), bf16_out(N, K)
    fp8.fp8_linear_dgrad_wgrad(to_dev_u8(G), to_dev_u8(Gt), scal(gs), to_dev_u8(Wt), scal(ws),
                               to_dev_u8(Xt), scal(xs), M, N, K, fp8.DELAYED, dx, dw)
    fp8.fp8_check_device_status()
    got_dx, got_dw = dx.float().cpu().numpy(), dw.float().cpu().numpy()
    rows = rng.choice(M, min(M, 96), replace=False)
    ii, jj = np.repeat(rows, K), np.tile(np.arange(K), len(rows))
    _, ref, bound = oracle.gemm_entries(G, Wt, gs, ws, ii, jj)
    assert oracle.gemm_tolerance_ok(got_dx[ii, jj], ref, bound).all()
    rows = rng.choice(N, min(N, 96), replace=False)
    ii, jj = np.repeat(rows, K), np.tile(np.arange(K), len(rows))
    _, ref, bound = oracle.gemm_entries(Gt, Xt, gs, xs, ii, jj)
    assert oracle.gemm_tolerance_ok(got_dw[ii, jj], ref, bound).all()
    # the single entry points (same kernel family) give the same bits
    got1 = run_tensor_gemm(G, Wt, gs, ws, which="dgrad")
    got2 = run_tensor_gemm(Gt, Xt, gs, xs, which="wgrad")
    assert np.array_equal(got1, got_dx) and np.array_equal(got2, got_dw)


def test_dgrad_wgrad_rejects_block_recipe():
    z = torch.zeros(128 * 128, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    out = bf16_out(128, 128)
    with pytest.raises(fp8.Fp8Error, match="FP8_ERR_UNSUPPORTED"):
        fp8.fp8_linear_dgrad_wgrad(z, z, s, z, s, z, s, 128, 128, 128, fp8.BLOCK, out, out)
