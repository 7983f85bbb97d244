"""Pins for the oracle's amax, scale rule, quantisation, tiling, GEMM and padding.

Each check compares the oracle with something other than itself: numpy or
torch library routines, brute force in exact integer / fraction arithmetic,
invariants that the pages fix (the amax/448 rule and the 448 maximum from the
AstrAI page "astrai/extension/fp8_state.py"; the multiple-of-16 token rule and
its printed failure from the SpecForge "Add training.fp8_linear" page) and
special cases where one recipe must reduce to another.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def _f32(h):
    return synth.bf16_bits_to_f32(h)


# ------------------------------------------------------------------ amax ---

def test_amax_matches_numpy_and_is_order_free():
    x = synth.normal_bf16((97, 131), 1.0, seed=3, tensor="x")
    ref = np.abs(_f32(x)).max()
    assert oracle.amax(x) == ref
    perm = np.random.default_rng(0).permutation(x.size)
    assert oracle.amax(x.ravel()[perm].copy()) == ref


def test_amax_special_values():
    h = synth.f32_to_bf16_bits(np.array([0.5, -3.0, 2.0], np.float32))
    assert oracle.amax(h) == 3.0
    assert oracle.amax(np.zeros(7, np.uint16)) == 0.0
    h = synth.f32_to_bf16_bits(np.array([0.5, -np.inf, 2.0], np.float32))
    assert oracle.amax(h) == np.inf
    nan = np.array([0x3F00, 0x7FC0, 0x4000], np.uint16)       # 0.5, NaN, 2.0
    assert np.isnan(oracle.amax(nan))
    assert oracle.amax(np.array([], np.uint16)) == 0.0


# ----------------------------------------------------------------- scale ---

def test_scale_rule_matches_torch_float32_division():
    """_update_delayed_scale with torch float32 tensor ops: clamp_min(1e-12),
    then the two quotients amax/448 and 448/amax, each one correctly rounded
    fp32 division (tensor / tensor).  torch's ``float / tensor`` shorthand
    computes reciprocal(amax) * 448 instead, which can be one ulp away; the
    plain quotient is the reading taken here."""
    m = GOLDEN["e4m3_max"]["value"]
    for a in [448.0, 1.0, 0.1, 3.7, 1e-3, 0.0, 1e-20, 5.0e4, 0.0998]:
        s, si = oracle.scale_from_amax(a)
        t = torch.tensor([a], dtype=torch.float32).clamp_min(GOLDEN["lag_clamp_min"]["value"])
        c = torch.full_like(t, m)
        assert s == torch.div(t, c).item()
        assert si == torch.div(c, t).item()
    s, si = oracle.scale_from_amax(448.0)
    assert s == 1.0 and si == 1.0


def test_scale_inv_is_not_reciprocal_of_scale():
    """scale_inv is 448/a computed directly; for some a it differs from
    1/scale in the last bit, so the rule is observable."""
    diffs = 0
    for a in np.linspace(0.01, 10.0, 2000, dtype=np.float32):
        s, si = oracle.scale_from_amax(a)
        if np.float32(1.0) / s != si:
            diffs += 1
            assert si == np.float32(448.0) / np.float32(a)
    assert diffs > 0


def test_current_scaling_maps_the_max_element_to_448():
    rng = np.random.default_rng(5)
    for trial in range(200):
        sigma = float(np.exp(rng.uniform(-12, 8)))
        x = synth.normal_bf16((33,), sigma, seed=trial, tensor="x")
        q, s, si, a = oracle.quantize_dynamic(x)
        big = np.argmax(np.abs(_f32(x)))
        assert q[big] & 0x7F == 0x7E
        # dequantised values stay within half an e4m3 step (2^-4 relative) of x
        table = oracle.e4m3_decode_table()
        deq = table[q] * float(s)
        xv = _f32(x).astype(np.float64)
        tol = np.maximum(np.abs(xv) * 2.0 ** -4, 2.0 ** -10 * float(s)) * (1 + 1e-6)
        assert np.all(np.abs(deq - xv) <= tol)


# -------------------------------------------------------------- quantise ---

def test_quantize_matches_torch_cast_of_the_scaled_value():
    x = synth.normal_bf16((64, 256), 1.0, seed=0, tensor="x")
    a = oracle.amax(x)
    _, si = oracle.scale_from_amax(a)
    q, amax = oracle.quantize(x, si)
    assert amax == a
    v = torch.from_numpy(_f32(x)) * torch.tensor(si, dtype=torch.float32)
    ref = v.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_quantize_saturates_beyond_the_scale():
    x = synth.f32_to_bf16_bits(np.array([1.0, -2.0, 1000.0, -1e30], np.float32))
    q, _ = oracle.quantize(x, np.float32(448.0))
    assert list(q) == [0x7E, 0xFE, 0x7E, 0xFE]


def test_transpose_u8_matches_numpy():
    q = np.random.default_rng(0).integers(0, 256, (37, 53), dtype=np.uint8)
    assert np.array_equal(oracle.transpose_u8(q), q.T)


# ---------------------------------------------------------- block tiles ---

def test_rowtiles_reduce_to_tensorwise_when_tile_amaxes_agree():
    """Put the same largest magnitude in every 1x128 tile: every tile scale
    equals the tensor scale and the bytes equal the tensorwise bytes."""
    x = synth.normal_bf16((8, 512), 1.0, seed=1, tensor="x")
    big = synth.f32_to_bf16_bits(np.array([9.5], np.float32))[0]
    x[:, ::128] = big
    q, s, si = oracle.quantize_rowtiles(x, 128)
    qd, sd, sid, _ = oracle.quantize_dynamic(x)
    assert np.all(s == sd) and np.all(si == sid)
    assert np.array_equal(q, qd)


def test_rowtile_scales_are_per_tile_amax():
    x = synth.normal_with_outliers_bf16((4, 384), 1.0, seed=2, tensor="x")
    q, s, si = oracle.quantize_rowtiles(x, 128)
    xv = _f32(x).reshape(4, 3, 128)
    for r in range(4):
        for t in range(3):
            a = np.float32(np.abs(xv[r, t]).max())
            s_ref, si_ref = oracle.scale_from_amax(a)
            assert s[r, t] == s_ref and si[r, t] == si_ref
            q_ref, _ = oracle.quantize(x[r, t * 128:(t + 1) * 128].copy(), si_ref)
            assert np.array_equal(q[r, t * 128:(t + 1) * 128], q_ref)


def test_coltiles_are_rowtiles_of_the_transpose():
    x = synth.normal_with_outliers_bf16((256, 48), 1.0, seed=4, tensor="g")
    qt, s, si = oracle.quantize_coltiles_t(x, 128)
    q2, s2, si2 = oracle.quantize_rowtiles(np.ascontiguousarray(x.T), 128)
    assert np.array_equal(qt, q2) and np.array_equal(s, s2) and np.array_equal(si, si2)


def test_sqtiles_reduce_to_tensorwise_when_tile_amaxes_agree():
    x = synth.normal_bf16((256, 384), 0.02, seed=5, tensor="w")
    big = synth.f32_to_bf16_bits(np.array([0.25], np.float32))[0]
    x[::128, ::128] = big
    q, s, si = oracle.quantize_sqtiles(x, 128)
    qd, sd, sid, _ = oracle.quantize_dynamic(x)
    assert s.shape == (2, 3) and np.all(s == sd) and np.all(si == sid)
    assert np.array_equal(q, qd)


def test_tile_scales_and_codes_worked_by_hand():
    """Closed forms chosen so that every product is exact.  e4m3 code =
    sign | exponent field (bias 7) << 3 | mantissa: 448 = 1.75 * 2^8 -> 0x7E,
    112 = 1.75 * 2^6 -> 0x6E, 64 -> 0x68, 72 -> 0x69, 80 -> 0x6A.
    Row tile 0 has amax 2.0 (scale_inv 448/2 = 224), row tile 1 amax 3.5
    (scale_inv 128); in tile 1, 0.59375 * 128 = 76 and 0.53125 * 128 = 68 are
    halfway between codes and go to the even mantissa (80 and 64)."""
    vals = np.zeros((1, 256), np.float32)
    vals[0, :128] = 0.5
    vals[0, 5] = 2.0
    vals[0, 7] = 0.30078125  # 0.3 in bf16; * 224 = 67.375 -> 64
    vals[0, 128:] = 0.59375
    vals[0, 130] = 3.5
    vals[0, 131] = 0.53125
    vals[0, 132] = -0.59375
    x = synth.f32_to_bf16_bits(vals)
    assert np.array_equal(_f32(x), vals)  # every value is exact in bf16
    q, s, si = oracle.quantize_rowtiles(x, 128)
    assert si[0, 0] == np.float32(224.0) and si[0, 1] == np.float32(128.0)
    assert s[0, 0] == np.float32(1.0 / 224.0) and s[0, 1] == np.float32(3.5 / 448.0)
    want = np.full(256, 0x6E, np.uint8)
    want[5], want[7] = 0x7E, 0x68
    want[128:] = 0x6A
    want[130], want[131], want[132] = 0x7E, 0x68, 0xEA
    assert np.array_equal(q[0], want), np.nonzero(q[0] != want)
    # the same values down a column give the same codes in the transposed copy
    qt, st, sit = oracle.quantize_coltiles_t(np.ascontiguousarray(x.T), 128)
    assert np.array_equal(qt[0], want) and np.array_equal(sit[0], si[0])  # scales [cols, rows/128]
    # one 128x128 weight tile whose largest magnitude is 1.0: scale_inv 448,
    # -0.25 * 448 = -112 -> 0xEE
    w = np.full((128, 128), -0.25, np.float32)
    w[17, 99] = 1.0
    qw, sw, siw = oracle.quantize_sqtiles(synth.f32_to_bf16_bits(w), 128)
    assert siw[0, 0] == np.float32(448.0) and sw[0, 0] == np.float32(1.0 / 448.0)
    assert qw[17, 99] == 0x7E and np.all(np.delete(qw.ravel(), 17 * 128 + 99) == 0xEE)


def test_sqtile_amax_brute_force():
    x = synth.normal_with_outliers_bf16((256, 256), 0.02, seed=6, tensor="w")
    _, s, _ = oracle.quantize_sqtiles(x, 128)
    xv = np.abs(_f32(x)).reshape(2, 128, 2, 128)
    for i in range(2):
        for j in range(2):
            assert s[i, j] == oracle.scale_from_amax(np.float32(xv[i, :, j, :].max()))[0]


# ------------------------------------------------------------------ GEMM ---

def _int_codes(rng, shape):
    """e4m3 codes whose values are the integers -16..16 (exactly representable)."""
    table = oracle.e4m3_decode_table()
    ints = {int(v): c for c, v in enumerate(table)
            if np.isfinite(v) and v == int(v) and abs(v) <= 16 and not (v == 0 and c == 0x80)}
    keys = np.array(sorted(ints))
    vals = rng.choice(keys, size=shape)
    codes = np.vectorize(lambda v: ints[int(v)])(vals).astype(np.uint8)
    return codes, vals.astype(np.int64)


def test_gemm_exact_on_integer_matrices():
    rng = np.random.default_rng(7)
    A, Ai = _int_codes(rng, (16, 32))
    B, Bi = _int_codes(rng, (16, 32))
    d, db, bound = oracle.gemm(A, B, np.float32(1.0), np.float32(1.0))
    assert np.array_equal(d, (Ai @ Bi.T).astype(np.float64))
    assert np.array_equal(bound, (np.abs(Ai) @ np.abs(Bi).T).astype(np.float64))
    # with scales: exact rational arithmetic, one fp64 rounding at the end
    sa, sb = np.float32(0.1), np.float32(3.3)
    d, db, _ = oracle.gemm(A, B, sa, sb)
    for i, j in [(0, 0), (3, 7), (15, 15)]:
        exact = Fraction(float(sa)) * Fraction(float(sb)) * int((Ai[i] * Bi[j]).sum())
        assert d[i, j] == float(exact)


def test_gemm_matches_library_matmul_and_is_transposition_consistent():
    rng = np.random.default_rng(8)
    A = rng.integers(0, 256, (24, 96), dtype=np.uint8)
    B = rng.integers(0, 256, (40, 96), dtype=np.uint8)
    A[(A & 0x7F) == 0x7F] = 0
    B[(B & 0x7F) == 0x7F] = 0
    sa, sb = np.float32(0.37), np.float32(1.9)
    d, db, bound = oracle.gemm(A, B, sa, sb)
    Ad = torch.from_numpy(A).view(torch.float8_e4m3fn).to(torch.float64)
    Bd = torch.from_numpy(B).view(torch.float8_e4m3fn).to(torch.float64)
    ref = (Ad @ Bd.T).numpy() * (float(sa) * float(sb))
    assert np.allclose(d, ref, rtol=1e-12, atol=0)
    dt, _, _ = oracle.gemm(B, A, sb, sa)
    assert np.array_equal(dt, d.T)
    # entries agree with the full product
    ii = rng.integers(0, 24, 50)
    jj = rng.integers(0, 40, 50)
    de, dbe, be = oracle.gemm_entries(A, B, sa, sb, ii, jj)
    assert np.array_equal(de, d[ii, jj]) and np.array_equal(be, bound[ii, jj])
    assert np.array_equal(dbe, db[ii, jj])
    # bf16 rounding of D equals torch's fp32->bf16 on values exact in fp32
    small = d[np.float32(d) == d]
    assert np.array_equal(db[np.float32(d) == d],
                          torch.from_numpy(small.astype(np.float32)).to(torch.bfloat16).double().numpy())


def test_gemm_bias_added_before_rounding():
    rng = np.random.default_rng(9)
    A, Ai = _int_codes(rng, (4, 32))
    B, Bi = _int_codes(rng, (8, 32))
    bias = synth.f32_to_bf16_bits(np.arange(8, dtype=np.float32) * 0.5)
    d, _, _ = oracle.gemm(A, B, np.float32(1.0), np.float32(1.0), bias)
    assert np.array_equal(d, (Ai @ Bi.T) + np.arange(8) * 0.5)


def test_gemm_tolerance_flags_a_planted_error():
    rng = np.random.default_rng(10)
    A = rng.integers(0, 0x7E, (8, 64), dtype=np.uint8)
    B = rng.integers(0, 0x7E, (8, 64), dtype=np.uint8)
    d, db, bound = oracle.gemm(A, B, np.float32(0.01), np.float32(0.02))
    assert oracle.gemm_tolerance_ok(db, db, bound).all()
    wrong = db.copy()
    wrong[3, 4] += 0.02 * bound[3, 4] + 1e-3
    assert not oracle.gemm_tolerance_ok(wrong, db, bound)[3, 4]


def test_block_gemm_brute_force_and_tensorwise_reduction():
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 256
    A, Ai = _int_codes(rng, (M, K))
    B, Bi = _int_codes(rng, (N, K))
    sa = rng.uniform(0.1, 2, (M, 2)).astype(np.float32)
    sb = rng.uniform(0.1, 2, (N, 2)).astype(np.float32)
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    d, _, _ = oracle.gemm_block_entries(A, B, sa, sb, 1, ii.ravel(), jj.ravel())
    for t, (i, j) in enumerate(zip(ii.ravel(), jj.ravel())):
        exact = sum(Fraction(float(sa[i, b])) * Fraction(float(sb[j, b]))
                    * int((Ai[i, b * 128:(b + 1) * 128] * Bi[j, b * 128:(b + 1) * 128]).sum())
                    for b in range(2))
        assert abs(d[t] - float(exact)) <= abs(float(exact)) * 2 ** -50
    # equal tile scales reduce to the tensorwise GEMM
    sa1 = np.full((M, 2), 0.25, np.float32)
    sb1 = np.full((1, 2), 0.5, np.float32)           # one 128-row weight tile row
    d1, _, _ = oracle.gemm_block_entries(A, B, sa1, sb1, 128, ii.ravel(), jj.ravel())
    dt, _, _ = oracle.gemm(A, B, np.float32(0.25), np.float32(0.5))
    assert np.array_equal(d1, dt.ravel())


# --------------------------------------------------------------- padding ---

def test_pad_rows_page_example():
    ex = GOLDEN["unaligned_token_count_example"]
    mult = GOLDEN["token_multiple"]["value"]
    rows = ex["rows"]
    assert rows % mult != 0 and str(rows) in ex["message"]
    x = synth.normal_bf16((rows, 32), 1.0, seed=0, tensor="x")
    p = oracle.pad_rows(x, mult)
    assert p.shape == (3872, 32) and p.shape[0] % mult == 0
    assert np.array_equal(p[:rows], x) and not p[rows:].any()
    # padded rows do not change amax, nor any real row of the quantised tensor
    assert oracle.amax(p) == oracle.amax(x)
    _, si = oracle.scale_from_amax(oracle.amax(x))
    qp, _ = oracle.quantize(p, si)
    q, _ = oracle.quantize(x, si)
    assert np.array_equal(qp[:rows], q) and not qp[rows:].any()


def test_padding_leaves_wgrad_and_real_rows_unchanged():
    """Zero rows add nothing: dW over padded tokens equals dW over the real
    ones, and real rows of Y are unchanged."""
    x = synth.normal_bf16((40, 64), 1.0, seed=1, tensor="x")
    g = synth.normal_bf16((40, 32), 1e-3, seed=1, tensor="g")
    w = synth.normal_bf16((32, 64), 0.02, seed=1, tensor="w")
    xp, gp = oracle.pad_rows(x, 16), oracle.pad_rows(g, 16)
    assert xp.shape[0] == 48
    _, sx, six, _ = oracle.quantize_dynamic(x)
    _, sg, sig, _ = oracle.quantize_dynamic(g)
    _, sw, siw, _ = oracle.quantize_dynamic(w)
    xq, _ = oracle.quantize(x, six)
    xpq, _ = oracle.quantize(xp, six)
    gq, _ = oracle.quantize(g, sig)
    gpq, _ = oracle.quantize(gp, sig)
    wq, _ = oracle.quantize(w, siw)
    dw, _, _ = oracle.gemm(oracle.transpose_u8(gq), oracle.transpose_u8(xq), sg, sx)
    dwp, _, _ = oracle.gemm(oracle.transpose_u8(gpq), oracle.transpose_u8(xpq), sg, sx)
    assert np.array_equal(dw, dwp)
    y, _, _ = oracle.gemm(xq, wq, sx, sw)
    yp, _, _ = oracle.gemm(xpq, wq, sx, sw)
    assert np.array_equal(yp[:40], y) and not yp[40:].any()


def test_fp8_storage_bytes_page_example():
    ex = GOLDEN["fp8_weight_storage_bytes"]
    q, _ = oracle.quantize(np.zeros((16, 16), np.uint16), np.float32(1.0))
    assert q.itemsize == ex["itemsize"]
    assert int(np.prod(ex["shape"])) * q.itemsize == ex["bytes"]


# -------------------------------------------------------------- bias grad ---
# dbias = column sums of the upstream gradient (the third output of the
# linear backward whose output mask the AstrAI page's fp8_linear_backward
# passes through).

def test_bias_grad_closed_form_on_integer_columns():
    rows, cols = 96, 40
    col_vals = np.arange(1, cols + 1, dtype=np.float32) * np.where(np.arange(cols) % 2, -1, 1)
    g = synth.f32_to_bf16_bits(np.tile(col_vals, (rows, 1)))
    d, db, mag = oracle.bias_grad(g)
    assert np.array_equal(d, rows * col_vals.astype(np.float64))
    assert np.array_equal(db, d)  # 96*k has at most 8 significant bits for k <= 40
    assert np.array_equal(mag, np.abs(d))
    # +v / -v alternating down a column cancels exactly
    alt = synth.f32_to_bf16_bits(np.outer(np.where(np.arange(rows) % 2, -1.0, 1.0),
                                          np.linspace(0.1, 7.0, cols)).astype(np.float32))
    d, db, mag = oracle.bias_grad(alt)
    assert not d.any() and not db.any() and (mag > 0).all()


def test_bias_grad_matches_library_sum_and_is_order_free():
    g = synth.normal_bf16((500, 72), 1e-3, seed=3, tensor="g")
    d, db, _ = oracle.bias_grad(g)
    ref = torch.from_numpy(_f32(g)).double().sum(0).numpy()
    assert np.array_equal(d, ref)  # exact: bf16 values sum exactly in fp64
    perm = np.random.default_rng(0).permutation(500)
    d2, db2, _ = oracle.bias_grad(np.ascontiguousarray(g[perm]))
    assert np.array_equal(d2, d) and np.array_equal(db2, db)
    assert all(db[i] == oracle.round_to_bf16(d[i]) for i in range(72))


def test_bias_grad_ignores_pad_rows_and_tolerance_catches_an_error():
    g = synth.normal_bf16((3858, 24), 1e-3, seed=4, tensor="g")
    gp = oracle.pad_rows(g, 16)
    d, db, mag = oracle.bias_grad(g)
    dp, dbp, magp = oracle.bias_grad(gp)
    assert np.array_equal(d, dp) and np.array_equal(db, dbp) and np.array_equal(mag, magp)
    assert oracle.bias_grad_tolerance_ok(db, db, mag, 3858).all()
    # a one-term error (one row's value counted twice) is far outside the bound
    bad = db + np.abs(_f32(g)[0]).astype(np.float64) * 8
    assert not oracle.bias_grad_tolerance_ok(bad, db, mag, 3858).all()


# ------------------------------------------------------ parallel padding ---

def test_pad_multiple_and_bshd_length_page_example():
    ex = GOLDEN["bshd_tp_example"]
    B, tp = ex["batch"], ex["tp_size"]
    # the review's point: B*T % (8*tp) == 0 alone lets T be a multiple of 2
    t8 = next(t for t in range(1, 64) if (B * t) % (8 * tp) == 0)
    assert t8 == ex["multiple_from_8_tp"] and t8 % tp != 0
    # our length splits over tp and gives every rank a multiple of 16 tokens
    t = oracle.padded_seq_len(B, 1, 1, tp)
    assert t % tp == 0 and (B * t // tp) % 16 == 0 and t == 4
    assert GOLDEN["thd_pad_multiple_formula"]["value"] == "8 * cp_size * tp_size"
    assert oracle.pad_multiple(1, 1) == GOLDEN["token_multiple"]["value"]
    # a packed batch padded to pad_multiple leaves each of the cp*tp ranks a
    # multiple of 16 tokens, and a smaller multiple would not for some size
    for cp in (1, 2, 4):
        for tp in (1, 2, 8):
            m = oracle.pad_multiple(cp, tp)
            assert (m // (cp * tp)) % 16 == 0 and m // 2 // (cp * tp) % 16 != 0


def test_padded_seq_len_matches_closed_form():
    from math import gcd
    for B in (1, 2, 3, 16, 24):
        for cp in (1, 2):
            for tp in (1, 2, 4):
                r = cp * tp
                step_b = 16 * r // gcd(B, 16 * r)   # B*T' % (16r) == 0  <=>  T' % step_b == 0
                L = r * step_b // gcd(r, step_b)
                for T in (0, 1, 7, 16, 100, 3858):
                    assert oracle.padded_seq_len(B, T, cp, tp) == -(-T // L) * L


def test_pad_bshd_rows():
    x = synth.normal_bf16((3, 5, 16), 1.0, seed=2, tensor="x")
    out = oracle.pad_bshd(x, 8)
    assert out.shape == (3, 8, 16)
    assert np.array_equal(out[:, :5], x) and not out[:, 5:].any()
    assert np.array_equal(oracle.pad_bshd(x, 5), x)
