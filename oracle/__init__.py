"""CPU oracle for the FP8 scaled linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (``scaled_linear_layers_gb300``) never imports it and shares no code with
it: the two meet only through the seeded input generators in ``synth``.

The arithmetic lives in ``fp8_oracle.c`` (plain single-threaded C, built with
gcc and ``-ffp-contract=off`` so every fp32 multiply and divide is one IEEE
operation).  This module is a thin numpy wrapper around it plus the scaling
state machine in ``state.py``.

Source of every rule: the AstrAI page "astrai/extension/fp8_state.py": its
E4M3 maximum of 448, its comment on the GEMM layout (D = A_SCALE * B_SCALE *
A * B, so a tensor's scale is amax/448 and quantising multiplies by the
inverse), its weight-meta and global-state classes and its delayed-scale
update.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compile fp8_oracle.c into liboracle.so next to it (gcc, -O2, no FP
    contraction, no fast-math).  Returns the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        F = ctypes.c_float
        sig = {
            "orc_bf16_to_f32": (F, [ctypes.c_uint16]),
            "orc_round_to_bf16": (ctypes.c_double, [ctypes.c_double]),
            "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [F]),
            "orc_amax_bf16": (F, [P, I]),
            "orc_scale_from_amax": (None, [F, P, P]),
            "orc_quantize": (F, [P, I, F, P]),
            "orc_transpose_u8": (None, [P, I, I, P]),
            "orc_quantize_rowtiles": (None, [P, I, I, I, P, P, P]),
            "orc_quantize_coltiles_t": (None, [P, I, I, I, P, P, P]),
            "orc_quantize_sqtiles": (None, [P, I, I, I, P, P, P]),
            "orc_gemm_entries": (None, [P, P, I, F, F, P, P, P, I, P, P, P]),
            "orc_gemm": (None, [P, P, I, I, I, F, F, P, P, P, P]),
            "orc_gemm_block_entries": (None, [P, P, I, I, P, P, I, P, P, I, P, P, P]),
            "orc_pad_rows": (I, [P, I, I, I, P]),
            "orc_bias_grad": (None, [P, I, I, P, P, P]),
            "orc_pad_bshd": (None, [P, I, I, I, I, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "bf16 tensors are passed as uint16 bit patterns"
    return x


# ------------------------------------------------------------------ codec ---

def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (vectorised through the C scalar)."""
    h = _bf16(h)
    lib = _load()
    return np.array([lib.orc_bf16_to_f32(int(v)) for v in h.ravel()],
                    dtype=np.float32).reshape(h.shape)


def round_to_bf16(x: float) -> float:
    return _load().orc_round_to_bf16(float(x))


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    """fp64 value of every one of the 256 codes (NaN for 0x7F and 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v: float) -> int:
    """Saturating round-to-nearest-even encode of one binary32 value."""
    return int(_load().orc_e4m3_encode(float(np.float32(v))))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    return np.array([lib.orc_e4m3_encode(float(t)) for t in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


# ------------------------------------------------------- amax and scales ---

def amax(x: np.ndarray) -> np.float32:
    x = _bf16(x)
    return np.float32(_load().orc_amax_bf16(_p(x), x.size))


def scale_from_amax(a) -> tuple[np.float32, np.float32]:
    """(scale, scale_inv) = (a/448, 448/a) with a = max(amax, 1e-12): the
    _update_delayed_scale rule, also used for current (dynamic) scaling."""
    s = np.zeros(1, np.float32)
    si = np.zeros(1, np.float32)
    _load().orc_scale_from_amax(float(np.float32(a)), _p(s), _p(si))
    return s[0], si[0]


# ------------------------------------------------------------- quantise ---

def quantize(x: np.ndarray, scale_inv) -> tuple[np.ndarray, np.float32]:
    """q = e4m3(fl32(x * scale_inv)) elementwise; also returns amax(x)."""
    x = _bf16(x)
    q = np.empty(x.shape, np.uint8)
    a = _load().orc_quantize(_p(x), x.size, float(np.float32(scale_inv)), _p(q))
    return q, np.float32(a)


def quantize_dynamic(x: np.ndarray):
    """Current (dynamic tensorwise) scaling: the scale comes from this
    tensor's own amax.  Returns (q, scale, scale_inv, amax)."""
    a = amax(x)
    s, si = scale_from_amax(a)
    q, _ = quantize(x, si)
    return q, s, si, a


def transpose_u8(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows, cols = q.shape
    qt = np.empty((cols, rows), np.uint8)
    _load().orc_transpose_u8(_p(q), rows, cols, _p(qt))
    return qt


def quantize_rowtiles(x: np.ndarray, tile: int = 128):
    """1 x tile scaling along the last dim.  Returns (q, scale, scale_inv)
    with scales [rows, cols/tile]."""
    x = _bf16(x)
    rows, cols = x.shape
    assert cols % tile == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // tile), np.float32)
    si = np.empty_like(s)
    _load().orc_quantize_rowtiles(_p(x), rows, cols, tile, _p(q), _p(s), _p(si))
    return q, s, si


def quantize_coltiles_t(x: np.ndarray, tile: int = 128):
    """tile x 1 scaling down the columns, written transposed.  Returns
    (qt [cols, rows], scale [cols, rows/tile], scale_inv)."""
    x = _bf16(x)
    rows, cols = x.shape
    assert rows % tile == 0
    qt = np.empty((cols, rows), np.uint8)
    s = np.empty((cols, rows // tile), np.float32)
    si = np.empty_like(s)
    _load().orc_quantize_coltiles_t(_p(x), rows, cols, tile, _p(qt), _p(s), _p(si))
    return qt, s, si


def quantize_sqtiles(x: np.ndarray, tile: int = 128):
    """tile x tile scaling (weights).  Returns (q, scale [rows/tile, cols/tile], scale_inv)."""
    x = _bf16(x)
    rows, cols = x.shape
    assert rows % tile == 0 and cols % tile == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // tile, cols // tile), np.float32)
    si = np.empty_like(s)
    _load().orc_quantize_sqtiles(_p(x), rows, cols, tile, _p(q), _p(s), _p(si))
    return q, s, si


# ----------------------------------------------------------------- GEMM ---

def gemm(A: np.ndarray, B: np.ndarray, s_a, s_b, bias=None):
    """D = s_a*s_b*dec(A)·dec(B)ᵀ (+bias) in fp64 for A [M,K], B [N,K] e4m3
    codes.  Returns (D, D rounded to bf16, bound) with bound =
    s_a*s_b*Σ_k|dec a||dec b|, all [M,N] fp64."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    d = np.empty((M, N), np.float64)
    db = np.empty_like(d)
    bd = np.empty_like(d)
    bias_p = None if bias is None else _p(_bf16(bias))
    _load().orc_gemm(_p(A), _p(B), M, N, K, float(np.float32(s_a)), float(np.float32(s_b)),
                     bias_p, _p(d), _p(db), _p(bd))
    return d, db, bd


def gemm_entries(A, B, s_a, s_b, ii, jj, bias=None):
    """As gemm() but only for the entries (ii[t], jj[t])."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    K = A.shape[1]
    assert B.shape[1] == K
    ii = np.ascontiguousarray(ii, np.int64)
    jj = np.ascontiguousarray(jj, np.int64)
    n = ii.size
    d = np.empty(n, np.float64)
    db = np.empty_like(d)
    bd = np.empty_like(d)
    bias_p = None if bias is None else _p(_bf16(bias))
    _load().orc_gemm_entries(_p(A), _p(B), K, float(np.float32(s_a)), float(np.float32(s_b)),
                             bias_p, _p(ii), _p(jj), n, _p(d), _p(db), _p(bd))
    return d, db, bd


def gemm_block_entries(A, B, sa, sb, b_rows, ii, jj, kb: int = 128):
    """Block-scaled D entries: sa [M, K/kb], sb [N/b_rows, K/kb]."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    K = A.shape[1]
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    assert sa.shape[1] == K // kb and sb.shape[1] == K // kb
    ii = np.ascontiguousarray(ii, np.int64)
    jj = np.ascontiguousarray(jj, np.int64)
    n = ii.size
    d = np.empty(n, np.float64)
    db = np.empty_like(d)
    bd = np.empty_like(d)
    _load().orc_gemm_block_entries(_p(A), _p(B), K, kb, _p(sa), _p(sb), b_rows,
                                   _p(ii), _p(jj), n, _p(d), _p(db), _p(bd))
    return d, db, bd


# -------------------------------------------------------------- padding ---

def pad_rows(x: np.ndarray, multiple: int = 16) -> np.ndarray:
    """Append zero rows up to the next multiple of ``multiple``."""
    x = _bf16(x)
    rows, cols = x.shape
    padded = (rows + multiple - 1) // multiple * multiple
    out = np.empty((padded, cols), np.uint16)
    got = _load().orc_pad_rows(_p(x), rows, cols, multiple, _p(out))
    assert got == padded
    return out


def pad_multiple(cp_size: int, tp_size: int) -> int:
    """Token multiple of a packed (THD) batch under context and tensor
    parallelism.  The FP8 GEMMs need every rank's token count to be a
    multiple of 16 (SpecForge page, Conclusion); with the tokens split over
    cp * tp ranks (the NeMo page "Add FP8 support for SALMAutomodel" review:
    the local linear sees M = B*T/tp, which is why its THD helper pads to
    8 * cp * tp for TE's 8) that is 16 * cp * tp of the whole batch."""
    return 16 * cp_size * tp_size


def padded_seq_len(batch: int, seq: int, cp_size: int = 1, tp_size: int = 1) -> int:
    """BSHD padding (same review): the smallest T' >= seq such that the
    sequence dim splits evenly over the cp * tp ranks (T' % (cp*tp) == 0) and
    every rank's token count batch * T' / (cp*tp) is a multiple of 16; found
    by search."""
    r = cp_size * tp_size
    t = seq
    while t % r or (batch * t) % (16 * r):
        t += 1
    return t


def pad_bshd(x: np.ndarray, seq_out: int) -> np.ndarray:
    """[B, T, H] bf16 -> [B, seq_out, H] with zero rows at each sequence's end."""
    x = np.ascontiguousarray(x, np.uint16)
    B, T, H = x.shape
    out = np.empty((B, seq_out, H), np.uint16)
    _load().orc_pad_bshd(_p(x), B, T, H, seq_out, _p(out))
    return out


def bias_grad(g: np.ndarray):
    """Column sums of the bf16 matrix g [rows, cols] (the bias gradient of a
    linear), exact in fp64: returns (exact sums, their bf16 roundings, column
    sums of |g|)."""
    g = _bf16(g)
    rows, cols = g.shape
    d, db, mag = (np.empty(cols, np.float64) for _ in range(3))
    _load().orc_bias_grad(_p(g), rows, cols, _p(d), _p(db), _p(mag))
    return d, db, mag


def bias_grad_tolerance_ok(got: np.ndarray, ref_bf16: np.ndarray, mag: np.ndarray, rows: int):
    """A GPU bias gradient summed in fp32 in a fixed order and rounded once to
    bf16 passes if |got - bf16(ref)| <= 2^-7 (1 + 2^-7) |ref| + (17 +
    ceil(rows/128)) * 2^-23 * sum|g|: bf16 keeps 8 significant bits, so each
    of got and bf16(ref) is within 2^-8 of its magnitude of the value it
    rounds, and a sum of k fp32 terms taken in at most 17 + rows/128
    sequential additions errs by at most that many units of 2^-24 times the
    sum of magnitudes (doubled for slack)."""
    got = np.asarray(got, np.float64)
    bound = (2.0 ** -7 * (1 + 2.0 ** -7) * np.abs(ref_bf16)
             + (17 + -(-rows // 128)) * 2.0 ** -23 * mag)
    return np.abs(got - ref_bf16) <= bound


def gemm_tolerance_ok(d_gpu: np.ndarray, d_ref_bf16: np.ndarray, bound: np.ndarray):
    """The stated GEMM bar: |D_gpu - bf16(D_ref)| <= 1e-2 * bound + 1e-3."""
    err = np.abs(d_gpu.astype(np.float64) - d_ref_bf16)
    return err <= 1e-2 * bound + 1e-3


def gemm_derived_ok(d_gpu: np.ndarray, d_ref_bf16: np.ndarray, bound: np.ndarray, k: int):
    """A tighter bar derived from the arithmetic of a scaled FP8 GEMM with an
    fp32 accumulator and a bf16 result:

        |D_gpu - bf16(D)| <= 2^-7 (1 + 2^-7) |bf16(D)| + (1 + 2^-8) k 2^-23 bound

    with D the exact result and bound = s_a s_b sum_k |a||b|.  Each product of
    two e4m3 values is exact in fp32; summing k of them in fp32 in any order
    with round-to-nearest errs by at most (k-1) 2^-24 / (1 - (k-1) 2^-24) times
    the sum of magnitudes, under k 2^-23 for any k below 2^22; the fp32
    product of the two scales and the fp32 multiply of the sum by it add two
    more relative roundings of 2^-24 (and a bias add in fp32 a third), which
    the (1 + 2^-7) factor covers.  bf16 keeps 8 significant bits, so rounding
    to it moves a value by at most 2^-8 of its magnitude; the two roundings
    (of the GPU's fp32 value and of D) together add 2^-7 |D|, and
    |D| <= |bf16(D)| / (1 - 2^-8).  The block recipe (per-128 partials scaled
    and summed in fp32) satisfies the same bound when bound carries the
    per-tile scales."""
    ref = np.asarray(d_ref_bf16, np.float64)
    err = np.abs(np.asarray(d_gpu, np.float64) - ref)
    lim = 2.0 ** -7 * (1 + 2.0 ** -7) * np.abs(ref) + (1 + 2.0 ** -8) * k * 2.0 ** -23 * bound
    return err <= lim
