"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/fp8linear.h declares, and rejects bad arguments on the host before
anything is enqueued (the rejection happens before the device is touched, so
these run on a CPU-only machine)."""
import ctypes
import json
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8linear.h")
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "page_facts.json")))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    from scaled_linear_layers_gb300 import _lib
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", text)) - {"fp8_meta", "fp8_status"})


def test_header_declares_the_expected_boundary():
    syms = declared_symbols()
    for name in ["fp8_quantize", "fp8_quantize_transpose", "fp8_linear_fprop", "fp8_linear_dgrad",
                 "fp8_linear_wgrad", "fp8_meta_record", "fp8_meta_refresh", "fp8_pad_tokens"]:
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    from scaled_linear_layers_gb300 import _lib
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_library_does_not_link_the_oracle(lib):
    from scaled_linear_layers_gb300 import _lib
    assert not hasattr(lib, "orc_e4m3_encode")
    with open(_lib.LIB_PATH, "rb") as f:
        assert b"orc_" not in f.read()


def test_version(lib):
    assert lib.fp8_version().decode().startswith("fp8linear")


def test_padded_rows_page_example(lib):
    ex = GOLDEN["unaligned_token_count_example"]
    m = GOLDEN["token_multiple"]["value"]
    assert lib.fp8_padded_rows(ex["rows"], m) == 3872
    assert lib.fp8_padded_rows(0, 16) == 0
    assert lib.fp8_padded_rows(16, 16) == 16
    assert lib.fp8_padded_rows(17, 16) == 32
    assert lib.fp8_padded_rows(-1, 16) == -1
    assert lib.fp8_padded_rows(5, 0) == -1


def test_gemm_rejects_unaligned_token_count_with_the_pages_message(lib):
    ex = GOLDEN["unaligned_token_count_example"]
    st = lib.fp8_linear_fprop(None, None, None, None, 4096, 4096, ex["rows"], 0, None, None, None)
    assert st == 3  # FP8_ERR_ALIGNMENT
    msg = lib.fp8_last_error().decode()
    assert f"Expected K to be divisible by 16, but got K={ex['rows']}" in msg
    st = lib.fp8_linear_wgrad(None, None, None, None, ex["rows"], 4096, 4096, 0, None, None)
    assert st == 3 and f"but got M={ex['rows']}" in lib.fp8_last_error().decode()


def test_gemm_block_recipe_needs_aligned_scale_pointers(lib):
    # host-side check only: the fake addresses are never dereferenced
    ok, off = 0x10000, 0x10004
    st = lib.fp8_linear_wgrad(ok, ok, ok, off, 256, 256, 256, 2, ok, None)
    assert st == 3 and "block scales are not 16-byte aligned" in lib.fp8_last_error().decode()
    st = lib.fp8_linear_fprop(ok, off, ok, ok, 256, 256, 256, 2, None, ok, None)
    assert st == 3 and "block scales are not 16-byte aligned" in lib.fp8_last_error().decode()


def test_gemm_block_recipe_needs_multiples_of_128(lib):
    st = lib.fp8_linear_fprop(None, None, None, None, 256, 256, 144, 2, None, None, None)
    assert st == 3 and "divisible by 128" in lib.fp8_last_error().decode()


def test_null_shape_and_alignment_errors(lib):
    assert lib.fp8_linear_fprop(None, None, None, None, 0, 16, 16, 0, None, None, None) == 2
    assert lib.fp8_linear_fprop(None, None, None, None, 16, 16, 16, 0, None, None, None) == 1
    assert "is NULL" in lib.fp8_last_error().decode()
    assert lib.fp8_quantize(None, 4, 4, 0, None, None, None, None, None) == 1
    assert lib.fp8_quantize(None, -1, 4, 0, None, None, None, None, None) == 2
    bad = ctypes.c_void_p(0x1001)  # never dereferenced: rejected on the host
    good = ctypes.c_void_p(0x2000)
    assert lib.fp8_quantize(bad, 4, 4, 0, None, good, good, None, None) == 3
    assert "16-byte aligned" in lib.fp8_last_error().decode()
    assert lib.fp8_quantize_transpose(good, 24, 16, 0, None, good, good, good, None, None, None,
                                      None) == 3
    assert lib.fp8_quantize_transpose(good, 16, 16, 9, None, good, good, good, None, None, None,
                                      None) == 2
    # dynamic scaling needs somewhere to put the amax
    assert lib.fp8_quantize(good, 4, 4, 1, good, good, good, None, None) == 1


def test_state_step_host_counter(lib):
    from scaled_linear_layers_gb300 import _lib
    cnt = ctypes.c_int64(0)
    for i in range(15):  # no refresh due before the 16th step: host only
        assert lib.fp8_state_step(ctypes.byref(cnt), 16, None, 0, None) == 0
    assert cnt.value == 15
    assert lib.fp8_state_step(ctypes.byref(cnt), 16, None, 0, None) == 0
    assert cnt.value == 16
    assert lib.fp8_state_step(ctypes.byref(cnt), 0, None, 0, None) == 2
    m = _lib.fp8_meta()
    assert lib.fp8_meta_record(ctypes.byref(m), 0, None, None) == 1


def test_pad_tokens_rejects_overlap_and_bad_multiple(lib):
    p = ctypes.c_void_p(0x10000)
    out_rows = ctypes.c_int64(0)
    assert lib.fp8_pad_tokens(p, 10, 16, 0, p, ctypes.byref(out_rows), None) == 2
    assert lib.fp8_pad_tokens(p, 10, 16, 16, p, ctypes.byref(out_rows), None) == 2
    assert "overlap" in lib.fp8_last_error().decode()
    assert out_rows.value == 16


def test_dbias_entry_point_host_checks(lib):
    good = ctypes.c_void_p(0x2000)
    bad = ctypes.c_void_p(0x2002)
    assert lib.fp8_dbias_workspace_bytes(4096, 4096) == 32 * 4096 * 4
    assert lib.fp8_dbias_workspace_bytes(3872, 48) == 31 * 48 * 4
    assert lib.fp8_dbias_workspace_bytes(0, 48) == 0
    args = lambda r, ws, db: (good, 256, 128, r, good, good, good, good, None, db, ws, None)
    assert lib.fp8_quantize_transpose_dbias(*args(2, good, good)) == 4  # block: unsupported
    assert lib.fp8_quantize_transpose_dbias(*args(0, None, good)) == 1  # no workspace
    assert lib.fp8_quantize_transpose_dbias(*args(0, good, None)) == 1  # no dbias
    assert lib.fp8_quantize_transpose_dbias(*args(0, good, bad)) == 3   # misaligned dbias
    assert lib.fp8_quantize_transpose_dbias(good, 250, 128, 0, good, good, good, good, None,
                                            good, good, None) == 3     # rows % 16


def test_meta_checkpoint_host_checks(lib):
    from scaled_linear_layers_gb300 import _lib
    assert lib.fp8_meta_state_bytes(16) == 24 + 4 * 24
    assert lib.fp8_meta_state_bytes(0) == 0 and lib.fp8_meta_state_bytes(2000) == 0
    m = _lib.fp8_meta()
    good = ctypes.c_void_p(0x2000)
    cnt = ctypes.c_int64(0)
    blob = ctypes.create_string_buffer(120)
    # an all-zero buffer is not a saved state
    assert lib.fp8_meta_load(ctypes.byref(m), good, ctypes.byref(cnt), blob, 120, None) == 2
    assert "not a saved fp8 meta state" in lib.fp8_last_error().decode()
    # a header with a bad idx
    hdr = (0x534D3846).to_bytes(4, "little") + (1).to_bytes(4, "little") + \
        (16).to_bytes(4, "little") + (16).to_bytes(4, "little") + (0).to_bytes(8, "little")
    blob = ctypes.create_string_buffer(hdr + bytes(96), 120)
    assert lib.fp8_meta_load(ctypes.byref(m), good, ctypes.byref(cnt), blob, 120, None) == 2
    # too short for its interval
    hdr = hdr[:12] + (3).to_bytes(4, "little") + hdr[16:]
    blob = ctypes.create_string_buffer(hdr + bytes(96), 120)
    assert lib.fp8_meta_load(ctypes.byref(m), good, ctypes.byref(cnt), blob, 100, None) == 2
    # save needs a big enough buffer
    m.dev, m.interval, m.idx = good, 16, 0
    assert lib.fp8_meta_save(ctypes.byref(m), 5, blob, 100, None) == 2


def test_parallel_padding_arithmetic_matches_the_oracle(lib):
    import oracle
    for cp in (1, 2, 3):
        for tp in (1, 2, 4, 8):
            assert lib.fp8_pad_multiple(cp, tp) == oracle.pad_multiple(cp, tp)
            for B in (1, 2, 5, 16, 24):
                for T in (0, 1, 9, 128, 3858):
                    assert lib.fp8_padded_seq_len(B, T, cp, tp) == \
                        oracle.padded_seq_len(B, T, cp, tp), (B, T, cp, tp)
    assert lib.fp8_pad_multiple(0, 1) == -1 and lib.fp8_padded_seq_len(0, 4, 1, 1) == -1
    good = ctypes.c_void_p(0x2000)
    out = ctypes.c_int64(0)
    assert lib.fp8_pad_tokens_bshd(good, 2, 5, 12, 1, 1, good, ctypes.byref(out), None) == 3
    assert lib.fp8_pad_tokens_bshd(good, 0, 5, 16, 1, 1, good, ctypes.byref(out), None) == 2


def test_multi_amax_host_checks(lib):
    P = ctypes.c_void_p
    ptrs = (P * 2)(0x2000, 0x2008)
    numel = (ctypes.c_int64 * 2)(16, 16)
    good = P(0x3000)
    assert lib.fp8_multi_amax_scales(ptrs, numel, 0, None, None, None, None) == 0
    assert lib.fp8_multi_amax_scales(ptrs, numel, 2, good, good, good, None) == 3  # misaligned w[1]
    ptrs[1] = None
    assert lib.fp8_multi_amax_scales(ptrs, numel, 2, good, good, good, None) == 1
    numel[1] = -1
    assert lib.fp8_multi_amax_scales(ptrs, numel, 2, good, good, good, None) == 2


def test_step_rejects_bad_flags_before_touching_the_counter(lib):
    from scaled_linear_layers_gb300 import _lib
    m = _lib.fp8_meta()
    good = 0x2000
    m.dev, m.interval, m.idx = good, 16, 0
    io = _lib.fp8_linear_step_io()
    for name in ("x", "w", "xq", "wq", "wqt", "amax", "y"):
        setattr(io, name, good)
    io.flags = 4
    cnt = ctypes.c_int64(7)
    st = lib.fp8_linear_step_delayed(ctypes.byref(m), ctypes.byref(cnt), ctypes.byref(io),
                                     16, 16, 16, None, None)
    assert st == 2 and "unknown flags" in lib.fp8_last_error().decode()
    assert cnt.value == 7  # nothing happened: the step counter is untouched
    io.flags = 1  # saving Xq from the forward needs xqt
    st = lib.fp8_linear_step_delayed(ctypes.byref(m), ctypes.byref(cnt), ctypes.byref(io),
                                     16, 16, 16, None, None)
    assert st == 1 and cnt.value == 7


def test_recipe_steps_host_checks(lib):
    from scaled_linear_layers_gb300 import _lib
    good = 0x2000
    io = _lib.fp8_linear_step_io()
    for name in ("x", "w", "xq", "wq", "wqt", "amax", "y"):
        setattr(io, name, good)
    P = ctypes.c_void_p
    # dynamic: scales and workspace are required; dbias and flags are not supported
    assert lib.fp8_linear_step_dynamic(ctypes.byref(io), None, P(good), 16, 16, 16, None) == 1
    io.dbias = good
    assert lib.fp8_linear_step_dynamic(ctypes.byref(io), P(good), P(good), 16, 16, 16, None) == 4
    io.dbias = None
    io.flags = 1
    assert lib.fp8_linear_step_dynamic(ctypes.byref(io), P(good), P(good), 16, 16, 16, None) == 2
    io.flags = 0
    assert lib.fp8_linear_step_dynamic(ctypes.byref(io), P(good), P(good), 16, 24, 16, None) == 3
    # block: dims multiples of 128, every scale array, no bias
    sc = _lib.fp8_block_step_scales()
    for name, _ in sc._fields_:
        setattr(sc, name, good)
    assert lib.fp8_linear_step_block(ctypes.byref(io), ctypes.byref(sc), 128, 128, 192, None) == 3
    io.bias = good
    assert lib.fp8_linear_step_block(ctypes.byref(io), ctypes.byref(sc), 128, 128, 128, None) == 4
    io.bias = None
    sc.g_scale_t = None
    assert lib.fp8_linear_step_block(ctypes.byref(io), ctypes.byref(sc), 128, 128, 128, None) == 1
    sc.g_scale_t = good + 4  # misaligned: rejected before the quantisers are enqueued
    assert lib.fp8_linear_step_block(ctypes.byref(io), ctypes.byref(sc), 128, 128, 128, None) == 3
    assert "scale array is not 16-byte aligned" in lib.fp8_last_error().decode()


# Host checks of the remaining entry points.  The fake addresses below are
# aligned (0x10000) or not (0x10004); none is dereferenced, because every
# call fails its argument checks before the device is touched.
OK_P, OFF_P = 0x10000, 0x10004


def test_amax_host_checks(lib):
    assert lib.fp8_amax(OK_P, -1, OK_P, None) == 2
    assert lib.fp8_amax(OK_P, 8, None, None) == 1
    assert lib.fp8_amax(None, 8, OK_P, None) == 1
    assert lib.fp8_amax(OFF_P, 8, OK_P, None) == 3
    assert "not 16-byte aligned" in lib.fp8_last_error().decode()


def test_dgrad_host_checks(lib):
    # dX [M,K] = Gq [M,N] . Wq [N,K]: each of M, N, K must be a multiple of 16
    st = lib.fp8_linear_dgrad(OK_P, OK_P, OK_P, OK_P, 4096, 3858, 4096, 0, OK_P, None)
    assert st == 3 and "Expected N to be divisible by 16, but got N=3858" in lib.fp8_last_error().decode()
    assert lib.fp8_linear_dgrad(OK_P, OK_P, OK_P, OK_P, 256, 256, 256, 0, None, None) == 1
    assert lib.fp8_linear_dgrad(OK_P, OK_P, OK_P, OK_P, 0, 256, 256, 0, OK_P, None) == 2
    assert lib.fp8_linear_dgrad(OK_P, OK_P, OK_P, OK_P, 256, 256, 256, 7, OK_P, None) == 2
    # block recipe: multiples of 128
    st = lib.fp8_linear_dgrad(OK_P, OK_P, OK_P, OK_P, 256, 144, 256, 2, OK_P, None)
    assert st == 3 and "divisible by 128" in lib.fp8_last_error().decode()


def test_dgrad_wgrad_host_checks(lib):
    args = [OK_P] * 7
    st = lib.fp8_linear_dgrad_wgrad(*args, 256, 256, 256, 2, OK_P, OK_P, None)
    assert st == 4 and "block recipe" in lib.fp8_last_error().decode()
    assert lib.fp8_linear_dgrad_wgrad(*args, 256, 256, 264, 0, OK_P, OK_P, None) == 3
    assert lib.fp8_linear_dgrad_wgrad(*args, 256, 256, 256, 0, OK_P, None, None) == 1
    assert lib.fp8_linear_dgrad_wgrad(*args, 256, 256, 256, 0, OFF_P, OK_P, None) == 3


def test_meta_init_and_refresh_host_checks(lib):
    from scaled_linear_layers_gb300 import _lib
    m = _lib.fp8_meta()
    assert lib.fp8_meta_init(None, OK_P, 16, None) == 1
    assert lib.fp8_meta_init(ctypes.byref(m), None, 16, None) == 1
    assert lib.fp8_meta_init(ctypes.byref(m), OFF_P, 16, None) == 3
    assert lib.fp8_meta_init(ctypes.byref(m), OK_P, 0, None) == 2
    assert lib.fp8_meta_init(ctypes.byref(m), OK_P, 1025, None) == 2
    assert m.dev is None  # nothing was initialised
    assert lib.fp8_meta_refresh(None, None) == 1
    assert lib.fp8_meta_refresh(ctypes.byref(m), None) == 1  # no device block
    m.dev, m.interval = OK_P, 0
    assert lib.fp8_meta_refresh(ctypes.byref(m), None) == 2


def test_fused_dynamic_host_checks(lib):
    assert lib.fp8_quantize_fused_workspace_bytes() == 16384
    f = lib.fp8_quantize_fused_dynamic
    assert f(OK_P, 100, 64, OK_P, OK_P, OK_P, None, OK_P, OK_P, None) == 3  # rows % 16
    assert f(OK_P, -16, 64, OK_P, OK_P, OK_P, None, OK_P, OK_P, None) == 2
    assert f(OK_P, 64, 64, OK_P, OK_P, None, None, OK_P, OK_P, None) == 1  # q and qt both NULL
    assert "both NULL" in lib.fp8_last_error().decode()
    assert f(OK_P, 64, 64, OK_P, OK_P, OK_P, None, OK_P, None, None) == 1  # no workspace
    assert f(OK_P, 64, 64, OK_P, OK_P, OK_P, None, OK_P, OFF_P, None) == 3
    assert f(OK_P, 64, 64, None, OK_P, OK_P, None, OK_P, OK_P, None) == 1  # no scale
    g = lib.fp8_quantize_fused_dynamic_noalloc
    assert g(OK_P, 100, 64, OK_P, OK_P, OK_P, None, OK_P, None) == 3
    assert g(OK_P, 64, 64, OK_P, OK_P, None, None, OK_P, None) == 1


def test_quantize_transpose_block_needs_column_scales(lib):
    f = lib.fp8_quantize_transpose
    # row+column tiles: the column-tile scales are required, the row-tile
    # ones only when q is written
    assert f(OK_P, 256, 256, 2, OK_P, OK_P, OK_P, OK_P, None, OK_P, None, None) == 1
    assert f(OK_P, 256, 256, 2, None, None, OK_P, OK_P, OK_P, OK_P, None, None) == 1
    assert f(OK_P, 256, 256, 9, OK_P, OK_P, OK_P, OK_P, OK_P, OK_P, None, None) == 2


def test_wait_limit_setter_returns_the_previous_limit(lib):
    default = 2_000_000_000
    prev = lib.fp8_set_wait_limit_ns(5000)
    assert prev == default
    assert lib.fp8_set_wait_limit_ns(0) == 5000       # 0 restores the default
    assert lib.fp8_set_wait_limit_ns(default) == default


def test_fused_dynamic_rejects_more_tiles_than_int32(lib):
    p = ctypes.c_void_p(0x1000)
    rows = cols = 1 << 24   # 2^34 tiles of 128 x 128
    for fn in (lib.fp8_quantize_fused_dynamic_noalloc,):
        assert fn(p, rows, cols, p, p, p, None, p, None) == 2   # FP8_ERR_SHAPE
    assert lib.fp8_quantize_fused_dynamic(p, rows, cols, p, p, p, None, p, p, None) == 2
    assert "tiles" in lib.fp8_last_error().decode()


def test_small_fprop_host_checks(lib):
    p = ctypes.c_void_p(0x1000)
    f = lib.fp8_linear_fprop_dynamic_small
    assert f(p, p, 144, 256, 256, None, p, None, None, None, p, None) == 4   # larger than a tile
    assert "one tile" in lib.fp8_last_error().decode()
    assert f(p, p, 64, 272, 256, None, p, None, None, None, p, None) == 4
    assert f(p, p, 64, 256, 528, None, p, None, None, None, p, None) == 4
    assert f(p, p, 64, 256, 24, None, p, None, None, None, p, None) == 3    # K % 16
    assert f(p, p, 0, 256, 256, None, p, None, None, None, p, None) == 2
    assert f(None, p, 64, 256, 256, None, p, None, None, None, p, None) == 1
    assert f(p, p, 64, 256, 256, None, p, None, ctypes.c_void_p(0x1001), None, p, None) == 3
