"""ctypes binding of libfp8linear.so: argument marshalling only.

Each function takes torch tensors (device memory owned by the caller), passes
their data pointers, sizes and the current CUDA stream to the C entry point of
the same name, and raises Fp8Error on a non-OK status.  No arithmetic of the
method happens here, and there is no fallback: if the library is missing the
import fails.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8linear.so")

FP8_OK, FP8_ERR_NULL, FP8_ERR_SHAPE, FP8_ERR_ALIGNMENT = 0, 1, 2, 3
FP8_ERR_UNSUPPORTED, FP8_ERR_CUDA, FP8_ERR_TIMEOUT = 4, 5, 6
STATUS_NAMES = {0: "FP8_OK", 1: "FP8_ERR_NULL", 2: "FP8_ERR_SHAPE", 3: "FP8_ERR_ALIGNMENT",
                4: "FP8_ERR_UNSUPPORTED", 5: "FP8_ERR_CUDA", 6: "FP8_ERR_TIMEOUT"}

DELAYED, DYNAMIC, BLOCK, BLOCK_2D = 0, 1, 2, 3
SLOT_W, SLOT_X, SLOT_G = 0, 1, 2
META_SCALE, META_SCALE_INV, META_X_SCALE, META_X_SCALE_INV = 0, 1, 2, 3
META_G_SCALE, META_G_SCALE_INV, META_HISTORY = 4, 5, 8


class Fp8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class fp8_meta(ctypes.Structure):
    _fields_ = [("dev", ctypes.c_void_p), ("interval", ctypes.c_int32), ("idx", ctypes.c_int32)]


class fp8_linear_step_io(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("x", "w", "g", "bias", "xq", "xqt", "wq", "wqt", "gq", "gqt", "amax", "y", "dx",
                 "dw", "dbias", "dbias_workspace")] + [("flags", ctypes.c_int32)]


class fp8_block_step_scales(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("x_scale", "x_scale_inv", "x_scale_t", "x_scale_inv_t", "w_scale", "w_scale_inv",
                 "g_scale", "g_scale_inv", "g_scale_t", "g_scale_inv_t")]


FP8_STEP_NEVENTS = 8
FP8_STEP_SAVE_XQ_FWD = 1

P, I64, I32, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
S = ctypes.c_int  # fp8_status / enums

SIGNATURES = {
    "fp8_amax": (S, [P, I64, P, P]),
    "fp8_quantize": (S, [P, I64, I64, S, P, P, P, P, P]),
    "fp8_quantize_transpose": (S, [P, I64, I64, S, P, P, P, P, P, P, P, P]),
    "fp8_dbias_workspace_bytes": (ctypes.c_size_t, [I64, I64]),
    "fp8_quantize_transpose_dbias": (S, [P, I64, I64, S, P, P, P, P, P, P, P, P]),
    "fp8_quantize_fused_workspace_bytes": (ctypes.c_size_t, []),
    "fp8_quantize_fused_dynamic": (S, [P, I64, I64, P, P, P, P, P, P, P]),
    "fp8_quantize_fused_dynamic_noalloc": (S, [P, I64, I64, P, P, P, P, P, P]),
    "fp8_linear_fprop": (S, [P, P, P, P, I64, I64, I64, S, P, P, P]),
    "fp8_linear_dgrad": (S, [P, P, P, P, I64, I64, I64, S, P, P]),
    "fp8_linear_wgrad": (S, [P, P, P, P, I64, I64, I64, S, P, P]),
    "fp8_linear_dgrad_wgrad": (S, [P, P, P, P, P, P, P, I64, I64, I64, S, P, P, P]),
    "fp8_meta_init": (S, [ctypes.POINTER(fp8_meta), P, I32, P]),
    "fp8_meta_record": (S, [ctypes.POINTER(fp8_meta), S, P, P]),
    "fp8_meta_refresh": (S, [ctypes.POINTER(fp8_meta), P]),
    "fp8_meta_state_bytes": (ctypes.c_size_t, [I32]),
    "fp8_meta_save": (S, [ctypes.POINTER(fp8_meta), I64, P, ctypes.c_size_t, P]),
    "fp8_meta_load": (S, [ctypes.POINTER(fp8_meta), P, ctypes.POINTER(I64), P, ctypes.c_size_t, P]),
    "fp8_state_step": (S, [ctypes.POINTER(I64), I32, ctypes.POINTER(fp8_meta), I32, P]),
    "fp8_linear_step_delayed": (S, [ctypes.POINTER(fp8_meta), ctypes.POINTER(I64),
                                    ctypes.POINTER(fp8_linear_step_io), I64, I64, I64, P, P]),
    "fp8_linear_step_dynamic": (S, [ctypes.POINTER(fp8_linear_step_io), P, P, I64, I64, I64, P]),
    "fp8_linear_fprop_dynamic_small": (S, [P, P, I64, I64, I64, P, P, P, P, P, P, P]),
    "fp8_linear_step_block": (S, [ctypes.POINTER(fp8_linear_step_io),
                                  ctypes.POINTER(fp8_block_step_scales), I64, I64, I64, P]),
    "fp8_padded_rows": (I64, [I64, I64]),
    "fp8_pad_multiple": (I64, [I32, I32]),
    "fp8_padded_seq_len": (I64, [I64, I64, I32, I32]),
    "fp8_pad_tokens_bshd": (S, [P, I64, I64, I64, I32, I32, P, ctypes.POINTER(I64), P]),
    "fp8_multi_amax_scales": (S, [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(I64), I32, P,
                                  P, P, P]),
    "fp8_pad_tokens": (S, [P, I64, I64, I64, P, ctypes.POINTER(I64), P]),
    "fp8_check_device_status": (S, [P]),
    "fp8_inject_launch_failures": (S, [I32]),
    "fp8_selftest_wait_timeout": (S, [U32, P]),
    "fp8_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "fp8_last_error": (ctypes.c_char_p, []),
    "fp8_version": (ctypes.c_char_p, []),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with __graft_entry__.build() "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib
