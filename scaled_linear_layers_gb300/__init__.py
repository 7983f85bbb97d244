"""GB300-native FP8 scaled linear layer: thin Python binding of libfp8linear.so.

Every function has the name of the C entry point it calls (see
include/fp8linear.h) and only marshals arguments: torch tensors in, their
device pointers, sizes and the current CUDA stream out to C.  All arithmetic
runs in the library's sm_103a kernels; torch provides device memory and
streams.  Importing this package requires the built library (no fallback).
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (BLOCK, BLOCK_2D, DELAYED, DYNAMIC, SLOT_G, SLOT_W, SLOT_X, Fp8Error,
                   META_G_SCALE, META_G_SCALE_INV, META_HISTORY, META_SCALE, META_SCALE_INV,
                   META_X_SCALE, META_X_SCALE_INV)

_LIB = _lib.load()

__all__ = [
    "fp8_amax", "fp8_quantize", "fp8_quantize_transpose", "fp8_linear_fprop",
    "fp8_linear_dgrad", "fp8_linear_wgrad", "fp8_linear_dgrad_wgrad", "fp8_meta_init",
    "fp8_dbias_workspace_bytes", "fp8_quantize_transpose_dbias", "fp8_pad_multiple",
    "fp8_padded_seq_len", "fp8_pad_tokens_bshd", "fp8_multi_amax_scales",
    "fp8_linear_step_dynamic", "DynamicStepState", "fp8_linear_step_block", "BlockStepScales",
    "fp8_linear_fprop_dynamic_small",
    "fp8_meta_record",
    "fp8_meta_refresh", "fp8_state_step", "fp8_padded_rows", "fp8_pad_tokens",
    "fp8_check_device_status", "fp8_selftest_wait_timeout", "fp8_set_wait_limit_ns",
    "fp8_version", "Fp8Meta",
    "fp8_linear_step_delayed", "LinearStep", "fp8_quantize_fused_dynamic",
    "fp8_quantize_fused_workspace_bytes", "fp8_quantize_fused_dynamic_noalloc",
    "Fp8Error", "DELAYED", "DYNAMIC", "BLOCK", "BLOCK_2D", "SLOT_W", "SLOT_X", "SLOT_G",
    "library_path",
]


def library_path() -> str:
    return _lib.LIB_PATH


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor or None, got {type(t)}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int):
    if status != 0:
        raise Fp8Error(status, _LIB.fp8_last_error().decode())


def _bf16(t):
    assert t.dtype == torch.bfloat16 and t.is_contiguous(), "bf16 contiguous tensor expected"
    return t


def _u8(t):
    if t is None:
        return None
    assert t.dtype in (torch.uint8, torch.float8_e4m3fn) and t.is_contiguous()
    return t


def fp8_version() -> str:
    return _LIB.fp8_version().decode()


def fp8_amax(x, amax_out, stream=None):
    _check(_LIB.fp8_amax(_ptr(_bf16(x)), x.numel(), _ptr(amax_out), _stream(stream)))


def fp8_quantize(x, recipe, scale, scale_inv, q, amax_out=None, stream=None):
    x2 = _bf16(x).reshape(-1, x.shape[-1]) if x.dim() != 1 else x.reshape(1, -1)
    _check(_LIB.fp8_quantize(_ptr(x2), x2.shape[0], x2.shape[1], recipe, _ptr(scale),
                             _ptr(scale_inv), _ptr(_u8(q)), _ptr(amax_out), _stream(stream)))


def fp8_quantize_transpose(x, recipe, scale, scale_inv, q, qt, scale_t=None, scale_inv_t=None,
                           amax_out=None, stream=None):
    _bf16(x)
    assert x.dim() == 2
    _check(_LIB.fp8_quantize_transpose(_ptr(x), x.shape[0], x.shape[1], recipe, _ptr(scale),
                                       _ptr(scale_inv), _ptr(_u8(q)), _ptr(_u8(qt)), _ptr(scale_t),
                                       _ptr(scale_inv_t), _ptr(amax_out), _stream(stream)))


def fp8_quantize_fused_workspace_bytes() -> int:
    return int(_LIB.fp8_quantize_fused_workspace_bytes())


def fp8_quantize_fused_dynamic(x, scale, scale_inv, q, qt, amax_out, workspace, stream=None):
    """Current scaling in one launch; ``workspace`` is a zeroed device tensor
    of fp8_quantize_fused_workspace_bytes() bytes (reusable across calls)."""
    _bf16(x)
    assert x.dim() == 2
    assert workspace.numel() * workspace.element_size() >= fp8_quantize_fused_workspace_bytes()
    _check(_LIB.fp8_quantize_fused_dynamic(_ptr(x), x.shape[0], x.shape[1], _ptr(scale),
                                           _ptr(scale_inv), _ptr(_u8(q)), _ptr(_u8(qt)),
                                           _ptr(amax_out), _ptr(workspace), _stream(stream)))


def fp8_quantize_fused_dynamic_noalloc(x, scale, scale_inv, q, qt, amax_out, stream=None):
    """fp8_quantize_fused_dynamic with the library's static scratch instead of
    a workspace, for callers that cannot allocate device memory (see the C
    header).  Calls share that scratch: keep them in one stream order."""
    _bf16(x)
    assert x.dim() == 2
    _check(_LIB.fp8_quantize_fused_dynamic_noalloc(_ptr(x), x.shape[0], x.shape[1], _ptr(scale),
                                                   _ptr(scale_inv), _ptr(_u8(q)), _ptr(_u8(qt)),
                                                   _ptr(amax_out), _stream(stream)))


def fp8_linear_fprop(xq, x_scale, wq, w_scale, M, N, K, recipe, bias, y, stream=None):
    _check(_LIB.fp8_linear_fprop(_ptr(_u8(xq)), _ptr(x_scale), _ptr(_u8(wq)), _ptr(w_scale), M, N,
                                 K, recipe, _ptr(bias), _ptr(y), _stream(stream)))


def fp8_linear_dgrad(gq, g_scale, wqt, w_scale, M, N, K, recipe, dx, stream=None):
    _check(_LIB.fp8_linear_dgrad(_ptr(_u8(gq)), _ptr(g_scale), _ptr(_u8(wqt)), _ptr(w_scale), M,
                                 N, K, recipe, _ptr(dx), _stream(stream)))


def fp8_linear_wgrad(gqt, g_scale, xqt, x_scale, M, N, K, recipe, dw, stream=None):
    _check(_LIB.fp8_linear_wgrad(_ptr(_u8(gqt)), _ptr(g_scale), _ptr(_u8(xqt)), _ptr(x_scale), M,
                                 N, K, recipe, _ptr(dw), _stream(stream)))


def fp8_dbias_workspace_bytes(rows, cols):
    return _LIB.fp8_dbias_workspace_bytes(rows, cols)


def fp8_quantize_transpose_dbias(g, recipe, scale, scale_inv, q, qt, dbias, workspace,
                                 amax_out=None, stream=None):
    rows, cols = g.shape
    _check(_LIB.fp8_quantize_transpose_dbias(_ptr(_bf16(g)), rows, cols, recipe, _ptr(scale),
                                             _ptr(scale_inv), _ptr(_u8(q)), _ptr(_u8(qt)),
                                             _ptr(amax_out),
                                             _ptr(dbias), _ptr(workspace), _stream(stream)))


def fp8_linear_dgrad_wgrad(gq, gqt, g_scale, wqt, w_scale, xqt, x_scale, M, N, K, recipe, dx, dw,
                           stream=None):
    _check(_LIB.fp8_linear_dgrad_wgrad(_ptr(_u8(gq)), _ptr(_u8(gqt)), _ptr(g_scale),
                                       _ptr(_u8(wqt)), _ptr(w_scale), _ptr(_u8(xqt)),
                                       _ptr(x_scale), M, N, K, recipe, _ptr(dx), _ptr(dw),
                                       _stream(stream)))


def fp8_linear_fprop_dynamic_small(x, w, scales, y, bias=None, amax=None, xq=None, wq=None,
                                   stream=None):
    """Current-scaling fprop of a one-tile linear in one launch (see the C
    header): x [M,K], w [N,K] bf16 -> y [M,N]; scales: 4 device floats."""
    _bf16(x)
    _bf16(w)
    M, K = x.shape
    N = w.shape[0]
    assert w.shape[1] == K and tuple(y.shape) == (M, N)
    _check(_LIB.fp8_linear_fprop_dynamic_small(_ptr(x), _ptr(w), M, N, K, _ptr(bias),
                                               _ptr(scales), _ptr(amax), _ptr(_u8(xq)),
                                               _ptr(_u8(wq)), _ptr(y), _stream(stream)))


class DynamicStepState:
    """Device scratch of fp8_linear_step_dynamic: the 6 scales and the three
    quantiser workspaces (zeroed once)."""

    def __init__(self, device="cuda"):
        self.scales = torch.empty(6, dtype=torch.float32, device=device)
        n = 3 * _LIB.fp8_quantize_fused_workspace_bytes() // 4
        self.workspace = torch.zeros(n, dtype=torch.int32, device=device)


def fp8_linear_step_dynamic(state: DynamicStepState, step: "LinearStep", stream=None):
    """One current-scaling training step (see the C header)."""
    _check(_LIB.fp8_linear_step_dynamic(ctypes.byref(step.io), _ptr(state.scales),
                                        _ptr(state.workspace), step.M, step.N, step.K,
                                        _stream(stream)))


class BlockStepScales:
    """The tile-scale arrays of fp8_linear_step_block for an [M, N, K] linear
    (torch float32 tensors this object owns, named as in the C struct)."""

    def __init__(self, M, N, K, device="cuda"):
        f = dict(dtype=torch.float32, device=device)
        shapes = {"x_scale": (M, K // 128), "x_scale_t": (M // 128, K),
                  "w_scale": (N // 128, K // 128), "g_scale": (M, N // 128),
                  "g_scale_t": (M // 128, N)}
        self.c = _lib.fp8_block_step_scales()
        for name, shape in shapes.items():
            inv = name.replace("_scale", "_scale_inv")
            for n in (name, inv):
                t = torch.empty(shape, **f)
                setattr(self, n, t)
                setattr(self.c, n, t.data_ptr())


def fp8_linear_step_block(scales: BlockStepScales, step: "LinearStep", stream=None):
    """One block-recipe training step (see the C header)."""
    _check(_LIB.fp8_linear_step_block(ctypes.byref(step.io), ctypes.byref(scales.c), step.M,
                                      step.N, step.K, _stream(stream)))


def fp8_pad_multiple(cp_size=1, tp_size=1):
    return _LIB.fp8_pad_multiple(cp_size, tp_size)


def fp8_padded_seq_len(batch, seq, cp_size=1, tp_size=1):
    return _LIB.fp8_padded_seq_len(batch, seq, cp_size, tp_size)


def fp8_pad_tokens_bshd(x, cp_size, tp_size, out, stream=None):
    """x [B, T, H] bf16 -> out [B, T', H]; returns T'."""
    _bf16(x)
    B, T, H = x.shape
    tp = ctypes.c_int64(0)
    _check(_LIB.fp8_pad_tokens_bshd(_ptr(x), B, T, H, cp_size, tp_size, _ptr(out),
                                    ctypes.byref(tp), _stream(stream)))
    return tp.value


def fp8_multi_amax_scales(ws, amax, scale, scale_inv, stream=None):
    """amax/scale/scale_inv: float32 device tensors of len(ws)."""
    n = len(ws)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in ws])
    numel = (ctypes.c_int64 * max(n, 1))(*[t.numel() for t in ws])
    for t in ws:
        _bf16(t)
    _check(_LIB.fp8_multi_amax_scales(ptrs, numel, n, _ptr(amax), _ptr(scale), _ptr(scale_inv),
                                      _stream(stream)))


class Fp8Meta:
    """One weight's delayed-scaling state: the C fp8_meta struct plus the
    device block it points to (a torch float32 tensor this object owns)."""

    def __init__(self, interval: int = 16, device="cuda", stream=None):
        self.block = torch.empty(8 + interval, dtype=torch.float32, device=device)
        self.c = _lib.fp8_meta()
        _check(_LIB.fp8_meta_init(ctypes.byref(self.c), _ptr(self.block), interval,
                                  _stream(stream)))

    def view(self, index: int):
        return self.block[index:index + 1]

    @property
    def scale(self):
        return self.view(META_SCALE)

    @property
    def scale_inv(self):
        return self.view(META_SCALE_INV)

    @property
    def x_scale(self):
        return self.view(META_X_SCALE)

    @property
    def x_scale_inv(self):
        return self.view(META_X_SCALE_INV)

    @property
    def g_scale(self):
        return self.view(META_G_SCALE)

    @property
    def g_scale_inv(self):
        return self.view(META_G_SCALE_INV)

    @property
    def history(self):
        return self.block[META_HISTORY:]

    def save(self, step_count: int = 0, stream=None) -> bytes:
        """The meta's checkpoint blob (fp8_meta_save; synchronises the stream)."""
        n = _LIB.fp8_meta_state_bytes(self.c.interval)
        buf = ctypes.create_string_buffer(n)
        _check(_LIB.fp8_meta_save(ctypes.byref(self.c), int(step_count), buf, n,
                                  _stream(stream)))
        return buf.raw

    @classmethod
    def load(cls, blob: bytes, device="cuda", stream=None):
        """A meta restored from a blob of save(); returns (meta, step_count)."""
        hdr = ctypes.create_string_buffer(blob, len(blob))
        interval = int.from_bytes(blob[8:12], "little", signed=True)
        if not 1 <= interval <= 1024:
            raise Fp8Error(2, "not a saved fp8 meta state")
        self = cls.__new__(cls)
        self.block = torch.empty(8 + interval, dtype=torch.float32, device=device)
        self.c = _lib.fp8_meta()
        cnt = ctypes.c_int64(0)
        _check(_LIB.fp8_meta_load(ctypes.byref(self.c), _ptr(self.block), ctypes.byref(cnt), hdr,
                                  len(blob), _stream(stream)))
        return self, cnt.value

    @property
    def idx(self) -> int:
        return self.c.idx


def fp8_meta_init(meta: Fp8Meta, interval: int = 16, stream=None):
    _check(_LIB.fp8_meta_init(ctypes.byref(meta.c), _ptr(meta.block), interval, _stream(stream)))


def fp8_meta_record(meta: Fp8Meta, which: int, amax_dev, stream=None):
    _check(_LIB.fp8_meta_record(ctypes.byref(meta.c), which, _ptr(amax_dev), _stream(stream)))


def fp8_meta_refresh(meta: Fp8Meta, stream=None):
    _check(_LIB.fp8_meta_refresh(ctypes.byref(meta.c), _stream(stream)))


def fp8_state_step(step_count: list, interval: int, metas, stream=None):
    """step_count is a one-element list holding the host counter (updated in place)."""
    arr = (_lib.fp8_meta * max(1, len(metas)))()
    for i, m in enumerate(metas):
        arr[i] = m.c
    cnt = ctypes.c_int64(step_count[0])
    _check(_LIB.fp8_state_step(ctypes.byref(cnt), interval, arr, len(metas), _stream(stream)))
    step_count[0] = cnt.value
    for i, m in enumerate(metas):
        m.c = arr[i]


class LinearStep:
    """Buffers of fp8_linear_step_delayed for one linear: the C io struct
    built once from torch tensors (the caller keeps them alive), so a step
    is a single C call.  ``set_inputs`` swaps the x / g / w pointers."""

    def __init__(self, M, N, K, device="cuda", backward=True, bias=None, dbias=False,
                 save_xq_fwd=False):
        u8 = dict(dtype=torch.uint8, device=device)
        bf = dict(dtype=torch.bfloat16, device=device)
        self.M, self.N, self.K = M, N, K
        self.xq, self.wq, self.wqt = (torch.empty((M, K), **u8), torch.empty((N, K), **u8),
                                      torch.empty((K, N), **u8))
        self.amax = torch.zeros(3, dtype=torch.float32, device=device)
        self.y = torch.empty((M, N), **bf)
        self.bias = bias
        if backward:
            self.xqt, self.gq, self.gqt = (torch.empty((K, M), **u8), torch.empty((M, N), **u8),
                                           torch.empty((N, M), **u8))
            self.dx, self.dw = torch.empty((M, K), **bf), torch.empty((N, K), **bf)
        else:
            self.xqt = self.gq = self.gqt = self.dx = self.dw = None
        self.dbias = self.dbias_workspace = None
        if backward and dbias:
            self.dbias = torch.empty(N, **bf)
            self.dbias_workspace = torch.empty(
                _LIB.fp8_dbias_workspace_bytes(M, N) // 4, dtype=torch.float32, device=device)
        self.io = _lib.fp8_linear_step_io()
        for name in ("xq", "xqt", "wq", "wqt", "gq", "gqt", "amax", "y", "dx", "dw", "bias",
                     "dbias", "dbias_workspace"):
            t = getattr(self, name)
            setattr(self.io, name, None if t is None else t.data_ptr())
        self.io.flags = _lib.FP8_STEP_SAVE_XQ_FWD if save_xq_fwd else 0

    def set_inputs(self, x, w, g=None):
        for t in (x, w) + ((g,) if g is not None else ()):
            _bf16(t)
        assert tuple(x.shape) == (self.M, self.K) and tuple(w.shape) == (self.N, self.K)
        self.io.x, self.io.w = x.data_ptr(), w.data_ptr()
        if g is not None:
            assert tuple(g.shape) == (self.M, self.N) and self.gq is not None
        self.io.g = None if g is None else g.data_ptr()


def fp8_linear_step_delayed(meta: Fp8Meta, step_count: list, step: LinearStep, events=None,
                            stream=None):
    """One delayed-scaling training step (see the C header).  ``events`` is
    None or a list of FP8_STEP_NEVENTS recorded torch.cuda.Event objects."""
    cnt = ctypes.c_int64(step_count[0])
    ev = None
    if events is not None:
        arr = (ctypes.c_void_p * _lib.FP8_STEP_NEVENTS)(*[e.cuda_event for e in events])
        ev = ctypes.cast(arr, ctypes.c_void_p)
    _check(_LIB.fp8_linear_step_delayed(ctypes.byref(meta.c), ctypes.byref(cnt),
                                        ctypes.byref(step.io), step.M, step.N, step.K, ev,
                                        _stream(stream)))
    step_count[0] = cnt.value


def fp8_padded_rows(rows: int, multiple: int = 16) -> int:
    return int(_LIB.fp8_padded_rows(rows, multiple))


def fp8_pad_tokens(x, multiple, out, stream=None) -> int:
    _bf16(x)
    padded = ctypes.c_int64(0)
    _check(_LIB.fp8_pad_tokens(_ptr(x), x.shape[0], x.shape[1], multiple, _ptr(out),
                               ctypes.byref(padded), _stream(stream)))
    return padded.value


def fp8_check_device_status(stream=None):
    _check(_LIB.fp8_check_device_status(_stream(stream)))


def fp8_selftest_wait_timeout(timeout_us: int, stream=None):
    _check(_LIB.fp8_selftest_wait_timeout(timeout_us, _stream(stream)))


def fp8_set_wait_limit_ns(limit_ns: int) -> int:
    """Limit of the kernels' bounded waits (0 restores the 2 s default);
    returns the previous limit."""
    return int(_LIB.fp8_set_wait_limit_ns(int(limit_ns)))
