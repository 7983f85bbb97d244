"""Scaling state machine and whole-step drivers of the oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows the AstrAI page "astrai/extension/fp8_state.py":

* ``Meta`` is FP8TensorMeta: every field a single fp32, all starting at 1;
  ``amax_history`` holds ``update_interval`` fp32 slots starting at 1;
  ``record`` writes the slot at ``idx`` and advances ``idx`` modulo the length;
  ``refresh`` takes the window max ``m`` and, only if ``m > 0``, sets
  scale = m/448 and scale_inv = 448/m.
* ``State`` is FP8State: ``step`` adds one to ``step_count`` and refreshes every
  meta when the count is a multiple of ``update_interval``.  It runs once per
  training step (once per fp8_autocast entry).  A second entry in the same
  step (wrapping backward in autocast too) would update twice; the NeMo review
  on the FP8 SALMAutomodel page warns about exactly that extra update.
* ``lag_update`` is _update_delayed_scale: a = max(amax, 1e-12),
  scale = a/448, scale_inv = 448/a, for the next call.
* ``linear_forward`` / ``linear_backward`` are fp8_linear_forward /
  fp8_linear_backward: x and w quantised with the meta's current scale_inv,
  GEMM scaled by the product of the two scales, then record(amax_w) and the lag
  update of x; in backward, g quantised with g_scale_inv, w and x quantised
  again (x with the x scale the forward just updated), dgrad with
  g_scale*scale, wgrad with g_scale*x_scale, then the lag update of g.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import (amax as _amax, quantize, scale_from_amax, transpose_u8, gemm,
               gemm_entries)

F32 = np.float32
_448 = F32(448.0)


@dataclass
class Meta:
    update_interval: int = 16
    scale: np.float32 = F32(1.0)
    scale_inv: np.float32 = F32(1.0)
    x_scale: np.float32 = F32(1.0)
    x_scale_inv: np.float32 = F32(1.0)
    g_scale: np.float32 = F32(1.0)
    g_scale_inv: np.float32 = F32(1.0)
    idx: int = 0
    amax_history: np.ndarray = field(default=None)

    def __post_init__(self):
        if self.amax_history is None:
            self.amax_history = np.ones(self.update_interval, np.float32)

    def record(self, amax) -> None:
        self.amax_history[self.idx] = F32(amax)
        self.idx = (self.idx + 1) % self.amax_history.size

    def refresh(self) -> None:
        m = self.amax_history.max()          # NaN-propagating max, as torch's
        if m > 0:
            self.scale = F32(m / _448)
            self.scale_inv = F32(_448 / m)

    def snapshot(self) -> dict:
        return dict(scale=self.scale, scale_inv=self.scale_inv, x_scale=self.x_scale,
                    x_scale_inv=self.x_scale_inv, g_scale=self.g_scale,
                    g_scale_inv=self.g_scale_inv, idx=self.idx,
                    amax_history=self.amax_history.copy())


@dataclass
class State:
    update_interval: int = 16
    step_count: int = 0
    metas: list = field(default_factory=list)

    def new_meta(self) -> Meta:
        m = Meta(self.update_interval)
        self.metas.append(m)
        return m

    def step(self) -> None:
        self.step_count += 1
        if self.step_count % self.update_interval == 0:
            for m in self.metas:
                m.refresh()


def lag_update(amax):
    """_update_delayed_scale: returns (scale, scale_inv) for the next call."""
    return scale_from_amax(amax)


def _gemm_out(A, B, s_a, s_b, entries, bias=None):
    if entries is None:
        return gemm(A, B, s_a, s_b, bias)
    ii, jj = entries
    return gemm_entries(A, B, s_a, s_b, ii, jj, bias)


def linear_forward(meta: Meta, x, w, entries=None, bias=None) -> dict:
    """Delayed-scaling forward.  x [M,K] and w [N,K] are bf16 bit patterns.
    entries=(ii, jj) limits the GEMM to those outputs."""
    used = dict(x_scale=meta.x_scale, x_scale_inv=meta.x_scale_inv,
                w_scale=meta.scale, w_scale_inv=meta.scale_inv)
    xq, amax_x = quantize(x, meta.x_scale_inv)
    wq, amax_w = quantize(w, meta.scale_inv)
    y = _gemm_out(xq, wq, meta.x_scale, meta.scale, entries, bias)
    meta.record(amax_w)
    meta.x_scale, meta.x_scale_inv = lag_update(amax_x)
    return dict(xq=xq, wq=wq, amax_x=amax_x, amax_w=amax_w, y=y, used=used)


def linear_backward(meta: Meta, g, x, w, entries_dx=None, entries_dw=None,
                    need=(True, True), saved=None) -> dict:
    """Delayed-scaling backward.  g [M,N]; need = (dX, dW).

    saved = (xq, x_scale) kept by the forward: the torchao float8 behaviour
    the SpecForge page ("Add training.fp8_linear", notes under the end-to-end
    table) credits for its memory saving, float8 activations saved for
    backward.  None re-quantises x with the current, just-updated x scale,
    as the AstrAI page's fp8_linear_backward does."""
    used = dict(g_scale=meta.g_scale, g_scale_inv=meta.g_scale_inv,
                w_scale=meta.scale, x_scale=meta.x_scale, x_scale_inv=meta.x_scale_inv)
    gq, amax_g = quantize(g, meta.g_scale_inv)
    wq, _ = quantize(w, meta.scale_inv)
    if saved is None:
        xq, _ = quantize(x, meta.x_scale_inv)
    else:
        xq, used["x_scale"] = saved
        used["x_scale_inv"] = None
    out = dict(gq=gq, amax_g=amax_g, xq_bwd=xq, used=used)
    if need[0]:
        # dX [M,K] = Gq [M,N] · Wq [N,K]: contraction over N, B operand = Wqᵀ [K,N]
        out["dx"] = _gemm_out(gq, transpose_u8(wq), meta.g_scale, meta.scale, entries_dx)
    if need[1]:
        # dW [N,K] = Gqᵀ [N,M] · Xq [M,K]: contraction over M
        out["dw"] = _gemm_out(transpose_u8(gq), transpose_u8(xq), meta.g_scale,
                              used["x_scale"], entries_dw)
    meta.g_scale, meta.g_scale_inv = lag_update(amax_g)
    return out


def delayed_training_step(state: State, meta: Meta, x, w, g, entries=None,
                          save_xq_fwd: bool = False) -> dict:
    """One training step: step() at autocast entry, forward, backward.
    entries = dict(y=(ii,jj), dx=(ii,jj), dw=(ii,jj)) or None for full.
    save_xq_fwd: the backward uses the forward's Xq and x scale (see
    linear_backward)."""
    state.step()
    e = entries or {}
    fwd = linear_forward(meta, x, w, e.get("y"))
    saved = (fwd["xq"], fwd["used"]["x_scale"]) if save_xq_fwd else None
    bwd = linear_backward(meta, g, x, w, e.get("dx"), e.get("dw"), saved=saved)
    return dict(fwd=fwd, bwd=bwd, step_count=state.step_count, meta=meta.snapshot())


def dynamic_linear_step(x, w, g, entries=None) -> dict:
    """Current (dynamic tensorwise) scaling: every tensor takes its scale from
    its own amax of this call, the lag rule applied to the current amax."""
    e = entries or {}
    out = {}
    for name, t in (("x", x), ("w", w), ("g", g)):
        a = _amax(t)
        s, si = scale_from_amax(a)
        q, _ = quantize(t, si)
        out[name] = dict(q=q, amax=a, scale=s, scale_inv=si)
    X, W, G = out["x"], out["w"], out["g"]
    out["y"] = _gemm_out(X["q"], W["q"], X["scale"], W["scale"], e.get("y"))
    out["dx"] = _gemm_out(G["q"], transpose_u8(W["q"]), G["scale"], W["scale"], e.get("dx"))
    out["dw"] = _gemm_out(transpose_u8(G["q"]), transpose_u8(X["q"]), G["scale"], X["scale"],
                          e.get("dw"))
    return out
