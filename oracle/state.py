"""Delayed and current scaling of one FP8 linear, and whole-step drivers.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Rules (AstrAI page "astrai/extension/fp8_state.py": the module docstring, the
comment on the GEMM layout, the weight-meta class, the global state class,
the delayed-scale update and the forward/backward functions), restated:

* Every scale is a pair (scale, scale_inv) of fp32 values, scale = a/448 and
  scale_inv = 448/a for some amax a.  All pairs start at (1, 1).
* Weight: each forward appends the weight's amax to a window of the last
  ``interval`` values; the window starts out filled with 1.0.  The weight pair
  changes only at a refresh, which takes the window's maximum m and, when
  m > 0, sets the pair from m; otherwise the pair is kept.
* Refreshes happen when a training step begins and the step count, advanced
  once per step, is a multiple of ``interval`` (16).  A second advance in the
  same step (entering the autocast context around backward too) would move
  the refresh earlier; the NeMo review on the SALMAutomodel FP8 page warns
  about that extra update.
* Activation x and gradient g: the pair used by a call comes from the amax
  the previous call of the same linear produced, a = max(amax, 1e-12).
* Forward: x quantised with the x pair, w with the weight pair, Y scaled by
  x_scale * w_scale; then the weight amax joins the window and the x pair
  moves to this call's amax.  Backward: g quantised with the g pair, w and x
  quantised again (x with the pair the forward has just set), dX scaled by
  g_scale * w_scale, dW by g_scale * x_scale; then the g pair moves.

Structure: ``WeightScaling`` keeps only logs (every weight amax recorded,
the number of records at each refresh, the last x and g amax); every scale
and the slot layout of the window are computed from those logs by the pure
functions below, so each can be checked against the rules on its own.
"""
from __future__ import annotations

import numpy as np

from . import (amax as _amax, quantize, scale_from_amax, transpose_u8, gemm,
               gemm_entries)

F32 = np.float32
UNIT = (F32(1.0), F32(1.0))


# ------------------------------------------------------ pure functions ---

def pair_from(a) -> tuple:
    """(a/448, 448/a) with a = max(a, 1e-12), correctly rounded fp32."""
    return scale_from_amax(a)


def window_values(w_log, interval: int) -> np.ndarray:
    """The values the window holds after the records in ``w_log``: the last
    ``interval`` records, plus the initial 1.0 in every slot no record has
    reached yet (in no particular order)."""
    recent = [F32(v) for v in list(w_log)[-interval:]]
    return np.array(recent + [F32(1.0)] * (interval - len(recent)), np.float32)


def window_slots(w_log, interval: int) -> np.ndarray:
    """The window in slot order, as a device ring holds it: record number r
    (0-based) lands in slot r mod interval, slots never written hold 1.0."""
    slots = np.ones(interval, np.float32)
    for r, v in enumerate(w_log):
        slots[r % interval] = F32(v)
    return slots


def refreshed_pair(window: np.ndarray, current: tuple) -> tuple:
    """A refresh: the window max m sets the pair when m > 0 (a NaN max is not
    > 0 and keeps the pair)."""
    m = F32(np.max(window))
    if m > 0:
        return F32(m / F32(448.0)), F32(F32(448.0) / m)
    return current


def weight_pair(w_log, refresh_counts, interval: int) -> tuple:
    """The weight pair after the refreshes, each of which saw the first
    ``refresh_counts[i]`` records of ``w_log``."""
    pair = UNIT
    for n in refresh_counts:
        pair = refreshed_pair(window_values(list(w_log)[:n], interval), pair)
    return pair


def lagged_pair(prev_amax) -> tuple:
    """The x or g pair of a call: from the previous call's amax, (1, 1) before
    the first call."""
    return UNIT if prev_amax is None else pair_from(prev_amax)


# ---------------------------------------------------------- the state ---

class WeightScaling:
    """The scaling state of one weight and its paired activation and
    gradient, kept as logs."""

    def __init__(self, interval: int = 16):
        self.interval = interval
        self.w_log = []            # weight amaxes, oldest first
        self.refresh_counts = []   # len(w_log) at each refresh
        self.x_amax = None         # amax of the last call's x
        self.g_amax = None         # amax of the last call's g

    # derived values
    @property
    def w_pair(self):
        return weight_pair(self.w_log, self.refresh_counts, self.interval)

    @property
    def x_pair(self):
        return lagged_pair(self.x_amax)

    @property
    def g_pair(self):
        return lagged_pair(self.g_amax)

    scale = property(lambda self: self.w_pair[0])
    scale_inv = property(lambda self: self.w_pair[1])
    x_scale = property(lambda self: self.x_pair[0])
    x_scale_inv = property(lambda self: self.x_pair[1])
    g_scale = property(lambda self: self.g_pair[0])
    g_scale_inv = property(lambda self: self.g_pair[1])

    @property
    def amax_history(self) -> np.ndarray:
        return window_slots(self.w_log, self.interval)

    @property
    def idx(self) -> int:
        """The slot the next record goes to."""
        return len(self.w_log) % self.interval

    # events
    def record(self, amax_w) -> None:
        self.w_log.append(F32(amax_w))

    def note_x(self, amax_x) -> None:
        self.x_amax = F32(amax_x)

    def note_g(self, amax_g) -> None:
        self.g_amax = F32(amax_g)

    def snapshot(self) -> dict:
        s, si = self.w_pair
        xs, xsi = self.x_pair
        gs, gsi = self.g_pair
        return dict(scale=s, scale_inv=si, x_scale=xs, x_scale_inv=xsi, g_scale=gs,
                    g_scale_inv=gsi, idx=self.idx, amax_history=self.amax_history)


class StepCounter:
    """The training-step count shared by every weight: ``step()`` once per
    training step, refreshing every weight when the count reaches a multiple
    of the interval."""

    def __init__(self, interval: int = 16):
        self.interval = interval
        self.step_count = 0
        self.weights = []

    def new_weight(self) -> WeightScaling:
        ws = WeightScaling(self.interval)
        self.weights.append(ws)
        return ws

    def step(self) -> None:
        self.step_count += 1
        if self.step_count % self.interval == 0:
            for ws in self.weights:
                ws.refresh_counts.append(len(ws.w_log))


# ------------------------------------------------------- the GEMM calls ---

def _gemm_out(A, B, s_a, s_b, entries, bias=None):
    if entries is None:
        return gemm(A, B, s_a, s_b, bias)
    ii, jj = entries
    return gemm_entries(A, B, s_a, s_b, ii, jj, bias)


def dgrad_operands(gq, wq):
    """dX [M,K] = Gq [M,N] · Wq [N,K]: A = Gq (rows M, contraction N),
    B = Wqᵀ [K,N] (rows K, contraction N)."""
    return gq, transpose_u8(wq)


def wgrad_operands(gq, xq):
    """dW [N,K] = Gqᵀ [N,M] · Xq [M,K]: A = Gqᵀ [N,M], B = Xqᵀ [K,M]
    (contraction over the M tokens)."""
    return transpose_u8(gq), transpose_u8(xq)


def linear_forward(ws: WeightScaling, x, w, entries=None, bias=None) -> dict:
    """Delayed-scaling forward.  x [M,K] and w [N,K] are bf16 bit patterns.
    entries=(ii, jj) limits the GEMM to those outputs."""
    (xs, xsi), (s, si) = ws.x_pair, ws.w_pair
    used = dict(x_scale=xs, x_scale_inv=xsi, w_scale=s, w_scale_inv=si)
    xq, amax_x = quantize(x, xsi)
    wq, amax_w = quantize(w, si)
    y = _gemm_out(xq, wq, xs, s, entries, bias)
    ws.record(amax_w)
    ws.note_x(amax_x)
    return dict(xq=xq, wq=wq, amax_x=amax_x, amax_w=amax_w, y=y, used=used)


def linear_backward(ws: WeightScaling, g, x, w, entries_dx=None, entries_dw=None,
                    need=(True, True), saved=None) -> dict:
    """Delayed-scaling backward.  g [M,N]; need = (dX, dW).

    saved = (xq, x_scale) kept by the forward: float8 activations saved for
    backward, the torchao behaviour the SpecForge page ("Add
    training.fp8_linear", notes under the end-to-end tables) credits for its
    memory saving.  None quantises x again with the x pair the forward has
    just set, as the AstrAI page's backward does."""
    (gs, gsi), (s, si), (xs, xsi) = ws.g_pair, ws.w_pair, ws.x_pair
    used = dict(g_scale=gs, g_scale_inv=gsi, w_scale=s, x_scale=xs, x_scale_inv=xsi)
    gq, amax_g = quantize(g, gsi)
    wq, _ = quantize(w, si)
    if saved is None:
        xq, _ = quantize(x, xsi)
    else:
        xq, used["x_scale"] = saved
        used["x_scale_inv"] = None
    out = dict(gq=gq, amax_g=amax_g, xq_bwd=xq, used=used)
    if need[0]:
        out["dx"] = _gemm_out(*dgrad_operands(gq, wq), gs, s, entries_dx)
    if need[1]:
        out["dw"] = _gemm_out(*wgrad_operands(gq, xq), gs, used["x_scale"], entries_dw)
    ws.note_g(amax_g)
    return out


def delayed_training_step(counter: StepCounter, ws: WeightScaling, x, w, g, entries=None,
                          save_xq_fwd: bool = False) -> dict:
    """One training step: the step count advances, then forward and backward.
    entries = dict(y=(ii,jj), dx=(ii,jj), dw=(ii,jj)) or None for full.
    save_xq_fwd: the backward uses the forward's Xq and x scale (see
    linear_backward)."""
    counter.step()
    e = entries or {}
    fwd = linear_forward(ws, x, w, e.get("y"))
    saved = (fwd["xq"], fwd["used"]["x_scale"]) if save_xq_fwd else None
    bwd = linear_backward(ws, g, x, w, e.get("dx"), e.get("dw"), saved=saved)
    return dict(fwd=fwd, bwd=bwd, step_count=counter.step_count, meta=ws.snapshot())


def dynamic_linear_step(x, w, g, entries=None) -> dict:
    """Current (dynamic tensorwise) scaling: every tensor takes its pair from
    its own amax of this call."""
    e = entries or {}
    out = {}
    for name, t in (("x", x), ("w", w), ("g", g)):
        a = _amax(t)
        s, si = pair_from(a)
        q, _ = quantize(t, si)
        out[name] = dict(q=q, amax=a, scale=s, scale_inv=si)
    X, W, G = out["x"], out["w"], out["g"]
    out["y"] = _gemm_out(X["q"], W["q"], X["scale"], W["scale"], e.get("y"))
    out["dx"] = _gemm_out(*dgrad_operands(G["q"], W["q"]), G["scale"], W["scale"], e.get("dx"))
    out["dw"] = _gemm_out(*wgrad_operands(G["q"], X["q"]), G["scale"], X["scale"], e.get("dw"))
    return out
