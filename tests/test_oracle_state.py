"""Pins for the oracle's delayed-scaling state and its step drivers.

Expected values are worked out by hand from the rules of the AstrAI page
"astrai/extension/fp8_state.py" (weight-meta class, global state class,
delayed-scale update, forward and backward functions): every scale pair and
every window slot starts at 1, each forward adds the weight amax to a window
of 16, the window max (when > 0) sets the weight pair when the step count
reaches a multiple of 16, and the x/g pairs come from the previous call's
amax.  The NeMo SALMAutomodel review warns that entering the autocast twice
per step adds an extra update; one test shows that the state sees that
difference.  The GEMM wiring of the step drivers (which operand, which
transpose, which pair of scales) is pinned against a product computed
independently: torch's own e4m3 decode and an fp64 matmul, with the scale
pairs derived from numpy amaxes and torch fp32 divisions.
"""
import json
import os

import numpy as np

import oracle
import synth
from oracle.state import (WeightScaling, StepCounter, linear_forward, linear_backward,
                          delayed_training_step)

F = np.float32
GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def test_meta_initial_state_matches_page():
    m = WeightScaling()
    assert m.interval == GOLDEN["update_interval_default"]["value"] == 16
    one = GOLDEN["meta_init_value"]["value"]
    assert m.amax_history.shape == (16,) and np.all(m.amax_history == one)
    assert m.scale == m.scale_inv == m.x_scale == m.x_scale_inv == m.g_scale == m.g_scale_inv == one
    assert m.idx == 0


def test_history_window_lags_and_keeps_the_initial_one_until_step_32():
    """Record 0.1 every step.  Steps 1..15 keep scale 1 (no refresh yet).  The
    refresh at step 16 runs before that step's record, so slot 15 still holds
    the initial 1.0 and the window max is 1: scale = 1/448.  At step 32 the
    window holds only 0.1s: scale = 0.1/448."""
    st = StepCounter(16)
    m = st.new_weight()
    a = F(0.1)
    seen = {}
    for t in range(1, 41):
        st.step()
        seen[t] = (m.scale, m.scale_inv)
        m.record(a)
    for t in range(1, 16):
        assert seen[t] == (F(1.0), F(1.0))
    assert seen[16] == (F(1.0) / F(448.0), F(448.0) / F(1.0))
    for t in range(17, 32):
        assert seen[t] == seen[16]
    assert seen[32] == (a / F(448.0), F(448.0) / a)
    assert seen[40] == seen[32]
    assert m.idx == 40 % 16


def test_history_wraps_and_takes_the_window_max():
    st = StepCounter(4)
    m = st.new_weight()
    for v in [3.0, 0.5, 0.25, 0.125]:
        m.record(F(v))
    st.step(); st.step(); st.step(); st.step()          # refresh at step 4
    assert m.scale == F(3.0) / F(448.0)
    m.record(F(0.75))                                   # overwrites the 3.0 (slot 0)
    assert m.amax_history[0] == F(0.75) and m.idx == 1
    for _ in range(4):
        st.step()                                       # refresh at step 8
    assert m.scale == F(0.75) / F(448.0) and m.scale_inv == F(448.0) / F(0.75)


def test_refresh_skips_a_zero_window():
    """A window max of 224 sets the pair (0.5, 2); a later window of zeros
    is skipped and the pair stays."""
    st = StepCounter(2)
    m = st.new_weight()
    m.record(F(224.0)); m.record(F(224.0))
    st.step(); st.step()
    assert (m.scale, m.scale_inv) == (F(0.5), F(2.0))
    m.record(F(0.0)); m.record(F(0.0))
    st.step(); st.step()
    assert np.all(m.amax_history == 0)
    assert (m.scale, m.scale_inv) == (F(0.5), F(2.0))


def test_refresh_touches_every_meta():
    st = StepCounter(2)
    a, b = st.new_weight(), st.new_weight()
    a.record(F(2.0)); a.record(F(1.0))
    b.record(F(4.0)); b.record(F(8.0))
    st.step(); st.step()
    assert a.scale == F(2.0) / F(448.0) and b.scale == F(8.0) / F(448.0)


def test_x_and_g_scales_lag_one_call():
    m = WeightScaling()
    w = synth.normal_bf16((16, 32), 0.02, seed=1, tensor="w")
    amax_seen = []
    for step in range(3):
        x = synth.normal_bf16((16, 32), 1.0 + step, seed=1, tensor="x", step=step)
        g = synth.normal_bf16((16, 16), 1e-3, seed=1, tensor="g", step=step)
        f = linear_forward(m, x, w)
        if step == 0:
            assert f["used"]["x_scale"] == F(1.0) and f["used"]["x_scale_inv"] == F(1.0)
        else:
            prev = amax_seen[-1][0]
            assert f["used"]["x_scale"] == prev / F(448.0)
            assert f["used"]["x_scale_inv"] == F(448.0) / prev
        # backward re-quantises x with the scale the forward just set
        b = linear_backward(m, g, x, w)
        assert b["used"]["x_scale"] == f["amax_x"] / F(448.0)
        if step == 0:
            assert b["used"]["g_scale"] == F(1.0)
        else:
            assert b["used"]["g_scale"] == amax_seen[-1][1] / F(448.0)
        amax_seen.append((f["amax_x"], b["amax_g"]))
        assert f["amax_x"] == oracle.amax(x) and b["amax_g"] == oracle.amax(g)
    assert m.idx == 3 and np.all(m.amax_history[:3] == oracle.amax(w))


def test_lag_update_clamps_a_zero_amax():
    m = WeightScaling()
    x = np.zeros((16, 32), np.uint16)
    w = synth.normal_bf16((16, 32), 0.02, seed=2, tensor="w")
    linear_forward(m, x, w)
    assert m.x_scale == F(1e-12) / F(448.0) and m.x_scale_inv == F(448.0) / F(1e-12)


def test_one_step_per_training_step_and_the_reentry_hazard():
    """Entering the autocast once per training step refreshes at step 16;
    entering it twice (forward and backward wrapped) refreshes at step 8,
    which changes the weight scale used by steps 8..15."""
    def run(entries_per_step):
        st = StepCounter(16)
        m = st.new_weight()
        scales = []
        for t in range(16):
            for _ in range(entries_per_step):
                st.step()
            scales.append(m.scale)
            m.record(F(0.1))
        return scales
    once, twice = run(1), run(2)
    assert all(s == F(1.0) for s in once[:15])
    assert twice[7] == F(1.0) / F(448.0)   # refreshed early: window still held ones
    assert once[7] == F(1.0)


def test_saved_forward_xq_agrees_when_the_x_scale_does_not_move():
    """Backward with the forward's saved Xq (the float8-activations-saved-for-
    backward behaviour of the SpecForge page) against the AstrAI page's
    re-quantisation: the two differ only through the x scale, so when this
    step's x has the same amax as the previous step's (the lag update then
    writes back the same scale) every byte and every dW entry agrees; when
    the amax moves, the re-quantised Xq follows the new scale and the saved
    one does not."""
    M, K, N = 48, 64, 32
    w = synth.normal_bf16((N, K), 0.02, seed=1, tensor="w")
    x0 = synth.normal_bf16((M, K), 1.0, seed=1, tensor="x", step=0)
    g = synth.normal_bf16((M, N), 1e-3, seed=1, tensor="g", step=1)
    # x1: a row permutation of x0 (same amax) -> the x scale does not move
    x1 = np.ascontiguousarray(x0[::-1])
    runs = {}
    for save in (False, True):
        st = StepCounter(16)
        m = st.new_weight()
        delayed_training_step(st, m, x0, w, g)
        runs[save] = delayed_training_step(st, m, x1, w, g, save_xq_fwd=save)
    a, b = runs[False]["bwd"], runs[True]["bwd"]
    assert np.array_equal(a["xq_bwd"], b["xq_bwd"])
    assert np.array_equal(a["dw"][0], b["dw"][0]) and np.array_equal(a["dx"][0], b["dx"][0])
    assert b["used"]["x_scale"] == runs[True]["fwd"]["used"]["x_scale"]
    # a step whose amax differs: the saved Xq keeps the forward scale
    x2 = synth.normal_bf16((M, K), 3.0, seed=1, tensor="x", step=2)
    outs = {}
    for save in (False, True):
        st = StepCounter(16)
        m = st.new_weight()
        delayed_training_step(st, m, x0, w, g)
        outs[save] = delayed_training_step(st, m, x2, w, g, save_xq_fwd=save)
    assert np.array_equal(outs[True]["bwd"]["xq_bwd"], outs[True]["fwd"]["xq"])
    assert not np.array_equal(outs[False]["bwd"]["xq_bwd"], outs[True]["bwd"]["xq_bwd"])


# ------------------------------------------ GEMM wiring, pinned independently

import pytest  # noqa: E402
import torch  # noqa: E402

from oracle import state as ost  # noqa: E402


def _f32(h):
    """bf16 bit patterns -> fp32 values (the exact widening, by bit shift)."""
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _np_amax(h):
    return F(np.max(np.abs(_f32(h))))


def _np_pair(a):
    """(a/448, 448/a) by numpy fp32 division, a clamped at 1e-12."""
    a = max(F(a), F(1e-12))
    return F(a) / F(448.0), F(448.0) / F(a)


def _dec(q):
    """e4m3 codes -> fp64 through torch's own float8_e4m3fn type."""
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64)


def _codes(h, scale_inv):
    """torch's e4m3 cast of fl32(x * scale_inv), clamped to +-448 first."""
    v = torch.from_numpy(_f32(h) * F(scale_inv)).clamp(-448.0, 448.0)
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _independent(a_dec, b_dec, s_a, s_b):
    """(s_a s_b A·B, s_a s_b |A|·|B|) in fp64 for A [R,k], B [k,C]."""
    s = float(s_a) * float(s_b)
    return (s * (a_dec @ b_dec)).numpy(), (s * (a_dec.abs() @ b_dec.abs())).numpy()


def _matches(oracle_out, indep):
    d, _, _ = oracle_out
    want, mag = indep
    return d.shape == want.shape and bool(np.all(np.abs(d - want) <= 1e-12 * mag))


def _two_steps(M, N, K, seed, save=False):
    """Two delayed steps with refresh interval 2, so that the second step has
    a refreshed weight pair, a lagged x pair and a lagged g pair that all
    differ from 1 and from one another.  W ~ N(0,1) puts amax_w above the
    window's initial 1.0."""
    w = synth.normal_bf16((N, K), 1.0, seed, "w")
    xs = [synth.normal_bf16((M, K), s, seed, "x", t) for t, s in enumerate((1.0, 2.5))]
    gs = [synth.normal_bf16((M, N), s, seed, "g", t) for t, s in enumerate((1e-3, 3e-3))]
    st = StepCounter(2)
    m = st.new_weight()
    delayed_training_step(st, m, xs[0], w, gs[0], save_xq_fwd=save)
    out = delayed_training_step(st, m, xs[1], w, gs[1], save_xq_fwd=save)
    return w, xs, gs, out


@pytest.mark.parametrize("save", [False, True])
def test_delayed_step_gemm_wiring_against_an_independent_product(save):
    M, N, K = 48, 80, 112
    w, xs, gs, out = _two_steps(M, N, K, 5, save)
    f, b = out["fwd"], out["bwd"]
    # the pairs the rules give for step 2
    w_pair = _np_pair(max(_np_amax(w), F(1.0)))      # refresh over [amax_w, 1.0]
    assert _np_amax(w) > 1.0
    x_fwd = _np_pair(_np_amax(xs[0]))                # lagged from step 1
    x_bwd = x_fwd if save else _np_pair(_np_amax(xs[1]))
    g_pair = _np_pair(_np_amax(gs[0]))               # lagged from step 1
    assert f["used"]["w_scale"] == w_pair[0] and f["used"]["x_scale"] == x_fwd[0]
    assert b["used"]["g_scale"] == g_pair[0] and b["used"]["x_scale"] == x_bwd[0]
    # the codes are the casts with those pairs
    assert np.array_equal(f["xq"], _codes(xs[1], x_fwd[1]))
    assert np.array_equal(f["wq"], _codes(w, w_pair[1]))
    assert np.array_equal(b["gq"], _codes(gs[1], g_pair[1]))
    xq_b = f["xq"] if save else _codes(xs[1], x_bwd[1])
    assert np.array_equal(b["xq_bwd"], xq_b)
    X, W, G = _dec(f["xq"]), _dec(f["wq"]), _dec(b["gq"])
    Xb = _dec(xq_b)
    assert _matches(f["y"], _independent(X, W.T, x_fwd[0], w_pair[0]))      # Y = X Wᵀ
    assert _matches(b["dx"], _independent(G, W, g_pair[0], w_pair[0]))     # dX = G W
    assert _matches(b["dw"], _independent(G.T, Xb, g_pair[0], x_bwd[0]))    # dW = Gᵀ X


def test_dynamic_step_gemm_wiring_against_an_independent_product():
    M, N, K = 48, 80, 112
    x = synth.normal_bf16((M, K), 1.0, 6, "x")
    w = synth.normal_bf16((N, K), 0.02, 6, "w")
    g = synth.normal_bf16((M, N), 1e-3, 6, "g")
    ref = ost.dynamic_linear_step(x, w, g)
    pairs = {n: _np_pair(_np_amax(h)) for n, h in (("x", x), ("w", w), ("g", g))}
    for n, h in (("x", x), ("w", w), ("g", g)):
        assert (ref[n]["scale"], ref[n]["scale_inv"]) == pairs[n]
        assert np.array_equal(ref[n]["q"], _codes(h, pairs[n][1]))
    X, W, G = _dec(ref["x"]["q"]), _dec(ref["w"]["q"]), _dec(ref["g"]["q"])
    assert _matches(ref["y"], _independent(X, W.T, pairs["x"][0], pairs["w"][0]))
    assert _matches(ref["dx"], _independent(G, W, pairs["g"][0], pairs["w"][0]))
    assert _matches(ref["dw"], _independent(G.T, X, pairs["g"][0], pairs["x"][0]))


def test_the_wiring_pin_rejects_plausible_mistakes(monkeypatch):
    """N = K, so the mistakes below are shape-valid and only the values can
    catch them: Wq passed un-transposed to dgrad (planted in the oracle's
    operand helper), dW scaled by the weight scale instead of the x scale,
    and dX scaled by the g pair of the wrong step."""
    M, N, K = 48, 80, 80
    w, xs, gs, out = _two_steps(M, N, K, 7)
    f, b = out["fwd"], out["bwd"]
    w_pair = _np_pair(max(_np_amax(w), F(1.0)))
    x_bwd, g_pair = _np_pair(_np_amax(xs[1])), _np_pair(_np_amax(gs[0]))
    X, W, G = _dec(b["xq_bwd"]), _dec(f["wq"]), _dec(b["gq"])
    want_dx = _independent(G, W, g_pair[0], w_pair[0])
    want_dw = _independent(G.T, X, g_pair[0], x_bwd[0])
    assert _matches(b["dx"], want_dx) and _matches(b["dw"], want_dw)
    # 1. un-transposed Wq, planted in the oracle
    monkeypatch.setattr(ost, "dgrad_operands", lambda gq, wq: (gq, wq))
    st = StepCounter(2)
    m = st.new_weight()
    delayed_training_step(st, m, xs[0], w, gs[0])
    bad = delayed_training_step(st, m, xs[1], w, gs[1])["bwd"]
    monkeypatch.undo()
    assert bad["dx"][0].shape == want_dx[0].shape
    assert not _matches(bad["dx"], want_dx)
    # 2. dW with the weight scale
    wrong = oracle.gemm(*ost.wgrad_operands(b["gq"], b["xq_bwd"]), g_pair[0], w_pair[0])
    assert not _matches(wrong, want_dw)
    # 3. dX with the g pair of this step's own amax (one step too late)
    late = _np_pair(_np_amax(gs[1]))
    wrong = oracle.gemm(*ost.dgrad_operands(b["gq"], f["wq"]), late[0], w_pair[0])
    assert not _matches(wrong, want_dx)


def _bf16_round(v32):
    return torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.bfloat16) \
        .to(torch.float64).numpy()


def test_derived_bound_accepts_fp32_accumulation_and_rejects_a_lagged_g_scale():
    """The derived GEMM bound (oracle.gemm_derived_ok) against an fp32
    emulation of the GPU arithmetic (exact e4m3 products summed in fp32 by
    numpy's matmul, one fp32 multiply by fl32(s_a s_b), bf16 rounding): the
    right g pair passes everywhere; the g pair of the step before (the amax
    two steps back) fails.  G's sigma changes every step, as in the GPU step
    tests, so the pairs of consecutive steps differ by a factor 1.5-3.  The
    stated tolerance is too loose to see that at these magnitudes."""
    M, N, K = 64, 96, 128
    w = synth.normal_bf16((N, K), 0.02, 8, "w")
    st = StepCounter(16)
    m = st.new_weight()
    amax_g = []
    for t in range(4):
        x = synth.normal_bf16((M, K), 1.0, 8, "x", t)
        g = synth.normal_bf16((M, N), 1e-3 * (1 + t % 3), 8, "g", t)
        out = delayed_training_step(st, m, x, w, g)
        f, b = out["fwd"], out["bwd"]
        amax_g.append(b["amax_g"])
        G32 = _dec(b["gq"]).to(torch.float32).numpy()
        W32 = _dec(f["wq"]).to(torch.float32).numpy()
        s_w = b["used"]["w_scale"]
        _, ref_b, bound = b["dx"]

        def emulate(g_scale):
            acc = np.matmul(G32, W32)            # fp32 sums of exact products
            return _bf16_round(acc * F(F(g_scale) * F(s_w)))
        assert oracle.gemm_derived_ok(emulate(b["used"]["g_scale"]), ref_b, bound, N).all()
        assert oracle.gemm_derived_ok(ref_b, ref_b, bound, N).all()
        if t >= 2:
            prev = _np_pair(amax_g[t - 2])[0]     # the pair one step too old
            assert prev != b["used"]["g_scale"]
            # all but the entries that cancel to almost nothing are rejected
            assert oracle.gemm_derived_ok(emulate(prev), ref_b, bound, N).mean() < 0.02
