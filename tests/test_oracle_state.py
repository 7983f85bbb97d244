"""Pins for the oracle's delayed-scaling state machine.

Expected values are worked out by hand from the AstrAI page
"astrai/extension/fp8_state.py": FP8TensorMeta starts every scale and every
history slot at 1, record() writes slot idx and advances it, refresh() takes
the window max and skips non-positive maxima, FP8State.step() refreshes when
the step count is a multiple of update_interval (16), and
_update_delayed_scale() sets the x/g scale for the next call.  The NeMo
SALMAutomodel review warns that entering the autocast twice per step adds an
extra update; one test shows that the state machine sees that difference.
"""
import json
import os

import numpy as np

import oracle
import synth
from oracle.state import Meta, State, linear_forward, linear_backward, delayed_training_step

F = np.float32
GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def test_meta_initial_state_matches_page():
    m = Meta()
    assert m.update_interval == GOLDEN["update_interval_default"]["value"] == 16
    one = GOLDEN["meta_init_value"]["value"]
    assert m.amax_history.shape == (16,) and np.all(m.amax_history == one)
    assert m.scale == m.scale_inv == m.x_scale == m.x_scale_inv == m.g_scale == m.g_scale_inv == one
    assert m.idx == 0


def test_history_window_lags_and_keeps_the_initial_one_until_step_32():
    """Record 0.1 every step.  Steps 1..15 keep scale 1 (no refresh yet).  The
    refresh at step 16 runs before that step's record, so slot 15 still holds
    the initial 1.0 and the window max is 1: scale = 1/448.  At step 32 the
    window holds only 0.1s: scale = 0.1/448."""
    st = State(16)
    m = st.new_meta()
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
    st = State(4)
    m = st.new_meta()
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
    st = State(2)
    m = st.new_meta()
    m.record(F(0.0)); m.record(F(0.0))
    m.scale, m.scale_inv = F(0.5), F(2.0)
    st.step(); st.step()
    assert (m.scale, m.scale_inv) == (F(0.5), F(2.0))


def test_refresh_touches_every_meta():
    st = State(2)
    a, b = st.new_meta(), st.new_meta()
    a.record(F(2.0)); a.record(F(1.0))
    b.record(F(4.0)); b.record(F(8.0))
    st.step(); st.step()
    assert a.scale == F(2.0) / F(448.0) and b.scale == F(8.0) / F(448.0)


def test_x_and_g_scales_lag_one_call():
    m = Meta()
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
    m = Meta()
    x = np.zeros((16, 32), np.uint16)
    w = synth.normal_bf16((16, 32), 0.02, seed=2, tensor="w")
    linear_forward(m, x, w)
    assert m.x_scale == F(1e-12) / F(448.0) and m.x_scale_inv == F(448.0) / F(1e-12)


def test_one_step_per_training_step_and_the_reentry_hazard():
    """Entering the autocast once per training step refreshes at step 16;
    entering it twice (forward and backward wrapped) refreshes at step 8,
    which changes the weight scale used by steps 8..15."""
    def run(entries_per_step):
        st = State(16)
        m = st.new_meta()
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


def test_delayed_training_step_end_to_end_small():
    st = State(16)
    m = st.new_meta()
    M, K, N = 32, 64, 48
    w = synth.normal_bf16((N, K), 0.02, seed=0, tensor="w")
    for t in range(3):
        x = synth.normal_bf16((M, K), 1.0, seed=0, tensor="x", step=t)
        g = synth.normal_bf16((M, N), 1e-3, seed=0, tensor="g", step=t)
        out = delayed_training_step(st, m, x, w, g)
        y, yb, yb_bound = out["fwd"]["y"]
        assert y.shape == (M, N)
        assert out["bwd"]["dx"][0].shape == (M, K) and out["bwd"]["dw"][0].shape == (N, K)
    assert st.step_count == 3


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
        st = State(16)
        m = st.new_meta()
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
        st = State(16)
        m = st.new_meta()
        delayed_training_step(st, m, x0, w, g)
        outs[save] = delayed_training_step(st, m, x2, w, g, save_xq_fwd=save)
    assert np.array_equal(outs[True]["bwd"]["xq_bwd"], outs[True]["fwd"]["xq"])
    assert not np.array_equal(outs[False]["bwd"]["xq_bwd"], outs[True]["bwd"]["xq_bwd"])
