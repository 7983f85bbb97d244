"""End-to-end parity of the five workloads against the oracle, through the C ABI.

1. one FP8 linear fprop, dynamic tensorwise scaling, X [64,256], W [256,256];
2. one FP8 linear fwd+dgrad+wgrad under delayed scaling for 20 steps
   (16-step weight amax history, X/G scales lagged one call) — all 20 steps at
   512^3 with full comparison, and the first steps at the full 4096^3 size
   with full quantised bytes / scales and sampled GEMM outputs;
3. a transformer MLP block (tokens 16384, hidden 4096, FFN 14336), dynamic
   scaling, every projection fwd+dgrad+wgrad, sampled outputs;
4. a packed THD batch of 64 sequences (lengths 128..4096) zero-padded to a
   multiple of 16: padded rows change no amax and no real output;
5. the block-scaled recipe at M=32768, K=N=8192, inputs with 1% outliers x50.

Bytes, amaxes and scales must be bit-exact; GEMM outputs within the stated
tolerance |D - bf16(D_ref)| <= 1e-2 * s_A s_B sum|a||b| + 1e-3 and, where the
contraction length is passed, within the tighter bound derived from fp32
accumulation and bf16 rounding (oracle.gemm_derived_ok), which sees a scale
taken from the wrong step.  The delayed-scaling tests change G's sigma every
step (x1, x2, x3 in turn), so the g pairs of consecutive steps differ by a
factor 1.5-3 and a g scale read one step off fails the derived bound."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import state as ost
from helpers import dev_bf16, host_u8, f32, u8, bf16_out, first_diff

import scaled_linear_layers_gb300 as fp8

pytestmark = pytest.mark.gpu


def f32bits(v):
    return np.float32(v).view(np.uint32)


def check_gemm(got_full, ref_tuple, ii=None, jj=None, k=None):
    """The stated tolerance, and the derived bound when the contraction
    length k is given."""
    _, ref, bound = ref_tuple
    got = got_full if ii is None else got_full[ii, jj]
    ok = oracle.gemm_tolerance_ok(got, ref, bound)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance"
    if k is not None:
        ok = oracle.gemm_derived_ok(got, ref, bound, k)
        assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the derived bound (k={k})"


def g_sigma(t):
    """G's sigma at step t: 1e-3 times 1, 2, 3 in turn."""
    return synth.CONFIG2["g_sigma"] * (1 + t % 3)


def sample_entries(rng, R, C, n=2048, panels=2):
    rows = rng.choice(R, panels, replace=False)
    ii = np.concatenate([rng.integers(0, R, n), np.repeat(rows, C)])
    jj = np.concatenate([rng.integers(0, C, n), np.tile(np.arange(C), panels)])
    return ii, jj


# ------------------------------------------------------------ workload 1 ---

def test_config1_dynamic_fprop():
    c = synth.CONFIG1
    M, K, N = c["M"], c["K"], c["N"]
    x = synth.normal_bf16((M, K), c["x_sigma"], c["seed"], "x")
    w = synth.normal_bf16((N, K), c["w_sigma"], c["seed"], "w")
    qx, qw = u8(M, K), u8(N, K)
    sx, six, ax = f32(), f32(), f32()
    sw, siw, aw = f32(), f32(), f32()
    fp8.fp8_quantize(dev_bf16(x), fp8.DYNAMIC, sx, six, qx, ax)
    fp8.fp8_quantize(dev_bf16(w), fp8.DYNAMIC, sw, siw, qw, aw)
    y = bf16_out(M, N)
    fp8.fp8_linear_fprop(qx, sx, qw, sw, M, N, K, fp8.DYNAMIC, None, y)
    rx = oracle.quantize_dynamic(x)
    rw = oracle.quantize_dynamic(w)
    assert np.array_equal(host_u8(qx), rx[0]) and np.array_equal(host_u8(qw), rw[0])
    assert sx.item() == rx[1] and sw.item() == rw[1]
    check_gemm(y.float().cpu().numpy(), oracle.gemm(rx[0], rw[0], rx[1], rw[1]))


# ------------------------------------------------------------ workload 2 ---

class GpuDelayedLinear:
    """The delayed-scaling call sequence of one training step through the C ABI."""

    def __init__(self, M, N, K, w):
        self.M, self.N, self.K = M, N, K
        self.w = w
        self.meta = fp8.Fp8Meta(16)
        self.count = [0]
        self.xq, self.xqt = u8(M, K), u8(K, M)
        self.wq, self.wqt = u8(N, K), u8(K, N)
        self.gq, self.gqt = u8(M, N), u8(N, M)
        self.y, self.dx, self.dw = bf16_out(M, N), bf16_out(M, K), bf16_out(N, K)
        self.ax, self.aw, self.ag = f32(), f32(), f32()

    def step(self, x, g):
        m, M, N, K = self.meta, self.M, self.N, self.K
        fp8.fp8_state_step(self.count, 16, [m])
        used = dict(x_scale=m.x_scale.item(), x_scale_inv=m.x_scale_inv.item(),
                    w_scale=m.scale.item(), g_scale=m.g_scale.item())
        fp8.fp8_quantize(x, fp8.DELAYED, None, m.x_scale_inv, self.xq, self.ax)
        fp8.fp8_quantize_transpose(self.w, fp8.DELAYED, None, m.scale_inv, self.wq, self.wqt,
                                   amax_out=self.aw)
        fp8.fp8_linear_fprop(self.xq, m.x_scale, self.wq, m.scale, M, N, K, fp8.DELAYED, None,
                             self.y)
        fp8.fp8_meta_record(m, fp8.SLOT_W, self.aw)
        fp8.fp8_meta_record(m, fp8.SLOT_X, self.ax)
        fp8.fp8_quantize_transpose(g, fp8.DELAYED, None, m.g_scale_inv, self.gq, self.gqt,
                                   amax_out=self.ag)
        fp8.fp8_quantize_transpose(x, fp8.DELAYED, None, m.x_scale_inv, None, self.xqt)
        used["x_scale_bwd"] = m.x_scale.item()
        fp8.fp8_linear_dgrad(self.gq, m.g_scale, self.wqt, m.scale, M, N, K, fp8.DELAYED, self.dx)
        fp8.fp8_linear_wgrad(self.gqt, m.g_scale, self.xqt, m.x_scale, M, N, K, fp8.DELAYED,
                             self.dw)
        fp8.fp8_meta_record(m, fp8.SLOT_G, self.ag)
        fp8.fp8_check_device_status()
        return used


def run_delayed(M, N, K, steps, full_gemm, seed=0):
    c = synth.CONFIG2
    rng = np.random.default_rng(seed)
    w = synth.normal_bf16((N, K), c["w_sigma"], seed, "w")
    gpu = GpuDelayedLinear(M, N, K, dev_bf16(w))
    st = ost.StepCounter(16)
    meta = st.new_weight()
    for t in range(steps):
        x = synth.normal_bf16((M, K), c["x_sigma"], seed, "x", t)
        g = synth.normal_bf16((M, N), g_sigma(t), seed, "g", t)
        used = gpu.step(dev_bf16(x), dev_bf16(g))
        if full_gemm:
            entries = None
        else:
            entries = dict(y=sample_entries(rng, M, N), dx=sample_entries(rng, M, K),
                           dw=sample_entries(rng, N, K))
        ref = ost.delayed_training_step(st, meta, x, w, g, entries)
        f, b = ref["fwd"], ref["bwd"]
        # scales used by this step, bit for bit
        assert f32bits(used["x_scale"]) == f32bits(f["used"]["x_scale"]), t
        assert f32bits(used["w_scale"]) == f32bits(f["used"]["w_scale"]), t
        assert f32bits(used["g_scale"]) == f32bits(b["used"]["g_scale"]), t
        assert f32bits(used["x_scale_bwd"]) == f32bits(b["used"]["x_scale"]), t
        # bytes and amaxes
        assert np.array_equal(host_u8(gpu.xq), f["xq"]), first_diff(host_u8(gpu.xq), f["xq"])
        assert np.array_equal(host_u8(gpu.wq), f["wq"])
        # Wqᵀ (from the backward launch, as Wq's bytes transposed): the bytes
        # the page's second quantisation of W with the same scale gives
        assert np.array_equal(host_u8(gpu.wqt), f["wq"].T)
        assert np.array_equal(host_u8(gpu.gq), b["gq"])
        assert np.array_equal(host_u8(gpu.xqt), b["xq_bwd"].T)
        assert f32bits(gpu.ax.item()) == f32bits(f["amax_x"])
        assert f32bits(gpu.aw.item()) == f32bits(f["amax_w"])
        assert f32bits(gpu.ag.item()) == f32bits(b["amax_g"])
        # state after the step
        snap = ref["meta"]
        blk = gpu.meta.block.cpu().numpy()
        assert np.array_equal(blk[8:].view(np.uint32), snap["amax_history"].view(np.uint32))
        assert gpu.meta.idx == snap["idx"]
        for k, i in (("scale", 0), ("scale_inv", 1), ("x_scale", 2), ("x_scale_inv", 3),
                     ("g_scale", 4), ("g_scale_inv", 5)):
            assert f32bits(blk[i]) == f32bits(snap[k]), (t, k)
        # GEMMs
        for name, out, k in (("y", gpu.y, K), ("dx", gpu.dx, N), ("dw", gpu.dw, M)):
            got = out.float().cpu().numpy()
            src = f if name == "y" else b
            if full_gemm:
                check_gemm(got, src[name], k=k)
            else:
                ii, jj = entries[name]
                check_gemm(got, src[name], ii, jj, k=k)
    return st


def test_config2_delayed_20_steps_small():
    st = run_delayed(512, 512, 512, steps=20, full_gemm=True)
    assert st.step_count == 20


def test_config2_delayed_full_size_first_steps():
    run_delayed(4096, 4096, 4096, steps=2, full_gemm=False)


@pytest.mark.parametrize("shape", [(256, 384, 512), (272, 400, 528)])
def test_composite_step_matches_oracle_20_steps(shape):
    """fp8_linear_step_delayed (one native call per training step) against
    the oracle's state machine: all 20 steps, full compare, at 256x384x512
    and at a shape with partial 128-row and 128-column tiles in every
    quantised tensor (the byte transpose that makes Wqᵀ included)."""
    c = synth.CONFIG2
    M, N, K = shape
    w = synth.normal_bf16((N, K), c["w_sigma"], 7, "w")
    wd = dev_bf16(w)
    step = fp8.LinearStep(M, N, K)
    meta = fp8.Fp8Meta(16)
    count = [0]
    st = ost.StepCounter(16)
    om = st.new_weight()
    for t in range(20):
        x = synth.normal_bf16((M, K), c["x_sigma"], 7, "x", t)
        g = synth.normal_bf16((M, N), g_sigma(t), 7, "g", t)
        xd, gd = dev_bf16(x), dev_bf16(g)
        step.set_inputs(xd, wd, gd)
        fp8.fp8_linear_step_delayed(meta, count, step)
        fp8.fp8_check_device_status()
        ref = ost.delayed_training_step(st, om, x, w, g)
        f, b = ref["fwd"], ref["bwd"]
        assert count[0] == st.step_count == t + 1
        assert np.array_equal(host_u8(step.xq), f["xq"]) and np.array_equal(host_u8(step.wq), f["wq"])
        assert np.array_equal(host_u8(step.wqt), f["wq"].T)
        assert np.array_equal(host_u8(step.gq), b["gq"]) and np.array_equal(host_u8(step.gqt), b["gq"].T)
        assert np.array_equal(host_u8(step.xqt), b["xq_bwd"].T)
        am = step.amax.cpu().numpy()
        assert [f32bits(v) for v in am] == [f32bits(f["amax_x"]), f32bits(f["amax_w"]),
                                            f32bits(b["amax_g"])]
        blk = meta.block.cpu().numpy()
        snap = ref["meta"]
        assert np.array_equal(blk[8:].view(np.uint32), snap["amax_history"].view(np.uint32))
        for k, i in (("scale", 0), ("scale_inv", 1), ("x_scale", 2), ("x_scale_inv", 3),
                     ("g_scale", 4), ("g_scale_inv", 5)):
            assert f32bits(blk[i]) == f32bits(snap[k]), (t, k)
        check_gemm(step.y.float().cpu().numpy(), f["y"], k=K)
        check_gemm(step.dx.float().cpu().numpy(), b["dx"], k=N)
        check_gemm(step.dw.float().cpu().numpy(), b["dw"], k=M)


def test_composite_step_full_size_as_benchmarked():
    """The benchmark's own launch configuration: fp8_linear_step_delayed at
    M=N=K=4096 (fprop on the 2-SM kernel, dgrad and wgrad sharing one 2-SM
    launch, the state update and backward quantisation on the second stream)
    for 3 steps, against the oracle's state machine: every byte, amax and
    scale, and the GEMMs on sampled entries and full row panels."""
    c = synth.CONFIG2
    M = N = K = 4096
    w = synth.normal_bf16((N, K), c["w_sigma"], c["seed"], "w")
    wd = dev_bf16(w)
    step = fp8.LinearStep(M, N, K)
    meta = fp8.Fp8Meta(16)
    count = [0]
    st = ost.StepCounter(16)
    om = st.new_weight()
    rng = np.random.default_rng(3)
    for t in range(3):
        x = synth.normal_bf16((M, K), c["x_sigma"], c["seed"], "x", t)
        g = synth.normal_bf16((M, N), g_sigma(t), c["seed"], "g", t)
        step.set_inputs(dev_bf16(x), wd, dev_bf16(g))
        fp8.fp8_linear_step_delayed(meta, count, step)
        fp8.fp8_check_device_status()
        ent = dict(y=sample_entries(rng, M, N), dx=sample_entries(rng, M, K),
                   dw=sample_entries(rng, N, K))
        ref = ost.delayed_training_step(st, om, x, w, g, ent)
        f, b = ref["fwd"], ref["bwd"]
        assert np.array_equal(host_u8(step.xq), f["xq"]) and np.array_equal(host_u8(step.wq), f["wq"])
        assert np.array_equal(host_u8(step.gq), b["gq"])
        assert np.array_equal(host_u8(step.xqt), b["xq_bwd"].T)
        am = step.amax.cpu().numpy()
        assert [f32bits(v) for v in am] == [f32bits(f["amax_x"]), f32bits(f["amax_w"]),
                                            f32bits(b["amax_g"])]
        blk = meta.block.cpu().numpy()
        for k, i in (("scale", 0), ("x_scale", 2), ("g_scale", 4)):
            assert f32bits(blk[i]) == f32bits(ref["meta"][k]), (t, k)
        check_gemm(step.y.float().cpu().numpy(), f["y"], *ent["y"], k=K)
        check_gemm(step.dx.float().cpu().numpy(), b["dx"], *ent["dx"], k=N)
        check_gemm(step.dw.float().cpu().numpy(), b["dw"], *ent["dw"], k=M)


def test_composite_step_with_bias_and_bias_gradient():
    """The step with a bias (added in fprop's epilogue) and the bias gradient
    fused into G's quantisation (a padded token count: 3872 = 3858 rounded up
    to 16, the SpecForge page's example, G's pad rows zero)."""
    M, N, K = 3872, 256, 384
    w = synth.normal_bf16((N, K), 0.02, 9, "w")
    b = synth.normal_bf16((N,), 0.1, 9, "bias")
    wd, bd = dev_bf16(w), dev_bf16(b)
    step = fp8.LinearStep(M, N, K, bias=bd, dbias=True)
    meta = fp8.Fp8Meta(16)
    count = [0]
    st = ost.StepCounter(16)
    om = st.new_weight()
    rng = np.random.default_rng(9)
    for t in range(3):
        x = synth.normal_bf16((M, K), 1.0, 9, "x", t)
        g = synth.normal_bf16((M, N), 1e-3, 9, "g", t)
        g[3858:] = 0
        step.set_inputs(dev_bf16(x), wd, dev_bf16(g))
        fp8.fp8_linear_step_delayed(meta, count, step)
        fp8.fp8_check_device_status()
        st.step()
        ey, edx, edw = sample_entries(rng, M, N), sample_entries(rng, M, K), sample_entries(rng, N, K)
        f = ost.linear_forward(om, x, w, ey, bias=b)
        bw = ost.linear_backward(om, g, x, w, edx, edw)
        check_gemm(step.y.float().cpu().numpy()[ey], f["y"], k=K)
        check_gemm(step.dx.float().cpu().numpy()[edx], bw["dx"], k=N)
        check_gemm(step.dw.float().cpu().numpy()[edw], bw["dw"], k=M)
        _, ref_db, mag = oracle.bias_grad(g)
        got = step.dbias.float().cpu().numpy().astype(np.float64)
        assert oracle.bias_grad_tolerance_ok(got, ref_db, mag, M).all(), t
        # the same bits as the stand-alone fused entry point on the same G
        db2 = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        ws2 = torch.empty_like(step.dbias_workspace)
        fp8.fp8_quantize_transpose_dbias(dev_bf16(g), fp8.DELAYED, None,
                                         torch.ones(1, device="cuda"), u8(M, N), u8(N, M), db2,
                                         ws2)
        assert torch.equal(db2, step.dbias)


def test_composite_step_with_saved_forward_xq():
    """FP8_STEP_SAVE_XQ_FWD: the backward takes the forward's Xqᵀ and x scale
    (no second read of X) and matches the oracle's saved-Xq variant."""
    c = synth.CONFIG2
    M, N, K = 256, 384, 512
    w = synth.normal_bf16((N, K), c["w_sigma"], 11, "w")
    wd = dev_bf16(w)
    step = fp8.LinearStep(M, N, K, save_xq_fwd=True)
    meta = fp8.Fp8Meta(16)
    count = [0]
    st = ost.StepCounter(16)
    om = st.new_weight()
    for t in range(18):
        x = synth.normal_bf16((M, K), c["x_sigma"] * (1 + t % 3), 11, "x", t)
        g = synth.normal_bf16((M, N), g_sigma(t + 1), 11, "g", t)
        step.set_inputs(dev_bf16(x), wd, dev_bf16(g))
        fp8.fp8_linear_step_delayed(meta, count, step)
        fp8.fp8_check_device_status()
        ref = ost.delayed_training_step(st, om, x, w, g, save_xq_fwd=True)
        f, b = ref["fwd"], ref["bwd"]
        assert np.array_equal(host_u8(step.xq), f["xq"])
        assert np.array_equal(host_u8(step.xqt), f["xq"].T)
        assert np.array_equal(host_u8(step.gq), b["gq"])
        blk = meta.block.cpu().numpy()
        for k, i in (("scale", 0), ("x_scale", 2), ("g_scale", 4)):
            assert f32bits(blk[i]) == f32bits(ref["meta"][k]), (t, k)
        check_gemm(step.y.float().cpu().numpy(), f["y"], k=K)
        check_gemm(step.dx.float().cpu().numpy(), b["dx"], k=N)
        check_gemm(step.dw.float().cpu().numpy(), b["dw"], k=M)


def test_meta_checkpoint_restore_continues_bit_for_bit():
    """fp8_meta_save after 10 steps, fp8_meta_load into a fresh meta: the
    next 10 steps (across the step-16 refresh) give the same bits as the
    run that saved it."""
    c = synth.CONFIG2
    M, N, K = 256, 256, 256
    w = synth.normal_bf16((N, K), c["w_sigma"], 12, "w")
    wd = dev_bf16(w)
    xs = [dev_bf16(synth.normal_bf16((M, K), c["x_sigma"], 12, "x", t)) for t in range(20)]
    gs = [dev_bf16(synth.normal_bf16((M, N), c["g_sigma"], 12, "g", t)) for t in range(20)]

    def run(meta, count, step, ts):
        outs = []
        for t in ts:
            step.set_inputs(xs[t], wd, gs[t])
            fp8.fp8_linear_step_delayed(meta, count, step)
            outs.append([step.y.clone(), step.dx.clone(), step.dw.clone(), meta.block.clone()])
        fp8.fp8_check_device_status()
        return outs

    meta, count, step = fp8.Fp8Meta(16), [0], fp8.LinearStep(M, N, K)
    run(meta, count, step, range(10))
    blob = meta.save(count[0])
    first = run(meta, count, step, range(10, 20))
    meta2, cnt = fp8.Fp8Meta.load(blob)
    assert cnt == 10 and meta2.c.idx == 10 and meta2.c.interval == 16
    second = run(meta2, [cnt], fp8.LinearStep(M, N, K), range(10, 20))
    for a, b in zip(first, second):
        for ta, tb in zip(a, b):
            assert torch.equal(ta, tb)


@pytest.mark.parametrize("shape", [(256, 384, 512), (272, 400, 528), (2048, 4096, 1024)])
def test_dynamic_step_one_call(shape):
    """fp8_linear_step_dynamic against the oracle's current-scaling step: every
    byte, amax and scale bit for bit, the GEMMs within the tolerance (all
    entries at the small shape, sampled at the larger one, where dgrad and
    wgrad share a 2-SM launch); a second call on new inputs reuses the
    scratch."""
    M, N, K = shape
    st = fp8.DynamicStepState()
    step = fp8.LinearStep(M, N, K)
    rng = np.random.default_rng(M)
    w = synth.normal_bf16((N, K), 0.02, 21, "w")
    for t in range(2):
        x = synth.normal_bf16((M, K), 1.0, 21, "x", t)
        g = synth.normal_bf16((M, N), 1e-3, 21, "g", t)
        step.set_inputs(dev_bf16(x), dev_bf16(w), dev_bf16(g))
        fp8.fp8_linear_step_dynamic(st, step)
        fp8.fp8_check_device_status()
        small = M * N * K <= 272 * 400 * 528
        ent = None if small else dict(y=sample_entries(rng, M, N), dx=sample_entries(rng, M, K),
                                      dw=sample_entries(rng, N, K))
        ref = ost.dynamic_linear_step(x, w, g, ent)
        sc = st.scales.cpu().numpy()
        am = step.amax.cpu().numpy()
        for i, name in enumerate(("x", "w", "g")):
            r = ref[name]
            assert f32bits(am[i]) == f32bits(r["amax"]), name
            assert f32bits(sc[2 * i]) == f32bits(r["scale"]) and \
                f32bits(sc[2 * i + 1]) == f32bits(r["scale_inv"]), name
        assert np.array_equal(host_u8(step.xq), ref["x"]["q"])
        assert np.array_equal(host_u8(step.wqt), ref["w"]["q"].T)
        assert np.array_equal(host_u8(step.gqt), ref["g"]["q"].T)
        assert np.array_equal(host_u8(step.xqt), ref["x"]["q"].T)
        if small:
            check_gemm(step.y.float().cpu().numpy(), ref["y"], k=K)
            check_gemm(step.dx.float().cpu().numpy(), ref["dx"], k=N)
            check_gemm(step.dw.float().cpu().numpy(), ref["dw"], k=M)
        else:
            check_gemm(step.y.float().cpu().numpy(), ref["y"], *ent["y"], k=K)
            check_gemm(step.dx.float().cpu().numpy(), ref["dx"], *ent["dx"], k=N)
            check_gemm(step.dw.float().cpu().numpy(), ref["dw"], *ent["dw"], k=M)


def test_block_step_one_call_matches_the_single_calls_and_the_oracle():
    """fp8_linear_step_block at 512x384x640 (ragged pair and group tails):
    the same bits as the quantise-transpose and GEMM calls it stands for, and
    every output within the tolerance of the oracle's block GEMMs."""
    M, N, K = 512, 384, 640
    xh = synth.normal_with_outliers_bf16((M, K), 1.0, 31, "x")
    wh = synth.normal_with_outliers_bf16((N, K), 1.0, 31, "w")
    gh = synth.normal_with_outliers_bf16((M, N), 1.0, 31, "g")
    x, w, g = dev_bf16(xh), dev_bf16(wh), dev_bf16(gh)
    step = fp8.LinearStep(M, N, K)
    step.set_inputs(x, w, g)
    sc = fp8.BlockStepScales(M, N, K)
    fp8.fp8_linear_step_block(sc, step)
    fp8.fp8_check_device_status()
    # the single calls
    xq, xqt = u8(M, K), u8(K, M)
    xs, xsi, xst, xsit = f32(M, K // 128), f32(M, K // 128), f32(M // 128, K), f32(M // 128, K)
    fp8.fp8_quantize_transpose(x, fp8.BLOCK, xs, xsi, xq, xqt, xst, xsit)
    wq, wqt = u8(N, K), u8(K, N)
    ws, wsi = f32(N // 128, K // 128), f32(N // 128, K // 128)
    fp8.fp8_quantize_transpose(w, fp8.BLOCK_2D, ws, wsi, wq, wqt)
    gq, gqt = u8(M, N), u8(N, M)
    gs, gsi, gst, gsit = f32(M, N // 128), f32(M, N // 128), f32(M // 128, N), f32(M // 128, N)
    fp8.fp8_quantize_transpose(g, fp8.BLOCK, gs, gsi, gq, gqt, gst, gsit)
    y, dx, dw = bf16_out(M, N), bf16_out(M, K), bf16_out(N, K)
    fp8.fp8_linear_fprop(xq, xs, wq, ws, M, N, K, fp8.BLOCK, None, y)
    fp8.fp8_linear_dgrad(gq, gs, wqt, ws, M, N, K, fp8.BLOCK, dx)
    fp8.fp8_linear_wgrad(gqt, gst, xqt, xst, M, N, K, fp8.BLOCK, dw)
    for a, b in ((step.xq, xq), (step.xqt, xqt), (step.wq, wq), (step.wqt, wqt), (step.gq, gq),
                 (step.gqt, gqt), (sc.x_scale, xs), (sc.x_scale_t, xst), (sc.w_scale, ws),
                 (sc.g_scale, gs), (sc.g_scale_t, gst), (step.y, y), (step.dx, dx),
                 (step.dw, dw)):
        assert torch.equal(a, b)
    # the oracle
    xq_ref, xs_ref, _ = oracle.quantize_rowtiles(xh, 128)
    wq_ref, ws_ref, _ = oracle.quantize_sqtiles(wh, 128)
    gq_ref, gs_ref, _ = oracle.quantize_rowtiles(gh, 128)
    gqt_ref, gst_ref, _ = oracle.quantize_coltiles_t(gh, 128)
    xqt_ref, xst_ref, _ = oracle.quantize_coltiles_t(xh, 128)
    assert np.array_equal(host_u8(step.xq), xq_ref) and np.array_equal(host_u8(step.wq), wq_ref)
    assert np.array_equal(host_u8(step.gqt), gqt_ref) and np.array_equal(host_u8(step.xqt), xqt_ref)
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    check_gemm(step.y.float().cpu().numpy().ravel(),
               oracle.gemm_block_entries(xq_ref, wq_ref, xs_ref, ws_ref, 128, ii.ravel(), jj.ravel()))
    ii, jj = np.meshgrid(np.arange(M), np.arange(K), indexing="ij")
    check_gemm(step.dx.float().cpu().numpy().ravel(),
               oracle.gemm_block_entries(gq_ref, wq_ref.T.copy(), gs_ref,
                                         np.ascontiguousarray(ws_ref.T), 128, ii.ravel(),
                                         jj.ravel()))
    ii, jj = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    check_gemm(step.dw.float().cpu().numpy().ravel(),
               oracle.gemm_block_entries(gqt_ref, xqt_ref, gst_ref, xst_ref, 1, ii.ravel(),
                                         jj.ravel()))


def test_composite_step_forward_only_and_events():
    M, N, K = 128, 256, 128
    x = synth.normal_bf16((M, K), 1.0, 8, "x")
    w = synth.normal_bf16((N, K), 0.02, 8, "w")
    step = fp8.LinearStep(M, N, K, backward=False)
    meta = fp8.Fp8Meta(16)
    count = [0]
    step.set_inputs(dev_bf16(x), dev_bf16(w))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    for e in ev:
        e.record()
    fp8.fp8_linear_step_delayed(meta, count, step, events=ev)
    torch.cuda.synchronize()
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0 for i in range(7))
    st = ost.StepCounter(16)
    om = st.new_weight()
    st.step()
    f = ost.linear_forward(om, x, w)
    check_gemm(step.y.float().cpu().numpy(), f["y"])
    assert meta.idx == 1 and count[0] == 1


# ------------------------------------------------------------ workload 3 ---

def dynamic_linear_gpu(x, w, g):
    """Dynamic tensorwise fwd+dgrad+wgrad of one projection on the GPU."""
    M, K = x.shape
    N = w.shape[0]
    res = {}
    for name, t in (("x", x), ("w", w), ("g", g)):
        r, c = t.shape
        q, qt = u8(r, c), u8(c, r)
        s, si, a = f32(), f32(), f32()
        fp8.fp8_quantize_transpose(t, fp8.DYNAMIC, s, si, q, qt, amax_out=a)
        res[name] = (q, qt, s, a)
    y, dx, dw = bf16_out(M, N), bf16_out(M, K), bf16_out(N, K)
    X, W, G = res["x"], res["w"], res["g"]
    fp8.fp8_linear_fprop(X[0], X[2], W[0], W[2], M, N, K, fp8.DYNAMIC, None, y)
    # the backward pair through the one-launch entry point, as the MLP workload runs it
    fp8.fp8_linear_dgrad_wgrad(G[0], G[1], G[2], W[1], W[2], X[1], X[2], M, N, K, fp8.DYNAMIC,
                               dx, dw)
    fp8.fp8_check_device_status()
    return res, y, dx, dw


def check_dynamic_projection(xh, wh, gh, res, y, dx, dw, rng, sample_rows=8):
    refq = {}
    for name, h in (("x", xh), ("w", wh), ("g", gh)):
        q, qt, s, a = res[name]
        amax = oracle.amax(h)
        rs, rsi = oracle.scale_from_amax(amax)
        assert f32bits(a.item()) == f32bits(amax) and f32bits(s.item()) == f32bits(rs)
        rows = rng.choice(h.shape[0], sample_rows, replace=False)
        rq, _ = oracle.quantize(np.ascontiguousarray(h[rows]), rsi)
        assert np.array_equal(host_u8(q[torch.from_numpy(rows).cuda()]), rq)
        cols = rng.choice(h.shape[1], sample_rows, replace=False)
        rqt, _ = oracle.quantize(np.ascontiguousarray(h[:, cols].T), rsi)
        assert np.array_equal(host_u8(qt[torch.from_numpy(cols).cuda()]), rqt)
        refq[name] = (host_u8(q), rs)
    X, W, G = refq["x"], refq["w"], refq["g"]
    M, K = xh.shape
    N = wh.shape[0]
    ii, jj = sample_entries(rng, M, N, 1024, 1)
    check_gemm(y.float().cpu().numpy(), oracle.gemm_entries(X[0], W[0], X[1], W[1], ii, jj), ii, jj,
               k=K)
    ii, jj = sample_entries(rng, M, K, 1024, 1)
    check_gemm(dx.float().cpu().numpy(),
               oracle.gemm_entries(G[0], oracle.transpose_u8(W[0]), G[1], W[1], ii, jj), ii, jj,
               k=N)
    ii, jj = sample_entries(rng, N, K, 1024, 1)
    check_gemm(dw.float().cpu().numpy(),
               oracle.gemm_entries(oracle.transpose_u8(G[0]), oracle.transpose_u8(X[0]), G[1],
                                   X[1], ii, jj), ii, jj, k=M)


@pytest.mark.parametrize("proj", ["gate_up", "down"])
def test_config3_mlp_projection(proj):
    c = synth.CONFIG3
    M, H, F = c["M"], c["hidden"], c["ffn"]
    K, N = (H, 2 * F) if proj == "gate_up" else (F, H)
    seed = c["seed"] + (0 if proj == "gate_up" else 1)
    xh = synth.normal_bf16((M, K), c["x_sigma"], seed, "x")
    wh = synth.normal_bf16((N, K), c["w_sigma"], seed, "w")
    gh = synth.normal_bf16((M, N), c["g_sigma"], seed, "g")
    res, y, dx, dw = dynamic_linear_gpu(dev_bf16(xh), dev_bf16(wh), dev_bf16(gh))
    check_dynamic_projection(xh, wh, gh, res, y, dx, dw, np.random.default_rng(seed))


# ------------------------------------------------------------ workload 4 ---

def test_config4_thd_padding():
    c = synth.CONFIG4
    lengths = synth.thd_lengths(c["seed"], c["n_seq"], c["lo"], c["hi"])
    T = int(lengths.sum())
    K, N = c["K"], c["N"]
    xh = synth.normal_bf16((T, K), c["x_sigma"], c["seed"], "x")
    wh = synth.normal_bf16((N, K), c["w_sigma"], c["seed"], "w")
    Tp = fp8.fp8_padded_rows(T, c["multiple"])
    assert Tp % 16 == 0 and Tp - T < 16
    gh = synth.normal_bf16((Tp, N), c["g_sigma"], c["seed"], "g")
    gh[T:] = 0  # gradients of pad tokens are zero
    xp = bf16_out(Tp, K)
    assert fp8.fp8_pad_tokens(dev_bf16(xh), 16, xp) == Tp
    res, y, dx, dw = dynamic_linear_gpu(xp, dev_bf16(wh), dev_bf16(gh))
    # padded rows do not change amax; the scale is the unpadded tensor's
    assert f32bits(res["x"][3].item()) == f32bits(oracle.amax(xh))
    # pad rows of the quantised input, of Y and of dX are zero
    assert not host_u8(res["x"][0][T:]).any()
    assert not (y[T:].float() != 0).any().item() and not (dx[T:].float() != 0).any().item()
    xph = np.concatenate([xh, np.zeros((Tp - T, K), np.uint16)])
    check_dynamic_projection(xph, wh, gh, res, y, dx, dw, np.random.default_rng(4))
    # dW over the padded batch equals dW over the real tokens (sampled)
    rng = np.random.default_rng(5)
    gq = host_u8(res["g"][0])[:T]
    xq = host_u8(res["x"][0])[:T]
    ii, jj = sample_entries(rng, N, K, 512, 1)
    ref = oracle.gemm_entries(oracle.transpose_u8(gq), oracle.transpose_u8(xq),
                              res["g"][2].item(), res["x"][2].item(), ii, jj)
    check_gemm(dw.float().cpu().numpy(), ref, ii, jj, k=T)


# ------------------------------------------------------------ workload 5 ---

def test_config5_block_recipe_full_size():
    c = synth.CONFIG5
    M, K, N = c["M"], c["K"], c["N"]
    rng = np.random.default_rng(c["seed"])
    xh = synth.normal_with_outliers_bf16((M, K), c["sigma"], c["seed"], "x", p=c["p"], factor=c["factor"])
    wh = synth.normal_with_outliers_bf16((N, K), c["sigma"], c["seed"], "w", p=c["p"], factor=c["factor"])
    gh = synth.normal_with_outliers_bf16((M, N), c["sigma"], c["seed"], "g", p=c["p"], factor=c["factor"])
    x, w, g = dev_bf16(xh), dev_bf16(wh), dev_bf16(gh)
    # X: 1x128 rows for fprop and 128x1 columns (transposed) for wgrad
    xq, xqt = u8(M, K), u8(K, M)
    xs, xsi, xst, xsit = f32(M, K // 128), f32(M, K // 128), f32(M // 128, K), f32(M // 128, K)
    fp8.fp8_quantize_transpose(x, fp8.BLOCK, xs, xsi, xq, xqt, xst, xsit)
    wq, wqt = u8(N, K), u8(K, N)
    ws, wsi = f32(N // 128, K // 128), f32(N // 128, K // 128)
    fp8.fp8_quantize_transpose(w, fp8.BLOCK_2D, ws, wsi, wq, wqt)
    gq, gqt = u8(M, N), u8(N, M)
    gs, gsi, gst, gsit = f32(M, N // 128), f32(M, N // 128), f32(M // 128, N), f32(M // 128, N)
    fp8.fp8_quantize_transpose(g, fp8.BLOCK, gs, gsi, gq, gqt, gst, gsit)
    y, dx, dw = bf16_out(M, N), bf16_out(M, K), bf16_out(N, K)
    fp8.fp8_linear_fprop(xq, xs, wq, ws, M, N, K, fp8.BLOCK, None, y)
    fp8.fp8_linear_dgrad(gq, gs, wqt, ws, M, N, K, fp8.BLOCK, dx)
    fp8.fp8_linear_wgrad(gqt, gst, xqt, xst, M, N, K, fp8.BLOCK, dw)
    fp8.fp8_check_device_status()
    # quantisers on sampled row / column blocks against the oracle
    rows = rng.choice(M // 128, 2, replace=False) * 128
    for r0 in rows:
        blk = np.ascontiguousarray(xh[r0:r0 + 128])
        q_ref, s_ref, _ = oracle.quantize_rowtiles(blk, 128)
        assert np.array_equal(host_u8(xq[r0:r0 + 128]), q_ref)
        assert np.array_equal(xs[r0:r0 + 128].cpu().numpy(), s_ref)
        qt_ref, st_ref, _ = oracle.quantize_coltiles_t(blk, 128)
        assert np.array_equal(host_u8(xqt[:, r0:r0 + 128]), qt_ref)
        assert np.array_equal(xst[r0 // 128].cpu().numpy(), st_ref[:, 0])
    wq_ref, ws_ref, _ = oracle.quantize_sqtiles(wh, 128)
    assert np.array_equal(host_u8(wq), wq_ref) and np.array_equal(ws.cpu().numpy(), ws_ref)
    # GEMMs on sampled entries, with the GPU's (verified) operands
    xqh, gqh, xqth, gqth = host_u8(xq), host_u8(gq), host_u8(xqt), host_u8(gqt)
    # the oracle takes column-tile scales as [rows of the operand, blocks]
    xsh, gsh = xs.cpu().numpy(), gs.cpu().numpy()
    xsth, gsth = np.ascontiguousarray(xst.cpu().numpy().T), np.ascontiguousarray(gst.cpu().numpy().T)
    ii, jj = sample_entries(rng, M, N, 1024, 1)
    check_gemm(y.float().cpu().numpy(),
               oracle.gemm_block_entries(xqh, wq_ref, xsh, ws_ref, 128, ii, jj), ii, jj, k=K)
    ii, jj = sample_entries(rng, M, K, 1024, 1)
    check_gemm(dx.float().cpu().numpy(),
               oracle.gemm_block_entries(gqh, host_u8(wqt), gsh, np.ascontiguousarray(ws_ref.T),
                                         128, ii, jj), ii, jj, k=N)
    ii, jj = sample_entries(rng, N, K, 1024, 1)
    check_gemm(dw.float().cpu().numpy(),
               oracle.gemm_block_entries(gqth, xqth, gsth, xsth, 1, ii, jj), ii, jj, k=M)
