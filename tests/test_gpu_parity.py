"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Exact-gradient cases (integer-valued inputs, so G is exact in fp32 in any
summation order) must match the oracle's float32 op-sequence mode bit for
bit in every variant, including stochastic-rounding decisions and 8-bit
codes. Random-input cases are held to the element-wise tolerance of
oracle/tolerance.py (a 1e-5 relative perturbation of the step's inputs,
the gradient's scaled by |dY|^T |X|) for fp32 outputs; a bf16 output must be
the storage rounding of a value within that tolerance (one bf16 ulp at most
where the tolerance is below an ulp), and 8-bit codes within one code, in at
most 1e-4 of the elements.
"""

import numpy as np
import pytest
import torch

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300 import synthetic as S
import oracle.forge_oracle as O

from forge_cases import HYPER, VARIANTS, assert_bit_exact, check_tolerance, gpu_step, oracle_step, to_np

pytestmark = pytest.mark.gpu

OPTS = ["adamw", "sgdm", "lion"]
# (D_out, D_in, BT): several tiles and a ragged token tail; ragged D; one tile.
SHAPES = [(256, 384, 200), (136, 200, 70), (128, 128, 64)]


def _prob(shape, seed, x_dtype, w, st, exact, fresh=False, zero_rows=0.0):
    d_out, d_in, bt = shape
    return S.linear_problem(d_out, d_in, bt, seed=seed, x_dtype=x_dtype, w_dtype=w, state=st, exact=exact,
                            fresh_moments=fresh, zero_row_fraction=zero_rows)


def _ok_shape(shape, st):
    return st != "q8" or shape[1] % 128 == 0


# ---------------------------------------------------------------------------
# Bit-exact against the float32 op-sequence oracle (exact gradients)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("opt", OPTS)
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: f"W{v[0]}-m{v[1]}")
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_gradient_bit_exact(opt, variant, shape):
    w, st = variant
    if not _ok_shape(shape, st):
        pytest.skip("8-bit blocks need D_in % 128 == 0")
    sr = w == "bf16"
    srm = st == "bf16"
    prob = _prob(shape, 11, "bf16", w, st, exact=True)
    for t in (1, 7):
        got = gpu_step(opt, prob, t, seed=1234, sr_w=sr, sr_moments=srm)
        ref = oracle_step(opt, prob, w, st, t, seed=1234, sr_w=sr, sr_moments=srm, mode="f32emu")
        assert_bit_exact(got, ref, opt)


@pytest.mark.parametrize("opt", OPTS)
@pytest.mark.parametrize("variant", [("bf16", "bf16"), ("f32", "q8")], ids=lambda v: f"W{v[0]}-m{v[1]}")
def test_exact_gradient_rne_stores(opt, variant):
    # Round-to-nearest-even stores of bf16 W / moments (no stochastic rounding).
    w, st = variant
    prob = _prob((256, 384, 130), 5, "bf16", w, st, exact=True)
    got = gpu_step(opt, prob, 3, seed=9)
    ref = oracle_step(opt, prob, w, st, 3, seed=9, mode="f32emu")
    assert_bit_exact(got, ref, opt)


# ---------------------------------------------------------------------------
# Random inputs against the float64 oracle within the stated tolerance
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("opt", OPTS)
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: f"W{v[0]}-m{v[1]}")
@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: "x".join(map(str, s)))
def test_random_inputs_within_tolerance(opt, variant, shape):
    w, st = variant
    if not _ok_shape(shape, st):
        pytest.skip("8-bit blocks need D_in % 128 == 0")
    sr = w == "bf16"
    prob = _prob(shape, 21, "bf16", w, st, exact=False)
    got = gpu_step(opt, prob, 2, seed=77, sr_w=sr)
    rep = check_tolerance(opt, prob, w, st, 2, got, seed=77, sr_w=sr)
    print(opt, w, st, shape, rep)


def test_adamw_tolerance_at_paper_verification_shape():
    # D_in = D_out = 512, BT = 256 (the paper's per-family numerical check, Appendix N).
    prob = _prob((512, 512, 256), 31, "bf16", "f32", "f32", exact=False)
    got = gpu_step("adamw", prob, 1)
    rep = check_tolerance("adamw", prob, "f32", "f32", 1, got)
    assert rep["W"] <= 1.0 and rep["m"] <= 1.0 and rep["v"] <= 1.0


# ---------------------------------------------------------------------------
# fp32 inputs (CUDA-core path): the 3-step fp32 AdamW problem
# ---------------------------------------------------------------------------

def test_fp32_three_steps_fresh_inputs():
    # W 256x256 ~N(0, 0.02), X and dY 128 x 256 ~N(0, 1) drawn fresh each step,
    # m = v = 0, AdamW lr 1e-3, betas (0.9, 0.999), eps 1e-8, wd 0.01, seed 0.
    d_out = d_in = 256
    bt = 128
    dev = "cuda:0"
    W0 = S.normal((d_out, d_in), 0.02, 0, S.STREAM_W, "f32")
    W = W0.clone().to(dev)
    m = torch.zeros_like(W); v = torch.zeros_like(W)
    st = O.State(W=W0.numpy().copy(), m=np.zeros((d_out, d_in), np.float32), v=np.zeros((d_out, d_in), np.float32))
    h = O.Hyper(**HYPER["adamw"])
    worst = 0.0
    from oracle import tolerance as T
    for t in (1, 2, 3):
        X, dY = S.step_inputs(d_out, d_in, bt, 0, t, "f32")
        F.wgrad_step_adamw(X.to(dev), dY.to(dev), W, m, v, step=t, **HYPER["adamw"])
        F.sync_status()
        Xn, dYn = X.numpy(), dY.numpy()
        G = O.wgrad_f64(dYn, Xn); A = O.abs_wgrad_f64(dYn, Xn)
        tw, tm, tv = T.adamw_tol(st.W, st.m, st.v, G, A, h, t)
        ref = O.step("adamw", Xn, dYn, st, h, t)
        for name, g, r, tol in (("W", W, ref.W, tw), ("m", m, ref.m, tm), ("v", v, ref.v, tv)):
            viol = T.rel_violation(to_np(g), r, tol)
            worst = max(worst, viol)
            assert viol <= 1.0, (t, name, viol)
        # continue the trajectory from the GPU's own state (the oracle is
        # held to one step at a time)
        st = O.State(W=to_np(W), m=to_np(m), v=to_np(v))
    print("fp32 3-step worst tolerance use", worst)


@pytest.mark.parametrize("opt", OPTS)
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: f"W{v[0]}-m{v[1]}")
def test_fp32_inputs_exact_bit_exact(opt, variant):
    w, st = variant
    prob = _prob((64, 256, 40), 4, "f32", w, st, exact=True)
    got = gpu_step(opt, prob, 2, seed=5, sr_w=w == "bf16", sr_moments=st == "bf16")
    ref = oracle_step(opt, prob, w, st, 2, seed=5, sr_w=w == "bf16", sr_moments=st == "bf16", mode="f32emu")
    assert_bit_exact(got, ref, opt)


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("opt", OPTS)
@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_empty_token_axis_is_a_zero_gradient_step(opt, x_dtype):
    prob = _prob((136, 256, 0), 2, x_dtype, "f32", "f32", exact=True)
    got = gpu_step(opt, prob, 4)
    ref = oracle_step(opt, prob, "f32", "f32", 4, mode="f32emu")
    assert_bit_exact(got, ref, opt)


@pytest.mark.parametrize("shape", [(8, 8, 1), (8, 128, 3), (264, 8, 65), (1000, 1024, 1)])
def test_degenerate_and_minimum_shapes(shape):
    prob = _prob(shape, 8, "bf16", "f32", "f32", exact=True)
    got = gpu_step("adamw", prob, 1)
    ref = oracle_step("adamw", prob, "f32", "f32", 1, mode="f32emu")
    assert_bit_exact(got, ref, "adamw")


def test_q8_zero_gradient_rows_keep_reserved_zero_codes():
    # 30% of W rows get an exactly zero gradient and start from zero moments.
    prob = _prob((512, 512, 256), 3, "bf16", "f32", "q8", exact=False, zero_rows=0.3)
    got = gpu_step("adamw", prob, 1)
    zr = prob.zero_rows
    assert np.all(got.m[zr] == 0) and np.all(got.v[zr] == 0)
    assert np.all(got.m_scale[:, zr] == 0) and np.all(got.v_scale[:, zr] == 0)
    decay = np.float32(1.0 - HYPER["adamw"]["lr"] * HYPER["adamw"]["weight_decay"])
    assert np.array_equal(got.W[zr], (decay * to_np(prob.W)[zr]).astype(np.float32))
    assert np.all(got.v[~zr] != 0)       # nonzero second moments never take code 0
    check_tolerance("adamw", prob, "f32", "q8", 1, got)


def test_sr_weight_store_is_unbiased_on_gpu():
    # The quarter-ulp example: lr chosen so every update is ~1/4 bf16 ulp.
    d_out, d_in = 256, 512
    dev = "cuda:0"
    X = torch.zeros((1, d_in), dtype=torch.bfloat16, device=dev)
    dY = torch.zeros((1, d_out), dtype=torch.bfloat16, device=dev)
    W = torch.full((d_out, d_in), 0.75, dtype=torch.bfloat16, device=dev)
    m = torch.full((d_out, d_in), 1.0, dtype=torch.float32, device=dev)   # SGDM with mu = 1, g = 0
    W_rne = W.clone(); m_rne = m.clone()
    for t in range(1, 101):
        F.wgrad_step_sgdm(X, dY, W, m, lr=1e-3, momentum=1.0, weight_decay=0.0, step=t, seed=1234, sr_w=True)
        F.wgrad_step_sgdm(X, dY, W_rne, m_rne, lr=1e-3, momentum=1.0, weight_decay=0.0, step=t)
    F.sync_status()
    assert torch.all(W_rne == 0.75)
    mean_change = float(W.float().mean() - 0.75)
    se = 10 * 2 ** -8 / 2 / np.sqrt(d_out * d_in)
    assert abs(mean_change - (-0.1)) < 5 * se, mean_change


# ---------------------------------------------------------------------------
# Invariances
# ---------------------------------------------------------------------------

def test_run_to_run_determinism():
    prob = _prob((512, 1024, 512), 9, "bf16", "bf16", "bf16", exact=False)
    a = gpu_step("adamw", prob, 3, seed=1, sr_w=True)
    b = gpu_step("adamw", prob, 3, seed=1, sr_w=True)
    assert_bit_exact(a, b, "adamw")


def test_row_shard_invariance():
    # A row block of W stepped on its own (the tensor-parallel shard of
    # Proposition 2 (i)) equals the same rows of the full step, bit for bit.
    dev = "cuda:0"
    prob = _prob((512, 384, 300), 12, "bf16", "f32", "f32", exact=False)
    full = gpu_step("adamw", prob, 2)
    X, dY = prob.X.to(dev), prob.dY.to(dev)
    W, m, v = prob.W.to(dev), prob.m.to(dev), prob.v.to(dev)
    for r0, r1 in ((0, 128), (128, 384), (384, 512)):
        F.wgrad_step_adamw(X, dY[:, r0:r1], W[r0:r1], m[r0:r1], v[r0:r1], step=2, **HYPER["adamw"])
    F.sync_status()
    assert np.array_equal(to_np(W).view(np.uint32), full.W.view(np.uint32))
    assert np.array_equal(to_np(m).view(np.uint32), full.m.view(np.uint32))
    assert np.array_equal(to_np(v).view(np.uint32), full.v.view(np.uint32))


@pytest.mark.parametrize("exact", [True, False])
def test_tile_width_invariance(exact):
    prob = _prob((256, 512, 192), 13, "bf16", "f32", "f32", exact=exact)
    a = gpu_step("adamw", prob, 1, flags=F.FLAG_TILE_N_128)
    b = gpu_step("adamw", prob, 1, flags=F.FLAG_TILE_N_64)
    assert_bit_exact(a, b, "adamw")


def test_checkpoint_resume_bit_identical():
    # 3 steps == 2 steps, copy the state out and back (a checkpoint), 1 step.
    dev = "cuda:0"
    prob = _prob((256, 384, 128), 14, "bf16", "bf16", "q8", exact=False)
    def run(n, state=None):
        W = prob.W.to(dev).clone(); m = prob.m.to(dev).clone(); v = prob.v.to(dev).clone()
        ms = prob.m_scale.to(dev).clone(); vs = prob.v_scale.to(dev).clone()
        if state is not None:
            for dst, src in zip((W, m, v, ms, vs), state):
                dst.copy_(src.to(dev))
        for t in n:
            F.wgrad_step_adamw(prob.X.to(dev), prob.dY.to(dev), W, m, v, m_scale=ms, v_scale=vs, step=t,
                               seed=42, sr_w=True, **HYPER["adamw"])
        F.sync_status()
        return [x.cpu() for x in (W, m, v, ms, vs)]
    a = run([1, 2, 3])
    ck = run([1, 2])
    b = run([3], state=ck)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ---------------------------------------------------------------------------
# Failure path: a bounded device wait that gives up (no fault, no hang)
# ---------------------------------------------------------------------------

def test_forced_device_timeout_reports_and_leaves_state():
    dev = "cuda:0"
    prob = _prob((256, 256, 64), 15, "bf16", "f32", "f32", exact=False)
    X, dY = prob.X.to(dev), prob.dY.to(dev)
    W, m, v = prob.W.to(dev), prob.m.to(dev), prob.v.to(dev)
    F.wgrad_step_adamw(X, dY, W, m, v, step=1, flags=F.FLAG_TEST_FORCE_TIMEOUT, **HYPER["adamw"])
    with pytest.raises(F.ForgeError) as ei:
        F.sync_status()
    assert ei.value.status == 5 and "test hook" in str(ei.value)
    assert torch.equal(W.cpu(), prob.W) and torch.equal(m.cpu(), prob.m) and torch.equal(v.cpu(), prob.v)
    # the context is healthy: the next call runs normally
    F.wgrad_step_adamw(X, dY, W, m, v, step=1, **HYPER["adamw"])
    F.sync_status()
    assert not torch.equal(W.cpu(), prob.W)


# ---------------------------------------------------------------------------
# Input gradient (Remark 1)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("w_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dx_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(256, 384, 200), (136, 200, 70), (1024, 512, 512), (2048, 1024, 64),
                                   (1024, 512, 640), (1024, 4000, 1300), (256, 10000, 200), (1000, 10000, 512)])
def test_dgrad_exact(w_dtype, dx_dtype, shape):
    # (1024, 4000, 1300): with bf16 weights, 128 x 256 tiles with ragged
    # token and feature tails. D_in 10000 on short token axes: the policy
    # takes all-token tiles for fp32 weights (2 / 4 blocks of 128 tokens, 79
    # columns of tiles, the last one ragged; D_out 1000: a ragged last
    # stage).
    d_out, d_in, bt = shape
    dev = "cuda:0"
    dY = S.small_integers((bt, d_out), -3, 3, 1, S.STREAM_DY, "bf16")
    W = S.small_integers((d_out, d_in), -3, 3, 1, S.STREAM_W, w_dtype)
    dX = torch.empty((bt, d_in), dtype=torch.bfloat16 if dx_dtype == "bf16" else torch.float32, device=dev)
    F.dgrad(dY.to(dev), W.to(dev), dX)
    F.sync_status()
    ref = O.dgrad_f64(dY.float().numpy(), W.float().numpy())
    got = dX.float().cpu().numpy()
    if dx_dtype == "bf16":
        ref = O.bf16_bits_to_f32(O.f64_to_bf16_rne(ref))
    assert np.array_equal(got, ref.astype(np.float32))


@pytest.mark.parametrize("w_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(8192, 2600, 512), (8192, 520, 200), (4096, 1000, 300), (136, 200, 70)],
                         ids=lambda s: "x".join(map(str, s)))
def test_dgrad_with_workspace_exact(w_dtype, shape):
    # forge_dgrad_ws: with the workspace the contraction is split over D_out
    # where the plan says so (all-token tiles at 2600 x 512, 128-token tiles
    # at 520 x 200), else the same kernel as forge_dgrad; exact inputs, so
    # dX is exact either way, and a second call gives the same bits.
    d_out, d_in, bt = shape
    dev = "cuda:0"
    dY = S.small_integers((bt, d_out), -3, 3, 7, S.STREAM_DY, "bf16")
    W = S.small_integers((d_out, d_in), -3, 3, 7, S.STREAM_W, w_dtype)
    ws = torch.empty(max(16, F.workspace_bytes(d_out, d_in, bt)), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(2):
        dX = torch.full((bt, d_in), float("nan"), dtype=torch.float32, device=dev)
        F.dgrad(dY.to(dev), W.to(dev), dX, workspace=ws)
        F.sync_status()
        outs.append(dX.cpu().numpy())
    ref = O.dgrad_f64(dY.float().numpy(), W.float().numpy())
    assert np.array_equal(outs[0], ref.astype(np.float32))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_dgrad_random_reads_pre_update_weights():
    d_out, d_in, bt = 1024, 512, 256
    dev = "cuda:0"
    prob = S.linear_problem(d_out, d_in, bt, seed=16, x_dtype="bf16", w_dtype="f32", state="f32",
                            w_bf16_representable=False)
    X, dY = prob.X.to(dev), prob.dY.to(dev)
    W, m, v = prob.W.to(dev), prob.m.to(dev), prob.v.to(dev)
    dX = torch.empty((bt, d_in), dtype=torch.float32, device=dev)
    F.dgrad(dY, W, dX)                                   # enqueued first (Remark 1)
    F.wgrad_step_adamw(X, dY, W, m, v, step=1, **HYPER["adamw"])
    F.sync_status()
    w16 = O.bf16_bits_to_f32(O.f32_to_bf16_rne(prob.W.numpy())).astype(np.float64)
    dYn = prob.dY.float().numpy()
    ref = dYn @ w16
    tol = 1e-5 * (np.abs(dYn) @ np.abs(w16))
    assert np.all(np.abs(dX.cpu().numpy() - ref) <= tol)


@pytest.mark.parametrize("shape", [(4096, 512, 256), (14336, 4096, 512), (2048, 4096, 512), (4096, 14336, 512)])
@pytest.mark.parametrize("tiles", ["auto", "tokens128", "all_tokens"])
def test_dgrad_f32_and_bf16_weights_agree_bit_for_bit(shape, tiles):
    # fp32 master weights that are bf16-representable must give exactly the
    # dX of the same weights stored as bf16 (the staging conversion is exact)
    # on the same tiles, on every repetition (no stale staging data). "auto":
    # forge_dgrad's own choice where both dtypes take the same tiles (the
    # 128-token tiles at these shapes, except the down-projection, where fp32
    # weights take all-token tiles); otherwise forced through
    # forge_backward_step's split path without a workspace (SGD with lr = 0:
    # W unchanged).
    d_out, d_in, bt = shape
    dev = "cuda:0"
    W16 = S.normal((d_out, d_in), 0.02, 2, S.STREAM_W, "bf16").to(dev)
    W32 = W16.float()
    dY = S.normal((bt, d_out), 1.0, 2, S.STREAM_DY, "bf16").to(dev)
    X = S.normal((bt, d_in), 1.0, 2, S.STREAM_X, "bf16").to(dev)

    def run(W, out):
        if tiles == "auto":
            F.dgrad(dY, W, out)
        else:
            fl = F.FLAG_DGRAD_TOKENS_128 if tiles == "tokens128" else F.FLAG_DGRAD_ALL_TOKENS
            F.backward_step("sgd", X, dY, W, None, None, out, lr=0.0, step=1, flags=fl | F.FLAG_BACKWARD_SPLIT)

    if tiles == "auto" and d_in == 14336:
        pytest.skip("fp32 and bf16 weights take different tiles here")
    ref = torch.empty((bt, d_in), dtype=torch.float32, device=dev)
    run(W16, ref)
    for _ in range(4):
        out = torch.empty_like(ref)
        run(W32, out)
        F.sync_status()
        assert torch.equal(out, ref), int((out != ref).sum())


# ---------------------------------------------------------------------------
# The remaining element-wise families (Appendix N (i))
# ---------------------------------------------------------------------------

NEW_OPTS = ["sgd", "rmsprop", "adagrad", "nadam", "radam"]
NEW_VARIANTS = [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16"), ("bf16", "f32")]


@pytest.mark.parametrize("opt", NEW_OPTS)
@pytest.mark.parametrize("variant", NEW_VARIANTS, ids=lambda v: f"W{v[0]}-m{v[1]}")
@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: "x".join(map(str, s)))
def test_more_families_exact_bit_exact(opt, variant, shape):
    w, st = variant
    prob = _prob(shape, 17, "bf16", w, st, exact=True)
    for t in (1, 7):   # RAdam: step 1 unrectified, step 7 rectified
        got = gpu_step(opt, prob, t, seed=99, sr_w=w == "bf16", sr_moments=st == "bf16")
        ref = oracle_step(opt, prob, w, st, t, seed=99, sr_w=w == "bf16", sr_moments=st == "bf16", mode="f32emu")
        assert_bit_exact(got, ref, opt)


@pytest.mark.parametrize("opt", NEW_OPTS)
@pytest.mark.parametrize("variant", [("f32", "f32"), ("bf16", "bf16")], ids=lambda v: f"W{v[0]}-m{v[1]}")
def test_more_families_random_within_tolerance(opt, variant):
    w, st = variant
    prob = _prob((256, 384, 200), 23, "bf16", w, st, exact=False)
    for t in (2, 9):
        got = gpu_step(opt, prob, t, seed=5, sr_w=w == "bf16")
        rep = check_tolerance(opt, prob, w, st, t, got, seed=5, sr_w=w == "bf16")
        print(opt, w, st, t, rep)


@pytest.mark.parametrize("opt", NEW_OPTS)
def test_more_families_fp32_inputs_bit_exact(opt):
    prob = _prob((64, 256, 40), 4, "f32", "f32", "f32", exact=True)
    got = gpu_step(opt, prob, 3)
    ref = oracle_step(opt, prob, "f32", "f32", 3, mode="f32emu")
    assert_bit_exact(got, ref, opt)


# ---------------------------------------------------------------------------
# 128 x 256 tiles (long token axes)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("opt", ["adamw", "lion", "sgdm", "nadam"])
@pytest.mark.parametrize("variant", [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16"), ("bf16", "f32")],
                         ids=lambda v: f"W{v[0]}-m{v[1]}")
@pytest.mark.parametrize("shape", [(384, 520, 1100), (136, 256, 70)], ids=lambda s: "x".join(map(str, s)))
def test_wide_tiles_exact(opt, variant, shape):
    # fp32 W + fp32 state streams 16-column chunks on these tiles (three
    # operand stages), the other storages 32-column ones.
    w, st = variant
    prob = _prob(shape, 17, "bf16", w, st, exact=True)
    sr, srm = w == "bf16", st == "bf16"
    got = gpu_step(opt, prob, 2, seed=5, sr_w=sr, sr_moments=srm, flags=F.FLAG_TILE_N_256)
    ref = oracle_step(opt, prob, w, st, 2, seed=5, sr_w=sr, sr_moments=srm, mode="f32emu")
    assert_bit_exact(got, ref, opt)


@pytest.mark.parametrize("opt", ["adamw", "lion", "sgdm", "nadam"])
@pytest.mark.parametrize("shape", [(264, 520, 300), (136, 200, 600), (384, 1024, 1100)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_state_64_column_chunks_exact(opt, shape):
    # bf16 W + bf16 moments on 128-column tiles below 768 tokens stream the
    # state in 64-column chunks (two- and three-stage operand rings at 300
    # and 600 tokens), elsewhere in 32-column ones; ragged D_in leaves a
    # chunk partly or wholly past the edge.
    prob = _prob(shape, 23, "bf16", "bf16", "bf16", exact=True)
    for flag in (F.FLAG_TILE_N_128, F.FLAG_TILE_N_256):
        got = gpu_step(opt, prob, 2, seed=9, sr_w=True, sr_moments=True, flags=flag)
        ref = oracle_step(opt, prob, "bf16", "bf16", 2, seed=9, sr_w=True, sr_moments=True, mode="f32emu")
        assert_bit_exact(got, ref, opt)


@pytest.mark.parametrize("opt", ["adamw", "lion", "sgdm", "nadam"])
@pytest.mark.parametrize("variant", [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16"), ("bf16", "f32")],
                         ids=lambda v: f"W{v[0]}-m{v[1]}")
@pytest.mark.parametrize("shape", [(384, 520, 1100), (136, 256, 70), (640, 776, 300)],
                         ids=lambda s: "x".join(map(str, s)))
def test_cta_pair_tiles_exact(opt, variant, shape):
    # 256 x 256 tiles shared by a cluster of two CTAs: ragged D_out leaves
    # the second CTA's half of the last tile row partly (136 rows) or wholly
    # (384 rows) past the edge; ragged D_in and token tails.
    w, st = variant
    prob = _prob(shape, 41, "bf16", w, st, exact=True)
    sr, srm = w == "bf16", st == "bf16"
    got = gpu_step(opt, prob, 2, seed=6, sr_w=sr, sr_moments=srm, flags=F.FLAG_TILE_PAIR_256)
    ref = oracle_step(opt, prob, w, st, 2, seed=6, sr_w=sr, sr_moments=srm, mode="f32emu")
    assert_bit_exact(got, ref, opt)


@pytest.mark.parametrize("variant", [("f32", "f32"), ("bf16", "bf16")], ids=lambda v: f"W{v[0]}-m{v[1]}")
@pytest.mark.parametrize("bt", [2048, 4160])
def test_cta_pair_tiles_match_single_cta_tiles(variant, bt):
    # Random inputs: the pair's M = 256 products give every gradient element
    # the same value as one CTA's 128 x 256 and 128 x 128 tiles, bit for bit
    # (fp32 state: four pair stages below 4096 tokens, five from there).
    w, st = variant
    prob = _prob((1024, 1280, bt), 43, "bf16", w, st, exact=False)
    sr = w == "bf16"
    a = gpu_step("adamw", prob, 1, seed=2, sr_w=sr, sr_moments=sr, flags=F.FLAG_TILE_PAIR_256)
    b = gpu_step("adamw", prob, 1, seed=2, sr_w=sr, sr_moments=sr, flags=F.FLAG_TILE_N_256)
    c = gpu_step("adamw", prob, 1, seed=2, sr_w=sr, sr_moments=sr, flags=F.FLAG_TILE_N_128)
    assert_bit_exact(a, b, "adamw")
    assert_bit_exact(a, c, "adamw")


@pytest.mark.parametrize("opt", ["lion", "adamw"])
def test_long_token_axis_automatic_tiles_exact(opt):
    # 2048 tokens on a layer with >= 152 tiles of 256 columns: the automatic
    # policy's tiles (CTA pairs) against the oracle's float32 sequence.
    prob = _prob((4096, 2048, 2048), 45, "bf16", "bf16", "bf16", exact=True)
    got = gpu_step(opt, prob, 3, seed=8, sr_w=True, sr_moments=True)
    ref = oracle_step(opt, prob, "bf16", "bf16", 3, seed=8, sr_w=True, sr_moments=True, mode="f32emu")
    assert_bit_exact(got, ref, opt)


def test_cta_pair_tiles_reject_8bit_state():
    prob = _prob((256, 512, 128), 44, "bf16", "f32", "q8", exact=False)
    with pytest.raises(F.ForgeError):
        gpu_step("adamw", prob, 1, flags=F.FLAG_TILE_PAIR_256)


@pytest.mark.parametrize("opt", ["adamw", "lion", "sgdm", "radam"])
def test_deep_ring_fp32_state_16_column_chunks_exact(opt):
    # fp32 W + fp32 state past 768 tokens on 128-column tiles: four operand
    # stages beside a ring of 16-column state chunks; ragged D_in and a
    # ragged token tail. Against the oracle and against 64-column tiles
    # (two stages, 32-column chunks).
    prob = _prob((264, 520, 800), 29, "bf16", "f32", "f32", exact=True)
    got = gpu_step(opt, prob, 2, seed=3, flags=F.FLAG_TILE_N_128)
    ref = oracle_step(opt, prob, "f32", "f32", 2, seed=3, mode="f32emu")
    assert_bit_exact(got, ref, opt)
    assert_bit_exact(gpu_step(opt, prob, 2, seed=3, flags=F.FLAG_TILE_N_64), ref, opt)


@pytest.mark.parametrize("exact", [True, False])
def test_tile_width_invariance_wide(exact):
    prob = _prob((512, 768, 1088), 18, "bf16", "f32", "f32", exact=exact)
    a = gpu_step("adamw", prob, 1, flags=F.FLAG_TILE_N_256)
    b = gpu_step("adamw", prob, 1, flags=F.FLAG_TILE_N_128)
    assert_bit_exact(a, b, "adamw")


def test_wide_tiles_random_within_tolerance():
    prob = _prob((640, 1024, 2048), 19, "bf16", "f32", "f32", exact=False)
    got = gpu_step("adamw", prob, 3, flags=F.FLAG_TILE_N_256)
    check_tolerance("adamw", prob, "f32", "f32", 3, got)


# ---------------------------------------------------------------------------
# Non-finite weights through the stochastic-rounding store
# ---------------------------------------------------------------------------

def _bf16_is_nan(b):
    b = np.asarray(b, np.uint16)
    return (b & 0x7FFF) > 0x7F80


@pytest.mark.parametrize("flag", ["n128", "n64"])
def test_sr_store_non_finite_weights(flag):
    # NaN and +-Inf weights (bf16 W, stochastic rounding): a NaN stays a NaN
    # (its payload is the arithmetic's, which differs between the GPU and the
    # host), an infinity stays that infinity, and every finite neighbour in
    # the same group of eight -- the kernel tests a group for NaN at once --
    # takes the oracle's draws bit for bit. Both chunk widths of the bf16
    # store (64 columns on 128-column tiles, 32 on 64-column ones).
    prob = _prob((256, 512, 200), 29, "bf16", "bf16", "bf16", exact=True)
    bits = prob.W.view(torch.int16).numpy().view(np.uint16)
    planted = {(0, 0): 0x7FC0, (0, 3): 0xFFC1, (5, 9): 0x7F81, (7, 16): 0x7F80, (7, 17): 0xFF80,
               (100, 200): 0x7F80, (130, 64): 0x7FC0, (255, 511): 0xFF80, (200, 130): 0xFFFF}
    for (i, j), b in planted.items():
        bits[i, j] = b
    flags = F.FLAG_TILE_N_128 if flag == "n128" else F.FLAG_TILE_N_64
    got = gpu_step("adamw", prob, 2, seed=9, sr_w=True, sr_moments=True, flags=flags)
    with np.errstate(invalid="ignore"):
        ref = oracle_step("adamw", prob, "bf16", "bf16", 2, seed=9, sr_w=True, sr_moments=True, mode="f32emu")
    nan_ref = _bf16_is_nan(ref.W)
    assert np.array_equal(_bf16_is_nan(got.W), nan_ref)
    assert int(nan_ref.sum()) == 5
    fin = ~nan_ref
    assert np.array_equal(np.asarray(got.W)[fin], np.asarray(ref.W)[fin])
    for (i, j), b in planted.items():
        if b in (0x7F80, 0xFF80):
            assert int(got.W[i, j]) == b
    assert_bit_exact(O.State(W=ref.W, m=got.m, v=got.v), ref, "adamw")


# ---------------------------------------------------------------------------
# AdamW with bf16 / 8-bit moments: operands outside the branch-free divide
# and square root's ranges take the guarded path
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("tiles", ["n128", "n64"])
def test_adamw_bf16_state_out_of_range_operands_bit_exact(tiles):
    # Zero rows (m' = v' = 0), second moments above 2^100 and below 2^-100,
    # first moments below 2^-60 and above 2^60, planted among ordinary
    # values: each group of eight that holds one is recomputed by the
    # guarded correctly rounded functions, and every value must still equal
    # the oracle's float32 op sequence bit for bit.
    prob = _prob((256, 512, 200), 37, "bf16", "bf16", "bf16", exact=True, zero_rows=0.1)
    m = prob.m.view(torch.int16).numpy().view(np.uint16)
    v = prob.v.view(torch.int16).numpy().view(np.uint16)
    plants = {(3, 5): ("v", 1e32), (3, 77): ("v", 3e35), (9, 8): ("v", 1e-33), (17, 100): ("m", 1e-25),
              (17, 101): ("m", -4e-30), (30, 200): ("m", 5e20), (31, 300): ("m", -2e24), (40, 9): ("v", 0.0),
              (40, 10): ("m", 0.0)}
    zr = np.flatnonzero(prob.zero_rows)
    for k, r in enumerate(zr[:4]):            # the same extremes on rows with no gradient
        plants[(int(r), 8 * k + 1)] = ("m", 3e-24)
        plants[(int(r), 8 * k + 40)] = ("v", 1e-34)
    for (i, j), (which, x) in plants.items():
        (m if which == "m" else v)[i, j] = int(O.f32_to_bf16_rne(np.array([x], np.float32))[0])
    flags = F.FLAG_TILE_N_128 if tiles == "n128" else F.FLAG_TILE_N_64
    for t in (1, 3):
        got = gpu_step("adamw", prob, t, seed=13, sr_w=True, sr_moments=True, flags=flags)
        ref = oracle_step("adamw", prob, "bf16", "bf16", t, seed=13, sr_w=True, sr_moments=True, mode="f32emu")
        assert_bit_exact(got, ref, "adamw")


def test_adamw_q8_state_out_of_range_operands_bit_exact():
    # 8-bit moments whose block scales put the decoded moments outside the
    # fast path's ranges: |m| above 2^60 (scale x 2^72) and v above 2^100
    # (square-root-domain scale x 2^62) on rows with a gradient; |m| below
    # 2^-60 (x 2^-55) and v below 2^-100 (x 2^-45) on rows with none, whose
    # codes are copied from a row that has a gradient. Bit-exact against the
    # float32 op sequence.
    prob = _prob((256, 512, 192), 38, "bf16", "f32", "q8", exact=True, zero_rows=0.1)
    m, v = prob.m.numpy(), prob.v.numpy()
    ms, vs = prob.m_scale.numpy(), prob.v_scale.numpy()
    zr = np.flatnonzero(prob.zero_rows)
    live = np.flatnonzero(~prob.zero_rows)
    ms[0, live[3]] *= np.float32(2.0 ** 72)
    ms[2, live[50]] *= np.float32(2.0 ** 72)
    vs[1, live[3]] *= np.float32(2.0 ** 62)
    vs[3, live[99]] *= np.float32(2.0 ** 62)
    for k, r in enumerate(zr[:3]):
        src = live[k]
        cols = slice(128 * k, 128 * (k + 1))
        m[r, cols] = m[src, cols]
        v[r, cols] = v[src, cols]
        ms[k, r] = ms[k, src] * np.float32(2.0 ** -55)
        vs[k, r] = vs[k, src] * np.float32(2.0 ** -45)
    for t in (1, 2):
        got = gpu_step("adamw", prob, t, seed=5, flags=F.FLAG_TILE_N_128)
        ref = oracle_step("adamw", prob, "f32", "q8", t, seed=5, mode="f32emu")
        assert_bit_exact(got, ref, "adamw")
