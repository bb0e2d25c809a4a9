"""GPU parity of the whole backward pass of a layer: dX = dY W_old and the
fused step (forge_backward_step), on the fused input-gradient path (one
read of W) and on the split path (dgrad, then the step).

Exact cases use integer-valued X, dY and W, so G and dX are exact in fp32
in any summation order: the new state must match the oracle's float32
op-sequence mode bit for bit and dX the float64 product (rounded once for
a bf16 dX). Random cases hold the state to the element-wise tolerance of
oracle/tolerance.py and dX to a 1e-5 relative perturbation of its terms,
|dX - dY W16| <= 1e-5 |dY| |W16| (W16 = W rounded to bf16, the operand
precision of the tensor cores), plus one ulp of a bf16 dX.
"""

import numpy as np
import pytest
import torch

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300 import synthetic as S
import oracle.forge_oracle as O

from forge_cases import HYPER, NSTATE, assert_bit_exact, check_tolerance, oracle_step, state_tensors, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
RULES = ["adamw", "sgdm", "lion", "sgd", "rmsprop", "adagrad", "nadam", "radam"]
VARIANTS = [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16"), ("bf16", "f32")]
# (D_out, D_in, BT): ragged D and tokens, one tile per CTA, several tiles per
# CTA with runs that cross tile columns, and the largest token count; the
# last two take fewer CTAs than SMs (2 tiles each: within a column, and
# across columns of 11 tiles).
SHAPES = [(256, 384, 200), (136, 200, 70), (1000, 520, 300), (2048, 1024, 768), (1408, 1024, 300)]


def _prob(shape, seed, w, st, exact):
    d_out, d_in, bt = shape
    prob = S.linear_problem(d_out, d_in, bt, seed=seed, x_dtype="bf16", w_dtype=w, state=st, exact=exact,
                            w_bf16_representable=exact or w == "bf16")
    if exact:
        prob.W = S.small_integers((d_out, d_in), -3, 3, seed, S.STREAM_W, w)
    return prob


def _hyper_kw(rule):
    hp = dict(HYPER[rule])
    return dict(lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"], weight_decay=hp["weight_decay"],
                momentum_decay=hp.get("momentum_decay", 4e-3))


def run_backward(rule, prob, t, *, dx_dtype="bf16", seed=0, sr_w=False, sr_moments=False, path="fused",
                 workspace=True, flags=0):
    """Copy the problem to the GPU, run forge_backward_step, return (state, dX) on the CPU."""
    X, dY, W = prob.X.to(DEV), prob.dY.to(DEV), prob.W.to(DEV)
    s0, s1 = state_tensors(rule, prob)
    s0 = s0.to(DEV) if s0 is not None else None
    s1 = s1.to(DEV) if s1 is not None else None
    bt, d_in = prob.X.shape
    dX = torch.full((bt, d_in), float("nan"), dtype=torch.bfloat16 if dx_dtype == "bf16" else torch.float32,
                    device=DEV)
    nbytes = F.workspace_bytes(prob.W.shape[0], d_in, bt)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV) if workspace else None
    if path == "fused":
        flags |= F.FLAG_BACKWARD_FUSED
    elif path == "split":
        flags |= F.FLAG_BACKWARD_SPLIT
    F.backward_step(rule, X, dY, W, s0, s1, dX, step=t, seed=seed, sr_w=sr_w, sr_moments=sr_moments,
                    workspace=ws, flags=flags, **_hyper_kw(rule))
    F.sync_status()
    st = O.State(W=to_np(W), m=to_np(s0) if s0 is not None else None, v=to_np(s1) if s1 is not None else None)
    return st, dX.float().cpu().numpy()


def _dx_ref(prob):
    w16 = O.bf16_bits_to_f32(O.f32_to_bf16_rne(prob.W.float().numpy())).astype(np.float64)
    dYn = prob.dY.float().numpy().astype(np.float64)
    return O.dgrad_f64(dYn, w16), np.abs(dYn) @ np.abs(w16)


def _check_dx(got, prob, dx_dtype, exact):
    ref, A = _dx_ref(prob)
    if exact:
        want = ref.astype(np.float32)
        if dx_dtype == "bf16":
            want = O.bf16_bits_to_f32(O.f64_to_bf16_rne(ref))
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"dX: {len(bad)} elements differ, first {bad[:3].tolist()}"
        return 0.0
    tol = 1e-5 * A
    if dx_dtype == "bf16":
        tol = tol + np.abs(ref) * 2.0 ** -8
    viol = float(np.max(np.abs(got - ref) / np.maximum(tol, 1e-300)))
    assert viol <= 1.0, f"dX: {viol:.3f} of the tolerance"
    return viol


# ---------------------------------------------------------------------------
# Fused path: bit-exact with exact inputs, every rule and storage variant
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: f"W{v[0]}-m{v[1]}")
@pytest.mark.parametrize("shape", SHAPES[:2] + [(264, 384, 512), (264, 384, 600)], ids=lambda s: "x".join(map(str, s)))
def test_fused_backward_exact(rule, variant, shape):
    # BT 200 / 70: short token axes (16-column state chunks for fp32 W and
    # two fp32 moments); BT 512: 16-column chunks for one-state fp32 rules
    # too, three operand stages with bf16 weights; BT 600: three operand
    # stages where they fit.
    w, st = variant
    prob = _prob(shape, 21, w, st, exact=True)
    sr, srm = w == "bf16", st == "bf16" and NSTATE[rule] > 0
    for t in (1, 4):
        got, dx = run_backward(rule, prob, t, seed=77, sr_w=sr, sr_moments=srm)
        ref = oracle_step(rule, prob, w, st, t, seed=77, sr_w=sr, sr_moments=srm, mode="f32emu")
        assert_bit_exact(got, ref, rule)
        _check_dx(dx, prob, "bf16", exact=True)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dx_dtype", ["bf16", "f32"])
def test_fused_backward_exact_adamw_shapes(shape, dx_dtype):
    prob = _prob(shape, 22, "f32", "f32", exact=True)
    got, dx = run_backward("adamw", prob, 2, dx_dtype=dx_dtype)
    ref = oracle_step("adamw", prob, "f32", "f32", 2, mode="f32emu")
    assert_bit_exact(got, ref, "adamw")
    _check_dx(dx, prob, dx_dtype, exact=True)


# ---------------------------------------------------------------------------
# Random inputs: tolerance, and agreement between the two paths
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("variant", [("f32", "f32"), ("bf16", "bf16")], ids=lambda v: f"W{v[0]}-m{v[1]}")
def test_fused_backward_random_within_tolerance(rule, variant):
    w, st = variant
    prob = _prob((512, 640, 384), 23, w, st, exact=False)
    sr = w == "bf16"
    got, dx = run_backward(rule, prob, 3, dx_dtype="f32", seed=5, sr_w=sr)
    check_tolerance(rule, prob, w, st, 3, got, seed=5, sr_w=sr)
    _check_dx(dx, prob, "f32", exact=False)


@pytest.mark.parametrize("shape", [(512, 640, 384), (2048, 1024, 512)], ids=lambda s: "x".join(map(str, s)))
def test_fused_and_split_paths_agree(shape):
    # Same products in the same token order: the new state is bit-identical;
    # dX differs only in the fp32 summation order over D_out.
    prob = _prob(shape, 24, "f32", "f32", exact=False)
    a, dxa = run_backward("adamw", prob, 2, dx_dtype="f32", path="fused")
    b, dxb = run_backward("adamw", prob, 2, dx_dtype="f32", path="split")
    assert_bit_exact(a, b, "adamw")
    _, A = _dx_ref(prob)
    assert np.all(np.abs(dxa.astype(np.float64) - dxb) <= 2e-5 * A)


def test_fused_backward_is_deterministic():
    prob = _prob((2048, 1024, 512), 25, "f32", "f32", exact=False)
    a, dxa = run_backward("adamw", prob, 1, dx_dtype="f32")
    b, dxb = run_backward("adamw", prob, 1, dx_dtype="f32")
    assert_bit_exact(a, b, "adamw")
    assert np.array_equal(dxa.view(np.uint32), dxb.view(np.uint32))


def test_fused_backward_one_token():
    prob = _prob((384, 256, 1), 26, "f32", "f32", exact=True)
    got, dx = run_backward("adamw", prob, 1)
    assert_bit_exact(got, oracle_step("adamw", prob, "f32", "f32", 1, mode="f32emu"), "adamw")
    _check_dx(dx, prob, "bf16", exact=True)


# ---------------------------------------------------------------------------
# Path selection, workspace contract, failure path
# ---------------------------------------------------------------------------

def test_workspace_bytes_geometry():
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def fused(d_out, d_in, bt):
        # one fp32 slab of ceil(BT/128)*128 x 64 per (CTA, tile column) of the fused pass
        if bt < 1 or bt > 768:
            return 0
        tm, tn = -(-d_out // 128), -(-d_in // 64)
        T = tm * tn
        G = min(T, sms)
        # the fewest CTAs with the same most tiles per CTA, if that idles >= 10 % of them
        per = -(-T // G)
        if 10 * -(-T // per) <= 9 * G:
            G = -(-T // per)
        runs = max((((c + 1) * T // G) - 1) // tm - (c * T // G) // tm + 1 for c in range(G))
        return G * runs * (-(-bt // 128) * 128 * 64) * 4

    def plan(d_out, d_in, bt, wbytes):
        # The input gradient's plan, costed by the bytes through the busiest
        # SM's shared memory: waves x multiply-adds per CTA (token blocks
        # padded to 128) x (2 / BN + (W bytes + 6 for fp32 W) / (128 MB)
        # + 2 / N + 2 / M for M x N products: 128 x BN, or 128 x 256 on
        # all-token tiles), x 1.2 for all-token tiles (x 1.4 for four blocks
        # with bf16 W), plus 740 KB for a split's fix-up. Candidates: 128-token
        # tiles (128 x 256 for bf16 W when those fill the GPU); the same split
        # in S = min(4, SMs // tiles) parts of >= 2048 rows where that puts
        # >= 1.5x as many SMs to work as 128 x 128 tiles (bf16 W on 128 x 256
        # tiles); all-token tiles (2 / 4 blocks of 128 tokens x 128 columns,
        # BT in (128, 512], 64-row stages) split in parts of >= 256 rows.
        def cost(mb, bn, bk, tiles_m, parts):
            tiles_n = -(-d_in // bn)
            P = parts if parts >= 2 else 1
            waves = -(-(tiles_m * tiles_n * P) // sms)
            operands = 2.0 / 256.0 + 2.0 / 128.0 if mb > 1 else 2.0 / bn + 2.0 / 128.0
            per_mac = 2.0 / bn + (wbytes + (6.0 if wbytes == 4 else 0.0)) / (128.0 * mb) + operands
            c = waves * (128.0 * mb * bn * (d_out / P)) * per_mac
            if mb > 1:
                c *= 1.4 if (mb == 4 and wbytes == 2) else 1.2
            if parts >= 2:
                c += 740e3
            nbytes = tiles_m * tiles_n * parts * 128 * mb * bn * 4 if parts >= 2 else 0
            return c, nbytes

        tm = -(-bt // 128)
        bn = 256 if wbytes == 2 and tm * -(-d_in // 256) >= sms else 128
        best = cost(1, bn, 128 if bn == 128 else 64, tm, 0)
        bn = 256 if wbytes == 2 else 128
        bk = 128 if bn == 128 else 64
        tiles, kb, tiles128 = tm * -(-d_in // bn), -(-d_out // bk), tm * -(-d_in // 128)
        parts = min(4, sms // tiles)
        while parts >= 2 and kb * (bk // 64) < 32 * parts:
            parts -= 1
        if parts >= 2 and 2 * tiles128 <= sms and 2 * tiles * parts >= 3 * tiles128:
            c = cost(1, bn, bk, tm, parts)
            if c[0] < best[0]:
                best = c
        if 128 < bt <= 512:
            mb, tiles_n, kb = (2 if bt <= 256 else 4), -(-d_in // 128), -(-d_out // 64)
            parts = min(4, sms // tiles_n)
            while parts >= 2 and kb * 64 < 256 * parts:
                parts -= 1
            c = cost(mb, 128, 64, 1, parts if parts >= 2 else 0)
            if c[0] < best[0]:
                best = c
        return best[1]

    def split(d_out, d_in, bt):
        return max(plan(d_out, d_in, bt, 4), plan(d_out, d_in, bt, 2)) if bt >= 1 else 0

    for shape in [(14336, 4096, 512), (4096, 14336, 512), (1024, 4096, 512), (136, 200, 70), (8, 8, 1),
                  (14336, 4096, 2048), (14336, 4096, 8192), (4096, 4096, 769), (14336, 4096, 256),
                  (14336, 4096, 128), (4096, 4096, 256), (8192, 2600, 512), (8192, 2600, 200), (8192, 520, 200),
                  (4096, 4096, 300), (14336, 4096, 129)]:
        assert F.workspace_bytes(*shape) == max(fused(*shape), split(*shape)), shape
    assert F.workspace_bytes(4096, 4096, 0) == 0


def test_forced_fused_without_workspace_is_an_error():
    prob = _prob((256, 256, 128), 27, "f32", "f32", exact=False)
    with pytest.raises(F.ForgeError) as ei:
        run_backward("adamw", prob, 1, workspace=False)
    assert ei.value.status == 1 and "workspace" in str(ei.value)


@pytest.mark.parametrize("bt", [800, 1024])
def test_long_token_axis_takes_the_split_path(bt):
    prob = _prob((256, 384, bt), 28, "f32", "f32", exact=True)
    with pytest.raises(F.ForgeError) as ei:
        run_backward("adamw", prob, 1, path="fused")
    assert ei.value.status == 2
    got, dx = run_backward("adamw", prob, 1, path="auto")
    assert_bit_exact(got, oracle_step("adamw", prob, "f32", "f32", 1, mode="f32emu"), "adamw")
    _check_dx(dx, prob, "bf16", exact=True)


def test_q8_state_takes_the_split_path():
    prob = S.linear_problem(256, 384, 128, seed=29, x_dtype="bf16", w_dtype="f32", state="q8", exact=True)
    X, dY, W = prob.X.to(DEV), prob.dY.to(DEV), prob.W.to(DEV)
    m, v, ms, vs = prob.m.to(DEV), prob.v.to(DEV), prob.m_scale.to(DEV), prob.v_scale.to(DEV)
    dX = torch.empty((128, 384), dtype=torch.bfloat16, device=DEV)
    # 8-bit state descriptors need their scales: go through the rule wrapper's descriptor path.
    tX, tdY, tW, tdX = (F.tensor_desc(t) for t in (X, dY, W, dX))
    tm, tv = F.tensor_desc(m, ms), F.tensor_desc(v, vs)
    import ctypes
    from backward_gemm_optimizer_gb300 import _lib
    h = _lib._hyper(1e-3, 0.9, 0.999, 1e-8, 0.01, False, False, F.FLAG_BACKWARD_FUSED)
    st = F.lib().forge_backward_step(0, ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tm),
                                     ctypes.byref(tv), ctypes.byref(tdX), ctypes.byref(h), 1, 0, None, 0,
                                     _lib._stream(None))
    assert st == 2


def test_auto_path_without_workspace_runs_split():
    prob = _prob((512, 384, 256), 30, "f32", "f32", exact=True)
    got, dx = run_backward("adamw", prob, 1, path="auto", workspace=False)
    assert_bit_exact(got, oracle_step("adamw", prob, "f32", "f32", 1, mode="f32emu"), "adamw")
    _check_dx(dx, prob, "bf16", exact=True)


def test_fused_forced_timeout_reports_and_leaves_state():
    prob = _prob((512, 512, 256), 31, "f32", "f32", exact=False)
    X, dY, W = prob.X.to(DEV), prob.dY.to(DEV), prob.W.to(DEV)
    m, v = prob.m.to(DEV), prob.v.to(DEV)
    dX = torch.empty((256, 512), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(F.workspace_bytes(512, 512, 256), dtype=torch.uint8, device=DEV)
    F.backward_step("adamw", X, dY, W, m, v, dX, step=1, workspace=ws,
                    flags=F.FLAG_BACKWARD_FUSED | F.FLAG_TEST_FORCE_TIMEOUT, **_hyper_kw("adamw"))
    with pytest.raises(F.ForgeError) as ei:
        F.sync_status()
    assert ei.value.status == 5
    assert torch.equal(W.cpu(), prob.W) and torch.equal(m.cpu(), prob.m) and torch.equal(v.cpu(), prob.v)
    F.backward_step("adamw", X, dY, W, m, v, dX, step=1, workspace=ws, flags=F.FLAG_BACKWARD_FUSED,
                    **_hyper_kw("adamw"))
    F.sync_status()
    assert not torch.equal(W.cpu(), prob.W)


@pytest.mark.parametrize("w", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(8192, 520, 200), (6144, 1024, 128)], ids=lambda s: "x".join(map(str, s)))
def test_split_path_input_gradient_split_contraction(w, shape):
    # Short token axes, long contraction: on the split path the input
    # gradient runs its contraction over D_out in parts on several SMs and a
    # second kernel adds the parts in a fixed order. Exact inputs: dX and the
    # state bit-exact; random inputs: within tolerance, run-to-run identical,
    # and equal to the one-kernel dgrad (forge_dgrad) up to summation order.
    d_out, d_in, bt = shape
    assert F.workspace_bytes(d_out, d_in, bt) > 0
    prob = _prob(shape, 29, w, w, exact=True)
    got, dx = run_backward("adamw", prob, 2, path="split", sr_w=w == "bf16", seed=3)
    ref = oracle_step("adamw", prob, w, w, 2, seed=3, sr_w=w == "bf16", mode="f32emu")
    assert_bit_exact(got, ref, "adamw")
    _check_dx(dx, prob, "bf16", exact=True)
    prob = _prob(shape, 30, w, w, exact=False)
    _, dx1 = run_backward("adamw", prob, 1, dx_dtype="f32", path="split", sr_w=w == "bf16")
    _, dx2 = run_backward("adamw", prob, 1, dx_dtype="f32", path="split", sr_w=w == "bf16")
    assert np.array_equal(dx1.view(np.uint32), dx2.view(np.uint32))
    _check_dx(dx1, prob, "f32", exact=False)
    dY, W = prob.dY.to(DEV), prob.W.to(DEV)
    dx3 = torch.empty((bt, d_in), dtype=torch.float32, device=DEV)
    F.dgrad(dY, W, dx3)
    F.sync_status()
    _, A = _dx_ref(prob)
    assert np.all(np.abs(dx1.astype(np.float64) - dx3.cpu().numpy()) <= 2e-5 * A)


@pytest.mark.parametrize("w", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(4096, 2600, 512), (4096, 2600, 300), (2048, 1000, 200), (1000, 520, 129)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("workspace", [True, False], ids=["split", "whole"])
def test_split_path_all_token_input_gradient(w, shape, workspace):
    # The input gradient on all-token tiles (FORGE_FLAG_DGRAD_ALL_TOKENS):
    # 4 blocks of 128 tokens (BT 512; BT 300: the last block empty, the third
    # ragged) or 2 (BT 200, 129), 128 features, ragged last column of tiles
    # and last stage (D_out 1000); with a workspace the contraction is split
    # in parts added by the fix-up kernel, without one each tile runs whole.
    # Exact inputs: state and dX bit-exact; random inputs: dX within
    # tolerance, run-to-run identical, and equal to the 128-token tiles'
    # dX up to summation order.
    d_out, d_in, bt = shape
    prob = _prob(shape, 31, w, w, exact=True)
    fl = F.FLAG_DGRAD_ALL_TOKENS
    got, dx = run_backward("adamw", prob, 2, path="split", sr_w=w == "bf16", seed=3, workspace=workspace, flags=fl)
    ref = oracle_step("adamw", prob, w, w, 2, seed=3, sr_w=w == "bf16", mode="f32emu")
    assert_bit_exact(got, ref, "adamw")
    _check_dx(dx, prob, "bf16", exact=True)
    prob = _prob(shape, 32, w, w, exact=False)
    kw = dict(dx_dtype="f32", path="split", sr_w=w == "bf16", workspace=workspace)
    _, dx1 = run_backward("adamw", prob, 1, flags=fl, **kw)
    _, dx2 = run_backward("adamw", prob, 1, flags=fl, **kw)
    assert np.array_equal(dx1.view(np.uint32), dx2.view(np.uint32))
    _check_dx(dx1, prob, "f32", exact=False)
    _, dx3 = run_backward("adamw", prob, 1, flags=F.FLAG_DGRAD_TOKENS_128, **kw)
    _, A = _dx_ref(prob)
    assert np.all(np.abs(dx1.astype(np.float64) - dx3) <= 2e-5 * A)


def test_all_token_input_gradient_needs_a_short_token_axis():
    prob = _prob((256, 256, 600), 33, "f32", "f32", exact=False)
    with pytest.raises(F.ForgeError) as ei:
        run_backward("adamw", prob, 1, path="split", flags=F.FLAG_DGRAD_ALL_TOKENS)
    assert ei.value.status == 2 and "all-token" in str(ei.value)
    with pytest.raises(F.ForgeError) as ei:
        run_backward("adamw", prob, 1, path="fused", flags=F.FLAG_DGRAD_TOKENS_128)
    assert ei.value.status == 1
