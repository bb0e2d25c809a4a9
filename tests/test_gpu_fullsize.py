"""Full-size parity at the Llama-3.1-8B linear shapes (up/gate 14336 x 4096,
down 4096 x 14336, q/o 4096 x 4096, k/v 1024 x 4096; BT = 512 and the BT
sweep), in the launch configuration the benchmarks time: one
forge_backward_step per layer with a workspace of workspace_bytes() and no
path flag, so the library takes the path it takes in the stack benchmark
(the fused input-gradient pass where it applies, dgrad + step elsewhere).
The whole layer runs on the GPU; the oracle recomputes a sample of rows
(every column of each sampled row, so every column tile and every 8-bit
block of those rows is covered) and a sample of dX rows (the full
contraction over D_out) from the same inputs. Hyper-parameters: AdamW as in
the fp32 problem, Lion and SGD-momentum from the paper's Appendix N,
Table 20."""

import numpy as np
import pytest
import torch

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300 import synthetic as S
import oracle.forge_oracle as O

from forge_cases import HYPER, assert_bit_exact, check_tolerance, oracle_state, to_np

pytestmark = pytest.mark.gpu

SHAPES = {"up": (14336, 4096), "down": (4096, 14336), "q": (4096, 4096), "k": (1024, 4096)}
SEED = 1234


def _sample_rows(d_out, n, seed):
    rs = np.random.RandomState(seed)
    rows = np.sort(rs.choice(d_out, size=n, replace=False))
    return np.unique(np.concatenate([rows, [0, 127, 128, d_out - 1]]))


def _row_problem(prob, rows):
    """The sampled rows of W / moments with all of X and the matching dY columns."""
    idx = torch.from_numpy(rows)
    sub = S.LinearProblem(X=prob.X, dY=prob.dY[:, idx].contiguous(), W=prob.W[idx],
                          m=prob.m[idx] if prob.m is not None else None,
                          v=prob.v[idx] if prob.v is not None else None)
    if prob.m_scale is not None:
        sub.m_scale = prob.m_scale[:, idx].contiguous()
        sub.v_scale = prob.v_scale[:, idx].contiguous() if prob.v_scale is not None else None
    return sub


def _gpu_backward(opt, prob, *, sr_w, t=1):
    """The layer's backward pass as the benchmarks launch it."""
    dev = "cuda:0"
    d_out, d_in = prob.W.shape
    X, dY, W = prob.X.to(dev), prob.dY.to(dev), prob.W.to(dev)
    m = prob.m.to(dev) if prob.m is not None else None
    v = prob.v.to(dev) if (prob.v is not None and O.NSTATE[opt] == 2) else None
    ms = prob.m_scale.to(dev) if prob.m_scale is not None else None
    vs = prob.v_scale.to(dev) if (prob.v_scale is not None and v is not None) else None
    dX = torch.empty((X.shape[0], d_in), dtype=torch.bfloat16, device=dev)
    hp = dict(HYPER[opt])
    common = dict(step=t, seed=SEED, sr_w=sr_w)
    if ms is None:
        ws = torch.empty(max(16, F.workspace_bytes(d_out, d_in, X.shape[0])), dtype=torch.uint8, device=dev)
        common["workspace"] = ws
        if opt == "adamw":
            F.backward_step("adamw", X, dY, W, m, v, dX, **hp, **common)
        elif opt == "lion":
            F.backward_step("lion", X, dY, W, m, None, dX, lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"],
                            weight_decay=hp["weight_decay"], **common)
        else:
            F.backward_step("sgdm", X, dY, W, m, None, dX, lr=hp["lr"], momentum=hp["beta1"],
                            weight_decay=hp["weight_decay"], **common)
    else:
        F.dgrad(dY, W, dX)
        F.wgrad_step_adamw(X, dY, W, m, v, m_scale=ms, v_scale=vs, **hp, **common)
    F.sync_status()
    return W, m, v, ms, vs, dX


def _gather(rows, W, m, v, ms, vs):
    idx = torch.from_numpy(rows).cuda()
    return O.State(W=to_np(W[idx]), m=to_np(m[idx]) if m is not None else None,
                   v=to_np(v[idx]) if v is not None else None,
                   m_scale=to_np(ms[:, idx]) if ms is not None else None,
                   v_scale=to_np(vs[:, idx]) if vs is not None else None)


def _check_dx(prob, dX, seed=6):
    """Sampled dX rows over the full D_out contraction with the pre-step W
    (Appendix A, Remark 1), rounded to bf16 as the tensor cores see it."""
    bt = prob.X.shape[0]
    toks = _sample_rows(bt, 8, seed) if bt > 8 else np.arange(bt)
    w16 = O.bf16_bits_to_f32(O.f32_to_bf16_rne(prob.W.float().numpy())).astype(np.float64)
    dYt = prob.dY[torch.from_numpy(toks)].float().numpy().astype(np.float64)
    ref = O.dgrad_f64(dYt, w16)
    tol = 1e-5 * (np.abs(dYt) @ np.abs(w16)) + np.abs(ref) * 2 ** -8      # bf16 output rounding
    gx = dX[torch.from_numpy(toks).cuda()].float().cpu().numpy()
    viol = float(np.max(np.abs(gx - ref) / np.maximum(tol, 1e-300)))
    assert viol <= 1.0, viol
    return viol


def _full_size_case(opt, name, w, st, bt, seed):
    d_out, d_in = SHAPES[name]
    zr = 0.3 if st == "q8" else 0.0
    prob = S.linear_problem(d_out, d_in, bt, seed=seed, x_dtype="bf16", w_dtype=w, state=st,
                            two_moments=O.NSTATE[opt] == 2, zero_row_fraction=zr)
    sr_w = w == "bf16"
    W, m, v, ms, vs, dX = _gpu_backward(opt, prob, sr_w=sr_w)
    rows = _sample_rows(d_out, 24, 5)
    got = _gather(rows, W, m, v, ms, vs)
    rep = check_tolerance(opt, _row_problem(prob, rows), w, st, 1, got, seed=SEED, sr_w=sr_w, rows=rows)
    rep["dX"] = _check_dx(prob, dX)
    print(opt, name, w, st, bt, rep)


@pytest.mark.parametrize("w,st,bt", [("f32", "f32", 512), ("bf16", "bf16", 512), ("bf16", "bf16", 2048),
                                     ("bf16", "bf16", 8192), ("f32", "q8", 512)],
                         ids=["f32state-bt512", "bf16state-bt512", "bf16state-bt2048", "bf16state-bt8192",
                              "q8state-bt512"])
def test_up_proj_full_size_sampled_rows(w, st, bt):
    _full_size_case("adamw", "up", w, st, bt, seed=2)


STACK_CASES = [(opt, name, st) for name in ("up", "down", "q", "k") for opt in ("adamw", "lion", "sgdm")
               for st in ("f32", "bf16") if not (name == "up" and opt == "adamw")]


@pytest.mark.parametrize("opt,name,st", STACK_CASES, ids=[f"{o}-{n}-{s}state" for o, n, s in STACK_CASES])
def test_stack_shapes_full_size_sampled_rows(opt, name, st):
    # Every shape and rule of the 224-linear stack benchmark, fp32 W + fp32
    # moments or bf16 W (stochastic rounding) + bf16 moments, BT = 512.
    _full_size_case(opt, name, "f32" if st == "f32" else "bf16", st, 512, seed=3)


def test_up_proj_q8_exact_gradient_codes_bit_exact():
    # Integer-valued X, dY: the gradient is exact, so the quantiser sees the
    # same fp32 inputs on both sides and every 8-bit code, scale and weight of
    # the sampled rows must equal the oracle's fp32 op sequence bit for bit.
    d_out, d_in = SHAPES["up"]
    prob = S.linear_problem(d_out, d_in, 512, seed=4, x_dtype="bf16", w_dtype="f32", state="q8", exact=True,
                            zero_row_fraction=0.3)
    W, m, v, ms, vs, dX = _gpu_backward("adamw", prob, sr_w=False)
    rows = _sample_rows(d_out, 24, 8)
    got = _gather(rows, W, m, v, ms, vs)
    sub = _row_problem(prob, rows)
    ref = O.step("adamw", sub.X.float().numpy(), sub.dY.float().numpy(), oracle_state(sub, "f32", "q8"),
                 O.Hyper(**HYPER["adamw"]), 1, mode="f32emu", rows=rows)
    assert_bit_exact(got, ref, "adamw")
    print("q8 exact full size: 0 of", got.m.size, "m codes and", got.v.size, "v codes differ")


def test_up_proj_accumulation_window_full_size():
    # The accumulation benchmark's window at full size: three micro-batches
    # through forge_backward_accumulate (dX and G_acc in one pass), the last
    # through forge_dgrad + forge_wgrad_step_accumulated. The sampled rows of
    # the new state must match one AdamW step on the concatenated batch, and
    # every micro-batch's sampled dX rows the product with the window's W.
    dev, nmb, bt = "cuda:0", 4, 512
    d_out, d_in = SHAPES["up"]
    prob = S.linear_problem(d_out, d_in, bt, seed=7, x_dtype="bf16", w_dtype="f32", state="f32")
    mbs = [(S.normal((bt, d_in), 1.0, 70 + i, S.STREAM_X, "bf16"), S.normal((bt, d_out), 1.0, 70 + i, S.STREAM_DY, "bf16"))
           for i in range(nmb)]
    W, m, v = prob.W.to(dev), prob.m.to(dev), prob.v.to(dev)
    G = torch.empty_like(W)
    ws = torch.empty(F.workspace_bytes(d_out, d_in, bt), dtype=torch.uint8, device=dev)
    dxs = []
    for i, (X, dY) in enumerate(mbs):
        Xd, dYd = X.to(dev), dY.to(dev)
        dX = torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev)
        if i < nmb - 1:
            F.backward_accumulate(Xd, dYd, W, G, dX, overwrite=(i == 0), workspace=ws, flags=F.FLAG_BACKWARD_FUSED)
        else:
            F.dgrad(dYd, W, dX)
            F.wgrad_step_accumulated("adamw", Xd, dYd, G, W, m, v, step=1, **HYPER["adamw"])
        dxs.append(dX)
    F.sync_status()
    rows = _sample_rows(d_out, 24, 5)
    idx = torch.from_numpy(rows).cuda()
    got = O.State(W=to_np(W[idx]), m=to_np(m[idx]), v=to_np(v[idx]))
    cat = S.LinearProblem(**{**prob.__dict__, "X": torch.cat([x for x, _ in mbs]),
                             "dY": torch.cat([d for _, d in mbs])})
    print("accumulation window", check_tolerance("adamw", _row_problem(cat, rows), "f32", "f32", 1, got))
    for (X, dY), dX in zip(mbs, dxs):
        _check_dx(S.LinearProblem(X=X, dY=dY, W=prob.W, m=None, v=None), dX)
