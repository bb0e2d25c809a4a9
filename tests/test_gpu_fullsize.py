"""Full-size parity at the Llama-3.1-8B up-projection shape (W 14336 x 4096,
BT = 512 and the BT sweep), in the launch configuration the benchmark
times (forge_backward_step with its workspace: the fused input-gradient
pass at BT 512): the whole layer runs on the GPU; the oracle recomputes a
sample of rows (every column of each sampled row, so every column tile and
every 8-bit block of those rows is covered) and a sample of dX rows (the
full contraction over D_out) from the same inputs."""

import numpy as np
import pytest
import torch

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300 import synthetic as S
import oracle.forge_oracle as O
import oracle.tolerance as T

from forge_cases import HYPER, check_tolerance, to_np

pytestmark = pytest.mark.gpu

D_OUT, D_IN = 14336, 4096


def _sample_rows(d_out, n, seed):
    rs = np.random.RandomState(seed)
    rows = np.sort(rs.choice(d_out, size=n, replace=False))
    return np.unique(np.concatenate([rows, [0, 127, 128, d_out - 1]]))


def _row_problem(prob, rows):
    """The sampled rows of W / moments with all of X and the matching dY columns."""
    sub = S.LinearProblem(X=prob.X, dY=prob.dY[:, torch.from_numpy(rows)].contiguous(),
                          W=prob.W[torch.from_numpy(rows)], m=prob.m[torch.from_numpy(rows)],
                          v=prob.v[torch.from_numpy(rows)] if prob.v is not None else None)
    if prob.m_scale is not None:
        sub.m_scale = prob.m_scale[:, torch.from_numpy(rows)].contiguous()
        sub.v_scale = prob.v_scale[:, torch.from_numpy(rows)].contiguous()
    return sub


def _gpu_full(prob, *, sr_w, t=1):
    """The layer's backward pass as the benchmark launches it. fp32 / bf16
    state: one forge_backward_step with a workspace of workspace_bytes() and
    no path flag (the fused input-gradient pass at BT 512; dgrad + step past
    768 tokens). 8-bit state: forge_dgrad, then the step."""
    dev = "cuda:0"
    X, dY, W, m, v = (prob.X.to(dev), prob.dY.to(dev), prob.W.to(dev), prob.m.to(dev), prob.v.to(dev))
    ms = prob.m_scale.to(dev) if prob.m_scale is not None else None
    vs = prob.v_scale.to(dev) if prob.v_scale is not None else None
    dX = torch.empty((X.shape[0], D_IN), dtype=torch.bfloat16, device=dev)
    if ms is None:
        ws = torch.empty(max(16, F.workspace_bytes(D_OUT, D_IN, X.shape[0])), dtype=torch.uint8, device=dev)
        F.backward_step("adamw", X, dY, W, m, v, dX, step=t, seed=1234, sr_w=sr_w, workspace=ws, **HYPER["adamw"])
    else:
        F.dgrad(dY, W, dX)
        F.wgrad_step_adamw(X, dY, W, m, v, m_scale=ms, v_scale=vs, step=t, seed=1234, sr_w=sr_w, **HYPER["adamw"])
    F.sync_status()
    return W, m, v, ms, vs, dX


@pytest.mark.parametrize("w,st,bt", [("f32", "f32", 512), ("bf16", "bf16", 512), ("bf16", "bf16", 2048),
                                     ("bf16", "bf16", 8192), ("f32", "q8", 512)],
                         ids=["f32state-bt512", "bf16state-bt512", "bf16state-bt2048", "bf16state-bt8192",
                              "q8state-bt512"])
def test_up_proj_full_size_sampled_rows(w, st, bt):
    zr = 0.3 if st == "q8" else 0.0
    prob = S.linear_problem(D_OUT, D_IN, bt, seed=2, x_dtype="bf16", w_dtype=w, state=st, zero_row_fraction=zr)
    W, m, v, ms, vs, dX = _gpu_full(prob, sr_w=(w == "bf16"))
    rows = _sample_rows(D_OUT, 24, 5)
    # the same rows, taken from the full-size GPU result
    got = O.State(W=to_np(W[torch.from_numpy(rows).cuda()]), m=to_np(m[torch.from_numpy(rows).cuda()]),
                  v=to_np(v[torch.from_numpy(rows).cuda()]),
                  m_scale=to_np(ms[:, torch.from_numpy(rows).cuda()]) if ms is not None else None,
                  v_scale=to_np(vs[:, torch.from_numpy(rows).cuda()]) if vs is not None else None)
    sub = _row_problem(prob, rows)
    # Stochastic rounding is keyed on the element index p * D_in + q of the
    # full matrix: check W by recomputing each row's draws at its own index.
    rep = check_tolerance("adamw", sub, w, st, 1, got, seed=1234, sr_w=False)  if w == "f32" else None
    if w == "bf16":
        h = O.Hyper(**HYPER["adamw"])
        st0 = O.State(W=to_np(sub.W), m=to_np(sub.m), v=to_np(sub.v), w_dtype=w, state=st)
        Xn, dYn = sub.X.float().numpy(), sub.dY.float().numpy()
        G = O.wgrad_f64(dYn, Xn); A = O.abs_wgrad_f64(dYn, Xn)
        W1, m1, v1 = O.adamw_f64(O.load_w(st0), O.load_m(st0), O.load_v(st0), G, h, 1)
        r16 = np.stack([O.sr_draws(1234, 1, O.SITE_W, 1, D_IN, row0=int(p), total_cols=D_IN)[0] for p in rows])
        ref_w = O.f32_to_bf16_sr(W1.astype(np.float32), r16)
        tw, tm, tv = T.adamw_tol(O.load_w(st0), O.load_m(st0), O.load_v(st0), G, A, h, 1)
        d = T.bf16_ulp_distance(got.W, ref_w)
        gv = O.bf16_bits_to_f32(got.W).astype(np.float64); rv = O.bf16_bits_to_f32(ref_w).astype(np.float64)
        assert T.rel_violation(gv, rv, tw + np.maximum(T.bf16_ulp(got.W), T.bf16_ulp(ref_w))) <= 1.0
        assert np.mean(d != 0) <= 1e-3, np.mean(d != 0)
        for name, g_, r_, tol in (("m", got.m, O.f64_to_bf16_rne(m1), tm), ("v", got.v, O.f64_to_bf16_rne(v1), tv)):
            gv = O.bf16_bits_to_f32(g_).astype(np.float64); rv = O.bf16_bits_to_f32(r_).astype(np.float64)
            assert T.rel_violation(gv, rv, tol + np.maximum(T.bf16_ulp(g_), T.bf16_ulp(r_))) <= 1.0, name
    # dX for the sampled token rows: the full contraction over D_out.
    toks = _sample_rows(bt, 8, 6)
    w16 = O.bf16_bits_to_f32(O.f32_to_bf16_rne(prob.W.float().numpy())).astype(np.float64)
    dYt = prob.dY[torch.from_numpy(toks)].float().numpy().astype(np.float64)
    ref = dYt @ w16
    tol = 1e-5 * (np.abs(dYt) @ np.abs(w16)) + np.abs(ref) * 2 ** -8      # bf16 output rounding
    gx = dX[torch.from_numpy(toks).cuda()].float().cpu().numpy()
    assert np.all(np.abs(gx - ref) <= tol)
    if rep is not None:
        print(w, st, bt, rep)


def test_up_proj_accumulation_window_full_size():
    # The accumulation benchmark's window at full size: three micro-batches
    # through forge_backward_accumulate (dX and G_acc in one pass), the last
    # through forge_dgrad + forge_wgrad_step_accumulated. The sampled rows of
    # the new state must match one AdamW step on the concatenated batch, and
    # every micro-batch's sampled dX rows the product with the window's W.
    dev, nmb, bt = "cuda:0", 4, 512
    prob = S.linear_problem(D_OUT, D_IN, bt, seed=7, x_dtype="bf16", w_dtype="f32", state="f32")
    mbs = [(S.normal((bt, D_IN), 1.0, 70 + i, S.STREAM_X, "bf16"), S.normal((bt, D_OUT), 1.0, 70 + i, S.STREAM_DY, "bf16"))
           for i in range(nmb)]
    W, m, v = prob.W.to(dev), prob.m.to(dev), prob.v.to(dev)
    G = torch.empty_like(W)
    ws = torch.empty(F.workspace_bytes(D_OUT, D_IN, bt), dtype=torch.uint8, device=dev)
    dxs = []
    for i, (X, dY) in enumerate(mbs):
        Xd, dYd = X.to(dev), dY.to(dev)
        dX = torch.empty((bt, D_IN), dtype=torch.bfloat16, device=dev)
        if i < nmb - 1:
            F.backward_accumulate(Xd, dYd, W, G, dX, overwrite=(i == 0), workspace=ws, flags=F.FLAG_BACKWARD_FUSED)
        else:
            F.dgrad(dYd, W, dX)
            F.wgrad_step_accumulated("adamw", Xd, dYd, G, W, m, v, step=1, **HYPER["adamw"])
        dxs.append(dX)
    F.sync_status()
    rows = _sample_rows(D_OUT, 24, 5)
    idx = torch.from_numpy(rows).cuda()
    got = O.State(W=to_np(W[idx]), m=to_np(m[idx]), v=to_np(v[idx]))
    cat = S.LinearProblem(**{**prob.__dict__, "X": torch.cat([x for x, _ in mbs]),
                             "dY": torch.cat([d for _, d in mbs])})
    print("accumulation window", check_tolerance("adamw", _row_problem(cat, rows), "f32", "f32", 1, got))
    w16 = O.bf16_bits_to_f32(O.f32_to_bf16_rne(prob.W.float().numpy())).astype(np.float64)
    toks = _sample_rows(bt, 8, 6)
    for (_, dY), dX in zip(mbs, dxs):
        dYt = dY[torch.from_numpy(toks)].float().numpy().astype(np.float64)
        ref = dYt @ w16
        tol = 1e-5 * (np.abs(dYt) @ np.abs(w16)) + np.abs(ref) * 2 ** -8      # bf16 output rounding
        gx = dX[torch.from_numpy(toks).cuda()].float().cpu().numpy()
        assert np.all(np.abs(gx - ref) <= tol)
