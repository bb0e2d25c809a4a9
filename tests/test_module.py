"""ForgeLinear / ForgeStepManager: the autograd layer over the C ABI.

GPU: its backward gives exactly what forge_dgrad and the fused step give
when called directly (bit for bit), the weight gradient is never formed,
and the manager drives the step counter and learning rate. CPU: there is
no CPU path, and misuse fails loudly."""

import pytest
import torch

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300.module import ForgeLinear, ForgeStepManager, StepConfig, replace_linears


def test_cpu_tensors_are_rejected():
    layer = ForgeLinear(16, 8)
    ForgeStepManager(layer).pre_step(lr=1e-3)
    with pytest.raises(RuntimeError, match="CUDA"):
        layer(torch.zeros(4, 16))


def test_unknown_rule_and_bias_rejected():
    with pytest.raises(ValueError):
        ForgeLinear(16, 8, rule="adafactor")
    with pytest.raises(ValueError):
        ForgeLinear.from_linear(torch.nn.Linear(16, 8, bias=True))


def test_manager_lists_non_fused_params():
    model = torch.nn.Sequential(torch.nn.Linear(16, 16, bias=False), torch.nn.LayerNorm(16),
                                torch.nn.Linear(16, 8, bias=False))
    cfg = replace_linears(model, rule="lion")
    mgr = ForgeStepManager(model, cfg)
    assert len(mgr.layers) == 2 and all(isinstance(m, ForgeLinear) for m in mgr.layers)
    assert {id(p) for p in mgr.get_non_fused_params()} == {id(p) for p in model[1].parameters()}
    mgr.pre_step(lr=3e-6)
    mgr.pre_step()
    assert cfg.step == 2 and cfg.lr == 3e-6
    sd = mgr.state_dict()
    cfg2 = StepConfig()
    ForgeStepManager(torch.nn.Sequential(ForgeLinear(4, 4, config=cfg2))).load_state_dict(sd)
    assert cfg2.step == 2 and cfg2.rule == "lion"


@pytest.mark.gpu
@pytest.mark.parametrize("path", ["auto", "fused"])
@pytest.mark.parametrize("rule", ["adamw", "sgdm", "lion", "nadam", "rmsprop"])
def test_backward_equals_direct_abi_calls(rule, path):
    torch.manual_seed(0)
    dev = "cuda:0"
    layer = ForgeLinear(384, 256, rule=rule, device=dev)
    mgr = ForgeStepManager(layer)
    mgr.config.lr, mgr.config.weight_decay = 1e-3, 0.01
    mgr.config.backward_flags = F.FLAG_BACKWARD_FUSED if path == "fused" else 0
    x = torch.randn(2, 100, 384, device=dev).bfloat16().requires_grad_(True)
    g = torch.randn(2, 100, 256, device=dev).bfloat16()
    W0 = layer.weight.detach().clone()
    s0 = None if layer.state0 is None else layer.state0.clone()
    s1 = None if layer.state1 is None else layer.state1.clone()
    for step in (1, 2):
        mgr.pre_step()
        if step == 2:
            W0 = layer.weight.detach().clone()
            s0 = None if layer.state0 is None else layer.state0.clone()
            s1 = None if layer.state1 is None else layer.state1.clone()
        x.grad = None
        y = layer(x)
        (y.float() * g.float()).sum().backward()
        F.sync_status()
    assert layer.weight.grad is None                      # the weight gradient never exists
    # the same step through the C ABI directly
    x2d, dy2d = x.detach().reshape(-1, 384), g.reshape(-1, 256).contiguous()
    dx = torch.empty_like(x2d)
    c = mgr.config
    ws = torch.empty(max(16, F.workspace_bytes(256, 384, x2d.shape[0])), dtype=torch.uint8, device=dev)
    F.backward_step(rule, x2d, dy2d, W0, s0, s1, dx, lr=c.lr, beta1=c.beta1, beta2=c.beta2, eps=c.eps,
                    weight_decay=c.weight_decay, momentum_decay=c.momentum_decay, step=2, seed=c.seed,
                    workspace=ws, flags=c.backward_flags)
    F.sync_status()
    assert torch.equal(layer.weight, W0)
    assert torch.equal(x.grad.reshape(-1, 384), dx)
    if s0 is not None:
        assert torch.equal(layer.state0, s0)
    if s1 is not None:
        assert torch.equal(layer.state1, s1)


@pytest.mark.gpu
def test_small_model_trains_with_fused_layers():
    torch.manual_seed(1)
    dev = "cuda:0"
    model = torch.nn.Sequential(torch.nn.Linear(256, 512, bias=False), torch.nn.GELU(),
                                torch.nn.Linear(512, 256, bias=False)).to(dev)
    cfg = replace_linears(model, rule="adamw", weight_dtype=torch.float32)
    mgr = ForgeStepManager(model, cfg)
    cfg.weight_decay = 0.0
    x = torch.randn(64, 256, device=dev).bfloat16()
    target = torch.randn(64, 256, device=dev).bfloat16()
    losses = []
    for step in range(30):
        mgr.pre_step(lr=1e-2 if step < 20 else 3e-3)
        y = model(x)
        loss = ((y.float() - target.float()) ** 2).mean()
        loss.backward()
        losses.append(float(loss.detach()))
    F.sync_status()
    assert losses[-1] < 0.7 * losses[0], losses
    assert all(m.weight.grad is None for m in mgr.layers)


@pytest.mark.gpu
@pytest.mark.parametrize("rule", ["adamw", "lion"])
def test_accumulation_window_equals_one_step_on_the_whole_batch(rule):
    # Exact gradient accumulation (Appendix L): K micro-batches through the
    # layer with accumulation_steps = K update W exactly as one step on the
    # concatenated batch (integer-valued inputs: every sum is exact).
    dev = "cuda:0"
    torch.manual_seed(3)
    K, d_in, d_out = 3, 256, 384
    xs = [torch.randint(-3, 4, (n, d_in), device=dev).bfloat16() for n in (64, 100, 37)]
    gs = [torch.randint(-3, 4, (n, d_out), device=dev).bfloat16() for n in (64, 100, 37)]
    acc = ForgeLinear(d_in, d_out, rule=rule, device=dev)
    one = ForgeLinear(d_in, d_out, rule=rule, device=dev)
    with torch.no_grad():
        one.weight.copy_(acc.weight)
    m_acc = ForgeStepManager(acc, accumulation_steps=K)
    m_one = ForgeStepManager(one)
    for cfg in (m_acc.config, m_one.config):
        cfg.lr, cfg.weight_decay = 1e-3, 0.01
    W0 = acc.weight.detach().clone()
    w16 = W0.bfloat16().double()
    for x, g in zip(xs, gs):
        m_acc.pre_step()
        x = x.clone().requires_grad_(True)
        (acc(x).float() * g.float()).sum().backward()
        if m_acc.config.micro < K - 1:
            assert torch.equal(acc.weight, W0)          # no step before the window's last micro-batch
        # dX of every micro-batch from the window's (unchanged) weights:
        # fp32 sums of the bf16 products, one bf16 rounding.
        ref = g.double() @ w16
        tol = 1e-5 * (g.double().abs() @ w16.abs()) + ref.abs() * 2.0 ** -8
        assert torch.all((x.grad.double() - ref).abs() <= tol)
    m_one.pre_step()
    xc = torch.cat(xs).requires_grad_(True)
    (one(xc).float() * torch.cat(gs).float()).sum().backward()
    F.sync_status()
    assert m_acc.config.step == m_one.config.step == 1
    assert torch.equal(acc.weight, one.weight)
    assert torch.equal(acc.state0, one.state0)
    if acc.state1 is not None:
        assert torch.equal(acc.state1, one.state1)


@pytest.mark.gpu
def test_backward_allocates_no_weight_gradient():
    # Proposition 3: the weight gradient never exists in HBM. Through the
    # layer: no W.grad, and the backward pass allocates only dX (4 MB here),
    # far below one fp32 gradient (64 MB). Through the C ABI with caller
    # buffers: the call allocates nothing, from torch or from the driver.
    dev = "cuda:0"
    d_in, d_out, bt = 4096, 4096, 512
    layer = ForgeLinear(d_in, d_out, device=dev)
    mgr = ForgeStepManager(layer)
    mgr.pre_step(lr=1e-3)
    x = torch.randn(bt, d_in, device=dev).bfloat16().requires_grad_(True)
    g = torch.randn(bt, d_out, device=dev).bfloat16()
    layer(x).backward(g)                              # first call creates the shared workspace
    mgr.pre_step()
    x.grad = None
    y = layer(x)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    y.backward(g)
    torch.cuda.synchronize()
    F.sync_status()
    assert layer.weight.grad is None
    assert torch.cuda.max_memory_allocated() - base < (d_out * d_in * 4) // 8

    X, dY = x.detach(), g
    W = layer.weight.detach()
    m, v = layer.state0, layer.state1
    dX = torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(F.workspace_bytes(d_out, d_in, bt), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    for flags in (F.FLAG_BACKWARD_FUSED, F.FLAG_BACKWARD_SPLIT):
        F.backward_step("adamw", X, dY, W, m, v, dX, lr=1e-3, step=3, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    F.sync_status()
    assert torch.cuda.max_memory_allocated() == base
    assert torch.cuda.mem_get_info()[0] > free0 - 8 * 2 ** 20     # no driver-level allocation either


@pytest.mark.gpu
@pytest.mark.parametrize("rule,wdt,sdt", [("adamw", torch.float32, torch.float32),
                                          ("lion", torch.bfloat16, torch.bfloat16),
                                          ("sgdm", torch.float32, torch.float32)],
                         ids=["adamw-f32", "lion-bf16-sr", "sgdm-f32"])
def test_layer_matches_oracle_over_steps_with_changing_lr(rule, wdt, sdt):
    # The user-facing layer (ForgeLinear + ForgeStepManager.pre_step(lr=...))
    # against the CPU oracle: three backward passes with a different learning
    # rate each, fresh seeded inputs each step. After every step the layer's
    # W and moments are one oracle step (at the manager's 1-based step count
    # and lr) from the state before it, and dX is dY W_old (Appendix A,
    # Remark 1). A wrong step counter, a stale lr or a dX from the updated
    # weights fails the comparison.
    import numpy as np
    import oracle.forge_oracle as O
    from backward_gemm_optimizer_gb300 import synthetic as S
    from forge_cases import HYPER, check_tolerance, to_np

    dev = "cuda:0"
    d_in, d_out, bt = 384, 256, 200
    torch.manual_seed(3)
    layer = ForgeLinear(d_in, d_out, rule=rule, weight_dtype=wdt, state_dtype=sdt, device=dev)
    hp = dict(HYPER[rule])
    mgr = ForgeStepManager(layer)
    c = mgr.config
    c.beta1, c.beta2, c.eps, c.weight_decay = hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"]
    c.sr_w, c.seed = wdt == torch.bfloat16, 99
    w_kind = "bf16" if wdt == torch.bfloat16 else "f32"
    s_kind = "bf16" if sdt == torch.bfloat16 else "f32"
    with torch.no_grad():   # non-zero moments from the start, so the bias corrections matter
        layer.state0.copy_(S.normal((d_out, d_in), 1e-3, 5, S.STREAM_M, s_kind).to(dev))
        if layer.state1 is not None:
            layer.state1.copy_(S.abs_normal((d_out, d_in), 1e-6, 5, S.STREAM_V, s_kind).to(dev))
    lrs = [hp["lr"], hp["lr"] * 0.5, hp["lr"] * 0.2]
    for t, lr in enumerate(lrs, start=1):
        X, dY = S.step_inputs(d_out, d_in, bt, 11, t, "bf16")
        prob = S.LinearProblem(X=X, dY=dY, W=layer.weight.detach().cpu().clone(),
                               m=layer.state0.detach().cpu().clone(),
                               v=None if layer.state1 is None else layer.state1.detach().cpu().clone())
        mgr.pre_step(lr=lr)
        assert c.step == t and c.lr == lr
        x = X.to(dev).requires_grad_(True)
        y = layer(x)
        y.backward(dY.to(dev))
        torch.cuda.synchronize()
        F.sync_status()
        assert layer.weight.grad is None
        got = O.State(W=to_np(layer.weight), m=to_np(layer.state0),
                      v=None if layer.state1 is None else to_np(layer.state1))
        rep = check_tolerance(rule, prob, w_kind, s_kind, t, got, seed=99, sr_w=c.sr_w,
                              hyper={**hp, "lr": lr})
        w16 = O.bf16_bits_to_f32(O.f32_to_bf16_rne(prob.W.float().numpy())).astype(np.float64)
        ref = O.dgrad_f64(dY.float().numpy(), w16)
        tol = 1e-5 * (np.abs(dY.float().numpy()).astype(np.float64) @ np.abs(w16)) + np.abs(ref) * 2 ** -8
        viol = float(np.max(np.abs(x.grad.float().cpu().numpy() - ref) / np.maximum(tol, 1e-300)))
        assert viol <= 1.0, (t, viol)
        print(rule, "step", t, "lr", lr, rep, "dX", viol)
