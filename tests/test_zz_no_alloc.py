"""forge_backward_step_no_alloc: the fused backward pass for callers that
cannot allocate device memory (a framework allocator that owns the whole
device, a plug-in handed tensors but no allocator, a host that forbids
allocation once training runs). Its scratch is an array built into the
library, so its results must be those of forge_backward_step given a
caller-allocated workspace, call after call, although the array keeps
whatever the previous call left in it.

This file is collected last, so a run that stops at the first failure has
already run every other test.
"""

import numpy as np
import pytest
import torch

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


@pytest.mark.parametrize("shape", [(2048, 1024, 512), (1000, 520, 300)], ids=lambda s: "x".join(map(str, s)))
def test_no_alloc_matches_backward_step_on_two_calls(shape):
    d_out, d_in, bt = shape
    prob = S.linear_problem(d_out, d_in, bt, seed=41, x_dtype="bf16", w_dtype="f32", state="f32",
                            w_bf16_representable=False)
    X, dY = prob.X.to(DEV), prob.dY.to(DEV)
    ref = [prob.W.to(DEV), prob.m.to(DEV), prob.v.to(DEV)]
    got = [t.clone() for t in ref]
    ws = torch.empty(F.workspace_bytes(d_out, d_in, bt), dtype=torch.uint8, device=DEV)
    for t in (1, 2):  # two calls in a row: the second sees the first call's leftovers in the array
        dx_ref = torch.empty((bt, d_in), dtype=torch.float32, device=DEV)
        dx_got = torch.full((bt, d_in), float("nan"), dtype=torch.float32, device=DEV)
        F.backward_step("adamw", X, dY, ref[0], ref[1], ref[2], dx_ref, step=t, workspace=ws,
                        flags=F.FLAG_BACKWARD_FUSED, **HP)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats(DEV)
        base = torch.cuda.max_memory_allocated(DEV)
        free0 = torch.cuda.mem_get_info(DEV)[0]
        F.backward_step_no_alloc("adamw", X, dY, got[0], got[1], got[2], dx_got, step=t, **HP)
        F.sync_status()
        if t == 2:
            # The defining property: once the array is loaded (first call), a
            # call allocates nothing, neither from torch's allocator nor from
            # the driver.
            assert torch.cuda.max_memory_allocated(DEV) == base
            assert torch.cuda.mem_get_info(DEV)[0] > free0 - (8 << 20)
        # Same kernels, same inputs, fixed summation order: identical bits.
        for a, b, name in zip(got + [dx_got], ref + [dx_ref], ("W", "m", "v", "dX")):
            assert np.array_equal(_bits(a), _bits(b)), f"call {t}: {name} differs"


def test_no_alloc_rejects_a_layer_beyond_its_scratch():
    # 128 x 29184 at BT 768: 456 one-tile columns spread over the CTAs, so a
    # CTA writes several partial slabs -- more than the 64 MiB array holds.
    d_out, d_in, bt = 128, 29184, 768
    need = F.workspace_bytes(d_out, d_in, bt)
    assert need > (64 << 20)
    X = torch.zeros((bt, d_in), dtype=torch.bfloat16, device=DEV)
    dY = torch.zeros((bt, d_out), dtype=torch.bfloat16, device=DEV)
    W = torch.ones((d_out, d_in), dtype=torch.float32, device=DEV)
    m, v = torch.zeros_like(W), torch.zeros_like(W)
    dX = torch.empty((bt, d_in), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(F.ForgeError) as ei:
        F.backward_step_no_alloc("adamw", X, dY, W, m, v, dX, step=1, **HP)
    assert ei.value.status == 2 and "scratch" in str(ei.value)
    F.sync_status()
    assert bool((W == 1).all())  # rejected before any work
