"""A PyTorch linear layer whose backward pass runs the fused step.

``ForgeLinear`` computes ``y = x W^T`` in its forward pass. Its backward
pass enqueues, on the current stream, one ``forge_backward_step``: the
input gradient ``dX = dY W`` from the weights before they change (FORGE
paper, Appendix A, Remark 1) and the fused weight-gradient + optimizer
step, which updates the weight and its optimizer state in place -- in one
pass over W where the library's policy takes the fused path (it gets a
workspace from a per-stream cache here), else as ``forge_dgrad`` followed
by ``forge_wgrad_step_<rule>``. ``W.grad`` is never formed:
the weight is a trainable parameter (so that autograd always reaches the
backward, whether or not the input needs a gradient), but the backward
returns no gradient for it.

``ForgeStepManager`` plays the role of the pages' optimizer manager: it
holds the hyper-parameters shared by the fused layers, and its
``pre_step(lr=...)`` advances the step counter (and optionally the
learning rate) before each forward/backward. With
``accumulation_steps = K > 1`` (exact gradient accumulation, FORGE
Appendix L) ``pre_step`` is called before every micro-batch: the first
K - 1 backward passes of a window add their weight gradients into a
per-layer fp32 accumulator, each in one pass with its input gradient
(``forge_backward_accumulate``), and the K-th fires
the fused step once on the whole window's gradient
(``forge_wgrad_step_accumulated``); the step counter advances once per
window.

Weights read by more than one backward path in a step (tied embeddings,
experts reduced across ranks) must not be fused (Remark 1); keep those on
a standard optimizer. The forward GEMM is a plain library GEMM
(``torch.nn.functional.linear``) on a bf16 view of the weights; every
backward computation runs in this library's kernels.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Iterable, List, Optional

import torch

from . import _lib as F

_RULES = ("adamw", "sgdm", "lion", "sgd", "rmsprop", "adagrad", "nadam", "radam")
_NSTATE = {"adamw": 2, "nadam": 2, "radam": 2, "sgdm": 1, "lion": 1, "rmsprop": 1, "adagrad": 1, "sgd": 0}


@dataclasses.dataclass
class StepConfig:
    """Hyper-parameters of the fused rule and the current step (1-based)."""

    rule: str = "adamw"
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    momentum_decay: float = 4e-3
    sr_w: bool = False
    sr_moments: bool = False
    seed: int = 0
    step: int = 0
    backward_flags: int = 0  # FLAG_BACKWARD_FUSED / FLAG_BACKWARD_SPLIT force a path; 0 = library policy
    accumulation_steps: int = 1  # micro-batches per optimizer step
    micro: int = 0               # 0-based micro-batch of the current window


# Workspaces of the fused backward path, one per (device, stream): calls on
# one stream run in order, so they can share one; grown on demand.
_WORKSPACES: Dict[tuple, torch.Tensor] = {}
_PATH_FLAGS = F.FLAG_BACKWARD_FUSED | F.FLAG_BACKWARD_SPLIT


def _workspace(device: torch.device, nbytes: int) -> Optional[torch.Tensor]:
    if nbytes <= 0:
        return None
    stream = torch.cuda.current_stream(device)
    key = (device.index, stream.cuda_stream)
    buf = _WORKSPACES.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _WORKSPACES[key] = buf
    return buf


class _ForgeLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x2d, weight, layer):
        ctx.layer = layer
        ctx.save_for_backward(x2d)
        w = weight if weight.dtype == x2d.dtype else weight.to(x2d.dtype)
        return torch.nn.functional.linear(x2d, w)

    @staticmethod
    def backward(ctx, dy2d):
        (x2d,) = ctx.saved_tensors
        layer: ForgeLinear = ctx.layer
        dy2d = dy2d.contiguous()
        dx = None
        if layer.config.accumulation_steps > 1:
            if ctx.needs_input_grad[0]:
                dx = torch.empty(x2d.shape, dtype=x2d.dtype, device=x2d.device)
            layer._accumulate(x2d, dy2d, dx)               # W is unchanged until the window's last micro-batch
        elif ctx.needs_input_grad[0]:
            dx = torch.empty(x2d.shape, dtype=x2d.dtype, device=x2d.device)
            layer._backward(x2d, dy2d, dx)                 # dX from W before the step (Remark 1)
        else:
            layer._fused_step(x2d, dy2d)
        return dx, None, None


class ForgeLinear(torch.nn.Module):
    """``y = x W^T`` (no bias) with the optimizer step fused into backward.

    weight_dtype: storage of W (float32 master weights or bfloat16).
    state_dtype: storage of the optimizer state (float32 or bfloat16).
    config: a StepConfig shared with a ForgeStepManager (one is made if None).
    """

    def __init__(self, in_features: int, out_features: int, *, rule: str = "adamw",
                 weight_dtype=torch.float32, state_dtype=torch.float32, config: Optional[StepConfig] = None,
                 device=None):
        super().__init__()
        if rule not in _RULES:
            raise ValueError(f"unknown rule {rule!r}; one of {_RULES}")
        self.in_features, self.out_features = in_features, out_features
        self.config = config if config is not None else StepConfig(rule=rule)
        self.config.rule = rule
        w = torch.empty((out_features, in_features), dtype=weight_dtype, device=device)
        torch.nn.init.normal_(w, std=0.02)
        self.weight = torch.nn.Parameter(w, requires_grad=True)
        n = _NSTATE[rule]
        for i, name in enumerate(("state0", "state1")):
            t = torch.zeros((out_features, in_features), dtype=state_dtype, device=device) if i < n else None
            self.register_buffer(name, t)

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, *, rule: str = "adamw", weight_dtype=torch.float32,
                    state_dtype=torch.float32, config: Optional[StepConfig] = None) -> "ForgeLinear":
        if linear.bias is not None:
            raise ValueError("ForgeLinear has no bias; keep biased layers on a standard optimizer")
        m = cls(linear.in_features, linear.out_features, rule=rule, weight_dtype=weight_dtype,
                state_dtype=state_dtype, config=config, device=linear.weight.device)
        with torch.no_grad():
            m.weight.copy_(linear.weight.to(weight_dtype))
        return m

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if not x.is_cuda:
            raise RuntimeError("ForgeLinear runs on CUDA tensors only (there is no CPU path)")
        if self.config.step < 1:
            raise RuntimeError("call ForgeStepManager.pre_step() (step counter is 0) before the first forward")
        shape = x.shape
        x2d = x.reshape(-1, self.in_features)
        if not x2d.is_contiguous():
            x2d = x2d.contiguous()
        y = _ForgeLinearFn.apply(x2d, self.weight, self)
        return y.reshape(*shape[:-1], self.out_features)

    def _accumulate(self, x2d: torch.Tensor, dy2d: torch.Tensor, dx: Optional[torch.Tensor]):
        c = self.config
        if getattr(self, "grad_acc", None) is None or self.grad_acc.shape != self.weight.shape:
            # The one gradient-shaped buffer of the accumulation mode, live for the run.
            self.grad_acc = torch.empty(self.weight.shape, dtype=torch.float32, device=self.weight.device)
        if c.micro < c.accumulation_steps - 1:
            if dx is None:
                F.wgrad_accumulate(x2d, dy2d, self.grad_acc, overwrite=(c.micro == 0))
            else:   # dX and the accumulation in one pass where the layer allows it
                ws = _workspace(x2d.device, F.workspace_bytes(self.out_features, self.in_features, x2d.shape[0]))
                F.backward_accumulate(x2d, dy2d, self.weight, self.grad_acc, dx, overwrite=(c.micro == 0),
                                      workspace=ws, flags=c.backward_flags & _PATH_FLAGS)
        else:
            if dx is not None:                             # from W before the step (Remark 1)
                ws = _workspace(x2d.device, F.workspace_bytes(self.out_features, self.in_features, x2d.shape[0]))
                F.dgrad(dy2d, self.weight, dx, workspace=ws)
            F.wgrad_step_accumulated(c.rule, x2d, dy2d, self.grad_acc, self.weight, self.state0, self.state1,
                                     lr=c.lr, beta1=c.beta1, beta2=c.beta2, eps=c.eps,
                                     weight_decay=c.weight_decay, momentum_decay=c.momentum_decay, step=c.step,
                                     seed=c.seed, sr_w=c.sr_w, sr_moments=c.sr_moments)

    def _backward(self, x2d: torch.Tensor, dy2d: torch.Tensor, dx: torch.Tensor):
        c = self.config
        ws = _workspace(x2d.device, F.workspace_bytes(self.out_features, self.in_features, x2d.shape[0]))
        F.backward_step(c.rule, x2d, dy2d, self.weight, self.state0, self.state1, dx, lr=c.lr, beta1=c.beta1,
                        beta2=c.beta2, eps=c.eps, weight_decay=c.weight_decay, momentum_decay=c.momentum_decay,
                        step=c.step, seed=c.seed, sr_w=c.sr_w, sr_moments=c.sr_moments, workspace=ws,
                        flags=c.backward_flags)

    def _fused_step(self, x2d: torch.Tensor, dy2d: torch.Tensor):
        c = self.config
        W, s0, s1 = self.weight, self.state0, self.state1
        common = dict(step=c.step, seed=c.seed, sr_w=c.sr_w)
        if c.rule == "adamw":
            F.wgrad_step_adamw(x2d, dy2d, W, s0, s1, lr=c.lr, beta1=c.beta1, beta2=c.beta2, eps=c.eps,
                               weight_decay=c.weight_decay, sr_moments=c.sr_moments, **common)
        elif c.rule == "sgdm":
            F.wgrad_step_sgdm(x2d, dy2d, W, s0, lr=c.lr, momentum=c.beta1, weight_decay=c.weight_decay,
                              sr_moments=c.sr_moments, **common)
        elif c.rule == "lion":
            F.wgrad_step_lion(x2d, dy2d, W, s0, lr=c.lr, beta1=c.beta1, beta2=c.beta2,
                              weight_decay=c.weight_decay, sr_moments=c.sr_moments, **common)
        elif c.rule == "sgd":
            F.wgrad_step_sgd(x2d, dy2d, W, lr=c.lr, weight_decay=c.weight_decay, **common)
        elif c.rule == "rmsprop":
            F.wgrad_step_rmsprop(x2d, dy2d, W, s0, lr=c.lr, alpha=c.beta2, eps=c.eps,
                                 weight_decay=c.weight_decay, sr_moments=c.sr_moments, **common)
        elif c.rule == "adagrad":
            F.wgrad_step_adagrad(x2d, dy2d, W, s0, lr=c.lr, eps=c.eps, weight_decay=c.weight_decay,
                                 sr_moments=c.sr_moments, **common)
        elif c.rule == "nadam":
            F.wgrad_step_nadam(x2d, dy2d, W, s0, s1, lr=c.lr, beta1=c.beta1, beta2=c.beta2, eps=c.eps,
                               weight_decay=c.weight_decay, momentum_decay=c.momentum_decay,
                               sr_moments=c.sr_moments, **common)
        else:
            F.wgrad_step_radam(x2d, dy2d, W, s0, s1, lr=c.lr, beta1=c.beta1, beta2=c.beta2, eps=c.eps,
                               weight_decay=c.weight_decay, sr_moments=c.sr_moments, **common)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, rule={self.config.rule}, "
                f"weight={self.weight.dtype}, state={None if self.state0 is None else self.state0.dtype}")


class ForgeStepManager:
    """Shared step configuration of a model's ForgeLinear layers.

    pre_step(lr=...) advances the 1-based step counter (and sets the learning
    rate) before the forward/backward in which the fused layers update.
    """

    def __init__(self, model: torch.nn.Module, config: Optional[StepConfig] = None, accumulation_steps: int = 1):
        if accumulation_steps < 1:
            raise ValueError("accumulation_steps must be >= 1")
        self.layers: List[ForgeLinear] = [m for m in model.modules() if isinstance(m, ForgeLinear)]
        self.config = config if config is not None else (self.layers[0].config if self.layers else StepConfig())
        for m in self.layers:
            m.config = self.config
        self.config.accumulation_steps = accumulation_steps
        self.config.micro = accumulation_steps - 1  # the first pre_step opens a window
        self._fused_ids = {id(m.weight) for m in self.layers}
        self._model = model

    def pre_step(self, lr: Optional[float] = None):
        """Call before each forward/backward (each micro-batch when accumulating)."""
        c = self.config
        if lr is not None:
            c.lr = float(lr)
        c.micro = (c.micro + 1) % c.accumulation_steps
        if c.micro == 0:
            c.step += 1

    def get_non_fused_params(self) -> Iterable[torch.nn.Parameter]:
        """Parameters a standard optimizer should still step (norms, embeddings...)."""
        return [p for p in self._model.parameters() if id(p) not in self._fused_ids and p.requires_grad]

    def fused_params(self) -> Iterable[torch.nn.Parameter]:
        """The weights stepped inside backward (leave them out of any other optimizer)."""
        return [m.weight for m in self.layers]

    def state_dict(self) -> Dict:
        return dataclasses.asdict(self.config)

    def load_state_dict(self, d: Dict):
        for k, v in d.items():
            setattr(self.config, k, v)


def replace_linears(model: torch.nn.Module, *, rule: str = "adamw", weight_dtype=torch.float32,
                    state_dtype=torch.float32, config: Optional[StepConfig] = None) -> StepConfig:
    """Swap every bias-free nn.Linear of `model` for a ForgeLinear sharing one StepConfig."""
    cfg = config if config is not None else StepConfig(rule=rule)
    for parent in list(model.modules()):
        for name, child in list(parent.named_children()):
            if isinstance(child, torch.nn.Linear) and child.bias is None:
                setattr(parent, name, ForgeLinear.from_linear(child, rule=rule, weight_dtype=weight_dtype,
                                                              state_dtype=state_dtype, config=cfg))
    return cfg
