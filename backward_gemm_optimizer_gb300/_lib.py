"""ctypes binding of ``libforge.so`` (argument marshalling only).

Every function here fills the C descriptors of ``include/forge.h`` from
torch tensors and calls the library; all arithmetic runs in the library's
CUDA kernels. If the library has not been built the import fails loudly:
there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch  # loads the CUDA runtime the library links against

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libforge.so")

F32, BF16, I8B128 = 0, 1, 2
FLAG_TILE_N_AUTO, FLAG_TILE_N_128, FLAG_TILE_N_64, FLAG_TILE_N_256, FLAG_TILE_PAIR_256 = 0, 1, 2, 3, 4
FLAG_TEST_FORCE_TIMEOUT = 0x100
FLAG_BACKWARD_FUSED, FLAG_BACKWARD_SPLIT = 0x200, 0x400
FLAG_DGRAD_TOKENS_128, FLAG_DGRAD_ALL_TOKENS = 0x800, 0x1000
RULES = {"adamw": 0, "sgdm": 1, "lion": 2, "sgd": 3, "rmsprop": 4, "adagrad": 5, "nadam": 6, "radam": 7}

STATUS_NAMES = {0: "FORGE_OK", 1: "FORGE_ERR_INVALID_ARG", 2: "FORGE_ERR_UNSUPPORTED",
                3: "FORGE_ERR_ALIGNMENT", 4: "FORGE_ERR_CUDA", 5: "FORGE_ERR_TIMEOUT"}

EXPORTED = ("forge_wgrad_step_adamw", "forge_wgrad_step_sgdm", "forge_wgrad_step_lion",
            "forge_wgrad_step_sgd", "forge_wgrad_step_rmsprop", "forge_wgrad_step_adagrad",
            "forge_wgrad_step_nadam", "forge_wgrad_step_radam",
            "forge_dgrad", "forge_dgrad_ws", "forge_backward_step", "forge_backward_step_no_alloc",
            "forge_wgrad_accumulate",
            "forge_backward_accumulate", "forge_wgrad_step_accumulated", "forge_sync_status", "forge_last_error", "forge_version",
            "forge_workspace_bytes", "forge_selftest_math")


class ForgeTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ld", ctypes.c_int64), ("scale", ctypes.c_void_p)]


class ForgeHyper(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("sr_w", ctypes.c_int32), ("sr_moments", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("momentum_decay", ctypes.c_double)]


class ForgeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()'). There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    T, H = ForgeTensor, ForgeHyper
    vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
    lib.forge_wgrad_step_adamw.argtypes = [P(T), P(T), P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_wgrad_step_sgdm.argtypes = [P(T), P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_wgrad_step_lion.argtypes = [P(T), P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_wgrad_step_sgd.argtypes = [P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_wgrad_step_rmsprop.argtypes = [P(T), P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_wgrad_step_adagrad.argtypes = [P(T), P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_wgrad_step_nadam.argtypes = [P(T), P(T), P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_wgrad_step_radam.argtypes = [P(T), P(T), P(T), P(T), P(T), P(H), i64, u64, vp]
    lib.forge_dgrad.argtypes = [P(T), P(T), P(T), vp]
    lib.forge_dgrad_ws.argtypes = [P(T), P(T), P(T), vp, ctypes.c_size_t, vp]
    lib.forge_backward_step.argtypes = [ctypes.c_int, P(T), P(T), P(T), P(T), P(T), P(T), P(H), i64, u64, vp,
                                        ctypes.c_size_t, vp]
    lib.forge_backward_step_no_alloc.argtypes = [ctypes.c_int, P(T), P(T), P(T), P(T), P(T), P(T), P(H), i64,
                                                 u64, vp]
    lib.forge_wgrad_accumulate.argtypes = [P(T), P(T), P(T), ctypes.c_int, vp]
    lib.forge_backward_accumulate.argtypes = [P(T), P(T), P(T), P(T), P(T), ctypes.c_int, ctypes.c_uint32, vp,
                                              ctypes.c_size_t, vp]
    lib.forge_wgrad_step_accumulated.argtypes = [ctypes.c_int, P(T), P(T), P(T), P(T), P(T), P(T), P(H), i64, u64,
                                                 vp]
    lib.forge_sync_status.argtypes = [vp]
    for f in ("forge_wgrad_step_adamw", "forge_wgrad_step_sgdm", "forge_wgrad_step_lion",
              "forge_wgrad_step_sgd", "forge_wgrad_step_rmsprop", "forge_wgrad_step_adagrad",
              "forge_wgrad_step_nadam", "forge_wgrad_step_radam", "forge_dgrad", "forge_dgrad_ws", "forge_backward_step",
              "forge_backward_step_no_alloc", "forge_wgrad_accumulate", "forge_backward_accumulate",
              "forge_wgrad_step_accumulated",
              "forge_sync_status"):
        getattr(lib, f).restype = ctypes.c_int
    lib.forge_last_error.restype = ctypes.c_char_p
    lib.forge_version.restype = ctypes.c_char_p
    lib.forge_workspace_bytes.argtypes = [i64, i64, i64]
    lib.forge_workspace_bytes.restype = ctypes.c_size_t
    lib.forge_selftest_math.argtypes = [ctypes.c_int, u64, u64, P(u64), P(u64)]
    lib.forge_selftest_math.restype = ctypes.c_int
    return lib


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _check(status: int):
    if status != 0:
        raise ForgeError(status, lib().forge_last_error().decode())


def _dtype_code(t: torch.Tensor, scale: Optional[torch.Tensor]) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.int8, torch.uint8):
        if scale is None:
            raise ValueError("8-bit moment codes need their fp32 scale tensor [D_in/128, D_out]")
        return I8B128
    raise TypeError(f"unsupported dtype {t.dtype}")


def tensor_desc(t: torch.Tensor, scale: Optional[torch.Tensor] = None) -> ForgeTensor:
    """Descriptor of a 2-D tensor with unit column stride (rows may be padded)."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.numel() > 0 and t.stride(1) != 1:
        raise ValueError("columns must be contiguous (stride(1) == 1)")
    if scale is not None and (scale.dtype != torch.float32 or not scale.is_contiguous()):
        raise ValueError("scale must be a contiguous float32 tensor")
    ld = t.stride(0) if t.shape[0] > 1 else max(t.shape[1], t.stride(0))
    return ForgeTensor(ctypes.c_void_p(t.data_ptr() if t.numel() else 0), _dtype_code(t, scale),
                       t.shape[0], t.shape[1], max(ld, t.shape[1]),
                       ctypes.c_void_p(scale.data_ptr() if scale is not None else 0))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _hyper(lr, beta1, beta2, eps, weight_decay, sr_w, sr_moments, flags, momentum_decay=0.0) -> ForgeHyper:
    return ForgeHyper(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                      int(bool(sr_w)), int(bool(sr_moments)), int(flags), float(momentum_decay))


def wgrad_step_adamw(X, dY, W, m, v, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                     step, seed=0, sr_w=False, sr_moments=False, m_scale=None, v_scale=None,
                     flags=0, stream=None):
    """Fused G = dY^T X and AdamW step on W, m, v in place (forge_wgrad_step_adamw)."""
    tX, tdY, tW = tensor_desc(X), tensor_desc(dY), tensor_desc(W)
    tm, tv = tensor_desc(m, m_scale), tensor_desc(v, v_scale)
    h = _hyper(lr, beta1, beta2, eps, weight_decay, sr_w, sr_moments, flags)
    _check(lib().forge_wgrad_step_adamw(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW),
                                        ctypes.byref(tm), ctypes.byref(tv), ctypes.byref(h),
                                        int(step), int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream)))


def wgrad_step_sgdm(X, dY, W, m, *, lr, momentum=0.9, weight_decay=0.0, step, seed=0,
                    sr_w=False, sr_moments=False, m_scale=None, flags=0, stream=None):
    """Fused G = dY^T X and SGD-momentum step on W, m in place (forge_wgrad_step_sgdm)."""
    tX, tdY, tW, tm = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(m, m_scale)
    h = _hyper(lr, momentum, 0.0, 0.0, weight_decay, sr_w, sr_moments, flags)
    _check(lib().forge_wgrad_step_sgdm(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW),
                                       ctypes.byref(tm), ctypes.byref(h), int(step),
                                       int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream)))


def wgrad_step_lion(X, dY, W, m, *, lr, beta1=0.9, beta2=0.99, weight_decay=0.0, step, seed=0,
                    sr_w=False, sr_moments=False, m_scale=None, flags=0, stream=None):
    """Fused G = dY^T X and Lion step on W, m in place (forge_wgrad_step_lion)."""
    tX, tdY, tW, tm = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(m, m_scale)
    h = _hyper(lr, beta1, beta2, 0.0, weight_decay, sr_w, sr_moments, flags)
    _check(lib().forge_wgrad_step_lion(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW),
                                       ctypes.byref(tm), ctypes.byref(h), int(step),
                                       int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream)))


def _seed(seed):
    return int(seed) & 0xFFFFFFFFFFFFFFFF


def wgrad_step_sgd(X, dY, W, *, lr, weight_decay=0.0, step, seed=0, sr_w=False, flags=0, stream=None):
    """Fused G = dY^T X and plain SGD step on W in place (forge_wgrad_step_sgd)."""
    tX, tdY, tW = tensor_desc(X), tensor_desc(dY), tensor_desc(W)
    h = _hyper(lr, 0.0, 0.0, 0.0, weight_decay, sr_w, False, flags)
    _check(lib().forge_wgrad_step_sgd(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(h),
                                      int(step), _seed(seed), _stream(stream)))


def wgrad_step_rmsprop(X, dY, W, v, *, lr, alpha=0.99, eps=1e-8, weight_decay=0.0, step, seed=0, sr_w=False,
                       sr_moments=False, flags=0, stream=None):
    """Fused G = dY^T X and RMSprop step on W, v in place (forge_wgrad_step_rmsprop)."""
    tX, tdY, tW, tv = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(v)
    h = _hyper(lr, 0.0, alpha, eps, weight_decay, sr_w, sr_moments, flags)
    _check(lib().forge_wgrad_step_rmsprop(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tv),
                                          ctypes.byref(h), int(step), _seed(seed), _stream(stream)))


def wgrad_step_adagrad(X, dY, W, v, *, lr, eps=1e-10, weight_decay=0.0, step, seed=0, sr_w=False,
                       sr_moments=False, flags=0, stream=None):
    """Fused G = dY^T X and AdaGrad step on W, v in place (forge_wgrad_step_adagrad)."""
    tX, tdY, tW, tv = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(v)
    h = _hyper(lr, 0.0, 0.0, eps, weight_decay, sr_w, sr_moments, flags)
    _check(lib().forge_wgrad_step_adagrad(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tv),
                                          ctypes.byref(h), int(step), _seed(seed), _stream(stream)))


def wgrad_step_nadam(X, dY, W, m, v, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                     momentum_decay=4e-3, step, seed=0, sr_w=False, sr_moments=False, flags=0, stream=None):
    """Fused G = dY^T X and NAdam step on W, m, v in place (forge_wgrad_step_nadam)."""
    tX, tdY, tW, tm, tv = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(m), tensor_desc(v)
    h = _hyper(lr, beta1, beta2, eps, weight_decay, sr_w, sr_moments, flags, momentum_decay)
    _check(lib().forge_wgrad_step_nadam(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tm),
                                        ctypes.byref(tv), ctypes.byref(h), int(step), _seed(seed), _stream(stream)))


def wgrad_step_radam(X, dY, W, m, v, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step, seed=0,
                     sr_w=False, sr_moments=False, flags=0, stream=None):
    """Fused G = dY^T X and RAdam step on W, m, v in place (forge_wgrad_step_radam)."""
    tX, tdY, tW, tm, tv = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(m), tensor_desc(v)
    h = _hyper(lr, beta1, beta2, eps, weight_decay, sr_w, sr_moments, flags)
    _check(lib().forge_wgrad_step_radam(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tm),
                                        ctypes.byref(tv), ctypes.byref(h), int(step), _seed(seed), _stream(stream)))


def dgrad(dY, W_old, dX, *, workspace=None, stream=None):
    """dX = dY W_old (forge_dgrad, or forge_dgrad_ws given a `workspace` device tensor of
    workspace_bytes(D_out, D_in, BT) bytes); enqueue before the step that overwrites W."""
    tdY, tW, tdX = tensor_desc(dY), tensor_desc(W_old), tensor_desc(dX)
    if workspace is None:
        _check(lib().forge_dgrad(ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tdX), _stream(stream)))
    else:
        ws_bytes = workspace.numel() * workspace.element_size()
        _check(lib().forge_dgrad_ws(ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tdX),
                                    ctypes.c_void_p(workspace.data_ptr() if ws_bytes else 0), ws_bytes,
                                    _stream(stream)))


def backward_step(rule, X, dY, W, s0, s1, dX, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                  momentum_decay=4e-3, momentum=None, alpha=None, step, seed=0, sr_w=False, sr_moments=False,
                  workspace=None, flags=0, stream=None, m_scale=None, v_scale=None):
    """dX = dY W_old and the fused step of `rule` on W and its state (forge_backward_step).

    s0 / s1 are the rule's state tensors as the wgrad_step_<rule> call takes
    them (None where the rule has fewer); m_scale / v_scale are their block
    scales for 8-bit state. `momentum` (SGD-momentum) and `alpha` (RMSprop)
    are aliases of beta1 / beta2. `workspace`: a device tensor of at least
    workspace_bytes(D_out, D_in, BT) bytes enables the fused input-gradient
    path, and on the split path (dgrad, then the step) lets the input
    gradient spread over all SMs.
    """
    if rule not in RULES:
        raise ValueError(f"unknown rule {rule!r}; one of {tuple(RULES)}")
    if momentum is not None:
        beta1 = momentum
    if alpha is not None:
        beta2 = alpha
    tX, tdY, tW, tdX = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(dX)
    t0 = tensor_desc(s0, m_scale) if s0 is not None else None
    t1 = tensor_desc(s1, v_scale) if s1 is not None else None
    h = _hyper(lr, beta1, beta2, eps, weight_decay, sr_w, sr_moments, flags, momentum_decay)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr() if workspace is not None and workspace.numel() else 0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().forge_backward_step(RULES[rule], ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW),
                                     ctypes.byref(t0) if t0 is not None else None,
                                     ctypes.byref(t1) if t1 is not None else None, ctypes.byref(tdX),
                                     ctypes.byref(h), int(step), _seed(seed), ws_ptr, ws_bytes, _stream(stream)))


def backward_step_no_alloc(rule, X, dY, W, s0, s1, dX, *, lr, beta1=0.9, beta2=0.999, eps=1e-8,
                           weight_decay=0.0, momentum_decay=4e-3, momentum=None, alpha=None, step, seed=0,
                           sr_w=False, sr_moments=False, flags=0, stream=None):
    """backward_step on the fused path with the library's built-in scratch array
    (forge_backward_step_no_alloc): for callers that cannot allocate device memory."""
    if rule not in RULES:
        raise ValueError(f"unknown rule {rule!r}; one of {tuple(RULES)}")
    if momentum is not None:
        beta1 = momentum
    if alpha is not None:
        beta2 = alpha
    tX, tdY, tW, tdX = tensor_desc(X), tensor_desc(dY), tensor_desc(W), tensor_desc(dX)
    t0 = tensor_desc(s0) if s0 is not None else None
    t1 = tensor_desc(s1) if s1 is not None else None
    h = _hyper(lr, beta1, beta2, eps, weight_decay, sr_w, sr_moments, flags, momentum_decay)
    _check(lib().forge_backward_step_no_alloc(RULES[rule], ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW),
                                              ctypes.byref(t0) if t0 is not None else None,
                                              ctypes.byref(t1) if t1 is not None else None, ctypes.byref(tdX),
                                              ctypes.byref(h), int(step), _seed(seed), _stream(stream)))


def wgrad_accumulate(X, dY, G_acc, *, overwrite=False, stream=None):
    """G_acc (+)= dY^T X for one micro-batch (forge_wgrad_accumulate); overwrite on the first."""
    tX, tdY, tG = tensor_desc(X), tensor_desc(dY), tensor_desc(G_acc)
    _check(lib().forge_wgrad_accumulate(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tG), int(bool(overwrite)),
                                        _stream(stream)))


def backward_accumulate(X, dY, W, G_acc, dX, *, overwrite=False, workspace=None, flags=0, stream=None):
    """dX = dY W and G_acc (+)= dY^T X for a micro-batch that is not the window's last
    (forge_backward_accumulate): one pass when `workspace` (workspace_bytes(D_out, D_in, BT)
    bytes) is given and the layer allows it, else dgrad and wgrad_accumulate."""
    tX, tdY, tW, tG, tdX = (tensor_desc(t) for t in (X, dY, W, G_acc, dX))
    ws_ptr = ctypes.c_void_p(workspace.data_ptr() if workspace is not None and workspace.numel() else 0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().forge_backward_accumulate(ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tW), ctypes.byref(tG),
                                           ctypes.byref(tdX), int(bool(overwrite)), int(flags), ws_ptr, ws_bytes,
                                           _stream(stream)))


def wgrad_step_accumulated(rule, X, dY, G_acc, W, s0, s1, *, lr, beta1=0.9, beta2=0.999, eps=1e-8,
                           weight_decay=0.0, momentum_decay=4e-3, momentum=None, alpha=None, step, seed=0,
                           sr_w=False, sr_moments=False, flags=0, stream=None):
    """The last micro-batch: G = G_acc + dY^T X per tile, then the fused step of `rule`
    (forge_wgrad_step_accumulated). s0 / s1 as for backward_step."""
    if rule not in RULES:
        raise ValueError(f"unknown rule {rule!r}; one of {tuple(RULES)}")
    if momentum is not None:
        beta1 = momentum
    if alpha is not None:
        beta2 = alpha
    tX, tdY, tG, tW = tensor_desc(X), tensor_desc(dY), tensor_desc(G_acc), tensor_desc(W)
    t0 = tensor_desc(s0) if s0 is not None else None
    t1 = tensor_desc(s1) if s1 is not None else None
    h = _hyper(lr, beta1, beta2, eps, weight_decay, sr_w, sr_moments, flags, momentum_decay)
    _check(lib().forge_wgrad_step_accumulated(RULES[rule], ctypes.byref(tX), ctypes.byref(tdY), ctypes.byref(tG),
                                              ctypes.byref(tW), ctypes.byref(t0) if t0 is not None else None,
                                              ctypes.byref(t1) if t1 is not None else None, ctypes.byref(h),
                                              int(step), _seed(seed), _stream(stream)))


def sync_status(stream=None):
    """Synchronise the stream and raise ForgeError if a kernel's bounded wait gave up."""
    _check(lib().forge_sync_status(_stream(stream)))


def version() -> str:
    return lib().forge_version().decode()


def workspace_bytes(d_out: int, d_in: int, bt: int) -> int:
    return int(lib().forge_workspace_bytes(d_out, d_in, bt))


def selftest_math(which: int, first: int, count: int):
    """(mismatches, declined) of forge_selftest_math (test hook)."""
    mism, decl = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(lib().forge_selftest_math(int(which), int(first), int(count), ctypes.byref(mism), ctypes.byref(decl)))
    return mism.value, decl.value
