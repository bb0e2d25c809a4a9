"""The C-ABI library: it loads, exports every entry point include/forge.h
declares, and rejects bad arguments on the host with the documented
status codes before any device work (CPU only, no compute calls)."""

import ctypes
import os
import re
import subprocess

import pytest

import backward_gemm_optimizer_gb300 as F
from backward_gemm_optimizer_gb300._lib import ForgeHyper, ForgeTensor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "forge.h")

OK, INVALID, UNSUPPORTED, ALIGNMENT = 0, 1, 2, 3


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(forge_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("forge_wgrad_step_adamw", "forge_wgrad_step_sgdm", "forge_wgrad_step_lion", "forge_dgrad",
              "forge_sync_status", "forge_last_error"):
        assert n in names


def test_binding_flags_match_the_header():
    # Every FORGE_FLAG_* value the header defines (the tile-width mask
    # aside) has a binding constant of the same value.
    src = open(HEADER).read()
    flags = dict(re.findall(r"#define FORGE_FLAG_([A-Z0-9_]+) (0x[0-9a-fA-F]+|[0-9]+)u", src))
    assert "TILE_PAIR_256" in flags and "DGRAD_ALL_TOKENS" in flags
    for name, val in flags.items():
        if name == "TILE_N_MASK":
            continue
        assert getattr(F, "FLAG_" + name) == int(val, 0), name


def test_library_exports_every_declared_symbol():
    lib = F.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", F.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (forge_\w+)", out))
    assert set(declared_functions()) <= exported
    assert set(F.EXPORTED) == set(declared_functions())


def test_version_and_workspace():
    assert re.match(r"\d+\.\d+\.\d+", F.version())
    assert F.workspace_bytes(14336, 4096, 512) == 0


def _t(data=0x1000, dtype=1, rows=4, cols=8, ld=None, scale=0):
    return ForgeTensor(ctypes.c_void_p(data), dtype, rows, cols, cols if ld is None else ld, ctypes.c_void_p(scale))


def _h(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, sr_w=0, sr_moments=0, flags=0)
    d.update(kw)
    return ForgeHyper(**d)


def _adamw(X, dY, W, m, v, h, step=1):
    lib = F.lib()
    r = lib.forge_wgrad_step_adamw(ctypes.byref(X), ctypes.byref(dY), ctypes.byref(W), ctypes.byref(m),
                                   ctypes.byref(v), ctypes.byref(h), step, 0, None)
    return r, lib.forge_last_error().decode()


def _shapes(bt=16, d_in=64, d_out=32, xdt=1, wdt=0, mdt=0):
    return (_t(dtype=xdt, rows=bt, cols=d_in), _t(dtype=xdt, rows=bt, cols=d_out),
            _t(dtype=wdt, rows=d_out, cols=d_in), _t(dtype=mdt, rows=d_out, cols=d_in),
            _t(dtype=mdt, rows=d_out, cols=d_in))


@pytest.mark.parametrize("step", [0, -3])
def test_step_must_be_positive(step):
    r, msg = _adamw(*_shapes(), _h(), step=step)
    assert r == INVALID and "step" in msg


def test_null_arguments():
    lib = F.lib()
    X, dY, W, m, v = _shapes()
    h = _h()
    r = lib.forge_wgrad_step_adamw(None, ctypes.byref(dY), ctypes.byref(W), ctypes.byref(m), ctypes.byref(v),
                                   ctypes.byref(h), 1, 0, None)
    assert r == INVALID
    r = lib.forge_dgrad(None, None, None, None)
    assert r == INVALID
    r = lib.forge_dgrad_ws(None, None, None, None, 0, None)
    assert r == INVALID


def test_shape_mismatch():
    X, dY, W, m, v = _shapes()
    W.rows = 31
    r, msg = _adamw(X, dY, W, m, v, _h())
    assert r == INVALID and "W" in msg


def test_mixed_input_dtypes_unsupported():
    X, dY, W, m, v = _shapes()
    dY.dtype = 0
    assert _adamw(X, dY, W, m, v, _h())[0] == UNSUPPORTED


def test_misaligned_base_and_pitch():
    X, dY, W, m, v = _shapes()
    X.data = ctypes.c_void_p(0x1008)
    assert _adamw(X, dY, W, m, v, _h())[0] == ALIGNMENT
    X, dY, W, m, v = _shapes()
    W.ld = 65                                   # 260-byte fp32 row pitch
    assert _adamw(X, dY, W, m, v, _h())[0] == ALIGNMENT


def test_dims_must_be_multiples_of_8():
    X, dY, W, m, v = _shapes(d_in=60, d_out=32)
    for t in (X, W, m, v):
        t.ld = 64
    assert _adamw(X, dY, W, m, v, _h())[0] == UNSUPPORTED


def test_q8_needs_scales_and_128_columns():
    X, dY, W, m, v = _shapes(d_in=64, mdt=2)
    m.scale = ctypes.c_void_p(0x2000); v.scale = ctypes.c_void_p(0x3000)
    assert _adamw(X, dY, W, m, v, _h())[0] == UNSUPPORTED       # 64 % 128 != 0
    X, dY, W, m, v = _shapes(d_in=128, mdt=2)
    assert _adamw(X, dY, W, m, v, _h())[0] == INVALID            # no scale arrays


def test_moment_dtypes_must_match_and_sr_needs_bf16():
    X, dY, W, m, v = _shapes()
    v.dtype = 1
    assert _adamw(X, dY, W, m, v, _h())[0] == UNSUPPORTED
    assert _adamw(*_shapes(), _h(sr_w=1))[0] == INVALID          # fp32 W
    assert _adamw(*_shapes(), _h(sr_moments=1))[0] == INVALID    # fp32 moments


def test_bad_hyper_parameters_and_flags():
    assert _adamw(*_shapes(), _h(lr=float("nan")))[0] == INVALID
    assert _adamw(*_shapes(), _h(beta2=1.0))[0] == INVALID
    assert _adamw(*_shapes(), _h(flags=0x8000))[0] == INVALID


def test_empty_weight_is_a_no_op():
    # D_out = 0: nothing to update, no device work, OK.
    assert _adamw(*_shapes(d_out=0), _h())[0] == OK


def test_dgrad_validation():
    lib = F.lib()
    dY, W, dX = _t(rows=16, cols=32), _t(dtype=0, rows=32, cols=64), _t(dtype=1, rows=16, cols=64)
    dY.dtype = 0
    assert lib.forge_dgrad(ctypes.byref(dY), ctypes.byref(W), ctypes.byref(dX), None) == UNSUPPORTED
    assert lib.forge_dgrad_ws(ctypes.byref(dY), ctypes.byref(W), ctypes.byref(dX), None, 0, None) == UNSUPPORTED
    dY.dtype = 1
    W.rows = 31
    assert lib.forge_dgrad(ctypes.byref(dY), ctypes.byref(W), ctypes.byref(dX), None) == INVALID
    assert lib.forge_dgrad_ws(ctypes.byref(dY), ctypes.byref(W), ctypes.byref(dX), None, 0, None) == INVALID


def test_backward_step_host_checks():
    lib = F.lib()
    X, dY, W, m, v = _shapes()
    dX = _t(dtype=1, rows=16, cols=64)
    h = _h()
    args = (ctypes.byref(X), ctypes.byref(dY), ctypes.byref(W), ctypes.byref(m), ctypes.byref(v),
            ctypes.byref(dX), ctypes.byref(h), 1, 0, None, 0, None)
    assert lib.forge_backward_step(99, *args) == INVALID                     # unknown rule
    assert lib.forge_backward_step(-1, *args) == INVALID
    h2 = _h(flags=F.FLAG_BACKWARD_FUSED | F.FLAG_BACKWARD_SPLIT)
    r = lib.forge_backward_step(0, ctypes.byref(X), ctypes.byref(dY), ctypes.byref(W), ctypes.byref(m),
                                ctypes.byref(v), ctypes.byref(dX), ctypes.byref(h2), 1, 0, None, 0, None)
    assert r == INVALID and "both" in lib.forge_last_error().decode()
    bad_dx = _t(dtype=2, rows=16, cols=64)
    r = lib.forge_backward_step(0, ctypes.byref(X), ctypes.byref(dY), ctypes.byref(W), ctypes.byref(m),
                                ctypes.byref(v), ctypes.byref(bad_dx), ctypes.byref(h), 1, 0, None, 0, None)
    assert r == UNSUPPORTED                                                  # dX must be bf16 or f32
    assert lib.forge_backward_step_no_alloc(7, None, None, None, None, None, None, None, 1, 0, None) == INVALID


def test_accumulation_host_checks():
    lib = F.lib()
    X, dY, W, m, v = _shapes()
    G = _t(dtype=0, rows=32, cols=64)
    h = _h()
    assert lib.forge_wgrad_accumulate(ctypes.byref(X), ctypes.byref(dY), None, 0, None) == INVALID
    G16 = _t(dtype=1, rows=32, cols=64)
    assert lib.forge_wgrad_accumulate(ctypes.byref(X), ctypes.byref(dY), ctypes.byref(G16), 0, None) == UNSUPPORTED
    Xf, dYf = _t(dtype=0, rows=16, cols=64), _t(dtype=0, rows=16, cols=32)
    assert lib.forge_wgrad_accumulate(ctypes.byref(Xf), ctypes.byref(dYf), ctypes.byref(G), 1, None) == UNSUPPORTED
    r = lib.forge_wgrad_step_accumulated(42, ctypes.byref(X), ctypes.byref(dY), ctypes.byref(G), ctypes.byref(W),
                                         ctypes.byref(m), ctypes.byref(v), ctypes.byref(h), 1, 0, None)
    assert r == INVALID
    r = lib.forge_wgrad_step_accumulated(0, ctypes.byref(X), ctypes.byref(dY), None, ctypes.byref(W),
                                         ctypes.byref(m), ctypes.byref(v), ctypes.byref(h), 1, 0, None)
    assert r == INVALID
    Gbad = _t(dtype=0, rows=31, cols=64)
    r = lib.forge_wgrad_step_accumulated(0, ctypes.byref(X), ctypes.byref(dY), ctypes.byref(Gbad), ctypes.byref(W),
                                         ctypes.byref(m), ctypes.byref(v), ctypes.byref(h), 1, 0, None)
    assert r == INVALID and "G_acc" in lib.forge_last_error().decode()


def test_backward_accumulate_host_checks():
    lib = F.lib()
    X, dY, W, m, v = _shapes()
    G = _t(dtype=0, rows=32, cols=64)
    dX = _t(dtype=1, rows=16, cols=64)
    b = ctypes.byref
    f = lib.forge_backward_accumulate
    assert f(b(X), b(dY), None, b(G), b(dX), 0, 0, None, 0, None) == INVALID             # null W
    assert f(b(X), b(dY), b(W), None, b(dX), 0, 0, None, 0, None) == INVALID             # null G_acc
    assert f(b(X), b(dY), b(W), b(G), b(dX), 0, 0x1, None, 0, None) == INVALID           # not a path flag
    both = F.FLAG_BACKWARD_FUSED | F.FLAG_BACKWARD_SPLIT
    assert f(b(X), b(dY), b(W), b(G), b(dX), 0, both, None, 0, None) == INVALID
    assert "both" in lib.forge_last_error().decode()
    bad_dx = _t(dtype=2, rows=16, cols=64)
    assert f(b(X), b(dY), b(W), b(G), b(bad_dx), 0, 0, None, 0, None) == UNSUPPORTED    # dX must be bf16 / f32
    short_dx = _t(dtype=1, rows=15, cols=64)
    assert f(b(X), b(dY), b(W), b(G), b(short_dx), 0, 0, None, 0, None) == INVALID      # dX is BT x D_in
    w8 = _t(dtype=2, rows=32, cols=64, scale=0x2000)
    assert f(b(X), b(dY), b(w8), b(G), b(dX), 0, 0, None, 0, None) == UNSUPPORTED       # W is f32 or bf16
    Xf, dYf = _t(dtype=0, rows=16, cols=64), _t(dtype=0, rows=16, cols=32)
    assert f(b(Xf), b(dYf), b(W), b(G), b(dX), 0, 0, None, 0, None) == UNSUPPORTED      # bf16 inputs only
    assert f(b(Xf), b(dYf), b(W), b(G), b(dX), 0, F.FLAG_BACKWARD_FUSED, None, 0, None) == UNSUPPORTED


def test_selftest_math_argument_checks():
    # Host-side checks only (no device work): a bad selector, range or
    # null output pointer is FORGE_ERR_INVALID_ARG.
    lib = F.lib()
    out = ctypes.c_uint64(0)
    assert lib.forge_selftest_math(3, 0, 1, ctypes.byref(out), ctypes.byref(out)) == INVALID
    assert lib.forge_selftest_math(0, 0, 1, None, ctypes.byref(out)) == INVALID
    assert lib.forge_selftest_math(0, 1 << 32, 1, ctypes.byref(out), ctypes.byref(out)) == INVALID
    assert lib.forge_selftest_math(2, (1 << 46) - 1, 2, ctypes.byref(out), ctypes.byref(out)) == INVALID
