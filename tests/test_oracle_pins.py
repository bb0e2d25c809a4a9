"""Pins of the CPU oracle against what the FORGE paper and the mathematics fix.

None of these tests compares the oracle with itself: each checks it
against brute force, a hand-computed example, a closed form, an exact
expectation, an independent implementation (Philox), or a bound the
paper proves. CPU only.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle.forge_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _hyper(d):
    return O.Hyper(lr=d["lr"], beta1=d["beta1"], beta2=d["beta2"], eps=d["eps"],
                   weight_decay=d["weight_decay"])


# ---------------------------------------------------------------------------
# Phase 1: the gradient against a brute-force triple loop (Eq. 3)
# ---------------------------------------------------------------------------

def test_wgrad_brute_force_triple_loop():
    rs = np.random.RandomState(1)
    for (bt, d_out, d_in) in [(1, 1, 1), (3, 2, 5), (7, 4, 3), (5, 6, 6)]:
        dY = rs.randn(bt, d_out)
        X = rs.randn(bt, d_in)
        G = O.wgrad_f64(dY, X)
        assert G.shape == (d_out, d_in)
        for p in range(d_out):
            for q in range(d_in):
                s = 0.0
                for t in range(bt):
                    s += dY[t, p] * X[t, q]
                assert abs(G[p, q] - s) <= 1e-12 * (1 + abs(s))
        A = O.abs_wgrad_f64(dY, X)
        assert np.all(A >= np.abs(G) - 1e-12)


def test_wgrad_empty_token_axis_is_zero():
    G = O.wgrad_f64(np.zeros((0, 3)), np.zeros((0, 4)))
    assert G.shape == (3, 4) and np.all(G == 0)


# ---------------------------------------------------------------------------
# Proposition 1: per-tile fused update == materialise-then-step, any tile
# partition and any token partition (brute force, exact integer inputs)
# ---------------------------------------------------------------------------

def _random_partition(n, rs):
    cuts = sorted(set(rs.randint(1, n, size=rs.randint(0, n)).tolist())) if n > 1 else []
    edges = [0] + cuts + [n]
    return [(edges[i], edges[i + 1]) for i in range(len(edges) - 1)]


@pytest.mark.parametrize("opt", ["adamw", "sgdm", "lion"])
@pytest.mark.parametrize("mode", ["f64", "f32emu"])
def test_prop1_tile_partition_exact(opt, mode):
    rs = np.random.RandomState(7)
    h = O.Hyper(lr=1e-2, beta1=0.9, beta2=0.99 if opt == "lion" else 0.999, eps=1e-8,
                weight_decay=0.1)
    for trial in range(6):
        d_out, d_in, bt = rs.randint(1, 17), rs.randint(1, 17), rs.randint(1, 9)
        dY = rs.randint(-3, 4, size=(bt, d_out)).astype(np.float64)
        X = rs.randint(-3, 4, size=(bt, d_in)).astype(np.float64)
        W = (rs.randn(d_out, d_in) * 0.02).astype(np.float32)
        m = (rs.randn(d_out, d_in) * 1e-3).astype(np.float32)
        v = np.abs(rs.randn(d_out, d_in) * 1e-6).astype(np.float32)
        st = O.State(W=W, m=m, v=v if opt == "adamw" else None)
        t = 3
        whole = O.step(opt, X, dY, st, h, t, mode=mode)

        # Tile-fused schedule: irregular row/column tiles, each tile's G
        # accumulated over an irregular token partition with scalar loops.
        Wt = np.empty_like(W); mt = np.empty_like(m); vt = np.empty_like(v)
        tokens = _random_partition(bt, rs)
        for (r0, r1) in _random_partition(d_out, rs):
            for (c0, c1) in _random_partition(d_in, rs):
                Gt = np.zeros((r1 - r0, c1 - c0))
                for (k0, k1) in tokens:
                    for tt in range(k0, k1):
                        for p in range(r0, r1):
                            for q in range(c0, c1):
                                Gt[p - r0, q - c0] += dY[tt, p] * X[tt, q]
                sub = O.State(W=W[r0:r1, c0:c1], m=m[r0:r1, c0:c1],
                              v=v[r0:r1, c0:c1] if opt == "adamw" else None)
                out = O.step(opt, None, None, sub, h, t, mode=mode, G=Gt)
                Wt[r0:r1, c0:c1] = out.W
                mt[r0:r1, c0:c1] = out.m
                if opt == "adamw":
                    vt[r0:r1, c0:c1] = out.v
        assert np.array_equal(Wt.view(np.uint32), whole.W.view(np.uint32))
        assert np.array_equal(mt.view(np.uint32), whole.m.view(np.uint32))
        if opt == "adamw":
            assert np.array_equal(vt.view(np.uint32), whole.v.view(np.uint32))


# ---------------------------------------------------------------------------
# lr = 0 leaves W unchanged (Algorithm 1's weight update with eta = 0)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("opt", ["adamw", "sgdm", "lion"])
@pytest.mark.parametrize("mode", ["f64", "f32emu"])
def test_lr_zero_keeps_w(opt, mode):
    rs = np.random.RandomState(3)
    dY = rs.randn(9, 6); X = rs.randn(9, 5)
    W = (rs.randn(6, 5) * 0.02).astype(np.float32)
    m = (rs.randn(6, 5) * 1e-3).astype(np.float32)
    v = np.abs(rs.randn(6, 5) * 1e-6).astype(np.float32)
    h = O.Hyper(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.5)
    out = O.step(opt, X, dY, O.State(W=W, m=m, v=v), h, 2, mode=mode)
    assert np.array_equal(out.W.view(np.uint32), W.view(np.uint32))
    # The moments still move.
    assert not np.array_equal(out.m, m)


# ---------------------------------------------------------------------------
# Hand-computed 2x2 examples (tests/golden/*_hand.json)
# ---------------------------------------------------------------------------

def test_adamw_hand_2x2():
    g = _load("adamw_2x2_hand.json")
    h = _hyper(g["hyper"])
    W1, m1, v1 = O.adamw_f64(g["W"], g["m"], g["v"], g["G"], h, g["t"])
    np.testing.assert_allclose(W1, g["W_new"], rtol=1e-15, atol=1e-18)
    np.testing.assert_allclose(m1, g["m_new"], rtol=1e-15, atol=1e-18)
    np.testing.assert_allclose(v1, g["v_new"], rtol=1e-14, atol=1e-18)


def test_sgdm_hand_2x2():
    g = _load("sgdm_2x2_hand.json")
    W1, m1 = O.sgdm_f64(g["W"], g["m"], g["G"], _hyper(g["hyper"]), g["t"])
    np.testing.assert_allclose(W1, g["W_new"], rtol=1e-14, atol=1e-18)
    np.testing.assert_allclose(m1, g["m_new"], rtol=1e-14, atol=1e-18)


def test_lion_hand_2x2():
    g = _load("lion_2x2_hand.json")
    W1, m1 = O.lion_f64(g["W"], g["m"], g["G"], _hyper(g["hyper"]), g["t"])
    np.testing.assert_allclose(W1, g["W_new"], rtol=1e-14, atol=1e-18)
    np.testing.assert_allclose(m1, g["m_new"], rtol=1e-14, atol=1e-18)


def test_hand_examples_in_f32emu_mode_within_ulps():
    g = _load("adamw_2x2_hand.json")
    h = _hyper(g["hyper"])
    s = O.fold_scalars("adamw", h, 1)
    f = lambda a: np.asarray(a, np.float32)
    W1, m1, v1 = O.adamw_f32(f(g["W"]), f(g["m"]), f(g["v"]), f(g["G"]), s)
    np.testing.assert_allclose(W1, g["W_new"], rtol=4e-7, atol=1e-12)
    np.testing.assert_allclose(m1, g["m_new"], rtol=2e-7)
    np.testing.assert_allclose(v1, g["v_new"], rtol=2e-7)


# ---------------------------------------------------------------------------
# Closed forms over several steps with a constant gradient
# ---------------------------------------------------------------------------

def test_adamw_constant_gradient_closed_form():
    # With g constant from m = v = 0, m_hat_t = g and v_hat_t = g^2 exactly
    # (geometric series), so each step moves W by -lr g / (|g| + eps).
    rs = np.random.RandomState(5)
    G = rs.randn(4, 7) * 3
    W = rs.randn(4, 7) * 0.02
    m = np.zeros_like(W); v = np.zeros_like(W)
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    Wk = W.copy()
    for t in range(1, 11):
        Wk, m, v = O.adamw_f64(Wk, m, v, G, h, t)
        expect = W - t * 1e-3 * G / (np.abs(G) + 1e-8)
        np.testing.assert_allclose(Wk, expect, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(m / (1 - 0.9 ** t), G, rtol=1e-12)
        np.testing.assert_allclose(v / (1 - 0.999 ** t), G * G, rtol=1e-10)


def test_sgdm_constant_gradient_closed_form():
    rs = np.random.RandomState(6)
    G = rs.randn(3, 5); W = rs.randn(3, 5)
    m = np.zeros_like(W)
    mu, lr = 0.9, 1e-2
    h = O.Hyper(lr=lr, beta1=mu, weight_decay=0.0)
    Wk = W.copy(); acc = np.zeros_like(W)
    for t in range(1, 9):
        Wk, m = O.sgdm_f64(Wk, m, G, h, t)
        mt = G * (1 - mu ** t) / (1 - mu)
        acc += mt
        np.testing.assert_allclose(m, mt, rtol=1e-12)
        np.testing.assert_allclose(Wk, W - lr * acc, rtol=1e-12, atol=1e-15)


def test_lion_step_is_lr_sized():
    rs = np.random.RandomState(8)
    G = rs.randn(6, 6); W = rs.randn(6, 6); m = rs.randn(6, 6) * 0.1
    G[0, 0] = 0.0; m[0, 0] = 0.0   # c = 0 -> sign 0 -> decay only
    h = O.Hyper(lr=3e-4, beta1=0.9, beta2=0.99, weight_decay=0.2)
    W1, _ = O.lion_f64(W, m, G, h, 1)
    d = np.abs(W1 - (1 - 3e-4 * 0.2) * W)
    assert d[0, 0] == 0.0
    mask = np.ones_like(d, bool); mask[0, 0] = False
    np.testing.assert_allclose(d[mask], 3e-4, rtol=1e-9)


# ---------------------------------------------------------------------------
# float32 emulation against float64 (random inputs)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("opt", ["adamw", "sgdm", "lion"])
def test_f32emu_close_to_f64(opt):
    rs = np.random.RandomState(11)
    dY = rs.randn(64, 32).astype(np.float32); X = rs.randn(64, 48).astype(np.float32)
    W = (rs.randn(32, 48) * 0.02).astype(np.float32)
    m = (rs.randn(32, 48) * 1e-3).astype(np.float32)
    v = np.abs(rs.randn(32, 48) * 1e-6).astype(np.float32)
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.99 if opt == "lion" else 0.999, eps=1e-8,
                weight_decay=0.01)
    st = O.State(W=W, m=m, v=v)
    a = O.step(opt, X, dY, st, h, 4, mode="f64")
    b = O.step(opt, X, dY, st, h, 4, mode="f32emu")
    W1, m1, v1, G = O.step_values(opt, X, dY, st, h, 4)
    # m' and v' carry a few float32 roundings of their terms.
    np.testing.assert_allclose(b.m, m1, rtol=0, atol=4 * 2 ** -24 * (np.abs(m) + np.abs(G)).max())
    # W': decay*W and lr*u are each a few ulps; Lion's sign(c) may only
    # differ where c is within rounding of 0 (none at these sizes).
    np.testing.assert_allclose(b.W, a.W, rtol=0, atol=8 * 2 ** -24 * np.abs(W).max() + 1e-10)


# ---------------------------------------------------------------------------
# bf16 rounding against independent routines
# ---------------------------------------------------------------------------

def test_bf16_rne_matches_torch_cast():
    rs = np.random.RandomState(2)
    x = np.concatenate([rs.randn(20000).astype(np.float32) * 10.0 ** rs.randint(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.4e38, -3.4e38],
                                 np.float32)]).astype(np.float32)
    # exact ties: low 16 bits 0x8000
    ties = (rs.randint(0, 2 ** 31, 2000).astype(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32)])
    x = x[np.isfinite(x) | np.isinf(x)]
    ours = O.f32_to_bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    finite = ~np.isnan(x)
    assert np.array_equal(ours[finite], ref[finite])


def test_bf16_rne_from_f64_brute_force():
    # All finite positive bf16 values, sorted; nearest-by-exact-distance.
    allb = np.arange(0, 0x7F80, dtype=np.uint32)
    vals = (allb << np.uint32(16)).view(np.float32).astype(np.float64)
    rs = np.random.RandomState(4)
    x = rs.randn(20000) * 10.0 ** rs.uniform(-20, 20, 20000)
    # exact midpoints between neighbours
    k = rs.randint(1, 0x7F7F, 500)
    mids = (vals[k] + vals[k + 1]) / 2
    x = np.concatenate([x, mids, -mids])
    ours = O.f64_to_bf16_rne(x)
    ax = np.abs(x)
    hi = np.searchsorted(vals, ax, side="left")
    lo = np.maximum(hi - 1, 0)
    hi = np.minimum(hi, vals.size - 1)
    exact = vals[hi] == ax
    d_lo = ax - vals[lo]; d_hi = vals[hi] - ax
    pick = np.where(exact, hi, np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi,
                    np.where(lo % 2 == 0, lo, hi))))
    ref = allb[pick] | np.where(x < 0, 0x8000, 0).astype(np.uint32)
    assert np.array_equal(ours.astype(np.uint32), ref)


# ---------------------------------------------------------------------------
# Stochastic rounding (Appendix C, Proposition 5)
# ---------------------------------------------------------------------------

def test_sr_exact_expectation_over_all_draws():
    # Averaging the SR result over every r16 in [0, 2^16) gives x exactly.
    rs = np.random.RandomState(9)
    xs = np.concatenate([rs.randn(40).astype(np.float32),
                         np.array([1e-30, -7.5, 0.75 - 2 ** -10], np.float32)])
    r = np.arange(65536, dtype=np.uint32)
    for x in xs:
        b = O.f32_to_bf16_sr(np.full(65536, x, np.float32), r)
        vals = O.bf16_bits_to_f32(b).astype(np.float64)
        assert vals.mean() == pytest.approx(float(x), rel=0, abs=abs(float(x)) * 2 ** -40)
        # and only the two bf16 neighbours occur
        assert np.unique(b).size <= 2


def test_sr_worked_example_quarter_ulp():
    # 100 updates of -1e-3 on a weight in [0.5, 1) (bf16 ulp 2^-8, so each
    # update is about a quarter ulp): round-to-nearest never moves, while
    # stochastic rounding moves -0.100 in expectation (Appendix C).
    trials, steps = 400, 100
    w_rne = np.full(trials, 0.75, np.float32)
    w_sr = np.full(trials, 0.75, np.float32)
    for t in range(1, steps + 1):
        w_rne = O.bf16_bits_to_f32(O.f32_to_bf16_rne(w_rne - np.float32(1e-3)))
        r16 = O.sr_draws(1234, t, O.SITE_W, 1, trials)[0]
        w_sr = O.bf16_bits_to_f32(O.f32_to_bf16_sr(w_sr - np.float32(1e-3), r16))
    assert np.all(w_rne == np.float32(0.75))
    mean = float(np.mean(w_sr.astype(np.float64) - 0.75))
    # std of one trial's total is below sqrt(100) * ulp / 2
    se = 10 * 2 ** -8 / 2 / np.sqrt(trials)
    assert abs(mean - (-0.1)) < 5 * se, mean


def test_sr_round_up_fraction_binomial():
    # P(round up) equals the discarded fraction f, checked with Philox draws.
    n = 200000
    x = np.float32(1.0 + 0.3 * 2 ** -7)     # f = 0.3 of a bf16 ulp above 1
    r16 = O.sr_draws(77, 5, O.SITE_W, 1, n)[0]
    b = O.f32_to_bf16_sr(np.full(n, x, np.float32), r16)
    up = np.mean(b == 0x3F81)
    f = (int(np.float32(x).view(np.uint32)) & 0xFFFF) / 65536.0
    assert abs(up - f) < 5 * np.sqrt(f * (1 - f) / n)


# ---------------------------------------------------------------------------
# Philox4x32-10 against an independent implementation (Triton's CPU
# interpreter), and the stream mapping of the draws
# ---------------------------------------------------------------------------

_TRITON_PHILOX = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def kern(c_ptr, out_ptr, seed, n: tl.constexpr):
    i = tl.arange(0, n)
    c0 = tl.load(c_ptr + 4 * i + 0).to(tl.uint32)
    c1 = tl.load(c_ptr + 4 * i + 1).to(tl.uint32)
    c2 = tl.load(c_ptr + 4 * i + 2).to(tl.uint32)
    c3 = tl.load(c_ptr + 4 * i + 3).to(tl.uint32)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3, n_rounds=10)
    tl.store(out_ptr + 4 * i + 0, a.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + 4 * i + 1, b.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + 4 * i + 2, c.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + 4 * i + 3, d.to(tl.int64) & 0xFFFFFFFF)

cfg = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cfg:
    c = torch.tensor(ctrs, dtype=torch.int64)
    o = torch.zeros_like(c)
    kern[(1,)](c, o, seed, c.shape[0])
    res.append(o.tolist())
print(json.dumps(res))
"""


def test_philox_matches_independent_implementation():
    pytest.importorskip("triton")
    rs = np.random.RandomState(12)
    cases = []
    for seed in [0, 1234, 0xFFFFFFFF, 0x123456789ABCDEF]:
        ctrs = rs.randint(0, 2 ** 32, size=(16, 4), dtype=np.uint64)
        ctrs[0] = 0
        ctrs[1] = 0xFFFFFFFF
        cases.append((int(seed), ctrs.astype(np.int64).tolist()))
    proc = subprocess.run([sys.executable, "-c", _TRITON_PHILOX], input=json.dumps(cases),
                          capture_output=True, text=True, timeout=600)
    if proc.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + proc.stderr[-300:])
    ref = json.loads(proc.stdout.strip().splitlines()[-1])
    for (seed, ctrs), r in zip(cases, ref):
        ours = O.philox4x32_10(np.array(ctrs, dtype=np.uint64), (seed & 0xFFFFFFFF, seed >> 32))
        assert np.array_equal(ours.astype(np.int64), np.array(r, dtype=np.int64)), seed


def test_sr_draw_stream_mapping():
    # Element idx takes half (idx % 2) of word (idx % 8) / 2 of the Philox
    # block idx / 8, counter (idx/8 lo, idx/8 hi, step, site), key = seed.
    seed, t, site, rows, cols = 0xABCDEF0123, 7, O.SITE_M, 3, 24
    r = O.sr_draws(seed, t, site, rows, cols)
    for p in range(rows):
        for q in range(cols):
            idx = p * cols + q
            ctr = np.array([[idx // 8, 0, t, site]], np.uint64)
            w = O.philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))[0]
            word = int(w[(idx % 8) // 2])
            assert r[p, q] == ((word >> (16 * (idx % 2))) & 0xFFFF)
    # sub-block draws agree with the whole-tensor draws
    sub = O.sr_draws(seed, t, site, 2, 5, row0=1, col0=9, total_cols=cols)
    assert np.array_equal(sub, r[1:3, 9:14])
    # different step / site / seed give different streams
    # a sample of whole rows draws what those rows of the whole tensor draw
    assert np.array_equal(O.row_draws(seed, t, site, (2, cols), rows=[0, 2]), r[[0, 2]])
    assert not np.array_equal(r, O.sr_draws(seed, t + 1, site, rows, cols))
    assert not np.array_equal(r, O.sr_draws(seed, t, site + 1, rows, cols))
    assert not np.array_equal(r, O.sr_draws(seed + 1, t, site, rows, cols))


# ---------------------------------------------------------------------------
# 8-bit block moments (Section 2.3, Appendix B, Proposition 4)
# ---------------------------------------------------------------------------

def test_q8_roundtrip_bounds_and_zero_codes():
    rs = np.random.RandomState(13)
    m = (rs.randn(8, 256) * 1e-3).astype(np.float32)
    m[0, :5] = 0.0
    m[1, :] = 0.0                      # an all-zero block row
    m[2, 7] = 1e-9                     # tiny nonzero: must not get code 0
    codes, s = O.quant_m(m)
    back = O.dequant_m(codes, s)
    srow = np.repeat(s.T, 128, axis=1)
    err = np.abs(back.astype(np.float64) - m)
    bumped = (codes != 0) & (np.abs(m) < srow / 2)
    assert np.all(err[~bumped] <= srow[~bumped] / 2 * (1 + 1e-6))
    assert np.all(err[bumped] <= srow[bumped] * (1 + 1e-6))
    assert np.all(codes[m == 0] == 0) and np.all(codes[m != 0] != 0)
    assert np.all(np.abs(codes.astype(int)) <= 127)
    assert np.all(s[:, 1] == 0)
    # the block absmax element gets code +-127
    for r in range(8):
        for b in range(2):
            blk = m[r, b * 128:(b + 1) * 128]
            if np.any(blk != 0):
                assert np.max(np.abs(codes[r, b * 128:(b + 1) * 128].astype(int))) == 127

    v = (np.abs(rs.randn(8, 256)) * 1e-6).astype(np.float32)
    v[0, :3] = 0.0
    v[3, 100] = 1e-30                  # tiny nonzero v: floored away from zero
    vc, vs = O.quant_v(v)
    assert np.all(vc[v == 0] == 0) and np.all(vc[v != 0] >= 1)
    u = np.sqrt(v.astype(np.float64))
    ub = np.sqrt(O.dequant_v(vc, vs).astype(np.float64))
    srow = np.repeat(vs.T, 128, axis=1)
    nz = v != 0
    floor = nz & (u < srow / 2)
    assert np.all(np.abs(ub - u)[nz & ~floor] <= srow[nz & ~floor] / 2 * (1 + 1e-5))
    assert np.all(np.abs(ub - u)[floor] <= srow[floor] * (1 + 1e-5))


def _exact_round_half_even(x, s):
    """round(x / s), ties to even, in exact rational arithmetic."""
    from fractions import Fraction
    return round(Fraction(float(x)) / Fraction(float(s)))


def _near_tie_pairs(rs, n, kmax):
    """(x, s) float32 pairs whose quotient lies on or within a few float32
    steps of a half-integer k + 1/2, |k| < kmax, plus exact ties."""
    xs, ss = [], []
    for _ in range(n):
        s = np.float32(rs.uniform(0.5, 1.0) * 2.0 ** rs.randint(-40, 10))
        k = rs.randint(-kmax, kmax)
        x0 = np.float32((k + 0.5) * float(s))
        x = x0
        for d in range(-3, 4):
            xs.append(x); ss.append(s)
            x = np.nextafter(x, np.float32(np.inf)) if d >= 0 else x
        xd = x0
        for _ in range(3):
            xd = np.nextafter(xd, np.float32(-np.inf))
            xs.append(xd); ss.append(s)
    # exact ties: s = 2^e * (odd / 2^j) with few bits, so (k + 1/2) s is a float32
    for k in range(-kmax, kmax):
        for e in (-30, -3, 0, 7):
            s = np.float32(2.0 ** e * 3.0)
            xs.append(np.float32((k + 0.5) * float(s))); ss.append(s)
    return np.array(xs, np.float32), np.array(ss, np.float32)


def test_q8_round_quotient_is_exact_on_near_ties():
    # q(x) = s * round(x / s) (Section 2.3; Appendix B, Proposition 4): the
    # oracle's rounding of x / s against exact rational arithmetic, on
    # quotients on and next to half-integers and on random pairs.
    rs = np.random.RandomState(41)
    x, s = _near_tie_pairs(rs, 400, 256)
    xr = (rs.randn(3000) * 1e-3).astype(np.float32)
    sr = (np.abs(rs.randn(3000)) * 1e-5 + 1e-7).astype(np.float32)
    keep = np.abs(xr.astype(np.float64) / sr) < 500
    x = np.concatenate([x, xr[keep]]); s = np.concatenate([s, sr[keep]])
    got = O.round_quotient(x, s)
    want = np.array([_exact_round_half_even(a, b) for a, b in zip(x, s)], np.float64)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]
    # the set really holds exact ties and near misses on both sides
    exact_tie = np.array([(2 * float(a)) / float(b) % 2 == 1 for a, b in zip(x, s)])
    assert exact_tie.sum() > 100


def _codes_by_rationals(x, which):
    """The paper's block quantiser written out element by element with exact
    rationals: scale s = fl32(absmax / 127) (m) or fl32(absmax(sqrt v) / 255)
    (v), code = clamp(round(x / s)), ties to even, reserved zero code."""
    rows, cols = x.shape
    codes = np.zeros((rows, cols), np.int64)
    for r in range(rows):
        for b in range(cols // 128):
            blk = x[r, b * 128:(b + 1) * 128]
            if which == "m":
                s = np.float32(np.float32(np.max(np.abs(blk))) / np.float32(127.0))
                for j, e in enumerate(blk):
                    if s == 0:
                        c = 0
                    else:
                        c = max(-127, min(127, _exact_round_half_even(e, s)))
                        if c == 0 and e != 0:
                            c = 1 if e > 0 else -1
                    codes[r, b * 128 + j] = c
            else:
                u = np.sqrt(blk.astype(np.float32))
                s = np.float32(np.float32(np.max(u)) / np.float32(255.0))
                for j, (e, ue) in enumerate(zip(blk, u)):
                    c = 0 if (s == 0 or e == 0) else max(1, min(255, _exact_round_half_even(ue, s)))
                    codes[r, b * 128 + j] = c
    return codes


def _planted_tie_block(rs, rows, which):
    """Rows of 128-element blocks whose values sit on and next to code
    boundaries of their own block scale (the largest element fixes s)."""
    out = np.zeros((rows, 256), np.float32)
    for r in range(rows):
        for b in range(2):
            top = np.float32(rs.uniform(0.5, 1.0) * 1e-3)
            lim = 127 if which == "m" else 255
            s = np.float32(top / np.float32(lim)) if which == "m" else np.float32(np.sqrt(top) / np.float32(lim))
            vals = [top if which == "m" else top]
            while len(vals) < 128:
                k = rs.randint(-126 if which == "m" else 0, lim - 1)
                t = np.float32((k + 0.5) * float(s))
                for _ in range(rs.randint(0, 3)):
                    t = np.nextafter(t, np.float32(np.inf if rs.rand() < 0.5 else -np.inf))
                vals.append(t if which == "m" else np.float32(t) * np.float32(t))
            blk = np.array(vals[:128], np.float32)
            if which == "v":
                blk = np.abs(blk)
                blk[rs.randint(1, 128)] = 0.0
            out[r, b * 128:(b + 1) * 128] = rs.permutation(blk)
    return out


def test_q8_codes_equal_the_exact_rule_elementwise():
    rs = np.random.RandomState(42)
    m = _planted_tie_block(rs, 6, "m")
    m[0, :3] = 0.0
    m[1, 128:] = 0.0
    codes, s = O.quant_m(m)
    assert np.array_equal(codes.astype(np.int64), _codes_by_rationals(m, "m"))
    v = _planted_tie_block(rs, 6, "v")
    vc, vs = O.quant_v(v)
    assert np.array_equal(vc.astype(np.int64), _codes_by_rationals(v, "v"))


def test_planted_reciprocal_quantiser_is_caught(monkeypatch):
    # x * fl(1/s) rounded in float32 (a cheaper sequence) moves codes next to
    # half-integers: the exact-rule pins must fail with it.
    def recip(x, s):
        x = np.asarray(x, np.float32); s = np.asarray(s, np.float32)
        return np.rint((x * (np.float32(1.0) / s)).astype(np.float32)).astype(np.float64)
    monkeypatch.setattr(O, "round_quotient", recip)
    with pytest.raises(AssertionError):
        test_q8_round_quotient_is_exact_on_near_ties()
    with pytest.raises(AssertionError):
        test_q8_codes_equal_the_exact_rule_elementwise()


def test_planted_half_away_rounding_is_caught(monkeypatch):
    def away(x, s):
        q = np.asarray(x, np.float32).astype(np.float64) / np.asarray(s, np.float32).astype(np.float64)
        return np.sign(q) * np.floor(np.abs(q) + 0.5)
    monkeypatch.setattr(O, "round_quotient", away)
    with pytest.raises(AssertionError):
        test_q8_round_quotient_is_exact_on_near_ties()


def test_q8_first_moment_drift_bound_prop4():
    # The stored 8-bit first moment stays within sum_k beta^(t-k) * e_k of the
    # fp32-state moment, with |e_k| <= s_k (s_k / 2 for round-to-nearest,
    # s_k for the reserved-zero bump): a damped, bounded drift.
    rs = np.random.RandomState(14)
    d_out, d_in, bt, steps = 16, 256, 32, 40
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    W = (rs.randn(d_out, d_in) * 0.02).astype(np.float32)
    st8 = O.State(W=W.copy(), m=np.zeros((d_out, d_in), np.int8),
                  v=np.zeros((d_out, d_in), np.uint8),
                  m_scale=np.zeros((d_in // 128, d_out), np.float32),
                  v_scale=np.zeros((d_in // 128, d_out), np.float32), state="q8")
    st32 = O.State(W=W.copy(), m=np.zeros((d_out, d_in), np.float32),
                   v=np.zeros((d_out, d_in), np.float32))
    bound = np.zeros((d_out, d_in))
    for t in range(1, steps + 1):
        dY = rs.randn(bt, d_out).astype(np.float32); X = rs.randn(bt, d_in).astype(np.float32)
        G = O.wgrad_f64(dY, X)
        st8 = O.step("adamw", None, None, st8, h, t, mode="f32emu", G=G)
        st32 = O.step("adamw", None, None, st32, h, t, mode="f32emu", G=G)
        s = np.repeat(st8.m_scale.T, 128, axis=1).astype(np.float64)
        bound = 0.9 * bound + s
        drift = np.abs(O.dequant_m(st8.m, st8.m_scale).astype(np.float64) - st32.m)
        assert np.all(drift <= bound * (1 + 1e-4) + 1e-12)
    # and the typical drift is about a quantisation step or less
    assert np.sqrt(np.mean(drift ** 2)) < np.mean(s)


def test_q8_zero_rows_keep_zero_state_and_decay_only():
    rs = np.random.RandomState(15)
    d_out, d_in = 6, 128
    W = (rs.randn(d_out, d_in) * 0.02).astype(np.float32)
    st = O.State(W=W, m=np.zeros((d_out, d_in), np.int8), v=np.zeros((d_out, d_in), np.uint8),
                 m_scale=np.zeros((1, d_out), np.float32), v_scale=np.zeros((1, d_out), np.float32),
                 state="q8")
    dY = rs.randn(4, d_out).astype(np.float32); dY[:, 2] = 0.0
    X = rs.randn(4, d_in).astype(np.float32)
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    for mode in ("f64", "f32emu"):
        out = O.step("adamw", X, dY, st, h, 1, mode=mode)
        assert np.all(out.m[2] == 0) and np.all(out.v[2] == 0)
        assert out.m_scale[0, 2] == 0 and out.v_scale[0, 2] == 0
        if mode == "f32emu":   # float32 scalar, one float32 product
            expect = (np.float32(1.0 - 1e-3 * 0.01) * W[2]).astype(np.float32)
        else:                  # exact product, rounded once
            expect = ((1.0 - 1e-3 * 0.01) * W[2].astype(np.float64)).astype(np.float32)
        assert np.array_equal(out.W[2], expect)


# ---------------------------------------------------------------------------
# The input gradient (Appendix A, Remark 1): dX = dY W_old
# ---------------------------------------------------------------------------

def test_dgrad_brute_force_triple_loop():
    rs = np.random.RandomState(51)
    for (bt, d_out, d_in) in [(1, 1, 1), (2, 3, 5), (4, 2, 3), (6, 5, 7)]:
        dY = rs.randn(bt, d_out)
        W = rs.randn(d_out, d_in)
        dX = O.dgrad_f64(dY, W)
        assert dX.shape == (bt, d_in)
        for t in range(bt):
            for q in range(d_in):
                acc = 0.0
                for p in range(d_out):
                    acc += dY[t, p] * W[p, q]
                assert abs(dX[t, q] - acc) <= 1e-12 * (1 + abs(acc))


def test_dgrad_hand_2x2():
    # dY = [[1, 2], [3, 4]], W = [[5, 6], [7, 8]]: dX = dY W = [[19, 22], [43, 50]]
    # (dY W^T would be [[17, 23], [39, 53]]).
    dX = O.dgrad_f64(np.array([[1.0, 2.0], [3.0, 4.0]]), np.array([[5.0, 6.0], [7.0, 8.0]]))
    assert np.array_equal(dX, np.array([[19.0, 22.0], [43.0, 50.0]]))


def test_planted_transposed_weight_in_dgrad_is_caught(monkeypatch):
    monkeypatch.setattr(O, "dgrad_f64", lambda dY, W: np.asarray(dY, float) @ np.asarray(W, float).T)
    with pytest.raises(AssertionError):
        test_dgrad_hand_2x2()


@pytest.mark.parametrize("opt", ["adamw", "sgdm", "lion"])
def test_backward_reads_the_weights_before_the_step(opt):
    # Remark 1: dX comes from W_old. With lr != 0 the step moves W, so dY W_old
    # and dY W_new differ; the oracle's backward pass must give the former.
    rs = np.random.RandomState(52)
    d_out, d_in, bt = 6, 5, 4
    X = rs.randint(-3, 4, size=(bt, d_in)).astype(np.float32)
    dY = rs.randint(-3, 4, size=(bt, d_out)).astype(np.float32)
    W = rs.randint(-3, 4, size=(d_out, d_in)).astype(np.float32) * np.float32(0.25)
    st = O.State(W=W.copy(), m=np.zeros((d_out, d_in), np.float32),
                 v=np.zeros((d_out, d_in), np.float32) if opt == "adamw" else None)
    h = O.Hyper(lr=0.5, beta1=0.9, beta2=0.99, eps=1e-8, weight_decay=0.1)
    dX, new = O.backward_step(opt, X, dY, st, h, 1)
    old = np.zeros((bt, d_in))
    for t in range(bt):
        for q in range(d_in):
            old[t, q] = sum(float(dY[t, p]) * float(W[p, q]) for p in range(d_out))
    assert np.array_equal(dX, old)
    assert not np.array_equal(dX, dY.astype(np.float64) @ new.W.astype(np.float64))
    # and the state is the plain step
    ref = O.step(opt, X, dY, st, h, 1)
    assert np.array_equal(new.W, ref.W)


# ---------------------------------------------------------------------------
# Planted mistakes: each plausible slip in the oracle fails a pin above.
# ---------------------------------------------------------------------------

def _pins_pass():
    try:
        test_adamw_hand_2x2()
        test_adamw_constant_gradient_closed_form()
        test_wgrad_brute_force_triple_loop()
        return True
    except AssertionError:
        return False


MUTANTS = {
    "no_bias_correction": lambda W, m, v, G, h, t: _adamw_mut(W, m, v, G, h, t, bc=False),
    "eps_inside_sqrt": lambda W, m, v, G, h, t: _adamw_mut(W, m, v, G, h, t, eps_in=True),
    "decay_after_update": lambda W, m, v, G, h, t: _adamw_mut(W, m, v, G, h, t, late_decay=True),
    "wrong_beta": lambda W, m, v, G, h, t: _adamw_mut(W, m, v, G, h, t, swap_beta=True),
}


def _adamw_mut(W, m, v, G, h, t, bc=True, eps_in=False, late_decay=False, swap_beta=False):
    W = np.asarray(W, float); m = np.asarray(m, float); v = np.asarray(v, float); G = np.asarray(G, float)
    b1, b2 = (h.beta2, h.beta1) if swap_beta else (h.beta1, h.beta2)
    m1 = b1 * m + (1 - b1) * G
    v1 = b2 * v + (1 - b2) * G * G
    mh = m1 / (1 - b1 ** t) if bc else m1
    vh = v1 / (1 - b2 ** t) if bc else v1
    den = np.sqrt(vh + h.eps) if eps_in else np.sqrt(vh) + h.eps
    if late_decay:
        W1 = (1 - h.lr * h.weight_decay) * (W - h.lr * mh / den)
    else:
        W1 = (1 - h.lr * h.weight_decay) * W - h.lr * mh / den
    return W1, m1, v1


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    assert _pins_pass()
    monkeypatch.setattr(O, "adamw_f64", MUTANTS[name])
    assert not _pins_pass(), name


def test_planted_transposed_gradient_is_caught(monkeypatch):
    monkeypatch.setattr(O, "wgrad_f64", lambda dY, X: np.asarray(X, float).T @ np.asarray(dY, float))
    with pytest.raises(AssertionError):
        test_wgrad_brute_force_triple_loop()


# ---------------------------------------------------------------------------
# The element-wise families against PyTorch's optimizers of the same name
# (float64, CPU): an independent library implementation of each rule.
# ---------------------------------------------------------------------------

def _torch_opt(name, p, h):
    kw = dict(lr=h.lr, weight_decay=h.weight_decay, foreach=False)
    if name == "adamw":
        return torch.optim.AdamW([p], betas=(h.beta1, h.beta2), eps=h.eps, **kw)
    if name == "sgdm":
        return torch.optim.SGD([p], momentum=h.beta1, **kw)
    if name == "sgd":
        return torch.optim.SGD([p], momentum=0.0, **kw)
    if name == "rmsprop":
        return torch.optim.RMSprop([p], alpha=h.beta2, eps=h.eps, **kw)
    if name == "adagrad":
        return torch.optim.Adagrad([p], eps=h.eps, **kw)
    if name == "nadam":
        return torch.optim.NAdam([p], betas=(h.beta1, h.beta2), eps=h.eps, momentum_decay=h.momentum_decay, **kw)
    if name == "radam":
        return torch.optim.RAdam([p], betas=(h.beta1, h.beta2), eps=h.eps, **kw)
    raise ValueError(name)


_TORCH_STATE = {"adamw": ("exp_avg", "exp_avg_sq"), "nadam": ("exp_avg", "exp_avg_sq"),
                "radam": ("exp_avg", "exp_avg_sq"), "sgdm": ("momentum_buffer",),
                "rmsprop": ("square_avg",), "adagrad": ("sum",), "sgd": ()}


@pytest.mark.parametrize("name", ["adamw", "sgdm", "sgd", "rmsprop", "adagrad", "nadam", "radam"])
def test_rules_match_torch_optim_float64(name):
    prev = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    try:
        rs = np.random.RandomState(21)
        W0 = rs.randn(5, 7) * 0.02
        h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.99 if name == "rmsprop" else 0.999, eps=1e-8,
                    weight_decay=0.01, momentum_decay=4e-3)
        p = torch.nn.Parameter(torch.tensor(W0))
        topt = _torch_opt(name, p, h)
        W = W0.copy()
        s0 = np.zeros_like(W0)
        s1 = np.zeros_like(W0)
        for t in range(1, 13):
            G = rs.randn(5, 7) * 3.0
            p.grad = torch.tensor(G)
            topt.step()
            if name == "adamw":
                W, s0, s1 = O.adamw_f64(W, s0, s1, G, h, t)
            elif name == "sgdm":
                W, s0 = O.sgdm_f64(W, s0, G, h, t)
            elif name == "sgd":
                W = O.sgd_f64(W, G, h, t)
            elif name == "rmsprop":
                W, s0 = O.rmsprop_f64(W, s0, G, h, t)
            elif name == "adagrad":
                W, s0 = O.adagrad_f64(W, s0, G, h, t)
            elif name == "nadam":
                W, s0, s1 = O.nadam_f64(W, s0, s1, G, h, t)
            else:
                W, s0, s1 = O.radam_f64(W, s0, s1, G, h, t)
            np.testing.assert_allclose(W, p.detach().numpy(), rtol=1e-12, atol=1e-15, err_msg=f"{name} W, t={t}")
            st = topt.state[p]
            for key, ours in zip(_TORCH_STATE[name], (s0, s1)):
                np.testing.assert_allclose(ours, st[key].numpy(), rtol=1e-12, atol=1e-18,
                                           err_msg=f"{name} {key}, t={t}")
    finally:
        torch.set_default_dtype(prev)


def test_radam_crosses_its_rectification_threshold():
    # With beta2 = 0.999 the rectification applies from step 6 on (rho_t > 5).
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999)
    flags = [O.radam_rect(h, t)[0] for t in range(1, 9)]
    assert flags == [False] * 5 + [True] * 3


def test_nadam_first_step_closed_form():
    # From zero state at t = 1 with constant g: m' = (1-b1) g, v' = (1-b2) g^2,
    # so W' = W - lr g / (|g| + eps) * (1 + mu_2 (1 - b1) / (1 - mu_1 mu_2)).
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, momentum_decay=4e-3)
    mu1 = 0.9 * (1 - 0.5 * 0.96 ** 0.004)
    mu2 = 0.9 * (1 - 0.5 * 0.96 ** 0.008)
    G = np.array([[2.0, -0.5]]); W = np.array([[0.1, 0.2]])
    W1, _, _ = O.nadam_f64(W, np.zeros_like(W), np.zeros_like(W), G, h, 1)
    factor = 1 + mu2 * 0.1 / (1 - mu1 * mu2)
    np.testing.assert_allclose(W1, W - 1e-3 * G / (np.abs(G) + 1e-8) * factor, rtol=1e-13)
    assert abs(factor - 1.0564522) < 1e-6


def test_accumulated_gradient_equals_the_concatenated_batch():
    # Appendix L: summing the micro-batch gradients is the gradient of the
    # whole effective batch, since G = dY^T X is a sum over tokens.
    rng = np.random.default_rng(7)
    sizes = [5, 1, 12, 7]
    mbs = [(rng.standard_normal((n, 6)), rng.standard_normal((n, 4))) for n in sizes]
    G = O.accumulated_gradient_f64(mbs)
    Xc = np.concatenate([x for x, _ in mbs]); dYc = np.concatenate([d for _, d in mbs])
    np.testing.assert_allclose(G, dYc.T @ Xc, rtol=1e-13, atol=1e-13)
    # brute force on one entry, and a single micro-batch is the plain gradient
    assert abs(G[2, 3] - sum(float(d[t, 2] * x[t, 3]) for x, d in mbs for t in range(len(x)))) < 1e-12
    np.testing.assert_array_equal(O.accumulated_gradient_f64(mbs[:1]), O.wgrad_f64(mbs[0][1], mbs[0][0]))


def test_accumulated_step_is_the_large_batch_step():
    # "Numerically identical to vanilla AdamW at the same effective batch":
    # the step fired once on the accumulated gradient equals the step on the
    # concatenated batch (exact here: integer inputs, float64 sums).
    rng = np.random.default_rng(8)
    mbs = [(rng.integers(-3, 4, (n, 8)).astype(np.float64), rng.integers(-3, 4, (n, 6)).astype(np.float64))
           for n in (3, 9, 4)]
    Xc = np.concatenate([x for x, _ in mbs]); dYc = np.concatenate([d for _, d in mbs])
    W = rng.standard_normal((6, 8)) * 0.02
    st = O.State(W=W.astype(np.float32), m=np.zeros((6, 8), np.float32), v=np.zeros((6, 8), np.float32),
                 w_dtype="f32", state="f32")
    h = O.Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    a = O.accumulated_step("adamw", mbs, st, h, 3)
    b = O.step("adamw", Xc, dYc, st, h, 3)
    for x, y in ((a.W, b.W), (a.m, b.m), (a.v, b.v)):
        np.testing.assert_array_equal(x, y)
