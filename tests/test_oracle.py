"""Pins for the fp64 oracle: checks against what the definitions fix, not
against the oracle itself.  CPU only.

Each group names the operation's page: fused add + RMSNorm ("optimize inner
persistent scheduler for static fusion", changes walkthrough, RMSNormAdd
benchmark with in-place update), RMSNorm / LayerNorm forward ("TMA inner
persistent scheduler", description), LayerNorm backward ("Llu/ln bwd").
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _ev(v):
    """Evaluate a closed-form entry from the hand-case fixture."""
    if isinstance(v, list):
        return [_ev(e) for e in v]
    if isinstance(v, str):
        return float(eval(v, {"__builtins__": {}}, {"sqrt": math.sqrt}))
    return float(v)


def _arr(v):
    return np.array(_ev(v), dtype=np.float64)


# ---------------------------------------------------------------- bf16 helpers

def _all_bf16_bits():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_widen_matches_torch_for_every_bf16_pattern():
    bits = _all_bf16_bits()
    ours = oracle.widen(bits)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(t)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], t[~nan])
    # signed zeros survive
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(t[~nan]))


def test_round_matches_torch_on_fp32_values():
    # fp32 values are exact in double, so one rounding from double must agree
    # with torch's fp32 -> bf16 conversion (round to nearest, ties to even).
    rng = np.random.default_rng(0)
    raw = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # force many exact ties: low 16 bits = 0x8000
    ties = (raw[:50_000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    f = np.concatenate([raw, ties]).view(np.float32)
    f = f[np.isfinite(f)]
    f = np.concatenate([f, np.float32([0.0, -0.0, 1.0, 3.3895314e38, 3.40e38, 1e-40, -1e-45])])
    ours = oracle.to_bf16(f.astype(np.float64))
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_double_against_brute_force_nearest():
    # Doubles that are not fp32 values: compare with the nearest entry of the
    # sorted table of all finite bf16 values, ties to the even pattern.
    rng = np.random.default_rng(1)
    d = np.concatenate([
        rng.standard_normal(20_000) * 10.0 ** rng.integers(-30, 30, 20_000),
        rng.standard_normal(2_000) * 1e-39,              # subnormal range
        1.0 + (np.arange(1, 512) / 512.0) * 2 ** -7,     # fine grid inside one bf16 spacing
    ])
    bits = _all_bf16_bits()
    vals = oracle.widen(bits)
    fin = np.isfinite(vals) & ~((vals == 0) & np.signbit(vals))
    order = np.argsort(vals[fin], kind="stable")
    table_v = vals[fin][order]
    table_b = bits[fin][order]
    got = oracle.to_bf16(d)
    for k in range(d.size):
        x = d[k]
        i = np.searchsorted(table_v, x)
        cands = [j for j in (i - 1, i) if 0 <= j < table_v.size]
        dist = [abs(table_v[j] - x) for j in cands]
        best = min(dist)
        near = [cands[n] for n in range(len(cands)) if dist[n] == best]
        if len(near) == 2:
            near = [j for j in near if table_b[j] % 2 == 0]
        want = table_b[near[0]]
        if table_v[near[0]] == 0.0 and x < 0:
            want = np.uint16(0x8000)
        assert got[k] == want, (x, got[k], want)


def test_round_overflow_and_nan():
    big = (2 - 2 ** -7) * 2.0 ** 127
    half_ulp = 2.0 ** (127 - 8)
    got = oracle.to_bf16(np.array([big, big + half_ulp * 0.99, big + half_ulp, -big - half_ulp,
                                   np.inf, -np.inf, np.nan]))
    assert list(got[:6]) == [0x7F7F, 0x7F7F, 0x7F80, 0xFF80, 0x7F80, 0xFF80]
    assert (got[6] & 0x7F80) == 0x7F80 and (got[6] & 0x7F) != 0


# ---------------------------------------------------------------- golden cases

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["rmsnorm_fwd"])
def test_golden_rmsnorm(case):
    y, _ = oracle.rmsnorm_fwd(_arr(case["x"]), _arr(case["w"]), case["eps"])
    np.testing.assert_allclose(y, _arr(case["y"]), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("case", _golden()["fused_add_rmsnorm"])
def test_golden_fused(case):
    s, y, _ = oracle.fused_add_rmsnorm(_arr(case["x"]), _arr(case["residual"]), _arr(case["w"]),
                                       case["eps"])
    np.testing.assert_allclose(s, _arr(case["residual_out"]), rtol=0, atol=0)
    np.testing.assert_allclose(y, _arr(case["x_out"]), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("case", _golden()["layernorm_fwd"])
def test_golden_layernorm_fwd(case):
    y, mean, rstd = oracle.layernorm_fwd(_arr(case["x"]), _arr(case["gamma"]), _arr(case["beta"]),
                                         case["eps"])
    np.testing.assert_allclose(y, _arr(case["y"]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(mean, _arr(case["mean"]), rtol=1e-15)
    np.testing.assert_allclose(rstd, _arr(case["rstd"]), rtol=1e-14)


@pytest.mark.parametrize("case", _golden()["layernorm_bwd"])
def test_golden_layernorm_bwd(case):
    dx, dg, db = oracle.layernorm_bwd(_arr(case["dy"]), _arr(case["x"]), _arr(case["mean"]),
                                      _arr(case["rstd"]), _arr(case["gamma"]))
    np.testing.assert_allclose(dx, _arr(case["dx"]), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dg, _arr(case["dgamma"]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(db, _arr(case["dbeta"]), rtol=0, atol=0)


@pytest.mark.parametrize("case", _golden()["rmsnorm_bwd"])
def test_golden_rmsnorm_bwd(case):
    dx, dw = oracle.rmsnorm_bwd(_arr(case["dy"]), _arr(case["x"]), _arr(case["rstd"]), _arr(case["w"]))
    np.testing.assert_allclose(dx, _arr(case["dx"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dw, _arr(case["dw"]), rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- RMSNorm pins

def test_rms_closed_form_mean_square():
    # w = 1: mean(y^2) = ms / (ms + eps) exactly, so about 1 - eps/ms.
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 4096)) * rng.uniform(0.01, 100, (64, 1))
    eps = 1e-6
    y, rstd = oracle.rmsnorm_fwd(x, np.ones(4096), eps)
    ms = (x ** 2).mean(axis=1)
    np.testing.assert_allclose((y ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, atol=1e-6 / ms.min() * 1.01)


def test_rms_scale_invariance_and_weight_linearity():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 1024))
    w = rng.standard_normal(1024)
    y1, _ = oracle.rmsnorm_fwd(x, w, 0.0)
    y2, _ = oracle.rmsnorm_fwd(-7.25 * x, w, 0.0)
    np.testing.assert_allclose(y2, -y1, rtol=1e-13, atol=1e-14)
    y3, _ = oracle.rmsnorm_fwd(x, 3.0 * w, 0.0)
    np.testing.assert_allclose(y3, 3.0 * y1, rtol=1e-14, atol=1e-15)


def test_rms_matches_torch_fp64():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((32, 2048)) * 3
    w = rng.standard_normal(2048)
    y, _ = oracle.rmsnorm_fwd(x, w, 1e-5)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (2048,), torch.from_numpy(w), eps=1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_rms_zero_row():
    y, rstd = oracle.rmsnorm_fwd(np.zeros((1, 8)), np.ones(8), 1e-6)
    assert np.all(y == 0) and rstd[0] == pytest.approx(1e3)


def test_fused_residual_is_exact_sum_and_reads_match():
    x, r, w = workloads.fused_inputs(16, 4096, residual_scale=4.0)
    xd, rd, wd = oracle.widen(x), oracle.widen(r), oracle.widen(w)
    s, y, rstd = oracle.fused_add_rmsnorm(x, r, w, 1e-6)
    assert np.array_equal(s, xd + rd)          # exact in fp64 for bf16 inputs
    y_ref, _ = oracle.rmsnorm_fwd(xd + rd, wd, 1e-6)
    np.testing.assert_allclose(y, y_ref, rtol=0, atol=0)
    # the other reading (normalize the rounded residual) is the same map on bf16(s)
    s2, y2, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-6, normalize_rounded=True)
    assert np.array_equal(s2, oracle.bf16_value(xd + rd))
    y2_ref, _ = oracle.rmsnorm_fwd(oracle.bf16_value(xd + rd), wd, 1e-6)
    np.testing.assert_allclose(y2, y2_ref, rtol=0, atol=0)
    # and the two readings are within half a bf16 ulp relative of each other
    assert np.max(np.abs(y2 - y) / np.maximum(np.abs(y), 1e-3)) < 2 ** -8 * 1.1


# ---------------------------------------------------------------- LayerNorm forward pins

def test_layernorm_moments():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 4096)) * 2 + 0.5
    eps = 1e-5
    y, mean, rstd = oracle.layernorm_fwd(x, np.ones(4096), np.zeros(4096), eps)
    var = x.var(axis=1)
    assert np.max(np.abs(y.mean(axis=1))) < 1e-12
    np.testing.assert_allclose(y.var(axis=1), var / (var + eps), rtol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-12)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(var + eps), rtol=1e-12)


def test_layernorm_shift_invariance_and_affine():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 1024))
    g = rng.standard_normal(1024)
    b = rng.standard_normal(1024)
    y1, m1, r1 = oracle.layernorm_fwd(x, g, b, 1e-5)
    y2, m2, r2 = oracle.layernorm_fwd(x + 3.0, g, b, 1e-5)
    np.testing.assert_allclose(y2, y1, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(m2, m1 + 3.0, rtol=1e-14)
    yn, _, _ = oracle.layernorm_fwd(x, np.ones(1024), np.zeros(1024), 1e-5)
    np.testing.assert_allclose(y1, yn * g + b, rtol=1e-13, atol=1e-14)


def test_layernorm_matches_torch_fp64():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((16, 4096)) * 2 + 0.5
    g = rng.standard_normal(4096)
    b = rng.standard_normal(4096)
    y, _, _ = oracle.layernorm_fwd(x, g, b, 1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (4096,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_layernorm_constant_row():
    g = np.arange(1, 9, dtype=np.float64)
    b = np.linspace(-1, 1, 8)
    y, mean, rstd = oracle.layernorm_fwd(np.full((2, 8), 5.0), g, b, 1e-5)
    np.testing.assert_allclose(y, np.tile(b, (2, 1)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(rstd, 1 / math.sqrt(1e-5), rtol=1e-15)


# ---------------------------------------------------------------- backward pins

def _ln_loss(x, dy, g, b, eps):
    y, _, _ = oracle.layernorm_fwd(x, g, b, eps)
    return float(np.sum(dy * y))


@pytest.mark.parametrize("rows,hidden", [(1, 4), (3, 8), (2, 5)])
def test_layernorm_bwd_finite_differences(rows, hidden):
    rng = np.random.default_rng(10 + rows * hidden)
    x = rng.standard_normal((rows, hidden))
    dy = rng.standard_normal((rows, hidden))
    g = rng.standard_normal(hidden)
    b = rng.standard_normal(hidden)
    eps = 1e-5
    _, mean, rstd = oracle.layernorm_fwd(x, g, b, eps)
    dx, dg, db = oracle.layernorm_bwd(dy, x, mean, rstd, g)
    h = 1e-6
    fd = np.zeros_like(x)
    for i in range(rows):
        for j in range(hidden):
            xp = x.copy(); xp[i, j] += h
            xm = x.copy(); xm[i, j] -= h
            fd[i, j] = (_ln_loss(xp, dy, g, b, eps) - _ln_loss(xm, dy, g, b, eps)) / (2 * h)
    np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-7)
    fdg = np.zeros(hidden)
    fdb = np.zeros(hidden)
    for j in range(hidden):
        gp = g.copy(); gp[j] += h
        gm = g.copy(); gm[j] -= h
        fdg[j] = (_ln_loss(x, dy, gp, b, eps) - _ln_loss(x, dy, gm, b, eps)) / (2 * h)
        bp = b.copy(); bp[j] += h
        bm = b.copy(); bm[j] -= h
        fdb[j] = (_ln_loss(x, dy, g, bp, eps) - _ln_loss(x, dy, g, bm, eps)) / (2 * h)
    np.testing.assert_allclose(dg, fdg, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(db, fdb, rtol=1e-6, atol=1e-8)


def test_layernorm_bwd_row_invariants_and_column_sums():
    rng = np.random.default_rng(11)
    rows, hidden = 16, 1024
    x = rng.standard_normal((rows, hidden)) * 2 + 0.5
    dy = rng.standard_normal((rows, hidden))
    _, mean, rstd = oracle.layernorm_fwd(x, np.ones(hidden), np.zeros(hidden), 1e-5)
    dx, dg, db = oracle.layernorm_bwd(dy, x, mean, rstd, np.ones(hidden))
    xhat = (x - mean[:, None]) * rstd[:, None]
    scale = np.abs(dx).max()
    # sum_j dx_j = 0 for any eps; sum_j dx_j * xhat_j = rstd * sum_j(g_j xhat_j) * eps/(var+eps)
    # (zero when eps = 0), with g = dy since gamma = 1.
    assert np.max(np.abs(dx.sum(axis=1))) < 1e-10 * scale * hidden
    var = x.var(axis=1)
    want = rstd * (dy * xhat).sum(axis=1) * 1e-5 / (var + 1e-5)
    np.testing.assert_allclose((dx * xhat).sum(axis=1), want, rtol=1e-6, atol=1e-10 * scale * hidden)
    _, mean0, rstd0 = oracle.layernorm_fwd(x, np.ones(hidden), np.zeros(hidden), 0.0)
    dx0, _, _ = oracle.layernorm_bwd(dy, x, mean0, rstd0, np.ones(hidden))
    xhat0 = (x - mean0[:, None]) * rstd0[:, None]
    assert np.max(np.abs((dx0 * xhat0).sum(axis=1))) < 1e-10 * scale * hidden
    # the column sums, by brute force over the rows
    bg = np.zeros(hidden)
    bb = np.zeros(hidden)
    for r in range(rows):
        bg += dy[r] * xhat[r]
        bb += dy[r]
    np.testing.assert_allclose(dg, bg, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, bb, rtol=1e-12, atol=1e-12)


def test_layernorm_bwd_matches_torch_autograd_fp64():
    rng = np.random.default_rng(12)
    rows, hidden = 8, 512
    x = torch.from_numpy(rng.standard_normal((rows, hidden))).requires_grad_()
    g = torch.from_numpy(rng.standard_normal(hidden) * 0.1 + 1).requires_grad_()
    b = torch.from_numpy(rng.standard_normal(hidden) * 0.1).requires_grad_()
    dy = rng.standard_normal((rows, hidden))
    y = torch.nn.functional.layer_norm(x, (hidden,), g, b, eps=1e-5)
    y.backward(torch.from_numpy(dy))
    _, mean, rstd = oracle.layernorm_fwd(x.detach().numpy(), g.detach().numpy(),
                                         b.detach().numpy(), 1e-5)
    dx, dg, db = oracle.layernorm_bwd(dy, x.detach().numpy(), mean, rstd, g.detach().numpy())
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dg, g.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(db, b.grad.numpy(), rtol=1e-12, atol=1e-12)


def _rms_loss(x, dy, w, eps):
    y, _ = oracle.rmsnorm_fwd(x, w, eps)
    return float(np.sum(dy * y))


@pytest.mark.parametrize("rows,hidden", [(1, 4), (3, 6)])
def test_rmsnorm_bwd_finite_differences(rows, hidden):
    rng = np.random.default_rng(20 + rows)
    x = rng.standard_normal((rows, hidden))
    dy = rng.standard_normal((rows, hidden))
    w = rng.standard_normal(hidden)
    eps = 1e-5
    _, rstd = oracle.rmsnorm_fwd(x, w, eps)
    dx, dw = oracle.rmsnorm_bwd(dy, x, rstd, w)
    h = 1e-6
    fd = np.zeros_like(x)
    for i in range(rows):
        for j in range(hidden):
            xp = x.copy(); xp[i, j] += h
            xm = x.copy(); xm[i, j] -= h
            fd[i, j] = (_rms_loss(xp, dy, w, eps) - _rms_loss(xm, dy, w, eps)) / (2 * h)
    np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-8)
    fdw = np.zeros(hidden)
    for j in range(hidden):
        wp = w.copy(); wp[j] += h
        wm = w.copy(); wm[j] -= h
        fdw[j] = (_rms_loss(x, dy, wp, eps) - _rms_loss(x, dy, wm, eps)) / (2 * h)
    np.testing.assert_allclose(dw, fdw, rtol=1e-6, atol=1e-8)


def test_rmsnorm_bwd_matches_torch_autograd_fp64():
    rng = np.random.default_rng(21)
    rows, hidden = 8, 512
    x = torch.from_numpy(rng.standard_normal((rows, hidden))).requires_grad_()
    w = torch.from_numpy(rng.standard_normal(hidden) * 0.1 + 1).requires_grad_()
    dy = rng.standard_normal((rows, hidden))
    y = torch.nn.functional.rms_norm(x, (hidden,), w, eps=1e-5)
    y.backward(torch.from_numpy(dy))
    _, rstd = oracle.rmsnorm_fwd(x.detach().numpy(), w.detach().numpy(), 1e-5)
    dx, dw = oracle.rmsnorm_bwd(dy, x.detach().numpy(), rstd, w.detach().numpy())
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dw, w.grad.numpy(), rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- outer normalization pins

def test_outer_norm_column_moments():
    rng = np.random.default_rng(30)
    x = rng.standard_normal((513, 64)) * rng.uniform(0.1, 5, 64) + rng.uniform(-3, 3, 64)
    eps = 1e-5
    y, mean, rstd = oracle.outer_norm_fwd(x, np.ones(64), np.zeros(64), eps)
    var = x.var(axis=0)
    assert np.max(np.abs(y.mean(axis=0))) < 1e-12
    np.testing.assert_allclose(y.var(axis=0), var / (var + eps), rtol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=0), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(var + eps), rtol=1e-12)


def test_outer_norm_matches_torch_batch_norm_fp64():
    rng = np.random.default_rng(31)
    rows, hidden = 300, 48
    x = torch.from_numpy(rng.standard_normal((rows, hidden)) * 2 + 0.5).requires_grad_()
    g = torch.from_numpy(rng.standard_normal(hidden) * 0.1 + 1).requires_grad_()
    b = torch.from_numpy(rng.standard_normal(hidden) * 0.1).requires_grad_()
    dy = rng.standard_normal((rows, hidden))
    y = torch.nn.functional.batch_norm(x, None, None, g, b, training=True, eps=1e-5)
    y.backward(torch.from_numpy(dy))
    yo, mean, rstd = oracle.outer_norm_fwd(x.detach().numpy(), g.detach().numpy(),
                                           b.detach().numpy(), 1e-5)
    np.testing.assert_allclose(yo, y.detach().numpy(), rtol=1e-11, atol=1e-12)
    dx, dg, db = oracle.outer_norm_bwd(dy, x.detach().numpy(), mean, rstd, g.detach().numpy())
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dg, g.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(db, b.grad.numpy(), rtol=1e-12, atol=1e-12)


def _outer_loss(x, dy, g, b, eps):
    y, _, _ = oracle.outer_norm_fwd(x, g, b, eps)
    return float(np.sum(dy * y))


def test_outer_norm_bwd_finite_differences():
    rng = np.random.default_rng(32)
    rows, hidden = 5, 3
    x = rng.standard_normal((rows, hidden))
    dy = rng.standard_normal((rows, hidden))
    g = rng.standard_normal(hidden)
    b = rng.standard_normal(hidden)
    eps = 1e-5
    _, mean, rstd = oracle.outer_norm_fwd(x, g, b, eps)
    dx, dg, db = oracle.outer_norm_bwd(dy, x, mean, rstd, g)
    h = 1e-6
    for i in range(rows):
        for j in range(hidden):
            xp = x.copy(); xp[i, j] += h
            xm = x.copy(); xm[i, j] -= h
            fd = (_outer_loss(xp, dy, g, b, eps) - _outer_loss(xm, dy, g, b, eps)) / (2 * h)
            assert dx[i, j] == pytest.approx(fd, rel=1e-6, abs=1e-8)
    for j in range(hidden):
        gp = g.copy(); gp[j] += h
        gm = g.copy(); gm[j] -= h
        fd = (_outer_loss(x, dy, gp, b, eps) - _outer_loss(x, dy, gm, b, eps)) / (2 * h)
        assert dg[j] == pytest.approx(fd, rel=1e-6, abs=1e-8)
        assert db[j] == pytest.approx(dy[:, j].sum(), rel=1e-12)


def test_outer_norm_hand_case():
    # one column (2, 4, 6): mean 4, var 8/3, rstd sqrt(3/8); eps = 0, gamma 2, beta 1
    y, mean, rstd = oracle.outer_norm_fwd(np.array([[2.0], [4.0], [6.0]]), [2.0], [1.0], 0.0)
    r = math.sqrt(3 / 8)
    np.testing.assert_allclose(y[:, 0], [1 - 4 * r, 1.0, 1 + 4 * r], rtol=1e-14)
    assert mean[0] == 4.0 and rstd[0] == pytest.approx(r, rel=1e-15)


# ---------------------------------------------------------------- fused add + RMSNorm backward pins

def _fused_loss(x, r, w, dy, dres, eps):
    s, y, _ = oracle.fused_add_rmsnorm(x, r, w, eps)
    return float(np.sum(dy * y) + np.sum(dres * s))


def test_fused_add_rmsnorm_bwd_finite_differences():
    rng = np.random.default_rng(40)
    rows, hidden = 3, 6
    x = rng.standard_normal((rows, hidden))
    r = rng.standard_normal((rows, hidden)) * 2
    w = rng.standard_normal(hidden) * 0.3 + 1
    dy = rng.standard_normal((rows, hidden))
    dres = rng.standard_normal((rows, hidden))
    eps = 1e-3
    ds, dw = oracle.fused_add_rmsnorm_bwd(dy, dres, x + r, w, eps)
    h = 1e-6
    for i in range(rows):
        for j in range(hidden):
            for which in (0, 1):  # both inputs get the same gradient
                xp, xm, rp, rm = x.copy(), x.copy(), r.copy(), r.copy()
                if which == 0:
                    xp[i, j] += h; xm[i, j] -= h
                else:
                    rp[i, j] += h; rm[i, j] -= h
                fd = (_fused_loss(xp, rp, w, dy, dres, eps) - _fused_loss(xm, rm, w, dy, dres, eps)) / (2 * h)
                assert ds[i, j] == pytest.approx(fd, rel=1e-6, abs=1e-8)
    for j in range(hidden):
        wp, wm = w.copy(), w.copy()
        wp[j] += h; wm[j] -= h
        fd = (_fused_loss(x, r, wp, dy, dres, eps) - _fused_loss(x, r, wm, dy, dres, eps)) / (2 * h)
        assert dw[j] == pytest.approx(fd, rel=1e-6, abs=1e-8)


def test_fused_add_rmsnorm_bwd_matches_torch_autograd_fp64():
    rng = np.random.default_rng(41)
    rows, hidden, eps = 17, 40, 1e-5
    x = torch.from_numpy(rng.standard_normal((rows, hidden))).requires_grad_()
    r = torch.from_numpy(rng.standard_normal((rows, hidden)) * 4).requires_grad_()
    w = torch.from_numpy(rng.standard_normal(hidden) * 0.1 + 1).requires_grad_()
    dy = rng.standard_normal((rows, hidden))
    dres = rng.standard_normal((rows, hidden))
    s = x + r
    y = s * torch.rsqrt((s * s).mean(dim=1, keepdim=True) + eps) * w
    ((torch.from_numpy(dy) * y).sum() + (torch.from_numpy(dres) * s).sum()).backward()
    ds, dw = oracle.fused_add_rmsnorm_bwd(dy, dres, (x + r).detach().numpy(), w.detach().numpy(), eps)
    np.testing.assert_allclose(ds, x.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ds, r.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dw, w.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_fused_add_rmsnorm_bwd_without_residual_gradient_is_rmsnorm_bwd():
    rng = np.random.default_rng(42)
    s = rng.standard_normal((9, 24))
    w = rng.standard_normal(24)
    dy = rng.standard_normal((9, 24))
    ds, dw = oracle.fused_add_rmsnorm_bwd(dy, None, s, w, 1e-6)
    # closed form of the RMSNorm gradient: ds = rstd * (g - s_hat * mean(g * s_hat)), g = dy * w
    rstd = 1 / np.sqrt((s * s).mean(axis=1) + 1e-6)
    sh = s * rstd[:, None]
    g = dy * w
    expect = rstd[:, None] * (g - sh * (g * sh).mean(axis=1)[:, None])
    np.testing.assert_allclose(ds, expect, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dw, (dy * sh).sum(axis=0), rtol=1e-12, atol=1e-13)
