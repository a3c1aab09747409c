"""GPU parity: every kernel family, through the C ABI, against the fp64
oracle on the same seeded inputs.

Small and ragged cases compare every element; the full-size workloads
(LLM prefill fused add+RMSNorm up to 65536 x 8192, LayerNorm forward
16384 x {1024, 4096, 12288}, LayerNorm backward 16384 x {1024, 4096, 8192})
run in the launch configuration the benchmark uses and compare sampled rows
(every row for the column sums of the backward pass).
"""
import numpy as np
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32, host_f64, ulp_diff_bf16

pytestmark = pytest.mark.gpu

FWD_PATHS = ("reg", "cluster", "bulk")
BWD_PATHS = ("reg", "bulk")
RAGGED_ROWS = (1, 3, 37, 152, 301)


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    nf.set_path("auto")
    yield
    nf.set_path("auto")


def _sample_rows(rows: int, n: int = 48, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = {0, rows - 1, rows // 2}
    pick.update(rng.integers(0, rows, size=min(n, rows)).tolist())
    return np.array(sorted(pick), dtype=np.int64)


# ---------------------------------------------------------------- fused add + RMSNorm

def _run_fused(rows, hidden, eps, path, residual_scale=1.0, draw_rows=None, seed=0):
    x, r, w = workloads.fused_inputs(rows, hidden, seed=seed, residual_scale=residual_scale,
                                     draw_rows=draw_rows)
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(x, r, w, eps)
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    with nf.forced_path(path):
        nf.fused_add_rmsnorm(xd, rd, wd, eps)
    torch.cuda.synchronize()
    return xd, rd, s_ref, y_ref


def _check_fused(xd, rd, s_ref, y_ref, tag):
    check_bf16(xd, y_ref, f"{tag} x_out")
    # residual out = bf16(fp32(x + r)); equals bf16(x + r) except where the
    # fp32 sum itself was inexact (double rounding): at most 1 ulp, rarely.
    d = ulp_diff_bf16(rd, oracle.to_bf16(s_ref))
    assert d.max() <= 1, (tag, int(d.max()))
    assert (d > 0).mean() < 1e-4, (tag, float((d > 0).mean()))


@pytest.mark.parametrize("path", FWD_PATHS + ("auto",))
def test_fused_decode_16x4096(path):
    # fused add+RMSNorm, 16 rows x 4096, eps 1e-6, seed 0
    xd, rd, s_ref, y_ref = _run_fused(16, 4096, 1e-6, path)
    _check_fused(xd, rd, s_ref, y_ref, f"16x4096/{path}")


@pytest.mark.parametrize("path", FWD_PATHS)
@pytest.mark.parametrize("hidden", workloads.HIDDEN_SET)
@pytest.mark.parametrize("rows", RAGGED_ROWS)
def test_fused_all_sizes(rows, hidden, path):
    xd, rd, s_ref, y_ref = _run_fused(rows, hidden, 1e-5, path, residual_scale=4.0, seed=rows)
    _check_fused(xd, rd, s_ref, y_ref, f"{rows}x{hidden}/{path}")


@pytest.mark.parametrize("hidden", (4096, 8192))
@pytest.mark.parametrize("rows", (1, 2, 4, 8, 32, 128))
def test_fused_small_batch_sweep(rows, hidden):
    # first `rows` rows of a 128-row draw, eps 1e-6, library's own path choice
    xd, rd, s_ref, y_ref = _run_fused(rows, hidden, 1e-6, "auto", draw_rows=128)
    _check_fused(xd, rd, s_ref, y_ref, f"sweep {rows}x{hidden}")


@pytest.mark.parametrize("hidden", (2048, 4096, 5120, 8192))
@pytest.mark.parametrize("rows", (4096, 16384, 65536))
def test_fused_prefill_full_size_sampled(rows, hidden):
    # LLM prefill sizes in the benchmark's launch configuration (auto path):
    # inputs drawn on the device, sampled rows copied out before the
    # in-place call, compared with the oracle row by row.
    x, r, w = workloads.fused_inputs(rows, hidden, residual_scale=4.0, device="cuda")
    idx = _sample_rows(rows, seed=rows + hidden)
    ti = torch.from_numpy(idx).cuda()
    xs, rs = x.index_select(0, ti).cpu(), r.index_select(0, ti).cpu()
    nf.fused_add_rmsnorm(x, r, w, 1e-5)
    torch.cuda.synchronize()
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(xs, rs, w.cpu(), 1e-5)
    _check_fused(x.index_select(0, ti), r.index_select(0, ti), s_ref, y_ref, f"{rows}x{hidden}")
    # a global property on every row: outputs are finite
    assert torch.isfinite(x.float()).all() and torch.isfinite(r.float()).all()


# ---------------------------------------------------------------- RMSNorm forward

@pytest.mark.parametrize("path", FWD_PATHS)
@pytest.mark.parametrize("hidden", workloads.HIDDEN_SET)
@pytest.mark.parametrize("rows", RAGGED_ROWS)
def test_rmsnorm_fwd_all_sizes(rows, hidden, path):
    x, w = workloads.rms_inputs(rows, hidden, seed=rows)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    xd, wd = x.cuda(), w.cuda()
    with nf.forced_path(path):
        y = nf.rmsnorm_fwd(xd, wd, 1e-6)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"rms {rows}x{hidden}/{path}")
    assert torch.equal(xd.cpu(), x)  # input untouched


@pytest.mark.parametrize("path", FWD_PATHS)
def test_rmsnorm_in_place(path):
    x, w = workloads.rms_inputs(77, 8192)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    xd = x.cuda()
    with nf.forced_path(path):
        nf.rmsnorm_fwd(xd, w.cuda(), 1e-6, out=xd)
    torch.cuda.synchronize()
    check_bf16(xd, y_ref, f"rms in place/{path}")


# ---------------------------------------------------------------- LayerNorm forward

def _check_ln_fwd(y, mean, rstd, x, g, b, eps, tag):
    y_ref, m_ref, r_ref = oracle.layernorm_fwd(x, g, b, eps)
    check_bf16(y, y_ref, f"{tag} y")
    check_f32(mean, m_ref, f"{tag} mean")
    check_f32(rstd, r_ref, f"{tag} rstd", rtol=1e-4)


@pytest.mark.parametrize("path", FWD_PATHS)
@pytest.mark.parametrize("hidden", workloads.HIDDEN_SET)
@pytest.mark.parametrize("rows", RAGGED_ROWS)
def test_layernorm_fwd_all_sizes(rows, hidden, path):
    x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, seed=rows)
    with nf.forced_path(path):
        y, mean, rstd = nf.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    _check_ln_fwd(y, mean, rstd, x, g, b, 1e-5, f"ln {rows}x{hidden}/{path}")


@pytest.mark.parametrize("hidden", (1024, 4096, 12288))
def test_layernorm_fwd_full_size_sampled(hidden):
    rows = 16384
    x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, device="cuda")
    y, mean, rstd = nf.layernorm_fwd(x, g, b, 1e-5)
    torch.cuda.synchronize()
    idx = torch.from_numpy(_sample_rows(rows, seed=hidden)).cuda()
    _check_ln_fwd(y.index_select(0, idx), mean.index_select(0, idx), rstd.index_select(0, idx),
                  x.index_select(0, idx).cpu(), g.cpu(), b.cpu(), 1e-5, f"ln full {hidden}")


@pytest.mark.parametrize("path", FWD_PATHS)
def test_layernorm_constant_rows(path):
    # var = 0: y = beta, rstd = 1/sqrt(eps), mean = the constant
    rows, hidden = 5, 4096
    x = torch.full((rows, hidden), 3.25, dtype=torch.bfloat16)
    _, g, b = workloads.layernorm_fwd_inputs(1, hidden)
    with nf.forced_path(path):
        y, mean, rstd = nf.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), b.expand(rows, hidden))
    assert torch.allclose(mean.cpu(), torch.full((rows,), 3.25))
    assert torch.allclose(rstd.cpu(), torch.full((rows,), 1e-5 ** -0.5), rtol=1e-5)


def test_rms_zero_and_large_rows():
    hidden = 4096
    x, w = workloads.rms_inputs(4, hidden)
    x[0] = 0
    x[1] = (x[1].float() * 1000).to(torch.bfloat16)
    x[2] = (x[2].float() * 1e-3).to(torch.bfloat16)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    for path in FWD_PATHS:
        with nf.forced_path(path):
            y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
        torch.cuda.synchronize()
        check_bf16(y, y_ref, f"rms extremes/{path}")
        assert torch.count_nonzero(y[0]) == 0


# ---------------------------------------------------------------- LayerNorm backward

def _ln_bwd_case(rows, hidden, seed=0, device="cpu"):
    x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, seed=seed, device=device)
    return x, dy, g


def _saved_stats(x_cpu, eps=1e-5, chunk=2048):
    """mean/rstd from the fp64 oracle forward, rounded to fp32."""
    hidden = x_cpu.shape[1]
    ones = np.ones(hidden)
    zeros = np.zeros(hidden)
    ms, rs = [], []
    for i in range(0, x_cpu.shape[0], chunk):
        _, m, r = oracle.layernorm_fwd(x_cpu[i:i + chunk], ones, zeros, eps)
        ms.append(m)
        rs.append(r)
    m = np.concatenate(ms).astype(np.float32)
    r = np.concatenate(rs).astype(np.float32)
    return torch.from_numpy(m), torch.from_numpy(r)


def _oracle_bwd_chunked(dy, x, mean, rstd, g, chunk=2048):
    hidden = x.shape[1]
    dgs, dbs, dxs = np.zeros(hidden), np.zeros(hidden), []
    for i in range(0, x.shape[0], chunk):
        dx, dg, db = oracle.layernorm_bwd(dy[i:i + chunk], x[i:i + chunk], mean[i:i + chunk],
                                          rstd[i:i + chunk], g)
        dxs.append(dx)
        dgs += dg
        dbs += db
    return np.concatenate(dxs), dgs, dbs


@pytest.mark.parametrize("path", BWD_PATHS)
@pytest.mark.parametrize("hidden", workloads.HIDDEN_SET)
@pytest.mark.parametrize("rows", (1, 3, 37, 152, 301, 1000))
def test_layernorm_bwd_all_sizes(rows, hidden, path):
    x, dy, g = _ln_bwd_case(rows, hidden, seed=rows)
    mean, rstd = _saved_stats(x)
    dx_ref, dg_ref, db_ref = oracle.layernorm_bwd(dy, x, mean, rstd, g)
    with nf.forced_path(path):
        dx, dg, db = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"ln bwd dx {rows}x{hidden}/{path}")
    check_f32(dg, dg_ref, f"ln bwd dgamma {rows}x{hidden}/{path}")
    check_f32(db, db_ref, f"ln bwd dbeta {rows}x{hidden}/{path}")


@pytest.mark.parametrize("path", ("auto",) + BWD_PATHS)
@pytest.mark.parametrize("hidden", (1024, 4096, 8192))
def test_layernorm_bwd_full_size(hidden, path):
    rows = 16384
    x, dy, g = _ln_bwd_case(rows, hidden)
    mean, rstd = _saved_stats(x)
    with nf.forced_path(path):
        dx, dg, db = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
    torch.cuda.synchronize()
    dx_ref, dg_ref, db_ref = _oracle_bwd_chunked(dy, x, mean, rstd, g)
    check_f32(dg, dg_ref, f"ln bwd full dgamma {hidden}/{path}")
    check_f32(db, db_ref, f"ln bwd full dbeta {hidden}/{path}")
    idx = _sample_rows(rows, seed=hidden)
    check_bf16(dx.cpu()[torch.from_numpy(idx)], dx_ref[idx], f"ln bwd full dx {hidden}/{path}")


@pytest.mark.parametrize("path", BWD_PATHS)
def test_layernorm_bwd_in_place_alias(path):
    rows, hidden = 640, 4096
    x, dy, g = _ln_bwd_case(rows, hidden, seed=5)
    mean, rstd = _saved_stats(x)
    dx_ref, dg_ref, db_ref = oracle.layernorm_bwd(dy, x, mean, rstd, g)
    dyd = dy.cuda()
    with nf.forced_path(path):
        dx, dg, db = nf.layernorm_bwd(dyd, x.cuda(), mean.cuda(), rstd.cuda(), g.cuda(), out=dyd)
    torch.cuda.synchronize()
    check_bf16(dyd, dx_ref, "ln bwd dx written over dy")
    check_f32(dg, dg_ref, "ln bwd dgamma (aliased)")


def test_layernorm_bwd_workspace_too_small():
    rows, hidden = 64, 1024
    x, dy, g = _ln_bwd_case(rows, hidden)
    mean, rstd = _saved_stats(x)
    need = nf.nf_layernorm_bwd_workspace_size(rows, hidden)
    # the query covers every family; the call needs its own plan's partials
    plan = nf.nf_plan_query("layernorm_bwd", rows, hidden)
    need_run = plan["partials"] * 2 * hidden * 4
    assert need >= need_run > 0
    ws = torch.empty(need_run - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nf.NFError) as e:
        nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda(), workspace=ws)
    assert e.value.status == nf.NF_ERR_WORKSPACE_TOO_SMALL


def test_layernorm_bwd_zero_rows_zeroes_grads():
    hidden = 4096
    dg = torch.full((hidden,), 7.0, device="cuda")
    db = torch.full((hidden,), 7.0, device="cuda")
    st = nf.nf_layernorm_bwd(0, dg.data_ptr(), db.data_ptr(), 0, 0, 0, 0, 0, 0, hidden, 0, 0,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == nf.NF_OK
    assert torch.count_nonzero(dg) == 0 and torch.count_nonzero(db) == 0


# ---------------------------------------------------------------- RMSNorm backward

def _rms_bwd_ref(dy, x, w, eps, chunk=2048):
    """fp64 oracle: rstd from the oracle forward, then the oracle backward."""
    hidden = x.shape[1]
    dxs, dws = [], np.zeros(hidden)
    for i in range(0, x.shape[0], chunk):
        _, rstd = oracle.rmsnorm_fwd(x[i:i + chunk], w, eps)
        dx, dw = oracle.rmsnorm_bwd(dy[i:i + chunk], x[i:i + chunk], rstd, w)
        dxs.append(dx)
        dws += dw
    return np.concatenate(dxs), dws


@pytest.mark.parametrize("path", BWD_PATHS)
@pytest.mark.parametrize("hidden", workloads.HIDDEN_SET)
@pytest.mark.parametrize("rows", (1, 3, 37, 152, 301, 1000))
def test_rmsnorm_bwd_all_sizes(rows, hidden, path):
    x, dy, w = workloads.rms_bwd_inputs(rows, hidden, seed=rows)
    dx_ref, dw_ref = _rms_bwd_ref(dy, x, w, 1e-6)
    with nf.forced_path(path):
        dx, dw = nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"rms bwd dx {rows}x{hidden}/{path}")
    check_f32(dw, dw_ref, f"rms bwd dw {rows}x{hidden}/{path}")


@pytest.mark.parametrize("path", ("auto",) + BWD_PATHS)
@pytest.mark.parametrize("hidden", (4096, 8192))
def test_rmsnorm_bwd_full_size(hidden, path):
    rows = 16384
    x, dy, w = workloads.rms_bwd_inputs(rows, hidden)
    with nf.forced_path(path):
        dx, dw = nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-5)
    torch.cuda.synchronize()
    dx_ref, dw_ref = _rms_bwd_ref(dy, x, w, 1e-5)
    check_f32(dw, dw_ref, f"rms bwd full dw {hidden}/{path}")
    idx = _sample_rows(rows, seed=hidden)
    check_bf16(dx.cpu()[torch.from_numpy(idx)], dx_ref[idx], f"rms bwd full dx {hidden}/{path}")


@pytest.mark.parametrize("hidden", (5120, 12288))
def test_rmsnorm_bwd_automatic_runtime_hidden(hidden):
    # from 1024 rows the automatic choice runs the RMSNorm and fused-add
    # backward at these sizes on the runtime-hidden kernels
    rows = 16384
    assert nf.nf_plan_query("rmsnorm_bwd", rows, hidden)["path"] == "dynamic"
    x, dy, w = workloads.rms_bwd_inputs(rows, hidden, seed=hidden)
    dx, dw = nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-5)
    torch.cuda.synchronize()
    dx_ref, dw_ref = _rms_bwd_ref(dy, x, w, 1e-5)
    check_f32(dw, dw_ref, f"rms bwd auto dw {hidden}")
    idx = _sample_rows(rows, seed=hidden)
    check_bf16(dx.cpu()[torch.from_numpy(idx)], dx_ref[idx], f"rms bwd auto dx {hidden}")
    # the fused-add backward on the same kernels (the residual gradient in the ring)
    rows = 2048
    s_, w2, dy2, dres = workloads.fused_bwd_inputs(rows, hidden, seed=hidden + 1)
    assert nf.nf_plan_query("rmsnorm_bwd", rows, hidden)["path"] == "dynamic"
    ds_ref, dw2_ref = oracle.fused_add_rmsnorm_bwd(dy2, dres, s_, w2, 1e-6)
    ds, dw2 = nf.fused_add_rmsnorm_bwd(dy2.cuda(), s_.cuda(), w2.cuda(), dres.cuda(), 1e-6)
    ds_b, dw2_b = nf.fused_add_rmsnorm_bwd(dy2.cuda(), s_.cuda(), w2.cuda(), dres.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(ds, ds_ref, f"fused bwd auto dx {hidden}")
    check_f32(dw2, dw2_ref, f"fused bwd auto dw {hidden}")
    assert torch.equal(ds, ds_b) and torch.equal(dw2, dw2_b)


@pytest.mark.parametrize("path", BWD_PATHS)
def test_rmsnorm_bwd_in_place_and_deterministic(path):
    rows, hidden = 640, 8192
    x, dy, w = workloads.rms_bwd_inputs(rows, hidden, seed=9)
    dx_ref, dw_ref = _rms_bwd_ref(dy, x, w, 1e-6)
    with nf.forced_path(path):
        dyd = dy.cuda()
        _, dw1 = nf.rmsnorm_bwd(dyd, x.cuda(), w.cuda(), 1e-6, out=dyd)
        _, dw2 = nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(dyd, dx_ref, f"rms bwd dx written over dy/{path}")
    check_f32(dw1, dw_ref, f"rms bwd dw/{path}")
    assert torch.equal(dw1, dw2)


def test_rmsnorm_bwd_zero_rows_and_small_workspace():
    hidden = 2048
    dw = torch.full((hidden,), 3.0, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert nf.nf_rmsnorm_bwd(0, dw.data_ptr(), 0, 0, 0, 0, hidden, 1e-6, 0, 0, s) == nf.NF_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw) == 0
    x, dy, w = workloads.rms_bwd_inputs(64, hidden)
    need = nf.nf_rmsnorm_bwd_workspace_size(64, hidden)
    need_run = nf.nf_plan_query("rmsnorm_bwd", 64, hidden)["partials"] * hidden * 4
    assert need >= need_run > 0
    ws = torch.empty(need_run - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nf.NFError) as e:
        nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-6, workspace=ws)
    assert e.value.status == nf.NF_ERR_WORKSPACE_TOO_SMALL


# ---------------------------------------------------------------- determinism, empty, status

@pytest.mark.parametrize("path", FWD_PATHS)
def test_determinism_bitwise_forward(path):
    rows, hidden = 1000, 8192
    x, res, w = workloads.fused_inputs(rows, hidden)
    outs = []
    for _ in range(2):
        xd, rd = x.cuda(), res.cuda()
        with nf.forced_path(path):
            nf.fused_add_rmsnorm(xd, rd, w.cuda(), 1e-6)
        outs.append((xd.cpu(), rd.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("path", BWD_PATHS)
def test_determinism_bitwise_backward(path):
    xb, dy, g = _ln_bwd_case(3000, 4096)
    mean, rstd = _saved_stats(xb)
    with nf.forced_path(path):
        r1 = nf.layernorm_bwd(dy.cuda(), xb.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
        r2 = nf.layernorm_bwd(dy.cuda(), xb.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
    for a, b in zip(r1, r2):
        assert torch.equal(a.cpu(), b.cpu())


def test_zero_rows_leaves_buffers_untouched():
    x = torch.randn(4, 4096, device="cuda").to(torch.bfloat16)
    before = x.clone()
    st = nf.nf_fused_add_rmsnorm(x.data_ptr(), x.data_ptr(), x.data_ptr(), 0, 4096, 1e-6,
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == nf.NF_OK and torch.equal(x, before)


def test_plan_query_matches_pure_planner():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for op in ("fused_add_rmsnorm", "layernorm_fwd", "layernorm_bwd"):
        for rows in (1, 16, 4096):
            assert nf.nf_plan_query(op, rows, 4096) == nf.nf_plan_compute(op, rows, 4096, sms)[1]
    with nf.forced_path("bulk"):
        assert nf.nf_plan_query("fused_add_rmsnorm", 4096, 8192)["path"] == "bulk"


def test_bounded_wait_reports_timeout_and_context_survives():
    s = torch.cuda.current_stream().cuda_stream
    assert nf.nf_get_device_status(s) == nf.NF_OK
    assert nf.nf_selftest_wait_timeout(2_000_000, s) == nf.NF_OK  # 2 ms
    assert nf.nf_get_device_status(s) == nf.NF_ERR_TIMEOUT
    assert nf.nf_get_device_status(s) == nf.NF_OK                  # cleared
    # the context still works
    x, w = workloads.rms_inputs(8, 1024)
    y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(y, oracle.rmsnorm_fwd(x, w, 1e-6)[0], "after timeout")


def test_floor_probes_run_and_copy_exactly():
    # the launch-floor probes the benchmark times: an empty dependent launch
    # and a plain copy of a small-batch call's bytes (one CTA and a ragged
    # multi-CTA size)
    s = torch.cuda.current_stream().cuda_stream
    assert nf.nf_selftest_floor(0, 0, 0, 0, s) == nf.NF_OK
    for nbytes in (16, 16384, 16 * 5000 + 16):
        src = torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), dtype=torch.int32, device="cuda")
        dst = torch.zeros_like(src)
        assert nf.nf_selftest_floor(1, dst.data_ptr(), src.data_ptr(), nbytes, s) == nf.NF_OK
        torch.cuda.synchronize()
        assert torch.equal(dst, src)
