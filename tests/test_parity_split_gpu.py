"""GPU parity of the split family (a row over any number of CTAs, row
statistics through the workspace) and of the grid family (the same rows held
on chip across one grid barrier) against the fp64 oracle: forced at short
and ragged rows, automatic beyond the cluster limits, more rows than one
grid dimension holds, in place, determinism, the bounded barrier wait, and
the workspace rules of the forward calls."""
import numpy as np
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32, ulp_diff_bf16

pytestmark = pytest.mark.gpu

FORCED = ((5, 8), (300, 1000), (33, 8200), (7, 20000))   # (rows, hidden); 8200 = two chunks, ragged
AUTO_FWD = ((2, 262152), (1, 1 << 20), (4, 1 << 22), (9, 1 << 20))
AUTO_BWD = ((3, 131080), (2, 1 << 20), (2, 1 << 22), (4, 1 << 22), (9, 1 << 20))
# forced onto the grid family: one vector in all (one CTA with columns),
# ragged slices, the row bound of 8, a million columns, few short rows
GRID_FORCED = ((1, 8), (5, 8), (3, 20000), (8, 8200), (7, 1 << 20), (2, 1000))
ONE_BLOCK = ((1, 8200),)                                 # forced, one row: one row block
# forced, more than 16 rows per row block: the row statistics go through the
# separate merge launch instead of being merged inside the apply pass
MANY_ROWS = ((5000, 8200),)


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    nf.set_path("auto")
    yield
    nf.set_path("auto")


def _path(rows, hidden, op):
    auto = (rows, hidden) in AUTO_FWD + AUTO_BWD
    return "auto" if auto else "split"


def _grid_fits(op, rows, hidden):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, _ = nf.nf_plan_compute(op, rows, hidden, sms, "grid")
    return st == nf.NF_OK


def _family(rows, hidden, op):
    """The family a call runs on: forced split, or the automatic choice
    (grid where the rows fit on chip, except for the RMSNorm backward, else
    split)."""
    if _path(rows, hidden, op) == "split" or op == "rmsnorm_bwd":
        return "split"
    return "grid" if _grid_fits(op, rows, hidden) else "split"


@pytest.mark.parametrize("rows,hidden", FORCED + AUTO_FWD)
def test_split_fused(rows, hidden):
    x, r, w = workloads.fused_inputs(rows, hidden, seed=rows + hidden, residual_scale=4.0)
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-5)
    xd, rd = x.cuda(), r.cuda()
    with nf.forced_path(_path(rows, hidden, "f")):
        assert nf.nf_plan_query("fused_add_rmsnorm", rows, hidden)["path"] == \
            _family(rows, hidden, "fused_add_rmsnorm")
        nf.fused_add_rmsnorm(xd, rd, w.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(xd, y_ref, f"split fused {rows}x{hidden}")
    d = ulp_diff_bf16(rd, oracle.to_bf16(s_ref))
    assert d.max() <= 1 and (d > 0).mean() < 1e-3


@pytest.mark.parametrize("rows,hidden", FORCED + AUTO_FWD)
def test_split_rmsnorm_fwd(rows, hidden):
    x, w = workloads.rms_inputs(rows, hidden, seed=rows + hidden)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    with nf.forced_path(_path(rows, hidden, "f")):
        y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"split rms {rows}x{hidden}")


@pytest.mark.parametrize("rows,hidden", FORCED + AUTO_FWD)
def test_split_layernorm_fwd(rows, hidden):
    x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, seed=rows + hidden)
    y_ref, m_ref, r_ref = oracle.layernorm_fwd(x, g, b, 1e-5)
    with nf.forced_path(_path(rows, hidden, "f")):
        y, mean, rstd = nf.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"split ln {rows}x{hidden}")
    check_f32(mean, m_ref, f"split ln mean {rows}x{hidden}")
    check_f32(rstd, r_ref, f"split ln rstd {rows}x{hidden}", rtol=1e-4)


@pytest.mark.parametrize("rows,hidden", FORCED + ONE_BLOCK + MANY_ROWS + AUTO_BWD)
def test_split_layernorm_bwd(rows, hidden):
    x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, seed=rows + hidden)
    _, m, r = oracle.layernorm_fwd(x, np.ones(hidden), np.zeros(hidden), 1e-5)
    mean, rstd = torch.from_numpy(m.astype(np.float32)), torch.from_numpy(r.astype(np.float32))
    dx_ref, dg_ref, db_ref = oracle.layernorm_bwd(dy, x, mean, rstd, g)
    with nf.forced_path(_path(rows, hidden, "b")):
        assert nf.nf_plan_query("layernorm_bwd", rows, hidden)["path"] == \
            _family(rows, hidden, "layernorm_bwd")
        dx, dg, db = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
        dx2, dg2, db2 = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"split ln bwd dx {rows}x{hidden}")
    check_f32(dg, dg_ref, f"split ln bwd dgamma {rows}x{hidden}")
    check_f32(db, db_ref, f"split ln bwd dbeta {rows}x{hidden}")
    assert torch.equal(dx, dx2) and torch.equal(dg, dg2) and torch.equal(db, db2)


@pytest.mark.parametrize("rows,hidden", FORCED + ONE_BLOCK + MANY_ROWS + AUTO_BWD)
@pytest.mark.parametrize("fused", (False, True))
def test_split_rmsnorm_bwd(rows, hidden, fused):
    if fused:
        s, w, dy, dres = workloads.fused_bwd_inputs(rows, hidden, seed=rows + hidden)
        dx_ref, dw_ref = oracle.fused_add_rmsnorm_bwd(dy, dres, s, w, 1e-6)
    else:
        s, dy, w = workloads.rms_bwd_inputs(rows, hidden, seed=rows + hidden)
        _, rstd = oracle.rmsnorm_fwd(s, w, 1e-6)
        dx_ref, dw_ref = oracle.rmsnorm_bwd(dy, s, rstd, w)
    with nf.forced_path(_path(rows, hidden, "b")):
        assert nf.nf_plan_query("rmsnorm_bwd", rows, hidden)["path"] == \
            _family(rows, hidden, "rmsnorm_bwd")
        if fused:
            dx, dw = nf.fused_add_rmsnorm_bwd(dy.cuda(), s.cuda(), w.cuda(), dres.cuda(), 1e-6)
        else:
            dx, dw = nf.rmsnorm_bwd(dy.cuda(), s.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"split rms bwd dx {rows}x{hidden} fused={fused}")
    check_f32(dw, dw_ref, f"split rms bwd dw {rows}x{hidden} fused={fused}")


def test_split_more_rows_than_one_grid_dimension():
    # 70000 rows: the (chunk, row) launches walk rows in steps of 65535
    rows, hidden = 70000, 16
    x, w = workloads.rms_inputs(rows, hidden, seed=9)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    with nf.forced_path("split"):
        y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
        xl, gl, bl = workloads.layernorm_fwd_inputs(rows, hidden, seed=10)
        yl, ml, rl = nf.layernorm_fwd(xl.cuda(), gl.cuda(), bl.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, "split rms 70000 rows")
    yl_ref, ml_ref, rl_ref = oracle.layernorm_fwd(xl, gl, bl, 1e-5)
    check_bf16(yl, yl_ref, "split ln 70000 rows")
    check_f32(ml, ml_ref, "split ln mean 70000 rows")


def test_split_forward_needs_a_workspace():
    rows, hidden = 2, 262152
    x = torch.zeros(rows, hidden, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(hidden, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    # the plain call has no workspace for the split plan
    assert nf.nf_rmsnorm_fwd(y.data_ptr(), x.data_ptr(), w.data_ptr(), rows, hidden, 1e-6, s) == \
        nf.NF_ERR_WORKSPACE_TOO_SMALL
    need = nf.nf_workspace_size(nf.NF_OP_RMSNORM_FWD, rows, hidden)
    assert need >= rows * 8 * (-(-hidden // 8192))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert nf.nf_rmsnorm_fwd_ws(y.data_ptr(), x.data_ptr(), w.data_ptr(), rows, hidden, 1e-6,
                                ws.data_ptr(), need - 16, s) == nf.NF_ERR_WORKSPACE_TOO_SMALL
    assert nf.nf_rmsnorm_fwd_ws(y.data_ptr(), x.data_ptr(), w.data_ptr(), rows, hidden, 1e-6,
                                ws.data_ptr() + 8, need, s) == nf.NF_ERR_MISALIGNED
    assert nf.nf_rmsnorm_fwd_ws(y.data_ptr(), x.data_ptr(), w.data_ptr(), rows, hidden, 1e-6,
                                ws.data_ptr(), need, s) == nf.NF_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0


def test_plain_forward_falls_back_to_the_cluster_family():
    # hidden 65536: automatic plan = grid; without a workspace the plain
    # call runs the cluster kernels (which hold the row) instead
    rows, hidden = 3, 65536
    assert nf.nf_plan_query("rmsnorm_fwd", rows, hidden)["path"] == "grid"
    x, w = workloads.rms_inputs(rows, hidden, seed=21)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    xd, wd = x.cuda(), w.cuda()
    y = torch.empty_like(xd)
    s = torch.cuda.current_stream().cuda_stream
    assert nf.nf_rmsnorm_fwd(y.data_ptr(), xd.data_ptr(), wd.data_ptr(), rows, hidden, 1e-6, s) == \
        nf.NF_OK
    torch.cuda.synchronize()
    check_bf16(y, y_ref, "plain rms fwd at 65536")


# ---------------------------------------------------------------- grid family

@pytest.mark.parametrize("rows,hidden", GRID_FORCED)
def test_grid_fused(rows, hidden):
    # the residual is stored bf16(x + residual), and the output normalizes
    # that stored value; both against the oracle's exact sum
    x, r, w = workloads.fused_inputs(rows, hidden, seed=rows + hidden, residual_scale=4.0)
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-5)
    _, y_rnd, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-5, normalize_rounded=True)
    xd, rd = x.cuda(), r.cuda()
    with nf.forced_path("grid"):
        assert nf.nf_plan_query("fused_add_rmsnorm", rows, hidden)["path"] == "grid"
        nf.fused_add_rmsnorm(xd, rd, w.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(xd, y_ref, f"grid fused {rows}x{hidden}")
    # against the oracle's reading of normalizing the stored residual: one
    # bf16 rounding apart at most
    assert ulp_diff_bf16(xd, oracle.to_bf16(y_rnd)).max() <= 1
    d = ulp_diff_bf16(rd, oracle.to_bf16(s_ref))
    assert d.max() <= 1 and (d > 0).mean() < 1e-3


@pytest.mark.parametrize("rows,hidden", GRID_FORCED)
def test_grid_rmsnorm_fwd_and_in_place(rows, hidden):
    x, w = workloads.rms_inputs(rows, hidden, seed=rows + hidden)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    xd, wd = x.cuda(), w.cuda()
    with nf.forced_path("grid"):
        y = nf.rmsnorm_fwd(xd, wd, 1e-6)
        nf.rmsnorm_fwd(xd, wd, 1e-6, out=xd)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"grid rms {rows}x{hidden}")
    assert torch.equal(xd, y)


@pytest.mark.parametrize("rows,hidden", GRID_FORCED)
def test_grid_layernorm_fwd_and_in_place(rows, hidden):
    # in place too: every CTA reads the row's first element (the shift)
    # before the barrier, so CTA 0 overwriting it afterwards changes nothing
    x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, seed=rows + hidden)
    y_ref, m_ref, r_ref = oracle.layernorm_fwd(x, g, b, 1e-5)
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    with nf.forced_path("grid"):
        y, mean, rstd = nf.layernorm_fwd(xd, gd, bd, 1e-5)
        y2, mean2, rstd2 = nf.layernorm_fwd(xd, gd, bd, 1e-5, out=xd)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"grid ln {rows}x{hidden}")
    check_f32(mean, m_ref, f"grid ln mean {rows}x{hidden}")
    check_f32(rstd, r_ref, f"grid ln rstd {rows}x{hidden}", rtol=1e-4)
    assert torch.equal(y2, y) and torch.equal(mean2, mean) and torch.equal(rstd2, rstd)


@pytest.mark.parametrize("rows,hidden", GRID_FORCED)
def test_grid_layernorm_bwd(rows, hidden):
    x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, seed=rows + hidden)
    _, m, r = oracle.layernorm_fwd(x, np.ones(hidden), np.zeros(hidden), 1e-5)
    mean, rstd = torch.from_numpy(m.astype(np.float32)), torch.from_numpy(r.astype(np.float32))
    dx_ref, dg_ref, db_ref = oracle.layernorm_bwd(dy, x, mean, rstd, g)
    dyd = dy.cuda()
    with nf.forced_path("grid"):
        assert nf.nf_plan_query("layernorm_bwd", rows, hidden)["path"] == "grid"
        dx, dg, db = nf.layernorm_bwd(dyd, x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
        dx2, dg2, db2 = nf.layernorm_bwd(dyd, x.cuda(), mean.cuda(), rstd.cuda(), g.cuda(), out=dyd)
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"grid ln bwd dx {rows}x{hidden}")
    check_f32(dg, dg_ref, f"grid ln bwd dgamma {rows}x{hidden}")
    check_f32(db, db_ref, f"grid ln bwd dbeta {rows}x{hidden}")
    # written over dy, and bit-identical to the first call
    assert torch.equal(dyd, dx) and torch.equal(dg, dg2) and torch.equal(db, db2)


@pytest.mark.parametrize("rows,hidden", GRID_FORCED)
@pytest.mark.parametrize("fused", (False, True))
def test_grid_rmsnorm_bwd(rows, hidden, fused):
    if fused:
        s, w, dy, dres = workloads.fused_bwd_inputs(rows, hidden, seed=rows + hidden)
        dx_ref, dw_ref = oracle.fused_add_rmsnorm_bwd(dy, dres, s, w, 1e-6)
    else:
        s, dy, w = workloads.rms_bwd_inputs(rows, hidden, seed=rows + hidden)
        _, rstd = oracle.rmsnorm_fwd(s, w, 1e-6)
        dx_ref, dw_ref = oracle.rmsnorm_bwd(dy, s, rstd, w)
    dyd = dy.cuda()
    with nf.forced_path("grid"):
        assert nf.nf_plan_query("rmsnorm_bwd", rows, hidden)["path"] == "grid"
        if fused:
            dresd = dres.cuda()
            dx, dw = nf.fused_add_rmsnorm_bwd(dyd, s.cuda(), w.cuda(), dresd, 1e-6)
            dx2, dw2 = nf.fused_add_rmsnorm_bwd(dyd, s.cuda(), w.cuda(), dresd, 1e-6, out=dresd)
            inplace = dresd
        else:
            dx, dw = nf.rmsnorm_bwd(dyd, s.cuda(), w.cuda(), 1e-6)
            dx2, dw2 = nf.rmsnorm_bwd(dyd, s.cuda(), w.cuda(), 1e-6, out=dyd)
            inplace = dyd
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"grid rms bwd dx {rows}x{hidden} fused={fused}")
    check_f32(dw, dw_ref, f"grid rms bwd dw {rows}x{hidden} fused={fused}")
    assert torch.equal(inplace, dx) and torch.equal(dw, dw2)


def test_grid_refuses_rows_that_do_not_fit():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for op in ("rmsnorm_fwd", "layernorm_bwd"):
        assert nf.nf_plan_compute(op, 9, 8192, sms, "grid")[0] == nf.NF_ERR_UNSUPPORTED_PATH
        assert nf.nf_plan_compute(op, 8, 1 << 22, sms, "grid")[0] == nf.NF_ERR_UNSUPPORTED_PATH
        assert nf.nf_plan_compute(op, 8, 1 << 21, sms, "grid")[0] == nf.NF_OK
    x, w = workloads.rms_inputs(9, 1024, seed=3)
    with nf.forced_path("grid"):
        with pytest.raises(nf.NFError) as e:
            nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
    assert e.value.status == nf.NF_ERR_UNSUPPORTED_PATH


def test_grid_barrier_wait_runs_out_and_context_survives():
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert nf.nf_get_device_status(s) == nf.NF_OK
    assert nf.nf_selftest_grid_timeout(0, 2_000_000, s) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_selftest_grid_timeout(ws.data_ptr() + 8, 2_000_000, s) == nf.NF_ERR_MISALIGNED
    assert nf.nf_selftest_grid_timeout(ws.data_ptr(), 2_000_000, s) == nf.NF_OK  # 2 ms
    assert nf.nf_get_device_status(s) == nf.NF_ERR_TIMEOUT
    assert nf.nf_get_device_status(s) == nf.NF_OK
    # both CTAs arrived before giving up
    assert int(ws[:4].view(torch.int32).item()) == 2
    # the context still works, on the grid family itself
    x, w = workloads.rms_inputs(4, 1 << 16, seed=4)
    with nf.forced_path("grid"):
        y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(y, oracle.rmsnorm_fwd(x, w, 1e-6)[0], "grid after timeout")


@pytest.mark.parametrize("family", ("grid", "split"))
def test_long_rows_degenerate_cases(family):
    # a constant LayerNorm row (var = 0: y = beta exactly, rstd = 1/sqrt(eps)),
    # an all-zero RMSNorm row (y = 0), rows scaled by 1e3 and 1e-3, and the
    # fused op with residual = -x (the stored sum is 0, so is the output)
    rows, hidden = 4, 1 << 20
    x = torch.full((rows, hidden), 3.25, dtype=torch.bfloat16)
    _, g, b = workloads.layernorm_fwd_inputs(1, hidden, seed=2)
    with nf.forced_path(family):
        y, mean, rstd = nf.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), b.expand(rows, hidden))
    assert torch.allclose(mean.cpu(), torch.full((rows,), 3.25))
    assert torch.allclose(rstd.cpu(), torch.full((rows,), 1e-5 ** -0.5), rtol=1e-5)

    xr, w = workloads.rms_inputs(rows, hidden, seed=3)
    xr[0] = 0
    xr[1] = (xr[1].float() * 1000).to(torch.bfloat16)
    xr[2] = (xr[2].float() * 1e-3).to(torch.bfloat16)
    y_ref, _ = oracle.rmsnorm_fwd(xr, w, 1e-6)
    with nf.forced_path(family):
        yr = nf.rmsnorm_fwd(xr.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(yr, y_ref, f"long rows rms extremes/{family}")
    assert torch.count_nonzero(yr[0]) == 0

    xf = xr.clone()
    rf = (-xf.float()).to(torch.bfloat16)
    xd, rd = xf.cuda(), rf.cuda()
    with nf.forced_path(family):
        nf.fused_add_rmsnorm(xd, rd, w.cuda(), 1e-6)
    torch.cuda.synchronize()
    assert torch.count_nonzero(rd) == 0 and torch.count_nonzero(xd) == 0
