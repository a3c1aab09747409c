"""GPU parity of the split family (a row over any number of CTAs, row
statistics through the workspace) against the fp64 oracle: forced at short
and ragged rows, automatic beyond the cluster limits, more rows than one
grid dimension holds, and the workspace rules of the forward calls."""
import numpy as np
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32, ulp_diff_bf16

pytestmark = pytest.mark.gpu

FORCED = ((5, 8), (300, 1000), (33, 8200), (7, 20000))   # (rows, hidden); 8200 = two chunks, ragged
AUTO_FWD = ((2, 262152), (1, 1 << 20))
AUTO_BWD = ((3, 131080), (2, 1 << 20), (2, 1 << 22))   # the last: one row block (no column reduction)
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


@pytest.mark.parametrize("rows,hidden", FORCED + AUTO_FWD)
def test_split_fused(rows, hidden):
    x, r, w = workloads.fused_inputs(rows, hidden, seed=rows + hidden, residual_scale=4.0)
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-5)
    xd, rd = x.cuda(), r.cuda()
    with nf.forced_path(_path(rows, hidden, "f")):
        assert nf.nf_plan_query("fused_add_rmsnorm", rows, hidden)["path"] == "split"
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
        assert nf.nf_plan_query("layernorm_bwd", rows, hidden)["path"] == "split"
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
        assert nf.nf_plan_query("rmsnorm_bwd", rows, hidden)["path"] == "split"
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
    # hidden 65536: automatic plan = split; without a workspace the plain
    # call runs the cluster kernels (which hold the row) instead
    rows, hidden = 3, 65536
    assert nf.nf_plan_query("rmsnorm_fwd", rows, hidden)["path"] == "split"
    x, w = workloads.rms_inputs(rows, hidden, seed=21)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    xd, wd = x.cuda(), w.cuda()
    y = torch.empty_like(xd)
    s = torch.cuda.current_stream().cuda_stream
    assert nf.nf_rmsnorm_fwd(y.data_ptr(), xd.data_ptr(), wd.data_ptr(), rows, hidden, 1e-6, s) == \
        nf.NF_OK
    torch.cuda.synchronize()
    check_bf16(y, y_ref, "plain rms fwd at 65536")
