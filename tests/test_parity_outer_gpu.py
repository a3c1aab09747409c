"""GPU parity of the outer (per-column) normalization kernels against the
fp64 oracle: column tiles with a ragged tail, row stripes of uneven length,
a single row, and determinism of the column sums.  The forward has two
forms: the three-launch streaming passes (the automatic choice; also under
a forced split family) and the single launch with the row stripes on chip
(forced with the grid family), both checked at every shape."""
import numpy as np
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32

pytestmark = pytest.mark.gpu

HIDDEN = (8, 264, 1000, 4096, 4104)
ROWS = (1, 7, 300, 5000)


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    yield


@pytest.mark.parametrize("form", ("split", "grid"))
@pytest.mark.parametrize("hidden", HIDDEN)
@pytest.mark.parametrize("rows", ROWS)
def test_outer_fwd(rows, hidden, form):
    x, _, g, b = workloads.outer_inputs(rows, hidden, seed=rows * 7 + hidden)
    y_ref, m_ref, r_ref = oracle.outer_norm_fwd(x, g, b, 1e-5)
    args = (x.cuda(), g.cuda(), b.cuda(), 1e-5)
    with nf.forced_path(form):
        y, mean, rstd = nf.outer_norm_fwd(*args)
        y2, mean2, rstd2 = nf.outer_norm_fwd(*args)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"outer fwd y {rows}x{hidden} {form}")
    check_f32(mean, m_ref, f"outer fwd mean {rows}x{hidden} {form}")
    check_f32(rstd, r_ref, f"outer fwd rstd {rows}x{hidden} {form}", rtol=1e-4)
    assert torch.equal(y, y2) and torch.equal(mean, mean2) and torch.equal(rstd, rstd2)


def test_outer_grid_form_refuses_stripes_too_long():
    # 65536 rows: a stripe of 432 rows does not fit two band buffers of the
    # narrowest band (16 vectors), so the grid form is refused
    rows, hidden = 65536, 1024
    x = torch.zeros(rows, hidden, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(hidden, dtype=torch.bfloat16, device="cuda")
    with nf.forced_path("grid"):
        with pytest.raises(nf.NFError) as e:
            nf.outer_norm_fwd(x, g, g, 1e-5)
    assert e.value.status == nf.NF_ERR_UNSUPPORTED_PATH


@pytest.mark.parametrize("hidden", HIDDEN)
@pytest.mark.parametrize("rows", ROWS)
def test_outer_bwd(rows, hidden):
    x, dy, g, b = workloads.outer_inputs(rows, hidden, seed=rows * 11 + hidden)
    _, m, r = oracle.outer_norm_fwd(x, g, b, 1e-5)
    mean, rstd = torch.from_numpy(m.astype(np.float32)), torch.from_numpy(r.astype(np.float32))
    dx_ref, dg_ref, db_ref = oracle.outer_norm_bwd(dy, x, mean, rstd, g)
    args = (dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
    dx, dg, db = nf.outer_norm_bwd(*args)
    dx2, dg2, db2 = nf.outer_norm_bwd(*args)
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"outer bwd dx {rows}x{hidden}")
    check_f32(dg, dg_ref, f"outer bwd dgamma {rows}x{hidden}")
    check_f32(db, db_ref, f"outer bwd dbeta {rows}x{hidden}")
    assert torch.equal(dx, dx2) and torch.equal(dg, dg2) and torch.equal(db, db2)


@pytest.mark.parametrize("form", ("split", "grid"))
def test_outer_in_place(form):
    rows, hidden = 600, 1032
    x, dy, g, b = workloads.outer_inputs(rows, hidden, seed=5)
    y_ref, m_ref, r_ref = oracle.outer_norm_fwd(x, g, b, 1e-5)
    xd = x.cuda()
    with nf.forced_path(form):
        y, mean, rstd = nf.outer_norm_fwd(xd, g.cuda(), b.cuda(), 1e-5, out=xd)
    torch.cuda.synchronize()
    assert y.data_ptr() == xd.data_ptr()
    check_bf16(xd, y_ref, "outer fwd in place")
    mean32, rstd32 = mean.cpu(), rstd.cpu()
    dx_ref, _, _ = oracle.outer_norm_bwd(dy, x, mean32, rstd32, g)
    dyd = dy.cuda()
    nf.outer_norm_bwd(dyd, x.cuda(), mean, rstd, g.cuda(), out=dyd)
    torch.cuda.synchronize()
    check_bf16(dyd, dx_ref, "outer bwd in place")


def test_outer_zero_rows():
    hidden = 64
    x = torch.empty(0, hidden, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(hidden, dtype=torch.bfloat16, device="cuda")
    y, _, _ = nf.outer_norm_fwd(x, g, g, 1e-5)
    mean = torch.zeros(hidden, device="cuda")
    dx, dg, db = nf.outer_norm_bwd(x, x, mean, mean, g)
    torch.cuda.synchronize()
    assert y.numel() == 0 and dx.numel() == 0
    assert torch.count_nonzero(dg).item() == 0 and torch.count_nonzero(db).item() == 0


@pytest.mark.parametrize("rows,hidden", ((65536, 1024), (16384, 4096)))
def test_outer_full_size(rows, hidden):
    x, dy, g, b = workloads.outer_inputs(rows, hidden, seed=3)
    y_ref, m_ref, r_ref = oracle.outer_norm_fwd(x, g, b, 1e-5)
    y, mean, rstd = nf.outer_norm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"outer fwd {rows}x{hidden}")
    check_f32(mean, m_ref, "outer fwd mean")
    check_f32(rstd, r_ref, "outer fwd rstd", rtol=1e-4)
    mean32, rstd32 = torch.from_numpy(m_ref.astype(np.float32)), torch.from_numpy(r_ref.astype(np.float32))
    dx_ref, dg_ref, db_ref = oracle.outer_norm_bwd(dy, x, mean32, rstd32, g)
    dx, dg, db = nf.outer_norm_bwd(dy.cuda(), x.cuda(), mean32.cuda(), rstd32.cuda(), g.cuda())
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"outer bwd dx {rows}x{hidden}")
    check_f32(dg, dg_ref, "outer bwd dgamma")
    check_f32(db, db_ref, "outer bwd dbeta")


@pytest.mark.parametrize("rows,hidden", ((16384, 4104), (40000, 1000)))
def test_outer_large(rows, hidden):
    # inputs of 134 / 80 MB per tensor (several column tiles with a ragged
    # last one; 152 and 38 row stripes), forward and backward
    x, dy, g, b = workloads.outer_inputs(rows, hidden, seed=rows + hidden)
    y_ref, m_ref, r_ref = oracle.outer_norm_fwd(x, g, b, 1e-5)
    y, mean, rstd = nf.outer_norm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"outer large fwd y {rows}x{hidden}")
    check_f32(mean, m_ref, f"outer large fwd mean {rows}x{hidden}")
    check_f32(rstd, r_ref, f"outer large fwd rstd {rows}x{hidden}", rtol=1e-4)
    m32, r32 = torch.from_numpy(m_ref.astype(np.float32)), torch.from_numpy(r_ref.astype(np.float32))
    dx_ref, dg_ref, db_ref = oracle.outer_norm_bwd(dy, x, m32, r32, g)
    dx, dg, db = nf.outer_norm_bwd(dy.cuda(), x.cuda(), m32.cuda(), r32.cuda(), g.cuda())
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"outer large bwd dx {rows}x{hidden}")
    check_f32(dg, dg_ref, f"outer large bwd dgamma {rows}x{hidden}")
    check_f32(db, db_ref, f"outer large bwd dbeta {rows}x{hidden}")
