"""GPU parity of the grid-parallel cluster kernels (runtime hidden) for long
rows against the fp64 oracle: forward hidden up to 262144, backward up to
131072, plus shorter sizes, all forced onto the cluster family."""
import numpy as np
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32, ulp_diff_bf16

pytestmark = pytest.mark.gpu

FWD_LONG = (32776, 65536, 100008, 262144)
BWD_LONG = (16392, 65536, 131072)
FORCED = (264, 3072, 8192)   # non-compiled, non-compiled, compiled (backward only)


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    nf.set_path("auto")
    yield
    nf.set_path("auto")


def _path(hidden, bwd):
    # the automatic choice for long rows is the split family (measured
    # faster); the cluster kernels are forced here
    return "cluster"


@pytest.mark.parametrize("hidden", FWD_LONG + FORCED[:2])
@pytest.mark.parametrize("rows", (1, 5, 64))
def test_long_fused(rows, hidden):
    x, r, w = workloads.fused_inputs(rows, hidden, seed=hidden + rows, residual_scale=4.0)
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-5)
    xd, rd = x.cuda(), r.cuda()
    with nf.forced_path(_path(hidden, False)):
        assert nf.nf_plan_query("fused_add_rmsnorm", rows, hidden)["path"] == "cluster"
        nf.fused_add_rmsnorm(xd, rd, w.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(xd, y_ref, f"long fused {rows}x{hidden}")
    d = ulp_diff_bf16(rd, oracle.to_bf16(s_ref))
    assert d.max() <= 1 and (d > 0).mean() < 1e-3


@pytest.mark.parametrize("hidden", FWD_LONG + FORCED[:2])
@pytest.mark.parametrize("rows", (1, 5, 64))
def test_long_rmsnorm_fwd(rows, hidden):
    x, w = workloads.rms_inputs(rows, hidden, seed=hidden + rows)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    with nf.forced_path(_path(hidden, False)):
        y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"long rms {rows}x{hidden}")


@pytest.mark.parametrize("hidden", FWD_LONG + FORCED[:2])
@pytest.mark.parametrize("rows", (1, 5, 64))
def test_long_layernorm_fwd(rows, hidden):
    x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, seed=hidden + rows)
    y_ref, m_ref, r_ref = oracle.layernorm_fwd(x, g, b, 1e-5)
    with nf.forced_path(_path(hidden, False)):
        y, mean, rstd = nf.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"long ln {rows}x{hidden}")
    check_f32(mean, m_ref, f"long ln mean {rows}x{hidden}")
    check_f32(rstd, r_ref, f"long ln rstd {rows}x{hidden}", rtol=1e-4)


@pytest.mark.parametrize("hidden", BWD_LONG + FORCED)
@pytest.mark.parametrize("rows", (3, 200))
def test_long_layernorm_bwd(rows, hidden):
    x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, seed=hidden + rows)
    _, m, r = oracle.layernorm_fwd(x, np.ones(hidden), np.zeros(hidden), 1e-5)
    mean, rstd = torch.from_numpy(m.astype(np.float32)), torch.from_numpy(r.astype(np.float32))
    dx_ref, dg_ref, db_ref = oracle.layernorm_bwd(dy, x, mean, rstd, g)
    with nf.forced_path(_path(hidden, True)):
        assert nf.nf_plan_query("layernorm_bwd", rows, hidden)["path"] == "cluster"
        dx, dg, db = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
        dx2, dg2, db2 = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"long ln bwd dx {rows}x{hidden}")
    check_f32(dg, dg_ref, f"long ln bwd dgamma {rows}x{hidden}")
    check_f32(db, db_ref, f"long ln bwd dbeta {rows}x{hidden}")
    assert torch.equal(dg, dg2) and torch.equal(db, db2)


@pytest.mark.parametrize("hidden", BWD_LONG + FORCED)
@pytest.mark.parametrize("rows", (3, 200))
def test_long_rmsnorm_bwd(rows, hidden):
    x, dy, w = workloads.rms_bwd_inputs(rows, hidden, seed=hidden + rows)
    _, rstd = oracle.rmsnorm_fwd(x, w, 1e-6)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(dy, x, rstd, w)
    with nf.forced_path(_path(hidden, True)):
        dx, dw = nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"long rms bwd dx {rows}x{hidden}")
    check_f32(dw, dw_ref, f"long rms bwd dw {rows}x{hidden}")
