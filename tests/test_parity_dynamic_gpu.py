"""GPU parity of the runtime-hidden (dynamic) kernels against the fp64
oracle: hidden sizes outside the compiled set (any multiple of 8), and the
compiled sizes forced onto the dynamic kernels."""
import numpy as np
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32, ulp_diff_bf16

pytestmark = pytest.mark.gpu

FWD_HIDDEN = (8, 264, 768, 1000, 3072, 6144, 14336, 32768)
BWD_HIDDEN = (8, 264, 768, 1000, 2056, 3072, 6144, 6152, 16384)   # 2056 / 6152: the first sizes with two / four vectors per thread
ROWS = (1, 37, 300)


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    nf.set_path("auto")
    yield
    nf.set_path("auto")


def _path_for(hidden):
    return "dynamic" if hidden in nf.HIDDEN_SET else "auto"


@pytest.mark.parametrize("hidden", FWD_HIDDEN + (1024, 8192))
@pytest.mark.parametrize("rows", ROWS)
def test_dynamic_fused(rows, hidden):
    x, r, w = workloads.fused_inputs(rows, hidden, seed=rows + hidden, residual_scale=4.0)
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-5)
    xd, rd = x.cuda(), r.cuda()
    with nf.forced_path(_path_for(hidden)):
        assert nf.nf_plan_query("fused_add_rmsnorm", rows, hidden)["path"] == "dynamic"
        nf.fused_add_rmsnorm(xd, rd, w.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(xd, y_ref, f"dyn fused {rows}x{hidden}")
    d = ulp_diff_bf16(rd, oracle.to_bf16(s_ref))
    assert d.max() <= 1 and (d > 0).mean() < 1e-3


@pytest.mark.parametrize("hidden", FWD_HIDDEN + (1024, 8192))
@pytest.mark.parametrize("rows", ROWS)
def test_dynamic_rmsnorm_fwd(rows, hidden):
    x, w = workloads.rms_inputs(rows, hidden, seed=rows + hidden)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    with nf.forced_path(_path_for(hidden)):
        y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"dyn rms {rows}x{hidden}")


@pytest.mark.parametrize("hidden", FWD_HIDDEN + (1024, 8192))
@pytest.mark.parametrize("rows", ROWS)
def test_dynamic_layernorm_fwd(rows, hidden):
    x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, seed=rows + hidden)
    y_ref, m_ref, r_ref = oracle.layernorm_fwd(x, g, b, 1e-5)
    with nf.forced_path(_path_for(hidden)):
        y, mean, rstd = nf.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"dyn ln {rows}x{hidden}")
    check_f32(mean, m_ref, f"dyn ln mean {rows}x{hidden}")
    check_f32(rstd, r_ref, f"dyn ln rstd {rows}x{hidden}", rtol=1e-4)


@pytest.mark.parametrize("hidden", (24, 264, 1000))
def test_dynamic_fwd_ring_walks_many_rows(hidden):
    # rows of one warp run as one wave of 32 resident CTAs per SM that walk
    # the rows through a two-stage copy ring: with more rows than CTAs each
    # CTA takes several rows, the stages alternate, and the last rows of the
    # walk leave empty copy groups behind
    rows = 10007
    for op in ("rmsnorm_fwd", "layernorm_fwd", "fused_add_rmsnorm"):
        p = nf.nf_plan_query(op, rows, hidden)
        assert p["path"] == "dynamic" and p["block"] == 32
        if op == "fused_add_rmsnorm" and hidden > 512:  # more than 2 KB of inputs a row: no ring
            assert p["smem_bytes"] == 0 and p["grid"] == rows
        else:
            assert p["smem_bytes"] > 0 and rows > p["grid"] > rows // 4
    x, r, w = workloads.fused_inputs(rows, hidden, seed=hidden + 10, residual_scale=4.0)
    s_ref, y_ref, _ = oracle.fused_add_rmsnorm(x, r, w, 1e-5)
    xd, rd = x.cuda(), r.cuda()
    nf.fused_add_rmsnorm(xd, rd, w.cuda(), 1e-5)  # in place: x becomes y, r the sum
    torch.cuda.synchronize()
    check_bf16(xd, y_ref, f"dyn fused ring {rows}x{hidden}")
    d = ulp_diff_bf16(rd, oracle.to_bf16(s_ref))
    assert d.max() <= 1 and (d > 0).mean() < 1e-3
    x, w = workloads.rms_inputs(rows, hidden, seed=hidden + 11)
    y_ref, _ = oracle.rmsnorm_fwd(x, w, 1e-6)
    y = nf.rmsnorm_fwd(x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"dyn rms ring {rows}x{hidden}")
    x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, seed=hidden + 12)
    y_ref, m_ref, r_ref = oracle.layernorm_fwd(x, g, b, 1e-5)
    xd = x.cuda()
    y, mean, rstd = nf.layernorm_fwd(xd, g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_bf16(y, y_ref, f"dyn ln ring {rows}x{hidden}")
    check_f32(mean, m_ref, f"dyn ln ring mean {rows}x{hidden}")
    check_f32(rstd, r_ref, f"dyn ln ring rstd {rows}x{hidden}", rtol=1e-4)
    # in place: y over x (each row is read, through the ring, before it is written)
    nf.layernorm_fwd(xd, g.cuda(), b.cuda(), 1e-5, out=xd)
    torch.cuda.synchronize()
    assert torch.equal(xd, y)


@pytest.mark.parametrize("hidden", BWD_HIDDEN + (1024, 8192))
@pytest.mark.parametrize("rows", ROWS + (2000,))
def test_dynamic_layernorm_bwd(rows, hidden):
    x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, seed=rows + hidden)
    _, m, r = oracle.layernorm_fwd(x, np.ones(hidden), np.zeros(hidden), 1e-5)
    mean, rstd = torch.from_numpy(m.astype(np.float32)), torch.from_numpy(r.astype(np.float32))
    dx_ref, dg_ref, db_ref = oracle.layernorm_bwd(dy, x, mean, rstd, g)
    with nf.forced_path(_path_for(hidden)):
        dx, dg, db = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
        dx2, dg2, db2 = nf.layernorm_bwd(dy.cuda(), x.cuda(), mean.cuda(), rstd.cuda(), g.cuda())
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"dyn ln bwd dx {rows}x{hidden}")
    check_f32(dg, dg_ref, f"dyn ln bwd dgamma {rows}x{hidden}")
    check_f32(db, db_ref, f"dyn ln bwd dbeta {rows}x{hidden}")
    assert torch.equal(dg, dg2) and torch.equal(db, db2) and torch.equal(dx, dx2)


@pytest.mark.parametrize("hidden", BWD_HIDDEN + (1024, 8192))
@pytest.mark.parametrize("rows", ROWS + (2000,))
def test_dynamic_rmsnorm_bwd(rows, hidden):
    x, dy, w = workloads.rms_bwd_inputs(rows, hidden, seed=rows + hidden)
    _, rstd = oracle.rmsnorm_fwd(x, w, 1e-6)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(dy, x, rstd, w)
    with nf.forced_path(_path_for(hidden)):
        dx, dw = nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-6)
        dx2, dw2 = nf.rmsnorm_bwd(dy.cuda(), x.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(dx, dx_ref, f"dyn rms bwd dx {rows}x{hidden}")
    check_f32(dw, dw_ref, f"dyn rms bwd dw {rows}x{hidden}")
    # fixed-order sums (with more than 256 partial slots at 2000 rows the
    # column reduction splits each column over four warps): bit-identical
    assert torch.equal(dw, dw2) and torch.equal(dx, dx2)


@pytest.mark.parametrize("hidden", (264, 3072, 14336))
def test_dynamic_degenerate_rows(hidden):
    # a constant LayerNorm row: var = 0, so y = beta exactly and rstd =
    # 1/sqrt(eps); an all-zero RMSNorm row gives y = 0; rows scaled by 1e3
    # and 1e-3 stay within the tolerance
    rows = 3
    x = torch.full((rows, hidden), -1.5, dtype=torch.bfloat16)
    _, g, b = workloads.layernorm_fwd_inputs(1, hidden, seed=hidden)
    y, mean, rstd = nf.layernorm_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert nf.nf_plan_query("layernorm_fwd", rows, hidden)["path"] == "dynamic"
    assert torch.equal(y.cpu(), b.expand(rows, hidden))
    assert torch.allclose(mean.cpu(), torch.full((rows,), -1.5))
    assert torch.allclose(rstd.cpu(), torch.full((rows,), 1e-5 ** -0.5), rtol=1e-5)
    xr, w = workloads.rms_inputs(rows, hidden, seed=hidden + 1)
    xr[0] = 0
    xr[1] = (xr[1].float() * 1000).to(torch.bfloat16)
    xr[2] = (xr[2].float() * 1e-3).to(torch.bfloat16)
    y_ref, _ = oracle.rmsnorm_fwd(xr, w, 1e-6)
    yr = nf.rmsnorm_fwd(xr.cuda(), w.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_bf16(yr, y_ref, f"dynamic rms extremes {hidden}")
    assert torch.count_nonzero(yr[0]) == 0
