"""The LayerNorm backward entry point that allocates nothing.

Some callers cannot allocate device memory where they run the backward
pass (inside regions where the framework's allocator must not be entered,
plugins that only get pre-allocated buffers, latency-critical code that
cannot take cudaMalloc's synchronization).  nf_layernorm_bwd_noalloc serves
them from a fixed scratch area inside the library.  This checks, through
the C ABI, that on several calls in a row it returns exactly what
nf_layernorm_bwd returns with a caller-owned workspace (the same kernels
on the same plan, so bit for bit) and that both agree with the fp64
oracle, including long rows on the grid family; and that a size needing
more scratch than the area is refused before anything runs.  Named to be
collected last."""
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    nf.set_path("auto")
    yield
    nf.set_path("auto")


def _case(rows, hidden, seed):
    x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, seed=seed, device="cuda")
    _, mean, rstd = nf.layernorm_fwd(x, g, torch.zeros_like(g), 1e-5)
    return x, dy, g, mean, rstd


def _noalloc(dx, dg, db, dy, x, mean, rstd, g, rows, hidden):
    return nf.nf_layernorm_bwd_noalloc(dx.data_ptr(), dg.data_ptr(), db.data_ptr(), dy.data_ptr(),
                                       x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), g.data_ptr(),
                                       rows, hidden, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_and_oracle():
    # calls in a row with different sizes and data: the shared scratch area
    # must carry nothing from one call into the next.  Hidden 12288 has the
    # largest partials of the compiled sizes (one slot per SM).
    for call, (rows, hidden) in enumerate(((4096, 4096), (1000, 8192), (300, 1024), (2048, 12288))):
        x, dy, g, mean, rstd = _case(rows, hidden, seed=100 + call)
        dx_ref, dg_ref, db_ref = nf.layernorm_bwd(dy, x, mean, rstd, g)
        dx = torch.empty_like(x)
        dg = torch.empty(hidden, device="cuda")
        db = torch.empty(hidden, device="cuda")
        st = _noalloc(dx, dg, db, dy, x, mean, rstd, g, rows, hidden)
        assert st == nf.NF_OK, nf.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(dx, dx_ref), f"dx differs from the workspace entry point (call {call})"
        assert torch.equal(dg, dg_ref), f"dgamma differs from the workspace entry point (call {call})"
        assert torch.equal(db, db_ref), f"dbeta differs from the workspace entry point (call {call})"
        # and against the fp64 oracle on the same saved statistics
        o_dx, o_dg, o_db = oracle.layernorm_bwd(dy, x, host_f64(mean), host_f64(rstd), g)
        check_bf16(dx, o_dx, f"noalloc dx call {call}")
        check_f32(dg, o_dg, f"noalloc dgamma call {call}")
        check_f32(db, o_db, f"noalloc dbeta call {call}")


def test_noalloc_takes_long_rows_on_the_grid_family():
    # 4 rows of 2^22 elements run on the grid family, whose workspace is the
    # row partials only (rows x SMs float2): they fit the area
    rows, hidden = 4, 1 << 22
    assert nf.nf_plan_query("layernorm_bwd", rows, hidden)["path"] == "grid"
    x, dy, g, mean, rstd = _case(rows, hidden, seed=6)
    dx = torch.empty_like(x)
    dg = torch.empty(hidden, device="cuda")
    db = torch.empty(hidden, device="cuda")
    st = _noalloc(dx, dg, db, dy, x, mean, rstd, g, rows, hidden)
    assert st == nf.NF_OK, nf.status_string(st)
    torch.cuda.synchronize()
    dx_ref, dg_ref, db_ref = nf.layernorm_bwd(dy, x, mean, rstd, g)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx_ref) and torch.equal(dg, dg_ref) and torch.equal(db, db_ref)
    o_dx, o_dg, o_db = oracle.layernorm_bwd(dy, x, host_f64(mean), host_f64(rstd), g)
    check_bf16(dx, o_dx, "noalloc grid dx")
    check_f32(dg, o_dg, "noalloc grid dgamma")
    check_f32(db, o_db, "noalloc grid dbeta")


def test_noalloc_refuses_sizes_beyond_the_area():
    # 9 rows of 2^22 elements run on the split family (more rows than the
    # grid family holds), whose column partials alone are 2 x 2^22 fp32 =
    # 32 MiB per row block: more than the 16 MiB area on any device
    rows, hidden = 9, 1 << 22
    assert nf.nf_plan_query("layernorm_bwd", rows, hidden)["path"] == "split"
    x, dy, g, mean, rstd = _case(rows, hidden, seed=7)
    dx = torch.full_like(x, 5.0)
    dg = torch.full((hidden,), 5.0, device="cuda")
    db = torch.full((hidden,), 5.0, device="cuda")
    st = _noalloc(dx, dg, db, dy, x, mean, rstd, g, rows, hidden)
    torch.cuda.synchronize()
    assert st == nf.NF_ERR_WORKSPACE_TOO_SMALL
    assert torch.all(dg == 5.0) and torch.all(db == 5.0) and torch.all(dx == 5.0)  # nothing ran
