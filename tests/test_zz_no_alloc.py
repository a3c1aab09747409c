"""The LayerNorm backward entry point that allocates nothing.

Some callers cannot allocate device memory where they run the backward
pass (inside regions where the framework's allocator must not be entered,
plugins that only get pre-allocated buffers, latency-critical code that
cannot take cudaMalloc's synchronization).  nf_layernorm_bwd_noalloc serves
them from a fixed scratch area inside the library.  This checks, through
the C ABI, that it gives the same results as nf_layernorm_bwd with a
caller-owned workspace on two calls in a row, and that a size needing more
scratch than the area is refused.  Named to be collected last."""
import pytest
import torch

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


def _need(rows, hidden):
    """Scratch bytes the plan of this call uses: partial slots x 2 planes x hidden fp32."""
    return nf.nf_plan_query("layernorm_bwd", rows, hidden)["partials"] * 2 * hidden * 4


def _case(rows, hidden, seed):
    x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, seed=seed, device="cuda")
    _, mean, rstd = nf.layernorm_fwd(x, g, torch.zeros_like(g), 1e-5)
    return x, dy, g, mean, rstd


def test_noalloc_matches_workspace_entry_point_twice():
    s = torch.cuda.current_stream().cuda_stream
    # two calls in a row, different sizes and data: the shared scratch area
    # must carry nothing from one call into the next
    for call, (rows, hidden) in enumerate(((4096, 4096), (1000, 8192))):
        x, dy, g, mean, rstd = _case(rows, hidden, seed=100 + call)
        assert _need(rows, hidden) <= nf.NOALLOC_SCRATCH_BYTES
        dx_ref, dg_ref, db_ref = nf.layernorm_bwd(dy, x, mean, rstd, g)
        dx = torch.empty_like(x)
        dg = torch.empty(hidden, device="cuda")
        db = torch.empty(hidden, device="cuda")
        st = nf.nf_layernorm_bwd_noalloc(dx.data_ptr(), dg.data_ptr(), db.data_ptr(), dy.data_ptr(),
                                         x.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                                         g.data_ptr(), rows, hidden, s)
        assert st == nf.NF_OK, nf.status_string(st)
        torch.cuda.synchronize()
        check_bf16(dx, host_f64(dx_ref), f"noalloc dx call {call}")
        check_f32(dg, host_f64(dg_ref), f"noalloc dgamma call {call}")
        check_f32(db, host_f64(db_ref), f"noalloc dbeta call {call}")


def test_noalloc_refuses_sizes_beyond_the_area():
    # the runtime-hidden backward at hidden 16384 needs more partial space
    # than the fixed area on a full GPU
    rows, hidden = 4096, 16384
    if _need(rows, hidden) <= nf.NOALLOC_SCRATCH_BYTES:
        pytest.skip("this device needs no more than the area at hidden 16384")
    x, dy, g, mean, rstd = _case(rows, hidden, seed=7)
    dx = torch.full_like(x, 5.0)
    dg = torch.full((hidden,), 5.0, device="cuda")
    db = torch.full((hidden,), 5.0, device="cuda")
    st = nf.nf_layernorm_bwd_noalloc(dx.data_ptr(), dg.data_ptr(), db.data_ptr(), dy.data_ptr(),
                                     x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), g.data_ptr(),
                                     rows, hidden, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == nf.NF_ERR_WORKSPACE_TOO_SMALL
    assert torch.all(dg == 5.0) and torch.all(db == 5.0)   # nothing ran
