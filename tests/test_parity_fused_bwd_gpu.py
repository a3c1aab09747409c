"""GPU parity of the fused residual-add + RMSNorm backward against the fp64
oracle, on every kernel family (register, bulk, runtime hidden, cluster),
with and without the residual-stream gradient, and in place."""
import numpy as np
import pytest
import torch

import oracle
import row_normalization_inner_gb300 as nf
import workloads
from gpu_helpers import check_bf16, check_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    nf.set_path("auto")
    yield
    nf.set_path("auto")


def _inputs(rows, hidden, seed):
    return workloads.fused_bwd_inputs(rows, hidden, seed=seed)


CASES = [("reg", 1024), ("reg", 4096), ("reg", 8192), ("bulk", 1024), ("bulk", 5120),
         ("bulk", 12288), ("dynamic", 3072), ("dynamic", 4096), ("cluster", 65536),
         ("cluster", 2048)]


@pytest.mark.parametrize("path,hidden", CASES)
@pytest.mark.parametrize("with_dres", (True, False))
def test_fused_bwd(path, hidden, with_dres):
    rows = 3 if path == "cluster" else 300
    s, w, dy, dres = _inputs(rows, hidden, seed=hidden + rows)
    ds_ref, dw_ref = oracle.fused_add_rmsnorm_bwd(dy, dres if with_dres else None, s, w, 1e-6)
    with nf.forced_path(path):
        assert nf.nf_plan_query("rmsnorm_bwd", rows, hidden)["path"] == path
        dx, dw = nf.fused_add_rmsnorm_bwd(dy.cuda(), s.cuda(), w.cuda(),
                                          dres.cuda() if with_dres else None, 1e-6)
        dx2, dw2 = nf.fused_add_rmsnorm_bwd(dy.cuda(), s.cuda(), w.cuda(),
                                            dres.cuda() if with_dres else None, 1e-6)
    torch.cuda.synchronize()
    check_bf16(dx, ds_ref, f"fused bwd dx {path} {rows}x{hidden}")
    check_f32(dw, dw_ref, f"fused bwd dw {path} {rows}x{hidden}")
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2)


@pytest.mark.parametrize("target", ("dres", "dy"))
def test_fused_bwd_in_place(target):
    rows, hidden = 257, 4096
    s, w, dy, dres = _inputs(rows, hidden, seed=11)
    ds_ref, dw_ref = oracle.fused_add_rmsnorm_bwd(dy, dres, s, w, 1e-6)
    dyd, dresd = dy.cuda(), dres.cuda()
    out = dresd if target == "dres" else dyd
    dx, dw = nf.fused_add_rmsnorm_bwd(dyd, s.cuda(), w.cuda(), dresd, 1e-6, out=out)
    torch.cuda.synchronize()
    assert dx.data_ptr() == out.data_ptr()
    check_bf16(out, ds_ref, f"fused bwd in place into {target}")
    check_f32(dw, dw_ref, "fused bwd dw in place")


def test_fused_bwd_full_size_sampled_rows():
    # the prefill batch: the whole call on the GPU, sampled rows against the oracle
    rows, hidden = 16384, 8192
    s, w, dy, dres = _inputs(rows, hidden, seed=5)
    dx, dw = nf.fused_add_rmsnorm_bwd(dy.cuda(), s.cuda(), w.cuda(), dres.cuda(), 1e-6)
    torch.cuda.synchronize()
    idx = np.random.default_rng(0).choice(rows, 64, replace=False)
    ds_ref, _ = oracle.fused_add_rmsnorm_bwd(dy[idx], dres[idx], s[idx], w, 1e-6)
    check_bf16(dx.cpu()[idx], ds_ref, "fused bwd sampled rows")
    _, dw_ref = oracle.fused_add_rmsnorm_bwd(dy, dres, s, w, 1e-6)
    check_f32(dw, dw_ref, "fused bwd dw full size")
