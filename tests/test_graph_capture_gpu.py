"""Every entry point captured into a CUDA graph and replayed gives the
eager result bit for bit (the kernels are launched as programmatic
dependents, so the captured graph carries programmatic edges), and calls
issued on two streams at once give the results of calls issued one after
another."""
import pytest
import torch

import row_normalization_inner_gb300 as nf
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    nf.set_path("auto")
    yield
    nf.set_path("auto")


def _ops(rows, hidden, dev="cuda"):
    """(name, fn) pairs: each fn runs one call on the current stream and
    returns the output tensors; inputs are preallocated so the calls can be
    captured."""
    x, r, w = workloads.fused_inputs(rows, hidden, seed=1, device=dev)
    lx, g, b = workloads.layernorm_fwd_inputs(rows, hidden, seed=2, device=dev)
    bx, dy, bg = workloads.layernorm_bwd_inputs(rows, hidden, seed=3, device=dev)
    _, mean, rstd = nf.layernorm_fwd(bx, bg, torch.zeros_like(bg), 1e-5)
    s, fw, fdy, dres = workloads.fused_bwd_inputs(rows, hidden, seed=4, device=dev)
    ox, odyo, og, ob = workloads.outer_inputs(rows, hidden, seed=5, device=dev)
    _, om, orr = nf.outer_norm_fwd(ox, og, ob, 1e-5)
    y = torch.empty_like(x)
    ws_ln = torch.empty(max(nf.nf_layernorm_bwd_workspace_size(rows, hidden), 16), dtype=torch.uint8, device=dev)
    ws_rms = torch.empty(max(nf.nf_rmsnorm_bwd_workspace_size(rows, hidden), 16), dtype=torch.uint8, device=dev)
    ws_out = torch.empty(max(nf.nf_outer_norm_workspace_size(rows, hidden), 16), dtype=torch.uint8, device=dev)
    ws_fwd = torch.empty(max([nf.nf_workspace_size(op, rows, hidden) for op in range(3)] + [16]),
                         dtype=torch.uint8, device=dev)
    xf, rf = x.clone(), r.clone()

    def fused():
        xf.copy_(x)
        rf.copy_(r)
        nf.fused_add_rmsnorm(xf, rf, w, 1e-6, workspace=ws_fwd)
        return xf, rf

    return [
        ("fused_add_rmsnorm", fused),
        ("rmsnorm_fwd", lambda: (nf.rmsnorm_fwd(x, w, 1e-6, out=y, workspace=ws_fwd),)),
        ("layernorm_fwd", lambda: nf.layernorm_fwd(lx, g, b, 1e-5, workspace=ws_fwd)),
        ("layernorm_bwd", lambda: nf.layernorm_bwd(dy, bx, mean, rstd, bg, workspace=ws_ln)),
        ("rmsnorm_bwd", lambda: nf.rmsnorm_bwd(dy, bx, bg, 1e-6, workspace=ws_rms)),
        ("fused_add_rmsnorm_bwd", lambda: nf.fused_add_rmsnorm_bwd(fdy, s, fw, dres, 1e-6, workspace=ws_rms)),
        ("outer_norm_fwd", lambda: nf.outer_norm_fwd(ox, og, ob, 1e-5, workspace=ws_out)),
        ("outer_norm_bwd", lambda: nf.outer_norm_bwd(odyo, ox, om, orr, og, workspace=ws_out)),
    ]


@pytest.mark.parametrize("rows,hidden,path", [(300, 4096, "auto"), (1000, 1024, "bulk"),
                                              (64, 3000, "auto"), (3, 70000, "auto"),
                                              (5, 8192, "split")])
def test_graph_replay_matches_eager(rows, hidden, path):
    with nf.forced_path(path):
        for name, fn in _ops(rows, hidden):
            if path != "auto" and name.startswith("outer"):
                continue
            eager = [t.clone() for t in fn()]
            torch.cuda.synchronize()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                fn()  # warm the allocator on the capture stream
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=s):
                    outs = fn()
            for _ in range(2):
                g.replay()
            torch.cuda.synchronize()
            for e, o in zip(eager, outs):
                assert torch.equal(e, o), (name, rows, hidden, path)


def test_two_streams_at_once_match_one_after_another():
    rows, hidden = 2048, 4096
    a = workloads.layernorm_bwd_inputs(rows, hidden, seed=7, device="cuda")
    b = workloads.layernorm_bwd_inputs(rows, hidden, seed=8, device="cuda")
    stats = [nf.layernorm_fwd(x, g, torch.zeros_like(g), 1e-5)[1:] for (x, _, g) in (a, b)]
    ref = [nf.layernorm_bwd(dy, x, m, r, g) for (x, dy, g), (m, r) in zip((a, b), stats)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    outs = []
    for (x, dy, g), (m, r), s in zip((a, b), stats, (s1, s2)):
        ws = torch.empty(nf.nf_layernorm_bwd_workspace_size(rows, hidden), dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(s):
            outs.append(nf.layernorm_bwd(dy, x, m, r, g, workspace=ws, stream=s) + (ws,))
    torch.cuda.synchronize()
    for (dx, dg, db, _), (rdx, rdg, rdb) in zip(outs, ref):
        assert torch.equal(dx, rdx) and torch.equal(dg, rdg) and torch.equal(db, rdb)
